// internal.h -- shared host/device declarations of the MoE FFN library:
// workspace layout, kernel parameter blocks and launch helpers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

namespace moe {

constexpr int kBM = 128;          // rows per tile = tcgen05 MMA M
constexpr int kBK = 64;           // K elements per pipeline stage (128 B of bf16)
constexpr int kRowPad = 128;      // per-expert row segments are padded to this
constexpr int kMaxExperts = 1024;
constexpr int kRouteTokPerBlock = 256;  // tokens per routing block (default; Workspace::route_tpb)
// From this many routed pairs per token on, the rows of a token are summed in
// fp32 (a [T, D] workspace accumulator, rounded to bf16 once at the end)
// instead of by bf16 reductions into out: each bf16 reduction rounds the
// running sum, and the rounding errors of k adds grow with k.
constexpr int kF32AccumMinK = 9;
inline bool f32_accum(int k) { return k >= kF32AccumMinK; }

// Device-side view of the caller's workspace.  Every region starts on a
// 256-byte boundary; sizes depend only on (T, E, D, H, k, pipeline).
struct Workspace {
  int* err;            // [8]   err[0] error bits, err[1] timeout site
  int* meta;           // [8]   meta[0] = number of 128-row blocks, meta[1] = number of block pairs,
                       //       meta[2], meta[3] = tile counters of the up and down kernels
  int* counts;         // [E]
  int* offsets;        // [E+1] unpadded exclusive scan of counts
  int* pad_offsets;    // [E+1] exclusive scan of counts rounded up to 128
  int* expert_of_rb;   // [max_rb]
  int* pair_info;      // [max_rb] (first row block << 1) | (second block of the same expert exists)
  int* row_tok;        // [S_max] token of each padded slot, -1 for padding
  float* slot_w;       // [S_max] routing weight of each padded slot, 0 for padding
  int* slot_of_pair;   // [P]   unpadded slot of pair p = t*k + j
  int* blk_base;       // [NB*E] per routing block: rank base within each expert
  int* rb_order;       // [max_rb] row blocks ordered by the token band of their first row (down kernels)
  int* pair_order;     // [max_rb] block pairs in the same order
  void* xg;            // [S_max, D] bf16 gathered rows (split pipeline)
  void* act;           // [S_max, H] bf16 activation (split pipeline)
  void* acc_f32;       // [T, D] fp32 reduction target (fused pipeline)
  void* ring;          // fused pipeline on clusters: act exchange ring (bf16, or e4m3)
  void* ring_sf;       // MXFP8 fused pipeline on clusters: scale tiles of the ring
  void* xg_sf;         // MXFP8: scales of xg in blocked 512-byte tiles (S_max * D/32 bytes)
  void* act_sf;        // MXFP8: scales of act in blocked tiles (S_max * H/32 bytes)
  size_t bytes;        // total bytes required
  int64_t S_max;       // padded slot capacity (multiple of 128)
  int max_rb;
  int route_tpb;       // tokens per routing block (MOE_OPT_ROUTE_TPB)
  int route_blocks;
  // Not a region of the workspace: the call's router logits [T, E] fp32 when
  // the call starts from them (moe_ffn_forward_logits), else nullptr.
  const float* router_logits;
  unsigned long long wait_limit_ns;  // bound of every device wait of the call
  float swiglu_limit;                // > 0: clamped SwiGLU (moe_ffn_forward_ex), else plain
  int route_stall_test;              // test hook: one routing block never reaches the grid barrier
  int l2_policy;                     // MOE_OPT_L2_POLICY bits (see api.cu)
  const void* prefetch_base;         // the gather prefetches [base, base + bytes) into L2
  int64_t prefetch_bytes;            //   while the routing finishes (0 = off)
};

// MOE_OPT_ROUTE_COOP: 1 (default) routes problems too large for the
// single-block kernel in one cooperative launch; 0 uses three launches.
extern std::atomic<int> g_route_coop;
// MOE_OPT_ROUTER_FUSED: 1 runs the router inside single-block routing
// launches; 0 (default) always launches it separately.
extern std::atomic<int> g_router_fused;
// MOE_OPT_ROUTE_SMALL_PAIRS: problems of at most this many pairs (and at most
// 256 experts) route in one single-block launch.
extern std::atomic<int64_t> g_route_small_pairs;

// pipeline = kRouteOnly plans only the routing regions (the common prefix of
// every layout).
constexpr int kRouteOnly = -1;
Workspace plan_workspace(void* base, int T, int E, int D, int H, int k, int pipeline, int dtype = 0);

// ----------------------------------------------------------------- kernels
struct GemmArgs {
  const int* meta;          // meta[0] = number of row blocks, meta[1] = number of block pairs
  const int* expert_of_rb;
  const int* pair_info;     // pairs of row blocks of one expert (see Workspace)
  const int* row_tok;
  const float* slot_w;
  void* act;                // up: bf16 [S_max, H] output
  void* out;                // down: bf16 [T, D] reduction target
  float* out_f32;           // down: non-null = fp32 [T, D] reduction target instead of out
  int* err;
  unsigned long long wait_limit_ns;
  int D, H;
  int n_col_tiles;          // column tiles per row block
  int k_blocks;             // reduction length / kBK
  int prefetch;             // k-blocks of L2 prefetch ahead of the smem ring (0 = off)
  int stall_test;           // test hook: the MMA issuer first waits on a barrier nothing arrives on
  const void* x;            // up with the cp.async gather: the token rows [T, D]
  int* tile_counter;        // dynamic tile scheduling: zeroed before the launch; nullptr = static
  const int* counts;        // routed rows per expert and padded segment starts: the
  const int* pad_offsets;   //   row count of each row block (swap-AB tail tiles)
  int swap_ab;              // 1: tail row blocks of <= 112 rows run as swap-AB tiles
  int pair_swap_max;        // CTA-pair down kernel: pairs with at most this many routed rows
                            //   run as swap-AB tiles (0 = never)
  int out_hint;             // 1: reductions into out carry an L2 evict_last hint
  float swiglu_limit;       // > 0: gate clamped to <= limit, up to [-limit, limit] before SwiGLU
  int l2_policy;            // bit 0: weight tiles loaded with an L2 evict_first policy
  const int* pair_order;    // down: nullptr, or the order in which the block pairs are processed
  int half_m128;            // CTA-pair down kernel: a half pair runs as one M = 128 pair MMA (else M = 256,
                            //   the odd CTA recomputing the first block and storing nothing)
  int down_epi8;            // CTA-pair down kernel: eight epilogue warps (else four)
  int up_swap;              // CTA-pair up kernel: half pairs run as swap-AB tiles
};

// Routing; when zero_out != nullptr the first launch also zero-fills
// zero_out[0 .. zero_bytes) (the reduction target of the GEMMs).
// pdl: the second and third routing launches start as programmatic dependents.
// With ws.router_logits set, the routing launch first runs the router over
// those [T, E] logits and writes topk_ids / topk_w (then caller outputs).
cudaError_t launch_route(const Workspace& ws, const int32_t* topk_ids, const float* topk_w, int T, int E, int k,
                         cudaStream_t stream, void* zero_out = nullptr, int64_t zero_bytes = 0, int zero_grid = 0,
                         bool pdl = false);
// Orders of the down projection's tiles by token band (reductions into a
// reduction target larger than L2 then find the rows of one band of tokens
// there): rb_order = the row blocks, pair_order = the block pairs, each sorted
// stably by band(token of its first row) = tok * n_bands / T.  One block,
// launched after the routing.
cudaError_t launch_band_order(const Workspace& ws, int T, int n_bands, cudaStream_t stream);
// The router alone: top-k ids (decreasing logit, ties to the lower id) and the
// softmax of the selected logits, for each of T tokens of logits [T, E].
cudaError_t launch_router_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                               cudaStream_t stream);
// ids_ext / w_ext [T, k + n_shared]: the routed ids and weights of each token,
// then the shared experts E .. E + n_shared - 1 at weight 1.
cudaError_t launch_extend_routing(const int32_t* ids, const float* w, int T, int E, int k, int n_shared,
                                  int32_t* ids_ext, float* w_ext, cudaStream_t stream);
// xg[padded slot of pair p] = x[p / k] for every routed pair, and (when
// out != nullptr) out[0 .. out_bytes) = 0, out_bytes a multiple of 16 * T.
// pdl: launched as a programmatic dependent of the routing launch.
cudaError_t launch_gather_zero(const Workspace& ws, const void* x, const int32_t* topk_ids, int T, int E, int k,
                               int D, void* out, int64_t out_bytes, int grid, cudaStream_t stream, bool pdl);
// gather: 0 = map_a is the pre-gathered xg [S_max, D]; 1 = map_a is x [T, D]
// with one-row boxes and the kernel gathers with TMA gather4; 2 = the kernel's
// cp.async warps gather rows of args.x (map_a unused).
// fold = gate (and up) rows per tile: kUpFold (N = 256) or kUpFoldNarrow (N =
// 128, gather 0 only); map_w1's boxes must be `fold` rows.
// bm = 64: 64-row tiles (gather 0 only; map_a boxes of 64 rows).
cudaError_t launch_up_bf16(const CUtensorMap& map_a, const CUtensorMap& map_w1, const GemmArgs& args, int grid,
                           cudaStream_t stream, int gather, int fold, bool pdl, int bm = kBM);
// Up-projection with two row blocks of one expert per tile sharing each W1
// tile (tiles = block pairs x column tiles).
cudaError_t launch_up_pair_bf16(const CUtensorMap& map_a, const CUtensorMap& map_w1, const GemmArgs& args, int grid,
                                cudaStream_t stream);
// The split GEMMs on CTA pairs (cta_group::2): tiles are (block pair, column
// tile); n_pairs pairs of CTAs are launched as two-CTA clusters.  Up: fold
// 128, map_w1 boxes of 128 rows.  Down: 256-column tiles, map_w2 boxes of 128
// rows.
// map_w1_64: W1 in boxes of 64 rows (the swap-AB half pairs, args.up_swap)
cudaError_t launch_up_pair2_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w1_64,
                                 const GemmArgs& args, int n_pairs, cudaStream_t stream, bool pdl);
cudaError_t launch_down_pair2_bf16(const CUtensorMap& map_act, const CUtensorMap& map_w2, const GemmArgs& args,
                                   int n_pairs, cudaStream_t stream, bool pdl);
// Co-resident two-CTA clusters of the pair kernels on the current device.
int pair_cluster_slots();
// The up projection on CTA pairs in 512-column tiles (act tiles 2g and 2g+1
// of one block pair; args.n_col_tiles = H / 128), map_w1 boxes of 128 rows.
cudaError_t launch_up_pair2_wide_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const GemmArgs& args,
                                      int n_pairs, cudaStream_t stream, bool pdl);
int pair_wide_cluster_slots();
// n = output columns per tile: kDownN, or kDownNNarrow when D % 256 != 0;
// map_w2's boxes must be n rows.
// bm = 64: 64-row tiles (map_act boxes of 64 rows).
cudaError_t launch_down_bf16(const CUtensorMap& map_act, const CUtensorMap& map_w2, const GemmArgs& args, int grid,
                             cudaStream_t stream, bool pdl, int n, int bm = kBM);

struct FusedArgs {
  const int* meta;
  const int* expert_of_rb;
  const int* row_tok;
  const float* slot_w;
  void* out_f32;            // fp32 [T, D], zeroed before the launch
  int* err;
  unsigned long long wait_limit_ns;
  int D, H;
  int n_slices;             // H / 128
  int stall_test;           // test hook (see GemmArgs)
  float swiglu_limit;       // > 0: gate clamped to <= limit, up to [-limit, limit] before SwiGLU
};

cudaError_t launch_fused_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w2,
                              const FusedArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_f32_to_bf16(const void* acc, void* out, int64_t n, int grid, cudaStream_t stream);

// Fused pipeline on clusters of C CTAs (one 128-row block per cluster at a
// time, the activation exchanged through an L2-resident ring).
constexpr int kFusedClusterN = 256;       // GEMM2 output columns per sub-chunk
constexpr int kFusedClusterMaxCtas = 160; // ring capacity: clusters <= this / C
struct FusedClusterArgs {
  const int* meta;
  const int* expert_of_rb;
  const int* row_tok;
  const float* slot_w;
  void* out;                // bf16 [T, D], zeroed before the launch
  void* ring;               // bf16 [n_clusters * 2 * 128, H]
  int* err;
  unsigned long long wait_limit_ns;
  int D, H;
  int csize;                // CTAs per cluster C (1, 2, 4 or 8)
  int h1;                   // act columns per GEMM1 sub-chunk (32, 64, 96 or 128)
  int s1;                   // GEMM1 sub-chunks per CTA: h1 * s1 = H / C
  int s2;                   // GEMM2 sub-chunks per CTA: 256 * s2 = D / C
  int stall_test;           // test hook (see GemmArgs)
  int out_hint;             // 1: reductions into out carry an L2 evict_last hint
  float swiglu_limit;       // > 0: gate clamped to <= limit, up to [-limit, limit] before SwiGLU
};
// Act columns per GEMM1 sub-chunk for cluster size C, or 0 if (D, H) cannot
// run on clusters of C.
inline int fused_cluster_h1(int D, int H, int C) {
  if (C != 1 && C != 2 && C != 4 && C != 8) return 0;
  if (D % (kFusedClusterN * C) || H % C) return 0;
  const int h = H / C;
  for (int h1 : {128, 96, 64, 32})
    if (h % h1 == 0) return h1;
  return 0;
}
inline bool fused_cluster_ok(int D, int H) {
  for (int C : {1, 2, 4, 8})
    if (fused_cluster_h1(D, H, C)) return true;
  return false;
}
// MXFP8 fused pipeline on clusters: act slices of 128 columns (one scale tile
// of K), GEMM2 sub-chunks of 256 output columns.
struct FusedClusterMxArgs {
  const int* meta;
  const int* expert_of_rb;
  const int* row_tok;
  const float* slot_w;
  void* out;                // bf16 [T, D], zeroed before the launch
  void* ring;               // e4m3 [n_clusters * 2 * 128, H]
  void* ring_sf;            // blocked scale tiles of the ring: [n_clusters * 2][H / 128] x 512 B
  const void* xg_sf;        // blocked scale tiles of xg
  const void* w1_sf;        // packed W1 scales
  const void* w2_sf;        // packed W2 scales
  int* err;
  unsigned long long wait_limit_ns;
  int D, H;
  int csize;                // CTAs per cluster C (1, 2, 4 or 8)
  int s1;                   // GEMM1 sub-chunks per CTA: 128 * s1 = H / C
  int s2;                   // GEMM2 sub-chunks per CTA: 256 * s2 = D / C
  int stall_test;           // test hook (see GemmArgs)
  int out_hint;             // 1: reductions into out carry an L2 evict_last hint
  float swiglu_limit;       // > 0: gate clamped to <= limit, up to [-limit, limit] before SwiGLU
};
inline bool fused_cluster_mx_fits(int D, int H, int C) {
  return (C == 1 || C == 2 || C == 4 || C == 8) && D % (256 * C) == 0 && H % (128 * C) == 0;
}
int fused_cluster_mx_max_clusters(int csize);
cudaError_t launch_fused_cluster_mxfp8(const CUtensorMap& map_xg, const CUtensorMap& map_w1,
                                       const CUtensorMap& map_w2, const CUtensorMap& map_ring,
                                       const FusedClusterMxArgs& args, int n_clusters, cudaStream_t stream);

// The fused pipeline on clusters with act kept in shared memory: each CTA's
// act slice (h = H / C columns, a multiple of 64, at most 256) stays in its own
// shared memory and GEMM2's K tiles move between the cluster's CTAs by
// shared-to-shared bulk copies.  h1 / s1 / s2 as for the ring kernel.
inline bool fused_dsmem_fits(int D, int H, int C) {
  if (!fused_cluster_h1(D, H, C)) return false;
  const int h = H / C;
  return h % 64 == 0 && h <= 256;
}
int fused_dsmem_max_clusters(int csize);
cudaError_t launch_fused_dsmem_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w2,
                                    const FusedClusterArgs& args, int n_clusters, cudaStream_t stream);
// Co-resident clusters of size csize on the current device (0 on failure).
int fused_cluster_max_clusters(int csize);
cudaError_t launch_fused_cluster_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w2,
                                      const CUtensorMap& map_ring, const FusedClusterArgs& args, int n_clusters,
                                      cudaStream_t stream);

struct MxArgs {
  const int* meta;
  const int* expert_of_rb;
  const int* row_tok;
  const float* slot_w;
  void* act;                // up: e4m3 [S_max, H] output
  void* act_sf;             // up: blocked scale tiles of act
  void* out;                // down: bf16 [T, D] reduction target
  float* out_f32;           // down: non-null = fp32 [T, D] reduction target instead of out
  const int* rb_order;      // down: nullptr, or the order in which the row blocks are processed
  const int* pair_info;     // CTA-pair kernels: pairs of row blocks of one expert (see Workspace)
  const int* pair_order;    // CTA-pair down kernel: nullptr, or the order of the block pairs
  const float* x_gs;        // NVFP4: global scales of x [1], of W1 and W2 per expert [E], of act [1]
  const float* w1_gs;
  const float* w2_gs;
  const float* act_gs;
  const void* sf_a;         // blocked scale tiles of the A operand
  const void* sf_b;         // blocked scale tiles of the weights
  int* err;
  unsigned long long wait_limit_ns;
  int D, H;
  int n_col_tiles;
  int k_blocks;             // K / 128
  int stall_test;           // test hook (see GemmArgs)
  int out_hint;             // 1: reductions into out carry an L2 evict_last hint
  float swiglu_limit;       // > 0: gate clamped to <= limit, up to [-limit, limit] before SwiGLU
};

// fp4w: the weight maps are MXFP4 (16U4_ALIGN16B tensor maps of packed E2M1 codes).
cudaError_t launch_up_mxfp8(const CUtensorMap& a, const CUtensorMap& w1, const MxArgs& args, int grid,
                            cudaStream_t stream, bool fp4w = false);
cudaError_t launch_down_mxfp8(const CUtensorMap& act, const CUtensorMap& w2, const MxArgs& args, int grid,
                              cudaStream_t stream, bool pdl, bool fp4w = false);
// nv: NVFP4 rows (D/2 bytes of packed codes, D/16 e4m3 scales) instead of MXFP8.
cudaError_t launch_gather_mx(const Workspace& ws, const void* x, const void* x_sf, const int32_t* topk_ids, int T,
                             int E, int k, int D, void* out, int64_t out_bytes, int grid, cudaStream_t stream,
                             bool pdl, bool nv = false);
// NVFP4 split GEMMs (k_blocks = K / 256; the maps read packed codes as bytes).
cudaError_t launch_up_nvfp4(const CUtensorMap& a, const CUtensorMap& w1, const MxArgs& args, int grid,
                            cudaStream_t stream);
cudaError_t launch_down_nvfp4(const CUtensorMap& act, const CUtensorMap& w2, const MxArgs& args, int grid,
                              cudaStream_t stream, bool pdl);
// MXFP8 GEMMs on CTA pairs (cta_group::2): map_a / map_b in boxes of 128 rows,
// sfa / sfb the blocked scale tiles as [tiles, 128] u32 maps (make_map_sf).
cudaError_t launch_up_mxfp8_pair(const CUtensorMap& a, const CUtensorMap& w1, const CUtensorMap& sfa,
                                 const CUtensorMap& sfb, const MxArgs& args, int n_pairs, cudaStream_t stream);
cudaError_t launch_down_mxfp8_pair(const CUtensorMap& act, const CUtensorMap& w2, const CUtensorMap& sfa,
                                   const CUtensorMap& sfb, const MxArgs& args, int n_pairs, cudaStream_t stream,
                                   bool pdl);
// co-resident two-CTA clusters of the MXFP8 pair kernels (0 on error)
int mx_pair_cluster_slots();
cudaError_t launch_pack_sf(const void* sf, void* packed, int64_t rows, int K, int grid, cudaStream_t stream);
cudaError_t launch_mx_quantize(const float* in, int64_t n, uint8_t* q, uint8_t* sf, cudaStream_t stream);

struct FusedMxArgs {
  const int* meta;
  const int* expert_of_rb;
  const int* row_tok;
  const float* slot_w;
  void* out_f32;            // fp32 [T, D], zeroed before the launch
  const void* xg_sf;        // blocked scale tiles of xg
  const void* w1_sf;        // packed W1 scales
  const void* w2_sf;        // packed W2 scales
  int* err;
  unsigned long long wait_limit_ns;
  int D, H;
  int stall_test;
  float swiglu_limit;       // > 0: gate clamped to <= limit, up to [-limit, limit] before SwiGLU
};
cudaError_t launch_fused_mxfp8(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w2,
                               const FusedMxArgs& args, int grid, cudaStream_t stream);

// tile shapes of the bf16 GEMMs (host and device agree on these)
constexpr int kUpFold = 128;      // gate rows + up rows per tile: N = 2 * kUpFold
constexpr int kUpStages = 4;
constexpr int kUpFoldNarrow = 64;    // narrow up tiles (N = 128) for problems with few row blocks
constexpr int kUpStagesNarrow = 6;
constexpr int kDownN = 256;
constexpr int kDownStages = 4;
constexpr int kDownNNarrow = 128;
constexpr int kDownStagesNarrow = 6;
// 64-row tiles: the token stage is 8 KB, so more weight stages fit
constexpr int kUpStagesM64 = 5;          // 8 + 32 KB
constexpr int kUpStagesM64Narrow = 8;    // 8 + 16 KB
constexpr int kDownStagesM64 = 5;        // 8 + 32 KB
constexpr int kDownStagesM64Narrow = 8;  // 8 + 16 KB

}  // namespace moe
