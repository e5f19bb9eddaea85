// api.cu -- the extern "C" entry points: argument checks, workspace layout,
// tensor-map encoding and the launch sequence of each pipeline.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/moe_ffn.h"
#include "internal.h"
#include "mx_swap.h"
#include "ptx.cuh"

namespace moe {
// The routing kernels the last launch_route call of this host thread launched
// ('+' between them; route.cu).
const char* last_route_kernels();
// MXFP4 weight codes widened to e4m3 codes (mx4.cu)
cudaError_t launch_widen_e2m1(const void* in, int64_t n_bytes, void* out, int grid, cudaStream_t stream);
}  // namespace moe

namespace moe {
namespace {

std::atomic<unsigned long long> g_wait_limit_ns{2000ull * 1000 * 1000};
std::atomic<int> g_gather_mode{0};  // MOE_OPT_GATHER: 0 gather kernel, 1 in-GEMM gather4, 2 in-GEMM cp.async
std::atomic<int> g_prefetch{0};     // MOE_OPT_L2_PREFETCH (measured slower on GB300: off)
std::atomic<int> g_stall_test{0};   // MOE_OPT_TEST_STALL
std::atomic<int> g_up_pairs{0};     // MOE_OPT_UP_PAIRS (measured slower on GB300: off)
std::atomic<int> g_dynamic_tiles{2};  // MOE_OPT_DYNAMIC_TILES: 0 off, 1 on, 2 small problems only
std::atomic<int> g_tile_cols{0};      // MOE_OPT_TILE_COLS: 0 auto, 128 or 256 (bf16 split GEMM tile width)
std::atomic<int> g_fused_cluster{1};  // MOE_OPT_FUSED_CLUSTER: 0 off, 1 automatic size, 2/4/8 that size
std::atomic<int> g_pair_mma{2};       // MOE_OPT_PAIR_MMA: 0 off, 1 on, 2 automatic (not for small problems)
std::atomic<int> g_swap_ab{0};        // MOE_OPT_SWAP_AB: swap-AB tail tiles (measured slower on GB300: off)
std::atomic<int> g_out_hint{0};       // MOE_OPT_OUT_L2_HINT: 0 off (measured no gain), 1 automatic, 2 always
std::atomic<int> g_gather_blocks{8};  // MOE_OPT_GATHER_BLOCKS: gather blocks per SM
std::atomic<int> g_l2_policy{0};      // MOE_OPT_L2_POLICY: bit 0 weights evict_first, bit 1 xg evict_last
std::atomic<int> g_prefetch_mb{0};    // MOE_OPT_PREFETCH_MB: weights prefetched into L2 during routing
std::atomic<int> g_pair_swap{0};      // MOE_OPT_PAIR_SWAP: max routed rows of a swap-AB pair tile (measured slower: off)
std::atomic<int> g_wide_up{0};        // MOE_OPT_WIDE_UP: 512-column up tiles on CTA pairs
std::atomic<int> g_down_bands{1};     // MOE_OPT_DOWN_BANDS: token bands of the down tiles' order (0 automatic, 1 off)
constexpr int kHostChunkTokens = 16384;  // moe_ffn_forward_host: automatic chunk size
std::atomic<int> g_host_ramp{1};      // MOE_OPT_HOST_RAMP: quarter chunks at both ends of a long host pipeline
std::atomic<int> g_mx_swap{0};        // MOE_OPT_MX_SWAP: swap-AB MXFP8 split GEMMs (0 off: measured slower, 1 on, 2 decode-sized problems)
std::atomic<int> g_up_swap{1};        // MOE_OPT_UP_SWAP: swap-AB half pairs in the CTA-pair up kernel
std::atomic<int> g_mx_pairs{0};       // MOE_OPT_MX_PAIRS: MXFP8 split GEMMs on CTA pairs (0 off: measured slower, 1 on, 2 automatic)
std::atomic<int> g_down_epi8{1};      // MOE_OPT_DOWN_EPI8: eight epilogue warps in the CTA-pair down kernel
std::atomic<int> g_half_m128{0};      // MOE_OPT_HALF_PAIR_M128: half pairs as M = 128 pair MMAs (measured no gain: off)
std::atomic<int> g_fused_dsmem{0};    // MOE_OPT_FUSED_DSMEM: act kept in shared memory in the cluster kernel (measured slower: off)
std::atomic<int> g_tile_m{0};         // MOE_OPT_TILE_M: rows per tile of the single-CTA split GEMMs (0 automatic)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Whether the reductions into out carry an L2 evict_last hint: automatic when
// out is no larger than about the L2 (it can then stay resident while the
// weights stream past; a much larger out would only push weights out).
constexpr int64_t kOutHintMaxBytes = 160ll << 20;
int out_hint_for(int64_t out_bytes) {
  const int opt = g_out_hint.load();
  return opt == 2 || (opt == 1 && out_bytes <= kOutHintMaxBytes) ? 1 : 0;
}

// Token bands of the down projection's tile order: the reductions into out
// then stay within the rows of one band at a time, which L2 holds while the
// weights stream past.  Automatic: bands of at most 48 MiB of out, when out
// is larger than 64 MiB.
int down_bands(int T, int D) {
  const int opt = g_down_bands.load();
  if (opt >= 1) return T >= opt ? opt : 1;
  const int64_t out_bytes = (int64_t)T * D * 2;
  if (out_bytes <= (64ll << 20)) return 1;
  const int64_t n = (out_bytes + (48ll << 20) - 1) / (48ll << 20);
  return (int)std::min<int64_t>(std::min<int64_t>(n, 64), T);
}

bool shape_ok(int T, int E, int D, int H, int k) {
  return T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && D >= 128 && H >= 128 && D % 128 == 0 && H % 128 == 0 &&
         (int64_t)T * k < (int64_t)1 << 30;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols] read in boxes of [box_rows, 64] with the
// 128-byte swizzle (64 bf16 = one 128-byte swizzle row).  box_rows == 1 is the
// one-row box tile::gather4 requires.
bool make_map_2d(CUtensorMap* m, CUtensorMapDataType type, int elem_bytes, const void* base, uint64_t rows,
                 uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elem_bytes};
  cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, box_rows);
}
// e4m3 bytes [rows, cols] in boxes of [box_rows, 128] (one 128-byte swizzle row).
bool make_map_fp8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, box_rows);
}
// E2M1 codes [rows, cols], two per byte (element 2j in the low four bits of
// byte j), loaded in boxes of [box_rows, 128 codes] into 128-byte swizzled
// shared-memory rows, every 16 codes (8 bytes) in a 16-byte slot
// (16U4_ALIGN16B: base 32-byte aligned, cols a multiple of 128).
bool make_map_fp4(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols / 2};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Blocked scale tiles [tiles x 512 bytes] seen as a [tiles, 128] u32 tensor,
// one tile per box (no swizzle: a tile lands in shared memory as stored).
bool make_map_sf(CUtensorMap* m, const void* base, uint64_t tiles) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, tiles};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Optional per-stage timing (benchmarking aid).
constexpr int kMaxProfileEvents = 8;
struct Profile {
  std::mutex mu;
  bool on = false;
  bool created = false;
  cudaEvent_t ev[kMaxProfileEvents] = {};
  int recorded = 0;  // events recorded by the last profiled call
  const char* kernel[kMaxProfileEvents] = {};  // main kernel of each stage of the last profiled call
} g_prof;

// Record the next stage boundary of the current call (no-op when disabled).
void prof_mark(cudaStream_t st, int idx) {
  if (!g_prof.on || !g_prof.created || idx >= kMaxProfileEvents) return;
  cudaEventRecord(g_prof.ev[idx], st);
  g_prof.recorded = idx + 1;
}

// Name the main kernel of a stage of the current call (no-op when disabled).
void prof_kernel(int stage, const char* name) {
  if (!g_prof.on || stage < 0 || stage >= kMaxProfileEvents) return;
  g_prof.kernel[stage] = name;
}

// The routing and gather stages, common to every pipeline.
void prof_front(bool mx) {
  prof_kernel(0, last_route_kernels());  // called after the routing launch
  prof_kernel(1, mx ? "gather_rows_mx" : "gather_tokens");
}

}  // namespace

std::atomic<int> g_route_coop{1};
std::atomic<int> g_router_fused{0};
std::atomic<int> g_route_tpb{0};  // MOE_OPT_ROUTE_TPB: tokens per routing block (0: 256)
std::atomic<int64_t> g_route_small_pairs{8192};

Workspace plan_workspace(void* base, int T, int E, int D, int H, int k, int pipeline, int dtype) {
  Workspace w{};
  w.wait_limit_ns = g_wait_limit_ns.load();
  w.route_stall_test = g_stall_test.load() == 2 ? 1 : 0;
  w.l2_policy = g_l2_policy.load();
  const int64_t P = (int64_t)T * k;
  const int64_t live_experts = P < E ? P : E;
  w.S_max = (int64_t)align_up((size_t)(P + live_experts * (kRowPad - 1)), kRowPad);
  if (w.S_max == 0) w.S_max = kRowPad;
  w.max_rb = (int)(w.S_max / kRowPad);
  // tokens per routing block: by option (64, 128 or 256), else the default
  w.route_tpb = g_route_tpb.load() ? g_route_tpb.load() : kRouteTokPerBlock;
  w.route_blocks = (T + w.route_tpb - 1) / w.route_tpb;
  if (w.route_blocks == 0) w.route_blocks = 1;
  uint8_t* b = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = b ? b + off : nullptr;
    off = align_up(off + bytes, 256);
    return p;
  };
  w.err = reinterpret_cast<int*>(take(32));
  w.meta = reinterpret_cast<int*>(take(32));
  w.counts = reinterpret_cast<int*>(take(sizeof(int) * E));
  w.offsets = reinterpret_cast<int*>(take(sizeof(int) * (E + 1)));
  w.pad_offsets = reinterpret_cast<int*>(take(sizeof(int) * (E + 1)));
  w.expert_of_rb = reinterpret_cast<int*>(take(sizeof(int) * w.max_rb));
  w.pair_info = reinterpret_cast<int*>(take(sizeof(int) * w.max_rb));
  w.row_tok = reinterpret_cast<int*>(take(sizeof(int) * w.S_max));
  w.slot_w = reinterpret_cast<float*>(take(sizeof(float) * w.S_max));
  w.slot_of_pair = reinterpret_cast<int*>(take(sizeof(int) * (P ? P : 1)));
  w.blk_base = reinterpret_cast<int*>(take(sizeof(int) * (size_t)w.route_blocks * E));
  w.rb_order = reinterpret_cast<int*>(take(sizeof(int) * w.max_rb));
  w.pair_order = reinterpret_cast<int*>(take(sizeof(int) * w.max_rb));
  if (pipeline == kRouteOnly) {
    // routing regions only
  } else if (dtype == MOE_NVFP4) {  // split only: packed codes and e4m3 scales per 16
    w.xg = take((size_t)w.S_max * D / 2);
    w.xg_sf = take((size_t)w.S_max * D / 16);
    w.act = take((size_t)w.S_max * H / 2);
    w.act_sf = take((size_t)w.S_max * H / 16);
    if (f32_accum(k)) w.acc_f32 = take((size_t)T * D * 4);
  } else if (dtype != MOE_BF16) {  // MXFP8 activations (e4m3 weights, or MXFP4 weights)
    w.xg = take((size_t)w.S_max * D);
    w.xg_sf = take((size_t)w.S_max * D / 32);
    if (pipeline == MOE_SPLIT) {
      w.act = take((size_t)w.S_max * H);
      w.act_sf = take((size_t)w.S_max * H / 32);
      if (f32_accum(k)) w.acc_f32 = take((size_t)T * D * 4);
    } else {
      w.acc_f32 = take((size_t)T * D * 4);
      int cmin = 0;  // ring capacity for the smallest cluster size that applies
      for (int C : {8, 4, 2, 1})
        if (fused_cluster_mx_fits(D, H, C)) cmin = C;
      if (cmin) {
        const size_t bufs = (size_t)(kFusedClusterMaxCtas / cmin) * 2;
        w.ring = take(bufs * kBM * H);
        w.ring_sf = take(bufs * (H / 128) * 512);
      }
    }
  } else if (pipeline == MOE_SPLIT) {
    w.xg = take((size_t)w.S_max * D * 2);
    w.act = take((size_t)w.S_max * H * 2);
    if (f32_accum(k)) w.acc_f32 = take((size_t)T * D * 4);
  } else {
    w.xg = take((size_t)w.S_max * D * 2);
    w.acc_f32 = take((size_t)T * D * 4);
    if (fused_cluster_ok(D, H)) {  // capacity for the smallest cluster size that applies
      int cmin = 0;
      for (int C : {8, 4, 2, 1})
        if (fused_cluster_h1(D, H, C)) cmin = C;
      w.ring = take((size_t)(kFusedClusterMaxCtas / cmin) * 2 * kBM * H * 2);
    }
  }
  w.bytes = off;
  return w;
}

namespace {

// Cluster size for the fused kernel: the one with the shortest estimated run,
// waves of row blocks over the co-resident clusters times the work of one row
// block per CTA (1/C of it; more when GEMM1's sub-chunks are narrower than 128
// act columns, i.e. more operand bytes per FLOP, and for single-CTA clusters,
// which measured slower on GB300 than their share).  The row-block count is
// estimated from the routed pairs (half a padded block per live expert).
int choose_cluster_size(int D, int H, int64_t pairs, int E, int max_rb, bool dsmem) {
  const int64_t live = std::min<int64_t>(pairs, E);
  const int64_t est_rb = std::min<int64_t>(max_rb, std::max<int64_t>(live, (pairs + kBM - 1) / kBM + live / 2));
  int best = 0;
  double best_cost = 0;
  for (int C : {1, 2, 4, 8}) {
    const int h1 = fused_cluster_h1(D, H, C);
    if (!h1 || (dsmem && !fused_dsmem_fits(D, H, C))) continue;
    const int ncl = std::min(dsmem ? fused_dsmem_max_clusters(C) : fused_cluster_max_clusters(C),
                             kFusedClusterMaxCtas / C);
    if (ncl <= 0) continue;
    const double waves = (double)((est_rb + ncl - 1) / ncl);
    const double narrow = h1 == 128 ? 1.0 : h1 == 96 ? 1.1 : h1 == 64 ? 1.25 : 1.6;
    const double cost = waves * narrow * (C == 1 ? 1.3 : 1.0) / C;
    if (!best || cost < best_cost) {
      best = C;
      best_cost = cost;
    }
  }
  return best;
}

// Fused pipeline on clusters: routing, gather (+ zero-fill of out), one GEMM
// kernel in which clusters of D/256 CTAs exchange act through an L2-resident
// ring and reduce finished rows into out.
moe_status_t forward_fused_cluster_bf16(const Workspace& ws, const void* x, const void* w1, const void* w2,
                                        const int32_t* topk_ids, const float* topk_w, void* out, int T, int E, int D,
                                        int H, int k, int sms, int C, bool dsmem, cudaStream_t st) {
  const int h1 = fused_cluster_h1(D, H, C);
  const int ncl_cap = kFusedClusterMaxCtas / C;
  const int ncl = std::min(std::min(dsmem ? fused_dsmem_max_clusters(C) : fused_cluster_max_clusters(C), ncl_cap),
                           ws.max_rb);
  if (ncl <= 0 || !h1) return MOE_ERR_CUDA;
  CUtensorMap map_xg, map_w1, map_w2, map_ring;
  if (!make_map_bf16(&map_xg, ws.xg, (uint64_t)ws.S_max, (uint64_t)D, kBM) ||
      !make_map_bf16(&map_w1, w1, (uint64_t)E * 2 * H, (uint64_t)D, (uint32_t)h1) ||
      !make_map_bf16(&map_w2, w2, (uint64_t)E * D, (uint64_t)H, kFusedClusterN) ||
      (!dsmem && !make_map_bf16(&map_ring, ws.ring, (uint64_t)ncl_cap * 2 * kBM, (uint64_t)H, kBM)))
    return MOE_ERR_CUDA;
  prof_mark(st, 0);
  cudaError_t e = launch_route(ws, topk_ids, topk_w, T, E, k, st, nullptr, 0, 0, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 1);
  e = launch_gather_zero(ws, x, topk_ids, T, E, k, D, out, (int64_t)T * D * 2, sms * g_gather_blocks.load(), st, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 2);
  FusedClusterArgs fa{};
  fa.meta = ws.meta;
  fa.expert_of_rb = ws.expert_of_rb;
  fa.row_tok = ws.row_tok;
  fa.slot_w = ws.slot_w;
  fa.out = out;
  fa.ring = ws.ring;
  fa.err = ws.err;
  fa.wait_limit_ns = g_wait_limit_ns.load();
  fa.D = D;
  fa.H = H;
  fa.csize = C;
  fa.out_hint = out_hint_for((int64_t)T * D * 2);
  fa.h1 = h1;
  fa.s1 = H / C / h1;
  fa.s2 = D / C / kFusedClusterN;
  fa.stall_test = g_stall_test.load() == 1 ? 1 : 0;
  fa.swiglu_limit = ws.swiglu_limit;
  prof_front(false);
  prof_kernel(2, dsmem ? "fused_dsmem_bf16" : "fused_cluster_bf16");
  prof_kernel(3, "none");
  e = dsmem ? launch_fused_dsmem_bf16(map_xg, map_w1, map_w2, fa, ncl, st)
            : launch_fused_cluster_bf16(map_xg, map_w1, map_w2, map_ring, fa, ncl, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 3);
  prof_mark(st, 4);  // no rounding pass: out is reduced in bf16 directly
  return MOE_OK;
}

// Fused pipeline: routing, gather (+ zero-fill of the fp32 accumulator), one
// GEMM kernel that keeps act on chip, rounding of the accumulator to bf16.
moe_status_t forward_fused_bf16(const Workspace& ws, const void* x, const void* w1, const void* w2,
                                const int32_t* topk_ids, const float* topk_w, void* out, int T, int E, int D, int H,
                                int k, int sms, cudaStream_t st) {
  const int opt = g_fused_cluster.load();
  // the cluster kernel reduces finished rows into out in bf16; for large k
  // the split-K kernel's fp32 accumulator is taken instead
  if (opt && fused_cluster_ok(D, H) && !f32_accum(k)) {
    // act kept in shared memory where a cluster size allows it, else the L2 ring
    bool dsmem = false;
    int C = 0;
    if (g_fused_dsmem.load()) {
      C = (opt > 1 && fused_dsmem_fits(D, H, opt)) ? opt : 0;
      if (!C && opt == 1) C = choose_cluster_size(D, H, (int64_t)T * k, E, ws.max_rb, true);
      dsmem = C != 0;
    }
    if (!C) C = (opt > 1 && fused_cluster_h1(D, H, opt)) ? opt : 0;
    if (!C) C = choose_cluster_size(D, H, (int64_t)T * k, E, ws.max_rb, false);
    if (C) return forward_fused_cluster_bf16(ws, x, w1, w2, topk_ids, topk_w, out, T, E, D, H, k, sms, C, dsmem, st);
  }
  CUtensorMap map_xg, map_w1, map_w2;
  if (!make_map_bf16(&map_xg, ws.xg, (uint64_t)ws.S_max, (uint64_t)D, kBM) ||
      !make_map_bf16(&map_w1, w1, (uint64_t)E * 2 * H, (uint64_t)D, kUpFold) ||
      !make_map_bf16(&map_w2, w2, (uint64_t)E * D, (uint64_t)H, kDownN))
    return MOE_ERR_CUDA;
  prof_mark(st, 0);
  cudaError_t e = launch_route(ws, topk_ids, topk_w, T, E, k, st, nullptr, 0, 0, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 1);
  e = launch_gather_zero(ws, x, topk_ids, T, E, k, D, ws.acc_f32, (int64_t)T * D * 4, sms * g_gather_blocks.load(), st, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 2);
  FusedArgs fa{};
  fa.meta = ws.meta;
  fa.expert_of_rb = ws.expert_of_rb;
  fa.row_tok = ws.row_tok;
  fa.slot_w = ws.slot_w;
  fa.out_f32 = ws.acc_f32;
  fa.err = ws.err;
  fa.wait_limit_ns = g_wait_limit_ns.load();
  fa.D = D;
  fa.H = H;
  fa.n_slices = H / 128;
  fa.stall_test = g_stall_test.load() == 1 ? 1 : 0;
  fa.swiglu_limit = ws.swiglu_limit;
  const int grid = (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * fa.n_slices);
  prof_front(false);
  prof_kernel(2, "fused_moe_bf16");
  prof_kernel(3, "f32_to_bf16");
  e = launch_fused_bf16(map_xg, map_w1, map_w2, fa, grid, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 3);
  e = launch_f32_to_bf16(ws.acc_f32, out, (int64_t)T * D, sms * 4, st);
  prof_mark(st, 4);
  return cuda_status(e);
}

// MXFP8 split pipeline: routing, gather of e4m3 rows and their scales (+ zero
// of out), block-scaled up-projection with SwiGLU and requantization,
// block-scaled down-projection with the weighted reduction.
moe_status_t forward_split_mxfp8(const Workspace& ws, const void* x, const void* x_sf, const void* w1,
                                 const void* w1_sf, const void* w2, const void* w2_sf, const int32_t* topk_ids,
                                 const float* topk_w, void* out, int T, int E, int D, int H, int k, int sms,
                                 cudaStream_t st, bool fp4w) {
  // CTA pairs (e4m3 weights) unless the problem is small: decode-sized
  // problems stream weights, and single CTAs spread over more SMs
  const int mxp_opt = g_mx_pairs.load();
  const bool small = (int64_t)ws.max_rb * (H / 128) < 8LL * sms;
  const bool pairs = !fp4w && (mxp_opt == 1 || (mxp_opt == 2 && !small));
  // swapped operands (weights on the MMA's M side) when an expert holds few
  // rows: by option, or automatically at <= 64 routed rows per live expert on
  // average; bf16 row sums only (k <= 8)
  const int swap_opt = g_mx_swap.load();
  const int64_t P = (int64_t)T * k;
  const bool swap = !pairs && !f32_accum(k) &&
                    (swap_opt == 1 || (swap_opt == 2 && P <= 64 * std::min<int64_t>(P, E)));
  CUtensorMap map_xg, map_w1, map_act, map_w2, sf_xg, sf_w1, sf_act, sf_w2, map_xg32, map_act32;
  auto make_w = fp4w ? make_map_fp4 : make_map_fp8;
  if (!make_map_fp8(&map_xg, ws.xg, (uint64_t)ws.S_max, (uint64_t)D, kBM) ||
      !make_w(&map_w1, w1, (uint64_t)E * 2 * H, (uint64_t)D, 128) ||
      !make_map_fp8(&map_act, ws.act, (uint64_t)ws.S_max, (uint64_t)H, kBM) ||
      !make_w(&map_w2, w2, (uint64_t)E * D, (uint64_t)H, (pairs || swap) ? 128 : 256))
    return MOE_ERR_CUDA;
  if (swap && (!make_map_fp8(&map_xg32, ws.xg, (uint64_t)ws.S_max, (uint64_t)D, 32) ||
               !make_map_fp8(&map_act32, ws.act, (uint64_t)ws.S_max, (uint64_t)H, 32)))
    return MOE_ERR_CUDA;
  if (pairs && (!make_map_sf(&sf_xg, ws.xg_sf, (uint64_t)(ws.S_max / 128) * (D / 128)) ||
                !make_map_sf(&sf_w1, w1_sf, (uint64_t)E * (2 * H / 128) * (D / 128)) ||
                !make_map_sf(&sf_act, ws.act_sf, (uint64_t)(ws.S_max / 128) * (H / 128)) ||
                !make_map_sf(&sf_w2, w2_sf, (uint64_t)E * (D / 128) * (H / 128))))
    return MOE_ERR_CUDA;
  const int mx_slots = pairs ? mx_pair_cluster_slots() : 0;
  if (pairs && mx_slots <= 0) return MOE_ERR_CUDA;
  prof_mark(st, 0);
  cudaError_t e = launch_route(ws, topk_ids, topk_w, T, E, k, st, nullptr, 0, 0, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 1);
  // large k: the rows of a token are summed in the fp32 accumulator
  float* acc = f32_accum(k) ? static_cast<float*>(ws.acc_f32) : nullptr;
  e = acc ? launch_gather_mx(ws, x, x_sf, topk_ids, T, E, k, D, acc, (int64_t)T * D * 4, sms * g_gather_blocks.load(),
                             st, !g_prof.on)
          : launch_gather_mx(ws, x, x_sf, topk_ids, T, E, k, D, out, (int64_t)T * D * 2, sms * g_gather_blocks.load(),
                             st, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const int bands = down_bands(T, D);
  if (bands > 1 && launch_band_order(ws, T, bands, st) != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 2);
  MxArgs ma{};
  ma.meta = ws.meta;
  ma.expert_of_rb = ws.expert_of_rb;
  ma.pair_info = ws.pair_info;
  ma.row_tok = ws.row_tok;
  ma.slot_w = ws.slot_w;
  ma.act = ws.act;
  ma.act_sf = ws.act_sf;
  ma.out = out;
  ma.out_f32 = acc;
  ma.err = ws.err;
  ma.wait_limit_ns = g_wait_limit_ns.load();
  ma.D = D;
  ma.H = H;
  ma.stall_test = g_stall_test.load() == 1 ? 1 : 0;
  ma.swiglu_limit = ws.swiglu_limit;
  ma.out_hint = out_hint_for((int64_t)T * D * 2);
  MxArgs up = ma;
  up.sf_a = ws.xg_sf;
  up.sf_b = w1_sf;
  up.n_col_tiles = H / 128;
  up.k_blocks = D / 128;
  prof_front(true);
  if (bands > 1) prof_kernel(1, "gather_rows_mx+band_order");
  prof_kernel(2, swap    ? (fp4w ? "up_swiglu_mxfp4w_swap" : "up_swiglu_mxfp8_swap")
                 : fp4w  ? "up_swiglu_mxfp4w"
                 : pairs ? "up_swiglu_mxfp8_pair2"
                         : "up_swiglu_mxfp8");
  prof_kernel(3, swap    ? (fp4w ? "down_reduce_mxfp4w_swap" : "down_reduce_mxfp8_swap")
                 : fp4w  ? (acc ? "down_reduce_mxfp4w+f32_to_bf16" : "down_reduce_mxfp4w")
                 : pairs ? (acc ? "down_reduce_mxfp8_pair2+f32_to_bf16" : "down_reduce_mxfp8_pair2")
                         : (acc ? "down_reduce_mxfp8+f32_to_bf16" : "down_reduce_mxfp8"));
  MxSwapArgs sw{};
  if (swap) {
    sw.meta = ws.meta;
    sw.expert_of_rb = ws.expert_of_rb;
    sw.counts = ws.counts;
    sw.pad_offsets = ws.pad_offsets;
    sw.row_tok = ws.row_tok;
    sw.slot_w = ws.slot_w;
    sw.act = ws.act;
    sw.act_sf = ws.act_sf;
    sw.out = out;
    sw.err = ws.err;
    sw.wait_limit_ns = ma.wait_limit_ns;
    sw.D = D;
    sw.H = H;
    sw.stall_test = ma.stall_test;
    sw.out_hint = ma.out_hint;
    sw.swiglu_limit = ma.swiglu_limit;
    MxSwapArgs su = sw;
    su.sf_x = ws.xg_sf;
    su.sf_w = w1_sf;
    su.n_col_tiles = H / 128;
    su.k_blocks = D / 128;
    e = launch_up_mx_swap(map_w1, map_xg32, su, (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * su.n_col_tiles), st,
                          fp4w);
  } else if (pairs)
    e = launch_up_mxfp8_pair(map_xg, map_w1, sf_xg, sf_w1, up,
                             (int)std::min<int64_t>(mx_slots, (int64_t)ws.max_rb * up.n_col_tiles), st);
  else
    e = launch_up_mxfp8(map_xg, map_w1, up, (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * up.n_col_tiles), st,
                        fp4w);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 3);
  MxArgs dn = ma;
  dn.rb_order = bands > 1 ? ws.rb_order : nullptr;
  dn.pair_order = bands > 1 ? ws.pair_order : nullptr;
  dn.sf_a = ws.act_sf;
  dn.sf_b = w2_sf;
  dn.n_col_tiles = D / 256;
  dn.k_blocks = H / 128;
  if (swap) {
    MxSwapArgs sd = sw;
    sd.sf_x = ws.act_sf;
    sd.sf_w = w2_sf;
    sd.n_col_tiles = D / 128;
    sd.k_blocks = H / 128;
    e = launch_down_mx_swap(map_w2, map_act32, sd, (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * sd.n_col_tiles), st,
                            !g_prof.on, fp4w);
  } else if (pairs)
    e = launch_down_mxfp8_pair(map_act, map_w2, sf_act, sf_w2, dn,
                               (int)std::min<int64_t>(mx_slots, (int64_t)ws.max_rb * dn.n_col_tiles), st, !g_prof.on);
  else
    e = launch_down_mxfp8(map_act, map_w2, dn, (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * dn.n_col_tiles), st,
                          !g_prof.on, fp4w);
  if (e == cudaSuccess && acc) e = launch_f32_to_bf16(acc, out, (int64_t)T * D, sms * 4, st);
  prof_mark(st, 4);
  return cuda_status(e);
}

// NVFP4 split pipeline: routing, gather of packed rows and their scale tiles
// (+ zero of out), block-scaled up projection with SwiGLU and NVFP4
// requantization of act, block-scaled down projection with the reduction.
moe_status_t forward_split_nvfp4(const Workspace& ws, const void* x, const void* x_sf, const void* w1,
                                 const void* w1_sf, const void* w2, const void* w2_sf, const moe_ffn_nvfp4_scales_t& gs,
                                 const int32_t* topk_ids, const float* topk_w, void* out, int T, int E, int D, int H,
                                 int k, int sms, cudaStream_t st) {
  CUtensorMap map_xg, map_w1, map_act, map_w2;  // packed codes read as bytes, 256 codes per 128-byte box row
  if (!make_map_fp8(&map_xg, ws.xg, (uint64_t)ws.S_max, (uint64_t)D / 2, kBM) ||
      !make_map_fp8(&map_w1, w1, (uint64_t)E * 2 * H, (uint64_t)D / 2, 128) ||
      !make_map_fp8(&map_act, ws.act, (uint64_t)ws.S_max, (uint64_t)H / 2, kBM) ||
      !make_map_fp8(&map_w2, w2, (uint64_t)E * D, (uint64_t)H / 2, 128))  // two 128-row boxes per stage
    return MOE_ERR_CUDA;
  prof_mark(st, 0);
  cudaError_t e = launch_route(ws, topk_ids, topk_w, T, E, k, st, nullptr, 0, 0, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 1);
  float* acc = f32_accum(k) ? static_cast<float*>(ws.acc_f32) : nullptr;
  e = acc ? launch_gather_mx(ws, x, x_sf, topk_ids, T, E, k, D, acc, (int64_t)T * D * 4, sms * g_gather_blocks.load(),
                             st, !g_prof.on, true)
          : launch_gather_mx(ws, x, x_sf, topk_ids, T, E, k, D, out, (int64_t)T * D * 2, sms * g_gather_blocks.load(),
                             st, !g_prof.on, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 2);
  MxArgs ma{};
  ma.meta = ws.meta;
  ma.expert_of_rb = ws.expert_of_rb;
  ma.row_tok = ws.row_tok;
  ma.slot_w = ws.slot_w;
  ma.act = ws.act;
  ma.act_sf = ws.act_sf;
  ma.out = out;
  ma.out_f32 = acc;
  ma.x_gs = gs.x_gs;
  ma.w1_gs = gs.w1_gs;
  ma.w2_gs = gs.w2_gs;
  ma.act_gs = gs.act_gs;
  ma.err = ws.err;
  ma.wait_limit_ns = g_wait_limit_ns.load();
  ma.D = D;
  ma.H = H;
  ma.stall_test = g_stall_test.load() == 1 ? 1 : 0;
  ma.swiglu_limit = ws.swiglu_limit;
  MxArgs up = ma;
  up.sf_a = ws.xg_sf;
  up.sf_b = w1_sf;
  up.n_col_tiles = H / 128;
  up.k_blocks = D / 256;
  prof_front(true);
  prof_kernel(1, "gather_rows_nv");
  prof_kernel(2, "up_swiglu_nvfp4");
  prof_kernel(3, acc ? "down_reduce_nvfp4+f32_to_bf16" : "down_reduce_nvfp4");
  e = launch_up_nvfp4(map_xg, map_w1, up, (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * up.n_col_tiles), st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 3);
  MxArgs dn = ma;
  dn.sf_a = ws.act_sf;
  dn.sf_b = w2_sf;
  dn.n_col_tiles = D / 256;
  dn.k_blocks = H / 256;
  e = launch_down_nvfp4(map_act, map_w2, dn, (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * dn.n_col_tiles), st,
                        !g_prof.on);
  if (e == cudaSuccess && acc) e = launch_f32_to_bf16(acc, out, (int64_t)T * D, sms * 4, st);
  prof_mark(st, 4);
  return cuda_status(e);
}

// Cluster size for the MXFP8 fused kernel (same estimate as the bf16 one; the
// act slices are always 128 columns wide).
int choose_cluster_size_mx(int D, int H, int64_t pairs, int E, int max_rb) {
  const int64_t live = std::min<int64_t>(pairs, E);
  const int64_t est_rb = std::min<int64_t>(max_rb, std::max<int64_t>(live, (pairs + kBM - 1) / kBM + live / 2));
  int best = 0;
  double best_cost = 0;
  for (int C : {1, 2, 4, 8}) {
    if (!fused_cluster_mx_fits(D, H, C)) continue;
    const int ncl = std::min(fused_cluster_mx_max_clusters(C), kFusedClusterMaxCtas / C);
    if (ncl <= 0) continue;
    const double cost = (double)((est_rb + ncl - 1) / ncl) * (C == 1 ? 1.3 : 1.0) / C;
    if (!best || cost < best_cost) {
      best = C;
      best_cost = cost;
    }
  }
  return best;
}

// MXFP8 fused pipeline on clusters: routing, gather of e4m3 rows and scales (+
// zero of out), one block-scaled GEMM kernel whose clusters exchange the
// requantized act through an L2-resident ring.
moe_status_t forward_fused_cluster_mxfp8(const Workspace& ws, const void* x, const void* x_sf, const void* w1,
                                         const void* w1_sf, const void* w2, const void* w2_sf,
                                         const int32_t* topk_ids, const float* topk_w, void* out, int T, int E, int D,
                                         int H, int k, int sms, int C, cudaStream_t st) {
  const int ncl_cap = kFusedClusterMaxCtas / C;
  const int ncl = std::min(std::min(fused_cluster_mx_max_clusters(C), ncl_cap), ws.max_rb);
  if (ncl <= 0) return MOE_ERR_CUDA;
  CUtensorMap map_xg, map_w1, map_w2, map_ring;
  if (!make_map_fp8(&map_xg, ws.xg, (uint64_t)ws.S_max, (uint64_t)D, kBM) ||
      !make_map_fp8(&map_w1, w1, (uint64_t)E * 2 * H, (uint64_t)D, 128) ||
      !make_map_fp8(&map_w2, w2, (uint64_t)E * D, (uint64_t)H, 256) ||
      !make_map_fp8(&map_ring, ws.ring, (uint64_t)ncl_cap * 2 * kBM, (uint64_t)H, kBM))
    return MOE_ERR_CUDA;
  prof_mark(st, 0);
  cudaError_t e = launch_route(ws, topk_ids, topk_w, T, E, k, st, nullptr, 0, 0, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 1);
  e = launch_gather_mx(ws, x, x_sf, topk_ids, T, E, k, D, out, (int64_t)T * D * 2, sms * g_gather_blocks.load(), st, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 2);
  FusedClusterMxArgs fa{};
  fa.meta = ws.meta;
  fa.expert_of_rb = ws.expert_of_rb;
  fa.row_tok = ws.row_tok;
  fa.slot_w = ws.slot_w;
  fa.out = out;
  fa.ring = ws.ring;
  fa.ring_sf = ws.ring_sf;
  fa.xg_sf = ws.xg_sf;
  fa.w1_sf = w1_sf;
  fa.w2_sf = w2_sf;
  fa.err = ws.err;
  fa.wait_limit_ns = g_wait_limit_ns.load();
  fa.D = D;
  fa.H = H;
  fa.csize = C;
  fa.out_hint = out_hint_for((int64_t)T * D * 2);
  fa.s1 = H / C / 128;
  fa.s2 = D / C / 256;
  fa.stall_test = g_stall_test.load() == 1 ? 1 : 0;
  fa.swiglu_limit = ws.swiglu_limit;
  prof_front(true);
  prof_kernel(2, "fused_cluster_mxfp8");
  prof_kernel(3, "none");
  e = launch_fused_cluster_mxfp8(map_xg, map_w1, map_w2, map_ring, fa, ncl, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 3);
  prof_mark(st, 4);  // no rounding pass: out is reduced in bf16 directly
  return MOE_OK;
}

// MXFP8 fused pipeline: routing, gather of e4m3 rows and scales (+ zero of the
// fp32 accumulator), one block-scaled GEMM kernel that keeps the requantized
// act on chip, rounding of the accumulator to bf16.
moe_status_t forward_fused_mxfp8(const Workspace& ws, const void* x, const void* x_sf, const void* w1,
                                 const void* w1_sf, const void* w2, const void* w2_sf, const int32_t* topk_ids,
                                 const float* topk_w, void* out, int T, int E, int D, int H, int k, int sms,
                                 cudaStream_t st) {
  const int opt = g_fused_cluster.load();
  if (opt && ws.ring && !f32_accum(k)) {
    int C = (opt > 1 && fused_cluster_mx_fits(D, H, opt)) ? opt : 0;
    if (!C) C = choose_cluster_size_mx(D, H, (int64_t)T * k, E, ws.max_rb);
    if (C)
      return forward_fused_cluster_mxfp8(ws, x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E, D, H, k,
                                         sms, C, st);
  }
  CUtensorMap map_xg, map_w1, map_w2;
  if (!make_map_fp8(&map_xg, ws.xg, (uint64_t)ws.S_max, (uint64_t)D, kBM) ||
      !make_map_fp8(&map_w1, w1, (uint64_t)E * 2 * H, (uint64_t)D, 128) ||
      !make_map_fp8(&map_w2, w2, (uint64_t)E * D, (uint64_t)H, 256))
    return MOE_ERR_CUDA;
  prof_mark(st, 0);
  cudaError_t e = launch_route(ws, topk_ids, topk_w, T, E, k, st, nullptr, 0, 0, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 1);
  e = launch_gather_mx(ws, x, x_sf, topk_ids, T, E, k, D, ws.acc_f32, (int64_t)T * D * 4, sms * g_gather_blocks.load(), st,
                       !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 2);
  FusedMxArgs fa{};
  fa.meta = ws.meta;
  fa.expert_of_rb = ws.expert_of_rb;
  fa.row_tok = ws.row_tok;
  fa.slot_w = ws.slot_w;
  fa.out_f32 = ws.acc_f32;
  fa.xg_sf = ws.xg_sf;
  fa.w1_sf = w1_sf;
  fa.w2_sf = w2_sf;
  fa.err = ws.err;
  fa.wait_limit_ns = g_wait_limit_ns.load();
  fa.D = D;
  fa.H = H;
  fa.stall_test = g_stall_test.load() == 1 ? 1 : 0;
  fa.swiglu_limit = ws.swiglu_limit;
  const int grid = (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * (H / 128));
  prof_front(true);
  prof_kernel(2, "fused_moe_mxfp8");
  prof_kernel(3, "f32_to_bf16");
  e = launch_fused_mxfp8(map_xg, map_w1, map_w2, fa, grid, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 3);
  e = launch_f32_to_bf16(ws.acc_f32, out, (int64_t)T * D, sms * 4, st);
  prof_mark(st, 4);
  return cuda_status(e);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_ffn_workspace_size(int T, int E, int D, int H, int k, int dtype, int pipeline) {
  if (dtype == MOE_NVFP4 && pipeline != MOE_SPLIT) return 0;
  if (!shape_ok(T, E, D, H, k) || (dtype != MOE_BF16 && dtype != MOE_MXFP8 && dtype != MOE_MXFP4W && dtype != MOE_NVFP4) ||
      (pipeline != MOE_FUSED && pipeline != MOE_SPLIT))
    return 0;
  return plan_workspace(nullptr, T, E, D, H, k, pipeline, dtype).bytes;
}

moe_status_t moe_ffn_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < 64) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, 64, static_cast<cudaStream_t>(stream)));
}

void moe_ffn_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1); }

moe_status_t moe_ffn_set_option(int option, long long value) {
  switch (option) {
    case MOE_OPT_GATHER:
      if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
      g_gather_mode.store((int)value);
      return MOE_OK;
    case MOE_OPT_TEST_STALL:
      if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
      g_stall_test.store((int)value);
      return MOE_OK;
    case MOE_OPT_FUSED_CLUSTER:
      if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return MOE_ERR_INVALID_ARG;
      g_fused_cluster.store((int)value);
      return MOE_OK;
    case MOE_OPT_PAIR_MMA:
      if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
      g_pair_mma.store((int)value);
      return MOE_OK;
    case MOE_OPT_SWAP_AB:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_swap_ab.store((int)value);
      return MOE_OK;
    case MOE_OPT_ROUTE_COOP:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_route_coop.store((int)value);
      return MOE_OK;
    case MOE_OPT_OUT_L2_HINT:
      if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
      g_out_hint.store((int)value);
      return MOE_OK;
    case MOE_OPT_GATHER_BLOCKS:
      if (value < 1 || value > 16) return MOE_ERR_INVALID_ARG;
      g_gather_blocks.store((int)value);
      return MOE_OK;
    case MOE_OPT_L2_POLICY:
      if (value < 0 || value > 3) return MOE_ERR_INVALID_ARG;
      g_l2_policy.store((int)value);
      return MOE_OK;
    case MOE_OPT_ROUTER_FUSED:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_router_fused.store((int)value);
      return MOE_OK;
    case MOE_OPT_PREFETCH_MB:
      if (value < 0 || value > 1024) return MOE_ERR_INVALID_ARG;
      g_prefetch_mb.store((int)value);
      return MOE_OK;
    case MOE_OPT_PAIR_SWAP:
      if (value < 0 || value > 256) return MOE_ERR_INVALID_ARG;
      g_pair_swap.store((int)value);
      return MOE_OK;
    case MOE_OPT_FUSED_DSMEM:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_fused_dsmem.store((int)value);
      return MOE_OK;
    case MOE_OPT_TILE_M:
      if (value != 0 && value != 64 && value != 128) return MOE_ERR_INVALID_ARG;
      g_tile_m.store((int)value);
      return MOE_OK;
    case MOE_OPT_DOWN_BANDS:
      if (value < 0 || value > 64) return MOE_ERR_INVALID_ARG;
      g_down_bands.store((int)value);
      return MOE_OK;
    case MOE_OPT_ROUTE_SMALL_PAIRS:
      if (value < 0 || value > (1 << 20)) return MOE_ERR_INVALID_ARG;
      g_route_small_pairs.store(value);
      return MOE_OK;
    case MOE_OPT_HOST_RAMP:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_host_ramp.store((int)value);
      return MOE_OK;
    case MOE_OPT_MX_SWAP:
      if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
      g_mx_swap.store((int)value);
      return MOE_OK;
    case MOE_OPT_ROUTE_TPB:
      if (value != 0 && value != 64 && value != 128 && value != 256) return MOE_ERR_INVALID_ARG;
      g_route_tpb.store((int)value);
      return MOE_OK;
    case MOE_OPT_UP_SWAP:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_up_swap.store((int)value);
      return MOE_OK;
    case MOE_OPT_MX_PAIRS:
      if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
      g_mx_pairs.store((int)value);
      return MOE_OK;
    case MOE_OPT_DOWN_EPI8:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_down_epi8.store((int)value);
      return MOE_OK;
    case MOE_OPT_HALF_PAIR_M128:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_half_m128.store((int)value);
      return MOE_OK;
    case MOE_OPT_WIDE_UP:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_wide_up.store((int)value);
      return MOE_OK;

    case MOE_OPT_TILE_COLS:
      if (value != 0 && value != 128 && value != 256) return MOE_ERR_INVALID_ARG;
      g_tile_cols.store((int)value);
      return MOE_OK;
    case MOE_OPT_DYNAMIC_TILES:
      if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
      g_dynamic_tiles.store((int)value);
      return MOE_OK;
    case MOE_OPT_UP_PAIRS:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      g_up_pairs.store((int)value);
      return MOE_OK;
    case MOE_OPT_L2_PREFETCH:
      if (value < 0 || value > 64) return MOE_ERR_INVALID_ARG;
      g_prefetch.store((int)value);
      return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status_t moe_ffn_route(const int32_t* topk_ids, const float* topk_w, int T, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* slot_of_pair, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || (int64_t)T * k >= ((int64_t)1 << 30)) return MOE_ERR_INVALID_ARG;
  if (!workspace || (T > 0 && (!topk_ids || !topk_w))) return MOE_ERR_INVALID_ARG;
  Workspace ws = plan_workspace(workspace, T, E, 128, 128, k, kRouteOnly);
  if (workspace_bytes < ws.bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    cudaError_t z = cudaSuccess;
    if (counts) z = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st);
    if (z == cudaSuccess && offsets) z = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
    return cuda_status(z);
  }
  cudaError_t e = launch_route(ws, topk_ids, topk_w, T, E, k, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (counts) e = cudaMemcpyAsync(counts, ws.counts, sizeof(int32_t) * E, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && offsets)
    e = cudaMemcpyAsync(offsets, ws.offsets, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && slot_of_pair)
    e = cudaMemcpyAsync(slot_of_pair, ws.slot_of_pair, sizeof(int32_t) * T * k, cudaMemcpyDeviceToDevice, st);
  return cuda_status(e);
}

int64_t moe_ffn_route_padded_slots(int T, int E, int k) {
  if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || (int64_t)T * k >= ((int64_t)1 << 30)) return 0;
  return plan_workspace(nullptr, T, E, 128, 128, k, kRouteOnly).S_max;
}

moe_status_t moe_ffn_route_padded(const int32_t* topk_ids, const float* topk_w, int T, int E, int k,
                                  int32_t* pad_offsets, int32_t* expert_of_rb, int32_t* pair_info, int32_t* row_tok,
                                  float* slot_w, int32_t* n_blocks, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (T < 1 || E < 1 || E > kMaxExperts || k < 1 || (int64_t)T * k >= ((int64_t)1 << 30)) return MOE_ERR_INVALID_ARG;
  if (!workspace || !topk_ids || !topk_w || !pad_offsets || !expert_of_rb || !pair_info || !row_tok || !slot_w ||
      !n_blocks)
    return MOE_ERR_INVALID_ARG;
  Workspace ws = plan_workspace(workspace, T, E, 128, 128, k, kRouteOnly);
  if (workspace_bytes < ws.bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_route(ws, topk_ids, topk_w, T, E, k, st);
  auto copy = [&](void* dst, const void* src, size_t bytes) {
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
  };
  copy(pad_offsets, ws.pad_offsets, sizeof(int32_t) * (E + 1));
  copy(expert_of_rb, ws.expert_of_rb, sizeof(int32_t) * ws.max_rb);
  copy(pair_info, ws.pair_info, sizeof(int32_t) * ws.max_rb);
  copy(row_tok, ws.row_tok, sizeof(int32_t) * ws.S_max);
  copy(slot_w, ws.slot_w, sizeof(float) * ws.S_max);
  copy(n_blocks, ws.meta, sizeof(int32_t) * 2);
  return cuda_status(e);
}

// The forward pass from top-k ids and weights, or (router_logits != nullptr)
// from router logits, the routing launch writing topk_ids / topk_w first.
static moe_status_t forward_entry(const void* x, const void* x_sf, const void* w1, const void* w1_sf, const void* w2,
                                  const void* w2_sf, const int32_t* topk_ids, const float* topk_w, void* out, int T,
                                  int E, int D, int H, int k, int dtype, int pipeline, void* workspace,
                                  size_t workspace_bytes, void* stream, const float* router_logits,
                                  float swiglu_limit = 0.f) {
  if (!shape_ok(T, E, D, H, k)) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 && dtype != MOE_MXFP8 && dtype != MOE_MXFP4W) return MOE_ERR_INVALID_ARG;
  if (pipeline != MOE_FUSED && pipeline != MOE_SPLIT) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w1 || !w2 || !topk_ids || !topk_w || !out || !workspace) return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_BF16 && (x_sf || w1_sf || w2_sf)) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 && (!x_sf || !w1_sf || !w2_sf)) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 && ((reinterpret_cast<uintptr_t>(x_sf) & 3u) || !aligned16(w1_sf) || !aligned16(w2_sf)))
    return MOE_ERR_MISALIGNED;
  // packed 4-bit weights: split pipeline only; their tensor maps want 32-byte aligned bases
  if (dtype == MOE_MXFP4W && pipeline != MOE_SPLIT) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_MXFP4W && (((reinterpret_cast<uintptr_t>(w1) | reinterpret_cast<uintptr_t>(w2)) & 31u) != 0))
    return MOE_ERR_MISALIGNED;
  if (!aligned16(x) || !aligned16(w1) || !aligned16(w2) || !aligned16(out) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(topk_ids) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u))
    return MOE_ERR_MISALIGNED;
  // fused and MXFP8 kernels write 256-column output tiles; the bf16 split
  // pipeline falls back to 128-column tiles
  if (D % kDownN != 0 && (dtype != MOE_BF16 || pipeline != MOE_SPLIT)) return MOE_ERR_UNSUPPORTED;
  Workspace ws = plan_workspace(workspace, T, E, D, H, k, pipeline, dtype);
  if (workspace_bytes < ws.bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  ws.router_logits = router_logits;
  ws.swiglu_limit = swiglu_limit;
  // the up projection's weights, from the first expert on (its first tiles)
  ws.prefetch_base = w1;
  ws.prefetch_bytes = std::min<int64_t>((int64_t)g_prefetch_mb.load() << 20,
                                        (int64_t)E * 2 * H * D * (dtype == MOE_BF16 ? 2 : 1)) & ~(int64_t)15;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == MOE_MXFP8 && pipeline == MOE_FUSED)
    return forward_fused_mxfp8(ws, x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E, D, H, k, sms, st);
  if (dtype != MOE_BF16)
    return forward_split_mxfp8(ws, x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E, D, H, k, sms, st,
                               dtype == MOE_MXFP4W);
  if (pipeline == MOE_FUSED) return forward_fused_bf16(ws, x, w1, w2, topk_ids, topk_w, out, T, E, D, H, k, sms, st);

  const int gather = g_gather_mode.load();
  const bool in_gemm_gather = gather != 0;
  // Narrow up tiles when the 256-wide tiles would not fill the GPU several
  // times over (decode-sized problems): the last wave of equal tiles leaves
  // SMs idle, and narrower tiles make the waves finer.
  const int cols = g_tile_cols.load();
  const int down_n = (D % kDownN != 0 || cols == 128) ? kDownNNarrow : kDownN;
  const bool narrow_ok = !in_gemm_gather && !g_up_pairs.load();
  // CTA pairs unless the problem is small (decode-sized: its GEMMs stream
  // weights, and the narrow single-CTA tiles fill the GPU better)
  const int pair_opt = g_pair_mma.load();
  const bool small_up = (int64_t)ws.max_rb * (H / kUpFold) < 8LL * sms;
  const bool pair_mma =
      (pair_opt == 1 || (pair_opt == 2 && !small_up)) && !in_gemm_gather && !g_up_pairs.load() && cols != 128;
  const int fold =
      (!pair_mma && narrow_ok && (cols == 128 || (cols == 0 && (int64_t)ws.max_rb * (H / kUpFold) < 8LL * sms)))
          ? kUpFoldNarrow
          : kUpFold;  // auto: narrow when the wide tiles make fewer than ~8 waves
  const bool pair_down = pair_mma && down_n == kDownN;
  // 64-row tiles for the single-CTA GEMMs: by option, or automatically when
  // an expert gets at most 64 routed rows on average
  const int tile_m_opt = g_tile_m.load();
  const int64_t P = (int64_t)T * k;
  const bool m64 = !pair_mma && !in_gemm_gather && !g_up_pairs.load() &&
                   (tile_m_opt == 64 || (tile_m_opt == 0 && P <= 64 * std::min<int64_t>(P, E)));
  const int bm = m64 ? 64 : kBM;
  CUtensorMap map_xg, map_w1, map_w1_64, map_act, map_w2;
  const bool map_a_ok = in_gemm_gather ? make_map_bf16(&map_xg, x, (uint64_t)T, (uint64_t)D, 1)
                                       : make_map_bf16(&map_xg, ws.xg, (uint64_t)ws.S_max, (uint64_t)D, bm);
  if (!map_a_ok ||
      !make_map_bf16(&map_w1, w1, (uint64_t)E * 2 * H, (uint64_t)D, fold) ||
      !make_map_bf16(&map_act, ws.act, (uint64_t)ws.S_max, (uint64_t)H, bm) ||
      !make_map_bf16(&map_w2, w2, (uint64_t)E * D, (uint64_t)H, pair_down ? 128 : down_n) ||
      (pair_mma && !make_map_bf16(&map_w1_64, w1, (uint64_t)E * 2 * H, (uint64_t)D, 64)))
    return MOE_ERR_CUDA;

  prof_mark(st, 0);
  // Large k: the rows of a token are summed in the fp32 accumulator, which is
  // zero-filled instead of out and rounded into out after the down kernel.
  float* acc = f32_accum(k) ? static_cast<float*>(ws.acc_f32) : nullptr;
  void* zero_target = acc ? static_cast<void*>(acc) : out;
  const int64_t zero_bytes = (int64_t)T * D * (acc ? 4 : 2);
  // With the in-GEMM gather the routing launch also zero-fills the target;
  // otherwise the gather kernel does.
  cudaError_t e = in_gemm_gather
                      ? launch_route(ws, topk_ids, topk_w, T, E, k, st, zero_target, zero_bytes, sms * 2, !g_prof.on)
                      : launch_route(ws, topk_ids, topk_w, T, E, k, st, nullptr, 0, 0, !g_prof.on);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 1);
  if (!in_gemm_gather) {
    e = launch_gather_zero(ws, x, topk_ids, T, E, k, D, zero_target, zero_bytes, sms * g_gather_blocks.load(), st,
                           !g_prof.on);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  // the CTA-pair down kernel walks its block pairs in token-band order
  const int bands = pair_down ? down_bands(T, D) : 1;
  if (bands > 1 && launch_band_order(ws, T, bands, st) != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 2);

  GemmArgs ga{};
  ga.meta = ws.meta;
  ga.expert_of_rb = ws.expert_of_rb;
  ga.pair_info = ws.pair_info;
  ga.row_tok = ws.row_tok;
  ga.slot_w = ws.slot_w;
  ga.act = ws.act;
  ga.out = out;
  ga.out_f32 = acc;
  ga.err = ws.err;
  ga.wait_limit_ns = g_wait_limit_ns.load();
  ga.D = D;
  ga.H = H;
  ga.prefetch = g_prefetch.load();
  ga.stall_test = g_stall_test.load() == 1 ? 1 : 0;
  ga.swiglu_limit = ws.swiglu_limit;
  ga.counts = ws.counts;
  ga.pad_offsets = ws.pad_offsets;
  // swap-AB tiles reduce bf16 rows only
  ga.swap_ab = acc ? 0 : g_swap_ab.load();
  ga.pair_swap_max = acc ? 0 : g_pair_swap.load();
  ga.out_hint = out_hint_for((int64_t)T * D * 2);
  ga.l2_policy = ws.l2_policy;
  ga.half_m128 = g_half_m128.load();
  ga.down_epi8 = g_down_epi8.load();
  ga.up_swap = g_up_swap.load();

  const int dyn_opt = g_dynamic_tiles.load();
  const bool small_problem = (int64_t)ws.max_rb * (H / kUpFold) < 8LL * sms;
  const bool dyn = dyn_opt == 1 || (dyn_opt == 2 && small_problem);
  GemmArgs up = ga;
  up.tile_counter = dyn ? ws.meta + 2 : nullptr;
  up.n_col_tiles = H / fold;
  up.k_blocks = D / kBK;
  const int up_grid = (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * up.n_col_tiles * (kBM / bm));
  up.x = x;
  const int pair_slots = pair_mma ? pair_cluster_slots() : 0;
  if (pair_mma && pair_slots <= 0) return MOE_ERR_CUDA;
  prof_front(false);
  if (in_gemm_gather) prof_kernel(1, bands > 1 ? "band_order" : "none");  // rows gathered by the up kernel
  else if (bands > 1) prof_kernel(1, "gather_tokens+band_order");
  const bool wide_up = pair_mma && g_wide_up.load() == 1;
  const int wide_slots = wide_up ? pair_wide_cluster_slots() : 0;
  if (wide_up && wide_slots <= 0) return MOE_ERR_CUDA;
  prof_kernel(2, wide_up    ? "up_swiglu_pair2_wide"
                 : pair_mma ? "up_swiglu_pair2"
                 : (gather == 0 && g_up_pairs.load()) ? "up_pair_bf16"
                 : m64      ? "up_swiglu_bf16_m64"
                            : "up_swiglu_bf16");
  prof_kernel(3, pair_down ? (acc ? "down_reduce_pair2+f32_to_bf16" : "down_reduce_pair2")
                           : m64 ? (acc ? "down_reduce_bf16_m64+f32_to_bf16" : "down_reduce_bf16_m64")
                                 : (acc ? "down_reduce_bf16+f32_to_bf16" : "down_reduce_bf16"));
  if (wide_up)
    e = launch_up_pair2_wide_bf16(map_xg, map_w1, up,
                                  (int)std::min<int64_t>(wide_slots, (int64_t)ws.max_rb * ((up.n_col_tiles + 1) / 2)),
                                  st, !g_prof.on);
  else if (pair_mma)
    e = launch_up_pair2_bf16(map_xg, map_w1, map_w1_64, up,
                             (int)std::min<int64_t>(pair_slots, (int64_t)ws.max_rb * up.n_col_tiles), st, !g_prof.on);
  else if (gather == 0 && g_up_pairs.load())
    e = launch_up_pair_bf16(map_xg, map_w1, up, up_grid, st);
  else
    e = launch_up_bf16(map_xg, map_w1, up, up_grid, st, gather, fold, !g_prof.on, bm);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_mark(st, 3);

  GemmArgs dn = ga;
  dn.pair_order = bands > 1 ? ws.pair_order : nullptr;
  dn.tile_counter = dyn ? ws.meta + 3 : nullptr;
  dn.n_col_tiles = D / down_n;
  dn.k_blocks = H / kBK;
  const int dn_grid = (int)std::min<int64_t>(sms, (int64_t)ws.max_rb * dn.n_col_tiles * (kBM / bm));
  if (pair_down)
    e = launch_down_pair2_bf16(map_act, map_w2, dn,
                               (int)std::min<int64_t>(pair_slots, (int64_t)ws.max_rb * dn.n_col_tiles), st,
                               !g_prof.on);
  else
    e = launch_down_bf16(map_act, map_w2, dn, dn_grid, st, !g_prof.on, down_n, bm);
  if (e == cudaSuccess && acc) e = launch_f32_to_bf16(acc, out, (int64_t)T * D, sms * 4, st);
  prof_mark(st, 4);
  return cuda_status(e);
}

moe_status_t moe_ffn_forward(const void* x, const void* x_sf, const void* w1, const void* w1_sf, const void* w2,
                             const void* w2_sf, const int32_t* topk_ids, const float* topk_w, void* out, int T, int E,
                             int D, int H, int k, int dtype, int pipeline, void* workspace, size_t workspace_bytes,
                             void* stream) {
  return forward_entry(x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E, D, H, k, dtype, pipeline,
                       workspace, workspace_bytes, stream, nullptr);
}

// ---------------------------------------------------------------- host buffers
// Forward pass from host memory, tokens in chunks: the copy in of chunk c + 1
// (copy stream 1), the forward pass of chunk c (the caller's stream) and the
// copy out of chunk c - 1 (copy stream 2) run at the same time; two sets of
// device staging buffers alternate.  The copy streams and events are created
// once per device; a host mutex keeps one call's enqueue sequence whole.
namespace {
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, in_ready[2] = {}, computed[2] = {}, out_done[2] = {};
  bool ok = false;
};
std::mutex g_host_mu;
HostPipe g_host_pipe[64];

HostPipe* host_pipe() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  HostPipe& p = g_host_pipe[dev];
  if (p.ok) return &p;
  bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess;
  for (int b = 0; ok && b < 2; ++b)
    ok = cudaEventCreateWithFlags(&p.in_ready[b], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p.computed[b], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p.out_done[b], cudaEventDisableTiming) == cudaSuccess;
  p.ok = ok;
  return ok ? &p : nullptr;
}

int host_chunk_tokens(int T, int chunk_tokens) {
  if (chunk_tokens > 0) return std::min(chunk_tokens, std::max(T, 1));
  // automatic: whole problems up to 8192 tokens (their copies are short, and
  // smaller chunks lose GEMM efficiency); above, T / 8 rounded up to 128
  // tokens, at least 4096 (every chunk streams the weights once more) and at
  // most 16384
  if (T <= 8192) return std::max(T, 1);
  const int c = (int)(((int64_t)T + 8 * 128 - 1) / (8 * 128) * 128);
  return std::min(kHostChunkTokens, std::max(4096, c));
}

struct HostLayout {
  size_t fwd = 0, x = 0, x_sf = 0, ids = 0, tw = 0, out = 0, set = 0, bytes = 0;
};
HostLayout host_layout(int Tc, int E, int D, int H, int k, int dtype, int pipeline) {
  HostLayout l;
  l.fwd = align_up(plan_workspace(nullptr, Tc, E, D, H, k, pipeline, dtype).bytes, 256);
  l.x = align_up((size_t)Tc * D * (dtype == MOE_BF16 ? 2 : 1), 256);
  l.x_sf = dtype == MOE_BF16 ? 0 : align_up((size_t)Tc * D / 32, 256);
  l.ids = align_up((size_t)Tc * k * 4, 256);
  l.tw = l.ids;
  l.out = align_up((size_t)Tc * D * 2, 256);
  l.set = l.x + l.x_sf + l.ids + l.tw + l.out;
  l.bytes = l.fwd + 2 * l.set;
  return l;
}
}  // namespace

size_t moe_ffn_host_workspace_size(int T, int chunk_tokens, int E, int D, int H, int k, int dtype, int pipeline) {
  if (chunk_tokens < 0 || (dtype != MOE_BF16 && dtype != MOE_MXFP8 && dtype != MOE_MXFP4W)) return 0;
  const int Tc = host_chunk_tokens(T, chunk_tokens);
  if (moe_ffn_workspace_size(Tc, E, D, H, k, dtype, pipeline) == 0) return 0;
  return host_layout(Tc, E, D, H, k, dtype, pipeline).bytes;
}

moe_status_t moe_ffn_forward_host(const void* x_host, const void* x_sf_host, const void* w1, const void* w1_sf,
                                  const void* w2, const void* w2_sf, const int32_t* topk_ids_host,
                                  const float* topk_w_host, void* out_host, int T, int E, int D, int H, int k,
                                  int dtype, int pipeline, int chunk_tokens, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (!shape_ok(T, E, D, H, k) || chunk_tokens < 0) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 && dtype != MOE_MXFP8 && dtype != MOE_MXFP4W) return MOE_ERR_INVALID_ARG;
  if (pipeline != MOE_FUSED && pipeline != MOE_SPLIT) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !topk_ids_host || !topk_w_host || !out_host || !workspace || (dtype != MOE_BF16 && !x_sf_host))
    return MOE_ERR_INVALID_ARG;
  const int Tc = host_chunk_tokens(T, chunk_tokens);
  const HostLayout l = host_layout(Tc, E, D, H, k, dtype, pipeline);
  if (workspace_bytes < l.bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const size_t row = (size_t)D * (dtype == MOE_BF16 ? 2 : 1), row_sf = (size_t)D / 32;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  struct Set {
    uint8_t *x, *x_sf, *ids, *tw, *out;
  } set[2];
  for (int b = 0; b < 2; ++b) {
    uint8_t* p = base + l.fwd + b * l.set;
    set[b].x = p;
    set[b].x_sf = p + l.x;
    set[b].ids = p + l.x + l.x_sf;
    set[b].tw = set[b].ids + l.ids;
    set[b].out = set[b].tw + l.tw;
  }
  std::lock_guard<std::mutex> lock(g_host_mu);
  HostPipe* hp = host_pipe();
  if (!hp) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint8_t* xh = static_cast<const uint8_t*>(x_host);
  const uint8_t* xsh = static_cast<const uint8_t*>(x_sf_host);
  uint8_t* oh = static_cast<uint8_t*>(out_host);
  // both copy streams start behind everything already queued on the caller's stream
  cudaError_t e = cudaEventRecord(hp->start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->in, hp->start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->start, 0);
  // chunk c covers tokens [t0, t0 + tn).  With eight or more chunks the
  // first and the last are a quarter chunk: the copy in that nothing overlaps
  // and the copy out that nothing overlaps are then short (measured: with
  // fewer chunks the extra chunk costs more than it saves).
  const int q = g_host_ramp.load() && T >= 8 * Tc && Tc >= 512 ? Tc / 4 : 0;
  auto chunk_at = [&](int t0) {
    const int rem = T - t0;
    if (!q) return std::min(Tc, rem);
    if (t0 == 0) return q;
    if (rem > Tc + q) return Tc;
    return rem > 2 * q ? rem - q : rem;  // the tail: [rem - q, q], or rem whole
  };
  moe_status_t rs = MOE_OK;
  int t0 = 0;
  for (int c = 0; t0 < T && e == cudaSuccess && rs == MOE_OK; ++c) {
    const int b = c & 1, tn = chunk_at(t0);
    Set& sb = set[b];
    // in: buffers of set b are free once chunk c - 2's forward pass has read them
    if (c >= 2) e = cudaStreamWaitEvent(hp->in, hp->computed[b], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(sb.x, xh + (size_t)t0 * row, (size_t)tn * row, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess && dtype != MOE_BF16)
      e = cudaMemcpyAsync(sb.x_sf, xsh + (size_t)t0 * row_sf, (size_t)tn * row_sf, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(sb.ids, topk_ids_host + (size_t)t0 * k, (size_t)tn * k * 4, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(sb.tw, topk_w_host + (size_t)t0 * k, (size_t)tn * k * 4, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess) e = cudaEventRecord(hp->in_ready[b], hp->in);
    // forward pass of chunk c on the caller's stream, into out set b once
    // chunk c - 2's copy out has read it
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp->in_ready[b], 0);
    if (e == cudaSuccess && c >= 2) e = cudaStreamWaitEvent(st, hp->out_done[b], 0);
    if (e != cudaSuccess) break;
    rs = forward_entry(sb.x, dtype == MOE_BF16 ? nullptr : sb.x_sf, w1, w1_sf, w2, w2_sf,
                       reinterpret_cast<const int32_t*>(sb.ids), reinterpret_cast<const float*>(sb.tw), sb.out, tn,
                       E, D, H, k, dtype, pipeline, workspace, l.fwd, stream, nullptr);
    if (rs != MOE_OK) break;
    e = cudaEventRecord(hp->computed[b], st);
    // out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->computed[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(oh + (size_t)t0 * D * 2, sb.out, (size_t)tn * D * 2, cudaMemcpyDeviceToHost, hp->out);
    if (e == cudaSuccess) e = cudaEventRecord(hp->out_done[b], hp->out);
    t0 += tn;
  }
  // the caller's stream waits for the last copies out (and the copy streams
  // are joined back, so the call is one unit of work on the caller's stream)
  if (e == cudaSuccess) e = cudaEventRecord(hp->start, hp->out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp->start, 0);
  if (e == cudaSuccess) e = cudaEventRecord(hp->in_ready[0], hp->in);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp->in_ready[0], 0);
  if (rs != MOE_OK) return rs;
  return cuda_status(e);
}

moe_status_t moe_ffn_forward_logits(const void* x, const void* x_sf, const void* w1, const void* w1_sf,
                                    const void* w2, const void* w2_sf, const float* router_logits,
                                    int32_t* topk_ids, float* topk_w, void* out, int T, int E, int D, int H, int k,
                                    int dtype, int pipeline, void* workspace, size_t workspace_bytes, void* stream) {
  if (k > E) return MOE_ERR_INVALID_ARG;
  if (T > 0 && !router_logits) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(router_logits) & 3u) return MOE_ERR_MISALIGNED;
  return forward_entry(x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E, D, H, k, dtype, pipeline,
                       workspace, workspace_bytes, stream, router_logits);
}

moe_status_t moe_ffn_router_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                                 void* stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_w) & 3u))
    return MOE_ERR_MISALIGNED;
  return cuda_status(launch_router_topk(logits, T, E, k, topk_ids, topk_w, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_ffn_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (on && !g_prof.created) {
    for (int i = 0; i < kMaxProfileEvents; ++i)
      if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) return MOE_ERR_CUDA;
    g_prof.created = true;
  }
  g_prof.on = on != 0;
  g_prof.recorded = 0;
  return MOE_OK;
}

moe_status_t moe_ffn_profile_read(float* ms, int capacity, int* n_stages) {
  if (!ms || !n_stages) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  *n_stages = 0;
  if (!g_prof.created || g_prof.recorded < 2) return MOE_OK;
  if (cudaEventSynchronize(g_prof.ev[g_prof.recorded - 1]) != cudaSuccess) return MOE_ERR_CUDA;
  int n = 0;
  for (int i = 0; i + 1 < g_prof.recorded && n < capacity; ++i, ++n)
    if (cudaEventElapsedTime(&ms[n], g_prof.ev[i], g_prof.ev[i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
  *n_stages = n;
  return MOE_OK;
}

// Workspace of a call with shared experts: the plan of the extended problem
// (E + n_shared experts, k + n_shared pairs per token) followed by the
// extended ids and weights [T, k + n_shared].
static size_t ex_workspace_bytes(int T, int E, int D, int H, int k, int n_shared, int dtype, int pipeline,
                                 size_t* ext_offset) {
  const size_t base = plan_workspace(nullptr, T, E + n_shared, D, H, k + n_shared, pipeline, dtype).bytes;
  if (ext_offset) *ext_offset = base;
  if (n_shared == 0) return base;
  const size_t one = align_up(sizeof(int32_t) * (size_t)T * (k + n_shared), 256);
  return base + 2 * one;
}

size_t moe_ffn_workspace_size_ex(int T, int E, int D, int H, int k, int n_shared, int dtype, int pipeline) {
  if (n_shared < 0 || E + n_shared > kMaxExperts || !shape_ok(T, E + n_shared, D, H, k + n_shared) ||
      (dtype != MOE_BF16 && dtype != MOE_MXFP8 && dtype != MOE_MXFP4W && dtype != MOE_NVFP4) ||
      (pipeline != MOE_FUSED && pipeline != MOE_SPLIT) || (dtype == MOE_NVFP4 && pipeline != MOE_SPLIT))
    return 0;
  return ex_workspace_bytes(T, E, D, H, k, n_shared, dtype, pipeline, nullptr);
}

moe_status_t moe_ffn_forward_ex(const void* x, const void* x_sf, const void* w1, const void* w1_sf, const void* w2,
                                const void* w2_sf, int32_t* topk_ids, float* topk_w, void* out, int T, int E, int D,
                                int H, int k, int dtype, int pipeline, const moe_ffn_extras_t* extras,
                                void* workspace, size_t workspace_bytes, void* stream) {
  const float limit = extras ? extras->swiglu_limit : 0.f;
  const int ns = extras ? extras->n_shared : 0;
  const float* logits = extras ? extras->router_logits : nullptr;
  if (!(limit >= 0.f) || ns < 0 || E + ns > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (logits && (k > E || (reinterpret_cast<uintptr_t>(logits) & 3u))) return MOE_ERR_INVALID_ARG;
  if (ns == 0)
    return forward_entry(x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E, D, H, k, dtype, pipeline,
                         workspace, workspace_bytes, stream, logits, limit);
  if (!shape_ok(T, E + ns, D, H, k + ns)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !topk_w || !workspace) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(topk_ids) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u))
    return MOE_ERR_MISALIGNED;
  size_t ext_off = 0;
  if (workspace_bytes < ex_workspace_bytes(T, E, D, H, k, ns, dtype, pipeline, &ext_off))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // routed ids and weights first (the router, when the call starts from
  // logits), then [T, k + n_shared] with every shared expert at weight 1
  int32_t* ids_ext = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + ext_off);
  float* w_ext = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ids_ext) +
                                          align_up(sizeof(int32_t) * (size_t)T * (k + ns), 256));
  cudaError_t e = cudaSuccess;
  if (logits) e = launch_router_topk(logits, T, E, k, topk_ids, topk_w, st);
  if (e == cudaSuccess) e = launch_extend_routing(topk_ids, topk_w, T, E, k, ns, ids_ext, w_ext, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return forward_entry(x, x_sf, w1, w1_sf, w2, w2_sf, ids_ext, w_ext, out, T, E + ns, D, H, k + ns, dtype, pipeline,
                       workspace, ext_off, stream, nullptr, limit);
}

const char* moe_ffn_profile_stage_kernel(int stage) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (stage < 0 || stage + 1 >= g_prof.recorded) return nullptr;
  return g_prof.kernel[stage];
}

moe_status_t moe_ffn_prepare_mxfp8_weights(const void* w1_sf, const void* w2_sf, void* w1_sf_packed,
                                           void* w2_sf_packed, int E, int D, int H, void* stream) {
  if (E < 1 || D < 128 || H < 128 || D % 128 || H % 128) return MOE_ERR_INVALID_ARG;
  if (!w1_sf || !w2_sf || !w1_sf_packed || !w2_sf_packed) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w1_sf) & 3u) || (reinterpret_cast<uintptr_t>(w2_sf) & 3u) ||
      !aligned16(w1_sf_packed) || !aligned16(w2_sf_packed))
    return MOE_ERR_MISALIGNED;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_pack_sf(w1_sf, w1_sf_packed, (int64_t)E * 2 * H, D, sms * 4, st);
  if (e == cudaSuccess) e = launch_pack_sf(w2_sf, w2_sf_packed, (int64_t)E * D, H, sms * 4, st);
  return cuda_status(e);
}

moe_status_t moe_ffn_widen_mxfp4_weights(const void* w_fp4, int64_t n_elems, void* w_e4m3, void* stream) {
  if (n_elems < 0 || n_elems % 32) return MOE_ERR_INVALID_ARG;
  if (n_elems == 0) return MOE_OK;
  if (!w_fp4 || !w_e4m3) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_fp4) || !aligned16(w_e4m3)) return MOE_ERR_MISALIGNED;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  return cuda_status(launch_widen_e2m1(w_fp4, n_elems / 2, w_e4m3, sms * 8, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_ffn_debug_mx_quantize(const float* in, int64_t n, uint8_t* q, uint8_t* sf, void* stream) {
  if (n < 0 || n % 32 || (n > 0 && (!in || !q || !sf))) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  return cuda_status(launch_mx_quantize(in, n, q, sf, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_ffn_prepare_nvfp4_weights(const void* w1_sf, const void* w2_sf, void* w1_sf_packed,
                                           void* w2_sf_packed, int E, int D, int H, void* stream) {
  if (E < 1 || D < 256 || H < 256 || D % 256 || H % 256) return MOE_ERR_INVALID_ARG;
  if (!w1_sf || !w2_sf || !w1_sf_packed || !w2_sf_packed) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w1_sf) & 3u) || (reinterpret_cast<uintptr_t>(w2_sf) & 3u) ||
      !aligned16(w1_sf_packed) || !aligned16(w2_sf_packed))
    return MOE_ERR_MISALIGNED;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the packing groups four scale bytes of a row per 512-byte tile: 4 x 32
  // elements of MXFP8 scales, or 4 x 16 elements of NVFP4 scales (K doubled)
  cudaError_t e = launch_pack_sf(w1_sf, w1_sf_packed, (int64_t)E * 2 * H, 2 * D, sms * 4, st);
  if (e == cudaSuccess) e = launch_pack_sf(w2_sf, w2_sf_packed, (int64_t)E * D, 2 * H, sms * 4, st);
  return cuda_status(e);
}

moe_status_t moe_ffn_forward_nvfp4(const void* x, const void* x_sf, const void* w1, const void* w1_sf, const void* w2,
                                   const void* w2_sf, const moe_ffn_nvfp4_scales_t* gs, const int32_t* topk_ids,
                                   const float* topk_w, void* out, int T, int E, int D, int H, int k,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (!shape_ok(T, E, D, H, k) || D % 256 || H % 256) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !x_sf || !w1 || !w1_sf || !w2 || !w2_sf || !gs || !topk_ids || !topk_w || !out || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (!gs->x_gs || !gs->w1_gs || !gs->w2_gs || !gs->act_gs) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w1) || !aligned16(w2) || !aligned16(out) || !aligned16(workspace) ||
      !aligned16(w1_sf) || !aligned16(w2_sf) || (reinterpret_cast<uintptr_t>(x_sf) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_ids) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u) ||
      (reinterpret_cast<uintptr_t>(gs->x_gs) & 3u) || (reinterpret_cast<uintptr_t>(gs->w1_gs) & 3u) ||
      (reinterpret_cast<uintptr_t>(gs->w2_gs) & 3u) || (reinterpret_cast<uintptr_t>(gs->act_gs) & 3u))
    return MOE_ERR_MISALIGNED;
  Workspace ws = plan_workspace(workspace, T, E, D, H, k, MOE_SPLIT, MOE_NVFP4);
  if (workspace_bytes < ws.bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  return forward_split_nvfp4(ws, x, x_sf, w1, w1_sf, w2, w2_sf, *gs, topk_ids, topk_w, out, T, E, D, H, k, sms,
                             static_cast<cudaStream_t>(stream));
}

moe_status_t moe_ffn_sync_status(void* workspace, void* stream) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int words[2] = {0, 0};
  // read and clear on the call's own stream (no legacy-default-stream sync)
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(words, workspace, sizeof words, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(workspace, 0, 64, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (words[0] & kErrLaunch) return MOE_ERR_CUDA;
  if (words[0] & kErrTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  if (words[0] & kErrBadRouting) return MOE_ERR_BAD_ROUTING;
  return MOE_OK;
}

const char* moe_ffn_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape, dtype or pipeline";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MOE_ERR_BAD_ROUTING: return "expert id outside [0, E)";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out; output is invalid";
    case MOE_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

}  // extern "C"
