// gemm_mxfp8.cu -- the MXFP8 variant of the split pipeline ("Prime Flash MoE"
// sec. 7 "The MXFP8 variant"): e4m3 data with one ue8m0 scale per 32 elements
// along K, tcgen05.mma kind::mxf8f6f4 block_scale, scales copied from shared
// memory into tensor memory with tcgen05.cp before the MMAs that read them.
//
// UP:   acc[128 x 256] = (xg * s_x) . ([W1 gate j | W1 up j] * s_w1)^T over K=D,
//       act = silu(gate) * up in fp32, requantized per 32 along H to e4m3 +
//       ue8m0 (sec. 7 "The epilogue also quantizes"), stored with its scale
//       tiles in the blocked layout the down kernel's tcgen05.cp expects
//       (sec. 7 "The split variant, in MXFP8").
// DOWN: acc[128 x 256] = (act * s_act) . (W2[e][n] * s_w2)^T over K=H, weighted
//       by the routing weight in fp32, rounded to bf16 and reduced into out
//       with one bulk reduction per row.
// A stage holds K = 128 (four MMAs of K = 32, one UTCCP group: sec. 7 "this is
// also the reason the MXFP8 kernel uses BK = 128").  The accumulator takes 256
// TMEM columns, so it is single-buffered and the scale sets sit behind it at
// columns 256 + 16 * stage_slot (sec. 7: the scale columns rotate so in-flight
// stages never overwrite each other's scales).  The epilogue frees the
// accumulator as soon as it has read it; eight epilogue warps (two per TMEM
// lane quadrant, each taking half of the columns) keep that window short.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

enum { kMxUp = 0, kMxDown = 1 };
constexpr int kMxBK = 128;                  // fp8 elements (bytes) per stage row
constexpr int kMxN = 256;
constexpr int kMxThreads = 64 + 256;   // producer warp, MMA warp, 8 epilogue warps
constexpr int kMxEpi = 256;            // two warps per TMEM lane quadrant, one per column half
constexpr uint64_t kMxDrainNs = 200ull * 1000 * 1000;

// FP4W: the weights (B operand) are MXFP4, E2M1 codes packed two per byte in
// global memory.  Their tensor map (16U4_ALIGN16B) spreads each 16 codes (8
// bytes) over a 16-byte slot of shared memory, so a B tile keeps the e4m3
// tile's geometry (128 K elements per 128-byte swizzled row, "Porting
// Block-Scaled GEMM Kernels" sec. 2.1: on sm_103a kind::mxf8f6f4 reads a 4-bit
// operand next to an 8-bit one from such 1-byte-per-element containers),
// while only the packed bytes cross from global memory: they are what the
// stage's transaction count expects.  The instruction descriptor gives B the
// E2M1 code of kind::mxf8f6f4, 5 (sec. 2.3).
template <int MODE, int STAGES, int FP4W = 0>
struct MxCfg {
  static constexpr int kA = kBM * kMxBK;          // 16 KB
  static constexpr int kB = kMxN * kMxBK;         // 32 KB of shared memory
  static constexpr int kSF = 512 * 3;             // SFA tile + two SFB tiles
  static constexpr int kTx = kA + (FP4W ? kB / 2 : kB) + kSF;
  // DOWN: each epilogue thread stages half an output row (128 bf16, +16 B so
  // a warp's rows fall on distinct banks) for its bulk reduction.
  static constexpr int kStageRowBytes = kMxN + 16;
  static constexpr int kStaging = MODE == kMxDown ? kMxEpi * kStageRowBytes : 0;
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmem = 1024 + STAGES * (kA + kB + kSF) + kStaging + kBarrierBytes;
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(256 + 16 * STAGES <= 512, "TMEM columns");
};

__device__ __forceinline__ float mx_u2f(uint32_t u) { return __uint_as_float(u); }
// silu(g) * u with the optional clamp (lim = +inf when off): g <= lim,
// -lim <= u <= lim.
__device__ __forceinline__ float mx_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

template <int MODE, int STAGES, int FP4W = 0>
__global__ void __launch_bounds__(kMxThreads, 1)
    grouped_gemm_mxfp8_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                              const MxArgs args) {
  using Cfg = MxCfg<MODE, STAGES, FP4W>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * Cfg::kA;
  uint8_t* sSF = sB + STAGES * Cfg::kB;
  uint8_t* sStage = sSF + STAGES * Cfg::kSF;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + Cfg::kStaging);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* never = drain + 1;  // no thread ever arrives here (failure-path test hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kMxEpi);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (MODE == kMxUp && threadIdx.x == 0) griddep_launch_dependents();

  const int num_rb = args.meta[0];
  const int n_tiles = num_rb * args.n_col_tiles;
  const int KB = args.k_blocks;             // K / 128
  // row block of a tile: in token-band order for DOWN when an order is given
  auto tile_rb = [&](int tile) {
    const int i = tile / args.n_col_tiles;
    return (MODE == kMxDown && args.rb_order) ? args.rb_order[i] : i;
  };
  const uint8_t* sf_a = static_cast<const uint8_t*>(args.sf_a);
  const uint8_t* sf_b = static_cast<const uint8_t*>(args.sf_b);

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    if (MODE == kMxDown) griddep_wait();
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[STAGES];
#pragma unroll
    for (int i = 0; i < STAGES; ++i) issued_phase[i] = -1;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
      const int rb = tile_rb(tile), j = tile % args.n_col_tiles;
      const int e = args.expert_of_rb[rb];
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&empty[s], ph ^ 1u, wc, 21))) break;
        mbar_arrive_expect_tx(&full[s], Cfg::kTx);
        issued_phase[s] = (int)ph;
        uint8_t* a = sA + s * Cfg::kA;
        uint8_t* b = sB + s * Cfg::kB;
        uint8_t* sf = sSF + s * Cfg::kSF;
        tma_load_2d(a, &map_a, &full[s], kb * kMxBK, rb * kBM);
        bulk_load(sf, sf_a + sf_tile_offset(rb, kb, KB), 512, &full[s]);
        if (MODE == kMxUp) {
          const int rt_gate = e * (2 * args.H / 128) + j;   // 128-row tiles of W1 [E*2H, D]
          const int rt_up = rt_gate + args.H / 128;
          tma_load_2d(b, &map_b, &full[s], kb * kMxBK, rt_gate * 128);
          tma_load_2d(b + 128 * kMxBK, &map_b, &full[s], kb * kMxBK, rt_up * 128);
          bulk_load(sf + 512, sf_b + sf_tile_offset(rt_gate, kb, KB), 512, &full[s]);
          bulk_load(sf + 1024, sf_b + sf_tile_offset(rt_up, kb, KB), 512, &full[s]);
        } else {
          const int rt0 = e * (args.D / 128) + j * 2;       // 128-row tiles of W2 [E*D, H]
          tma_load_2d(b, &map_b, &full[s], kb * kMxBK, rt0 * 128);
          bulk_load(sf + 512, sf_b + sf_tile_offset(rt0, kb, KB), 512, &full[s]);
          bulk_load(sf + 1024, sf_b + sf_tile_offset(rt0 + 1, kb, KB), 512, &full[s]);
        }
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      for (int i = 0; i < STAGES; ++i)
        if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kMxDrainNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_mxf8(kBM, kMxN) | (FP4W ? kFmtE2M1 << 10 : 0u);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 92);  // runs out after the wait limit
    int it = 0;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++it) {
      if (!(ok = mbar_wait(tempty, ((uint32_t)it & 1u) ^ 1u, wc, 22))) break;
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&full[s], ph, wc, 23))) break;
        tc_fence_after();
        // scale tiles of this stage -> TMEM columns reserved for this ring slot
        const uint32_t sfa_col = tmem_base + 256 + 16 * s, sfb_col = sfa_col + 4;
        const uint32_t sf_smem = smem_addr(sSF + s * Cfg::kSF);
        utccp_sf(sfa_col, sdesc_sf_tile(sf_smem));
        utccp_sf(sfb_col, sdesc_sf_tile(sf_smem + 512));
        utccp_sf(sfb_col + 4, sdesc_sf_tile(sf_smem + 1024));
        const uint64_t ad = sdesc_sw128(smem_addr(sA + s * Cfg::kA));
        const uint64_t bd = sdesc_sw128(smem_addr(sB + s * Cfg::kB));
#pragma unroll
        for (int kk = 0; kk < kMxBK / 32; ++kk)
          umma_mxf8(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc_with_sf_id(idesc, kk), sfa_col, sfb_col,
                    (kb | kk) != 0);
        umma_commit(&empty[s]);
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit(tfull);
    }
    if (!ok) {
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kMxDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;      // which half of the accumulator columns
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_stage = sStage + (half * kBM + row) * Cfg::kStageRowBytes;
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      if (!mbar_wait(tfull, (uint32_t)it & 1u, wc, 24)) break;
      tc_fence_after();
      const int rb = tile_rb(tile), j = tile % args.n_col_tiles;
      const int64_t slot = (int64_t)rb * kBM + row;
      const int tok = args.row_tok[slot];
      if (MODE == kMxUp) {
        // columns [64 half, 64 half + 64) of gate (0..127) and of up (128..255)
        float act[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t g[32], u[32];
          const int col = half * 64 + c * 32;
          tmem_ld_x32_pair(lane_base + col, lane_base + 128 + col, g, u);
#pragma unroll
          for (int i = 0; i < 32; ++i) act[c * 32 + i] = mx_swiglu(mx_u2f(g[i]), mx_u2f(u[i]), swiglu_lim);
        }
        tc_fence_before();
        mbar_arrive(tempty);  // the accumulator is free once all 256 threads have read it
        if (tok >= 0) {
          uint8_t* dst = static_cast<uint8_t*>(args.act) + slot * args.H + j * 128 + half * 64;
          uint32_t sfw = 0;
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            uint32_t q[8];
            const uint32_t sfb = mx_quantize32(act + blk * 32, q);
            sfw |= sfb << (8 * blk);
            st_global_v4(dst + blk * 32, q[0], q[1], q[2], q[3]);
            st_global_v4(dst + blk * 32 + 16, q[4], q[5], q[6], q[7]);
          }
          uint8_t* sfdst = static_cast<uint8_t*>(args.act_sf) + sf_tile_offset(rb, j, args.H / 128) + sf_in_tile(row) +
                           half * 2;
          *reinterpret_cast<uint16_t*>(sfdst) = (uint16_t)sfw;
        }
      } else if (args.out_f32) {
        // fp32 reduction target: this thread's 128 columns read at once (the
        // accumulator is then free), staged and reduced as two 256-byte chunks
        const float w = args.slot_w[slot];
        uint32_t v[4][32];
        tmem_ld_x32_pair(lane_base + half * 128, lane_base + half * 128 + 32, v[0], v[1]);
        tmem_ld_x32_pair(lane_base + half * 128 + 64, lane_base + half * 128 + 96, v[2], v[3]);
        tc_fence_before();
        mbar_arrive(tempty);
        if (tok >= 0) {
          float* frow = args.out_f32 + (int64_t)tok * args.D + j * kMxN + half * 128;
#pragma unroll
          for (int c = 0; c < 4; c += 2) {
            bulk_wait_read_all();
            stage_scaled_f32x32(my_stage, w, v[c]);
            stage_scaled_f32x32(my_stage + 128, w, v[c + 1]);
            fence_proxy_async_smem();
            bulk_reduce_add_f32(frow + c * 32, my_stage, 256);
            bulk_commit();
          }
        }
      } else {
        const float w = args.slot_w[slot];
        bulk_wait_read_all();
#pragma unroll 1
        for (int c = 0; c < 4; c += 2) {   // 4 chunks of 32 columns = this thread's half
          uint32_t v0[32], v1[32];
          const int col = half * 128 + c * 32;
          tmem_ld_x32_pair(lane_base + col, lane_base + col + 32, v0, v1);
          if (tok >= 0) {
#pragma unroll
            for (int qd = 0; qd < 4; ++qd)
              st_shared_v4(my_stage + c * 64 + qd * 16, pack_bf16x2(w * mx_u2f(v0[8 * qd]), w * mx_u2f(v0[8 * qd + 1])),
                           pack_bf16x2(w * mx_u2f(v0[8 * qd + 2]), w * mx_u2f(v0[8 * qd + 3])),
                           pack_bf16x2(w * mx_u2f(v0[8 * qd + 4]), w * mx_u2f(v0[8 * qd + 5])),
                           pack_bf16x2(w * mx_u2f(v0[8 * qd + 6]), w * mx_u2f(v0[8 * qd + 7])));
#pragma unroll
            for (int qd = 0; qd < 4; ++qd)
              st_shared_v4(my_stage + (c + 1) * 64 + qd * 16,
                           pack_bf16x2(w * mx_u2f(v1[8 * qd]), w * mx_u2f(v1[8 * qd + 1])),
                           pack_bf16x2(w * mx_u2f(v1[8 * qd + 2]), w * mx_u2f(v1[8 * qd + 3])),
                           pack_bf16x2(w * mx_u2f(v1[8 * qd + 4]), w * mx_u2f(v1[8 * qd + 5])),
                           pack_bf16x2(w * mx_u2f(v1[8 * qd + 6]), w * mx_u2f(v1[8 * qd + 7])));
          }
        }
        tc_fence_before();
        mbar_arrive(tempty);
        if (tok >= 0) {
          fence_proxy_async_smem();
          bulk_reduce_add_bf16_hint(static_cast<__nv_bfloat16*>(args.out) + (int64_t)tok * args.D + j * kMxN + half * 128,
                               my_stage, kMxN, args.out_hint != 0, l2_policy_evict_last());
          bulk_commit();
        }
      }
    }
    if (MODE == kMxDown) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int MODE, int STAGES, int FP4W = 0>
cudaError_t launch_mx(const CUtensorMap& a, const CUtensorMap& b, const MxArgs& args, int grid, cudaStream_t stream,
                      bool pdl) {
  using Cfg = MxCfg<MODE, STAGES, FP4W>;
  auto kern = grouped_gemm_mxfp8_kernel<MODE, STAGES, FP4W>;
  // once per device: not a stream operation, so it stays out of graph capture
  static bool smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (err != cudaSuccess) return err;
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMxThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, b, args);
}

// Token-major gather of e4m3 rows: one warp per (token, 4 KB chunk of its code
// row); the chunk is read once (16-byte loads, eight per lane) and written to
// each of the token's k padded slots, so x is read once rather than k times.
// The same warps zero-fill the token's row of `out` (the reduction target).
// Then the scales: row-major x_sf[T, D/32] into the blocked 512-byte tiles of
// xg_sf, slot by slot (padding rows get scale 1.0; their codes are never
// written: each GEMM output row depends only on its own input row and padding
// rows are dropped by the epilogues).  Launched as a programmatic dependent of
// the routing.
constexpr int kMxGatherChunkVecs = 256;

__global__ void __launch_bounds__(256)
    gather_tokens_mx_kernel(const uint4* __restrict__ x, const uint32_t* __restrict__ x_sf,
                            const int32_t* __restrict__ ids, const int* __restrict__ slot_of_pair,
                            const int* __restrict__ offsets, const int* __restrict__ pad_offsets,
                            const int* __restrict__ row_tok, const int* __restrict__ meta, int T, int E, int k,
                            int vec_per_row, int kt_per_row, uint4* __restrict__ xg, uint8_t* __restrict__ xg_sf,
                            uint4* __restrict__ out, int out_vecs_per_row, uint32_t pad_sf) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_chunks = (vec_per_row + kMxGatherChunkVecs - 1) / kMxGatherChunkVecs;
  const int zero_per = (out_vecs_per_row + n_chunks - 1) / n_chunks;
  const int64_t items = (int64_t)T * n_chunks;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t gwarp = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  for (int64_t it = gwarp; it < items; it += nwarps) {
    const int t = (int)(it / n_chunks), c = (int)(it % n_chunks);
    const int v0 = c * kMxGatherChunkVecs;
    const uint4* src = x + (int64_t)t * vec_per_row + v0;
    uint4 v[kMxGatherChunkVecs / 32];
#pragma unroll
    for (int i = 0; i < kMxGatherChunkVecs / 32; ++i)
      if (v0 + i * 32 + lane < vec_per_row) v[i] = __ldg(src + i * 32 + lane);
    for (int j0 = 0; j0 < k; j0 += 32) {
      int ps = -1;  // lane l resolves the padded slot of pair j0 + l
      if (j0 + lane < k) {
        const int64_t p = (int64_t)t * k + j0 + lane;
        const int e = ids[p], s = slot_of_pair[p];
        if (s >= 0 && (unsigned)e < (unsigned)E) ps = s - offsets[e] + pad_offsets[e];
      }
      const int nj = min(32, k - j0);
      for (int jj = 0; jj < nj; ++jj) {
        const int slot = __shfl_sync(0xffffffffu, ps, jj);
        if (slot < 0) continue;
        uint4* dst = xg + (int64_t)slot * vec_per_row + v0;
#pragma unroll
        for (int i = 0; i < kMxGatherChunkVecs / 32; ++i)
          if (v0 + i * 32 + lane < vec_per_row) dst[i * 32 + lane] = v[i];
      }
    }
    if (out) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      uint4* orow = out + (int64_t)t * out_vecs_per_row;
      const int z1 = min(out_vecs_per_row, (c + 1) * zero_per);
      for (int i = c * zero_per + lane; i < z1; i += 32) orow[i] = z;
    }
  }
  // scales: one warp per (row block, K tile) writes the blocked 512-byte tile
  // with coalesced 16-byte stores, lane l gathering the 4-byte scale words of
  // rows l, l + 32, l + 64, l + 96 (padding rows: pad_sf, an e8m0 scale of 1.0
  // for MXFP8, a zero e4m3 scale for NVFP4)
  const int64_t n_sf_tiles = (int64_t)meta[0] * kt_per_row;
  for (int64_t q = gwarp; q < n_sf_tiles; q += nwarps) {
    const int64_t rb = q / kt_per_row;
    const int kt = (int)(q % kt_per_row);
    uint32_t wv[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int tok = row_tok[rb * kRowPad + g * 32 + lane];
      wv[g] = tok >= 0 ? __ldg(x_sf + (int64_t)tok * kt_per_row + kt) : pad_sf;
    }
    *reinterpret_cast<uint4*>(xg_sf + sf_tile_offset(rb, kt, kt_per_row) + lane * 16) =
        make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
}

// Row-major scales sf[rows, K/32] -> blocked tiles (rows % 128 == 0).
__global__ void __launch_bounds__(256) pack_sf_kernel(const uint32_t* __restrict__ sf, uint8_t* __restrict__ packed,
                                                      int64_t rows, int K) {
  const int kt_per_row = K / 128;
  const int64_t n = rows * kt_per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / kt_per_row;
    const int kt = (int)(i % kt_per_row);
    *reinterpret_cast<uint32_t*>(packed + sf_tile_offset(row / 128, kt, kt_per_row) + sf_in_tile((int)(row % 128))) =
        sf[i];
  }
}

// Test hook: the epilogue's requantization applied to n fp32 values.
__global__ void mx_quantize_kernel(const float* __restrict__ in, int64_t n_blocks, uint8_t* __restrict__ q,
                                   uint8_t* __restrict__ sf) {
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks; b += (int64_t)gridDim.x * blockDim.x) {
    float a[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] = in[b * 32 + i];
    uint32_t qq[8];
    sf[b] = (uint8_t)mx_quantize32(a, qq);
#pragma unroll
    for (int i = 0; i < 8; ++i) reinterpret_cast<uint32_t*>(q + b * 32)[i] = qq[i];
  }
}

}  // namespace

cudaError_t launch_up_mxfp8(const CUtensorMap& a, const CUtensorMap& w1, const MxArgs& args, int grid,
                            cudaStream_t stream, bool fp4w) {
  if (fp4w) return launch_mx<kMxUp, 4, 1>(a, w1, args, grid, stream, false);
  return launch_mx<kMxUp, 4>(a, w1, args, grid, stream, false);
}
cudaError_t launch_down_mxfp8(const CUtensorMap& act, const CUtensorMap& w2, const MxArgs& args, int grid,
                              cudaStream_t stream, bool pdl, bool fp4w) {
  if (fp4w) return launch_mx<kMxDown, 3, 1>(act, w2, args, grid, stream, pdl);
  return launch_mx<kMxDown, 3>(act, w2, args, grid, stream, pdl);
}
cudaError_t launch_gather_mx(const Workspace& ws, const void* x, const void* x_sf, const int32_t* topk_ids, int T,
                             int E, int k, int D, void* out, int64_t out_bytes, int grid, cudaStream_t stream,
                             bool pdl, bool nv) {
  if (T == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gather_tokens_mx_kernel, static_cast<const uint4*>(x),
                            static_cast<const uint32_t*>(x_sf), topk_ids, static_cast<const int*>(ws.slot_of_pair),
                            static_cast<const int*>(ws.offsets), static_cast<const int*>(ws.pad_offsets),
                            static_cast<const int*>(ws.row_tok), static_cast<const int*>(ws.meta), T, E, k,
                            nv ? D / 32 : D / 16, nv ? D / 64 : D / 128, static_cast<uint4*>(ws.xg),
                            static_cast<uint8_t*>(ws.xg_sf), static_cast<uint4*>(out),
                            out ? (int)(out_bytes / 16 / T) : 0, nv ? 0u : 0x7f7f7f7fu);
}
cudaError_t launch_pack_sf(const void* sf, void* packed, int64_t rows, int K, int grid, cudaStream_t stream) {
  pack_sf_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint32_t*>(sf), static_cast<uint8_t*>(packed), rows, K);
  return cudaGetLastError();
}
cudaError_t launch_mx_quantize(const float* in, int64_t n, uint8_t* q, uint8_t* sf, cudaStream_t stream) {
  const int64_t nb = n / 32;
  const int grid = (int)std::min<int64_t>((nb + 127) / 128, 4096);
  mx_quantize_kernel<<<grid > 0 ? grid : 1, 128, 0, stream>>>(in, nb, q, sf);
  return cudaGetLastError();
}

}  // namespace moe
