// gemm_fused_mx.cu -- the fused pipeline in MXFP8 ("Prime Flash MoE" sec. 7:
// the pipeline, the split-K and the shared ring carry over from bf16, the
// epilogue requantizes act, and the down loop runs its jobs one after another
// on a single accumulator).
//
// Per tile (128-row block rb, 128-wide slice j of H):
//   GEMM1  acc[128 x 256] = (xg * s_x) . ([W1 gate j | up j] * s_w1)^T over K=D,
//          block-scaled kind::mxf8f6f4, scales copied to TMEM per stage;
//   SwiGLU in fp32, requantized per 32 columns to e4m3 + ue8m0 straight into
//          shared memory: the codes in the 128-byte-swizzled K-major layout of
//          GEMM2's A operand, the scales as one 512-byte tile for tcgen05.cp
//          (sec. 7 "The epilogue also quantizes": the intermediate never
//          leaves the SM);
//   GEMM2  for each 256-column chunk n of D: acc = (act * s_act) . (W2[e][n
//          rows, slice j] * s_w2)^T (K = 128, one stage);
//   reduce w * acc in fp32 into out_f32 with cp.reduce.async.bulk .add.f32
//          (fp32 for the same accuracy reason as the bf16 fused kernel).
// The accumulator takes TMEM columns [0, 256) and every job (GEMM1 or one
// GEMM2 chunk) waits for the epilogue to drain the previous one; the scale
// sets of the ring slots sit at 256 + 16 * slot.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kXStages = 3;
constexpr int kXThreads = 192;
constexpr int kXEpi = 128;
constexpr int kXBK = 128;                        // fp8 bytes per K stage
constexpr int kXA = kBM * kXBK;                  // 16 KB
constexpr int kXB = 256 * kXBK;                  // 32 KB
constexpr int kXSF = 3 * 512;                    // A tile + two B tiles
constexpr int kXActBytes = kBM * 128;            // act codes: 128 rows x 128 e4m3
constexpr int kXActSF = 512;                     // act scale tile
constexpr int kXRedCols = 64;                    // fp32 columns per bulk reduction
constexpr int kXRedRow = kXRedCols * 4 + 16;
constexpr int kXRed = kBM * kXRedRow;
constexpr int kXSmem = 1024 + kXStages * (kXA + kXB + kXSF) + kXActBytes + kXActSF + kXRed + 256;
static_assert(kXSmem <= 232448, "shared memory");
static_assert(256 + 16 * kXStages <= 512, "TMEM columns");
constexpr uint64_t kXDrainNs = 200ull * 1000 * 1000;

__device__ __forceinline__ float x_u2f(uint32_t u) { return __uint_as_float(u); }
// silu(g) * u with the optional clamp (lim = +inf when off): g <= lim,
// -lim <= u <= lim.
__device__ __forceinline__ float x_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__global__ void __launch_bounds__(kXThreads, 1)
    fused_moe_mxfp8_kernel(const __grid_constant__ CUtensorMap map_xg, const __grid_constant__ CUtensorMap map_w1,
                           const __grid_constant__ CUtensorMap map_w2, const FusedMxArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                            // SW128 operands first: 1024-byte aligned
  uint8_t* sB = sA + kXStages * kXA;
  uint8_t* act = sB + kXStages * kXB;
  uint8_t* sSF = act + kXActBytes;
  uint8_t* act_sf = sSF + kXStages * kXSF;
  uint8_t* red = act_sf + kXActSF;
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kXRed);
  uint64_t* empty = full + kXStages;
  uint64_t* tfull = empty + kXStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* act_full = tempty + 1;
  uint64_t* drain = act_full + 1;
  uint64_t* never = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kXStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kXEpi);
    mbar_init(act_full, kXEpi);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_xg);
    prefetch_tmap(&map_w1);
    prefetch_tmap(&map_w2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int NS = args.H / 128;              // slices
  const int n_tiles = args.meta[0] * NS;
  const int K1 = args.D / kXBK;             // GEMM1 stages per tile
  const int NO = args.D / 256;              // GEMM2 jobs per tile
  const uint8_t* xg_sf = static_cast<const uint8_t*>(args.xg_sf);
  const uint8_t* w1_sf = static_cast<const uint8_t*>(args.w1_sf);
  const uint8_t* w2_sf = static_cast<const uint8_t*>(args.w2_sf);

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[kXStages] = {-1, -1, -1};
    bool ok = true;
    auto acquire = [&](uint32_t bytes) -> bool {
      if (!mbar_wait(&empty[s], ph ^ 1u, wc, 41)) return false;
      mbar_arrive_expect_tx(&full[s], bytes);
      issued_phase[s] = (int)ph;
      return true;
    };
    auto advance = [&]() {
      if (++s == kXStages) {
        s = 0;
        ph ^= 1u;
      }
    };
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
      const int rb = tile / NS, j = tile % NS;
      const int e = args.expert_of_rb[rb];
      const int rt_gate = e * (2 * args.H / 128) + j, rt_up = rt_gate + args.H / 128;
      for (int kb = 0; ok && kb < K1; ++kb) {
        if (!(ok = acquire(kXA + kXB + kXSF))) break;
        uint8_t* b = sB + s * kXB;
        uint8_t* sf = sSF + s * kXSF;
        tma_load_2d(sA + s * kXA, &map_xg, &full[s], kb * kXBK, rb * kBM);
        tma_load_2d(b, &map_w1, &full[s], kb * kXBK, rt_gate * 128);
        tma_load_2d(b + 128 * kXBK, &map_w1, &full[s], kb * kXBK, rt_up * 128);
        bulk_load(sf, xg_sf + sf_tile_offset(rb, kb, K1), 512, &full[s]);
        bulk_load(sf + 512, w1_sf + sf_tile_offset(rt_gate, kb, K1), 512, &full[s]);
        bulk_load(sf + 1024, w1_sf + sf_tile_offset(rt_up, kb, K1), 512, &full[s]);
        advance();
      }
      for (int n = 0; ok && n < NO; ++n) {
        if (!(ok = acquire(kXB + 1024))) break;
        const int rt0 = e * (args.D / 128) + 2 * n;   // 128-row tiles of W2 [E*D, H]
        uint8_t* sf = sSF + s * kXSF;
        tma_load_2d(sB + s * kXB, &map_w2, &full[s], j * kXBK, rt0 * 128);
        bulk_load(sf + 512, w2_sf + sf_tile_offset(rt0, j, NS), 512, &full[s]);
        bulk_load(sf + 1024, w2_sf + sf_tile_offset(rt0 + 1, j, NS), 512, &full[s]);
        advance();
      }
    }
    if (!ok) {
      for (int i = 0; i < kXStages; ++i)
        if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kXDrainNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_mxf8(kBM, 256);
    int s = 0;
    uint32_t ph = 0;
    uint32_t q = 0;  // jobs issued (each job owns the accumulator until drained)
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 94);
    const uint32_t act_addr = smem_addr(act), act_sf_addr = smem_addr(act_sf);
    auto stage_mmas = [&](uint64_t ad, bool a_from_act, int kb_first) {
      const uint32_t sfa_col = tmem_base + 256 + 16 * s, sfb_col = sfa_col + 4;
      const uint32_t sf_smem = smem_addr(sSF + s * kXSF);
      utccp_sf(sfa_col, sdesc_sf_tile(a_from_act ? act_sf_addr : sf_smem));
      utccp_sf(sfb_col, sdesc_sf_tile(sf_smem + 512));
      utccp_sf(sfb_col + 4, sdesc_sf_tile(sf_smem + 1024));
      const uint64_t bd = sdesc_sw128(smem_addr(sB + s * kXB));
#pragma unroll
      for (int kk = 0; kk < kXBK / 32; ++kk)
        umma_mxf8(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc_with_sf_id(idesc, kk), sfa_col, sfb_col,
                  (kb_first | kk) != 0);
      umma_commit(&empty[s]);
      if (++s == kXStages) {
        s = 0;
        ph ^= 1u;
      }
    };
    int it = 0;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++it) {
      if (!(ok = mbar_wait(tempty, (q & 1u) ^ 1u, wc, 42))) break;
      tc_fence_after();
      for (int kb = 0; kb < K1; ++kb) {
        if (!(ok = mbar_wait(&full[s], ph, wc, 43))) break;
        tc_fence_after();
        stage_mmas(sdesc_sw128(smem_addr(sA + s * kXA)), false, kb);
      }
      if (!ok) break;
      umma_commit(tfull);
      ++q;
      if (!(ok = mbar_wait(act_full, (uint32_t)it & 1u, wc, 44))) break;
      tc_fence_after();
      for (int n = 0; ok && n < NO; ++n) {
        if (!(ok = mbar_wait(tempty, (q & 1u) ^ 1u, wc, 45))) break;
        tc_fence_after();
        if (!(ok = mbar_wait(&full[s], ph, wc, 46))) break;
        tc_fence_after();
        stage_mmas(sdesc_sw128(act_addr), true, 0);
        umma_commit(tfull);
        ++q;
      }
    }
    if (!ok) {
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kXDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_red = red + row * kXRedRow;
    float* out_f32 = static_cast<float*>(args.out_f32);
    uint32_t q = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
      const int rb = tile / NS;
      const int64_t slot = (int64_t)rb * kBM + row;
      const int tok = args.row_tok[slot];
      const float w = args.slot_w[slot];
      // GEMM1 -> SwiGLU -> MXFP8 act tile in shared memory
      if (!(ok = mbar_wait(tfull, q & 1u, wc, 47))) break;
      tc_fence_after();
      // one 32-column block at a time: SwiGLU, requantize, swizzled store
      uint8_t* arow = act + row * 128;
      uint32_t sfw = 0;
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        uint32_t g[32], u[32];
        tmem_ld_x32_pair(lane_base + blk * 32, lane_base + 128 + blk * 32, g, u);
        float a[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = x_swiglu(x_u2f(g[i]), x_u2f(u[i]), swiglu_lim);
        uint32_t qv[8];
        sfw |= mx_quantize32(a, qv) << (8 * blk);
        // 32 codes = 16-byte chunks 2*blk and 2*blk+1 of the 128-byte row, swizzled
        st_shared_v4(arow + (((2 * blk) ^ (row & 7)) << 4), qv[0], qv[1], qv[2], qv[3]);
        st_shared_v4(arow + (((2 * blk + 1) ^ (row & 7)) << 4), qv[4], qv[5], qv[6], qv[7]);
      }
      tc_fence_before();
      mbar_arrive(tempty);
      ++q;
      *reinterpret_cast<uint32_t*>(act_sf + sf_in_tile(row)) = sfw;
      fence_proxy_async_smem();
      mbar_arrive(act_full);
      // GEMM2 chunks -> fp32 reductions
      for (int n = 0; n < (args.D / 256); ++n) {
        if (!(ok = mbar_wait(tfull, q & 1u, wc, 48))) break;
        tc_fence_after();
#pragma unroll 1
        for (int h = 0; h < 256 / kXRedCols; ++h) {
          uint32_t v0[32], v1[32];
          tmem_ld_x32_pair(lane_base + h * kXRedCols, lane_base + h * kXRedCols + 32, v0, v1);
          if (tok >= 0) {
            bulk_wait_read_all();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_shared_v4(my_red + i * 16, __float_as_uint(w * x_u2f(v0[4 * i])), __float_as_uint(w * x_u2f(v0[4 * i + 1])),
                           __float_as_uint(w * x_u2f(v0[4 * i + 2])), __float_as_uint(w * x_u2f(v0[4 * i + 3])));
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_shared_v4(my_red + 128 + i * 16, __float_as_uint(w * x_u2f(v1[4 * i])),
                           __float_as_uint(w * x_u2f(v1[4 * i + 1])), __float_as_uint(w * x_u2f(v1[4 * i + 2])),
                           __float_as_uint(w * x_u2f(v1[4 * i + 3])));
            fence_proxy_async_smem();
            bulk_reduce_add_f32(out_f32 + (int64_t)tok * args.D + n * 256 + h * kXRedCols, my_red, kXRedCols * 4);
            bulk_commit();
          }
        }
        tc_fence_before();
        mbar_arrive(tempty);
        ++q;
      }
    }
    bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace

cudaError_t launch_fused_mxfp8(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w2,
                               const FusedMxArgs& args, int grid, cudaStream_t stream) {
  // once per device: not a stream operation, so it stays out of graph capture
  static bool smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    cudaError_t err = cudaFuncSetAttribute(fused_moe_mxfp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmem);
    if (err != cudaSuccess) return err;
    smem_set[dev] = true;
  }
  fused_moe_mxfp8_kernel<<<grid, kXThreads, kXSmem, stream>>>(map_xg, map_w1, map_w2, args);
  return cudaGetLastError();
}

}  // namespace moe
