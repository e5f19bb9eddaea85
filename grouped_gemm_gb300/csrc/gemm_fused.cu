// gemm_fused.cu -- the fused pipeline's GEMM kernel: for one (128-row block,
// 128-wide slice j of the intermediate dimension) per tile it runs GEMM1 with
// the SwiGLU epilogue, keeps the activation tile in shared memory, and runs
// GEMM2 on it as a split-K partial of the down projection ("Prime Flash MoE"
// sec. 2 "Trick 2: Cut the intermediate": CTA j owns intermediate columns
// [128j, 128j+128) and adds its partial output rows into out).
//
//   GEMM1: acc1[128 x 256] = xg[rb rows] . [W1 gate rows j*128.. | up rows H+j*128..]^T
//   SwiGLU epilogue: act = silu(gate) * up (fp32) -> bf16 written into shared
//          memory in the 128-byte-swizzled K-major layout GEMM2's A operand
//          expects (sec. 5 "SwiGLU - which never leaves the SM": fp32 in
//          tensor memory -> registers -> bf16 in smem -> tensor core).
//   GEMM2: for every 256-column chunk n of D, acc2[128 x 256] = act . W2[e][n
//          cols, j slice]^T (K = 128), the routing weight applied in fp32.
//   Reduction: each row is staged in shared memory and added into an fp32
//          accumulator out_f32[row_tok, n cols] with cp.reduce.async.bulk
//          .add.f32 (sec. 5 "Three jobs - one instruction": the top-k sum, the
//          split-K sum over slices and the scatter back to token order).  fp32,
//          not bf16: with C = H/128 slices and k experts, C*k bf16 roundings per
//          element exceed the accuracy the pipeline must keep.  A final pass
//          rounds out_f32 to bf16 out.
// One ring of TMA stages serves both GEMMs (sec. 4 "One ring, both GEMMs"):
// GEMM1 stages carry an xg tile and a W1 tile, GEMM2 stages a W2 tile.
// Accumulators use two 256-column TMEM slots in job order (GEMM1, then one job
// per output chunk), so the epilogue of one job overlaps the MMAs of the next.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kFThreads = 192;
constexpr int kFEpiThreads = 128;
constexpr int kFStages = 3;
constexpr int kSlice = 128;                        // intermediate columns per tile
constexpr int kN2 = 256;                           // GEMM2 output columns per job
constexpr int kFA = kBM * kBK * 2;                 // 16 KB
constexpr int kFB = 256 * kBK * 2;                 // 32 KB (W1 gate+up, or W2 256 rows)
constexpr int kFStage = kFA + kFB;
constexpr int kActBytes = 2 * kBM * kBK * 2;       // 128 x 128 bf16: two SW128 K-blocks
constexpr int kRedCols = 64;                       // fp32 columns per bulk reduction
constexpr int kRedRowBytes = kRedCols * 4 + 16;    // padded: rows of a warp on distinct banks
constexpr int kRedBytes = kBM * kRedRowBytes;
constexpr int kFBarrierBytes = 256;
constexpr int kFSmem = 1024 + kFStages * kFStage + kActBytes + kRedBytes + kFBarrierBytes;
static_assert(kFSmem <= 232448, "shared memory");
static_assert((2 * kFStages + 7) * 8 + 8 <= kFBarrierBytes, "barrier area");
constexpr uint64_t kFDrainNs = 200ull * 1000 * 1000;

__device__ __forceinline__ float f_u2f(uint32_t u) { return __uint_as_float(u); }
// silu(g) * u with the optional clamp (lim = +inf when off): g <= lim,
// -lim <= u <= lim.
__device__ __forceinline__ float f_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__global__ void __launch_bounds__(kFThreads, 1)
    fused_moe_bf16_kernel(const __grid_constant__ CUtensorMap map_xg, const __grid_constant__ CUtensorMap map_w1,
                          const __grid_constant__ CUtensorMap map_w2, const FusedArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* act = smem + kFStages * kFStage;
  uint8_t* red = act + kActBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kRedBytes);
  uint64_t* empty = full + kFStages;
  uint64_t* tfull = empty + kFStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* act_full = tempty + 2;
  uint64_t* drain = act_full + 1;
  uint64_t* never = drain + 1;  // no thread ever arrives here (failure-path test hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kFEpiThreads);
    }
    mbar_init(act_full, kFEpiThreads);
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

  const int NS = args.n_slices;            // H / 128
  const int n_tiles = args.meta[0] * NS;
  const int K1 = args.D / kBK;             // GEMM1 k-blocks
  const int NO = args.D / kN2;             // GEMM2 output chunks
  constexpr int K2 = kSlice / kBK;         // GEMM2 k-blocks per chunk (2)

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[kFStages] = {-1, -1, -1};
    bool ok = true;
    auto acquire = [&](uint32_t bytes) -> bool {
      if (!mbar_wait(&empty[s], ph ^ 1u, wc, 11)) return false;
      mbar_arrive_expect_tx(&full[s], bytes);
      issued_phase[s] = (int)ph;
      return true;
    };
    auto advance = [&]() {
      if (++s == kFStages) {
        s = 0;
        ph ^= 1u;
      }
    };
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
      const int rb = tile / NS, j = tile % NS;
      const int e = args.expert_of_rb[rb];
      const int w1_row = e * 2 * args.H + j * kSlice;
      for (int kb = 0; ok && kb < K1; ++kb) {
        if (!(ok = acquire(kFStage))) break;
        uint8_t* st = ring + s * kFStage;
        tma_load_2d(st, &map_xg, &full[s], kb * kBK, rb * kBM);
        tma_load_2d(st + kFA, &map_w1, &full[s], kb * kBK, w1_row);
        tma_load_2d(st + kFA + kSlice * kBK * 2, &map_w1, &full[s], kb * kBK, w1_row + args.H);
        advance();
      }
      for (int n = 0; ok && n < NO; ++n) {
        for (int kb = 0; kb < K2; ++kb) {
          if (!(ok = acquire(kFB))) break;
          tma_load_2d(ring + s * kFStage + kFA, &map_w2, &full[s], j * kSlice + kb * kBK, e * args.D + n * kN2);
          advance();
        }
      }
    }
    if (!ok) {
      for (int i = 0; i < kFStages; ++i)
        if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kFDrainNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, 256);
    int s = 0;
    uint32_t ph = 0;
    uint32_t q = 0;  // accumulator job counter
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 91);  // runs out after the wait limit
    int it = 0;
    const uint32_t act_addr = smem_addr(act);
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++it) {
      // GEMM1
      {
        const uint32_t slot = q & 1u;
        if (!(ok = mbar_wait(&tempty[slot], ((q >> 1) & 1u) ^ 1u, wc, 12))) break;
        tc_fence_after();
        const uint32_t d = tmem_base + slot * 256;
        for (int kb = 0; kb < K1; ++kb) {
          if (!(ok = mbar_wait(&full[s], ph, wc, 13))) break;
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_addr(ring + s * kFStage));
          const uint64_t bd = sdesc_sw128(smem_addr(ring + s * kFStage + kFA));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) umma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          umma_commit(&empty[s]);
          if (++s == kFStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[slot]);
        ++q;
      }
      // the SwiGLU epilogue has written act into shared memory
      if (!(ok = mbar_wait(act_full, (uint32_t)it & 1u, wc, 14))) break;
      tc_fence_after();
      // GEMM2, one job per 256-column output chunk
      for (int n = 0; ok && n < NO; ++n) {
        const uint32_t slot = q & 1u;
        if (!(ok = mbar_wait(&tempty[slot], ((q >> 1) & 1u) ^ 1u, wc, 15))) break;
        tc_fence_after();
        const uint32_t d = tmem_base + slot * 256;
        for (int kb = 0; kb < K2; ++kb) {
          if (!(ok = mbar_wait(&full[s], ph, wc, 16))) break;
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(act_addr + kb * (kBM * kBK * 2));
          const uint64_t bd = sdesc_sw128(smem_addr(ring + s * kFStage + kFA));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) umma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          umma_commit(&empty[s]);
          if (++s == kFStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[slot]);
        ++q;
      }
    }
    if (!ok) {
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kFDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_red = red + row * kRedRowBytes;
    float* out_f32 = static_cast<float*>(args.out_f32);
    uint32_t q = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
      const int rb = tile / NS;
      const int64_t slot_row = (int64_t)rb * kBM + row;
      const int tok = args.row_tok[slot_row];
      const float w = args.slot_w[slot_row];
      // SwiGLU: TMEM -> registers -> bf16 act tile in shared memory
      {
        const uint32_t slot = q & 1u;
        if (!(ok = mbar_wait(&tfull[slot], (q >> 1) & 1u, wc, 17))) break;
        tc_fence_after();
        const uint32_t t = lane_base + slot * 256;
#pragma unroll 1
        for (int c = 0; c < kSlice / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_x32_pair(t + c * 32, t + kSlice + c * 32, g, u);
          uint8_t* kblk = act + (c >> 1) * (kBM * kBK * 2) + row * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t p[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int v = i * 8 + m * 2;
              p[m] = pack_bf16x2(f_swiglu(f_u2f(g[v]), f_u2f(u[v]), swiglu_lim), f_swiglu(f_u2f(g[v + 1]), f_u2f(u[v + 1]), swiglu_lim));
            }
            const int chunk = (c & 1) * 4 + i;  // 16-byte chunk within the 128-byte row
            st_shared_v4(kblk + ((chunk ^ (row & 7)) << 4), p[0], p[1], p[2], p[3]);
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[slot]);
        ++q;
        fence_proxy_async_smem();  // act is read by the tensor core (async proxy)
        mbar_arrive(act_full);
      }
      // GEMM2 partial rows -> fp32 bulk reductions into out_f32
      for (int n = 0; n < NO; ++n) {
        const uint32_t slot = q & 1u;
        if (!(ok = mbar_wait(&tfull[slot], (q >> 1) & 1u, wc, 18))) break;
        tc_fence_after();
        const uint32_t t = lane_base + slot * 256;
#pragma unroll 1
        for (int h = 0; h < kN2 / kRedCols; ++h) {
          uint32_t v0[32], v1[32];
          tmem_ld_x32_pair(t + h * kRedCols, t + h * kRedCols + 32, v0, v1);
          if (tok >= 0) {
            bulk_wait_read_all();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_shared_v4(my_red + i * 16, __float_as_uint(w * f_u2f(v0[4 * i])), __float_as_uint(w * f_u2f(v0[4 * i + 1])),
                           __float_as_uint(w * f_u2f(v0[4 * i + 2])), __float_as_uint(w * f_u2f(v0[4 * i + 3])));
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_shared_v4(my_red + 128 + i * 16, __float_as_uint(w * f_u2f(v1[4 * i])),
                           __float_as_uint(w * f_u2f(v1[4 * i + 1])), __float_as_uint(w * f_u2f(v1[4 * i + 2])),
                           __float_as_uint(w * f_u2f(v1[4 * i + 3])));
            fence_proxy_async_smem();
            bulk_reduce_add_f32(out_f32 + (int64_t)tok * args.D + n * kN2 + h * kRedCols, my_red, kRedCols * 4);
            bulk_commit();
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[slot]);
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

// out[i] = bf16(acc[i]), 8 elements per thread-iteration.
__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float4* __restrict__ acc, uint4* __restrict__ out,
                                                          int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    out[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
}

}  // namespace

cudaError_t launch_fused_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w2,
                              const FusedArgs& args, int grid, cudaStream_t stream) {
  // once per device: not a stream operation, so it stays out of graph capture
  static bool smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    cudaError_t err = cudaFuncSetAttribute(fused_moe_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmem);
    if (err != cudaSuccess) return err;
    smem_set[dev] = true;
  }
  fused_moe_bf16_kernel<<<grid, kFThreads, kFSmem, stream>>>(map_xg, map_w1, map_w2, args);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const void* acc, void* out, int64_t n, int grid, cudaStream_t stream) {
  f32_to_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const float4*>(acc), static_cast<uint4*>(out), n / 8);
  return cudaGetLastError();
}

}  // namespace moe
