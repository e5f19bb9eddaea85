// gemm_pair.cu -- up-projection + SwiGLU with two row blocks per tile.
//
// Same computation as the UP mode of gemm_bf16.cu, but each tile covers a pair
// of consecutive 128-row blocks of one expert (the routing emits the pairs)
// against one [gate j | up j] W1 tile: every weight byte brought into shared
// memory feeds two MMAs ("Prime Flash MoE" sec. 5 "BPC and CPC": BPC lets one
// CTA process two row tiles against the same weight tiles; sec. 6 uses the
// idea in the split pipeline's down kernel).  Per 64-wide K step a stage holds
// A0 (16 KB), A1 (16 KB) and the 256-row W1 tile (32 KB), so a CTA needs a
// third fewer bytes per FLOP than with one row block -- the up kernel is bound
// by how many bytes it can keep in flight, not by the tensor core.
// The two 256-column accumulators fill tensor memory, so they are not double
// buffered; eight epilogue warps (two per TMEM lane quadrant, one per
// accumulator) drain them in parallel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPStages = 3;
constexpr int kPThreads = 64 + 256;
constexpr int kPEpi = 256;
constexpr int kPA = kBM * kBK * 2;               // 16 KB per row block
constexpr int kPB = 256 * kBK * 2;               // 32 KB: gate j (128 rows) | up j (128 rows)
constexpr int kPStage = 2 * kPA + kPB;           // 64 KB
constexpr int kPSmem = 1024 + kPStages * kPStage + 256;
static_assert(kPSmem <= 232448, "shared memory");
constexpr uint64_t kPDrainNs = 200ull * 1000 * 1000;

__device__ __forceinline__ float p_u2f(uint32_t u) { return __uint_as_float(u); }
// silu(g) * u with the optional clamp (lim = +inf when off): g <= lim,
// -lim <= u <= lim.
__device__ __forceinline__ float p_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__global__ void __launch_bounds__(kPThreads, 1)
    up_pair_bf16_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPStages * kPStage);
  uint64_t* empty = full + kPStages;
  uint64_t* tfull = empty + kPStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* never = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kPEpi);
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
  if (threadIdx.x == 0) griddep_launch_dependents();

  const int NJ = args.n_col_tiles;
  const int n_tiles = args.meta[1] * NJ;
  const int KB = args.k_blocks;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[kPStages] = {-1, -1, -1};
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
      const int info = args.pair_info[tile / NJ], j = tile % NJ;
      const int rb0 = info >> 1, two = info & 1;
      const int e = args.expert_of_rb[rb0];
      const int row0 = e * 2 * args.H + j * kUpFold;
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&empty[s], ph ^ 1u, wc, 31))) break;
        mbar_arrive_expect_tx(&full[s], (two ? 2 : 1) * kPA + kPB);
        issued_phase[s] = (int)ph;
        uint8_t* st = smem + s * kPStage;
        tma_load_2d(st, &map_a, &full[s], kb * kBK, rb0 * kBM);
        if (two) tma_load_2d(st + kPA, &map_a, &full[s], kb * kBK, (rb0 + 1) * kBM);
        tma_load_2d(st + 2 * kPA, &map_b, &full[s], kb * kBK, row0);
        tma_load_2d(st + 2 * kPA + kUpFold * kBK * 2, &map_b, &full[s], kb * kBK, row0 + args.H);
        if (++s == kPStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      for (int i = 0; i < kPStages; ++i)
        if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kPDrainNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, 2 * kUpFold);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 93);
    int it = 0;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++it) {
      const int two = args.pair_info[tile / NJ] & 1;
      if (!(ok = mbar_wait(tempty, ((uint32_t)it & 1u) ^ 1u, wc, 32))) break;
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&full[s], ph, wc, 33))) break;
        tc_fence_after();
        const uint32_t st = smem_addr(smem + s * kPStage);
        const uint64_t a0 = sdesc_sw128(st), a1 = sdesc_sw128(st + kPA), bd = sdesc_sw128(st + 2 * kPA);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          umma_bf16(tmem_base, a0 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          if (two) umma_bf16(tmem_base + 256, a1 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
        }
        umma_commit(&empty[s]);
        if (++s == kPStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit(tfull);
    }
    if (!ok) {
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kPDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int sel = (warp - 2) >> 2;  // accumulator (row block of the pair) this warp drains
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t tacc = tmem_base + ((uint32_t)(quad * 32) << 16) + sel * 256;
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      if (!mbar_wait(tfull, (uint32_t)it & 1u, wc, 34)) break;
      tc_fence_after();
      const int info = args.pair_info[tile / NJ], j = tile % NJ;
      const int two = info & 1;
      if (sel == 0 || two) {
        const int64_t slot = (int64_t)((info >> 1) + sel) * kBM + row;
        const int tok = args.row_tok[slot];
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(args.act) + slot * args.H + j * kUpFold;
#pragma unroll 1
        for (int c = 0; c < kUpFold / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_x32_pair(tacc + c * 32, tacc + kUpFold + c * 32, g, u);
          if (tok >= 0) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(p_swiglu(p_u2f(g[2 * i]), p_u2f(u[2 * i]), swiglu_lim),
                                  p_swiglu(p_u2f(g[2 * i + 1]), p_u2f(u[2 * i + 1]), swiglu_lim));
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_global_v4(dst + c * 32 + q * 8, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty);
    }
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

cudaError_t launch_up_pair_bf16(const CUtensorMap& map_a, const CUtensorMap& map_w1, const GemmArgs& args, int grid,
                                cudaStream_t stream) {
  // once per device: not a stream operation, so it stays out of graph capture
  static bool smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    cudaError_t err = cudaFuncSetAttribute(up_pair_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
    if (err != cudaSuccess) return err;
    smem_set[dev] = true;
  }
  up_pair_bf16_kernel<<<grid, kPThreads, kPSmem, stream>>>(map_a, map_w1, args);
  return cudaGetLastError();
}

}  // namespace moe
