// gemm_pair2_wide.cu -- the split pipeline's up-projection (GEMM1 + SwiGLU) on
// CTA pairs with 512-column tiles: each tile is one block pair (M = 256 rows,
// 128 per CTA) by two 256-column halves, [gate j0 | up j0] and
// [gate j0+1 | up j0+1], accumulated side by side in the pair's 512 TMEM
// columns.  Per K step of 64 a CTA brings in its 128 A rows (16 KB) and its
// 128 rows of each half's B tile (2 x 16 KB): 48 KB for 128 x 512 outputs
// instead of the 256-column tiles' 32 KB for 128 x 256, a quarter fewer
// operand bytes per FLOP (Pearl "Optimizing Grouped GEMM for MoE on
// Blackwell": 2-CTA tiles 256 rows by 512 columns at large batch).
//
// The two halves of the accumulator are released separately (Pearl, the
// split tensor-memory slots of its 512-wide tiles): the epilogue reads half 0,
// frees it, then reads half 1.  The MMA issuer of the next tile starts on
// half 0 as soon as it is free and runs up to kWLag K steps ahead on it,
// holding those stages, before it needs half 1; the epilogue's read of half 1
// overlaps those MMAs.
//
// Roles (192 threads): warp 0 lane 0 loads (both CTAs); warp 1 allocates
// tensor memory and its lane 0 issues the pair MMAs (even CTA); warps 2..5
// read the accumulator, apply SwiGLU, round to bf16 and store act rows with
// bulk copies (both CTAs).  Both CTAs' loads complete on the even CTA's full[]
// barriers; MMA commits are multicast to both CTAs; each CTA's epilogue warps
// arrive on the even CTA's tempty[half] barriers.  Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kWStages = 4;
constexpr int kWLag = kWStages - 1;          // K steps the issuer may run ahead on half 0
constexpr int kWThreads = 192;
constexpr int kWA = kBM * kBK * 2;           // 16 KB: this CTA's 128 rows of A
constexpr int kWB = 128 * kBK * 2;           // 16 KB: this CTA's 128 rows of one half's B tile
constexpr int kWStage = kWA + 2 * kWB;       // 48 KB
constexpr int kWStageRow = 256 + 16;         // staging row: 128 act values (+16 B: distinct banks)
constexpr int kWStaging = kBM * kWStageRow;
constexpr int kWBarrierBytes = 256;
constexpr int kWSmem = kWStages * kWStage + kWStaging + kWBarrierBytes;
static_assert(kWSmem <= 232448, "shared memory");
static_assert((2 * kWStages + 6) * 8 + 8 <= kWBarrierBytes, "barrier area");
constexpr uint64_t kWDrainNs = 200ull * 1000 * 1000;
constexpr uint64_t kWSettleNs = 2ull * 1000 * 1000;

__device__ __forceinline__ float w_u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ float w_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__global__ void __launch_bounds__(kWThreads, 1)
    gemm_up_wide_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_addr(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(args.err, kErrLaunch);
    return;
  }
  uint8_t* sStage = smem_raw + kWStages * kWStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + kWStaging);
  uint64_t* empty = full + kWStages;
  uint64_t* tfull = empty + kWStages;
  uint64_t* tempty = tfull + 1;  // [2]: half 0, half 1
  uint64_t* drain = tempty + 2;
  uint64_t* never = drain + 1;   // no thread ever arrives here (failure-path test hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto sA = [&](int s) { return smem_raw + s * kWStage; };
  auto sB = [&](int s, int h) { return smem_raw + s * kWStage + kWA + h * kWB; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_slot = (int)blockIdx.x >> 1, n_pair_slots = (int)gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(&tempty[0], 8);  // even CTA: four epilogue warps of each CTA
    mbar_init(&tempty[1], 8);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();

  const int NJ = args.n_col_tiles;   // 128-column act tiles
  const int NG = (NJ + 1) >> 1;      // column groups of two tiles
  const int n_tiles = args.meta[1] * NG;
  const int KB = args.k_blocks;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[kWStages];
#pragma unroll
    for (int i = 0; i < kWStages; ++i) issued_phase[i] = -1;
    bool ok = true;
    for (int tile = pair_slot; ok && tile < n_tiles; tile += n_pair_slots) {
      const int info = args.pair_info[tile / NG], g = tile % NG;
      const int rb0 = info >> 1, two = info & 1;
      const int my_rb = rb0 + (int)(rank & (uint32_t)two);  // the odd CTA of a half pair reloads rb0
      const int e = args.expert_of_rb[rb0];
      const bool has1 = 2 * g + 1 < NJ;
      // even CTA: gate rows of both halves; odd CTA: up rows
      const int brow = e * 2 * args.H + (int)rank * args.H + 2 * g * 128;
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&empty[s], ph ^ 1u, wc, 71))) break;
        if (leader) mbar_arrive_expect_tx(&full[s], 2 * (kWA + (has1 ? 2 : 1) * kWB));
        const uint32_t fb = mapa_shared(smem_addr(&full[s]), 0);
        tma_load_2d_pair(sA(s), &map_a, fb, kb * kBK, my_rb * kBM);
        tma_load_2d_pair(sB(s, 0), &map_b, fb, kb * kBK, brow);
        if (has1) tma_load_2d_pair(sB(s, 1), &map_b, fb, kb * kBK, brow + 128);
        issued_phase[s] = (int)ph;
        if (++s == kWStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      if (leader) {
        for (int i = 0; i < kWStages; ++i)
          if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kWDrainNs);
      } else {
        spin_ns(kWSettleNs);
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, 256);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 98);
    int it = 0;
    for (int tile = pair_slot; ok && tile < n_tiles; tile += n_pair_slots, ++it) {
      const bool has1 = 2 * (tile % NG) + 1 < NJ;
      const uint32_t tph = ((uint32_t)it & 1u) ^ 1u;  // phase of tempty[] that frees this tile's halves
      if (!(ok = mbar_wait_cluster(&tempty[0], tph, wc, 72))) break;
      tc_fence_after();
      bool half1_free = !has1;
      int pend_s[kWLag];
      int n_pend = 0;
      // MMAs of half 1 for the stages held so far; then release those stages
      auto flush_half1 = [&]() {
        for (int i = 0; i < n_pend; ++i) {
          const uint64_t adesc = sdesc_sw128(smem_addr(sA(pend_s[i])));
          const uint64_t bdesc = sdesc_sw128(smem_addr(sB(pend_s[i], 1)));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_pair(tmem_base + 256, adesc + 2 * kk, bdesc + 2 * kk, idesc, (i | kk) != 0);
          umma_commit_pair(&empty[pend_s[i]], 0x3);
        }
        n_pend = 0;
      };
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&full[s], ph, wc, 73))) break;
        tc_fence_after();
        const uint64_t adesc = sdesc_sw128(smem_addr(sA(s)));
        const uint64_t bdesc0 = sdesc_sw128(smem_addr(sB(s, 0)));
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_bf16_pair(tmem_base, adesc + 2 * kk, bdesc0 + 2 * kk, idesc, (kb | kk) != 0);
        if (!half1_free && mbar_try_wait_acq_cluster(&tempty[1], tph)) {
          half1_free = true;
          tc_fence_after();
          flush_half1();
        }
        if (half1_free) {
          if (has1) {
            const uint64_t bdesc1 = sdesc_sw128(smem_addr(sB(s, 1)));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_bf16_pair(tmem_base + 256, adesc + 2 * kk, bdesc1 + 2 * kk, idesc, (kb | kk) != 0);
          }
          umma_commit_pair(&empty[s], 0x3);
        } else {
          pend_s[n_pend++] = s;  // kb == n_pend - 1: half 1 has not started yet
          if (n_pend == kWLag || kb + 1 == KB) {
            if (!(ok = mbar_wait_cluster(&tempty[1], tph, wc, 74))) break;
            tc_fence_after();
            half1_free = true;
            flush_half1();
          }
        }
        if (++s == kWStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit_pair(tfull, 0x3);
    }
    if (!ok) {
      umma_commit_pair(drain, 0x1);
      mbar_wait_drain(drain, 0, kWDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_stage = sStage + row * kWStageRow;
    const uint32_t tempty_leader = mapa_shared(smem_addr(&tempty[0]), 0);
    int it = 0;
    for (int tile = pair_slot; tile < n_tiles; tile += n_pair_slots, ++it) {
      if (!mbar_wait(tfull, (uint32_t)it & 1u, wc, 75)) break;
      tc_fence_after();
      const int info = args.pair_info[tile / NG], g = tile % NG;
      const bool has1 = 2 * g + 1 < NJ;
      const bool valid = rank == 0 || (info & 1);
      const int64_t slot = (int64_t)((info >> 1) + (int)rank) * kBM + row;
      const int tok = valid ? args.row_tok[slot] : -1;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[64];
        if (h == 0 || has1) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t gv[32], uv[32];
            tmem_ld_x32_pair(lane_base + h * 256 + c * 32, lane_base + h * 256 + 128 + c * 32, gv, uv);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[c * 16 + i] = pack_bf16x2(w_swiglu(w_u2f(gv[2 * i]), w_u2f(uv[2 * i]), swiglu_lim),
                                           w_swiglu(w_u2f(gv[2 * i + 1]), w_u2f(uv[2 * i + 1]), swiglu_lim));
          }
        }
        // this warp has read half h: the next tile's MMAs may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader + h * 8);
        if ((h == 0 || has1) && tok >= 0) {
          bulk_wait_read_all();  // the previous store has left the staging row
#pragma unroll
          for (int q = 0; q < 16; ++q)
            st_shared_v4(my_stage + q * 16, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          fence_proxy_async_smem();
          bulk_store(static_cast<__nv_bfloat16*>(args.act) + slot * args.H + (2 * g + h) * 128, my_stage, 256);
          bulk_commit();
        }
      }
    }
    bulk_wait_all();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

}  // namespace

int pair_wide_cluster_slots() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev]) return cache[dev];
  if (cudaFuncSetAttribute(gemm_up_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kWThreads);
  cfg.dynamicSmemBytes = kWSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_up_wide_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cache[dev] = n;
  return n;
}

cudaError_t launch_up_pair2_wide_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const GemmArgs& args,
                                      int n_pairs, cudaStream_t stream, bool pdl) {
  if (pair_wide_cluster_slots() <= 0) return cudaErrorInvalidConfiguration;  // also sets the smem attribute
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n_pairs);
  cfg.blockDim = dim3(kWThreads);
  cfg.dynamicSmemBytes = kWSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_up_wide_kernel, map_xg, map_w1, args);
}

}  // namespace moe
