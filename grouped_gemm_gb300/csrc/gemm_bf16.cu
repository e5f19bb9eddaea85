// gemm_bf16.cu -- persistent grouped GEMMs of the split pipeline on tcgen05.
//
// UP  (GEMM1 + SwiGLU): for each 128-row block rb of the sorted, padded token
//     order (expert e = expert_of_rb[rb]) and each column tile j, the
//     accumulator holds [gate rows j*G .. +G | up rows H + j*G .. +G] of
//     W1[e] times the 128 routed rows, so both halves of every SwiGLU pair sit
//     in the same TMEM accumulator ("Prime Flash MoE", sec. 2 "Trick 1": gate
//     and up interleaved per 128-row block; here the interleave is two TMA
//     boxes into adjacent shared-memory rows).  The 128 token rows arrive
//     either with tile::gather4 straight from x (four rows per instruction,
//     sec. 3 "For the tokens: TMA gathers them too") or as a plain tile of the
//     pre-gathered xg (sec. 6).  The epilogue computes act = silu(gate) * up
//     in fp32, rounds to bf16 and stores act[slot, j*G..] (sec. 5 "SwiGLU",
//     sec. 6: the split pipeline writes act once).
// DOWN (GEMM2 + weighted reduce): for each row block and 256-column tile of
//     D, acc = act[rb rows, :] * W2[e][cols, :]^T over all of H (sec. 6 "The
//     down-projection kernel": C = 1, no split-K).  The epilogue scales row r
//     by its routing weight in fp32, rounds to bf16 into a padded shared
//     staging row and reduces the whole 512-byte row into out[row_tok[r]] with
//     one cp.reduce.async.bulk .add.bf16 (sec. 5 "Three jobs - one
//     instruction": the top-k sum and the scatter back to token order).
//
// Warp roles (192 threads, one CTA per SM, persistent over a static tile list):
//   warp 0      TMA producer: A and B tiles into a STAGES-deep ring
//   warp 1      TMEM allocator; one lane issues tcgen05.mma (M=128, K=16)
//   warps 2..5  epilogue: tcgen05.ld of the warp's 32 TMEM lanes (= rows)
// The accumulator is double-buffered in TMEM (2 x N columns) so the epilogue
// of tile i overlaps the main loop of tile i+1.  Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

enum { kModeUp = 0, kModeDown = 1 };

template <int MODE, int N, int STAGES>
struct GemmCfg {
  static constexpr int kABytes = kBM * kBK * 2;             // 16 KB
  static constexpr int kBBytes = N * kBK * 2;               // N rows of 128 B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * N;                   // double-buffered accumulator
  // DOWN stages each output row (N bf16) in shared memory for the bulk
  // reduction; +16 B per row keeps the 32 rows of a warp on distinct banks.
  static constexpr int kStageRowBytes = N * 2 + 16;
  static constexpr int kStagingBytes = MODE == kModeDown ? kBM * kStageRowBytes : 0;
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmemBytes = 1024 /*align slack*/ + STAGES * kStageBytes + kStagingBytes + kBarrierBytes;
  static_assert(N % 32 == 0 && N >= 32 && N <= 256, "MMA N");
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns: power of two <= 512");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert((2 * STAGES + 6) * 8 + 8 <= kBarrierBytes, "barrier area");
};

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;  // 200 ms

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

template <int MODE, int N, int STAGES, bool GATHER>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_bf16_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                             const GemmArgs args) {
  using Cfg = GemmCfg<MODE, N, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::kABytes;
  uint8_t* sStage = smem + STAGES * Cfg::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + Cfg::kStagingBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* never = drain + 1;  // no thread ever arrives here (failure-path test hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiThreads);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (MODE == kModeUp && threadIdx.x == 0) griddep_launch_dependents();

  const int num_rb = args.meta[0];
  const int n_tiles = num_rb * args.n_col_tiles;
  const int KB = args.k_blocks;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (MODE == kModeDown && lane == 0) griddep_wait();  // act is written by the previous grid
    __syncwarp();
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[STAGES];
#pragma unroll
    for (int i = 0; i < STAGES; ++i) issued_phase[i] = -1;
    bool ok = true;
    // L2 prefetch cursor: runs args.prefetch k-blocks ahead of the loads
    // (across tile boundaries) so that tiles land in L2 before the ring needs
    // them -- more bytes in flight than the shared-memory ring can hold.
    int pf_tile = blockIdx.x, pf_kb = 0, pf_e = pf_tile < n_tiles ? args.expert_of_rb[pf_tile / args.n_col_tiles] : 0;
    auto prefetch_one = [&]() {
      if (pf_tile >= n_tiles) return;
      const int prb = pf_tile / args.n_col_tiles, pj = pf_tile % args.n_col_tiles;
      if (!GATHER) tma_prefetch_2d(&map_a, pf_kb * kBK, prb * kBM);
      if (MODE == kModeUp) {
        constexpr int G = N / 2;
        const int row0 = pf_e * 2 * args.H + pj * G;
        tma_prefetch_2d(&map_b, pf_kb * kBK, row0);
        tma_prefetch_2d(&map_b, pf_kb * kBK, row0 + args.H);
      } else {
        tma_prefetch_2d(&map_b, pf_kb * kBK, pf_e * args.D + pj * N);
      }
      if (++pf_kb == KB) {
        pf_kb = 0;
        pf_tile += gridDim.x;
        if (pf_tile < n_tiles) pf_e = args.expert_of_rb[pf_tile / args.n_col_tiles];
      }
    };
    if (lane == 0)
      for (int i = 0; i < args.prefetch; ++i) prefetch_one();
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
      const int rb = tile / args.n_col_tiles, j = tile % args.n_col_tiles;
      const int e = args.expert_of_rb[rb];
      int g0 = 0, g1 = 0, g2 = 0, g3 = 0;
      if (GATHER) {  // lane l fetches tile rows 4l..4l+3; padding rows read row 0
        const int* rt = args.row_tok + (int64_t)rb * kBM + lane * 4;
        g0 = max(rt[0], 0);
        g1 = max(rt[1], 0);
        g2 = max(rt[2], 0);
        g3 = max(rt[3], 0);
      }
      for (int kb = 0; kb < KB; ++kb) {
        int got = 1;
        if (lane == 0) {
          got = mbar_wait(&empty[s], ph ^ 1u, wc, 1) ? 1 : 0;
          if (got) mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        if (GATHER) {
          tma_gather4(sA + s * Cfg::kABytes + lane * 4 * kBK * 2, &map_a, &full[s], kb * kBK, g0, g1, g2, g3);
        } else if (lane == 0) {
          tma_load_2d(sA + s * Cfg::kABytes, &map_a, &full[s], kb * kBK, rb * kBM);
        }
        if (lane == 0) {
          if (args.prefetch > 0) prefetch_one();
          if (MODE == kModeUp) {
            constexpr int G = N / 2;
            const int row0 = e * 2 * args.H + j * G;
            tma_load_2d(sB + s * Cfg::kBBytes, &map_b, &full[s], kb * kBK, row0);
            tma_load_2d(sB + s * Cfg::kBBytes + G * kBK * 2, &map_b, &full[s], kb * kBK, row0 + args.H);
          } else {
            tma_load_2d(sB + s * Cfg::kBBytes, &map_b, &full[s], kb * kBK, e * args.D + j * N);
          }
          issued_phase[s] = (int)ph;
        }
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {  // let every copy already in flight land before the CTA exits
      for (int i = 0; i < STAGES; ++i)
        if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kDrainNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, N);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 90);  // runs out after the wait limit
    int it = 0;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(&tempty[acc], aph ^ 1u, wc, 2)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * N;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&full[s], ph, wc, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = sdesc_sw128(smem_addr(sA + s * Cfg::kABytes));
        const uint64_t bdesc = sdesc_sw128(smem_addr(sB + s * Cfg::kBBytes));
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // +32 bytes per K step of 16 bf16 = +2 in the descriptor's address field
          umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
        }
        umma_commit(&empty[s]);  // frees the smem stage once these MMAs are done
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit(&tfull[acc]);  // accumulator ready for the epilogue
    }
    if (!ok) {  // wait for every MMA already issued before TMEM is released
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_stage = sStage + row * Cfg::kStageRowBytes;
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(&tfull[acc], aph, wc, 4)) break;
      tc_fence_after();
      const int rb = tile / args.n_col_tiles, j = tile % args.n_col_tiles;
      const int64_t slot = (int64_t)rb * kBM + row;
      const int tok = args.row_tok[slot];
      const uint32_t tacc = lane_base + acc * N;
      if (MODE == kModeUp) {
        constexpr int G = N / 2;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(args.act) + slot * args.H + j * G;
#pragma unroll 1
        for (int c = 0; c < G / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_x32_pair(tacc + c * 32, tacc + G + c * 32, g, u);
          if (tok >= 0) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(swiglu(u2f(g[2 * i]), u2f(u[2 * i])), swiglu(u2f(g[2 * i + 1]), u2f(u[2 * i + 1])));
#pragma unroll
            for (int q = 0; q < 4; ++q) st_global_v4(dst + c * 32 + q * 8, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      } else {
        const float w = args.slot_w[slot];
        bulk_wait_read_all();  // the previous tile's reduction has left the staging row
#pragma unroll 1
        for (int c = 0; c < N / 32; c += 2) {
          uint32_t v0[32], v1[32];
          tmem_ld_x32_pair(tacc + c * 32, tacc + (c + 1) * 32, v0, v1);
          if (tok >= 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(my_stage + c * 64 + q * 16, pack_bf16x2(w * u2f(v0[8 * q + 0]), w * u2f(v0[8 * q + 1])),
                           pack_bf16x2(w * u2f(v0[8 * q + 2]), w * u2f(v0[8 * q + 3])),
                           pack_bf16x2(w * u2f(v0[8 * q + 4]), w * u2f(v0[8 * q + 5])),
                           pack_bf16x2(w * u2f(v0[8 * q + 6]), w * u2f(v0[8 * q + 7])));
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(my_stage + (c + 1) * 64 + q * 16,
                           pack_bf16x2(w * u2f(v1[8 * q + 0]), w * u2f(v1[8 * q + 1])),
                           pack_bf16x2(w * u2f(v1[8 * q + 2]), w * u2f(v1[8 * q + 3])),
                           pack_bf16x2(w * u2f(v1[8 * q + 4]), w * u2f(v1[8 * q + 5])),
                           pack_bf16x2(w * u2f(v1[8 * q + 6]), w * u2f(v1[8 * q + 7])));
          }
        }
        if (tok >= 0) {
          fence_proxy_async_smem();
          bulk_reduce_add_bf16(static_cast<__nv_bfloat16*>(args.out) + (int64_t)tok * args.D + j * N, my_stage,
                               N * 2);
          bulk_commit();
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
    if (MODE == kModeDown) bulk_wait_all();  // reductions complete before the CTA exits
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

template <int MODE, int N, int STAGES, bool GATHER>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& args, int grid,
                        cudaStream_t stream, bool pdl) {
  using Cfg = GemmCfg<MODE, N, STAGES>;
  auto kern = grouped_gemm_bf16_kernel<MODE, N, STAGES, GATHER>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, b, args);
}

}  // namespace

cudaError_t launch_up_bf16(const CUtensorMap& map_a, const CUtensorMap& map_w1, const GemmArgs& args, int grid,
                           cudaStream_t stream, bool gather4) {
  if (gather4) return launch_gemm<kModeUp, 2 * kUpFold, kUpStages, true>(map_a, map_w1, args, grid, stream, false);
  return launch_gemm<kModeUp, 2 * kUpFold, kUpStages, false>(map_a, map_w1, args, grid, stream, false);
}

cudaError_t launch_down_bf16(const CUtensorMap& map_act, const CUtensorMap& map_w2, const GemmArgs& args, int grid,
                             cudaStream_t stream, bool pdl) {
  return launch_gemm<kModeDown, kDownN, kDownStages, false>(map_act, map_w2, args, grid, stream, pdl);
}

}  // namespace moe
