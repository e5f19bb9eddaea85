// gemm_pair2.cu -- the split pipeline's GEMMs on CTA pairs (tcgen05
// cta_group::2): one MMA of M = 256 rows (two row blocks of one expert) by
// N = 256 columns is issued by the even CTA of a two-CTA cluster; each CTA
// holds its own 128 rows of A and half (128 rows) of the B tile in shared
// memory and receives its 128 rows of the accumulator in its own tensor
// memory.  Per K step a CTA brings in 32 KB (16 KB of A, 16 KB of B) for the
// same 128 x 256 block of output as the single-CTA kernel's 48 KB: a third
// fewer bytes per FLOP, six stages in the same shared memory, one and a half
// times the work in flight per SM (Pearl "Optimizing Grouped GEMM for MoE on
// Blackwell": 2-CTA 256-row tiles at large batch; "Prime Flash MoE" sec. 5
// "BPC and CPC": two row tiles against the same weight tile).
//
// UP  (GEMM1 + SwiGLU): B = [W1 gate rows j*128 .. +128 (even CTA) | up rows
//     H + j*128 .. +128 (odd CTA)], so each CTA's accumulator holds gate in
//     columns [0, 128) and up in [128, 256) for its row block; the epilogue
//     is the single-CTA kernel's (act row staged, one bulk store).
// DOWN (GEMM2 + weighted reduce): B = W2[e] rows j*256 + 128 * rank .. +128;
//     the epilogue scales by the routing weight and reduces half rows into out
//     with bulk .add.bf16.
// Tiles are (block pair, column tile j).  A pair whose second block does not
// exist (an expert with an odd number of row blocks: a half pair) still runs
// both CTAs.  UP: the odd CTA loads the first block's rows again and stores
// nothing.  DOWN (args.half_m128): it runs as one M = 128 pair MMA, 64 rows of
// the block in each CTA, so no tensor-core work goes to a missing block.
// Measured layout of that shape: each CTA's 64 accumulator rows take all 128
// TMEM lanes, lanes 0..63 holding columns [0, N/2) of rows 0..63 and lanes
// 64..127 columns [N/2, N) of the same rows, so each lane reduces a half row.
// (The same for UP, with [gate 64 | up 64] B tiles per CTA, measured the up
// kernel 3-12% slower over all tiles and is not built.)
//
// Swap-AB pair tiles (DOWN, args.pair_swap_max > 0): a pair whose blocks hold
// at most pair_swap_max routed rows -- typically a half pair, an expert's odd
// last block -- runs with the operands swapped: the 256 W2 rows are the MMA's
// M side (each CTA its own 128, the rows it loads anyway) and the pair's
// routed rows its N = ns (rounded up to 16, half of them in each CTA), so the
// tensor cores do 256 x ns instead of 256 x 256 multiply-adds per K step and
// an idle half pair costs almost nothing ("Porting Block-Scaled GEMM Kernels"
// sec. 5.1 and Pearl: swap-AB for small per-expert M).  The epilogue reads the
// transposed accumulator (lane = output column, column = routed row) into the
// staging tile row by row and reduces each staged row into out as usual.
//
// Swap-AB half pairs (UP, args.up_swap): an expert's odd last row block holds
// at most 128 routed rows, yet a half pair pays for a full 256 x 256 MMA.  With
// the operands swapped the tensor cores do 256 x ns per K step (ns = the
// block's routed rows rounded up to 16): the M side is 256 W1 rows, each CTA
// loading [gate 64 | up 64] rows for its 64 act columns c (two 64-row boxes),
// and the N side the block's routed rows, ns / 2 in each CTA.  A CTA's
// accumulator then holds gate column c in lane c and up column c in lane
// 64 + c, routed row r in TMEM column r: the warps of lane quadrants 2 and 3
// pass their up values through shared memory (fp32) to the warps of quadrants
// 0 and 1, which form silu(gate) * up and store act.
//
// Synchronization: both CTAs' TMA loads complete on the even CTA's full[]
// barrier (which expects the pair's bytes); the MMA commits arrive on empty[]
// and tfull[] of both CTAs (multicast); each CTA's epilogue warps arrive on the
// even CTA's tempty[] (release, cluster scope).  Every wait is bounded; both
// CTAs meet at a cluster barrier before the pair releases tensor memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

enum { kPairUp = 0, kPairDown = 1 };
constexpr int kQA = kBM * kBK * 2;          // 16 KB: this CTA's 128 rows of A
constexpr int kQB = 128 * kBK * 2;          // 16 KB: this CTA's half of the 256-row B tile
constexpr int kQStage = kQA + kQB;
constexpr int kQBarrierBytes = 256;
// NEPI epilogue warps.  Four: one per TMEM lane quadrant, each thread one
// accumulator row, staged and reduced as two half rows in turn (staging row of
// 256 B + 16 B, so a warp's 32 rows fall on distinct banks), six stages.
// Eight (down projection): two warps per quadrant, one per half row; a warp
// reads its 128 columns into registers and releases the accumulator before it
// stages anything, so the MMAs of the next tile but one never wait for the
// reductions; both half rows of a row share one 528-byte staging row (two
// 256-byte halves + 16 B), five stages.
template <int NEPI>
struct PairCfg {
  static_assert(NEPI == 4 || NEPI == 8, "epilogue warps");
  static constexpr int kStages = NEPI == 8 ? 5 : 6;
  static constexpr int kThreads = 64 + 32 * NEPI;
  static constexpr int kStageRow = NEPI == 8 ? 2 * 256 + 16 : 256 + 16;
  static constexpr int kStaging = kBM * kStageRow;
  static constexpr int kSmem = kStages * kQStage + kStaging + kQBarrierBytes;
  static_assert(kSmem <= 232448, "shared memory");
  static_assert((2 * kStages + 7) * 8 + 8 <= kQBarrierBytes, "barrier area");
};
constexpr uint64_t kQDrainNs = 200ull * 1000 * 1000;
constexpr uint64_t kQSettleNs = 2ull * 1000 * 1000;  // abort path: copies in flight land well within this

__device__ __forceinline__ float q_u2f(uint32_t u) { return __uint_as_float(u); }
// silu(g) * u with the optional clamp (lim = +inf when off): g <= lim,
// -lim <= u <= lim.
__device__ __forceinline__ float q_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// N of a swap-AB up tile: a half pair's routed rows rounded up to 16, or 0
// for a normal tile (every role of both CTAs derives it from the same tables).
__device__ __forceinline__ int up_swap_ns(const GemmArgs& a, int info) {
  if (!a.up_swap || (info & 1)) return 0;
  const int rb0 = info >> 1, e = a.expert_of_rb[rb0];
  const int rows = min(kBM, a.counts[e] - (rb0 * kBM - a.pad_offsets[e]));
  return (rows + 15) & ~15;
}

// N of a swap-AB pair tile (routed rows of the pair rounded up to 16), or 0
// for a normal tile.  Every role of both CTAs derives it from the same tables.
__device__ __forceinline__ int pair_swap_ns(const GemmArgs& a, int info) {
  if (a.pair_swap_max <= 0) return 0;
  const int rb0 = info >> 1, e = a.expert_of_rb[rb0];
  const int rows = min(2 * kBM, a.counts[e] - (rb0 * kBM - a.pad_offsets[e]));
  return rows <= a.pair_swap_max ? (rows + 15) & ~15 : 0;
}

template <int MODE, int NEPI>
__global__ void __launch_bounds__(PairCfg<NEPI>::kThreads, 1)
    gemm_pair2_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                      const __grid_constant__ CUtensorMap map_b64, const GemmArgs args) {
  using Cfg = PairCfg<NEPI>;
  constexpr int kQStages = Cfg::kStages;
  constexpr int kQStageRow = Cfg::kStageRow;
  static_assert(MODE == kPairDown || NEPI == 4, "eight epilogue warps: down projection only");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_addr(smem_raw) & 1023u) {  // the same in every CTA: all of them return here
    if (threadIdx.x == 0) atomicOr(args.err, kErrLaunch);
    return;
  }
  uint8_t* sA = smem_raw;
  uint8_t* sB = sA + kQStages * kQA;
  uint8_t* sStage = sB + kQStages * kQB;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + Cfg::kStaging);
  uint64_t* empty = full + kQStages;
  uint64_t* tfull = empty + kQStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* never = drain + 1;  // no thread ever arrives here (failure-path test hook)
  uint64_t* epi_bar = never + 1;  // this CTA's four epilogue warps (swap-AB staging)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_slot = (int)blockIdx.x >> 1, n_pair_slots = (int)gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&full[s], 1);   // even CTA: its producer's arrive + both CTAs' bytes
      mbar_init(&empty[s], 1);  // the pair MMA's commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * NEPI);  // even CTA: every epilogue warp of each CTA
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    mbar_init(epi_bar, 128);  // the four warps of epilogue half 0
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
    if (MODE == kPairUp && args.up_swap) prefetch_tmap(&map_b64);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // both CTAs' barriers and tensor memory exist
  const uint32_t tmem_base = *tmem_slot;
  // launched as a programmatic dependent: the prologue above overlapped the
  // previous grid; everything below reads its outputs
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();

  const int NJ = args.n_col_tiles;
  const int n_tiles = args.meta[1] * NJ;  // (block pair, column tile)
  const int KB = args.k_blocks;
  // pair_info of the i-th block pair processed: in token-band order for DOWN
  // when an order is given (the reductions then stay within one band of out)
  auto tile_pair = [&](int i) {
    return args.pair_info[(MODE == kPairDown && args.pair_order) ? args.pair_order[i] : i];
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[kQStages];
#pragma unroll
    for (int i = 0; i < kQStages; ++i) issued_phase[i] = -1;
    bool ok = true;
    for (int tile = pair_slot; ok && tile < n_tiles; tile += n_pair_slots) {
      const int info = tile_pair(tile / NJ), j = tile % NJ;
      const int rb0 = info >> 1, two = info & 1;
      const int e = args.expert_of_rb[rb0];
      const int brow = MODE == kPairUp ? e * 2 * args.H + (int)rank * args.H + j * 128
                                       : e * args.D + j * 256 + (int)rank * 128;
      // swap-AB: this CTA's half of the ns routed rows (the TMA box still moves
      // 128 rows; the MMA reads the first ns / 2)
      const int ns = MODE == kPairDown ? pair_swap_ns(args, info) : up_swap_ns(args, info);
      // swap-AB UP: gate and up rows of this CTA's 64 act columns of tile j
      const int wrow = e * 2 * args.H + j * 128 + (int)rank * 64;
      // DOWN half pair (M = 128): this CTA's 64 rows of the block (the box
      // moves 128 rows; the MMA reads the first 64)
      const bool m128 = MODE == kPairDown && !two && !ns && args.half_m128;
      const int arow = ns     ? rb0 * kBM + (int)rank * (ns >> 1)
                       : m128 ? rb0 * kBM + (int)rank * 64
                              : (rb0 + (int)(rank & (uint32_t)two)) * kBM;  // the odd CTA of a half pair reloads rb0
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&empty[s], ph ^ 1u, wc, 61))) break;
        if (leader) mbar_arrive_expect_tx(&full[s], 2 * kQStage);
        const uint32_t fb = mapa_shared(smem_addr(&full[s]), 0);
        tma_load_2d_pair(sA + s * kQA, &map_a, fb, kb * kBK, arow);
        if (MODE == kPairUp && ns) {
          tma_load_2d_pair(sB + s * kQB, &map_b64, fb, kb * kBK, wrow);
          tma_load_2d_pair(sB + s * kQB + kQB / 2, &map_b64, fb, kb * kBK, wrow + args.H);
        } else if (args.l2_policy & 1)  // weight tiles are read by one pair: evict them first
          tma_load_2d_pair_hint(sB + s * kQB, &map_b, fb, kb * kBK, brow, l2_policy_evict_first());
        else
          tma_load_2d_pair(sB + s * kQB, &map_b, fb, kb * kBK, brow);
        issued_phase[s] = (int)ph;
        if (++s == kQStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {  // let every copy already in flight land before the CTA exits
      if (leader) {
        for (int i = 0; i < kQStages; ++i)
          if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kQDrainNs);
      } else {
        spin_ns(kQSettleNs);  // this CTA's loads complete on the even CTA's barriers
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, 256);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 97);  // runs out after the wait limit
    int it = 0;
    for (int tile = pair_slot; ok && tile < n_tiles; tile += n_pair_slots, ++it) {
      const int acc = it & 1;
      if (!(ok = mbar_wait_cluster(&tempty[acc], ((uint32_t)(it >> 1) & 1u) ^ 1u, wc, 62))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * 256;
      const int ns = MODE == kPairDown ? pair_swap_ns(args, tile_pair(tile / NJ)) : up_swap_ns(args, tile_pair(tile / NJ));
      const uint32_t idesc_swap = idesc_bf16_f32(2 * kBM, ns ? ns : 16);
      // DOWN: a half pair runs as one M = 128 pair MMA (64 rows in each CTA)
      const bool m128_t = MODE == kPairDown && !ns && args.half_m128 && !(tile_pair(tile / NJ) & 1);
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&full[s], ph, wc, 63))) break;
        tc_fence_after();
        const uint64_t adesc = sdesc_sw128(smem_addr(sA + s * kQA));
        const uint64_t bdesc = sdesc_sw128(smem_addr(sB + s * kQB));
        if (ns) {  // swap-AB: weight rows are M, the routed rows are N
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_pair(d_tmem, bdesc + 2 * kk, adesc + 2 * kk, idesc_swap, (kb | kk) != 0);
        } else if (m128_t) {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc_bf16_f32(kBM, 256), (kb | kk) != 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
        }
        umma_commit_pair(&empty[s], 0x3);  // frees this stage in both CTAs
        if (++s == kQStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit_pair(&tfull[acc], 0x3);  // both CTAs' accumulators ready
    }
    if (!ok) {  // wait for every MMA already issued before tensor memory is released
      umma_commit_pair(drain, 0x1);
      mbar_wait_drain(drain, 0, kQDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;  // TMEM lanes this warp may access
    const int row = quad * 32 + lane;
    const int ehalf = NEPI == 8 ? (warp - 2) >> 2 : 0;  // eight warps: the half row (128 columns) this warp takes
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_stage = sStage + row * kQStageRow + ehalf * 256;
    const uint32_t tempty_leader0 = mapa_shared(smem_addr(&tempty[0]), 0);
    // barrier of this CTA's 128 epilogue threads (bounded, unlike bar.sync)
    uint32_t epi_ph = 0;
    auto epi_sync = [&](int site) -> bool {
      mbar_arrive(epi_bar);
      const bool got = mbar_wait(epi_bar, epi_ph, wc, site);
      epi_ph ^= 1u;
      return got;
    };
    int it = 0;
    for (int tile = pair_slot; tile < n_tiles; tile += n_pair_slots, ++it) {
      const int acc = it & 1;
      if (!mbar_wait(&tfull[acc], (uint32_t)(it >> 1) & 1u, wc, 64)) break;
      tc_fence_after();
      const int info = tile_pair(tile / NJ), j = tile % NJ;
      const uint32_t tacc = lane_base + acc * 256;
      const int ns = MODE == kPairDown ? pair_swap_ns(args, info) : up_swap_ns(args, info);
      const bool m128 = MODE == kPairDown && !(info & 1) && !ns && args.half_m128;
      // m128: TMEM lane row (0..127) holds columns [128 * half, +128) of tile row
      // (row & 63), the block's row rank * 64 + (row & 63)
      const int half = row >> 6;
      const int64_t slot = m128 ? (int64_t)(info >> 1) * kBM + (int)rank * 64 + (row & 63)
                                : (int64_t)((info >> 1) + (int)rank) * kBM + row;
      const int tok = (m128 || rank == 0 || (info & 1)) ? args.row_tok[slot] : -1;
      const bool valid = tok >= 0;
      bool released = false;  // this warp has already told the MMA issuer it read the accumulator
      if (MODE == kPairDown && m128) {
        // output columns j*256 + 128*half .. +128 of the row (the four warps of
        // epilogue half 0; with eight warps the others have nothing to read)
        if (ehalf == 0) {
          const float w = valid ? args.slot_w[slot] : 0.f;
          uint32_t v[4][32];
          tmem_ld_x32_pair(tacc, tacc + 32, v[0], v[1]);
          tmem_ld_x32_pair(tacc + 64, tacc + 96, v[2], v[3]);
          if (tok >= 0) {
            const int64_t col0 = (int64_t)tok * args.D + j * 256 + half * 128;
            if (args.out_f32) {
#pragma unroll
              for (int c = 0; c < 4; c += 2) {
                bulk_wait_read_all();
                stage_scaled_f32x32(my_stage, w, v[c]);
                stage_scaled_f32x32(my_stage + 128, w, v[c + 1]);
                fence_proxy_async_smem();
                bulk_reduce_add_f32(args.out_f32 + col0 + c * 32, my_stage, 256);
                bulk_commit();
              }
            } else {
              bulk_wait_read_all();
#pragma unroll
              for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  st_shared_v4(my_stage + c * 64 + q * 16, pack_bf16x2(w * q_u2f(v[c][8 * q + 0]), w * q_u2f(v[c][8 * q + 1])),
                               pack_bf16x2(w * q_u2f(v[c][8 * q + 2]), w * q_u2f(v[c][8 * q + 3])),
                               pack_bf16x2(w * q_u2f(v[c][8 * q + 4]), w * q_u2f(v[c][8 * q + 5])),
                               pack_bf16x2(w * q_u2f(v[c][8 * q + 6]), w * q_u2f(v[c][8 * q + 7])));
              fence_proxy_async_smem();
              bulk_reduce_add_bf16_hint(static_cast<__nv_bfloat16*>(args.out) + col0, my_stage, 256,
                                        args.out_hint != 0, l2_policy_evict_last());
              bulk_commit();
            }
          }
        }
      } else if (MODE == kPairDown && ns > 0 && ehalf != 0) {
        // swap-AB tiles are read by the four warps of epilogue half 0
      } else if (MODE == kPairDown && ns > 0) {
        // Swap-AB tile: TMEM lane `row` is output column j*256 + 128*rank + row,
        // column c is routed row c of the pair (slot (info >> 1) * 128 + c).
        // 128 routed rows at a time go transposed into the staging tile (staging
        // row c = routed row c); thread c then reduces staging row c into out.
        const int64_t slot0 = (int64_t)(info >> 1) * kBM;
        const int col = j * 256 + (int)rank * 128;
        bool failed = false;
#pragma unroll 1
        for (int h0 = 0; h0 < ns; h0 += kBM) {
          const int cn = min(ns - h0, kBM);
          bulk_wait_read_all();  // this thread's last reduction has left its staging row
          if (!epi_sync(67)) {
            failed = true;
            break;
          }
#pragma unroll 1
          for (int c0 = 0; c0 < cn; c0 += 64) {
            uint32_t a0[32], a1[32];
            tmem_ld_x32_pair(tacc + h0 + c0, tacc + h0 + c0 + 32, a0, a1);
            const int ci = h0 + c0 + lane;
            const float w0 = ci < ns ? args.slot_w[slot0 + ci] : 0.f;
            const float w1 = ci + 32 < ns ? args.slot_w[slot0 + ci + 32] : 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              st_shared_b16(sStage + (c0 + i) * kQStageRow + row * 2, __shfl_sync(0xffffffffu, w0, i) * q_u2f(a0[i]));
#pragma unroll
            for (int i = 0; i < 32; ++i)
              st_shared_b16(sStage + (c0 + 32 + i) * kQStageRow + row * 2,
                            __shfl_sync(0xffffffffu, w1, i) * q_u2f(a1[i]));
          }
          fence_proxy_async_smem();
          if (!epi_sync(68)) {
            failed = true;
            break;
          }
          if (row < cn) {
            const int tok = args.row_tok[slot0 + h0 + row];
            if (tok >= 0) {
              bulk_reduce_add_bf16_hint(static_cast<__nv_bfloat16*>(args.out) + (int64_t)tok * args.D + col,
                                   sStage + row * kQStageRow, 256, args.out_hint != 0, l2_policy_evict_last());
              bulk_commit();
            }
          }
        }
        if (failed) break;
      } else if (MODE == kPairUp && ns > 0) {
        // Swap-AB half pair: lane c / 64 + c hold gate / up of act column
        // 64 * rank + c, TMEM column r routed row r of the block.  U[r][c]
        // (fp32, 256 B a row) stages the up values in the staging area.
        const int64_t slot0 = (int64_t)(info >> 1) * kBM;
        float* U = reinterpret_cast<float*>(sStage);
        bulk_wait_read_all();  // this thread's last store has left its staging row
        if (!epi_sync(69)) break;  // every staging row free, the previous tile's U reads done
        if (quad >= 2) {
#pragma unroll 1
          for (int r0 = 0; r0 < ns; r0 += 32) {
            uint32_t a[32];
            tmem_ld_x32(tacc + r0, a);
#pragma unroll
            for (int i = 0; i < 32; ++i) U[(r0 + i) * 64 + (row - 64)] = q_u2f(a[i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty_leader0 + acc * 8);
          released = true;
        }
        if (!epi_sync(70)) break;  // U complete
        if (quad < 2) {
          __nv_bfloat16* acol = static_cast<__nv_bfloat16*>(args.act) + j * 128 + (int)rank * 64 + row;
#pragma unroll 1
          for (int r0 = 0; r0 < ns; r0 += 32) {
            uint32_t a[32];
            tmem_ld_x32(tacc + r0, a);
            const int tk = r0 + lane < ns ? args.row_tok[slot0 + r0 + lane] : -1;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int tki = __shfl_sync(0xffffffffu, tk, i);
              if (tki >= 0)
                acol[(slot0 + r0 + i) * args.H] = __float2bfloat16(q_swiglu(q_u2f(a[i]), U[(r0 + i) * 64 + row], swiglu_lim));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty_leader0 + acc * 8);
          released = true;
        }
        if (!epi_sync(71)) break;  // U read: the staging area is free for the next tile
      } else if (MODE == kPairUp) {
        if (tok >= 0) bulk_wait_read_all();  // the previous tile's store has left the staging row
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_x32_pair(tacc + c * 32, tacc + 128 + c * 32, g, u);
          if (tok >= 0) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(q_swiglu(q_u2f(g[2 * i]), q_u2f(u[2 * i]), swiglu_lim),
                                  q_swiglu(q_u2f(g[2 * i + 1]), q_u2f(u[2 * i + 1]), swiglu_lim));
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(my_stage + c * 64 + q * 16, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        if (tok >= 0) {  // act[slot, j*128 .. +128): one 256-byte bulk copy of the staged row
          fence_proxy_async_smem();
          bulk_store(static_cast<__nv_bfloat16*>(args.act) + slot * args.H + j * 128, my_stage, 256);
          bulk_commit();
        }
      } else if (args.out_f32) {
        // fp32 reduction target: quarter rows of 64 columns (256 bytes staged
        // each), all four by one warp, or two by each of a quadrant's two warps
        const float w = valid ? args.slot_w[slot] : 0.f;
        float* frow = args.out_f32 + (int64_t)(tok < 0 ? 0 : tok) * args.D + j * 256;
#pragma unroll 1
        for (int q = 4 / (NEPI / 4) * ehalf; q < 4 / (NEPI / 4) * (ehalf + 1); ++q) {
          bulk_wait_read_all();        // the previous reduction has left the staging row
          uint32_t v0[32], v1[32];
          tmem_ld_x32_pair(tacc + q * 64, tacc + q * 64 + 32, v0, v1);
          if (tok >= 0) {
            stage_scaled_f32x32(my_stage, w, v0);
            stage_scaled_f32x32(my_stage + 128, w, v1);
            fence_proxy_async_smem();
            bulk_reduce_add_f32(frow + q * 64, my_stage, 256);
            bulk_commit();
          }
        }
      } else if (NEPI == 8) {
        // this warp's half row: 128 columns into registers, the accumulator
        // released, then staged and reduced while the MMAs go on
        const float w = valid ? args.slot_w[slot] : 0.f;
        uint32_t v[4][32];
        const uint32_t tcol = tacc + ehalf * 128;
        tmem_ld_x32_pair(tcol, tcol + 32, v[0], v[1]);
        tmem_ld_x32_pair(tcol + 64, tcol + 96, v[2], v[3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader0 + acc * 8);
        released = true;
        if (tok >= 0) {
          bulk_wait_read_all();  // the previous tile's reduction has left the staging half row
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(my_stage + c * 64 + q * 16, pack_bf16x2(w * q_u2f(v[c][8 * q + 0]), w * q_u2f(v[c][8 * q + 1])),
                           pack_bf16x2(w * q_u2f(v[c][8 * q + 2]), w * q_u2f(v[c][8 * q + 3])),
                           pack_bf16x2(w * q_u2f(v[c][8 * q + 4]), w * q_u2f(v[c][8 * q + 5])),
                           pack_bf16x2(w * q_u2f(v[c][8 * q + 6]), w * q_u2f(v[c][8 * q + 7])));
          fence_proxy_async_smem();
          bulk_reduce_add_bf16_hint(static_cast<__nv_bfloat16*>(args.out) + (int64_t)tok * args.D + j * 256 + ehalf * 128,
                                    my_stage, 256, args.out_hint != 0, l2_policy_evict_last());
          bulk_commit();
        }
      } else {
        const float w = valid ? args.slot_w[slot] : 0.f;
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tok < 0 ? 0 : tok) * args.D + j * 256;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {  // two half rows of 128 columns
          bulk_wait_read_all();        // the previous reduction has left the staging row
#pragma unroll 1
          for (int c = h * 4; c < h * 4 + 4; c += 2) {
            uint32_t v0[32], v1[32];
            tmem_ld_x32_pair(tacc + c * 32, tacc + (c + 1) * 32, v0, v1);
            if (tok >= 0) {
              uint8_t* st0 = my_stage + (c - h * 4) * 64;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                st_shared_v4(st0 + q * 16, pack_bf16x2(w * q_u2f(v0[8 * q + 0]), w * q_u2f(v0[8 * q + 1])),
                             pack_bf16x2(w * q_u2f(v0[8 * q + 2]), w * q_u2f(v0[8 * q + 3])),
                             pack_bf16x2(w * q_u2f(v0[8 * q + 4]), w * q_u2f(v0[8 * q + 5])),
                             pack_bf16x2(w * q_u2f(v0[8 * q + 6]), w * q_u2f(v0[8 * q + 7])));
#pragma unroll
              for (int q = 0; q < 4; ++q)
                st_shared_v4(st0 + 64 + q * 16, pack_bf16x2(w * q_u2f(v1[8 * q + 0]), w * q_u2f(v1[8 * q + 1])),
                             pack_bf16x2(w * q_u2f(v1[8 * q + 2]), w * q_u2f(v1[8 * q + 3])),
                             pack_bf16x2(w * q_u2f(v1[8 * q + 4]), w * q_u2f(v1[8 * q + 5])),
                             pack_bf16x2(w * q_u2f(v1[8 * q + 6]), w * q_u2f(v1[8 * q + 7])));
            }
          }
          if (tok >= 0) {
            fence_proxy_async_smem();
            bulk_reduce_add_bf16_hint(orow + h * 128, my_stage, 256, args.out_hint != 0, l2_policy_evict_last());
            bulk_commit();
          }
        }
      }
      // this warp has read the accumulator: tell the even CTA's MMA issuer
      if (!released) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader0 + acc * 8);
      }
    }
    bulk_wait_all();  // bulk stores / reductions complete before the CTA exits
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still use its barriers or shared memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

template <int MODE, int NEPI>
cudaError_t launch_pair2(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b64, const GemmArgs& args,
                         int n_pairs, cudaStream_t stream, bool pdl) {
  auto kern = gemm_pair2_kernel<MODE, NEPI>;
  constexpr int kQSmem = PairCfg<NEPI>::kSmem;
  // once per device: not a stream operation, so it stays out of graph capture
  static bool smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
    if (err != cudaSuccess) return err;
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n_pairs);
  cfg.blockDim = dim3(PairCfg<NEPI>::kThreads);
  cfg.dynamicSmemBytes = kQSmem;
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
  return cudaLaunchKernelEx(&cfg, kern, a, b, b64, args);
}

}  // namespace

int pair_cluster_slots() {
  // once per device: not a stream operation
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev]) return cache[dev];
  auto kern = gemm_pair2_kernel<kPairUp, 4>;
  constexpr int kQSmem = PairCfg<4>::kSmem;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(PairCfg<4>::kThreads);
  cfg.dynamicSmemBytes = kQSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cache[dev] = n;
  return n;
}

cudaError_t launch_up_pair2_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w1_64,
                                 const GemmArgs& args, int n_pairs, cudaStream_t stream, bool pdl) {
  return launch_pair2<kPairUp, 4>(map_xg, map_w1, map_w1_64, args, n_pairs, stream, pdl);
}

cudaError_t launch_down_pair2_bf16(const CUtensorMap& map_act, const CUtensorMap& map_w2, const GemmArgs& args,
                                   int n_pairs, cudaStream_t stream, bool pdl) {
  return args.down_epi8 ? launch_pair2<kPairDown, 8>(map_act, map_w2, map_w2, args, n_pairs, stream, pdl)
                        : launch_pair2<kPairDown, 4>(map_act, map_w2, map_w2, args, n_pairs, stream, pdl);
}

}  // namespace moe
