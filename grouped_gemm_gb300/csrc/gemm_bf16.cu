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
constexpr int kTileSlots = 4;   // depth of the producer -> consumers tile-index ring

template <int MODE, int N, int STAGES, int BM = kBM>
struct GemmCfg {
  static constexpr int kABytes = BM * kBK * 2;              // 16 KB (8 KB for 64-row tiles)
  static constexpr int kBBytes = N * kBK * 2;               // N rows of 128 B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * N;                   // double-buffered accumulator
  // DOWN stages half an output row (N/2 bf16) at a time in shared memory for
  // the bulk reduction; +16 B per row keeps the 32 rows of a warp on distinct
  // banks.  Half rows leave room for a 4-stage ring.
  // UP stages its row of N/2 act values the same way and writes it with one
  // bulk copy.
  static constexpr int kStageRowBytes = N + 16;
  static constexpr int kStagingBytes = BM * kStageRowBytes;
  static constexpr int kBarrierBytes = STAGES > 6 ? 512 : 256;
  // No alignment slack: dynamic shared memory starts 1024-byte aligned (the
  // kernel checks and reports an error otherwise).
  static constexpr int kSmemBytes = STAGES * kStageBytes + kStagingBytes + kBarrierBytes;
  static_assert(N % 32 == 0 && N >= 32 && N <= 256, "MMA N");
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns: power of two <= 512");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert((2 * STAGES + 7 + 2 * kTileSlots) * 8 + 8 + 8 * kTileSlots <= kBarrierBytes, "barrier area");
};

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kGatherThreads = 128;   // extra producer warps 6..9 of the cp.async gather
enum { kGatherTile = 0, kGatherTma4 = 1, kGatherCpAsync = 2 };
template <int GATHER>
constexpr int threads_for() { return GATHER == kGatherCpAsync ? kThreads + kGatherThreads : kThreads; }
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;  // 200 ms

// Swap-AB tail tiles.  The last row block of an expert holds v < 128 routed
// rows; with M fixed at 128 rows a normal tile spends (128 - v) / 128 of its
// MMA work on padding.  With the operands swapped the weight tile is the
// M = 128 side and the routed rows are N = ns = v rounded up to 16: two MMAs
// (weight rows 0..127 and 128..255 of the stage) accumulate transposed
// results into TMEM columns [0, ns) and [128, 128 + ns), for 256 * ns instead
// of 128 * 256 multiply-adds per K step ("Prime Flash MoE" and Pearl
// "Optimizing Grouped GEMM for MoE on Blackwell": swap-AB for small
// per-expert M).  Only the 256-row B stages (N = 256) have two 128-row halves.
constexpr int kSwapMaxN = 112;

// Rows of row block rb (of expert e) that hold routed pairs; the rest is padding.
__device__ __forceinline__ int rb_rows(const GemmArgs& a, int rb, int e) {
  return min(kBM, a.counts[e] - (rb * kBM - a.pad_offsets[e]));
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// silu(g) * u = g / (1 + e^-g) * u; fast reciprocal division (the result is
// rounded to bf16 right after).
// silu(g) * u with the optional clamp (lim = +inf when off): g <= lim,
// -lim <= u <= lim.
__device__ __forceinline__ float swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// BM = 64: 64-row tiles (tcgen05.mma M = 64), for problems with few routed
// rows per expert (Pearl "Optimizing Grouped GEMM for MoE on Blackwell":
// tile_m = 64 in 1-CTA mode halves the token stage, so more weight stages fit).
// Each 128-row block is two 64-row halves; tiles are ordered all first halves,
// then all second halves, and a second half without routed rows is skipped.
// The M = 64 accumulator sits in TMEM lanes 0..15 of each 32-lane quadrant
// (row r in lane 32 * (r / 16) + r % 16), so epilogue lanes 16..31 idle.
template <int MODE, int N, int STAGES, int GATHER, int BM = kBM>
__global__ void __launch_bounds__(threads_for<GATHER>(), 1)
    grouped_gemm_bf16_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                             const GemmArgs args) {
  static_assert(BM == kBM || (BM == 64 && GATHER == kGatherTile), "64-row tiles read the pre-gathered rows");
  using Cfg = GemmCfg<MODE, N, STAGES, BM>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_addr(smem_raw) & 1023u) {  // SW128 tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(args.err, kErrLaunch);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::kABytes;
  uint8_t* sStage = smem + STAGES * Cfg::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + Cfg::kStagingBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* never = drain + 1;  // no thread ever arrives here (failure-path test hook)
  uint64_t* epi_bar = never + 1;  // the epilogue warps' barrier around the swap-AB staging tile
  uint64_t* tile_full = epi_bar + 1;
  uint64_t* tile_empty = tile_full + kTileSlots;
  volatile int* tile_ring = reinterpret_cast<volatile int*>(tile_empty + kTileSlots);
  volatile int* tile_ns = tile_ring + kTileSlots;  // swap-AB width of each published tile, 0 = normal
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(tile_ns) + kTileSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};
  // Tile sequence: warp 0 draws tile indices (from a global atomic counter
  // when args.tile_counter is set -- CTAs that finish early take more tiles --
  // else the static round-robin blockIdx.x + i * gridDim.x) and publishes them
  // through a small ring; the MMA issuer, the epilogue and the gather warps
  // read the same sequence.  An index >= n_tiles ends the sequence.
  constexpr int kTileReaders = 1 + kEpiThreads + (GATHER == kGatherCpAsync ? kGatherThreads : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // with the cp.async gather, each of its threads also arrives once per stage
      mbar_init(&full[s], GATHER == kGatherCpAsync ? 1 + kGatherThreads : 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiThreads);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    mbar_init(epi_bar, kEpiThreads);
    for (int i = 0; i < kTileSlots; ++i) {
      mbar_init(&tile_full[i], 1);
      mbar_init(&tile_empty[i], kTileReaders);
    }
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
  // Launched as a programmatic dependent, the prologue above overlaps the
  // previous grid; everything below reads its outputs (xg or act, and the
  // routing tables, complete before that grid began).
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();

  const int num_rb = args.meta[0];
  constexpr int kHalves = kBM / BM;  // row tiles per 128-row block
  const int n_tiles = num_rb * kHalves * args.n_col_tiles;
  const int KB = args.k_blocks;
  // the 128-row block of a tile and the first padded slot of its rows
  auto tile_rb = [&](int tile) {
    const int rbh = tile / args.n_col_tiles;
    return kHalves == 1 ? rbh : (rbh >= num_rb ? rbh - num_rb : rbh);
  };
  auto tile_row0 = [&](int tile) -> int64_t {
    const int rbh = tile / args.n_col_tiles;
    return kHalves == 1 ? (int64_t)rbh * kBM : (int64_t)tile_rb(tile) * kBM + (rbh >= num_rb ? BM : 0);
  };

  // consumer side of the tile ring: the next tile index, or -1 if aborting;
  // t_ns gets the tile's swap-AB width (0 = normal tile)
  int t_slot = 0;
  uint32_t t_phase = 0;
  int t_ns = 0;
  auto take_tile = [&](int site) -> int {
    if (!mbar_wait(&tile_full[t_slot], t_phase, wc, site)) return -1;
    const int t = tile_ring[t_slot];
    t_ns = tile_ns[t_slot];
    mbar_arrive(&tile_empty[t_slot]);
    if (++t_slot == kTileSlots) {
      t_slot = 0;
      t_phase ^= 1u;
    }
    return t;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
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
      if (BM != kBM || pf_tile >= n_tiles) return;
      const int prb = pf_tile / args.n_col_tiles, pj = pf_tile % args.n_col_tiles;
      if (GATHER == kGatherTile) tma_prefetch_2d(&map_a, pf_kb * kBK, prb * kBM);
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
    int tile = -1;
    while (ok) {
      // publish the next tile index to the other roles (warp 0, lane 0)
      int next = 0;
      if (lane == 0) {
        if (!mbar_wait(&tile_empty[t_slot], t_phase ^ 1u, wc, 6)) {
          next = -1;
        } else {
          next = args.tile_counter ? atomicAdd(args.tile_counter, 1)
                                   : (tile < 0 ? (int)blockIdx.x : tile + (int)gridDim.x);
          // 64-row tiles: skip a second half that holds no routed rows
          while (BM != kBM && next < n_tiles && next >= num_rb * args.n_col_tiles) {
            const int nrb = tile_rb(next);
            if (rb_rows(args, nrb, args.expert_of_rb[nrb]) > BM) break;
            next = args.tile_counter ? atomicAdd(args.tile_counter, 1) : next + (int)gridDim.x;
          }
          int ns = 0;
          if (BM == kBM && N == 256 && args.swap_ab && next < n_tiles) {
            const int nrb = next / args.n_col_tiles;
            const int v = rb_rows(args, nrb, args.expert_of_rb[nrb]);
            if (v < kBM && ((v + 15) & ~15) <= kSwapMaxN) ns = (v + 15) & ~15;
          }
          tile_ring[t_slot] = next;
          tile_ns[t_slot] = ns;
          mbar_arrive(&tile_full[t_slot]);
        }
      }
      next = __shfl_sync(0xffffffffu, next, 0);
      if (++t_slot == kTileSlots) {
        t_slot = 0;
        t_phase ^= 1u;
      }
      if (next < 0) {
        ok = false;
        break;
      }
      if (next >= n_tiles) break;
      tile = next;
      const int rb = tile_rb(tile), j = tile % args.n_col_tiles;
      const int e = args.expert_of_rb[rb];
      const int a_row0 = (int)tile_row0(tile);
      int g0 = 0, g1 = 0, g2 = 0, g3 = 0;
      if (GATHER == kGatherTma4) {  // lane l fetches tile rows 4l..4l+3; padding rows read row 0
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
          if (got)
            mbar_arrive_expect_tx(&full[s], GATHER == kGatherCpAsync ? Cfg::kBBytes : Cfg::kStageBytes);
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        if (GATHER == kGatherTma4) {
          tma_gather4(sA + s * Cfg::kABytes + lane * 4 * kBK * 2, &map_a, &full[s], kb * kBK, g0, g1, g2, g3);
        } else if (GATHER == kGatherTile && lane == 0) {
          tma_load_2d(sA + s * Cfg::kABytes, &map_a, &full[s], kb * kBK, a_row0);
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
    constexpr uint32_t idesc = idesc_bf16_f32(BM, N);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 90);  // runs out after the wait limit
    int it = 0;
    for (; ok; ++it) {
      const int tile = take_tile(7);
      if (tile < 0) {
        ok = false;
        break;
      }
      if (tile >= n_tiles) break;
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(&tempty[acc], aph ^ 1u, wc, 2)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * N;
      const int ns = t_ns;
      const uint32_t idesc_swap = idesc_bf16_f32(kBM, ns > 0 ? ns : 16);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&full[s], ph, wc, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = sdesc_sw128(smem_addr(sA + s * Cfg::kABytes));
        const uint64_t bdesc = sdesc_sw128(smem_addr(sB + s * Cfg::kBBytes));
        if (BM == kBM && N == 256 && ns > 0) {
          // swap-AB: weight rows are M, the tile's routed rows are N
          const uint64_t bdesc_hi = sdesc_sw128(smem_addr(sB + s * Cfg::kBBytes + kBM * kBK * 2));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            umma_bf16(d_tmem, bdesc + 2 * kk, adesc + 2 * kk, idesc_swap, (kb | kk) != 0);
            umma_bf16(d_tmem + kBM, bdesc_hi + 2 * kk, adesc + 2 * kk, idesc_swap, (kb | kk) != 0);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // +32 bytes per K step of 16 bf16 = +2 in the descriptor's address field
            umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
          }
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
  } else if (GATHER == kGatherCpAsync && warp >= 6) {
    // ------------------------------------------------------------ row gather
    // 128 threads copy the tile's 128 token rows straight from x: thread t
    // moves 16-byte chunk t%8 of rows t/8 + 16i (i < 8), written at its
    // 128-byte-swizzle position, so each warp instruction covers four whole
    // 128-byte row segments.  A stage is released to the MMA issuer
    // (fence.proxy.async, then an arrive on full[]) kLag stages after it was
    // issued, when cp.async.wait_group shows its copies have landed.
    constexpr int kLag = STAGES - 1;
    const int gt = threadIdx.x - kThreads;
    const int chunk = gt & 7, r0 = gt >> 3;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(args.x);
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    bool ok = true;
    while (ok) {
      const int tile = take_tile(8);
      if (tile < 0) {
        ok = false;
        break;
      }
      if (tile >= n_tiles) break;
      const int rb = tile / args.n_col_tiles;
      const __nv_bfloat16* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        src[i] = x + (int64_t)max(args.row_tok[(int64_t)rb * kBM + r0 + 16 * i], 0) * args.D + chunk * 8;
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&empty[s], ph ^ 1u, wc, 5))) break;
        uint8_t* a = sA + s * Cfg::kABytes;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = r0 + 16 * i;
          cp_async_16(a + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + kb * kBK);
        }
        cp_async_commit();
        if (issued >= kLag) {
          cp_async_wait_group<kLag>();
          fence_proxy_async_smem();
          mbar_arrive(&full[(issued - kLag) % STAGES]);
        }
        ++issued;
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    cp_async_wait_group<0>();
    if (ok) {  // release the last stages
      fence_proxy_async_smem();
      for (int n = max(issued - kLag, 0); n < issued; ++n) mbar_arrive(&full[n % STAGES]);
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may access
    // the tile row this thread's TMEM lane holds (64-row tiles: lanes 0..15 only)
    const bool row_lane = BM == kBM || lane < 16;
    const int row = BM == kBM ? quad * 32 + lane : quad * 16 + (lane & 15);
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_stage = sStage + row * Cfg::kStageRowBytes;
    // barrier of the 128 epilogue threads (bounded, unlike bar.sync)
    uint32_t epi_ph = 0;
    auto epi_sync = [&](int site) -> bool {
      mbar_arrive(epi_bar);
      const bool got = mbar_wait(epi_bar, epi_ph, wc, site);
      epi_ph ^= 1u;
      return got;
    };
    int it = 0;
    for (;; ++it) {
      const int tile = take_tile(9);
      if (tile < 0 || tile >= n_tiles) break;
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(&tfull[acc], aph, wc, 4)) break;
      tc_fence_after();
      const int rb = tile_rb(tile), j = tile % args.n_col_tiles;
      const int64_t slot = tile_row0(tile) + row;
      const int tok = row_lane ? args.row_tok[slot] : -1;
      const uint32_t tacc = lane_base + acc * N;
      const int ns = t_ns;
      if (BM == kBM && N == 256 && ns > 0) {
        // Swap-AB tile: this thread's TMEM lane is weight row `row` of each
        // 128-row half and the columns are the tile's rows c < ns.  The values
        // go transposed into the staging tile (staging row c = tile row c),
        // then thread c moves staging row c with one bulk operation, as in a
        // normal tile.  Staging rows of padding slots are written, not moved.
        bool failed = false;
        if (MODE == kModeUp) {
          constexpr int G = N / 2;
          bulk_wait_read_all();  // this thread's last store has left the staging tile
          if (!epi_sync(12)) break;
#pragma unroll 1
          for (int c0 = 0; c0 < ns; c0 += 32) {
            uint32_t g[32], u[32];
            tmem_ld_x32_pair(tacc + c0, tacc + kBM + c0, g, u);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              st_shared_b16(sStage + (c0 + i) * Cfg::kStageRowBytes + row * 2, swiglu(u2f(g[i]), u2f(u[i]), swiglu_lim));
          }
          fence_proxy_async_smem();
          if (!epi_sync(13)) break;
          if (tok >= 0) {
            bulk_store(static_cast<__nv_bfloat16*>(args.act) + slot * args.H + j * G, my_stage, G * 2);
            bulk_commit();
          }
        } else {
          const float* wrow = args.slot_w + (int64_t)rb * kBM;
          __nv_bfloat16* orow =
              static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tok < 0 ? 0 : tok) * args.D + j * N;
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {  // D columns j*N + hh*128 .. +128
            bulk_wait_read_all();
            if (!epi_sync(12)) {
              failed = true;
              break;
            }
#pragma unroll 1
            for (int c0 = 0; c0 < ns; c0 += 64) {
              uint32_t a0[32], a1[32];
              tmem_ld_x32_pair(tacc + hh * kBM + c0, tacc + hh * kBM + c0 + 32, a0, a1);
              const float w0 = wrow[c0 + lane], w1 = wrow[c0 + 32 + lane];
#pragma unroll
              for (int i = 0; i < 32; ++i)
                st_shared_b16(sStage + (c0 + i) * Cfg::kStageRowBytes + row * 2,
                              __shfl_sync(0xffffffffu, w0, i) * u2f(a0[i]));
#pragma unroll
              for (int i = 0; i < 32; ++i)
                st_shared_b16(sStage + (c0 + 32 + i) * Cfg::kStageRowBytes + row * 2,
                              __shfl_sync(0xffffffffu, w1, i) * u2f(a1[i]));
            }
            fence_proxy_async_smem();
            if (!epi_sync(13)) {
              failed = true;
              break;
            }
            if (tok >= 0) {
              bulk_reduce_add_bf16_hint(orow + hh * kBM, my_stage, kBM * 2, args.out_hint != 0, l2_policy_evict_last());
              bulk_commit();
            }
          }
        }
        if (failed) break;
      } else if (MODE == kModeUp) {
        constexpr int G = N / 2;
        if (tok >= 0) bulk_wait_read_all();  // the previous tile's store has left the staging row
#pragma unroll 1
        for (int c = 0; c < G / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_x32_pair(tacc + c * 32, tacc + G + c * 32, g, u);
          if (tok >= 0) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(swiglu(u2f(g[2 * i]), u2f(u[2 * i]), swiglu_lim), swiglu(u2f(g[2 * i + 1]), u2f(u[2 * i + 1]), swiglu_lim));
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(my_stage + c * 64 + q * 16, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        if (tok >= 0) {  // act[slot, j*G .. +G): one 2G-byte bulk copy of the staged row
          fence_proxy_async_smem();
          bulk_store(static_cast<__nv_bfloat16*>(args.act) + slot * args.H + j * G, my_stage, G * 2);
          bulk_commit();
        }
      } else if (args.out_f32) {
        // fp32 reduction target: four chunks of N/4 columns (N bytes staged each)
        constexpr int CW = N / 4;
        const float w = args.slot_w[slot];
        float* frow = args.out_f32 + (int64_t)(tok < 0 ? 0 : tok) * args.D + j * N;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          bulk_wait_read_all();          // the previous reduction has left the staging row
#pragma unroll 1
          for (int c = 0; c < CW / 32; ++c) {
            uint32_t v[32];
            tmem_ld_x32(tacc + q * CW + c * 32, v);
            if (tok >= 0) stage_scaled_f32x32(my_stage + c * 128, w, v);
          }
          if (tok >= 0) {
            fence_proxy_async_smem();
            bulk_reduce_add_f32(frow + q * CW, my_stage, CW * 4);
            bulk_commit();
          }
        }
      } else {
        const float w = args.slot_w[slot];
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tok < 0 ? 0 : tok) * args.D + j * N;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {     // two half rows of N/2 columns
          bulk_wait_read_all();          // the previous reduction has left the staging row
#pragma unroll 1
          for (int c = h * (N / 64); c < (h + 1) * (N / 64); c += 2) {
            uint32_t v0[32], v1[32];
            tmem_ld_x32_pair(tacc + c * 32, tacc + (c + 1) * 32, v0, v1);
            if (tok >= 0) {
              uint8_t* st0 = my_stage + (c - h * (N / 64)) * 64;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                st_shared_v4(st0 + q * 16, pack_bf16x2(w * u2f(v0[8 * q + 0]), w * u2f(v0[8 * q + 1])),
                             pack_bf16x2(w * u2f(v0[8 * q + 2]), w * u2f(v0[8 * q + 3])),
                             pack_bf16x2(w * u2f(v0[8 * q + 4]), w * u2f(v0[8 * q + 5])),
                             pack_bf16x2(w * u2f(v0[8 * q + 6]), w * u2f(v0[8 * q + 7])));
#pragma unroll
              for (int q = 0; q < 4; ++q)
                st_shared_v4(st0 + 64 + q * 16, pack_bf16x2(w * u2f(v1[8 * q + 0]), w * u2f(v1[8 * q + 1])),
                             pack_bf16x2(w * u2f(v1[8 * q + 2]), w * u2f(v1[8 * q + 3])),
                             pack_bf16x2(w * u2f(v1[8 * q + 4]), w * u2f(v1[8 * q + 5])),
                             pack_bf16x2(w * u2f(v1[8 * q + 6]), w * u2f(v1[8 * q + 7])));
            }
          }
          if (tok >= 0) {
            fence_proxy_async_smem();
            bulk_reduce_add_bf16_hint(orow + h * (N / 2), my_stage, N, args.out_hint != 0, l2_policy_evict_last());
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
    bulk_wait_all();  // bulk stores / reductions complete before the CTA exits
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

template <int MODE, int N, int STAGES, int GATHER, int BM = kBM>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& args, int grid,
                        cudaStream_t stream, bool pdl) {
  using Cfg = GemmCfg<MODE, N, STAGES, BM>;
  auto kern = grouped_gemm_bf16_kernel<MODE, N, STAGES, GATHER, BM>;
  // once per device: not a stream operation, so it stays out of graph capture
  static bool smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (err != cudaSuccess) return err;
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads_for<GATHER>());
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
                           cudaStream_t stream, int gather, int fold, bool pdl, int bm) {
  if (bm == 64) {  // 64-row tiles (map_a boxes of 64 rows), pre-gathered rows
    if (fold == kUpFoldNarrow)
      return launch_gemm<kModeUp, 2 * kUpFoldNarrow, kUpStagesM64Narrow, kGatherTile, 64>(map_a, map_w1, args, grid,
                                                                                        stream, pdl);
    return launch_gemm<kModeUp, 2 * kUpFold, kUpStagesM64, kGatherTile, 64>(map_a, map_w1, args, grid, stream, pdl);
  }
  if (fold == kUpFoldNarrow)  // 64 gate + 64 up rows per tile, 6-stage ring
    return launch_gemm<kModeUp, 2 * kUpFoldNarrow, kUpStagesNarrow, kGatherTile>(map_a, map_w1, args, grid, stream,
                                                                                pdl);
  if (gather == kGatherTma4)
    return launch_gemm<kModeUp, 2 * kUpFold, kUpStages, kGatherTma4>(map_a, map_w1, args, grid, stream, pdl);
  if (gather == kGatherCpAsync)
    return launch_gemm<kModeUp, 2 * kUpFold, kUpStages, kGatherCpAsync>(map_a, map_w1, args, grid, stream, pdl);
  return launch_gemm<kModeUp, 2 * kUpFold, kUpStages, kGatherTile>(map_a, map_w1, args, grid, stream, pdl);
}

cudaError_t launch_down_bf16(const CUtensorMap& map_act, const CUtensorMap& map_w2, const GemmArgs& args, int grid,
                             cudaStream_t stream, bool pdl, int n, int bm) {
  if (bm == 64) {  // 64-row tiles (map_act boxes of 64 rows)
    if (n == kDownNNarrow)
      return launch_gemm<kModeDown, kDownNNarrow, kDownStagesM64Narrow, kGatherTile, 64>(map_act, map_w2, args, grid,
                                                                                        stream, pdl);
    return launch_gemm<kModeDown, kDownN, kDownStagesM64, kGatherTile, 64>(map_act, map_w2, args, grid, stream, pdl);
  }
  if (n == kDownNNarrow)  // D % 256 != 0: 128-column output tiles
    return launch_gemm<kModeDown, kDownNNarrow, kDownStagesNarrow, kGatherTile>(map_act, map_w2, args, grid, stream,
                                                                              pdl);
  return launch_gemm<kModeDown, kDownN, kDownStages, kGatherTile>(map_act, map_w2, args, grid, stream, pdl);
}

}  // namespace moe
