// gemm_mx_swap.cu -- the MXFP8 split pipeline's GEMMs with the operands
// swapped, for decode-sized problems: the weights are the M side of
// tcgen05.mma kind::mxf8f6f4.block_scale (128 rows per MMA) and a row
// block's routed rows the N side (ns = its routed rows rounded up to 16), so
// the tensor cores do 128 x ns rather than 128 x 256 multiply-adds per K
// step when an expert holds a few dozen rows ("Porting Block-Scaled GEMM
// Kernels" sec. 5.1 and Pearl "Optimizing Grouped GEMM for MoE on Blackwell":
// swap-AB for small per-expert M).  The weights may be e4m3 or E2M1 (MXFP4,
// read at 4 bits through a 16U4_ALIGN16B map; its format code 5 now sits in
// the A field of the instruction descriptor, bits 7-9).
//
// UP:   tile (row block rb, act columns j*128 .. +128).  Two accumulators in
//       tensor memory, G = W1 gate rows j*128.. x xg^T and U = W1 up rows
//       H + j*128.. x xg^T, so lane c of both holds act column c and TMEM
//       column r routed row r: silu(G) * U needs no exchange between lanes.
//       The requantization to MXFP8 per 32 act columns takes the 32 lanes of
//       one warp: a warp-wide max of |act| gives the block's ue8m0 exponent
//       (the same rule, in fp32, as the single-CTA kernel), each lane
//       converts its own value, and lane 0 writes the scale byte.
// DOWN: tile (row block rb, output columns j*128 .. +128): D = W2 rows x
//       act^T; each warp stages its 32 output columns of every routed row
//       (w times the accumulator, bf16) into a shared-memory row, and thread r
//       reduces staged row r into out[token of r] with one bulk .add.bf16.
//
// Scale factors: the weights' 128-row scale tiles are the A scales as
// prepared for the other kernels; the routed rows' tile (xg_sf / act_sf of
// the row block) holds the B scales of its first ns rows, which an N <= 128
// MMA reads from the same lanes as the first 128 columns of an N = 256 one.
// Every wait is bounded; warp 0 issues TMA, one lane of warp 1 the MMAs,
// warps 2..5 drain tensor memory (one per lane quadrant).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "mx.cuh"
#include "mx_swap.h"
#include "ptx.cuh"

namespace moe {
namespace {

enum { kSwUp = 0, kSwDown = 1 };
constexpr int kSwThreads = 192;
constexpr int kSwXBox = 32;                      // routed rows per TMA box of the N-side operand
constexpr uint64_t kSwDrainNs = 200ull * 1000 * 1000;

template <int MODE>
struct SwCfg {
  static constexpr int kStages = 4;
  static constexpr int kNA = MODE == kSwUp ? 2 : 1;   // weight tiles per stage (gate + up, or one)
  static constexpr int kA = 128 * 128;                // 16 KB of shared memory per weight tile
  static constexpr int kX = 128 * 128;                // up to 128 routed rows x 128 K (four boxes)
  static constexpr int kSF = 512 * (kNA + 1);         // weight scale tile(s) + the routed rows' tile
  static constexpr int kStage = kNA * kA + kX + kSF;
  static constexpr int kStageRow = 256 + 16;          // DOWN staging row: 128 bf16 + 16 B (distinct banks)
  static constexpr int kStaging = MODE == kSwDown ? 128 * kStageRow : 0;
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmem = 1024 + kStages * kStage + kStaging + kBarrierBytes;
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(128 * kNA + 16 * kStages <= 512, "TMEM columns");
};

__device__ __forceinline__ float sw_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Routed rows of row block rb: a prefix of the block (the padding rows of an
// expert's segment come last).  Rounded up to 16 it is the MMAs' N.
__device__ __forceinline__ int sw_rows(const MxSwapArgs& a, int rb) {
  const int e = a.expert_of_rb[rb];
  return min(kBM, a.counts[e] - (rb * kBM - a.pad_offsets[e]));
}

template <int MODE, int FP4W>
__global__ void __launch_bounds__(kSwThreads, 1)
    gemm_mx_swap_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                        const MxSwapArgs args) {
  using Cfg = SwCfg<MODE>;
  constexpr int ST = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                              // [ST][kNA][kA]
  uint8_t* sX = sA + ST * Cfg::kNA * Cfg::kA;      // [ST][kX]
  uint8_t* sSF = sX + ST * Cfg::kX;                // [ST][kSF]
  uint8_t* sStage = sSF + ST * Cfg::kSF;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + Cfg::kStaging);
  uint64_t* empty = full + ST;
  uint64_t* tfull = empty + ST;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* never = drain + 1;
  uint64_t* epi_bar = never + 1;  // the four epilogue warps (DOWN staging)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 4);  // one arrive per epilogue warp
    mbar_init(drain, 1);
    mbar_init(never, 1);
    mbar_init(epi_bar, 128);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_w);
    prefetch_tmap(&map_x);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (MODE == kSwUp && threadIdx.x == 0) griddep_launch_dependents();
  if (MODE == kSwDown) {  // programmatic dependent of the up kernel: act is read below
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();
  }

  const int NJ = args.n_col_tiles;
  const int n_tiles = args.meta[0] * NJ;
  const int KB = args.k_blocks;
  const uint8_t* sf_x = static_cast<const uint8_t*>(args.sf_x);
  const uint8_t* sf_w = static_cast<const uint8_t*>(args.sf_w);
  constexpr int kABytes = FP4W ? Cfg::kA / 2 : Cfg::kA;  // bytes a weight tile moves (packed E2M1: half)

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[ST];
#pragma unroll
    for (int i = 0; i < ST; ++i) issued_phase[i] = -1;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
      const int rb = tile / NJ, j = tile % NJ;
      const int e = args.expert_of_rb[rb];
      const int nbox = (sw_rows(args, rb) + kSwXBox - 1) / kSwXBox;
      // 128-row weight tiles: gate and up rows of act columns j*128.. (UP), W2 rows j*128.. (DOWN)
      const int rt0 = MODE == kSwUp ? e * (2 * args.H / 128) + j : e * (args.D / 128) + j;
      const int rt1 = rt0 + args.H / 128;  // UP: the up rows
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&empty[s], ph ^ 1u, wc, 111))) break;
        mbar_arrive_expect_tx(&full[s], Cfg::kNA * kABytes + nbox * kSwXBox * 128 + Cfg::kSF);
        issued_phase[s] = (int)ph;
        uint8_t* a = sA + s * Cfg::kNA * Cfg::kA;
        uint8_t* x = sX + s * Cfg::kX;
        uint8_t* sf = sSF + s * Cfg::kSF;
        tma_load_2d(a, &map_w, &full[s], kb * 128, rt0 * 128);
        bulk_load(sf, sf_w + sf_tile_offset(rt0, kb, KB), 512, &full[s]);
        if (MODE == kSwUp) {
          tma_load_2d(a + Cfg::kA, &map_w, &full[s], kb * 128, rt1 * 128);
          bulk_load(sf + 512, sf_w + sf_tile_offset(rt1, kb, KB), 512, &full[s]);
        }
        for (int bx = 0; bx < nbox; ++bx)
          tma_load_2d(x + bx * kSwXBox * 128, &map_x, &full[s], kb * 128, rb * kBM + bx * kSwXBox);
        bulk_load(sf + Cfg::kNA * 512, sf_x + sf_tile_offset(rb, kb, KB), 512, &full[s]);
        if (++s == ST) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      for (int i = 0; i < ST; ++i)
        if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kSwDrainNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 112);
    int it = 0;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++it) {
      const int ns = (sw_rows(args, tile / NJ) + 15) & ~15;
      // A = weights (E2M1 or e4m3 in the A format field), B = routed rows (e4m3)
      const uint32_t idesc = idesc_mxf8(128, ns) | (FP4W ? kFmtE2M1 << 7 : 0u);
      if (!(ok = mbar_wait(tempty, ((uint32_t)it & 1u) ^ 1u, wc, 113))) break;
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&full[s], ph, wc, 114))) break;
        tc_fence_after();
        // scale tiles -> the TMEM columns of this ring slot: weights (one or
        // two tiles) then the routed rows
        const uint32_t sf_col = tmem_base + 128 * Cfg::kNA + 16 * s;
        const uint32_t sf_smem = smem_addr(sSF + s * Cfg::kSF);
#pragma unroll
        for (int t = 0; t <= Cfg::kNA; ++t) utccp_sf(sf_col + 4 * t, sdesc_sf_tile(sf_smem + 512 * t));
        const uint32_t sfx_col = sf_col + 4 * Cfg::kNA;
        const uint64_t xd = sdesc_sw128(smem_addr(sX + s * Cfg::kX));
#pragma unroll
        for (int t = 0; t < Cfg::kNA; ++t) {
          const uint64_t ad = sdesc_sw128(smem_addr(sA + (s * Cfg::kNA + t) * Cfg::kA));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_mxf8(tmem_base + 128 * t, ad + 2 * kk, xd + 2 * kk, idesc_with_sf_id(idesc, kk), sf_col + 4 * t,
                      sfx_col, (kb | kk) != 0);
        }
        umma_commit(&empty[s]);
        if (++s == ST) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit(tfull);
    }
    if (!ok) {
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kSwDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int col = quad * 32 + lane;  // this thread's TMEM lane: act / output column of the tile
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint32_t epi_ph = 0;
    auto epi_sync = [&](int site) -> bool {
      mbar_arrive(epi_bar);
      const bool got = mbar_wait(epi_bar, epi_ph, wc, site);
      epi_ph ^= 1u;
      return got;
    };
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      if (!mbar_wait(tfull, (uint32_t)it & 1u, wc, 115)) break;
      tc_fence_after();
      const int rb = tile / NJ, j = tile % NJ;
      const int rows = sw_rows(args, rb);
      const int64_t slot0 = (int64_t)rb * kBM;
      if (MODE == kSwUp) {
        uint8_t* act = static_cast<uint8_t*>(args.act) + j * 128 + col;
        uint8_t* act_sf = static_cast<uint8_t*>(args.act_sf) + sf_tile_offset(rb, j, args.H / 128) + quad;
#pragma unroll 1
        for (int r0 = 0; r0 < rows; r0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld_x32_pair(lane_base + r0, lane_base + 128 + r0, g, u);
          if (r0 + 32 >= rows) {  // the last chunk: the accumulators are free
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int r = r0 + i;
            if (r >= rows) continue;  // the same for the whole warp
            const float a = sw_swiglu(__uint_as_float(g[i]), __uint_as_float(u[i]), swiglu_lim);
            // ue8m0 exponent of the 32 act columns of this warp (the single-CTA
            // kernel's rule): the smallest e with amax * 2^-e <= 448
            const uint32_t bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(a)));
            int ex = 0;
            if (bits != 0) {
              const int p = (int)((bits >> 23) & 0xff) - 127;
              ex = max(p - 8 + ((bits & 0x7fffff) > 0x600000u ? 1 : 0), -127);
            }
            const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);
            act[(slot0 + r) * args.H] = (uint8_t)(cvt_e4m3x2(a * inv, 0.f) & 0xffu);
            if (lane == 0) act_sf[sf_in_tile(r)] = (uint8_t)(ex + 127);
          }
        }
        if (rows <= 0) {  // (no row block has zero rows; kept for the barrier count)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty);
        }
      } else {
        // DOWN: stage w * acc (bf16) of every routed row, then one bulk
        // reduction per row (thread r reduces row r)
        bool failed = false;
        bulk_wait_read_all();       // this thread's last reduction has left its staging row
        if (!epi_sync(116)) break;  // every staging row free
#pragma unroll 1
        for (int r0 = 0; r0 < rows; r0 += 32) {
          uint32_t v[32];
          tmem_ld_x32(lane_base + r0, v);
          if (r0 + 32 >= rows) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
          }
          const float wl = r0 + lane < rows ? args.slot_w[slot0 + r0 + lane] : 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float w = __shfl_sync(0xffffffffu, wl, i);
            if (r0 + i < rows) st_shared_b16(sStage + (r0 + i) * Cfg::kStageRow + col * 2, w * __uint_as_float(v[i]));
          }
        }
        if (rows <= 0) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty);
        }
        fence_proxy_async_smem();
        if (!epi_sync(117)) failed = true;
        if (failed) break;
        const int r = quad * 32 + lane;  // this thread's staged row
        if (r < rows) {
          const int tok = args.row_tok[slot0 + r];
          if (tok >= 0) {
            bulk_reduce_add_bf16_hint(static_cast<__nv_bfloat16*>(args.out) + (int64_t)tok * args.D + j * 128,
                                      sStage + r * Cfg::kStageRow, 256, args.out_hint != 0, l2_policy_evict_last());
            bulk_commit();
          }
        }
      }
    }
    if (MODE == kSwDown) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int MODE, int FP4W>
cudaError_t launch_sw(const CUtensorMap& w, const CUtensorMap& x, const MxSwapArgs& args, int grid,
                      cudaStream_t stream, bool pdl) {
  using Cfg = SwCfg<MODE>;
  auto kern = gemm_mx_swap_kernel<MODE, FP4W>;
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
  cfg.blockDim = dim3(kSwThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, w, x, args);
}

}  // namespace

cudaError_t launch_up_mx_swap(const CUtensorMap& map_w1, const CUtensorMap& map_xg, const MxSwapArgs& args, int grid,
                              cudaStream_t stream, bool fp4w) {
  return fp4w ? launch_sw<kSwUp, 1>(map_w1, map_xg, args, grid, stream, false)
              : launch_sw<kSwUp, 0>(map_w1, map_xg, args, grid, stream, false);
}
cudaError_t launch_down_mx_swap(const CUtensorMap& map_w2, const CUtensorMap& map_act, const MxSwapArgs& args,
                                int grid, cudaStream_t stream, bool pdl, bool fp4w) {
  return fp4w ? launch_sw<kSwDown, 1>(map_w2, map_act, args, grid, stream, pdl)
              : launch_sw<kSwDown, 0>(map_w2, map_act, args, grid, stream, pdl);
}

}  // namespace moe
