// gemm_mxfp8_pair.cu -- the MXFP8 split pipeline's GEMMs on CTA pairs
// (tcgen05 cta_group::2, kind::mxf8f6f4.block_scale): one MMA of M = 256 rows
// (two row blocks of one expert) by N = 256 columns by K = 32, issued by the
// even CTA of a two-CTA cluster.  Each CTA holds its own 128 rows of A and
// 128 of the 256 B rows in shared memory, so per K step of 128 a CTA brings
// in 32 KB of e4m3 data for the 128 x 256 output block that costs the
// single-CTA kernel 48 KB ("Prime Flash MoE" sec. 7 "The MXFP8 variant";
// Pearl "Optimizing Grouped GEMM for MoE on Blackwell": 2-CTA tiles).
//
// Scale factors, measured on GB300: in a pair MMA each CTA's tensor core
// reads the A scales of its own 128 rows and the B scales of all 256 columns
// from its OWN tensor memory, both in the single-CTA N = 256 layout (columns
// [0, 128) at the B scale address, [128, 256) four TMEM columns further), and
// a tcgen05.cp.cta_group::2 issued by the even CTA copies each CTA's own
// shared-memory tile into that CTA's own tensor memory.  So every CTA loads
// its A rows' scale tile and BOTH 128-row scale tiles of the B tile (1.5 KB a
// stage), and the even CTA issues three pair copies before the four MMAs.
//
// UP  (GEMM1 + SwiGLU + requantization): B = [W1 gate rows j*128 .. +128
//     (even CTA) | up rows H + j*128 .. +128 (odd CTA)]: each CTA's
//     accumulator holds gate in columns [0, 128) and up in [128, 256) of its
//     row block; act = silu(gate) * up is requantized per 32 to e4m3 + ue8m0
//     as in the single-CTA kernel.
// DOWN (GEMM2 + weighted reduce): B = W2[e] rows j*256 + 128 * rank .. +128;
//     the epilogue scales by the routing weight and reduces half rows into out.
// A half pair (an expert's odd last row block) runs both CTAs: the odd CTA
// loads the first block's rows again and stores nothing.
//
// The accumulator takes 256 of the 512 TMEM columns and the scale sets of the
// stages the rest (16 columns a stage), so it is single-buffered: eight
// epilogue warps per CTA (two per lane quadrant, one per column half) read it
// into registers and release it before they quantize or reduce.
// Synchronization as in the bf16 pair kernels: all loads of both CTAs complete
// on the even CTA's full[] barrier; MMA commits arrive on empty[] / tfull[] of
// both CTAs; the epilogue warps of both CTAs arrive on the even CTA's tempty.
// Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

enum { kMpUp = 0, kMpDown = 1 };
constexpr int kMpBK = 128;                 // e4m3 elements (bytes) per stage row
constexpr int kMpThreads = 64 + 256;       // producer warp, MMA warp, eight epilogue warps
constexpr uint64_t kMpDrainNs = 200ull * 1000 * 1000;
constexpr uint64_t kMpSettleNs = 2ull * 1000 * 1000;

template <int MODE>
struct MpCfg {
  static constexpr int kStages = MODE == kMpUp ? 6 : 4;
  static constexpr int kA = kBM * kMpBK;           // 16 KB: this CTA's 128 rows
  static constexpr int kB = 128 * kMpBK;           // 16 KB: this CTA's half of the 256 B rows
  static constexpr int kSF = 3 * 512;              // A scale tile + both B scale tiles
  static constexpr int kTx = kA + kB + kSF;        // bytes one CTA brings in per stage
  // DOWN: a 528-byte staging row per accumulator row (two 256-byte half rows,
  // one per epilogue warp of the quadrant, + 16 B: a warp's rows on distinct banks)
  static constexpr int kStageRow = 2 * 256 + 16;
  static constexpr int kStaging = MODE == kMpDown ? kBM * kStageRow : 0;
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmem = 1024 + kStages * (kA + kB + kSF) + kStaging + kBarrierBytes;
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(256 + 16 * kStages <= 512, "TMEM columns");
  static_assert((2 * kStages + 5) * 8 + 8 <= kBarrierBytes, "barrier area");
};

__device__ __forceinline__ float mp_u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ float mp_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// TMEM <- each CTA's own 512-byte scale tile (pair-wide copy, even CTA issues).
__device__ __forceinline__ void utccp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void umma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// map_a / map_b: e4m3 operands (boxes of 128 rows x 128 bytes); map_sfa /
// map_sfb: the blocked scale tiles seen as [tiles, 128] u32 (one 512-byte
// tile per box, tile index = row tile * K/128 + K tile).
template <int MODE>
__global__ void __launch_bounds__(kMpThreads, 1)
    gemm_mxfp8_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                           const __grid_constant__ CUtensorMap map_sfa, const __grid_constant__ CUtensorMap map_sfb,
                           const MxArgs args) {
  using Cfg = MpCfg<MODE>;
  constexpr int ST = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  // the same offset in both CTAs (same kernel, same dynamic shared memory base)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + ST * Cfg::kA;
  uint8_t* sSF = sB + ST * Cfg::kB;
  uint8_t* sStage = sSF + ST * Cfg::kSF;
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + Cfg::kStaging);
  uint64_t* empty = full + ST;
  uint64_t* tfull = empty + ST;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* never = drain + 1;  // no thread ever arrives here (failure-path test hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_slot = (int)blockIdx.x >> 1, n_pair_slots = (int)gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);   // even CTA: its producer's arrive + both CTAs' bytes
      mbar_init(&empty[s], 1);  // the pair MMA's commit
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 16);  // even CTA: the eight epilogue warps of each CTA
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
    prefetch_tmap(&map_sfa);
    prefetch_tmap(&map_sfb);
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
  // launched as a programmatic dependent (DOWN): everything below reads the
  // previous grid's outputs
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();

  const int NJ = args.n_col_tiles;
  const int n_tiles = args.meta[1] * NJ;  // (block pair, column tile)
  const int KB = args.k_blocks;           // K / 128
  auto tile_pair = [&](int i) {
    return args.pair_info[(MODE == kMpDown && args.pair_order) ? args.pair_order[i] : i];
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[ST];
#pragma unroll
    for (int i = 0; i < ST; ++i) issued_phase[i] = -1;
    bool ok = true;
    for (int tile = pair_slot; ok && tile < n_tiles; tile += n_pair_slots) {
      const int info = tile_pair(tile / NJ), j = tile % NJ;
      const int rb0 = info >> 1, two = info & 1;
      const int e = args.expert_of_rb[rb0];
      const int rb = rb0 + (int)(rank & (uint32_t)two);  // the odd CTA of a half pair reloads rb0
      // 128-row tiles of the weights: this CTA's B rows and the two B scale tiles
      int rt_mine, rt0, rt1;
      if (MODE == kMpUp) {
        rt0 = e * (2 * args.H / 128) + j;  // gate rows of column tile j
        rt1 = rt0 + args.H / 128;          // up rows
      } else {
        rt0 = e * (args.D / 128) + 2 * j;
        rt1 = rt0 + 1;
      }
      rt_mine = rank ? rt1 : rt0;
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&empty[s], ph ^ 1u, wc, 71))) break;
        if (leader) mbar_arrive_expect_tx(&full[s], 2 * Cfg::kTx);
        const uint32_t fb = mapa_shared(smem_addr(&full[s]), 0);
        uint8_t* sf = sSF + s * Cfg::kSF;
        tma_load_2d_pair(sA + s * Cfg::kA, &map_a, fb, kb * kMpBK, rb * kBM);
        tma_load_2d_pair(sB + s * Cfg::kB, &map_b, fb, kb * kMpBK, rt_mine * 128);
        tma_load_2d_pair(sf, &map_sfa, fb, 0, rb * KB + kb);
        tma_load_2d_pair(sf + 512, &map_sfb, fb, 0, rt0 * KB + kb);
        tma_load_2d_pair(sf + 1024, &map_sfb, fb, 0, rt1 * KB + kb);
        issued_phase[s] = (int)ph;
        if (++s == ST) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {  // let every copy already in flight land before the CTA exits
      if (leader) {
        for (int i = 0; i < ST; ++i)
          if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kMpDrainNs);
      } else {
        spin_ns(kMpSettleNs);  // this CTA's loads complete on the even CTA's barriers
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_mxf8(2 * kBM, 256);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 93);  // runs out after the wait limit
    int it = 0;
    for (int tile = pair_slot; ok && tile < n_tiles; tile += n_pair_slots, ++it) {
      if (!(ok = mbar_wait_cluster(tempty, ((uint32_t)it & 1u) ^ 1u, wc, 72))) break;
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb) {
        if (!(ok = mbar_wait(&full[s], ph, wc, 73))) break;
        tc_fence_after();
        // scale tiles of this stage -> the TMEM columns of this ring slot, in both CTAs
        const uint32_t sfa_col = tmem_base + 256 + 16 * s, sfb_col = sfa_col + 4;
        const uint32_t sf_smem = smem_addr(sSF + s * Cfg::kSF);
        utccp_sf_pair(sfa_col, sdesc_sf_tile(sf_smem));
        utccp_sf_pair(sfb_col, sdesc_sf_tile(sf_smem + 512));
        utccp_sf_pair(sfb_col + 4, sdesc_sf_tile(sf_smem + 1024));
        const uint64_t ad = sdesc_sw128(smem_addr(sA + s * Cfg::kA));
        const uint64_t bd = sdesc_sw128(smem_addr(sB + s * Cfg::kB));
#pragma unroll
        for (int kk = 0; kk < kMpBK / 32; ++kk)
          umma_mxf8_pair(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc_with_sf_id(idesc, kk), sfa_col, sfb_col,
                         (kb | kk) != 0);
        umma_commit_pair(&empty[s], 0x3);  // frees this stage in both CTAs
        if (++s == ST) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit_pair(tfull, 0x3);  // both CTAs' accumulators ready
    }
    if (!ok) {  // wait for every MMA already issued before tensor memory is released
      umma_commit_pair(drain, 0x1);
      mbar_wait_drain(drain, 0, kMpDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;             // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;      // which half of the accumulator columns
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_stage = sStage + row * Cfg::kStageRow + half * 256;
    const uint32_t tempty_leader = mapa_shared(smem_addr(tempty), 0);
    int it = 0;
    for (int tile = pair_slot; tile < n_tiles; tile += n_pair_slots, ++it) {
      if (!mbar_wait(tfull, (uint32_t)it & 1u, wc, 74)) break;
      tc_fence_after();
      const int info = tile_pair(tile / NJ), j = tile % NJ;
      const int rb = (info >> 1) + (int)rank;
      const int64_t slot = (int64_t)rb * kBM + row;
      const int tok = (rank == 0 || (info & 1)) ? args.row_tok[slot] : -1;
      if (MODE == kMpUp) {
        // columns [64 half, 64 half + 64) of gate (0..127) and of up (128..255)
        float act[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t g[32], u[32];
          const int col = half * 64 + c * 32;
          tmem_ld_x32_pair(lane_base + col, lane_base + 128 + col, g, u);
#pragma unroll
          for (int i = 0; i < 32; ++i) act[c * 32 + i] = mp_swiglu(mp_u2f(g[i]), mp_u2f(u[i]), swiglu_lim);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader);  // this warp has read the accumulator
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
      } else {
        // this warp's half row: 128 columns into registers, the accumulator
        // released, then staged and reduced while the next tile's MMAs run
        const float w = tok >= 0 ? args.slot_w[slot] : 0.f;
        uint32_t v[4][32];
        const uint32_t tcol = lane_base + half * 128;
        tmem_ld_x32_pair(tcol, tcol + 32, v[0], v[1]);
        tmem_ld_x32_pair(tcol + 64, tcol + 96, v[2], v[3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader);
        if (tok >= 0) {
          if (args.out_f32) {
            float* frow = args.out_f32 + (int64_t)tok * args.D + j * 256 + half * 128;
#pragma unroll
            for (int c = 0; c < 4; c += 2) {
              bulk_wait_read_all();  // the previous reduction has left the staging half row
              stage_scaled_f32x32(my_stage, w, v[c]);
              stage_scaled_f32x32(my_stage + 128, w, v[c + 1]);
              fence_proxy_async_smem();
              bulk_reduce_add_f32(frow + c * 32, my_stage, 256);
              bulk_commit();
            }
          } else {
            bulk_wait_read_all();  // the previous tile's reduction has left the staging half row
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int q = 0; q < 4; ++q)
                st_shared_v4(my_stage + c * 64 + q * 16,
                             pack_bf16x2(w * mp_u2f(v[c][8 * q + 0]), w * mp_u2f(v[c][8 * q + 1])),
                             pack_bf16x2(w * mp_u2f(v[c][8 * q + 2]), w * mp_u2f(v[c][8 * q + 3])),
                             pack_bf16x2(w * mp_u2f(v[c][8 * q + 4]), w * mp_u2f(v[c][8 * q + 5])),
                             pack_bf16x2(w * mp_u2f(v[c][8 * q + 6]), w * mp_u2f(v[c][8 * q + 7])));
            fence_proxy_async_smem();
            bulk_reduce_add_bf16_hint(static_cast<__nv_bfloat16*>(args.out) + (int64_t)tok * args.D + j * 256 +
                                          half * 128,
                                      my_stage, 256, args.out_hint != 0, l2_policy_evict_last());
            bulk_commit();
          }
        }
      }
    }
    if (MODE == kMpDown) bulk_wait_all();  // reductions complete before the CTA exits
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

template <int MODE>
cudaError_t set_smem_once() {
  // once per device: not a stream operation, so it stays out of graph capture
  static bool smem_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    cudaError_t err = cudaFuncSetAttribute(gemm_mxfp8_pair_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           MpCfg<MODE>::kSmem);
    if (err != cudaSuccess) return err;
    smem_set[dev] = true;
  }
  return cudaSuccess;
}

template <int MODE>
cudaError_t launch_mp(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa, const CUtensorMap& sfb,
                      const MxArgs& args, int n_pairs, cudaStream_t stream, bool pdl) {
  cudaError_t err = set_smem_once<MODE>();
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n_pairs);
  cfg.blockDim = dim3(kMpThreads);
  cfg.dynamicSmemBytes = MpCfg<MODE>::kSmem;
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
  return cudaLaunchKernelEx(&cfg, gemm_mxfp8_pair_kernel<MODE>, a, b, sfa, sfb, args);
}

}  // namespace

int mx_pair_cluster_slots() {
  // once per device: not a stream operation
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev]) return cache[dev];
  // the larger of the two kernels' shared memory decides the residency
  constexpr int kMode = MpCfg<kMpUp>::kSmem >= MpCfg<kMpDown>::kSmem ? kMpUp : kMpDown;
  if (set_smem_once<kMode>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kMpThreads);
  cfg.dynamicSmemBytes = MpCfg<kMode>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_mxfp8_pair_kernel<kMode>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cache[dev] = n;
  return n;
}

cudaError_t launch_up_mxfp8_pair(const CUtensorMap& a, const CUtensorMap& w1, const CUtensorMap& sfa,
                                 const CUtensorMap& sfb, const MxArgs& args, int n_pairs, cudaStream_t stream) {
  return launch_mp<kMpUp>(a, w1, sfa, sfb, args, n_pairs, stream, false);
}
cudaError_t launch_down_mxfp8_pair(const CUtensorMap& act, const CUtensorMap& w2, const CUtensorMap& sfa,
                                   const CUtensorMap& sfb, const MxArgs& args, int n_pairs, cudaStream_t stream,
                                   bool pdl) {
  return launch_mp<kMpDown>(act, w2, sfa, sfb, args, n_pairs, stream, pdl);
}

}  // namespace moe
