// gemm_fused_cluster_mx.cu -- the MXFP8 fused pipeline on thread-block
// clusters: the structure of the bf16 cluster kernel (a cluster of C CTAs owns
// one 128-row block at a time, CTA c computes act columns [c*h, (c+1)*h) and
// output columns [c*dsl, (c+1)*dsl), act meets in a per-cluster L2-resident
// ring) with block-scaled MMAs ("Prime Flash MoE" sec. 7 "The MXFP8 variant":
// e4m3 data, one ue8m0 scale per 32 along K, tcgen05.mma kind::mxf8f6f4
// block_scale with the scales copied into tensor memory by tcgen05.cp).
//
//   GEMM1 (sub-chunk s of 128 act columns): acc1[128 x 256] = (xg * s_x) .
//          ([W1 gate rows | up rows] * s_w1)^T, K = D in stages of 128.
//   SwiGLU in fp32, requantized per 32 columns to e4m3 + ue8m0 (sec. 7 "The
//          epilogue also quantizes"): codes into the ring's [128 x H] e4m3
//          buffer, the four scale bytes of each row into the ring's blocked
//          512-byte scale tile of that 128-column K tile.
//   GEMM2 (sub-chunk s of 256 output columns): acc[128 x 256] = (act * s_act)
//          . (W2[e][rows] * s_w2)^T, K = H, once every act slice is in the ring.
//   Reduction: w * acc in fp32 -> bf16 -> bulk .add.bf16 into out, as in the
//          split pipeline's down projection.
// TMEM: one accumulator at columns [0, 256) for every job, the scale tiles of
// ring slot s at 256 + 16 s (A: 4 columns, B: 8), so in-flight stages never
// share scale columns (sec. 7: the MXFP8 loop is serialized).  Two 256-column
// accumulators would leave no columns for the scales, and a narrower GEMM2
// needs more operand bytes per FLOP than the kernel can stream; instead eight
// epilogue warps (two per TMEM lane quadrant, one per column half) read the
// accumulator and release it before they quantize or reduce, so the next job
// waits only for the tensor-memory reads.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kMThreads = 64 + 256;          // producer warp, MMA warp, 8 epilogue warps
constexpr int kMEpi = 256;
constexpr int kMStages = 3;
constexpr int kMBK = 128;                      // e4m3 bytes per K stage
constexpr int kMA = kBM * kMBK;                // 16 KB: xg or act tile
constexpr int kMB = 256 * kMBK;                // 32 KB: W1 or W2 tile of 256 rows
constexpr int kMSF = 3 * 512;                  // A scale tile + two B scale tiles
constexpr int kMN2 = 256;                      // GEMM2 output columns per sub-chunk
constexpr int kMStageCols = 128;               // reduction staging: an epilogue thread's half row
constexpr int kMStageRow = kMStageCols * 2 + 16;
constexpr int kMStaging = kMEpi * kMStageRow;
constexpr int kMBarrierBytes = 256;
constexpr int kMSmem = kMStages * (kMA + kMB + kMSF) + kMStaging + kMBarrierBytes;
static_assert(kMSmem <= 232448, "shared memory");
static_assert((2 * kMStages + 8) * 8 + 8 <= kMBarrierBytes, "barrier area");
constexpr uint32_t kMSfCol = 256;
static_assert(kMSfCol + 16 * kMStages <= 512, "TMEM columns");
constexpr uint64_t kMDrainNs = 200ull * 1000 * 1000;

__device__ __forceinline__ float m_u2f(uint32_t u) { return __uint_as_float(u); }
// silu(g) * u with the optional clamp (lim = +inf when off): g <= lim,
// -lim <= u <= lim.
__device__ __forceinline__ float m_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Rounds as in the bf16 cluster kernel: round r interleaves the GEMM1 jobs of
// row block r with the GEMM2 jobs of row block r - 1.
__device__ __forceinline__ int mx_round_jobs(int r, int n, int s1, int s2) {
  return (r < n ? s1 : 0) + (r >= 1 ? s2 : 0);
}
__device__ __forceinline__ bool mx_cluster_job(int r, int j, int n, int s1, int s2, int* it, int* sub) {
  const int n1 = r < n ? s1 : 0, n2 = r >= 1 ? s2 : 0;
  const int m = min(n1, n2);
  bool g2;
  if (j < 2 * m) {
    g2 = (j & 1) != 0;
    *sub = j >> 1;
  } else {
    g2 = n2 > n1;
    *sub = m + (j - 2 * m);
  }
  *it = g2 ? r - 1 : r;
  return g2;
}

__global__ void __launch_bounds__(kMThreads, 1)
    fused_cluster_mxfp8_kernel(const __grid_constant__ CUtensorMap map_xg, const __grid_constant__ CUtensorMap map_w1,
                               const __grid_constant__ CUtensorMap map_w2, const __grid_constant__ CUtensorMap map_ring,
                               const FusedClusterMxArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_addr(smem_raw) & 1023u) {  // the same in every CTA: all of them return here
    if (threadIdx.x == 0) atomicOr(args.err, kErrLaunch);
    return;
  }
  uint8_t* sA = smem_raw;                      // SW128 tiles first: 1024-byte aligned
  uint8_t* sB = sA + kMStages * kMA;
  uint8_t* sSF = sB + kMStages * kMB;
  uint8_t* staging = sSF + kMStages * kMSF;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + kMStaging);
  uint64_t* empty = full + kMStages;
  uint64_t* tfull = empty + kMStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* ready = tempty + 1;    // [2] all act slices of ring buffer b written (8 warps x s1 x C CTAs)
  uint64_t* freeb = ready + 2;     // [2] ring buffer b loaded by every CTA (C arrivals)
  uint64_t* drain = freeb + 2;
  uint64_t* never = drain + 1;     // no thread ever arrives here (failure-path test hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};
  const int C = args.csize;
  const int crank = (int)blockIdx.x % C, cid = (int)blockIdx.x / C, ncl = (int)gridDim.x / C;
  const int s1 = args.s1, s2 = args.s2;
  const int h = 128 * s1;                      // act columns of this CTA
  const int dsl = kMN2 * s2;                   // output columns of this CTA
  const int KT_H = args.H / 128;               // K tiles of GEMM2 (and scale tiles per ring row block)
  const int KT_D = args.D / 128;               // K tiles of GEMM1

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kMEpi);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ready[b], 8 * C * s1);
      mbar_init(&freeb[b], C);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_xg);
    prefetch_tmap(&map_w1);
    prefetch_tmap(&map_w2);
    prefetch_tmap(&map_ring);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive
  const uint32_t tmem_base = *tmem_slot;

  const int num_rb = args.meta[0];
  const int n_it = cid < num_rb ? (num_rb - cid + ncl - 1) / ncl : 0;
  const int n_rounds = n_it > 0 ? n_it + 1 : 0;
  const uint8_t* xg_sf = static_cast<const uint8_t*>(args.xg_sf);
  const uint8_t* w1_sf = static_cast<const uint8_t*>(args.w1_sf);
  const uint8_t* w2_sf = static_cast<const uint8_t*>(args.w2_sf);
  uint8_t* ring_sf = static_cast<uint8_t*>(args.ring_sf);

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[kMStages];
#pragma unroll
    for (int i = 0; i < kMStages; ++i) issued_phase[i] = -1;
    bool ok = true;
    for (int r = 0; ok && r < n_rounds; ++r) {
      const int nj = mx_round_jobs(r, n_it, s1, s2);
      for (int j = 0; ok && j < nj; ++j) {
        int it, sub;
        const bool g2 = mx_cluster_job(r, j, n_it, s1, s2, &it, &sub);
        const int rb = cid + it * ncl;
        const int e = args.expert_of_rb[rb];
        const int b = it & 1;
        if (g2) {  // every CTA of the cluster has written its act slices of this row block
          if (!(ok = mbar_wait_cluster(&ready[b], (uint32_t)(it >> 1) & 1u, wc, 51))) break;
          fence_proxy_async_global();
        }
        // 128-row tiles of W1 [E*2H, D] and of W2 [E*D, H]
        const int rt_gate = e * (2 * KT_H) + (crank * h) / 128 + sub;
        const int rt_up = rt_gate + KT_H;
        const int rt2 = e * KT_D + (crank * dsl + sub * kMN2) / 128;
        const int KB = g2 ? KT_H : KT_D;
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = mbar_wait(&empty[s], ph ^ 1u, wc, 52))) break;
          uint8_t* a = sA + s * kMA;
          uint8_t* bt = sB + s * kMB;
          uint8_t* sf = sSF + s * kMSF;
          if (!g2) {
            mbar_arrive_expect_tx(&full[s], kMA + kMB + 3 * 512);
            tma_load_2d(a, &map_xg, &full[s], kb * kMBK, rb * kBM);
            tma_load_2d(bt, &map_w1, &full[s], kb * kMBK, rt_gate * 128);
            tma_load_2d(bt + 128 * kMBK, &map_w1, &full[s], kb * kMBK, rt_up * 128);
            bulk_load(sf, xg_sf + sf_tile_offset(rb, kb, KT_D), 512, &full[s]);
            bulk_load(sf + 512, w1_sf + sf_tile_offset(rt_gate, kb, KT_D), 512, &full[s]);
            bulk_load(sf + 1024, w1_sf + sf_tile_offset(rt_up, kb, KT_D), 512, &full[s]);
          } else {
            mbar_arrive_expect_tx(&full[s], kMA + kMB + 3 * 512);
            tma_load_2d(a, &map_ring, &full[s], kb * kMBK, (cid * 2 + b) * kBM);
            bulk_load(sf, ring_sf + sf_tile_offset(cid * 2 + b, kb, KT_H), 512, &full[s]);
            tma_load_2d(bt, &map_w2, &full[s], kb * kMBK, rt2 * 128);
            bulk_load(sf + 512, w2_sf + sf_tile_offset(rt2, kb, KT_H), 512, &full[s]);
            bulk_load(sf + 1024, w2_sf + sf_tile_offset(rt2 + 1, kb, KT_H), 512, &full[s]);
          }
          issued_phase[s] = (int)ph;
          if (++s == kMStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (!ok) {  // let every copy already in flight land before the CTA exits
      for (int i = 0; i < kMStages; ++i)
        if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kMDrainNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_mxf8(kBM, 256);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 96);  // runs out after the wait limit
    int nq = 0;  // jobs issued: each owns the accumulator until the epilogue has read it
    for (int r = 0; ok && r < n_rounds; ++r) {
      const int nj = mx_round_jobs(r, n_it, s1, s2);
      for (int j = 0; ok && j < nj; ++j) {
        int it, sub;
        const bool g2 = mx_cluster_job(r, j, n_it, s1, s2, &it, &sub);
        if (!(ok = mbar_wait(tempty, ((uint32_t)nq & 1u) ^ 1u, wc, 53))) break;
        tc_fence_after();
        const int KB = g2 ? KT_H : KT_D;
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = mbar_wait(&full[s], ph, wc, 54))) break;
          tc_fence_after();
          // scale tiles of this stage -> TMEM columns reserved for this ring slot
          const uint32_t sfa_col = tmem_base + kMSfCol + 16 * s, sfb_col = sfa_col + 4;
          const uint32_t sf_smem = smem_addr(sSF + s * kMSF);
          utccp_sf(sfa_col, sdesc_sf_tile(sf_smem));
          utccp_sf(sfb_col, sdesc_sf_tile(sf_smem + 512));
          utccp_sf(sfb_col + 4, sdesc_sf_tile(sf_smem + 1024));
          const uint64_t ad = sdesc_sw128(smem_addr(sA + s * kMA));
          const uint64_t bd = sdesc_sw128(smem_addr(sB + s * kMB));
#pragma unroll
          for (int kk = 0; kk < kMBK / 32; ++kk)
            umma_mxf8(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc_with_sf_id(idesc, kk), sfa_col, sfb_col,
                      (kb | kk) != 0);
          umma_commit(&empty[s]);
          if (++s == kMStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (g2 && sub == s2 - 1) {
          // every act tile of this row block has landed in shared memory: the
          // cluster may rewrite ring buffer it & 1
          const uint32_t fa = smem_addr(&freeb[it & 1]);
          for (int q = 0; q < C; ++q) mbar_arrive_cluster(mapa_shared(fa, (uint32_t)q));
        }
        ++nq;
        umma_commit(tfull);  // accumulator ready for the epilogue
      }
    }
    if (!ok) {  // wait for every MMA already issued before TMEM is released
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kMDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogues
    const int quad = warp & 3;             // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;      // which half of the accumulator's columns
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_stage = staging + (half * kBM + row) * kMStageRow;
    uint8_t* ring = static_cast<uint8_t*>(args.ring);
    int nq = 0;
    bool ok = true;
    for (int r = 0, j = 0; ok && r < n_rounds;) {
      if (j == mx_round_jobs(r, n_it, s1, s2)) {  // next round (a round has at least one job)
        ++r;
        j = 0;
        if (r == n_rounds) break;
      }
      int it, sub;
      const bool g2 = mx_cluster_job(r, j++, n_it, s1, s2, &it, &sub);
      const int rb = cid + it * ncl;
      const int64_t slot = (int64_t)rb * kBM + row;
      const int tok = args.row_tok[slot];
      const int b = it & 1;
      if (!(ok = mbar_wait(tfull, (uint32_t)nq & 1u, wc, 55))) break;
      tc_fence_after();
      ++nq;
      if (!g2) {
        // SwiGLU of act columns [64 half, 64 half + 64) of the sub-chunk: gate
        // at accumulator columns 64 half .., up at 128 + 64 half ..
        float a[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t g[32], u[32];
          const int col = half * 64 + c * 32;
          tmem_ld_x32_pair(lane_base + col, lane_base + 128 + col, g, u);
#pragma unroll
          for (int i = 0; i < 32; ++i) a[c * 32 + i] = m_swiglu(m_u2f(g[i]), m_u2f(u[i]), swiglu_lim);
        }
        tc_fence_before();
        mbar_arrive(tempty);  // the accumulator is free once all 256 threads have read it
        // ring buffer b was loaded by every CTA for row block it - 2
        if (it >= 2 && !(ok = mbar_wait_cluster(&freeb[b], ((uint32_t)(it >> 1) & 1u) ^ 1u, wc, 56))) break;
        const int col0 = crank * h + sub * 128;  // first act column of this sub-chunk (K tile col0 / 128)
        if (tok >= 0) {  // padding rows: their GEMM2 rows are dropped
          uint8_t* dst = ring + ((int64_t)(cid * 2 + b) * kBM + row) * args.H + col0 + half * 64;
          uint32_t sfw = 0;
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            uint32_t q[8];
            sfw |= mx_quantize32(a + blk * 32, q) << (8 * blk);
            st_global_v4(dst + blk * 32, q[0], q[1], q[2], q[3]);
            st_global_v4(dst + blk * 32 + 16, q[4], q[5], q[6], q[7]);
          }
          *reinterpret_cast<uint16_t*>(ring_sf + sf_tile_offset(cid * 2 + b, col0 / 128, KT_H) + sf_in_tile(row) +
                                       half * 2) = (uint16_t)sfw;
        }
        // publish this warp's act rows to every CTA of the cluster
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) {
          const uint32_t ra = smem_addr(&ready[b]);
          for (int q = 0; q < C; ++q) mbar_arrive_cluster(mapa_shared(ra, (uint32_t)q));
        }
      } else {
        // weighted reduction of output columns [128 half, 128 half + 128)
        const float w = args.slot_w[slot];
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tok < 0 ? 0 : tok) * args.D +
                              crank * dsl + sub * kMN2 + half * kMStageCols;
        uint32_t v[4][32];
        tmem_ld_x32_pair(lane_base + half * 128, lane_base + half * 128 + 32, v[0], v[1]);
        tmem_ld_x32_pair(lane_base + half * 128 + 64, lane_base + half * 128 + 96, v[2], v[3]);
        tc_fence_before();
        mbar_arrive(tempty);  // the accumulator is free once all 256 threads have read it
        if (tok >= 0) {
          bulk_wait_read_all();  // the previous reduction has left the staging row
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int qd = 0; qd < 4; ++qd)
              st_shared_v4(my_stage + c * 64 + qd * 16, pack_bf16x2(w * m_u2f(v[c][8 * qd]), w * m_u2f(v[c][8 * qd + 1])),
                           pack_bf16x2(w * m_u2f(v[c][8 * qd + 2]), w * m_u2f(v[c][8 * qd + 3])),
                           pack_bf16x2(w * m_u2f(v[c][8 * qd + 4]), w * m_u2f(v[c][8 * qd + 5])),
                           pack_bf16x2(w * m_u2f(v[c][8 * qd + 6]), w * m_u2f(v[c][8 * qd + 7])));
          }
          fence_proxy_async_smem();
          bulk_reduce_add_bf16_hint(orow, my_stage, kMStageCols * 2, args.out_hint != 0, l2_policy_evict_last());
          bulk_commit();
        }
      }
    }
    bulk_wait_all();  // bulk reductions complete before the CTA exits
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while another may still arrive on its barriers
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

cudaError_t mx_set_smem_once() {
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(fused_cluster_mxfp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMSmem);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

int fused_cluster_mx_max_clusters(int csize) {
  // once per (device, cluster size): not a stream operation
  static int cache[64][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int slot = csize == 1 ? 0 : csize == 2 ? 1 : csize == 4 ? 2 : csize == 8 ? 3 : -1;
  if (slot < 0) return 0;
  if (cache[dev][slot]) return cache[dev][slot];
  if (mx_set_smem_once() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize);
  cfg.blockDim = dim3(kMThreads);
  cfg.dynamicSmemBytes = kMSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fused_cluster_mxfp8_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cache[dev][slot] = n;
  return n;
}

cudaError_t launch_fused_cluster_mxfp8(const CUtensorMap& map_xg, const CUtensorMap& map_w1,
                                       const CUtensorMap& map_w2, const CUtensorMap& map_ring,
                                       const FusedClusterMxArgs& args, int n_clusters, cudaStream_t stream) {
  cudaError_t e = mx_set_smem_once();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_clusters * args.csize);
  cfg.blockDim = dim3(kMThreads);
  cfg.dynamicSmemBytes = kMSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = args.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_cluster_mxfp8_kernel, map_xg, map_w1, map_w2, map_ring, args);
}

}  // namespace moe
