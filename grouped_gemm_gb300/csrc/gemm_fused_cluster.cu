// gemm_fused_cluster.cu -- the fused pipeline on thread-block clusters: one
// launch computes out += w * W2 . SwiGLU(W1 . x) for every routed row, and the
// activation never exists as an [S x H] tensor.
//
// A cluster of C CTAs owns one 128-row block rb (expert e) at a time ("Prime
// Flash MoE" sec. 2 "Trick 2: Cut the intermediate": the intermediate
// dimension is split over CTAs; here the split stays inside a cluster, so the
// down projection needs no split-K sum over CTAs).  CTA c owns act columns
// [c*h, (c+1)*h), h = H / C, in s1 sub-chunks of h1 (2*h1 <= 256), and output
// columns [c*dsl, (c+1)*dsl), dsl = D / C, in s2 sub-chunks of 256:
//   GEMM1 (sub-chunk s): acc1[128 x 2*h1] = xg[rb] . [W1 gate rows c*h + s*h1
//          .. +h1 | the matching up rows]^T, K = D.
//   SwiGLU epilogue: act[:, c*h + s*h1 .. +h1] = silu(gate) * up (fp32) -> bf16
//          into a per-cluster ring buffer of 128 x H bf16 (two buffers per
//          cluster, a few MB for the whole grid, so they stay in L2), then an
//          arrive on the "ready" barrier of every CTA of the cluster.
//   GEMM2 (sub-chunk s): acc2[128 x 256] = act[rb, all H] . W2[e][c*dsl + s*256
//          .. +256, :]^T once all slices of act are in the ring (TMA loads
//          from L2).
//   Reduction epilogue: rows scaled by their routing weight in fp32, rounded to
//          bf16 and added into out[row_tok, ..] with one bulk .add.bf16
//          reduction per half row (sec. 5 "Three jobs - one instruction"),
//          exactly as the split pipeline's down projection.
// Jobs run in rounds: round r interleaves the GEMM1 jobs of row block r with
// the GEMM2 jobs of row block r - 1 (G1, G2, G1, G2, ...), so the MMAs of one
// GEMM cover the other's epilogue, and the cluster-wide exchange of a row
// block's act is covered by a whole round.  acc1 lives at TMEM columns
// [0, 2*h1), acc2 at [256, 512).  One TMA ring of 48 KB stages serves both
// GEMMs (sec. 4 "One ring, both GEMMs").  Smaller clusters with more
// sub-chunks per CTA occupy more SMs (clusters must fit in a GPC) at the same
// bytes per FLOP.
// Ring buffer b = it & 1 is rewritten for row block it + 2 only after every CTA
// of the cluster has loaded it for GEMM2 (the "free" barriers).
// Every wait is bounded; every CTA reaches the final cluster barrier, so no CTA
// exits while another may still arrive on its barriers.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kCThreads = 192;
constexpr int kCEpi = 128;
constexpr int kCStages = 4;
constexpr int kCA = kBM * kBK * 2;            // 16 KB: xg or act tile
constexpr int kCB = 256 * kBK * 2;            // 32 KB: W1 (2h <= 256 rows) or W2 (256 rows) tile
constexpr int kCStage = kCA + kCB;
constexpr int kCStageRow = kFusedClusterN + 16;  // staging row: half of 256 bf16 + 16 B (distinct banks)
constexpr int kCStaging = kBM * kCStageRow;
constexpr int kCBarrierBytes = 256;
constexpr int kCSmem = kCStages * kCStage + kCStaging + kCBarrierBytes;
static_assert(kCSmem <= 232448, "shared memory");
static_assert((2 * kCStages + 10) * 8 + 8 <= kCBarrierBytes, "barrier area");
constexpr uint32_t kAcc2Col = 256;
constexpr uint64_t kCDrainNs = 200ull * 1000 * 1000;

__device__ __forceinline__ float c_u2f(uint32_t u) { return __uint_as_float(u); }
// silu(g) * u with the optional clamp (lim = +inf when off): g <= lim,
// -lim <= u <= lim.
__device__ __forceinline__ float c_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Job j of round r (row blocks 0 .. n-1; r in 0 .. n): GEMM1 sub-chunks of row
// block r and GEMM2 sub-chunks of row block r - 1, alternating while both
// remain.  Returns true for GEMM2; *it = row block, *sub = sub-chunk.
__device__ __forceinline__ int round_jobs(int r, int n, int s1, int s2) {
  return (r < n ? s1 : 0) + (r >= 1 ? s2 : 0);
}
__device__ __forceinline__ bool cluster_job(int r, int j, int n, int s1, int s2, int* it, int* sub) {
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

__global__ void __launch_bounds__(kCThreads, 1)
    fused_cluster_bf16_kernel(const __grid_constant__ CUtensorMap map_xg, const __grid_constant__ CUtensorMap map_w1,
                              const __grid_constant__ CUtensorMap map_w2, const __grid_constant__ CUtensorMap map_ring,
                              const FusedClusterArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_addr(smem_raw) & 1023u) {  // the same in every CTA: all of them return here
    if (threadIdx.x == 0) atomicOr(args.err, kErrLaunch);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* staging = smem + kCStages * kCStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + kCStaging);
  uint64_t* empty = full + kCStages;
  uint64_t* tfull1 = empty + kCStages;
  uint64_t* tempty1 = tfull1 + 1;
  uint64_t* tfull2 = tempty1 + 1;
  uint64_t* tempty2 = tfull2 + 1;
  uint64_t* ready = tempty2 + 1;   // [2] all act slices of ring buffer b written (4 warps x s1 x C CTAs)
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
  const int h1 = args.h1, s1 = args.s1, s2 = args.s2;
  const int h = h1 * s1;                    // act columns of this CTA
  const int dsl = kFusedClusterN * s2;      // output columns of this CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < kCStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull1, 1);
    mbar_init(tempty1, kCEpi);
    mbar_init(tfull2, 1);
    mbar_init(tempty2, kCEpi);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ready[b], 4 * C * s1);
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
  griddep_wait();

  const int num_rb = args.meta[0];
  const int n_it = cid < num_rb ? (num_rb - cid + ncl - 1) / ncl : 0;
  const int n_rounds = n_it > 0 ? n_it + 1 : 0;
  const int KB1 = args.D / kBK, KB2 = args.H / kBK;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[kCStages];
#pragma unroll
    for (int i = 0; i < kCStages; ++i) issued_phase[i] = -1;
    bool ok = true;
    for (int r = 0; ok && r < n_rounds; ++r) {
      const int nj = round_jobs(r, n_it, s1, s2);
      for (int j = 0; ok && j < nj; ++j) {
        int it, sub;
        const bool g2 = cluster_job(r, j, n_it, s1, s2, &it, &sub);
        const int rb = cid + it * ncl;
        const int e = args.expert_of_rb[rb];
        const int b = it & 1;
        if (g2) {  // every CTA of the cluster has written its act slices of this row block
          if (!(ok = mbar_wait_cluster(&ready[b], (uint32_t)(it >> 1) & 1u, wc, 41))) break;
          fence_proxy_async_global();
        }
        const int KB = g2 ? KB2 : KB1;
        const int w1_row = e * 2 * args.H + crank * h + sub * h1;
        const int w2_row = e * args.D + crank * dsl + sub * kFusedClusterN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = mbar_wait(&empty[s], ph ^ 1u, wc, 42))) break;
          uint8_t* st = smem + s * kCStage;
          if (!g2) {
            mbar_arrive_expect_tx(&full[s], kCA + 2 * h1 * kBK * 2);
            tma_load_2d(st, &map_xg, &full[s], kb * kBK, rb * kBM);
            tma_load_2d(st + kCA, &map_w1, &full[s], kb * kBK, w1_row);
            tma_load_2d(st + kCA + h1 * kBK * 2, &map_w1, &full[s], kb * kBK, w1_row + args.H);
          } else {
            mbar_arrive_expect_tx(&full[s], kCA + kCB);
            tma_load_2d(st, &map_ring, &full[s], kb * kBK, (cid * 2 + b) * kBM);
            tma_load_2d(st + kCA, &map_w2, &full[s], kb * kBK, w2_row);
          }
          issued_phase[s] = (int)ph;
          if (++s == kCStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (!ok) {  // let every copy already in flight land before the CTA exits
      for (int i = 0; i < kCStages; ++i)
        if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kCDrainNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc1 = idesc_bf16_f32(kBM, 2 * h1);
    constexpr uint32_t idesc2 = idesc_bf16_f32(kBM, kFusedClusterN);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 95);  // runs out after the wait limit
    int n1 = 0, n2 = 0;
    for (int r = 0; ok && r < n_rounds; ++r) {
      const int nj = round_jobs(r, n_it, s1, s2);
      for (int j = 0; ok && j < nj; ++j) {
        int it, sub;
        const bool g2 = cluster_job(r, j, n_it, s1, s2, &it, &sub);
        const int cnt = g2 ? n2 : n1;
        if (!(ok = mbar_wait(g2 ? tempty2 : tempty1, ((uint32_t)cnt & 1u) ^ 1u, wc, 43))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (g2 ? kAcc2Col : 0u);
        const uint32_t idesc = g2 ? idesc2 : idesc1;
        const int KB = g2 ? KB2 : KB1;
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = mbar_wait(&full[s], ph, wc, 44))) break;
          tc_fence_after();
          const uint64_t adesc = sdesc_sw128(smem_addr(smem + s * kCStage));
          const uint64_t bdesc = sdesc_sw128(smem_addr(smem + s * kCStage + kCA));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
          umma_commit(&empty[s]);
          if (++s == kCStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (g2) {
          if (sub == s2 - 1) {
            // every act tile of this row block has landed in shared memory:
            // the cluster may rewrite ring buffer it & 1
            const uint32_t fa = smem_addr(&freeb[it & 1]);
            for (int q = 0; q < C; ++q) mbar_arrive_cluster(mapa_shared(fa, (uint32_t)q));
          }
          ++n2;
        } else {
          ++n1;
        }
        umma_commit(g2 ? tfull2 : tfull1);  // accumulator ready for the epilogue
      }
    }
    if (!ok) {  // wait for every MMA already issued before TMEM is released
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kCDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogues
    const int quad = warp & 3;  // TMEM lanes this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_stage = staging + row * kCStageRow;
    __nv_bfloat16* ring = static_cast<__nv_bfloat16*>(args.ring);
    int n1 = 0, n2 = 0;
    bool ok = true;
    for (int r = 0, j = 0; ok && r < n_rounds;) {
      if (j == round_jobs(r, n_it, s1, s2)) {  // next round (a round has at least one job)
        ++r;
        j = 0;
        if (r == n_rounds) break;
      }
      int it, sub;
      const bool g2 = cluster_job(r, j++, n_it, s1, s2, &it, &sub);
      const int rb = cid + it * ncl;
      const int64_t slot = (int64_t)rb * kBM + row;
      const int tok = args.row_tok[slot];
      const int b = it & 1;
      if (!g2) {
        // SwiGLU: gate in columns [0, h1), up in [h1, 2*h1) of this thread's lane
        if (!(ok = mbar_wait(tfull1, (uint32_t)n1 & 1u, wc, 45))) break;
        tc_fence_after();
        // ring buffer b was loaded by every CTA for row block it - 2
        if (it >= 2 && !(ok = mbar_wait_cluster(&freeb[b], ((uint32_t)(it >> 1) & 1u) ^ 1u, wc, 46))) break;
        __nv_bfloat16* dst = ring + ((int64_t)(cid * 2 + b) * kBM + row) * args.H + crank * h + sub * h1;
#pragma unroll 1
        for (int c = 0; c < h1; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld_x32_pair(lane_base + c, lane_base + h1 + c, g, u);
          if (tok >= 0) {  // padding rows: their GEMM2 rows are dropped, the ring row is not read for them
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(c_swiglu(c_u2f(g[2 * i]), c_u2f(u[2 * i]), swiglu_lim),
                                  c_swiglu(c_u2f(g[2 * i + 1]), c_u2f(u[2 * i + 1]), swiglu_lim));
#pragma unroll
            for (int v = 0; v < 4; ++v)
              st_global_v4(dst + c + v * 8, pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
        tc_fence_before();
        mbar_arrive(tempty1);
        ++n1;
        // publish this warp's act rows to every CTA of the cluster
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) {
          const uint32_t ra = smem_addr(&ready[b]);
          for (int r = 0; r < C; ++r) mbar_arrive_cluster(mapa_shared(ra, (uint32_t)r));
        }
      } else {
        // weighted reduction of 256 output columns, two half rows of 128
        if (!(ok = mbar_wait(tfull2, (uint32_t)n2 & 1u, wc, 47))) break;
        tc_fence_after();
        const float w = args.slot_w[slot];
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tok < 0 ? 0 : tok) * args.D +
                              crank * dsl + sub * kFusedClusterN;
        const uint32_t tacc = lane_base + kAcc2Col;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          bulk_wait_read_all();  // the previous reduction has left the staging row
#pragma unroll 1
          for (int c = hh * 4; c < hh * 4 + 4; c += 2) {
            uint32_t v0[32], v1[32];
            tmem_ld_x32_pair(tacc + c * 32, tacc + (c + 1) * 32, v0, v1);
            if (tok >= 0) {
              uint8_t* st0 = my_stage + (c - hh * 4) * 64;
#pragma unroll
              for (int v = 0; v < 4; ++v)
                st_shared_v4(st0 + v * 16, pack_bf16x2(w * c_u2f(v0[8 * v + 0]), w * c_u2f(v0[8 * v + 1])),
                             pack_bf16x2(w * c_u2f(v0[8 * v + 2]), w * c_u2f(v0[8 * v + 3])),
                             pack_bf16x2(w * c_u2f(v0[8 * v + 4]), w * c_u2f(v0[8 * v + 5])),
                             pack_bf16x2(w * c_u2f(v0[8 * v + 6]), w * c_u2f(v0[8 * v + 7])));
#pragma unroll
              for (int v = 0; v < 4; ++v)
                st_shared_v4(st0 + 64 + v * 16, pack_bf16x2(w * c_u2f(v1[8 * v + 0]), w * c_u2f(v1[8 * v + 1])),
                             pack_bf16x2(w * c_u2f(v1[8 * v + 2]), w * c_u2f(v1[8 * v + 3])),
                             pack_bf16x2(w * c_u2f(v1[8 * v + 4]), w * c_u2f(v1[8 * v + 5])),
                             pack_bf16x2(w * c_u2f(v1[8 * v + 6]), w * c_u2f(v1[8 * v + 7])));
            }
          }
          if (tok >= 0) {
            fence_proxy_async_smem();
            bulk_reduce_add_bf16_hint(orow + hh * (kFusedClusterN / 2), my_stage, kFusedClusterN, args.out_hint != 0, l2_policy_evict_last());
            bulk_commit();
          }
        }
        tc_fence_before();
        mbar_arrive(tempty2);
        ++n2;
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

cudaError_t set_smem_once() {
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fused_cluster_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCSmem);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

int fused_cluster_max_clusters(int csize) {
  // once per (device, cluster size): not a stream operation
  static int cache[64][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int slot = csize == 1 ? 0 : csize == 2 ? 1 : csize == 4 ? 2 : csize == 8 ? 3 : -1;
  if (slot < 0) return 0;
  if (cache[dev][slot]) return cache[dev][slot];
  if (set_smem_once() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize);
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = kCSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fused_cluster_bf16_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cache[dev][slot] = n;
  return n;
}

cudaError_t launch_fused_cluster_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w2,
                                      const CUtensorMap& map_ring, const FusedClusterArgs& args, int n_clusters,
                                      cudaStream_t stream) {
  cudaError_t e = set_smem_once();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_clusters * args.csize);
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = kCSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = args.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_cluster_bf16_kernel, map_xg, map_w1, map_w2, map_ring, args);
}

}  // namespace moe
