// gemm_fused_dsmem.cu -- the fused pipeline on thread-block clusters with the
// activation kept in shared memory: out += w * W2 . SwiGLU(W1 . x) for every
// routed row in one launch, and no byte of act is written to or read from
// global memory ("Prime Flash MoE" sec. 5 "SwiGLU - which never leaves the
// SM"; sec. 2 "Trick 2": the intermediate dimension is split over CTAs).
//
// A cluster of C CTAs owns one 128-row block rb (expert e) at a time.  CTA c
// owns act columns [c*h, (c+1)*h), h = H / C (a multiple of 64, at most 256),
// and output columns [c*dsl, (c+1)*dsl), dsl = D / C:
//   GEMM1 (s1 sub-chunks of h1 columns): acc[128 x 2*h1] = xg[rb] . [W1 gate |
//          W1 up rows of the sub-chunk]^T over K = D.
//   SwiGLU epilogue: silu(gate) * up in fp32, rounded to bf16 and stored into
//          this CTA's act buffer in shared memory: h/64 tiles of 128 rows x 64
//          columns in the 128-byte-swizzled K-major layout the tensor core
//          reads, i.e. already GEMM2's A operand.
//   GEMM2 (s2 sub-chunks of 256 output columns): acc[128 x 256] = act[rb, all
//          H] . W2[e][cols, :]^T over K = H in 64-column K tiles.  A K tile
//          owned by this CTA is read by the MMA straight from the act buffer;
//          a tile owned by CTA q is copied by this CTA's producer warp from q's
//          shared memory (distributed shared memory loads, 16 KB) into the
//          A slot of its own pipeline stage.
//   Reduction epilogue: rows scaled by their routing weight in fp32, rounded
//          to bf16 and added into out[row_tok, ..] with bulk .add.bf16
//          reductions (sec. 5 "Three jobs - one instruction").
// Job order per round r: the GEMM2 sub-chunks of row block r - 1, then the
// GEMM1 sub-chunks of row block r; consecutive jobs alternate between the two
// 256-column TMEM accumulators, so each job's epilogue overlaps the next job's
// MMAs.  The act buffer is single: GEMM1's epilogue of row block r waits until
// every copy of row block r - 1's tiles has landed and this CTA's MMAs have
// read its own tiles.
//
// Flow control, once per row block (no handshake per K tile):
//   act_ready  (local) the four epilogue warps of each GEMM1 sub-chunk have
//                      stored their act rows (and fenced them for the async proxy);
//   peers_ready (each CTA) every other CTA of the cluster arrives once its act
//                      of the row block is stored: its tiles may be read;
//   act_free   (owner) each other CTA arrives once per K tile of this owner
//                      it has copied; the owner's MMA issuer commits once after
//                      its last own-tile MMA of the block.
// Every wait is bounded; every CTA reaches the final cluster barrier.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kDThreads = 192;
constexpr int kDEpi = 128;
constexpr int kDStages = 3;
constexpr int kDA = kBM * kBK * 2;            // 16 KB: an xg tile or a pushed act tile
constexpr int kDB = 256 * kBK * 2;            // 32 KB: W1 (2*h1 <= 256 rows) or W2 (256 rows)
constexpr int kDStage = kDA + kDB;
constexpr int kDChunk = 64;                   // output columns per staged reduction
constexpr int kDStageRow = kDChunk * 2 + 16;  // staging row (+16 B: a warp's rows on distinct banks)
constexpr int kDStaging = kBM * kDStageRow;
constexpr int kDBarrierBytes = 256;
constexpr int kDActMax = 4 * kDA;             // act buffer: up to four 64-column tiles (h <= 256)
constexpr int kDSmem = kDStages * kDStage + kDActMax + kDStaging + kDBarrierBytes;
static_assert(kDSmem <= 232448, "shared memory");
static_assert((2 * kDStages + 11) * 8 + 8 <= kDBarrierBytes, "barrier area");
constexpr uint64_t kDDrainNs = 200ull * 1000 * 1000;

__device__ __forceinline__ float d_u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ float d_swiglu(float g, float u, float lim) {
  g = fminf(g, lim);
  u = fminf(fmaxf(u, -lim), lim);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// 16 bytes from another CTA's shared memory (a shared::cluster address)
__device__ __forceinline__ uint4 ld_dsmem_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// One 16 KB act tile of a peer (src: shared::cluster address) into this CTA's
// shared memory, layout unchanged; the 32 lanes of the calling warp each move
// 512 bytes, eight 16-byte loads in flight per lane at a time.
__device__ __forceinline__ void pull_tile(uint8_t* dst, uint32_t src, int lane) {
#pragma unroll 1
  for (int i0 = 0; i0 < 32; i0 += 8) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ld_dsmem_v4(src + (uint32_t)(((i0 + i) * 32 + lane) * 16));
#pragma unroll
    for (int i = 0; i < 8; ++i) st_shared_v4(dst + ((i0 + i) * 32 + lane) * 16, v[i].x, v[i].y, v[i].z, v[i].w);
  }
}

// Jobs of round r (row blocks 0 .. n-1 of this cluster; r in 0 .. n): the
// GEMM2 sub-chunks of row block r - 1, then the GEMM1 sub-chunks of row block r.
__device__ __forceinline__ int d_round_jobs(int r, int n, int s1, int s2) {
  return (r >= 1 ? s2 : 0) + (r < n ? s1 : 0);
}
__device__ __forceinline__ bool d_job(int r, int j, int s2, int* it, int* sub) {
  const int n2 = r >= 1 ? s2 : 0;
  if (j < n2) {
    *it = r - 1;
    *sub = j;
    return true;
  }
  *it = r;
  *sub = j - n2;
  return false;
}

__global__ void __launch_bounds__(kDThreads, 1)
    fused_dsmem_bf16_kernel(const __grid_constant__ CUtensorMap map_xg, const __grid_constant__ CUtensorMap map_w1,
                            const __grid_constant__ CUtensorMap map_w2, const FusedClusterArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_addr(smem_raw) & 1023u) {  // the same in every CTA: all of them return here
    if (threadIdx.x == 0) atomicOr(args.err, kErrLaunch);
    return;
  }
  uint8_t* stages = smem_raw;
  uint8_t* actbuf = smem_raw + kDStages * kDStage;
  uint8_t* staging = actbuf + kDActMax;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + kDStaging);
  uint64_t* empty = full + kDStages;
  uint64_t* peers_ready = empty + kDStages;
  uint64_t* tfull = peers_ready + 1;   // [2]
  uint64_t* tempty = tfull + 2;        // [2]
  uint64_t* act_ready = tempty + 2;
  uint64_t* act_free = act_ready + 1;
  uint64_t* drain = act_free + 1;
  uint64_t* never = drain + 1;         // no thread ever arrives here (failure-path test hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float swiglu_lim = args.swiglu_limit > 0.f ? args.swiglu_limit : __int_as_float(0x7f800000);
  const WaitCtl wc{abort_flag, args.err, args.wait_limit_ns};
  const int C = args.csize;
  const int crank = (int)blockIdx.x % C, cid = (int)blockIdx.x / C, ncl = (int)gridDim.x / C;
  const int h1 = args.h1, s1 = args.s1, s2 = args.s2;
  const int h = h1 * s1;                    // act columns of this CTA
  const int n_kt = h / kBK;                 // K tiles of act owned by each CTA
  const int dsl = kFusedClusterN * s2;      // output columns of this CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(peers_ready, C - 1 > 0 ? C - 1 : 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kDEpi);
    }
    mbar_init(act_ready, 4 * s1);
    mbar_init(act_free, (C - 1) * n_kt * s2 + 1);
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
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive or copy
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();

  const int num_rb = args.meta[0];
  const int n_it = cid < num_rb ? (num_rb - cid + ncl - 1) / ncl : 0;
  const int n_rounds = n_it > 0 ? n_it + 1 : 0;
  const int KB1 = args.D / kBK, KT = args.H / kBK;
  (void)KT;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (lane 0 issues the
    // loads; the whole warp copies the act tiles of peers)
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[kDStages];
#pragma unroll
    for (int i = 0; i < kDStages; ++i) issued_phase[i] = -1;
    bool ok = true;
    int ready_cnt = 0;               // row blocks whose act this CTA and its peers have stored
    auto warp_wait = [&](uint64_t* bar, uint32_t parity, int site, bool cluster) -> bool {
      int got = 1;
      if (lane == 0) got = (cluster ? mbar_wait_cluster(bar, parity, wc, site) : mbar_wait(bar, parity, wc, site)) ? 1 : 0;
      return __shfl_sync(0xffffffffu, got, 0) != 0;
    };
    for (int r = 0; ok && r < n_rounds; ++r) {
      const int nj = d_round_jobs(r, n_it, s1, s2);
      for (int j = 0; ok && j < nj; ++j) {
        int it, sub;
        const bool g2 = d_job(r, j, s2, &it, &sub);
        const int rb = cid + it * ncl;
        const int e = args.expert_of_rb[rb];
        if (g2 && sub == 0) {
          // this CTA's act tiles of row block it are stored: tell the peers, then
          // wait until every peer's are
          if (!(ok = warp_wait(act_ready, (uint32_t)ready_cnt & 1u, 51, false))) break;
          if (lane == 0)
            for (int p = 0; p < C; ++p)
              if (p != crank) mbar_arrive_cluster(mapa_shared(smem_addr(peers_ready), (uint32_t)p));
          if (C > 1 && !(ok = warp_wait(peers_ready, (uint32_t)ready_cnt & 1u, 53, true))) break;
          ++ready_cnt;
        }
        const int KB = g2 ? KT : KB1;
        const int w1_row = e * 2 * args.H + crank * h + sub * h1;
        const int w2_row = e * args.D + crank * dsl + sub * kFusedClusterN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = warp_wait(&empty[s], ph ^ 1u, 52, false))) break;
          uint8_t* st = stages + s * kDStage;
          if (!g2) {
            if (lane == 0) {
              mbar_arrive_expect_tx(&full[s], kDA + 2 * h1 * kBK * 2);
              tma_load_2d(st, &map_xg, &full[s], kb * kBK, rb * kBM);
              tma_load_2d(st + kDA, &map_w1, &full[s], kb * kBK, w1_row);
              tma_load_2d(st + kDA + h1 * kBK * 2, &map_w1, &full[s], kb * kBK, w1_row + args.H);
            }
          } else {
            const int q = kb / n_kt;
            if (lane == 0) tma_load_2d(st + kDA, &map_w2, &full[s], kb * kBK, w2_row);
            if (q != crank) {
              // a peer's K tile: copy it into this stage's A slot (the MMA reads
              // an own tile in place), then release it to its owner
              pull_tile(st, mapa_shared(smem_addr(actbuf + (kb - q * n_kt) * kDA), (uint32_t)q), lane);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_addr(act_free), (uint32_t)q));
            }
            // armed after the copy: the phase completes when the W2 tile lands
            if (lane == 0) mbar_arrive_expect_tx(&full[s], kDB);
          }
          issued_phase[s] = (int)ph;
          if (++s == kDStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (!ok && lane == 0) {  // let every copy already in flight land before the CTA exits
      for (int i = 0; i < kDStages; ++i)
        if (issued_phase[i] >= 0) mbar_wait_drain(&full[i], (uint32_t)issued_phase[i], kDDrainNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc1 = idesc_bf16_f32(kBM, 2 * h1);
    constexpr uint32_t idesc2 = idesc_bf16_f32(kBM, kFusedClusterN);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (args.stall_test) ok = mbar_wait(never, 0, wc, 99);  // runs out after the wait limit
    int J = 0;
    int ready_cnt = 0;
    for (int r = 0; ok && r < n_rounds; ++r) {
      const int nj = d_round_jobs(r, n_it, s1, s2);
      for (int j = 0; ok && j < nj; ++j, ++J) {
        int it, sub;
        const bool g2 = d_job(r, j, s2, &it, &sub);
        const int acc = J & 1;
        if (!(ok = mbar_wait(&tempty[acc], ((uint32_t)(J >> 1) & 1u) ^ 1u, wc, 54))) break;
        tc_fence_after();
        if (g2 && sub == 0) {  // own act tiles stored (fenced for the async proxy)
          if (!(ok = mbar_wait(act_ready, (uint32_t)ready_cnt & 1u, wc, 55))) break;
          ++ready_cnt;
        }
        const uint32_t d_tmem = tmem_base + acc * 256;
        const uint32_t idesc = g2 ? idesc2 : idesc1;
        const int KB = g2 ? KT : KB1;
        for (int kb = 0; kb < KB; ++kb) {
          if (!(ok = mbar_wait(&full[s], ph, wc, 56))) break;
          tc_fence_after();
          const int q = g2 ? kb / n_kt : crank;
          const uint8_t* a_tile = (g2 && q == crank) ? actbuf + (kb - q * n_kt) * kDA : stages + s * kDStage;
          const uint64_t adesc = sdesc_sw128(smem_addr(a_tile));
          const uint64_t bdesc = sdesc_sw128(smem_addr(stages + s * kDStage + kDA));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
          umma_commit(&empty[s]);
          if (++s == kDStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (g2 && sub == s2 - 1) umma_commit(act_free);  // this CTA's MMAs on its own tiles are done
        umma_commit(&tfull[acc]);
      }
    }
    if (!ok) {  // wait for every MMA already issued before TMEM is released
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kDDrainNs);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogues
    const int quad = warp & 3;  // TMEM lanes this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    uint8_t* my_stage = staging + row * kDStageRow;
    bool ok = true;
    int J = 0;
    for (int r = 0; ok && r < n_rounds; ++r) {
      const int nj = d_round_jobs(r, n_it, s1, s2);
      for (int j = 0; ok && j < nj; ++j, ++J) {
        int it, sub;
        const bool g2 = d_job(r, j, s2, &it, &sub);
        const int acc = J & 1;
        const int rb = cid + it * ncl;
        const int64_t slot = (int64_t)rb * kBM + row;
        const int tok = args.row_tok[slot];
        if (!(ok = mbar_wait(&tfull[acc], (uint32_t)(J >> 1) & 1u, wc, 57))) break;
        tc_fence_after();
        const uint32_t tacc = lane_base + acc * 256;
        if (!g2) {
          // the act buffer still holds row block it - 1 until every copy of it landed
          if (it >= 1 && sub == 0 &&
              !(ok = mbar_wait_cluster(act_free, (uint32_t)(it - 1) & 1u, wc, 58)))
            break;
          // SwiGLU of columns [sub*h1, (sub+1)*h1) of this CTA's slice; gate in
          // accumulator columns [0, h1), up in [h1, 2*h1)
#pragma unroll 1
          for (int c = 0; c < h1; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld_x32_pair(tacc + c, tacc + h1 + c, g, u);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(d_swiglu(d_u2f(g[2 * i]), d_u2f(u[2 * i]), swiglu_lim),
                                  d_swiglu(d_u2f(g[2 * i + 1]), d_u2f(u[2 * i + 1]), swiglu_lim));
            // four 16-byte chunks of 8 act columns each, at their swizzled places
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int col = sub * h1 + c + v * 8;            // local act column
              const int kt = col >> 6, ch = (col & 63) >> 3;
              st_shared_v4(actbuf + kt * kDA + row * 128 + ((ch ^ (row & 7)) << 4), pk[4 * v], pk[4 * v + 1],
                           pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
          fence_proxy_async_smem();  // act rows visible to the tensor core and the bulk copies
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          __syncwarp();
          if (lane == 0) mbar_arrive(act_ready);
        } else {
          // weighted reduction of 256 output columns in chunks of 64
          const float w = args.slot_w[slot];
          __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.out) + (int64_t)(tok < 0 ? 0 : tok) * args.D +
                                crank * dsl + sub * kFusedClusterN;
#pragma unroll 1
          for (int c0 = 0; c0 < kFusedClusterN; c0 += kDChunk) {
            uint32_t v0[32], v1[32];
            tmem_ld_x32_pair(tacc + c0, tacc + c0 + 32, v0, v1);
            if (tok >= 0) {
              bulk_wait_read_all();  // the previous reduction has left the staging row
#pragma unroll
              for (int v = 0; v < 4; ++v)
                st_shared_v4(my_stage + v * 16, pack_bf16x2(w * d_u2f(v0[8 * v + 0]), w * d_u2f(v0[8 * v + 1])),
                             pack_bf16x2(w * d_u2f(v0[8 * v + 2]), w * d_u2f(v0[8 * v + 3])),
                             pack_bf16x2(w * d_u2f(v0[8 * v + 4]), w * d_u2f(v0[8 * v + 5])),
                             pack_bf16x2(w * d_u2f(v0[8 * v + 6]), w * d_u2f(v0[8 * v + 7])));
#pragma unroll
              for (int v = 0; v < 4; ++v)
                st_shared_v4(my_stage + 64 + v * 16, pack_bf16x2(w * d_u2f(v1[8 * v + 0]), w * d_u2f(v1[8 * v + 1])),
                             pack_bf16x2(w * d_u2f(v1[8 * v + 2]), w * d_u2f(v1[8 * v + 3])),
                             pack_bf16x2(w * d_u2f(v1[8 * v + 4]), w * d_u2f(v1[8 * v + 5])),
                             pack_bf16x2(w * d_u2f(v1[8 * v + 6]), w * d_u2f(v1[8 * v + 7])));
              fence_proxy_async_smem();
              bulk_reduce_add_bf16_hint(orow + c0, my_stage, kDChunk * 2, args.out_hint != 0,
                                        l2_policy_evict_last());
              bulk_commit();
            }
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
        }
      }
    }
    bulk_wait_all();  // bulk reductions complete before the CTA exits
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while another may still arrive on or copy into it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

cudaError_t dsmem_smem_once() {
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fused_dsmem_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmem);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

int fused_dsmem_max_clusters(int csize) {
  // once per (device, cluster size): not a stream operation
  static int cache[64][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int slot = csize == 1 ? 0 : csize == 2 ? 1 : csize == 4 ? 2 : csize == 8 ? 3 : -1;
  if (slot < 0) return 0;
  if (cache[dev][slot]) return cache[dev][slot];
  if (dsmem_smem_once() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize);
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = kDSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fused_dsmem_bf16_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cache[dev][slot] = n;
  return n;
}

cudaError_t launch_fused_dsmem_bf16(const CUtensorMap& map_xg, const CUtensorMap& map_w1, const CUtensorMap& map_w2,
                                    const FusedClusterArgs& args, int n_clusters, cudaStream_t stream) {
  cudaError_t e = dsmem_smem_once();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_clusters * args.csize);
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = kDSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = args.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_dsmem_bf16_kernel, map_xg, map_w1, map_w2, args);
}

}  // namespace moe
