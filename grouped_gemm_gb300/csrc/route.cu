// route.cu -- the routing permutation and the row gather.
//
// Routing ("Prime Flash MoE", sec. 3 "For the tokens: TMA gathers them too"
// and sec. 6 "The down-projection kernel": tokens are processed in sorted,
// per-expert order with each expert's segment padded to 128 rows):
//   counts[e]      = #pairs p = t*k + j with topk_ids[p] == e
//   offsets        = exclusive scan of counts               (E+1 entries)
//   pad_offsets    = exclusive scan of counts rounded up to 128
//   slot_of_pair[p]= offsets[e] + #{p' < p : topk_ids[p'] == e}  (stable)
//   row_tok[s], slot_w[s] for the padded slot s = pad_offsets[e] + rank,
//   -1 / 0 for padding rows; expert_of_rb[rb] for each 128-row block.
// Three kernels, all deterministic (no order-dependent atomics on results):
//   1. per-block histograms,
//   2. one block: scans over blocks and over experts, padding, block->expert,
//   3. per-block stable scatter using warp match + per-warp prefix counts.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <map>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kScatterWarps = 8;

// ---------------------------------------------------------------- router
// Top-k of one token's router logits by one warp, and the softmax of the
// selected logits.  This is the step upstream of the path: "Prime Flash MoE"
// sec. 1 takes each token's k experts and their weights (which sum to one) as
// given, and the workloads produce them from per-(token, expert) logits, the
// k largest with a softmax over just those k.
//   order: decreasing logit, ties to the lower expert id, NaN read as -inf;
//   w[j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) in fp32 (l_0 the largest);
//   every weight is 1/k when l_0 is -inf.
// Lane l holds experts l, l + 32, ... (EPL of them); the expert selected
// j-th is kept by lane j % 32 in slot j / 32.
template <int EPL>
__device__ __forceinline__ void router_warp_topk(const float* __restrict__ lrow, int E, int k, int32_t* ids,
                                                 float* w) {
  const int lane = threadIdx.x & 31;
  float v[EPL];
  uint32_t avail = 0;  // bit i: expert lane + 32 i exists and is not taken yet
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    const float x = e < E ? lrow[e] : -INFINITY;
    v[i] = x != x ? -INFINITY : x;
    if (e < E) avail |= 1u << i;
  }
  float selv[EPL];
  int seli[EPL];
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    selv[q] = -INFINITY;
    seli[q] = 0;
  }
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = INT_MAX;  // none yet: loses to any expert, even one at -inf
#pragma unroll
    for (int i = 0; i < EPL; ++i)  // ascending ids: strict > keeps the lower id on ties
      if (((avail >> i) & 1u) && (bi == INT_MAX || v[i] > bv)) {
        bv = v[i];
        bi = lane + 32 * i;
      }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
    if ((j & 31) == lane) {
#pragma unroll
      for (int q = 0; q < EPL; ++q)
        if (q == (j >> 5)) {
          selv[q] = bv;
          seli[q] = bi;
        }
    }
  }
  const float m = __shfl_sync(0xffffffffu, selv[0], 0);
  const bool flat = m == -INFINITY;
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < EPL; ++q)
    if (q * 32 + lane < k) s += flat ? 1.f : expf(selv[q] - m);
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int j = q * 32 + lane;
    if (j < k) {
      ids[j] = seli[q];
      w[j] = (flat ? 1.f : expf(selv[q] - m)) / s;
    }
  }
}

// Experts per lane for E experts (a power of two, E <= 32 * result).
__host__ __device__ constexpr int router_epl(int E) {
  return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : E <= 512 ? 16 : 32;
}

// Tokens [t0, t1) by the block's warps: top-k ids and weights written to
// ids / w [T, k].
template <int EPL>
__device__ void router_tokens(const float* __restrict__ logits, int E, int k, int t0, int t1, int32_t* ids,
                              float* w) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int t = t0 + warp; t < t1; t += nw)
    router_warp_topk<EPL>(logits + (int64_t)t * E, E, k, ids + (int64_t)t * k, w + (int64_t)t * k);
}

__device__ void router_tokens_any(const float* __restrict__ logits, int E, int k, int t0, int t1, int32_t* ids,
                                  float* w) {
  switch (router_epl(E)) {
    case 1: router_tokens<1>(logits, E, k, t0, t1, ids, w); break;
    case 2: router_tokens<2>(logits, E, k, t0, t1, ids, w); break;
    case 4: router_tokens<4>(logits, E, k, t0, t1, ids, w); break;
    case 8: router_tokens<8>(logits, E, k, t0, t1, ids, w); break;
    case 16: router_tokens<16>(logits, E, k, t0, t1, ids, w); break;
    default: router_tokens<32>(logits, E, k, t0, t1, ids, w); break;
  }
}

// The router alone: one warp per token.
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                          int32_t* __restrict__ ids, float* __restrict__ w) {
  const int per_block = blockDim.x >> 5;
  const int t0 = blockIdx.x * per_block;
  router_tokens_any(logits, E, k, t0, min(T, t0 + per_block), ids, w);
}

__global__ void __launch_bounds__(256) route_count_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int k,
                                                          int NB, int tpb, int* __restrict__ blk_counts,
                                                          int* __restrict__ err, uint4* __restrict__ zero_out,
                                                          int64_t zero_vecs) {
  extern __shared__ int hist[];
  if (zero_out) {  // every block of the (possibly wider) grid helps zero-fill the reduction target
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < zero_vecs;
         i += (int64_t)gridDim.x * blockDim.x)
      zero_out[i] = z;
  }
  if ((int)blockIdx.x >= NB) return;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t p0 = (int64_t)blockIdx.x * tpb * k;
  const int64_t p1 = min(P, p0 + (int64_t)tpb * k);
  bool bad = false;
  for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = ids[p];
    if ((unsigned)e < (unsigned)E) atomicAdd(&hist[e], 1);
    else bad = true;
  }
  if (bad) atomicOr(err, kErrBadRouting);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blk_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// Exclusive scan of one int per thread over a 1024-thread block; *total gets the sum.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int base = warp ? warp_sums[warp - 1] : 0;
  *total = warp_sums[31];
  __syncthreads();
  return base + x - v;
}

// Pairs of consecutive row blocks of one expert: expert e with nrb blocks owns
// ceil(nrb/2) pairs; pair_info = (first block << 1) | (1 if the pair is full).
__device__ void fill_pairs(int e, int lane, int po, int pc, int pair_off, int* pair_info) {
  const int rb0 = po / kRowPad, nrb = pc / kRowPad;
  for (int q = lane; q < (nrb + 1) / 2; q += 32)
    pair_info[pair_off + q] = ((rb0 + 2 * q) << 1) | (2 * q + 1 < nrb ? 1 : 0);
}

__global__ void __launch_bounds__(1024) route_scan_kernel(int NB, int E, int* __restrict__ blk, int* counts,
                                                          int* offsets, int* pad_offsets, int* meta,
                                                          int* expert_of_rb, int* pair_info, int* row_tok,
                                                          float* slot_w) {
  __shared__ int seg_sum[1024];
  __shared__ int cnt_s[kMaxExperts];
  __shared__ int warp_sums[32];
  griddep_wait();  // programmatic dependent of the histogram launch
  griddep_launch_dependents();
  const int tid = threadIdx.x;
  int Ep = 1;
  while (Ep < E) Ep <<= 1;
  const int nseg = 1024 / Ep;
  const int e = tid % Ep, seg = tid / Ep;
  const int per = (NB + nseg - 1) / nseg;
  const int b0 = min(NB, seg * per), b1 = min(NB, b0 + per);
  // pass 1: per-segment sums of the block histograms
  int run = 0;
  if (e < E) {
#pragma unroll 8
    for (int b = b0; b < b1; ++b) run += blk[(int64_t)b * E + e];
  }
  seg_sum[tid] = run;
  __syncthreads();
  if (seg == 0 && e < E) {
    int acc = 0;
    for (int s = 0; s < nseg; ++s) {
      const int v = seg_sum[s * Ep + e];
      seg_sum[s * Ep + e] = acc;
      acc += v;
    }
    cnt_s[e] = acc;
  }
  __syncthreads();
  // pass 2: per-block rank bases (exclusive scan over blocks, per expert)
  if (e < E) {
    int acc = seg_sum[tid];
#pragma unroll 8
    for (int b = b0; b < b1; ++b) {
      const int c = blk[(int64_t)b * E + e];
      blk[(int64_t)b * E + e] = acc;
      acc += c;
    }
  }
  // scans over experts
  const int cnt = tid < E ? cnt_s[tid] : 0;
  const int padc = (cnt + kRowPad - 1) / kRowPad * kRowPad;
  int tot, ptot, qtot;
  const int off = block_exclusive_scan(cnt, warp_sums, &tot);
  const int poff = block_exclusive_scan(padc, warp_sums, &ptot);
  const int qoff = block_exclusive_scan((padc / kRowPad + 1) / 2, warp_sums, &qtot);
  __shared__ int pair_off_s[kMaxExperts];
  if (tid < E) {
    counts[tid] = cnt;
    offsets[tid] = off;
    pad_offsets[tid] = poff;
    seg_sum[tid] = poff;  // reuse: padded offset of each expert
    pair_off_s[tid] = qoff;
  }
  if (tid == 0) {
    offsets[E] = tot;
    pad_offsets[E] = ptot;
    meta[0] = ptot / kRowPad;
    meta[1] = qtot;
    meta[2] = 0;  // tile counters of the GEMM kernels that follow
    meta[3] = 0;
  }
  __syncthreads();
  // padding rows and block -> expert, one warp per expert
  const int warp = tid >> 5, lane = tid & 31;
  for (int e = warp; e < E; e += 32) {
    const int c = cnt_s[e], po = seg_sum[e];
    const int pc = (c + kRowPad - 1) / kRowPad * kRowPad;
    for (int s2 = po + c + lane; s2 < po + pc; s2 += 32) {
      row_tok[s2] = -1;
      slot_w[s2] = 0.f;
    }
    for (int rb = po / kRowPad + lane; rb < (po + pc) / kRowPad; rb += 32) expert_of_rb[rb] = e;
    fill_pairs(e, lane, po, pc, pair_off_s[e], pair_info);
  }
}

// Stable scatter of one warp's contiguous pair range [q0, q1): 32 pairs per
// step, ranks from __match_any_sync, the running per-expert base in `mine`.
// ids and weights are fetched eight steps at a time so the loop is not a chain
// of dependent global loads.
// kFresh: ids and weights were written earlier in the same launch (the router
// runs first in the block), so they are read with volatile loads from L2,
// never through the read-only path.
template <bool kFresh = false>
__device__ __forceinline__ int load_i32(const int32_t* p) {
  if constexpr (kFresh) return *reinterpret_cast<const volatile int32_t*>(p);
  else return *p;
}
template <bool kFresh = false>
__device__ __forceinline__ float load_f32(const float* p) {
  if constexpr (kFresh) return *reinterpret_cast<const volatile float*>(p);
  else return *p;
}

template <bool kFresh = false>
__device__ __forceinline__ void scatter_range(const int32_t* ids, const float* topk_w,
                                              int64_t q0, int64_t q1, int E, int k, int* mine, const int* s_off,
                                              const int* s_poff, int* __restrict__ row_tok,
                                              float* __restrict__ slot_w, int* __restrict__ slot_of_pair) {
  const int lane = threadIdx.x & 31;
  constexpr int kBatch = 8;
  for (int64_t b0 = q0; b0 < q1; b0 += 32 * kBatch) {
    int ev[kBatch];
    float wv[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int64_t p = b0 + i * 32 + lane;
      ev[i] = p < q1 ? load_i32<kFresh>(ids + p) : -1;
      wv[i] = p < q1 ? load_f32<kFresh>(topk_w + p) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int64_t p = b0 + i * 32 + lane;
      if (b0 + i * 32 >= q1) break;  // warp-uniform
      const bool in = p < q1;
      const int e = ev[i];
      const bool valid = in && (unsigned)e < (unsigned)E;
      const int key = valid ? e : E + lane;  // invalid lanes never match anyone
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int r = valid ? mine[e] + rank : 0;
      __syncwarp();
      if (valid && rank == 0) mine[e] += __popc(peers);
      __syncwarp();
      if (valid) {
        const int ps = s_poff[e] + r;
        row_tok[ps] = (int)(p / k);
        slot_w[ps] = wv[i];
        slot_of_pair[p] = s_off[e] + r;
      } else if (in) {
        slot_of_pair[p] = -1;
      }
    }
  }
}

__global__ void __launch_bounds__(kScatterWarps * 32)
    route_scatter_kernel(const int32_t* __restrict__ ids, const float* __restrict__ topk_w, int64_t P, int E, int k,
                         int tpb, const int* __restrict__ blk_base, const int* __restrict__ offsets,
                         const int* __restrict__ pad_offsets, int* __restrict__ row_tok, float* __restrict__ slot_w,
                         int* __restrict__ slot_of_pair) {
  extern __shared__ int wcnt[];  // [kScatterWarps][E], then offsets[E], pad_offsets[E]
  int* s_off = wcnt + kScatterWarps * E;
  int* s_poff = s_off + E;
  griddep_wait();  // programmatic dependent of the scan launch
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t p0 = (int64_t)blockIdx.x * tpb * k;
  const int64_t p1 = min(P, p0 + (int64_t)tpb * k);
  const int64_t sub = (p1 - p0 + kScatterWarps - 1) / kScatterWarps;
  const int64_t q0 = min(p1, p0 + warp * sub), q1 = min(p1, q0 + sub);
  for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) wcnt[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    s_off[e] = offsets[e];
    s_poff[e] = pad_offsets[e];
  }
  __syncthreads();
  for (int64_t p = q0 + lane; p < q1; p += 32) {
    const int e = ids[p];
    if ((unsigned)e < (unsigned)E) atomicAdd(&wcnt[warp * E + e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int acc = blk_base[(int64_t)blockIdx.x * E + e];
    for (int w = 0; w < kScatterWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = acc;
      acc += c;
    }
  }
  __syncthreads();
  scatter_range(ids, topk_w, q0, q1, E, k, wcnt + warp * E, s_off, s_poff, row_tok, slot_w, slot_of_pair);
}

// The whole routing permutation in one 1024-thread block, for small problems
// (P <= g_route_small_pairs, E <= kRouteSmallMaxExperts): per-warp histograms
// of 32 contiguous pair ranges, scans over warps and experts, padding and
// block->expert tables, then the same stable warp-match scatter as above.
constexpr int kRouteSmallWarps = 32;
constexpr int kRouteSmallMaxExperts = 256;

// kRouter: the block first runs the router over all T tokens (logits [T, E]),
// writing ids / topk_w, and then routes what it wrote.
template <bool kRouter>
__global__ void __launch_bounds__(1024)
    route_small_kernel(const int32_t* ids, const float* topk_w, int P, int E, int k,
                       int* __restrict__ err, int* __restrict__ counts, int* __restrict__ offsets,
                       int* __restrict__ pad_offsets, int* __restrict__ meta, int* __restrict__ expert_of_rb,
                       int* __restrict__ pair_info, int* __restrict__ row_tok, float* __restrict__ slot_w,
                       int* __restrict__ slot_of_pair, const float* __restrict__ logits, int32_t* ids_out,
                       float* w_out) {
  __shared__ int wcnt[kRouteSmallWarps * kRouteSmallMaxExperts];
  __shared__ int s_off[kRouteSmallMaxExperts], s_poff[kRouteSmallMaxExperts], s_cnt[kRouteSmallMaxExperts];
  __shared__ int s_qoff[kRouteSmallMaxExperts];
  __shared__ int warp_sums[32];
  // the gather that follows may start now: it waits for this grid before
  // reading the routing tables, and meanwhile prefetches weights into L2
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = (P + kRouteSmallWarps - 1) / kRouteSmallWarps;
  const int q0 = min(P, warp * sub), q1 = min(P, q0 + sub);
  for (int i = threadIdx.x; i < kRouteSmallWarps * E; i += blockDim.x) wcnt[i] = 0;
  if constexpr (kRouter) {
    router_tokens_any(logits, E, k, 0, P / k, ids_out, w_out);
    ids = ids_out;
    topk_w = w_out;
  }
  __syncthreads();  // also orders the router's global writes before the reads below
  bool bad = false;
  for (int b0 = q0; b0 < q1; b0 += 32 * 8) {  // eight independent loads in flight per lane
    int ev[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int p = b0 + i * 32 + lane;
      ev[i] = p < q1 ? load_i32<kRouter>(ids + p) : 0;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (b0 + i * 32 + lane >= q1) continue;
      if ((unsigned)ev[i] < (unsigned)E) atomicAdd(&wcnt[warp * E + ev[i]], 1);
      else bad = true;
    }
  }
  if (bad) atomicOr(err, kErrBadRouting);
  __syncthreads();
  // exclusive prefix over warps, per expert; totals = counts
  int cnt = 0;
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    for (int w = 0; w < kRouteSmallWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = cnt;
      cnt += c;
    }
  }
  const int padc = (cnt + kRowPad - 1) / kRowPad * kRowPad;
  int tot, ptot, qtot;
  const int off = block_exclusive_scan(cnt, warp_sums, &tot);
  const int poff = block_exclusive_scan(padc, warp_sums, &ptot);
  const int qoff = block_exclusive_scan((padc / kRowPad + 1) / 2, warp_sums, &qtot);
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    counts[e] = cnt;
    offsets[e] = off;
    pad_offsets[e] = poff;
    s_off[e] = off;
    s_poff[e] = poff;
    s_cnt[e] = cnt;
    s_qoff[e] = qoff;
  }
  if (threadIdx.x == 0) {
    offsets[E] = tot;
    pad_offsets[E] = ptot;
    meta[0] = ptot / kRowPad;
    meta[1] = qtot;
    meta[2] = 0;  // tile counters of the GEMM kernels that follow
    meta[3] = 0;
  }
  __syncthreads();
  // padding rows and block -> expert, one warp per expert
  for (int e = warp; e < E; e += kRouteSmallWarps) {
    const int c = s_cnt[e], po = s_poff[e];
    const int pc = (c + kRowPad - 1) / kRowPad * kRowPad;
    for (int s2 = po + c + lane; s2 < po + pc; s2 += 32) {
      row_tok[s2] = -1;
      slot_w[s2] = 0.f;
    }
    for (int rb = po / kRowPad + lane; rb < (po + pc) / kRowPad; rb += 32) expert_of_rb[rb] = e;
    fill_pairs(e, lane, po, pc, s_qoff[e], pair_info);
  }
  // stable scatter
  scatter_range<kRouter>(ids, topk_w, q0, q1, E, k, wcnt + warp * E, s_off, s_poff, row_tok, slot_w, slot_of_pair);
}

// ---------------------------------------------------------------- one launch
// The whole routing permutation in ONE cooperative launch of NB = route_blocks
// blocks (all co-resident), for problems too large for the single-block
// kernel: the three phases of the three-kernel path separated by two grid
// barriers instead of two kernel boundaries.
//   A. per-warp histograms of contiguous pair ranges; block totals to
//      blk[b][e].  Block 0 sets meta to
//      "no row blocks" and every block marks its pairs' slots and its share
//      of the padded slots -1, so that if a barrier ever runs out the GEMMs
//      that follow find nothing to do rather than stale tables.
//   B. (more than 64 blocks only) one block per expert scans its column:
//      blk[.][e] becomes the exclusive prefix over blocks, counts[e] the
//      total.  With at most 64 blocks phase C reads the whole table instead,
//      and the second barrier is skipped.
//   C. every block scans counts over experts (offsets, padded offsets);
//      block 0 writes the expert tables (offsets, pad_offsets, expert_of_rb,
//      pair_info, padding rows, meta); every block scatters its own pairs with
//      the stable warp-match scatter.
// Grid barrier: err[4] counts arrivals, err[5] is the generation; both are
// zero at rest (status words, cleared with them).  Waits are bounded.
constexpr int kCoopWarps = 8;

struct CoopRouteArgs {
  const int32_t* ids;
  const float* topk_w;
  int64_t P;
  int E, k, NB;
  int tpb;  // tokens per block
  int* err;
  unsigned long long wait_limit_ns;
  int* blk;
  int* counts;
  int* offsets;
  int* pad_offsets;
  int* meta;
  int* expert_of_rb;
  int* pair_info;
  int* row_tok;
  float* slot_w;
  int* slot_of_pair;
  int64_t S_max;
  int stall_test;  // test hook: block 0 leaves before the first barrier
};

__device__ bool coop_grid_sync(const CoopRouteArgs& a, int site) {
  __syncthreads();
  int ok = 1;
  if (threadIdx.x == 0) {
    volatile int* gen = a.err + 5;
    const int g = *gen;
    __threadfence();
    if (atomicAdd(a.err + 4, 1) == a.NB - 1) {
      atomicExch(a.err + 4, 0);
      __threadfence();
      atomicAdd(a.err + 5, 1);
    } else {
      const uint64_t t0 = globaltimer_ns();
      for (uint32_t it = 1; *gen == g; ++it) {
        if ((it & 63) == 0 && globaltimer_ns() - t0 > a.wait_limit_ns) {
          atomicOr(a.err, kErrTimeout);
          atomicCAS(a.err + 1, 0, site);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
  }
  return __syncthreads_and(ok) != 0;
}

__global__ void __launch_bounds__(kCoopWarps * 32) route_coop_kernel(const CoopRouteArgs a) {
  if (threadIdx.x == 0) griddep_launch_dependents();  // see route_small_kernel
  extern __shared__ int sm[];
  int* wcnt = sm;                       // [kCoopWarps][E] per-warp counts, then bases
  int* s_off = wcnt + kCoopWarps * a.E;  // [E]
  int* s_poff = s_off + a.E;            // [E]
  int* s_cnt = s_poff + a.E;            // [E]
  int* s_qoff = s_cnt + a.E;            // [E]
  __shared__ int warp_sums[32];
  const int E = a.E, k = a.k, b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t p0 = (int64_t)b * a.tpb * k;
  const int64_t p1 = min(a.P, p0 + (int64_t)a.tpb * k);
  const int64_t sub = (p1 - p0 + kCoopWarps - 1) / kCoopWarps;
  const int64_t q0 = min(p1, p0 + warp * sub), q1 = min(p1, q0 + sub);
  const int32_t* ids = a.ids;
  const float* tw = a.topk_w;

  // ---- A
  if (b == 0 && threadIdx.x == 0) {
    a.meta[0] = 0;
    a.meta[1] = 0;
  }
  for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) a.slot_of_pair[p] = -1;
  for (int64_t r = (int64_t)b * blockDim.x + threadIdx.x; r < a.S_max; r += (int64_t)a.NB * blockDim.x)
    a.row_tok[r] = -1;
  for (int i = threadIdx.x; i < kCoopWarps * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  bool bad = false;
  for (int64_t p = q0 + lane; p < q1; p += 32) {
    const int e = ids[p];
    if ((unsigned)e < (unsigned)E) atomicAdd(&wcnt[warp * E + e], 1);
    else bad = true;
  }
  if (bad) atomicOr(a.err, kErrBadRouting);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int t = 0;
    for (int w = 0; w < kCoopWarps; ++w) t += wcnt[w * E + e];
    a.blk[(int64_t)b * E + e] = t;
  }
  if (a.stall_test && b == 0) return;  // the others' first barrier wait runs out
  if (!coop_grid_sync(a, 80)) return;

  // With few blocks (NB <= 64) every block reads the whole [NB, E] table of
  // block counts after the first barrier and derives the totals and its own
  // prefix itself (one barrier); otherwise phase B scans the columns first.
  const bool one_barrier = a.NB <= 64;
  if (!one_barrier) {
    // ---- B: exclusive prefix over blocks of each expert's column, one block
    // per expert, 256 blocks per step
    for (int e = b; e < E; e += a.NB) {
      int carry = 0;
      for (int c0 = 0; c0 < a.NB; c0 += blockDim.x) {
        const int bb = c0 + threadIdx.x;
        const int v = bb < a.NB ? a.blk[(int64_t)bb * E + e] : 0;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        int wbase = 0, tot = 0;
        for (int w = 0; w < kCoopWarps; ++w) {
          const int sw = warp_sums[w];
          if (w < warp) wbase += sw;
          tot += sw;
        }
        if (bb < a.NB) a.blk[(int64_t)bb * E + e] = carry + wbase + x - v;
        carry += tot;
        __syncthreads();
      }
      if (threadIdx.x == 0) a.counts[e] = carry;
    }
    if (!coop_grid_sync(a, 81)) return;
  }

  // ---- C: scans over experts (every block), tables (block 0), scatter (all)
  int warp_tot[3];
  if (one_barrier) {
    // totals and this block's prefix over blocks, straight from blk; the
    // prefix waits in s_qoff until the per-warp bases are formed below
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int tot = 0, mine = 0;
      for (int bb = 0; bb < a.NB; ++bb) {
        const int c = a.blk[(int64_t)bb * E + e];
        mine += bb < b ? c : 0;
        tot += c;
      }
      s_cnt[e] = tot;
      s_qoff[e] = mine;
      if (b == 0) a.counts[e] = tot;
    }
  } else {
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = a.counts[e];
  }
  __syncthreads();
  // one_barrier: this block's prefix of expert e, held by the thread that
  // forms e's per-warp bases below (s_qoff is reused for the pair offsets)
  int my_prefix[(kMaxExperts + kCoopWarps * 32 - 1) / (kCoopWarps * 32)];
#pragma unroll
  for (int q = 0; q < (kMaxExperts + kCoopWarps * 32 - 1) / (kCoopWarps * 32); ++q) {
    const int e = threadIdx.x + q * kCoopWarps * 32;
    my_prefix[q] = (one_barrier && e < E) ? s_qoff[e] : 0;
  }
  __syncthreads();
  // serial-in-thread chunks: thread i owns experts [i*per, (i+1)*per)
  const int per = (E + blockDim.x - 1) / blockDim.x;
  int c_sum = 0, pc_sum = 0, q_sum = 0;
  const int e0 = threadIdx.x * per;
  for (int e = e0; e < min(E, e0 + per); ++e) {
    const int c = s_cnt[e], pc = (c + kRowPad - 1) / kRowPad * kRowPad;
    c_sum += c;
    pc_sum += pc;
    q_sum += (pc / kRowPad + 1) / 2;
  }
  // block-wide exclusive scans of the three per-thread sums
  int vals[3] = {c_sum, pc_sum, q_sum}, excl[3];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    int x = vals[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    int wbase = 0, tot = 0;
    for (int w = 0; w < kCoopWarps; ++w) {
      const int sw = warp_sums[w];
      if (w < warp) wbase += sw;
      tot += sw;
    }
    excl[q] = wbase + x - vals[q];
    warp_tot[q] = tot;
    __syncthreads();
  }
  {
    int off = excl[0], poff = excl[1], qoff = excl[2];
    for (int e = e0; e < min(E, e0 + per); ++e) {
      const int c = s_cnt[e], pc = (c + kRowPad - 1) / kRowPad * kRowPad;
      s_off[e] = off;
      s_poff[e] = poff;
      s_qoff[e] = qoff;
      if (b == 0) {
        a.offsets[e] = off;
        a.pad_offsets[e] = poff;
      }
      off += c;
      poff += pc;
      qoff += (pc / kRowPad + 1) / 2;
    }
  }
  __syncthreads();
  if (b == 0) {
    // padding rows, block -> expert and pairs of every expert, one warp per expert
    for (int e = warp; e < E; e += kCoopWarps) {
      const int c = s_cnt[e], po = s_poff[e];
      const int pc = (c + kRowPad - 1) / kRowPad * kRowPad;
      for (int s2 = po + c + lane; s2 < po + pc; s2 += 32) a.slot_w[s2] = 0.f;  // row_tok is -1 already
      for (int rb = po / kRowPad + lane; rb < (po + pc) / kRowPad; rb += 32) a.expert_of_rb[rb] = e;
      fill_pairs(e, lane, po, pc, s_qoff[e], a.pair_info);
    }
    if (threadIdx.x == 0) {
      a.offsets[E] = warp_tot[0];
      a.pad_offsets[E] = warp_tot[1];
      a.meta[2] = 0;  // tile counters of the GEMM kernels that follow
      a.meta[3] = 0;
      a.meta[1] = warp_tot[2];
      __threadfence();
      a.meta[0] = warp_tot[1] / kRowPad;
    }
  }
  // this block's per-warp bases: its prefix over blocks + earlier warps
#pragma unroll
  for (int q = 0; q < (kMaxExperts + kCoopWarps * 32 - 1) / (kCoopWarps * 32); ++q) {
    const int e = threadIdx.x + q * kCoopWarps * 32;
    if (e >= E) break;
    int acc = one_barrier ? my_prefix[q] : a.blk[(int64_t)b * E + e];
    for (int w = 0; w < kCoopWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = acc;
      acc += c;
    }
  }
  __syncthreads();
  scatter_range(ids, tw, q0, q1, E, k, wcnt + warp * E, s_off, s_poff, a.row_tok, a.slot_w, a.slot_of_pair);
}

// Token-major gather: xg[padded slot of pair p, :] = x[t, :] for the k pairs
// p = t*k + j of every token t.  One warp per (token, 4 KB chunk of its row):
// the chunk is read once into registers (16-byte vector loads, eight per lane)
// and written to each of the token's k slots, so x is read once rather than k
// times.  The padded slot is slot_of_pair[p] - offsets[e] + pad_offsets[e].
// Padding rows of xg are never written: each GEMM output row depends only on
// its own input row, and padding rows are dropped by the epilogues.  The same
// warp zero-fills its share of the token's row of `out` (the reduction target
// of the down projection).  Launched as a programmatic dependent of the
// routing: it waits for the routing grid before reading its tables.
constexpr int kGatherChunkVecs = 256;  // 4 KB per warp work item

__global__ void __launch_bounds__(256)
    gather_tokens_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ ids,
                         const int* __restrict__ slot_of_pair, const int* __restrict__ offsets,
                         const int* __restrict__ pad_offsets, int T, int E, int k, int vec_per_row,
                         uint4* __restrict__ xg, uint4* __restrict__ out, int out_vecs_per_row, int keep_xg,
                         const uint8_t* __restrict__ pf_base, int64_t pf_bytes) {
  // keep_xg: the gathered rows are stored with an L2 evict_last policy, so
  // that more of them are still in L2 when the up projection reads them
  const uint64_t pol = l2_policy_evict_last();
  // While the routing finishes (latency-bound, HBM idle), each block asks L2
  // for its share of the first pf_bytes of the up projection's weights: the
  // first tiles of the up kernel then find them in L2.
  if (pf_bytes > 0 && threadIdx.x == 0) {
    const int64_t chunk = ((pf_bytes + gridDim.x - 1) / gridDim.x + 15) & ~(int64_t)15;
    const int64_t b0 = (int64_t)blockIdx.x * chunk;
    const int64_t n = min(chunk, pf_bytes - b0);
    if (n > 0) bulk_prefetch_l2(pf_base + b0, (uint32_t)n);
  }
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_chunks = (vec_per_row + kGatherChunkVecs - 1) / kGatherChunkVecs;
  const int zero_per = (out_vecs_per_row + n_chunks - 1) / n_chunks;
  const int64_t items = (int64_t)T * n_chunks;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t it = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp; it < items; it += nwarps) {
    const int t = (int)(it / n_chunks), c = (int)(it % n_chunks);
    const int v0 = c * kGatherChunkVecs;
    const uint4* src = x + (int64_t)t * vec_per_row + v0;
    uint4 v[kGatherChunkVecs / 32];
#pragma unroll
    for (int i = 0; i < kGatherChunkVecs / 32; ++i)
      if (v0 + i * 32 + lane < vec_per_row) v[i] = __ldg(src + i * 32 + lane);
    for (int j0 = 0; j0 < k; j0 += 32) {
      // lane l resolves the padded slot of pair j0 + l
      int ps = -1;
      if (j0 + lane < k) {
        const int64_t p = (int64_t)t * k + j0 + lane;
        const int e = ids[p], s = slot_of_pair[p];
        if (s >= 0 && (unsigned)e < (unsigned)E) ps = s - offsets[e] + pad_offsets[e];
      }
      const int nj = min(32, k - j0);
      for (int jj = 0; jj < nj; ++jj) {
        const int slot = __shfl_sync(0xffffffffu, ps, jj);
        if (slot < 0) continue;
        uint4* dst = xg + (int64_t)slot * vec_per_row + v0;
        if (keep_xg) {
#pragma unroll
          for (int i = 0; i < kGatherChunkVecs / 32; ++i)
            if (v0 + i * 32 + lane < vec_per_row) st_global_v4_hint(dst + i * 32 + lane, v[i], pol);
        } else {
#pragma unroll
          for (int i = 0; i < kGatherChunkVecs / 32; ++i)
            if (v0 + i * 32 + lane < vec_per_row) dst[i * 32 + lane] = v[i];
        }
      }
    }
    if (out) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      uint4* orow = out + (int64_t)t * out_vecs_per_row;
      const int z1 = min(out_vecs_per_row, (c + 1) * zero_per);
      for (int i = c * zero_per + lane; i < z1; i += 32) orow[i] = z;
    }
  }
}

}  // namespace

namespace {

thread_local const char* t_route_kernels = "none";

size_t route_coop_smem(int E) { return sizeof(int) * (size_t)(kCoopWarps + 4) * E; }

// Whether NB routing blocks can all be resident at once (checked once per
// device and expert count; a cooperative launch also refuses otherwise).
bool route_coop_fits(int NB, int E) {
  if (g_route_coop.load() == 0) return false;
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> cap;  // (device, E) -> resident blocks
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_pair(dev, E);
  auto it = cap.find(key);
  if (it == cap.end()) {
    int per_sm = 0, sms = 0, coop = 0;
    const size_t smem = route_coop_smem(E);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(route_coop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_coop_kernel, kCoopWarps * 32, smem) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    it = cap.emplace(key, coop ? per_sm * sms : 0).first;
  }
  return NB >= 2 && NB <= it->second;
}

}  // namespace

const char* last_route_kernels() { return t_route_kernels; }

cudaError_t launch_route(const Workspace& ws, const int32_t* topk_ids, const float* topk_w, int T, int E, int k,
                         cudaStream_t stream, void* zero_out, int64_t zero_bytes, int zero_grid, bool pdl) {
  const int64_t P = (int64_t)T * k;
  const float* logits = ws.router_logits;
  // with the router, topk_ids / topk_w are the caller's output arrays
  int32_t* ids_out = logits ? const_cast<int32_t*>(topk_ids) : nullptr;
  float* w_out = logits ? const_cast<float*>(topk_w) : nullptr;
  const bool small = !zero_out && P <= g_route_small_pairs.load() && E <= kRouteSmallMaxExperts;
  if (logits && (!small || !g_router_fused.load())) {
    // the router as its own wide launch (one warp per token): inside a
    // routing launch of a few blocks it would run on a small share of the GPU
    cudaError_t e = launch_router_topk(logits, T, E, k, ids_out, w_out, stream);
    if (e != cudaSuccess) return e;
    logits = nullptr;
  }
  const bool router_first = ws.router_logits && !logits;
  if (small) {
    t_route_kernels = router_first ? "router_topk+route_small" : "route_small";
    if (logits)
      route_small_kernel<true><<<1, 1024, 0, stream>>>(
          topk_ids, topk_w, (int)P, E, k, ws.err, ws.counts, ws.offsets, ws.pad_offsets, ws.meta, ws.expert_of_rb,
          ws.pair_info, ws.row_tok, ws.slot_w, ws.slot_of_pair, logits, ids_out, w_out);
    else
      route_small_kernel<false><<<1, 1024, 0, stream>>>(
          topk_ids, topk_w, (int)P, E, k, ws.err, ws.counts, ws.offsets, ws.pad_offsets, ws.meta, ws.expert_of_rb,
          ws.pair_info, ws.row_tok, ws.slot_w, ws.slot_of_pair, nullptr, nullptr, nullptr);
    return cudaGetLastError();
  }
  const int NB = ws.route_blocks;
  if (!zero_out && route_coop_fits(NB, E)) {
    t_route_kernels = router_first ? "router_topk+route_coop" : "route_coop";
    CoopRouteArgs ca{};
    ca.ids = topk_ids;
    ca.topk_w = topk_w;
    ca.P = P;
    ca.E = E;
    ca.k = k;
    ca.NB = NB;
    ca.tpb = ws.route_tpb;
    ca.err = ws.err;
    ca.wait_limit_ns = ws.wait_limit_ns;
    ca.blk = ws.blk_base;
    ca.counts = ws.counts;
    ca.offsets = ws.offsets;
    ca.pad_offsets = ws.pad_offsets;
    ca.meta = ws.meta;
    ca.expert_of_rb = ws.expert_of_rb;
    ca.pair_info = ws.pair_info;
    ca.row_tok = ws.row_tok;
    ca.slot_w = ws.slot_w;
    ca.slot_of_pair = ws.slot_of_pair;
    ca.S_max = ws.S_max;
    ca.stall_test = ws.route_stall_test;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NB);
    cfg.blockDim = dim3(kCoopWarps * 32);
    cfg.dynamicSmemBytes = route_coop_smem(E);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_coop_kernel, ca);
  }
  const int grid = zero_out ? (NB > zero_grid ? NB : zero_grid) : NB;
  t_route_kernels = router_first ? "router_topk+route_count+route_scan+route_scatter"
                                 : "route_count+route_scan+route_scatter";
  route_count_kernel<<<grid, 256, E * sizeof(int), stream>>>(topk_ids, P, E, k, NB, ws.route_tpb, ws.blk_base,
                                                             ws.err, static_cast<uint4*>(zero_out), zero_bytes / 16);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the scan and the scatter start as programmatic dependents (their launch
  // overlaps the previous kernel; each waits for it before reading)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  e = cudaLaunchKernelEx(&cfg, route_scan_kernel, NB, E, ws.blk_base, ws.counts, ws.offsets, ws.pad_offsets, ws.meta,
                         ws.expert_of_rb, ws.pair_info, ws.row_tok, ws.slot_w);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(NB);
  cfg.blockDim = dim3(kScatterWarps * 32);
  cfg.dynamicSmemBytes = (kScatterWarps + 2) * E * sizeof(int);
  return cudaLaunchKernelEx(&cfg, route_scatter_kernel, static_cast<const int32_t*>(topk_ids), topk_w, P, E, k,
                            ws.route_tpb, static_cast<const int*>(ws.blk_base), static_cast<const int*>(ws.offsets),
                            static_cast<const int*>(ws.pad_offsets), ws.row_tok, ws.slot_w, ws.slot_of_pair);
}

namespace {
__global__ void __launch_bounds__(256) extend_routing_kernel(const int32_t* __restrict__ ids,
                                                             const float* __restrict__ w, int64_t T, int E, int k,
                                                             int n_shared, int32_t* __restrict__ ids_ext,
                                                             float* __restrict__ w_ext) {
  const int kx = k + n_shared;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < T * kx; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / kx;
    const int j = (int)(i % kx);
    // a routed id outside [0, E) would name a shared expert (ids E ..
    // E + n_shared - 1 of the extended problem): -1 keeps it out of range so
    // the routing reports it as a bad id
    int id = E + (j - k);
    if (j < k) {
      id = ids[t * k + j];
      if (id < 0 || id >= E) id = -1;
    }
    ids_ext[i] = id;
    w_ext[i] = j < k ? w[t * k + j] : 1.f;
  }
}
}  // namespace

cudaError_t launch_extend_routing(const int32_t* ids, const float* w, int T, int E, int k, int n_shared,
                                  int32_t* ids_ext, float* w_ext, cudaStream_t stream) {
  const int64_t n = (int64_t)T * (k + n_shared);
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 4096);
  extend_routing_kernel<<<grid > 0 ? grid : 1, 256, 0, stream>>>(ids, w, T, E, k, n_shared, ids_ext, w_ext);
  return cudaGetLastError();
}

namespace {
// Band of a row block: that of the token of its first row (always a routed
// row: padding rows sit at the end of each expert's segment).
__device__ __forceinline__ int block_band(const int* row_tok, int rb, int T, int n_bands) {
  const int tok = row_tok[(int64_t)rb * kRowPad];
  return (int)((int64_t)(tok < 0 ? 0 : tok) * n_bands / T);
}

__global__ void __launch_bounds__(1024) band_order_kernel(const int* __restrict__ meta, const int* __restrict__ row_tok,
                                                          const int* __restrict__ pair_info, int T, int n_bands,
                                                          int* __restrict__ rb_order, int* __restrict__ pair_order) {
  __shared__ int warp_sums[32];
  griddep_wait();
  const int n_rb = meta[0], n_pq = meta[1];
  for (int which = 0; which < 2; ++which) {
    const int n = which ? n_pq : n_rb;
    int* out = which ? pair_order : rb_order;
    // thread t owns the contiguous items [i0, i1): a stable counting sort by band
    const int per = (n + (int)blockDim.x - 1) / (int)blockDim.x;
    const int i0 = min(n, (int)threadIdx.x * per), i1 = min(n, i0 + per);
    auto band = [&](int i) { return block_band(row_tok, which ? pair_info[i] >> 1 : i, T, n_bands); };
    int base = 0;  // items of the lower bands
    for (int b = 0; b < n_bands; ++b) {
      int c = 0;
      for (int i = i0; i < i1; ++i) c += band(i) == b;
      int tot;
      int pos = base + block_exclusive_scan(c, warp_sums, &tot);
      for (int i = i0; i < i1; ++i)
        if (band(i) == b) out[pos++] = i;
      base += tot;
    }
  }
}
}  // namespace

cudaError_t launch_band_order(const Workspace& ws, int T, int n_bands, cudaStream_t stream) {
  if (T <= 0 || n_bands < 1) return cudaSuccess;
  band_order_kernel<<<1, 1024, 0, stream>>>(ws.meta, ws.row_tok, ws.pair_info, T, n_bands, ws.rb_order,
                                           ws.pair_order);
  return cudaGetLastError();
}

cudaError_t launch_router_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                               cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  constexpr int kWarps = 8;
  router_topk_kernel<<<(T + kWarps - 1) / kWarps, kWarps * 32, 0, stream>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

cudaError_t launch_gather_zero(const Workspace& ws, const void* x, const int32_t* topk_ids, int T, int E, int k,
                               int D, void* out, int64_t out_bytes, int grid, cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gather_tokens_kernel, static_cast<const uint4*>(x), topk_ids,
                            static_cast<const int*>(ws.slot_of_pair), static_cast<const int*>(ws.offsets),
                            static_cast<const int*>(ws.pad_offsets), T, E, k, D / 8, static_cast<uint4*>(ws.xg),
                            static_cast<uint4*>(out), out ? (int)(out_bytes / 16 / T) : 0,
                            (ws.l2_policy & 2) ? 1 : 0, static_cast<const uint8_t*>(ws.prefetch_base),
                            ws.prefetch_bytes);
}

}  // namespace moe
