/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) routed Mixture-of-Experts SwiGLU
 * feed-forward forward pass.
 *
 * What it computes ("Prime Flash MoE - Faster MoE Kernels optimized for
 * Blackwell", sec. 1 "The computation"): for every token t and each of its k
 * routed experts e = topk_ids[t][j] with routing weight w = topk_w[t][j],
 *
 *     gate = W1[e][0:H]  x_t        up = W1[e][H:2H] x_t       (W1 output-major)
 *     act  = silu(gate) * up        (fp32, rounded to bf16 before the next GEMM)
 *     y    = W2[e] act
 *     out[t] = sum_j w * y          (the weight is applied before the sum)
 *
 * Layouts (all row-major, contiguous, device memory):
 *     x         [T, D]        bf16
 *     w1        [E, 2H, D]    bf16, rows 0..H-1 of each expert = gate, H..2H-1 = up
 *     w2        [E, D, H]     bf16
 *     topk_ids  [T, k]        int32, each in [0, E); repeats within a token allowed
 *     topk_w    [T, k]        float32
 *     out       [T, D]        bf16, OVERWRITTEN (the library zero-fills it)
 * Requirements: T >= 0 (T == 0 is a no-op), 1 <= k, 1 <= E <= 1024,
 * D % 128 == 0, H % 128 == 0, every pointer 16-byte aligned; the fused
 * pipeline and MXFP8 also need D % 256 == 0 (else MOE_ERR_UNSUPPORTED).
 *
 * Ownership: the caller owns every buffer, including the workspace; the
 * library allocates no device memory.  A workspace serves one call at a time:
 * calls that may run concurrently on the device (different streams) need
 * workspaces of their own.  Calls are asynchronous on `stream` (a
 * cudaStream_t passed as void*, NULL = legacy default stream) and may be
 * captured in CUDA graphs.  Host-detectable errors are returned immediately;
 * errors found on the device (an expert id out of range, a bounded wait that
 * ran out) are recorded in the workspace's status words, are sticky, and are
 * returned and cleared by moe_ffn_sync_status().  No C++ exception crosses
 * this interface.
 */
#ifndef MOE_FFN_H_
#define MOE_FFN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, negative size, k < 1 ... */
  MOE_ERR_UNSUPPORTED = 2,         /* shape or dtype/pipeline combination not built */
  MOE_ERR_MISALIGNED = 3,          /* a pointer is not 16-byte aligned */
  MOE_ERR_BAD_ROUTING = 4,         /* device saw an expert id outside [0, E) */
  MOE_ERR_WORKSPACE_TOO_SMALL = 5,
  MOE_ERR_DEVICE_TIMEOUT = 6,      /* a bounded device wait ran out; output invalid */
  MOE_ERR_CUDA = 7                 /* a CUDA runtime call failed */
} moe_status_t;

typedef enum { MOE_BF16 = 0, MOE_MXFP8 = 1, MOE_MXFP4W = 2, MOE_NVFP4 = 3 } moe_dtype_t;

/* MOE_FUSED: one GEMM kernel per call, the activation never leaves the SM
 *            ("Prime Flash MoE" sec. 2 "Trick 2", sec. 4).
 * MOE_SPLIT: gather, up-projection + SwiGLU writing the activation once, then
 *            the down projection with C = 1 ("Prime Flash MoE" sec. 6). */
typedef enum { MOE_FUSED = 0, MOE_SPLIT = 1 } moe_pipeline_t;

/* Bytes of workspace moe_ffn_forward needs for this problem.  Returns 0 for
 * an invalid shape.  The first 64 bytes are the status words: zero them once
 * before first use (moe_ffn_workspace_init does so). */
size_t moe_ffn_workspace_size(int T, int E, int D, int H, int k, int dtype, int pipeline);

/* Zero the workspace's status words (asynchronous on stream). */
moe_status_t moe_ffn_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* The forward pass described above.  x_sf, w1_sf, w2_sf are the MXFP8 scale
 * arrays and must be NULL for MOE_BF16.
 *
 * MOE_MXFP8 ("Prime Flash MoE" sec. 7; both pipelines): x, w1, w2 hold OCP
 * e4m3 codes (one byte per element, same shapes as above); every 32
 * consecutive elements along the contiguous (reduction) dimension share one
 * ue8m0 scale byte s (value 2^(s-127)).  x_sf is row-major [T, D/32] (4-byte
 * aligned); w1_sf and w2_sf are the weight scales already repacked by
 * moe_ffn_prepare_mxfp8_weights.  The activation is requantized to MXFP8
 * (per 32 along H) between the two GEMMs; out stays bf16.
 *
 * MOE_MXFP4W (split pipeline only; MOE_ERR_UNSUPPORTED for MOE_FUSED): x and
 * its scales as for MOE_MXFP8; w1 [E, 2H, D/2] and w2 [E, D, H/2] hold MXFP4
 * weights, E2M1 codes packed two per byte along the reduction dimension
 * (element 2j in bits 0..3 of byte j), one ue8m0 scale per 32 elements
 * (the routed-weight format of "GC-MoE on SM120" sec. 2.2), scales repacked by
 * moe_ffn_prepare_mxfp8_weights as for MOE_MXFP8.  The codes stay 4-bit in
 * HBM: the GEMMs read them with 4-bit tensor maps and multiply them as the
 * E2M1 operand of kind::mxf8f6f4 ("Porting Block-Scaled GEMM Kernels from
 * Blackwell to Rubin" sec. 2.1, 2.3).  w1 and w2 must be 32-byte aligned
 * (MOE_ERR_MISALIGNED otherwise). */
moe_status_t moe_ffn_forward(const void* x, const void* x_sf, const void* w1, const void* w1_sf, const void* w2,
                             const void* w2_sf, const int32_t* topk_ids, const float* topk_w, void* out, int T, int E,
                             int D, int H, int k, int dtype, int pipeline, void* workspace, size_t workspace_bytes,
                             void* stream);

/* NVFP4 operands ("Porting Block-Scaled GEMM Kernels from Blackwell to
 * Rubin" sec. 1.2: one scale per 16 elements along K; sec. 6.1: UE4M3 block
 * scales paired with fp32 global scales, per expert in MoE kernels): every
 * element is an E2M1 code c (packed two per byte along K, element 2j in bits
 * 0..3 of byte j), its 16-element block carries a non-negative E4M3 scale s,
 * and its tensor (each expert, for the weights) an fp32 global scale G: the
 * value is e2m1(c) * e4m3(s) * G.  act between the GEMMs is requantized the
 * same way with the global scale act_gs (per 16: s = the E4M3 code nearest to
 * amax / (6 act_gs), codes = the E2M1 values nearest to v / (e4m3(s) act_gs),
 * ties to even, saturating at 448 and 6).  All four are device pointers:
 *   x_gs [1], w1_gs [E], w2_gs [E], act_gs [1]  float32, 4-byte aligned. */
typedef struct {
  const float* x_gs;
  const float* w1_gs;
  const float* w2_gs;
  const float* act_gs;
} moe_ffn_nvfp4_scales_t;

/* One-time repacking of NVFP4 weight scales into the 512-byte tiles the
 * kernels copy into tensor memory (128 rows x 4 scales, i.e. 64 elements of K
 * per tile).  w1_sf [E, 2H, D/16] and w2_sf [E, D, H/16] row-major e4m3 bytes
 * (4-byte aligned); w1_sf_packed (E*2H*D/16 bytes) and w2_sf_packed (E*D*H/16
 * bytes) 16-byte aligned caller buffers.  D and H multiples of 256. */
moe_status_t moe_ffn_prepare_nvfp4_weights(const void* w1_sf, const void* w2_sf, void* w1_sf_packed,
                                           void* w2_sf_packed, int E, int D, int H, void* stream);

/* The forward pass with NVFP4 operands, split pipeline: x [T, D/2] packed
 * codes with x_sf [T, D/16] e4m3 scales (row-major), W1 [E, 2H, D/2] and
 * W2 [E, D, H/2] packed codes with scales repacked by
 * moe_ffn_prepare_nvfp4_weights, the global scales in *gs; out [T, D] bf16,
 * overwritten.  GEMMs on tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
 * with both operands packed in shared memory.  Requires D and H multiples of
 * 256; workspace of moe_ffn_workspace_size(..., MOE_NVFP4, MOE_SPLIT).
 * Errors as moe_ffn_forward. */
moe_status_t moe_ffn_forward_nvfp4(const void* x, const void* x_sf, const void* w1, const void* w1_sf, const void* w2,
                                   const void* w2_sf, const moe_ffn_nvfp4_scales_t* gs, const int32_t* topk_ids,
                                   const float* topk_w, void* out, int T, int E, int D, int H, int k,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* The forward pass from and to HOST memory (the library's own entry point:
 * "Prime Flash MoE" sec. 8 times the kernels with inputs resident on the GPU
 * and defines no host-buffer call; each chunk computes what moe_ffn_forward
 * does, the operation of sec. 1).  x (and x_sf), topk_ids and
 * topk_w are read from host memory, out is written to host memory; the
 * weights (and their scales) and the workspace are device memory as for
 * moe_ffn_forward.  The tokens are processed in chunks of chunk_tokens
 * (0: automatic: the whole problem up to 8192 tokens, else T / 8 rounded up
 * to a multiple of 128, within [4096, 16384]; the last chunk may be shorter;
 * with eight chunks or more the first and the last are a quarter chunk, so
 * the copy in and the copy out that nothing overlaps are short): while chunk c runs on `stream`, chunk c + 1
 * is copied in and chunk c - 1 copied out on two copy streams of the library,
 * through two sets of device staging buffers in the workspace.  Each chunk is
 * one moe_ffn_forward call, so each output row is exactly what
 * moe_ffn_forward gives for that token.
 *   Layouts as moe_ffn_forward (dtype MOE_BF16, MOE_MXFP8 or MOE_MXFP4W).
 *   Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister):
 *   copies from or to pageable memory are correct but block the calling
 *   thread and do not overlap the computation.
 *   workspace: moe_ffn_host_workspace_size(T, chunk_tokens, ...) bytes of
 *   device memory; its first bytes are the forward workspace of a chunk, so
 *   moe_ffn_sync_status(workspace) reads the call's status words.
 * Asynchronous on stream: the work queued on stream before the call comes
 * first, and everything the call does (copies included) completes before the
 * work queued on stream after it; the host buffers must stay valid and out
 * unread until then.  Calls on one device are serialized on the host (one
 * mutex) while they enqueue; their device work is ordered by `stream`.  Not
 * for stream capture: the library's copy streams are not part of a graph
 * (capture moe_ffn_forward with the caller's own copies instead).
 * Errors as moe_ffn_forward; MOE_ERR_INVALID_ARG for a negative
 * chunk_tokens or a NULL host pointer. */
size_t moe_ffn_host_workspace_size(int T, int chunk_tokens, int E, int D, int H, int k, int dtype, int pipeline);
moe_status_t moe_ffn_forward_host(const void* x_host, const void* x_sf_host, const void* w1, const void* w1_sf,
                                  const void* w2, const void* w2_sf, const int32_t* topk_ids_host,
                                  const float* topk_w_host, void* out_host, int T, int E, int D, int H, int k,
                                  int dtype, int pipeline, int chunk_tokens, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* The router step upstream of the path ("Prime Flash MoE" sec. 1 takes each
 * token's k experts and their weights, which sum to one, as given; the
 * workloads produce them from per-(token, expert) logits: the k largest, with
 * a softmax over just those k).
 *   logits    [T, E] float32 (4-byte aligned; a NaN logit is read as -inf)
 *   topk_ids  [T, k] int32 output: the k experts with the largest logits, in
 *             order of decreasing logit, ties going to the lower expert id
 *   topk_w    [T, k] float32 output: w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0)
 *             over the selected logits (l_0 the largest), computed in fp32;
 *             every weight is 1/k when l_0 is -inf
 * Requires 1 <= k <= E <= 1024.  Device pointers, asynchronous on stream.
 * The ids are a deterministic function of the logits (no atomics). */
moe_status_t moe_ffn_router_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                                 void* stream);

/* moe_ffn_forward starting from router logits: the router of
 * moe_ffn_router_topk runs over each token first (a launch of one warp per
 * token, right before the routing launch; see MOE_OPT_ROUTER_FUSED) and
 * writes topk_ids / topk_w (caller arrays [T, k], outputs here); then the
 * forward pass proceeds exactly as moe_ffn_forward with those ids and
 * weights.  Same workspace, requirements
 * and errors as moe_ffn_forward, plus k <= E and router_logits [T, E] float32
 * (4-byte aligned). */
moe_status_t moe_ffn_forward_logits(const void* x, const void* x_sf, const void* w1, const void* w1_sf,
                                    const void* w2, const void* w2_sf, const float* router_logits,
                                    int32_t* topk_ids, float* topk_w, void* out, int T, int E, int D, int H, int k,
                                    int dtype, int pipeline, void* workspace, size_t workspace_bytes, void* stream);

/* Optional extras of a forward call (moe_ffn_forward_ex); zero-initialize
 * and set what is needed.
 *   swiglu_limit   > 0: the clamped SwiGLU of the gpt-oss-style expert
 *                  ("Porting Block-Scaled GEMM Kernels from Blackwell to
 *                  Rubin" sec. 5.3): gate = min(gate, limit),
 *                  up = min(max(up, -limit), limit), then silu(gate) * up.
 *                  0: the plain SwiGLU.
 *   n_shared       >= 0 shared experts ("GC-MoE on SM120" sec. 4.7: every
 *                  token uses a shared expert): experts E .. E + n_shared - 1
 *                  of w1 / w2 (and of their MXFP8 scales), stored after the E
 *                  routed ones, are added for every token with weight 1, in
 *                  the same launches as the routed experts (each token gets
 *                  k + n_shared pairs).  Requires E + n_shared <= 1024.
 *   router_logits  optional [T, E] float32: the call starts from router
 *                  logits as moe_ffn_forward_logits does; topk_ids / topk_w
 *                  are then outputs. */
typedef struct {
  float swiglu_limit;
  int n_shared;
  const float* router_logits;
} moe_ffn_extras_t;

/* Workspace bytes of moe_ffn_forward_ex with n_shared shared experts (equal
 * to moe_ffn_workspace_size when n_shared == 0); 0 for an invalid shape. */
size_t moe_ffn_workspace_size_ex(int T, int E, int D, int H, int k, int n_shared, int dtype, int pipeline);

/* moe_ffn_forward with the extras above (extras may be NULL: then it is
 * moe_ffn_forward).  topk_ids / topk_w [T, k] hold the routed experts (or
 * receive them, with router_logits); the workspace must hold
 * moe_ffn_workspace_size_ex bytes.  Same requirements, layouts and errors as
 * moe_ffn_forward; MOE_ERR_INVALID_ARG for a negative limit or n_shared. */
moe_status_t moe_ffn_forward_ex(const void* x, const void* x_sf, const void* w1, const void* w1_sf, const void* w2,
                                const void* w2_sf, int32_t* topk_ids, float* topk_w, void* out, int T, int E, int D,
                                int H, int k, int dtype, int pipeline, const moe_ffn_extras_t* extras,
                                void* workspace, size_t workspace_bytes, void* stream);

/* One-time repacking of MXFP8 weight scales into the 512-byte tile layout the
 * kernels copy into tensor memory ("Prime Flash MoE" sec. 7 "Scales are
 * piped through tensor memory"; 128 rows x 4 K-scales per tile).
 *   w1_sf [E, 2H, D/32] and w2_sf [E, D, H/32] row-major ue8m0 (4-byte aligned);
 *   w1_sf_packed (E*2H*D/32 bytes) and w2_sf_packed (E*D*H/32 bytes) are
 *   caller buffers, 16-byte aligned, written asynchronously on stream. */
moe_status_t moe_ffn_prepare_mxfp8_weights(const void* w1_sf, const void* w2_sf, void* w1_sf_packed,
                                           void* w2_sf_packed, int E, int D, int H, void* stream);

/* MXFP4 expert weights for the MXFP8 path.  An MXFP4 weight is an E2M1 code
 * (1 sign, 2 exponent bits with bias 1, 1 mantissa bit: magnitudes 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6) with one ue8m0 scale per 32 consecutive elements along the
 * reduction dimension, the routed-weight format of "GC-MoE on SM120" sec. 2.2
 * (scale formats).  This call widens the codes once, at weight-load time, to
 * e4m3 codes of the same values (exact: every E2M1 value is an e4m3 value);
 * the scale arrays stay as they are and go through
 * moe_ffn_prepare_mxfp8_weights, and moe_ffn_forward then runs with
 * MOE_MXFP8.  The weights then occupy one byte per element in HBM, not half;
 * MOE_MXFP4W runs the packed codes as they are, at half a byte per element.
 *   w_fp4   n_elems/2 bytes, two codes per byte along the contiguous dimension:
 *           element 2j in bits 0..3 of byte j, element 2j+1 in bits 4..7;
 *           16-byte aligned (W1 [E, 2H, D/2] and W2 [E, D, H/2] row-major)
 *   w_e4m3  n_elems bytes output, element i in byte i, 16-byte aligned
 *           (W1 [E, 2H, D], W2 [E, D, H])
 * n_elems a multiple of 32 (0 does nothing).  Device pointers, asynchronous
 * on stream; the input is only read.  Errors: MOE_ERR_INVALID_ARG (n_elems
 * negative or not a multiple of 32, NULL pointer), MOE_ERR_MISALIGNED,
 * MOE_ERR_CUDA (launch failure). */
moe_status_t moe_ffn_widen_mxfp4_weights(const void* w_fp4, int64_t n_elems, void* w_e4m3, void* stream);

/* Test hook: the MXFP8 requantization the up-projection epilogue applies to
 * act, run on n fp32 values (n % 32 == 0): per 32 values, scale exponent
 * e = ceil(log2(amax/448)) (0 for amax == 0, at least -127), scale byte
 * sf = e + 127, codes q = e4m3_rne_satfinite(v * 2^-e).  Device pointers. */
moe_status_t moe_ffn_debug_mx_quantize(const float* in, int64_t n, uint8_t* q, uint8_t* sf, void* stream);

/* The routing permutation alone ("Prime Flash MoE" sec. 3 and 6: tokens are
 * processed in per-expert sorted order).  Writes, into caller device arrays:
 *   counts[E]         pairs routed to each expert
 *   offsets[E+1]      exclusive prefix sum of counts
 *   slot_of_pair[T*k] offsets[e] + number of earlier pairs (p' < p, p = t*k+j)
 *                     routed to the same expert: a stable counting sort.
 * Any output pointer may be NULL.  Bit-exact by construction (no
 * order-dependent atomics).  Uses the same workspace as moe_ffn_forward. */
moe_status_t moe_ffn_route(const int32_t* topk_ids, const float* topk_w, int T, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* slot_of_pair, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Capacity, in padded slots, of the padded routing tables of a problem:
 * S_max = T*k + min(E, T*k)*127 rounded up to a multiple of 128 (every
 * expert's segment padded to whole 128-row blocks fits in it).  0 for an
 * invalid shape. */
int64_t moe_ffn_route_padded_slots(int T, int E, int k);

/* The padded routing tables the grouped GEMMs consume, written to caller
 * arrays for bit-exact checks.  "Prime Flash MoE" sec. 3 and sec. 6: the
 * routed rows are sorted by expert and every expert's segment is padded to
 * whole 128-row blocks, so a row block never straddles two experts; the
 * padding rows are dropped in the epilogues.
 *   pad_offsets  [E+1]  exclusive scan of counts[e] rounded up to 128
 *   expert_of_rb [S_max/128]  expert of row block rb, for rb < n_blocks[0]
 *   pair_info    [S_max/128]  the CTA-pair kernels' schedule, for i < n_blocks[1]:
 *                       (first row block << 1) | (1 if the next row block
 *                       belongs to the same expert); pairs cover each expert's
 *                       blocks in order, two at a time
 *   row_tok      [S_max]  token t of padded slot s (its pair t*k+j sits at
 *                       pad_offsets[e] + its rank within expert e), -1 for
 *                       padding; entries from pad_offsets[E] on are unspecified
 *   slot_w       [S_max]  topk_w[t, j] of that pair, 0 for padding
 *   n_blocks     [2]   number of row blocks (pad_offsets[E] / 128), number of pairs
 * S_max = moe_ffn_route_padded_slots(T, E, k).  All arrays are device memory
 * owned by the caller; the workspace is sized as for moe_ffn_route.  Requires
 * T >= 1.  Errors: MOE_ERR_INVALID_ARG (shape or a null pointer),
 * MOE_ERR_WORKSPACE_TOO_SMALL, MOE_ERR_CUDA; a bad id is reported through
 * moe_ffn_sync_status. */
moe_status_t moe_ffn_route_padded(const int32_t* topk_ids, const float* topk_w, int T, int E, int k,
                                  int32_t* pad_offsets, int32_t* expert_of_rb, int32_t* pair_info, int32_t* row_tok,
                                  float* slot_w, int32_t* n_blocks, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* The routing permutation, for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point.
 *
 * Same results as moe_ffn_route, but the scratch lives in a fixed 6 MiB
 * device array inside this library instead of a caller workspace, for callers
 * that cannot call cudaMalloc or hand over a buffer of their own (graph
 * capture under an allocator that forbids new allocations, runtimes whose
 * device memory is planned ahead of time).  Inputs and the output arrays are
 * still the caller's.  Limits: T*k <= 131072 pairs and E <= 1024; larger
 * problems return MOE_ERR_WORKSPACE_TOO_SMALL without launching anything.
 * status_bits (optional, device int32) receives the call's device error bits:
 * 0 when the call succeeded; bit 0 (value 1) when an expert id was outside
 * [0, E) (those pairs are dropped); bit 1 (value 2) when a bounded device wait
 * ran out (problems of more than 8192 pairs route in one cooperative launch
 * whose blocks meet at a grid barrier): counts, offsets and slot_of_pair are
 * then invalid.
 * The first call on each device looks up the array's device address (setup
 * done once per device, with that device current); make that first call
 * before any stream capture.  The call allocates nothing.  All calls on a
 * device share the array and it keeps the last call's contents: calls that
 * overlap on the GPU (several streams or host threads at once) race and give
 * wrong results. */
moe_status_t moe_ffn_route_noalloc(const int32_t* topk_ids, const float* topk_w, int T, int E, int k,
                                   int32_t* counts, int32_t* offsets, int32_t* slot_of_pair, int32_t* status_bits,
                                   void* stream);

/* Synchronize `stream`, then return (and clear) the device status recorded in
 * the workspace since the last call: MOE_OK, MOE_ERR_BAD_ROUTING or
 * MOE_ERR_DEVICE_TIMEOUT.  MOE_ERR_CUDA if synchronization itself failed. */
moe_status_t moe_ffn_sync_status(void* workspace, void* stream);

/* Upper bound, in nanoseconds, of every wait inside the kernels (default 2 s).
 * Process-wide; affects launches made after the call. */
void moe_ffn_set_wait_limit_ns(uint64_t ns);

/* Process-wide tuning options (affect calls made afterwards).
 *   MOE_OPT_GATHER  0 (default): a gather kernel first materializes x in
 *                   sorted order (16-byte vector copies) and the up kernel
 *                   reads plain 128-row tiles of it ("Prime Flash MoE" sec. 6);
 *                   1: the up-projection kernel fetches its token rows itself
 *                   with TMA tile::gather4, four rows per instruction (sec. 3
 *                   "For the tokens: TMA gathers them too").  Measured on
 *                   GB300, option 1 makes the up kernel 2-3.5x slower.
 *                   2: four extra warps of the up-projection kernel copy the
 *                   token rows from x with 16-byte cp.async into the
 *                   swizzled operand tile (no gathered copy of x in HBM).
 *   MOE_OPT_L2_PREFETCH  0..64 (default 0): how many K-blocks ahead of the
 *                   shared-memory ring the GEMM producers prefetch operand
 *                   tiles into L2 (cp.async.bulk.prefetch.tensor); 0 = off.
 *                   Measured on GB300, prefetching slowed every workload.
 *   MOE_OPT_TEST_STALL  0 (default), 1 or 2: test hooks for failure
 *                   detection.  With 1, each GEMM kernel's MMA issuer first
 *                   waits on a barrier that nothing ever arrives on; the wait
 *                   runs out after the wait limit, the kernel records
 *                   MOE_ERR_DEVICE_TIMEOUT and exits cleanly (no fault, no
 *                   hang), so the status path can be tested on a GPU.  With 2,
 *                   one block of the one-launch routing leaves before its
 *                   first grid barrier; the other blocks' waits run out, the
 *                   routing records MOE_ERR_DEVICE_TIMEOUT and leaves tables
 *                   with no row blocks, so the GEMMs that follow do nothing.
 *                   After a timeout, moe_ffn_sync_status (which clears the
 *                   status words, including the routing barrier's state) must
 *                   be called before the workspace is used again.
 *   MOE_OPT_UP_PAIRS  0 (default) or 1: with 1 (and MOE_OPT_GATHER 0) each
 *                   tile of the bf16 up-projection takes two row blocks of
 *                   one expert against one weight tile ("Prime Flash MoE"
 *                   sec. 5 "BPC and CPC").  Measured on GB300 it is 7-17%
 *                   slower (its accumulators fill TMEM, so the epilogue no
 *                   longer overlaps the next tile's MMAs).
 *   MOE_OPT_DYNAMIC_TILES  0, 1 or 2 (default): with 1 the split pipeline's
 *                   bf16 GEMM kernels take their tiles from a global atomic
 *                   counter (CTAs that finish early take more work; "Porting
 *                   Block-Scaled GEMM Kernels" sec. 7 hands out work ids from
 *                   an atomic counter); 0 = static round-robin; 2 = dynamic
 *                   only when the problem has fewer than about eight waves of
 *                   up-projection tiles.  Measured on GB300: 2% faster at
 *                   decode, 3-5% slower at prefill and large_skewed.
 *   MOE_OPT_TILE_COLS  0 (default: automatic), 128 or 256: output columns per
 *                   tile of the bf16 split GEMMs (up: 64+64 or 128+128 gate/up
 *                   rows; down: 128 or 256 columns of D).  Automatic picks
 *                   128-wide up tiles when the 256-wide ones would fill the
 *                   GPU fewer than about eight times, and 256-wide down tiles
 *                   whenever D % 256 == 0.
 *   MOE_OPT_SWAP_AB  0 (default) or 1: with 1 the bf16 split GEMMs with
 *                   256-row weight tiles run the last row block of an expert
 *                   as a swap-AB tile when it holds at most 112 routed rows:
 *                   the weight rows become the MMA's M = 128 side and the
 *                   routed rows its N (rounded up to 16), so padding rows
 *                   cost no tensor-core work.  Measured on GB300: 1-3% slower
 *                   at prefill, large_skewed and decode (those GEMMs are
 *                   bound by operand traffic, not by tensor-core work).
 *   MOE_OPT_FUSED_CLUSTER  1 (default: automatic size), 2, 4, 8 or 0: the
 *                   bf16 fused pipeline runs on thread-block clusters of C
 *                   CTAs (D % (256 C) == 0, H/C a multiple of 32): each CTA
 *                   computes H/C columns of act for the cluster's row block,
 *                   the slices meet in an L2-resident ring, and each CTA
 *                   reduces D/C finished output columns into out in bf16.
 *                   1 picks C from the shape and the number of clusters that
 *                   fit on the device; 2, 4 or 8 request that size (automatic
 *                   when it does not apply).  With 0 (or a shape no C fits)
 *                   the fused pipeline splits H over CTAs and sums partial
 *                   rows in an fp32 buffer.
 *   MOE_OPT_PAIR_MMA  2 (default: automatic), 1 or 0: with 1 the bf16 split
 *                   pipeline's up and down GEMMs run on CTA pairs (two-CTA
 *                   clusters sharing one tcgen05 MMA of 256 rows,
 *                   cta_group::2): each CTA loads half of every weight tile, a
 *                   third fewer operand bytes per FLOP.  Two row blocks of one
 *                   expert form a tile; an expert with an odd number of row
 *                   blocks pays one idle half.  2 uses pairs unless the
 *                   problem is decode-sized (fewer than about eight waves of
 *                   up tiles).  Measured on GB300: prefill 0.360 -> 0.335 ms,
 *                   large_skewed 7.47 -> 6.83 ms, decode unchanged.
 *   MOE_OPT_PAIR_SWAP  0 (default) .. 256: with CTA pairs, a down-
 *                   projection tile whose two row blocks hold at most this
 *                   many routed rows (an expert's odd last block, or a small
 *                   expert) runs swap-AB: the 256 weight rows are the MMA's M
 *                   side and the routed rows, rounded up to 16, its N, so the
 *                   idle or padded rows of the pair cost no tensor-core work.
 *                   Measured on GB300 at prefill: down kernel 0.115 ms with
 *                   0, 0.121 with 128, 0.141 with 256 (the transposing
 *                   epilogue costs more than the MMA work saved; the kernel
 *                   is bound by streaming the weights).
 *   MOE_OPT_ROUTE_COOP  1 (default) or 0: routing of problems too large for
 *                   the single-block kernel (more than 8192 pairs or 256
 *                   experts) runs as ONE cooperative launch whose blocks meet
 *                   at two bounded grid barriers (the workspace's status
 *                   words hold the barrier state), when all its blocks fit on
 *                   the device at once; 0 (or too many blocks) uses three
 *                   launches (histograms, scans, scatter).
 *   MOE_OPT_OUT_L2_HINT  0 (default), 1 or 2: the bulk reductions into out
 *                   carry an L2 evict_last hint, so that an out of about the
 *                   L2's size may stay resident while the weights stream past
 *                   it instead of being read and written back for each of a
 *                   token's k contributions.  1 applies it when out is at
 *                   most 160 MiB, 2 always, 0 never.  Measured on GB300 at
 *                   mxfp8 (out 134 MB): split 2.12 -> 2.10 ms, fused 2.28 ->
 *                   2.34 ms; large_skewed unchanged.
 *   MOE_OPT_GATHER_BLOCKS  1..16 (default 8): blocks per SM of the row-gather
 *                   kernels (bytes in flight against HBM latency).  Measured
 *                   on GB300 at large_skewed: 4 -> 0.94 ms, 8 -> 0.87 ms.
 *   MOE_OPT_L2_POLICY  0 (default) .. 3, bits: 1 = the CTA-pair GEMMs load
 *                   weight tiles (read by one pair each) with an L2
 *                   evict_first policy; 2 = the row gather stores the
 *                   gathered rows (read right after by the up projection)
 *                   with evict_last.
 *   MOE_OPT_ROUTER_FUSED  0 (default) or 1: with router logits, 1 runs the
 *                   router inside the routing launch when that launch is a
 *                   single block (small problems), else as its own launch of
 *                   one warp per token; 0 always launches it separately.
 *                   Measured on GB300 at decode from logits: 0.422 ms fused,
 *                   0.413 ms separate (one block has too few warps for the
 *                   tokens' logits).
 *   MOE_OPT_PREFETCH_MB  0 (default) .. 1024: while the routing launch runs
 *                   (its latency leaves HBM idle), the bf16 row-gather's
 *                   blocks ask L2 for the first this-many MiB of w1, the
 *                   weights of the up projection's first tiles.  Measured on
 *                   GB300: decode 0.410 ms with 0, 0.408 with 32, 0.409 with
 *                   64; prefill 0.345 with 0, 0.348 with 96 (no gain, off).
 *   MOE_OPT_WIDE_UP  0 (default) or 1: with CTA pairs, 1 runs the up
 *                   projection in 512-column tiles (two 256-column halves of
 *                   the pair's accumulator, the act tiles j and j+1 of one
 *                   block pair) whose halves the epilogue frees one after the
 *                   other, so the next tile's MMAs start on half 0 while half
 *                   1 is still being read: a quarter fewer operand bytes per
 *                   FLOP than 256-column tiles, four 48 KB stages instead of
 *                   six 32 KB ones.
 *   MOE_OPT_TILE_M  0 (default: automatic, 64 when the routed pairs are at
 *                   most 64 per expert on average), 64 or 128: rows per tile
 *                   of the single-CTA split GEMMs (the CTA-pair kernels always
 *                   take 128 per CTA).  64-row tiles (tcgen05.mma M = 64)
 *                   halve the token stage so that more weight stages fit in
 *                   shared memory; a 128-row block's second half is skipped
 *                   when it holds no routed rows.  Measured on GB300 at
 *                   decode (16 rows per expert): step 0.410 ms with 128,
 *                   0.387 with 64 (up kernel 0.266 -> 0.250 ms, 0.97 of the
 *                   measured HBM copy rate).
 *   MOE_OPT_FUSED_DSMEM  0 (default) or 1: with 1 the bf16 fused pipeline on
 *                   clusters keeps act in shared memory (each CTA's slice of
 *                   H / C columns; the producer warp of every CTA copies the
 *                   other CTAs' K tiles of GEMM2's A operand from their shared
 *                   memory into its own pipeline stages) whenever a cluster
 *                   size gives slices of 64 to 256 columns in steps of 64;
 *                   0, or any other shape, exchanges act through an
 *                   L2-resident ring in global memory instead.  Measured on
 *                   GB300 (fused GEMM kernel): decode 1.19 against 0.41 ms,
 *                   prefill 0.85 against 0.37 ms, large_skewed 19.4 against
 *                   7.1 ms (three pipeline stages where the ring kernel has
 *                   four, and every CTA copies (C - 1) / C of the act K tiles
 *                   once per 256 output columns); a first form in which each
 *                   owner pushed its tiles into the other CTAs' stages by
 *                   shared-to-shared bulk copies, with a handshake per tile,
 *                   measured 1.26 / 0.66 / 15.9 ms.
 *   MOE_OPT_HALF_PAIR_M128  0 (default) or 1: with 1, in the CTA-pair down
 *                   projection, an expert's odd last row block (a pair
 *                   without its second block) runs as one M = 128 pair MMA
 *                   with 64 of its rows in each CTA; 0 runs it at M = 256 with
 *                   the odd CTA repeating the first block and storing nothing.
 *                   Measured on GB300, same box: prefill down kernel 0.117 /
 *                   0.123 ms with 1 against 0.115 / 0.121 with 0, large_skewed
 *                   2.78 against 2.73 ms (the kernel is not bound by MMA work).
 *   MOE_OPT_ROUTE_SMALL_PAIRS  0 .. 1048576 (default 8192): problems of at
 *                   most this many routed pairs (and at most 256 experts)
 *                   route in one single-block launch instead of the
 *                   cooperative one.
 *   MOE_OPT_DOWN_BANDS  1 (default: off), 0 (automatic: bands of at most
 *                   48 MiB of out when out exceeds 64 MiB) or 2 .. 64: the
 *                   split pipeline's down projection (CTA-pair bf16 kernel,
 *                   MXFP8 kernel) processes its tiles ordered by the token band
 *                   of their first row (band = token * bands / T; stable, so
 *                   expert order within a band), so that its reductions into
 *                   an out larger than L2 meet the rows of one band at a time
 *                   in L2; the weights are then read once per band.
 *   MOE_OPT_DOWN_EPI8  1 (default) or 0: eight epilogue warps in the
 *                   CTA-pair down projection (two per TMEM lane quadrant, one
 *                   per half row: each reads its 128 accumulator columns into
 *                   registers and releases the accumulator before it stages
 *                   and reduces them; five pipeline stages), or four (one per
 *                   quadrant, each row staged and reduced as two half rows in
 *                   turn while the accumulator is held; six stages).
 *   MOE_OPT_MX_PAIRS  0 (default: off), 1 or 2 (automatic): the MXFP8 split
 *                   pipeline's GEMMs (e4m3 weights) on CTA pairs
 *                   (tcgen05 cta_group::2, M = 256 rows of two row blocks of
 *                   one expert, each CTA holding half of the weight tile; the
 *                   A scales of a CTA's rows and the B scales of all 256
 *                   columns copied into each CTA's tensor memory); automatic
 *                   uses them unless the problem is decode-sized (fewer than
 *                   8 x SMs row-block x column tiles).  Measured on GB300,
 *                   mxfp8 workload, same box: step 2.20 ms with pairs against
 *                   2.13 ms without (up kernel 1.30 against 1.22 ms, down
 *                   0.79-0.81 against 0.78-0.80 ms): off.
 *   MOE_OPT_UP_SWAP  1 (default) or 0: in the CTA-pair up projection an
 *                   expert's odd last row block (a half pair) runs with the
 *                   operands swapped: 256 W1 rows ([gate 64 | up 64] of each
 *                   CTA's 64 act columns) as the MMA's M side and the block's
 *                   routed rows, rounded up to 16, as its N side, so the
 *                   tensor cores do 256 x ns rather than 256 x 256 per K
 *                   step; 0 runs it as a full pair whose odd CTA repeats the
 *                   block and stores nothing.
 *   MOE_OPT_ROUTE_TPB  0 (default: 256), 64, 128 or 256: tokens per block of
 *                   the multi-block routing (the cooperative launch and the
 *                   three-launch fallback); set before sizing the workspace
 *                   (the per-block count table takes blocks x E ints).
 *   MOE_OPT_MX_SWAP  0 (default: off), 1 or 2 (automatic): the MXFP8 split
 *                   pipeline's GEMMs (e4m3 or MXFP4 weights) with the operands
 *                   swapped: 128 weight rows as the MMA's M side and a row
 *                   block's routed rows, rounded up to 16, as its N side (up:
 *                   gate and up in two accumulators, so each act column's pair
 *                   shares a TMEM lane).  Automatic: at most 64 routed rows
 *                   per live expert on average and k <= 8.  Measured on GB300,
 *                   decode shape with MXFP4 weights: step 0.195 ms against
 *                   0.174 (up kernel 0.113 against 0.102, down 0.074 against
 *                   0.065): off.
 *   MOE_OPT_HOST_RAMP  1 (default) or 0: moe_ffn_forward_host with eight
 *                   chunks or more makes its first and last chunks a quarter
 *                   chunk; 0 keeps every chunk full (the last one ragged).
 *   (MOE_OPT_L2_POLICY measured at prefill: 0.343 ms with 0, 0.349 with 1,
 *                   0.342 with 2, 0.348 with 3: no gain, off.) */
typedef enum {
  MOE_OPT_GATHER = 0,
  MOE_OPT_L2_PREFETCH = 1,
  MOE_OPT_TEST_STALL = 2,
  MOE_OPT_UP_PAIRS = 3,
  MOE_OPT_DYNAMIC_TILES = 4,
  MOE_OPT_TILE_COLS = 5,
  MOE_OPT_SWAP_AB = 6,
  MOE_OPT_FUSED_CLUSTER = 7,
  MOE_OPT_PAIR_MMA = 8,
  MOE_OPT_PAIR_SWAP = 9,
  MOE_OPT_ROUTE_COOP = 10,
  MOE_OPT_OUT_L2_HINT = 11,
  MOE_OPT_GATHER_BLOCKS = 12,
  MOE_OPT_L2_POLICY = 13,
  MOE_OPT_ROUTER_FUSED = 14,
  MOE_OPT_PREFETCH_MB = 15,
  MOE_OPT_WIDE_UP = 16,
  MOE_OPT_TILE_M = 17,
  MOE_OPT_FUSED_DSMEM = 18,
  MOE_OPT_HALF_PAIR_M128 = 19,
  MOE_OPT_ROUTE_SMALL_PAIRS = 20,
  MOE_OPT_DOWN_BANDS = 21,
  MOE_OPT_DOWN_EPI8 = 22,
  MOE_OPT_MX_PAIRS = 23,
  MOE_OPT_UP_SWAP = 24,
  MOE_OPT_ROUTE_TPB = 25,
  MOE_OPT_MX_SWAP = 26,
  MOE_OPT_HOST_RAMP = 27
} moe_option_t;
moe_status_t moe_ffn_set_option(int option, long long value);

/* Per-stage timing of later moe_ffn_forward calls (a benchmarking aid, off by
 * default; process-wide state, for single-threaded use).  While enabled, each call records CUDA events on its stream
 * between its stages; the split pipeline's stages are
 *   0 routing (three kernels), 1 gather + zero-fill of out,
 *   2 up-projection + SwiGLU, 3 down-projection + weighted reduction.
 * Events are created lazily on the current device.  Recording events between
 * the up and down kernels stops them overlapping, so time the step itself
 * with profiling off. */
moe_status_t moe_ffn_profile_enable(int on);

/* Synchronize on the most recent profiled call and write its stage durations
 * in milliseconds to ms[0 .. *n_stages) (at most `capacity`). */
moe_status_t moe_ffn_profile_read(float* ms, int capacity, int* n_stages);

/* Name of the main kernel that ran in stage `stage` of the most recent
 * profiled call (for example "up_swiglu_pair2", "fused_cluster_bf16",
 * "none" for a stage that launches nothing), or NULL when that call recorded
 * no such stage.  The string is static; the caller does not free it. */
const char* moe_ffn_profile_stage_kernel(int stage);

/* Static description of a status code. */
const char* moe_ffn_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H_ */
