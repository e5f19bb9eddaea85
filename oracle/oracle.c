/*
 * oracle.c -- CPU oracle for the routed MoE SwiGLU feed-forward forward pass.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the benchmark's cpu_baseline / reference legs may load this library.  It
 * shares no code with the CUDA path (no headers, tables or helpers).
 *
 * Everything here is deliberately plain: fp64 arithmetic, straight loops in
 * the order the method states them, OpenMP only across independent tokens.
 *
 * Sources (page titles and sections):
 *  - "Prime Flash MoE - Faster MoE Kernels optimized for Blackwell", sec. 1
 *    "The computation": per routed (token, expert) pair, gate_up = W1[e] x_t
 *    with W1 output-major, gate = first H outputs, up = last H outputs
 *    (chunk(2)), act = silu(gate) * up, y = W2[e] act, and the routing weight
 *    is applied to y before the top-k outputs are summed into out[t].
 *  - same page, sec. 5 "The two epilogues": act is rounded to bf16 before the
 *    down projection; sec. 7 "The MXFP8 variant", "The epilogue also
 *    quantizes": in MXFP8 mode act is requantized to e4m3 with one e8m0
 *    scale per 32 contiguous elements along H.
 *  - "Porting Block-Scaled GEMM Kernels from Blackwell to Rubin", sec. 6.2:
 *    on sm_100/sm_103 the scale byte is obtained by rounding amax/448 up to
 *    a power of two (cvt.rp ... ue8m0), then values are multiplied by the
 *    reciprocal scale and converted to e4m3 with round-to-nearest-even and
 *    saturation.
 *  - OCP Microscaling (MX) format: E4M3 is bias 7, no infinities, S.1111.111
 *    is NaN, max finite 448, subnormal step 2^-9; E8M0 encodes 2^(s-127).
 *
 * Readings where the pages are silent are listed in the design notes; the ones
 * that change arithmetic are repeated at the functions they affect.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* binary32 -> bf16, round to nearest, ties to even (NaN stays NaN). */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    /* Add just under half an ulp of bf16, plus one if the kept lsb is odd. */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* OCP E4M3 (FN variant): s.eeee.mmm, bias 7, exponent field 0 = subnormal,
 * 0x7f / 0xff = NaN, no infinities. */
double oracle_e4m3_to_f64(uint8_t q) {
    int s = q >> 7, ef = (q >> 3) & 0xf, m = q & 7;
    double v;
    if (ef == 0xf && m == 7) return NAN;
    if (ef == 0) v = ldexp((double)m, -9);              /* m/8 * 2^(1-7) */
    else         v = ldexp(1.0 + m / 8.0, ef - 7);
    return s ? -v : v;
}

/* Real number -> E4M3, round to nearest even, saturating to +-448. */
uint8_t oracle_f64_to_e4m3(double v) {
    uint8_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x80 : 0x00;
    double a = fabs(v);
    if (isnan(v)) return 0x7f;
    if (a >= 448.0) return sign | 0x7e;                 /* satfinite */
    if (a < ldexp(1.0, -6)) {
        /* Subnormal grid: multiples of 2^-9.  A result of 8 is 2^-6, which
         * is exactly the encoding of the smallest normal (0x08). */
        double n = nearbyint(ldexp(a, 9));
        return sign | (uint8_t)n;
    }
    int ex;
    double f = frexp(a, &ex);                           /* a = f 2^ex, f in [0.5,1) */
    int e = ex - 1;                                     /* a = (2f) 2^e, 2f in [1,2) */
    double mant = nearbyint((2.0 * f - 1.0) * 8.0);     /* 3 fraction bits, RNE */
    if (mant == 8.0) { mant = 0.0; e += 1; }
    if (e > 8 || (e == 8 && mant > 6.0)) return sign | 0x7e;
    return sign | (uint8_t)(((e + 7) << 3) | (int)mant);
}

double oracle_e8m0_to_f64(uint8_t s) {
    if (s == 0xff) return NAN;
    return ldexp(1.0, (int)s - 127);
}

/*
 * Scale exponent for one MX block: the smallest integer e with
 * amax * 2^-e <= 448, i.e. e = ceil(log2(amax / 448)), which is what rounding
 * amax/448 up to a power of two gives.  Written without logarithms: with
 * amax = m 2^p, m in [1,2), and 448 = 1.75 2^8,
 *   e = p - 8 + (m > 1.75).
 * amax == 0 yields e = 0 (scale byte 127).
 */
int oracle_mx_scale_exponent(double amax) {
    if (amax == 0.0) return 0;
    int ex;
    double f = frexp(amax, &ex);
    double m = 2.0 * f;
    int p = ex - 1;
    return p - 8 + (m > 1.75 ? 1 : 0);
}

/*
 * Quantize n values (n a multiple of 32) to MXFP8: per block of 32, the scale
 * exponent above, scale byte e + 127, codes e4m3(a * 2^-e).  The values are
 * first rounded to binary32, the precision in which the kernel holds act when
 * it takes this decision (fp32 accumulators read from tensor memory).
 * deq (optional) receives q * 2^e.
 */
void oracle_mx_quantize(const double* a, int n, uint8_t* q, uint8_t* sf, double* deq) {
    for (int b = 0; b < n / 32; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            double v = (double)(float)a[b * 32 + i];
            if (fabs(v) > amax) amax = fabs(v);
        }
        int e = oracle_mx_scale_exponent(amax);
        sf[b] = (uint8_t)(e + 127);
        for (int i = 0; i < 32; ++i) {
            double v = (double)(float)a[b * 32 + i];
            uint8_t c = oracle_f64_to_e4m3(ldexp(v, -e));
            q[b * 32 + i] = c;
            if (deq) deq[b * 32 + i] = ldexp(oracle_e4m3_to_f64(c), e);
        }
    }
}

/*
 * OCP E2M1 (the MXFP4 element; routed expert weights in "GC-MoE on SM120"
 * sec. 2.2, scale formats, one UE8M0 scale per 32 elements): s.ee.m in the
 * low four bits of a byte, bias 1, exponent field 0 = subnormal (0 or 0.5),
 * no infinities or NaN; the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4 and 6.
 */
double oracle_e2m1_to_f64(uint8_t code) {
    int s = (code >> 3) & 1, ef = (code >> 1) & 3, m = code & 1;
    double v = ef == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, ef - 1);
    return s ? -v : v;
}

/* Real number -> E2M1 (low four bits), round to nearest with ties to the even
 * code (mantissa bit 0), saturating to +-6.  (NaN is not representable; it
 * maps to the largest magnitude.) */
uint8_t oracle_f64_to_e2m1(double v) {
    uint8_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x8 : 0x0;
    double a = fabs(v);
    if (isnan(v) || a >= 6.0) return sign | 0x7;
    if (a < 1.0) {
        /* subnormal grid: multiples of 0.5 (1.0 is the smallest normal, code 2) */
        double n = nearbyint(a * 2.0);
        return sign | (uint8_t)n;
    }
    int ex;
    double f = frexp(a, &ex);                           /* a = f 2^ex, f in [0.5,1) */
    int e = ex - 1;                                     /* a = (2f) 2^e, 2f in [1,2) */
    double mant = nearbyint((2.0 * f - 1.0) * 2.0);     /* 1 fraction bit, RNE */
    if (mant == 2.0) { mant = 0.0; e += 1; }
    if (e > 2) return sign | 0x7;
    return sign | (uint8_t)(((e + 1) << 1) | (int)mant);
}

/*
 * Scale exponent for one MXFP4 block: the smallest integer e with
 * amax * 2^-e <= 6, i.e. ceil(log2(amax / 6)).  With amax = m 2^p, m in
 * [1,2), and 6 = 1.5 2^2:  e = p - 2 + (m > 1.5).  amax == 0 yields 0.
 */
int oracle_mx4_scale_exponent(double amax) {
    if (amax == 0.0) return 0;
    int ex;
    double f = frexp(amax, &ex);
    double m = 2.0 * f;
    int p = ex - 1;
    return p - 2 + (m > 1.5 ? 1 : 0);
}

/* ------------------------------------------------------------------------ */
/* Routing permutation                                                      */
/* ------------------------------------------------------------------------ */

/*
 * Counting sort of the routed pairs p = t*k + j by expert id.
 *   counts[e]       number of pairs routed to expert e
 *   offsets[0..E]   exclusive prefix sum of counts
 *   slot_of_pair[p] offsets[e] + (number of earlier pairs p' < p with the
 *                   same expert): the stable order within each expert.
 * The padded variant gives every expert a segment rounded up to a multiple of
 * `pad` rows (empty experts get none) and the slot of each pair in it.
 * Returns 0, or -1 if an id lies outside [0, E).
 */
int oracle_route(int T, int E, int k, const int32_t* ids, int pad,
                 int64_t* counts, int64_t* offsets, int64_t* slot_of_pair,
                 int64_t* pad_offsets, int64_t* pad_slot_of_pair) {
    int64_t P = (int64_t)T * k;
    for (int64_t p = 0; p < P; ++p)
        if (ids[p] < 0 || ids[p] >= E) return -1;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) counts[ids[p]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    if (pad_offsets) {
        pad_offsets[0] = 0;
        for (int e = 0; e < E; ++e)
            pad_offsets[e + 1] = pad_offsets[e] + (counts[e] + pad - 1) / pad * pad;
    }
    int64_t* seen = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    if (!seen) return -2;
    for (int64_t p = 0; p < P; ++p) {
        int e = ids[p];
        if (slot_of_pair) slot_of_pair[p] = offsets[e] + seen[e];
        if (pad_slot_of_pair && pad_offsets) pad_slot_of_pair[p] = pad_offsets[e] + seen[e];
        seen[e] += 1;
    }
    free(seen);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The router step before the path                                          */
/* ------------------------------------------------------------------------ */

/*
 * Top-k selection with normalized weights, the step upstream of the path
 * ("Prime Flash MoE" sec. 1 starts from each token's k experts and weights
 * summing to one, produced beforehand; the workloads produce them from
 * per-(token, expert) logits: the k largest, with a softmax over those k).
 *
 * For each token t, with l[e] = logits[t][e] (a NaN logit is read as -inf):
 *   ids[t][0..k-1]: the k experts with the largest l[e], in order of
 *                   decreasing l, ties going to the lower expert id; found
 *                   by k passes, each taking the best expert not yet taken.
 *   w[t][j] = exp(l[ids[t][j]] - m) / sum_i exp(l[ids[t][i]] - m), with
 *             m = l[ids[t][0]] (the largest), in double.  If m is -inf
 *             (every selected logit is -inf) each weight is 1/k.
 * Returns 0, or -1 for a bad argument (k outside [1, E]).
 */
int oracle_router_topk(int T, int E, int k, const float* logits, int32_t* ids, double* w) {
    if (T < 0 || E < 1 || k < 1 || k > E) return -1;
    char* taken = (char*)malloc((size_t)E);
    if (!taken) return -2;
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (int64_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            double bv = 0.0;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                double v = isnan(l[e]) ? -INFINITY : (double)l[e];
                if (best < 0 || v > bv) {  /* strict: an equal later id never wins */
                    best = e;
                    bv = v;
                }
            }
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
        }
        double m = isnan(l[ids[(int64_t)t * k]]) ? -INFINITY : (double)l[ids[(int64_t)t * k]];
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            double v = isnan(l[ids[(int64_t)t * k + j]]) ? -INFINITY : (double)l[ids[(int64_t)t * k + j]];
            double p = (m == -INFINITY) ? 1.0 : exp(v - m);
            w[(int64_t)t * k + j] = p;
            sum += p;
        }
        for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] /= sum;
    }
    free(taken);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The forward pass                                                         */
/* ------------------------------------------------------------------------ */

enum { ORACLE_IN_BF16 = 0, ORACLE_IN_MXFP8 = 1, ORACLE_IN_MXFP4W = 2 };
enum { ORACLE_ACT_EXACT = 0, ORACLE_ACT_BF16 = 1, ORACLE_ACT_MXFP8 = 2 };

/* Element i of a row-major operand, dequantized exactly to double.
 * bf16: the value itself.  MXFP8: e4m3(q[i]) * 2^(sf[i/32] - 127), the scale
 * blocks running along the last (contiguous, reduction) dimension. */
static double elem(int in_mode, const void* v, const uint8_t* sf, int64_t i) {
    if (in_mode == ORACLE_IN_BF16) return oracle_bf16_to_f64(((const uint16_t*)v)[i]);
    return oracle_e4m3_to_f64(((const uint8_t*)v)[i]) * oracle_e8m0_to_f64(sf[i / 32]);
}

/* Element i of a weight operand.  MXFP4 weights: E2M1 codes packed two to a
 * byte along the last dimension (element 2j in the low four bits of byte j,
 * element 2j + 1 in the high four), scaled by 2^(sf[i/32] - 127); the
 * activations stay MXFP8 in that mode. */
static double welem(int in_mode, const void* v, const uint8_t* sf, int64_t i) {
    if (in_mode != ORACLE_IN_MXFP4W) return elem(in_mode, v, sf, i);
    uint8_t byte = ((const uint8_t*)v)[i / 2];
    uint8_t code = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xf);
    return oracle_e2m1_to_f64(code) * oracle_e8m0_to_f64(sf[i / 32]);
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/*
 * out[n][d] for each requested token t = tokens[n] (all T tokens when tokens
 * is NULL):
 *
 *   acc = 0
 *   for j = 0 .. k-1 (ascending):
 *     e = ids[t][j], w = topk_w[t][j]
 *     g[h] = sum_d W1[e][h][d]   x[t][d]        h < H   (gate rows 0..H-1)
 *     u[h] = sum_d W1[e][H+h][d] x[t][d]                (up rows H..2H-1)
 *     (clamped variant, swiglu_limit L > 0: g[h] = min(g[h], L),
 *      u[h] = min(max(u[h], -L), L) first -- an upper bound on the gate, a
 *      bound on both sides of the up projection: the gpt-oss-style
 *      activation of "Porting Block-Scaled GEMM Kernels from Blackwell to
 *      Rubin" sec. 5.3)
 *     a[h] = silu(g[h]) * u[h]
 *     a    = act_round(a)                               (see below)
 *     y[d] = sum_h W2[e][d][h] a[h]
 *     acc[d] += w * y[d]
 *   out[n] = acc
 *
 * act_round: EXACT keeps fp64; BF16 rounds each a[h] to binary32 then to bf16
 * (RNE); MXFP8 requantizes a to e4m3 with one scale per 32 consecutive h.
 * Shapes: x[T][D], W1[E][2H][D], W2[E][D][H], ids/topk_w[T][k]; MXFP8 scale
 * arrays have one byte per 32 elements of the last dimension.  in_mode
 * MXFP4W: x as MXFP8, W1 / W2 as MXFP4 (see welem; D and H multiples of 32).
 * Returns 0, or -1 for an expert id outside [0, E) or a bad argument.
 */
int oracle_moe_ffn(int T, int E, int D, int H, int k, int in_mode,
                   const void* x, const uint8_t* x_sf,
                   const void* w1, const uint8_t* w1_sf,
                   const void* w2, const uint8_t* w2_sf,
                   const int32_t* ids, const float* topk_w,
                   int act_mode, const int32_t* tokens, int n_tokens,
                   double* out, int n_threads, double swiglu_limit) {
    if (T < 0 || E < 1 || D < 1 || H < 1 || k < 1) return -1;
    if (act_mode == ORACLE_ACT_MXFP8 && H % 32) return -1;
    if ((in_mode == ORACLE_IN_MXFP8 || in_mode == ORACLE_IN_MXFP4W) && (D % 32 || H % 32)) return -1;
    int n = tokens ? n_tokens : T;
    for (int i = 0; i < n; ++i) {
        int t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) return -1;
        for (int j = 0; j < k; ++j)
            if (ids[(int64_t)t * k + j] < 0 || ids[(int64_t)t * k + j] >= E) return -1;
    }
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double* xd = (double*)malloc(sizeof(double) * (size_t)D);
        double* g = (double*)malloc(sizeof(double) * (size_t)H);
        double* u = (double*)malloc(sizeof(double) * (size_t)H);
        double* a = (double*)malloc(sizeof(double) * (size_t)H);
        uint8_t* aq = (uint8_t*)malloc((size_t)H);
        uint8_t* asf = (uint8_t*)malloc((size_t)H / 32 + 1);
        if (!xd || !g || !u || !a || !aq || !asf) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int i = 0; i < n; ++i) {
                int t = tokens ? tokens[i] : i;
                double* acc = out + (int64_t)i * D;
                for (int d = 0; d < D; ++d) {
                    acc[d] = 0.0;
                    xd[d] = elem(in_mode == ORACLE_IN_MXFP4W ? ORACLE_IN_MXFP8 : in_mode, x, x_sf,
                                 (int64_t)t * D + d);
                }
                for (int j = 0; j < k; ++j) {
                    int e = ids[(int64_t)t * k + j];
                    double w = (double)topk_w[(int64_t)t * k + j];
                    int64_t w1e = (int64_t)e * 2 * H * D;
                    for (int h = 0; h < H; ++h) {
                        double sg = 0.0, su = 0.0;
                        int64_t rg = w1e + (int64_t)h * D, ru = w1e + (int64_t)(H + h) * D;
                        for (int d = 0; d < D; ++d) {
                            sg += welem(in_mode, w1, w1_sf, rg + d) * xd[d];
                            su += welem(in_mode, w1, w1_sf, ru + d) * xd[d];
                        }
                        g[h] = sg;
                        u[h] = su;
                    }
                    if (swiglu_limit > 0.0) {
                        for (int h = 0; h < H; ++h) {
                            if (g[h] > swiglu_limit) g[h] = swiglu_limit;
                            if (u[h] > swiglu_limit) u[h] = swiglu_limit;
                            if (u[h] < -swiglu_limit) u[h] = -swiglu_limit;
                        }
                    }
                    for (int h = 0; h < H; ++h) a[h] = silu(g[h]) * u[h];
                    if (act_mode == ORACLE_ACT_BF16) {
                        for (int h = 0; h < H; ++h) a[h] = oracle_bf16_to_f64(oracle_f32_to_bf16((float)a[h]));
                    } else if (act_mode == ORACLE_ACT_MXFP8) {
                        oracle_mx_quantize(a, H, aq, asf, a);
                    }
                    int64_t w2e = (int64_t)e * D * H;
                    for (int d = 0; d < D; ++d) {
                        double y = 0.0;
                        int64_t r = w2e + (int64_t)d * H;
                        for (int h = 0; h < H; ++h) y += welem(in_mode, w2, w2_sf, r + h) * a[h];
                        acc[d] += w * y;
                    }
                }
            }
        }
        free(xd); free(g); free(u); free(a); free(aq); free(asf);
    }
    return failed ? -2 : 0;
}

/* ------------------------------------------------------------------------ */
/* NVFP4                                                                    */
/* ------------------------------------------------------------------------ */

/*
 * NVFP4 ("Porting Block-Scaled GEMM Kernels from Blackwell to Rubin": sec. 1.2
 * counts 16 scales per 256-element row, i.e. one scale per 16 elements along
 * K; sec. 6.1: UE4M3 block scales of amax / 6 paired with a per-tensor fp32
 * global scale, per expert in MoE kernels; sec. 5.3 dequantizes gate and up
 * by the expert's global scale alpha):
 * an element is an E2M1 code c, its 16-element block carries an E4M3 scale
 * s (a non-negative code), and the whole operand (for the weights: each
 * expert) one fp32 global scale G, so the value is
 *     e2m1(c) * e4m3(s) * G.
 * Codes are packed two per byte along K, element 2j in the low four bits.
 */
static double nv4_elem(const uint8_t* v, const uint8_t* sf, int64_t i) {
    uint8_t byte = v[i / 2];
    uint8_t code = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xf);
    return oracle_e2m1_to_f64(code) * oracle_e4m3_to_f64(sf[i / 16]);
}

/*
 * Quantize n values (n a multiple of 16) to NVFP4 with global scale gs > 0.
 * Reading (the pages give the format, not the recipe): per block of 16, on
 * the values rounded to binary32 (the precision of the accumulators the
 * kernel quantizes from), the block scale is the e4m3 code nearest to
 * amax / (6 gs) (round to nearest even, saturating at 448), so that the
 * largest element lands near the top of the E2M1 range; each element is
 * then the E2M1 code nearest to v / (e4m3(s) gs) (ties to the even code,
 * saturating at 6).  A block whose scale rounds to 0 is all zeros.
 * codes: n/2 bytes (packed as above), sf: n/16 bytes, deq (optional): the
 * dequantized values e2m1 * e4m3(s) * gs.
 */
void oracle_nv4_quantize(const double* a, int n, double gs, uint8_t* codes, uint8_t* sf, double* deq) {
    for (int b = 0; b < n / 16; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 16; ++i) {
            double v = (double)(float)a[b * 16 + i];
            if (fabs(v) > amax) amax = fabs(v);
        }
        uint8_t s = oracle_f64_to_e4m3(amax / (6.0 * gs));
        double scale = oracle_e4m3_to_f64(s) * gs;
        sf[b] = s;
        for (int i = 0; i < 16; ++i) {
            int idx = b * 16 + i;
            double v = (double)(float)a[idx];
            uint8_t c = scale > 0.0 ? oracle_f64_to_e2m1(v / scale) : 0;
            if (idx & 1) codes[idx / 2] = (uint8_t)((codes[idx / 2] & 0x0f) | (c << 4));
            else         codes[idx / 2] = (uint8_t)((codes[idx / 2] & 0xf0) | c);
            if (deq) deq[idx] = oracle_e2m1_to_f64(c) * scale;
        }
    }
}

enum { ORACLE_ACT_NVFP4 = 3 };

/*
 * The forward pass of oracle_moe_ffn with NVFP4 operands: x [T, D/2] codes,
 * x_sf [T, D/16], global x_gs; W1 [E, 2H, D/2], w1_sf [E, 2H, D/16], one
 * global w1_gs[e] per expert; W2 [E, D, H/2], w2_sf [E, D, H/16], w2_gs[e].
 * Every element is dequantized exactly (nv4_elem times its global scale) and
 * the arithmetic is that of oracle_moe_ffn in fp64.  act_mode: EXACT keeps
 * act in fp64; NVFP4 requantizes act per 16 along H with the global scale
 * act_gs (oracle_nv4_quantize) before the down projection; BF16 rounds act
 * to bf16 as in oracle_moe_ffn.  D and H multiples of 32.
 * Returns 0, or -1 for an expert id outside [0, E) or a bad argument.
 */
int oracle_moe_ffn_nvfp4(int T, int E, int D, int H, int k,
                         const uint8_t* x, const uint8_t* x_sf, double x_gs,
                         const uint8_t* w1, const uint8_t* w1_sf, const float* w1_gs,
                         const uint8_t* w2, const uint8_t* w2_sf, const float* w2_gs,
                         const int32_t* ids, const float* topk_w,
                         int act_mode, double act_gs, const int32_t* tokens, int n_tokens,
                         double* out, int n_threads, double swiglu_limit) {
    if (T < 0 || E < 1 || D < 1 || H < 1 || k < 1 || D % 32 || H % 32) return -1;
    if (act_mode != ORACLE_ACT_EXACT && act_mode != ORACLE_ACT_BF16 && act_mode != ORACLE_ACT_NVFP4) return -1;
    if (act_mode == ORACLE_ACT_NVFP4 && !(act_gs > 0.0)) return -1;
    int n = tokens ? n_tokens : T;
    for (int i = 0; i < n; ++i) {
        int t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) return -1;
        for (int j = 0; j < k; ++j)
            if (ids[(int64_t)t * k + j] < 0 || ids[(int64_t)t * k + j] >= E) return -1;
    }
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double* xd = (double*)malloc(sizeof(double) * (size_t)D);
        double* g = (double*)malloc(sizeof(double) * (size_t)H);
        double* u = (double*)malloc(sizeof(double) * (size_t)H);
        double* a = (double*)malloc(sizeof(double) * (size_t)H);
        uint8_t* aq = (uint8_t*)calloc((size_t)H / 2 + 1, 1);
        uint8_t* asf = (uint8_t*)malloc((size_t)H / 16 + 1);
        if (!xd || !g || !u || !a || !aq || !asf) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int i = 0; i < n; ++i) {
                int t = tokens ? tokens[i] : i;
                double* acc = out + (int64_t)i * D;
                for (int d = 0; d < D; ++d) {
                    acc[d] = 0.0;
                    xd[d] = nv4_elem(x, x_sf, (int64_t)t * D + d) * x_gs;
                }
                for (int j = 0; j < k; ++j) {
                    int e = ids[(int64_t)t * k + j];
                    double w = (double)topk_w[(int64_t)t * k + j];
                    double g1 = (double)w1_gs[e], g2 = (double)w2_gs[e];
                    int64_t w1e = (int64_t)e * 2 * H * D;
                    for (int h = 0; h < H; ++h) {
                        double sg = 0.0, su = 0.0;
                        int64_t rg = w1e + (int64_t)h * D, ru = w1e + (int64_t)(H + h) * D;
                        for (int d = 0; d < D; ++d) {
                            sg += nv4_elem(w1, w1_sf, rg + d) * g1 * xd[d];
                            su += nv4_elem(w1, w1_sf, ru + d) * g1 * xd[d];
                        }
                        g[h] = sg;
                        u[h] = su;
                    }
                    if (swiglu_limit > 0.0) {
                        for (int h = 0; h < H; ++h) {
                            if (g[h] > swiglu_limit) g[h] = swiglu_limit;
                            if (u[h] > swiglu_limit) u[h] = swiglu_limit;
                            if (u[h] < -swiglu_limit) u[h] = -swiglu_limit;
                        }
                    }
                    for (int h = 0; h < H; ++h) a[h] = silu(g[h]) * u[h];
                    if (act_mode == ORACLE_ACT_BF16) {
                        for (int h = 0; h < H; ++h) a[h] = oracle_bf16_to_f64(oracle_f32_to_bf16((float)a[h]));
                    } else if (act_mode == ORACLE_ACT_NVFP4) {
                        oracle_nv4_quantize(a, H, act_gs, aq, asf, a);
                    }
                    int64_t w2e = (int64_t)e * D * H;
                    for (int d = 0; d < D; ++d) {
                        double y = 0.0;
                        int64_t r = w2e + (int64_t)d * H;
                        for (int h = 0; h < H; ++h) y += nv4_elem(w2, w2_sf, r + h) * g2 * a[h];
                        acc[d] += w * y;
                    }
                }
            }
        }
        free(xd); free(g); free(u); free(a); free(aq); free(asf);
    }
    return failed ? -2 : 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
