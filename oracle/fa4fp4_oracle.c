/*
 * fa4fp4_oracle.c -- plain, slow CPU definition of block-scaled FP4 attention
 * with Direct-P ("Hardware-Aware FP4 FlashAttention-4", arXiv:2609.04105).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes, links or
 * calls this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark load it.  It shares no code, header, table or
 * constant generator with the CUDA path.
 *
 * Everything is computed in FP64, except the steps the method defines in FP32
 * (the score s that Direct-P classifies, and the FMA that forms the scaled
 * offset from the running maximum), which use C's float and fmaf.
 *
 * Sources (page "Hardware-Aware FP4 FlashAttention-4", gist.science technical
 * summary, and the arXiv abstract):
 *   - Problem Statement, "Numerical Range": E2M1 payloads, MXFP4/NVFP4.
 *   - Methodology 1, "Direct Mapping": scores mapped to the 8 non-negative E2M1
 *     magnitudes by classification instead of exp-then-round.
 *   - Methodology 1, "Consistent Normalization": the denominator is summed
 *     from the same rounded codes the P.V product consumes.
 *   - Methodology 1, "Format Selection": MXFP4 (one power-of-two scale for every
 *     32 consecutive elements) for P and V; Q and K use MXFP4 here as well.
 *   - Methodology 2, "Quantized Causal Backward": forward saves quantized Q/K,
 *     scales and the LSE; backward rebuilds P from them and uses FP8
 *     row/column views of Q, K, V for the gradient products.
 *   - Abstract: FP8 gradient operands.
 * Readings of the points the pages leave open are stated beside each function.
 *
 * Parity status: every function here is pinned by the CPU tests
 * (tests/test_oracle_*.py) against closed forms, brute force, library
 * routines or invariants; none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Element formats (Problem Statement, "Numerical Range")                    */
/* ------------------------------------------------------------------------ */

/* E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.  The eight
 * non-negative magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Decoded here from
 * the bit fields, not from a table, so the table pin is a real check. */
ORC_API double orc_e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* OCP FP8 E4M3 ("fn"): bias 7, no infinities, S.1111.111 is NaN, max 448. */
ORC_API double orc_e4m3_value(int code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);          /* m/8 * 2^-6 */
    else mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* E8M0 block scale: byte b is 2^(b-127); 255 is NaN. */
ORC_API double orc_e8m0_value(int byte) {
    if (byte == 255) return NAN;
    return ldexp(1.0, byte - 127);
}

/* Round |y| to the nearest representable magnitude of the element format,
 * ties to the even code (the code's lowest bit is the mantissa's lowest bit,
 * so this is round-half-to-even).  Values above the largest finite magnitude
 * saturate to it.  Implemented as a scan over all codes of the format so
 * that it is independent of any binade arithmetic. */
static int nearest_code(double ay, int fmt) {
    int ncodes = fmt == 0 ? 8 : 127;   /* E2M1: 0..7; E4M3: 0..126 (127 = NaN) */
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c < ncodes; ++c) {
        double v = fmt == 0 ? orc_e2m1_value(c) : orc_e4m3_value(c);
        double dd = fabs(ay - v);
        if (dd < bestd || (dd == bestd && (c & 1) == 0)) { best = c; bestd = dd; }
    }
    return best;
}

/* Quantize one value y (already divided by the block scale) to a code with
 * its sign kept: a negative value that rounds to zero gives negative zero. */
ORC_API int orc_round_to_code(double y, int fmt) {
    int mag = nearest_code(fabs(y), fmt);
    int signbit = signbit(y) ? 1 : 0;
    return fmt == 0 ? (signbit << 3) | mag : (signbit << 7) | mag;
}

/* Shared block exponent X for one block, following the OCP Microscaling (MX)
 * v1.0 rule: X = floor(log2(amax)) - emax_elem, clamped to the E8M0 range.
 * floor(log2(amax)) is read from the FP32 exponent field of amax (the inputs
 * are bf16, exact in FP32); a zero or subnormal amax has field 0.
 * Reading: the pages name E8M0 block scales but no rule; the OCP MX rule is
 * the published definition of MXFP4/MXFP8. */
ORC_API int orc_block_exponent(float amax, int fmt) {
    uint32_t bits;
    memcpy(&bits, &amax, 4);
    int E = (int)((bits >> 23) & 0xff);
    int emax = fmt == 0 ? 2 : 8;
    int X = E - 127 - emax;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    return X;
}

/* Block exponent of an E4M3 probability block (P of the FP8 P/V forward and
 * of the backward): the smallest X with amax <= 448 * 2^X, i.e.
 * X = ceil(log2(amax / 448)), clamped to the E8M0 range.  It is the OCP
 * exponent, or one more where the OCP exponent would put amax above 448.
 * Reading: the pages fix no scale rule.  Under the OCP rule a block maximum
 * whose significand is above 1.75 saturates to 448 (up to 12.5 % low), and
 * a probability 1 computed a few ulps low (a row with one key) falls to
 * 0.875 while exactly 1 stays 1; this rule has neither effect. */
ORC_API int orc_p_block_exponent(float amax) {
    int X = orc_block_exponent(amax, 1);
    if (X < 127 && (double)amax > ldexp(448.0, X)) X += 1;
    return X;
}

/* Quantize a logical [B,H,N,d] FP32 tensor (holding bf16 values) in blocks of
 * 32 along one axis.
 *   fmt  : 0 = MXFP4 (E2M1 codes, two per byte, element 2i in the low nibble)
 *          1 = MXFP8 E4M3 (one byte per element)
 *   axis : 0 = blocks along d, output [B,H,N,d] elements, scales [B,H,N,d/32]
 *          1 = blocks along N, output transposed [B,H,d,Np] elements and
 *              scales [B,H,d,Np/32], Np = N rounded up to a multiple of 128;
 *              positions beyond N hold +0 and count as zero in the amax.
 * Per block: amax over the block, X from orc_block_exponent, scale byte X+127,
 * each element y = x * 2^-X rounded by orc_round_to_code. */
ORC_API void orc_quantize(const float* x, int B, int H, int N, int d, int fmt, int axis,
                          uint8_t* codes, uint8_t* scales) {
    int Np = ((N + 127) / 128) * 128;
    long BH = (long)B * H;
    int L = axis == 0 ? d : Np;          /* length of a row along the block axis */
    int R = axis == 0 ? N : d;           /* rows per (b,h) */
    int nb = L / 32;
    #pragma omp parallel for schedule(static)
    for (long bh = 0; bh < BH; ++bh) {
        for (int r = 0; r < R; ++r) {
            for (int blk = 0; blk < nb; ++blk) {
                float vals[32];
                for (int t = 0; t < 32; ++t) {
                    int pos = blk * 32 + t;
                    float v;
                    if (axis == 0) v = x[(bh * N + r) * (long)d + pos];
                    else v = pos < N ? x[(bh * N + pos) * (long)d + r] : 0.0f;
                    vals[t] = v;
                }
                float amax = 0.0f;
                for (int t = 0; t < 32; ++t) if (fabsf(vals[t]) > amax) amax = fabsf(vals[t]);
                int X = orc_block_exponent(amax, fmt);
                scales[(bh * R + r) * (long)nb + blk] = (uint8_t)(X + 127);
                for (int t = 0; t < 32; ++t) {
                    int code = orc_round_to_code(ldexp((double)vals[t], -X), fmt);
                    long e = (bh * R + r) * (long)L + blk * 32 + t;
                    if (fmt == 1) {
                        codes[e] = (uint8_t)code;
                    } else {
                        uint8_t* byte = &codes[e / 2];
                        if ((e & 1) == 0) *byte = (uint8_t)((*byte & 0xf0) | code);
                        else *byte = (uint8_t)((*byte & 0x0f) | (code << 4));
                    }
                }
            }
        }
    }
}

/* Inverse view: expand codes+scales back to a logical [B,H,N,d] FP32 tensor
 * (every dequantized value is exact in FP32). */
ORC_API void orc_dequantize(const uint8_t* codes, const uint8_t* scales, int B, int H, int N,
                            int d, int fmt, int axis, float* out) {
    int Np = ((N + 127) / 128) * 128;
    long BH = (long)B * H;
    int L = axis == 0 ? d : Np;
    int R = axis == 0 ? N : d;
    int nb = L / 32;
    #pragma omp parallel for schedule(static)
    for (long bh = 0; bh < BH; ++bh) {
        for (int n = 0; n < N; ++n) {
            for (int c = 0; c < d; ++c) {
                int r = axis == 0 ? n : c, pos = axis == 0 ? c : n;
                long e = (bh * R + r) * (long)L + pos;
                int code = fmt == 1 ? codes[e] : ((codes[e / 2] >> (4 * (e & 1))) & 0xf);
                double v = fmt == 1 ? orc_e4m3_value(code) : orc_e2m1_value(code);
                double s = orc_e8m0_value(scales[(bh * R + r) * (long)nb + pos / 32]);
                out[(bh * N + n) * (long)d + c] = (float)(v * s);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* NVFP4 (Methodology 1, "Format Selection": NVFP4 for Q and K, for its      */
/* fine-grained scaling)                                                     */
/* ------------------------------------------------------------------------ */

/* The pages name NVFP4 but give no rule.  Reading: the public NVFP4 format,
 * E2M1 elements with one unsigned E4M3 scale per 16 consecutive elements along
 * d and one FP32 scale per tensor, every step an FP32 operation rounded to
 * nearest:
 *   amax_t = max |x| over the tensor; ts = amax_t / 2688 (2688 = 6 * 448: the
 *   tensor's largest block then takes the largest E2M1 value under the
 *   largest E4M3 scale); ts = 1 for an all-zero tensor;
 *   per block of 16: sb = E4M3(amax_b / (6 * ts)) (RNE, saturating);
 *   each element: code = E2M1(x / (sb * ts)) (RNE, saturating, sign kept); a
 *   block whose scale rounds to zero gets signed-zero codes.
 * A value dequantizes to e2m1(code) * sb * ts. */
ORC_API float orc_nvfp4_tensor_scale(const float* x, long n) {
    float amax = 0.0f;
    for (long i = 0; i < n; ++i) if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    return amax > 0.0f ? amax / 2688.0f : 1.0f;
}

/* x logical [B,H,N,d] FP32 (bf16 values); codes [B,H,N,d/2] (element 2i in
 * the low nibble), scales [B,H,N,d/16] E4M3 bytes, ts from
 * orc_nvfp4_tensor_scale of the same tensor. */
ORC_API void orc_quantize_nvfp4(const float* x, int B, int H, int N, int d, float ts, uint8_t* codes,
                                uint8_t* scales) {
    long rows = (long)B * H * N;
    int nb = d / 16;
    const float six_ts = 6.0f * ts;
    #pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        for (int blk = 0; blk < nb; ++blk) {
            const float* v = x + r * d + blk * 16;
            float amax = 0.0f;
            for (int t = 0; t < 16; ++t) if (fabsf(v[t]) > amax) amax = fabsf(v[t]);
            const float sbf = amax / six_ts;
            const int sbc = orc_round_to_code((double)sbf, 1);
            scales[r * nb + blk] = (uint8_t)sbc;
            const float den = (float)orc_e4m3_value(sbc) * ts;
            for (int t = 0; t < 16; ++t) {
                int code;
                if (den == 0.0f) code = signbit(v[t]) ? 0x8 : 0x0;
                else code = orc_round_to_code((double)(v[t] / den), 0);
                long e = r * d + blk * 16 + t;
                uint8_t* byte = &codes[e / 2];
                if ((e & 1) == 0) *byte = (uint8_t)((*byte & 0xf0) | code);
                else *byte = (uint8_t)((*byte & 0x0f) | (code << 4));
            }
        }
    }
}

ORC_API void orc_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales, float ts, int B, int H,
                                  int N, int d, float* out) {
    long n = (long)B * H * N * d;
    #pragma omp parallel for schedule(static)
    for (long e = 0; e < n; ++e) {
        int code = (codes[e / 2] >> (4 * (e & 1))) & 0xf;
        double sb = orc_e4m3_value(scales[e / 16]);
        out[e] = (float)(orc_e2m1_value(code) * sb * (double)ts);
    }
}

/* ------------------------------------------------------------------------ */
/* Direct-P (Methodology 1, "Direct Mapping")                                */
/* ------------------------------------------------------------------------ */

/* Reading: the probability code of a score s under running maximum m is
 * RNE_E2M1(6 * 2^x) with x = c*(s-m), c = softmax_scale*log2(e); the factor 6
 * places the row maximum on the largest E2M1 magnitude, and P blocks carry the
 * unit E8M0 scale.  x is formed as the single FP32 FMA fmaf(s, c, -fl32(m*c)).
 * The map is then a comparison of x against seven constants T_1..T_7, where
 * T_k is the smallest FP32 value with RNE_E2M1(6*2^T_k) >= (k-th magnitude).
 * They are found here by bisection over the ordered FP32 values, with the
 * predicate evaluated in FP64. */
static int e2m1_code_of_6exp2(float x) {
    return nearest_code(6.0 * exp2((double)x), 0);
}

static int32_t float_to_ordered(float f) {
    int32_t i;
    memcpy(&i, &f, 4);
    return i >= 0 ? i : (int32_t)(0x80000000u - (uint32_t)i) ;
}

static float ordered_to_float(int32_t o) {
    int32_t i = o >= 0 ? o : (int32_t)(0x80000000u - (uint32_t)o);
    float f;
    memcpy(&f, &i, 4);
    return f;
}

ORC_API void orc_directp_thresholds(float T[7]) {
    for (int k = 1; k <= 7; ++k) {
        /* predicate(x) = code(x) >= k is monotone in x; bracket on [-64, 0]. */
        int32_t lo = float_to_ordered(-64.0f), hi = float_to_ordered(0.0f);
        /* invariant: code(lo) < k <= code(hi) */
        while (hi - lo > 1) {
            int32_t mid = lo + (hi - lo) / 2;
            if (e2m1_code_of_6exp2(ordered_to_float(mid)) >= k) hi = mid;
            else lo = mid;
        }
        T[k - 1] = ordered_to_float(hi);
    }
}

static float g_T[7];
static int g_T_ready = 0;

static const float* thresholds(void) {
    if (!g_T_ready) {
        #pragma omp critical(orc_thresholds)
        {
            if (!g_T_ready) { orc_directp_thresholds(g_T); g_T_ready = 1; }
        }
    }
    return g_T;
}

/* The scaled offset of s from the running max, as the method forms it. */
ORC_API float orc_directp_x(float s, float m, float c) {
    float mc = m * c;               /* fl32(m*c) */
    return fmaf(s, c, -mc);
}

/* code = #{k : x >= T_k}, in 0..7. */
ORC_API int orc_directp_code_of_x(float x) {
    const float* T = thresholds();
    int code = 0;
    for (int k = 0; k < 7; ++k) code += (x >= T[k]);
    return code;
}

ORC_API int orc_directp_code(float s, float m, float c) {
    return orc_directp_code_of_x(orc_directp_x(s, m, c));
}

/* Vector form of orc_directp_code_of_x for the dense-grid pin. */
ORC_API void orc_directp_codes_of_x(const float* x, long n, uint8_t* out) {
    const float* T = thresholds();
    #pragma omp parallel for schedule(static)
    for (long e = 0; e < n; ++e) {
        int code = 0;
        for (int k = 0; k < 7; ++k) code += (x[e] >= T[k]);
        out[e] = (uint8_t)code;
    }
}

/* ------------------------------------------------------------------------ */
/* Forward (Methodology 1; Problem Statement)                                */
/* ------------------------------------------------------------------------ */

#define ORC_BC 128   /* key tile: 128 consecutive keys, visited in ascending order */

/* Forward attention for a chosen list of query rows.
 * Q [B,Hq,N,d], K and V [B,Hkv,N,d]: dequantized values (or raw values for
 * the identity-quantizer mode).  kv head of query head h is h / (Hq/Hkv).
 * rows[r] = (b*Hq + h)*N + i selects the query rows to compute; O_out[r*d..]
 * and LSE_out[r] receive the results.
 * mode 0 (the method): s = fl32(exact dot product); per key tile j in
 *   ascending order, m_j = max(m_{j-1}, max valid s in tile j); codes against
 *   m_j; alpha = 2^(c*(m_{j-1}-m_j)); l <- alpha*l + sum value(code);
 *   O <- alpha*O + sum value(code)*V.  Output O/l, LSE = scale*m + ln(l/6).
 *   Reading: the rescale is applied every time m grows (eager), and the code
 *   of a key is fixed against the running max of its own tile.
 * mode 1 (textbook reduction for pins): same loop with s in FP64 and
 *   p = exp2(c*(s-m)) in place of the code value (no factor 6; LSE = scale*m +
 *   ln l).
 * mode 2 (the FP8 P/V training route; "Stability Constraint" of the technical
 *   summary: the retained training route keeps FP8 probabilities and values):
 *   s and the running max as in mode 0; p = fl32(2^x) with x =
 *   fl32(fl32(s - m_j) * c) (the difference first: it is exact near the max,
 *   so the row max gets x = 0 and p = 1 exactly); p rounded to E4M3 with one
 *   E8M0 scale per 32 keys from orc_p_block_exponent (blocks aligned to
 *   absolute key positions 32a) as the P V operand;
 *   l <- alpha*l + sum deq(p8) (the normalizer from the same rounded values
 *   the product consumes); O <- alpha*O + sum deq(p8)*V, V being the
 *   dequantized MXFP8 V.  Output O/l, LSE = scale*m + ln l.
 * Causal: key n is valid for query i iff n <= i; key tiles wholly above the
 * diagonal are skipped. */
static void mxfp8_roundtrip(double* v, int n, long stride);
static void p_e4m3_roundtrip(double* v, int n);
ORC_API void orc_fwd(const float* Q, const float* K, const float* V, int B, int Hq, int Hkv,
                     int N, int d, float softmax_scale, int causal, int mode, long nrows,
                     const int64_t* rows, double* O_out, double* LSE_out) {
    if (softmax_scale <= 0.0f) softmax_scale = (float)(1.0 / sqrt((double)d));
    const float c = (float)((double)softmax_scale * 1.4426950408889634);   /* fl32(scale*log2 e) */
    /* mode 1 is the real-arithmetic textbook form: c unrounded */
    const double cr = mode != 1 ? (double)c : (double)softmax_scale * 1.4426950408889634;
    const int group = Hq / Hkv;
    #pragma omp parallel for schedule(dynamic, 4)
    for (long r = 0; r < nrows; ++r) {
        int64_t row = rows[r];
        int i = (int)(row % N);
        int h = (int)((row / N) % Hq);
        int b = (int)(row / ((int64_t)N * Hq));
        int hk = h / group;
        const float* q = Q + row * (long)d;
        const float* Kh = K + ((long)b * Hkv + hk) * (long)N * d;
        const float* Vh = V + ((long)b * Hkv + hk) * (long)N * d;
        double* o = O_out + r * (long)d;
        for (int t = 0; t < d; ++t) o[t] = 0.0;
        double l = 0.0;
        double m = -INFINITY;              /* running max (FP32 value in mode 0) */
        int last = causal ? i : N - 1;
        double* s = (double*)malloc(sizeof(double) * ORC_BC);
        for (int j0 = 0; j0 <= last; j0 += ORC_BC) {
            int j1 = j0 + ORC_BC - 1;
            if (j1 > last) j1 = last;
            int cnt = j1 - j0 + 1;
            double tmax = -INFINITY;
            for (int n = 0; n < cnt; ++n) {
                double acc = 0.0;
                const float* kr = Kh + (long)(j0 + n) * d;
                for (int t = 0; t < d; ++t) acc += (double)q[t] * (double)kr[t];
                s[n] = mode != 1 ? (double)(float)acc : acc;
                if (s[n] > tmax) tmax = s[n];
            }
            double mnew = m > tmax ? m : tmax;
            double alpha = (m == -INFINITY) ? 1.0 : exp2(cr * (m - mnew));
            l *= alpha;
            for (int t = 0; t < d; ++t) o[t] *= alpha;
            if (mode == 2) {
                /* p = fl32(2^x), x = fl32(fl32(s - m) * c), for the valid keys,
                 * then E4M3 in 32-key blocks under orc_p_block_exponent */
                for (int n = 0; n < cnt; ++n) {
                    const float dx = (float)s[n] - (float)mnew;
                    const float x = dx * c;
                    s[n] = (double)(float)exp2((double)x);
                }
                for (int a0 = 0; a0 < cnt; a0 += 32) {
                    int nb = cnt - a0 < 32 ? cnt - a0 : 32;
                    p_e4m3_roundtrip(s + a0, nb);
                }
            }
            for (int n = 0; n < cnt; ++n) {
                double p;
                if (mode == 0) p = orc_e2m1_value(orc_directp_code((float)s[n], (float)mnew, c));
                else if (mode == 2) p = s[n];
                else p = exp2(cr * (s[n] - mnew));
                if (p == 0.0) continue;
                l += p;
                const float* vr = Vh + (long)(j0 + n) * d;
                for (int t = 0; t < d; ++t) o[t] += p * (double)vr[t];
            }
            m = mnew;
        }
        free(s);
        for (int t = 0; t < d; ++t) o[t] /= l;
        LSE_out[r] = (double)softmax_scale * m + log(mode == 0 ? l / 6.0 : l);   /* modes 1, 2: ln l */
    }
}

/* ------------------------------------------------------------------------ */
/* Backward (Methodology 2, "Quantized Causal Backward"; abstract)           */
/* ------------------------------------------------------------------------ */

/* MXFP8 round trip of one 32-element block (OCP MX rule, E4M3 elements).
 * v[t*stride] for t < n are the valid elements; the rest of the block counts
 * as zero.  Values are replaced by their dequantized FP8 values. */
static void mxfp8_roundtrip(double* v, int n, long stride) {
    float amax = 0.0f;
    for (int t = 0; t < n; ++t) {
        float a = fabsf((float)v[t * stride]);
        if (a > amax) amax = a;
    }
    int X = orc_block_exponent(amax, 1);
    for (int t = 0; t < n; ++t) {
        double y = ldexp((double)(float)v[t * stride], -X);
        v[t * stride] = ldexp(orc_e4m3_value(orc_round_to_code(y, 1)), X);
    }
}

/* E4M3 round trip of one block of probabilities v[0..n) (n <= 32, the rest
 * of the block counts as zero) under orc_p_block_exponent. */
static void p_e4m3_roundtrip(double* v, int n) {
    float amax = 0.0f;
    for (int t = 0; t < n; ++t) {
        float a = fabsf((float)v[t]);
        if (a > amax) amax = a;
    }
    int X = orc_p_block_exponent(amax);
    for (int t = 0; t < n; ++t) {
        double y = ldexp((double)(float)v[t], -X);
        v[t] = ldexp(orc_e4m3_value(orc_round_to_code(y, 1)), X);
    }
}

/* Gradients of the forward above for a chosen set of rows.
 *
 * Inputs (logical [B,H,N,d] float arrays):
 *   Q4 [B,Hq], K4 [B,Hkv]   dequantized MXFP4 Q/K saved by the forward
 *   Q8 [B,Hq], K8 [B,Hkv]   dequantized MXFP8 views blocked along N (columns)
 *   V8 [B,Hkv]              dequantized MXFP8 view of V blocked along d (rows)
 *   O [B,Hq], dO [B,Hq]     forward output (FP32) and upstream gradient (bf16)
 *   LSE [B,Hq,N]            forward log-sum-exp (natural log)
 * mode 0 (the method):
 *   P = 2^x, x = fmaf(s, c, -fl32(LSE*fl32(log2 e))), s = fl32(Q4.K4);
 *   D_i = sum_t dO_it*O_it;
 *   dO is quantized twice: blocks along d (row view, feeds dP) and blocks of
 *   32 queries (column view, feeds dV);
 *   dP = dO_row . V8;  dS = P*(dP - D) with the FP32 P;
 *   Pq: P in blocks of 32 queries, E4M3 under orc_p_block_exponent; dS_row:
 *   blocks of 32 keys; dS_col: blocks of 32 queries (MXFP8, OCP rule);
 *   dV = sum_q Pq^T dO_col;  dK = scale * sum_q dS_col^T Q8;
 *   dQ = scale * sum_k dS_row K8; dK, dV summed over a GQA group.
 *   Blocks of 32 are aligned to absolute positions 32a and cover masked or
 *   out-of-range positions as zeros.
 * mode 1 (identity quantizers, pins): no quantization anywhere, s in FP64,
 *   P = exp(scale*s - LSE).
 *
 * qrows[r] = (b*Hq + h)*N + i selects rows of dQ (dQ_out[r*d..]);
 * krows[r] = (b*Hkv + hk)*N + n selects rows of dK/dV (dK_out, dV_out).
 * A P or dS block along queries needs the 32 queries of its block, and a
 * dS_row block needs its 32 keys, so each selected row recomputes the
 * 32x(all) or (all)x32 strip it depends on.  Slow and plain on purpose. */

typedef struct {
    const float *Q4, *K4, *Q8, *K8, *V8, *O, *dO, *LSE;
    int B, Hq, Hkv, N, d, causal, mode;
    float scale, c, lse2e;
} bwd_ctx;

static double dot_f(const float* a, const float* b, int d) {
    double acc = 0.0;
    for (int t = 0; t < d; ++t) acc += (double)a[t] * (double)b[t];
    return acc;
}

/* P and dS for query i of head (b,h) against key n (unquantized, FP32-valued
 * in mode 0).  Returns 0 for masked or out-of-range pairs. */
static void p_ds(const bwd_ctx* x, int b, int h, int i, int n, const double* Drow,
                 const double* dOrow, double* P, double* dS) {
    *P = 0.0;
    *dS = 0.0;
    if (i >= x->N || n >= x->N || (x->causal && n > i)) return;
    int hk = h / (x->Hq / x->Hkv);
    long qoff = (((long)b * x->Hq + h) * x->N + i) * x->d;
    long koff = (((long)b * x->Hkv + hk) * x->N + n) * x->d;
    double s = dot_f(x->Q4 + qoff, x->K4 + koff, x->d);
    double lse = x->LSE[((long)b * x->Hq + h) * x->N + i];
    double p;
    if (x->mode == 0) {
        float xs = fmaf((float)s, x->c, -(float)((float)lse * x->lse2e));
        p = (double)(float)exp2((double)xs);
    } else {
        p = exp((double)x->scale * s - lse);
    }
    /* dP from the dO row view (already round-tripped in mode 0) and V8 */
    double dp = 0.0;
    const float* v = x->V8 + koff;
    for (int t = 0; t < x->d; ++t) dp += dOrow[t] * (double)v[t];
    *P = p;
    *dS = p * (dp - *Drow);
}

/* dO row view (blocks along d) and D for query i of head (b,h). */
static void drow_of(const bwd_ctx* x, int b, int h, int i, double* dOrow, double* D) {
    long off = (((long)b * x->Hq + h) * x->N + i) * x->d;
    double acc = 0.0;
    for (int t = 0; t < x->d; ++t) {
        dOrow[t] = x->dO[off + t];
        acc += (double)x->dO[off + t] * (double)x->O[off + t];
    }
    *D = acc;
    if (x->mode == 0)
        for (int blk = 0; blk < x->d; blk += 32) mxfp8_roundtrip(dOrow + blk, 32, 1);
}

ORC_API void orc_bwd(const float* Q4, const float* K4, const float* Q8, const float* K8,
                     const float* V8, const float* O, const float* dO, const float* LSE,
                     int B, int Hq, int Hkv, int N, int d, float softmax_scale, int causal,
                     int mode, long nq, const int64_t* qrows, double* dQ_out, long nk,
                     const int64_t* krows, double* dK_out, double* dV_out) {
    bwd_ctx x;
    x.Q4 = Q4; x.K4 = K4; x.Q8 = Q8; x.K8 = K8; x.V8 = V8; x.O = O; x.dO = dO; x.LSE = LSE;
    x.B = B; x.Hq = Hq; x.Hkv = Hkv; x.N = N; x.d = d; x.causal = causal; x.mode = mode;
    if (softmax_scale <= 0.0f) softmax_scale = (float)(1.0 / sqrt((double)d));
    x.scale = softmax_scale;
    x.c = (float)((double)softmax_scale * 1.4426950408889634);
    x.lse2e = (float)1.4426950408889634;
    const int group = Hq / Hkv;

    /* dQ rows: dQ_i = scale * sum_n q8(dS_i,n; blocks of 32 keys) * K8_n */
    #pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < nq; ++r) {
        int64_t row = qrows[r];
        int i = (int)(row % N), h = (int)((row / N) % Hq), b = (int)(row / ((int64_t)N * Hq));
        int hk = h / group;
        double* dOrow = (double*)malloc(sizeof(double) * d);
        double* ds = (double*)malloc(sizeof(double) * (((N + 31) / 32) * 32));
        double D;
        drow_of(&x, b, h, i, dOrow, &D);
        int nkeys = ((N + 31) / 32) * 32;
        for (int n = 0; n < nkeys; ++n) {
            double P;
            p_ds(&x, b, h, i, n, &D, dOrow, &P, &ds[n]);
        }
        if (mode == 0)
            for (int blk = 0; blk < nkeys; blk += 32) mxfp8_roundtrip(ds + blk, 32, 1);
        double* out = dQ_out + r * (long)d;
        for (int t = 0; t < d; ++t) out[t] = 0.0;
        for (int n = 0; n < N; ++n) {
            if (ds[n] == 0.0) continue;
            const float* k = K8 + (((long)b * Hkv + hk) * N + n) * (long)d;
            for (int t = 0; t < d; ++t) out[t] += ds[n] * (double)k[t];
        }
        for (int t = 0; t < d; ++t) out[t] *= (double)softmax_scale;
        free(dOrow);
        free(ds);
    }

    /* dK/dV rows: for key n, sum over the heads of the group and all queries.
     * P and dS are quantized in blocks of 32 queries (one block = one strip of
     * 32 queries against this key); the dO column view is quantized in the
     * same 32-query blocks, per channel. */
    #pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < nk; ++r) {
        int64_t row = krows[r];
        int n = (int)(row % N), hk = (int)((row / N) % Hkv), b = (int)(row / ((int64_t)N * Hkv));
        double* dk = dK_out + r * (long)d;
        double* dv = dV_out + r * (long)d;
        for (int t = 0; t < d; ++t) { dk[t] = 0.0; dv[t] = 0.0; }
        double* dOrow = (double*)malloc(sizeof(double) * d);
        double* dOcol = (double*)malloc(sizeof(double) * 32 * d);
        double Pb[32], dSb[32];
        for (int hh = 0; hh < group; ++hh) {
            int h = hk * group + hh;
            for (int i0 = 0; i0 < N; i0 += 32) {
                int cnt = N - i0 < 32 ? N - i0 : 32;
                for (int u = 0; u < 32; ++u) {
                    Pb[u] = 0.0;
                    dSb[u] = 0.0;
                    for (int t = 0; t < d; ++t) dOcol[u * d + t] = 0.0;
                    if (u >= cnt) continue;
                    int i = i0 + u;
                    double D;
                    drow_of(&x, b, h, i, dOrow, &D);
                    p_ds(&x, b, h, i, n, &D, dOrow, &Pb[u], &dSb[u]);
                    long off = (((long)b * Hq + h) * N + i) * (long)d;
                    for (int t = 0; t < d; ++t) dOcol[u * d + t] = dO[off + t];
                }
                if (mode == 0) {
                    p_e4m3_roundtrip(Pb, 32);
                    mxfp8_roundtrip(dSb, 32, 1);
                    for (int t = 0; t < d; ++t) mxfp8_roundtrip(dOcol + t, 32, d);
                }
                for (int u = 0; u < cnt; ++u) {
                    const float* q = Q8 + (((long)b * Hq + h) * N + i0 + u) * (long)d;
                    for (int t = 0; t < d; ++t) {
                        dv[t] += Pb[u] * dOcol[u * d + t];
                        dk[t] += dSb[u] * (double)q[t];
                    }
                }
            }
        }
        for (int t = 0; t < d; ++t) dk[t] *= (double)softmax_scale;
        free(dOrow);
        free(dOcol);
    }
}

/* Unquantized FP64 softmax attention for the error report (not a parity
 * reference): O = softmax(scale * Q K^T [masked]) V on raw inputs. */
ORC_API void orc_attention_fp64(const float* Q, const float* K, const float* V, int B, int Hq,
                                int Hkv, int N, int d, float softmax_scale, int causal,
                                long nrows, const int64_t* rows, double* O_out) {
    if (softmax_scale <= 0.0f) softmax_scale = (float)(1.0 / sqrt((double)d));
    const int group = Hq / Hkv;
    #pragma omp parallel for schedule(dynamic, 4)
    for (long r = 0; r < nrows; ++r) {
        int64_t row = rows[r];
        int i = (int)(row % N), h = (int)((row / N) % Hq), b = (int)(row / ((int64_t)N * Hq));
        int hk = h / group;
        const float* q = Q + row * (long)d;
        int last = causal ? i : N - 1;
        double* s = (double*)malloc(sizeof(double) * (last + 1));
        double mx = -INFINITY;
        for (int n = 0; n <= last; ++n) {
            s[n] = softmax_scale * dot_f(q, K + (((long)b * Hkv + hk) * N + n) * (long)d, d);
            if (s[n] > mx) mx = s[n];
        }
        double l = 0.0;
        double* o = O_out + r * (long)d;
        for (int t = 0; t < d; ++t) o[t] = 0.0;
        for (int n = 0; n <= last; ++n) {
            double p = exp(s[n] - mx);
            l += p;
            const float* v = V + (((long)b * Hkv + hk) * N + n) * (long)d;
            for (int t = 0; t < d; ++t) o[t] += p * (double)v[t];
        }
        for (int t = 0; t < d; ++t) o[t] /= l;
        free(s);
    }
}

ORC_API int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
