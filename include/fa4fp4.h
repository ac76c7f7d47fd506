/*
 * fa4fp4.h -- C ABI of the GB300 (sm_103a) block-scaled FP4 attention library
 * with Direct-P.
 *
 * The method is the one described in "Hardware-Aware FP4 FlashAttention-4"
 * (arXiv:2609.04105; gist.science technical summary and the arXiv abstract):
 * Q and K quantized to E2M1 with power-of-two (E8M0) scales per 32 elements,
 * S = Q K^T on FP4 tensor cores, each score's offset from the running row max
 * mapped straight to an E2M1 probability code, P V on FP4 tensor cores with an
 * online-softmax rescale of O, and a causal backward that rebuilds P from the
 * saved quantized Q and K and uses FP8 E4M3 operands.
 *
 * Conventions shared by every call:
 *   - Pointers are DEVICE pointers, allocated and owned by the caller, except
 *     the host buffers of fa4fp4_fwd_host.  The library never allocates or
 *     frees memory and never synchronizes, except in fa4fp4_sync_status.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every compute call is asynchronous on it; the return value
 *     reports host-side argument validation and launch errors only.  Device
 *     watchdog errors (a pipeline wait that ran out of time) are reported by
 *     fa4fp4_sync_status.
 *   - Tensors are dense and row-major in the layouts stated below; every
 *     pointer must be 16-byte aligned (FA4FP4_ERR_ALIGNMENT otherwise).
 *   - Supported shapes: d in {64, 128}; N >= 1; B, H >= 0; Hq % Hkv == 0;
 *     causal attention uses the same N for queries and keys, aligned top-left
 *     (key n is visible to query i iff n <= i).
 *   - An empty problem (B == 0, or H == 0 / Hq == 0) is a no-op: the call
 *     checks its shape and options, then returns FA4FP4_OK without inspecting
 *     its pointers (they may be NULL) and without launching anything.
 *   - softmax_scale <= 0 selects 1/sqrt(d).
 *   - No C++ exception crosses this boundary; there is no CPU fallback.
 *
 * Quantized tensor layouts ("qtensor": a codes buffer plus a scales buffer):
 *   blocks along d (FA4FP4_BLOCKS_ALONG_D), logical x[B][H][N][d]:
 *       codes  [B][H][N][d/2] bytes (MXFP4: two E2M1 codes per byte, element
 *              2i in the low nibble) or [B][H][N][d] bytes (MXFP8: E4M3)
 *       scales [B][H][N][d/32] E8M0 bytes
 *   blocks along N (FA4FP4_BLOCKS_ALONG_N), stored transposed, Np = N rounded
 *   up to a multiple of 128, positions >= N hold +0:
 *       codes  [B][H][d][Np/2] (MXFP4) or [B][H][d][Np] (MXFP8)
 *       scales [B][H][d][Np/32]
 */
#ifndef FA4FP4_H
#define FA4FP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA4FP4_API __attribute__((visibility("default")))
#else
#define FA4FP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA4FP4_OK = 0,
  FA4FP4_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad enum */
  FA4FP4_ERR_UNSUPPORTED = 2,    /* d not in {64,128}, Hq % Hkv != 0, ... */
  FA4FP4_ERR_ALIGNMENT = 3,      /* a pointer is not 16-byte aligned */
  FA4FP4_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
  FA4FP4_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait expired */
  FA4FP4_ERR_WORKSPACE = 6       /* workspace missing or too small */
} fa4fp4_status;

typedef enum { FA4FP4_FMT_MXFP4 = 0, FA4FP4_FMT_MXFP8_E4M3 = 1 } fa4fp4_format;
typedef enum { FA4FP4_BLOCKS_ALONG_D = 0, FA4FP4_BLOCKS_ALONG_N = 1 } fa4fp4_axis;
typedef enum { FA4FP4_OUT_F32 = 0, FA4FP4_OUT_BF16 = 1 } fa4fp4_out_dtype;

/* Bytes of the codes buffer of a quantized tensor; *scale_bytes (if not NULL)
 * receives the bytes of its scales buffer.  Returns 0 for invalid arguments. */
FA4FP4_API size_t fa4fp4_qtensor_bytes(int B, int H, int N, int d, int fmt, int axis, size_t* scale_bytes);

/* Block quantization (technical summary, Methodology 1 "Format Selection";
 * Methodology 2 "Gradient Formats").  x_bf16 is [B][H][N][d] bf16.  Each block
 * of 32 elements along `axis` gets the E8M0 exponent X = floor(log2(amax)) -
 * emax (emax 2 for E2M1, 8 for E4M3; OCP MX rule; clamped to [-127,127]); each
 * element is x * 2^-X rounded to nearest-even on the element grid, saturating,
 * with its sign kept.  Writes codes/scales in the layouts above. */
FA4FP4_API fa4fp4_status fa4fp4_quantize(const void* x_bf16, int B, int H, int N, int d, int fmt, int axis,
                              void* codes, void* scales, void* stream);

/* The three forward inputs in one launch: q [B][Hq][N][d] and k [B][Hkv][N][d]
 * to MXFP4 with blocks along d, v [B][Hkv][N][d] to MXFP4 with blocks along N
 * (the transposed V^T layout), byte for byte what fa4fp4_quantize writes for
 * each of them (same rule, layouts and sizes: fa4fp4_qtensor_bytes);
 * technical summary, Methodology 1 ("Format Selection": MXFP4 Q, K and V).
 * The transposes of V share the grid with the row blocks of Q and K.  All
 * buffers are device memory owned by the caller, 16-byte aligned; errors as
 * fa4fp4_fwd's dimension checks (d in {64,128}, Hq a multiple of Hkv). */
FA4FP4_API fa4fp4_status fa4fp4_quantize_qkv(const void* q_bf16, const void* k_bf16, const void* v_bf16,
                                             int B, int Hq, int Hkv, int N, int d, void* q_codes,
                                             void* q_scales, void* k_codes, void* k_scales,
                                             void* vt_codes, void* vt_scales, void* stream);

/* Direct-P forward (technical summary, Methodology 1 "Direct Mapping" and
 * "Consistent Normalization"; abstract).
 *   q: MXFP4 along d, [B][Hq][N][d];  k: MXFP4 along d, [B][Hkv][N][d];
 *   vt: MXFP4 along N (transposed V), [B][Hkv][d][Np].
 *   Query head h reads kv head h / (Hq/Hkv).
 * Per 128-query tile, key tiles of 128 are visited in ascending order; for
 * key tile j the running max m_j = max(m_{j-1}, row max of S_j); each score s
 * gets the E2M1 code #{k : fmaf(s, c, -fl32(m_j*c)) >= T_k}, c =
 * fl32(softmax_scale*log2 e), T_k the smallest FP32 x with RNE_E2M1(6*2^x) >=
 * the k-th E2M1 magnitude; P blocks carry the unit E8M0 scale; O and the
 * normalizer l are rescaled by 2^(c(m_{j-1}-m_j)) before P_j V_j is added and
 * l accumulates the same code values.  Output o = O/l ([B][Hq][N][d], f32 or
 * bf16 per out_dtype) and, if lse != NULL, lse[B][Hq][N] = softmax_scale*m +
 * ln(l/6) (f32). */
FA4FP4_API fa4fp4_status fa4fp4_fwd(const void* q_codes, const void* q_scales, const void* k_codes,
                         const void* k_scales, const void* vt_codes, const void* vt_scales,
                         int B, int Hq, int Hkv, int N, int d, float softmax_scale, int causal,
                         void* o, int out_dtype, float* lse, void* stream);

/* The inference step end to end on HOST buffers: bf16 q [B][Hq][N][d] and k,
 * v [B][Hkv][N][d] in host memory, o (f32 or bf16 per out_dtype,
 * [B][Hq][N][d]) and lse (nullable, f32 [B][Hq][N]) written to host memory;
 * on the device, fa4fp4_quantize_qkv and fa4fp4_fwd (technical summary,
 * Methodology 1: MXFP4 Q, K, V and the Direct-P forward), with the same
 * results as those two calls on the same data.  The pages have no
 * counterpart; this is the library's end-to-end entry point.  The work is cut
 * into chunks of consecutive (batch element, kv head) units with their query
 * heads, the last chunk a single unit; each chunk's inputs are copied in on
 * an internal stream, quantized and attended alternately on `stream` and a
 * second internal stream, and copied out on a third, two chunks' staging
 * buffers in flight, so that the copies overlap the compute.
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to overlap; q, k, v, o must be 16-byte aligned and lse 4-byte
 * aligned.  `workspace` is DEVICE memory of at least
 * fa4fp4_fwd_host_workspace_bytes(B, Hq, Hkv, N, d) bytes, 16-byte aligned
 * (FA4FP4_ERR_WORKSPACE if missing or too small), used as staging; calls in
 * flight at the same time need their own workspaces.  The call is
 * asynchronous on `stream`: later work on `stream` sees o and lse in host
 * memory, and the call starts after earlier work on `stream`.  The first call
 * on a device creates three streams and seven events on it, kept until the
 * process exits.  Other errors as fa4fp4_fwd's; all checks are made before
 * anything is enqueued, and a CUDA failure while enqueuing returns
 * FA4FP4_ERR_CUDA with the chunks before it already enqueued. */
FA4FP4_API size_t fa4fp4_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int N, int d);
FA4FP4_API fa4fp4_status fa4fp4_fwd_host(const void* q_host, const void* k_host, const void* v_host, int B,
                                         int Hq, int Hkv, int N, int d, float softmax_scale, int causal,
                                         void* o_host, int out_dtype, float* lse_host, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* The FP8 P/V training route of the forward (technical summary, Methodology 2
 * "Stability Constraint" and Training Performance: the retained training route
 * keeps FP8 probabilities and values).  Same arguments, layouts and errors as
 * fa4fp4_fwd except V: v8_codes/v8_scales is V quantized to MXFP8 with blocks
 * along N (fa4fp4_quantize with FA4FP4_FMT_MXFP8_E4M3, FA4FP4_BLOCKS_ALONG_N:
 * E4M3 codes [B][Hkv][d][Np], scales [B][Hkv][d][Np/32]).  Per 128-key tile
 * in ascending order: S = Q K^T on FP4 tensor cores, running max m, p =
 * 2^x with x = fl32(fl32(s - m) c) in FP32 (hardware exponential; the row max
 * gets p = 1 exactly), P rounded to E4M3
 * with one E8M0 scale per 32 keys (the least X with amax <= 448 * 2^X, so no
 * element saturates), O += P V and l += P 1 on
 * FP8 tensor cores (kind::mxf8f6f4), eager rescale when m grows.  Outputs
 * O / l and LSE = softmax_scale * m + ln(l). */
FA4FP4_API fa4fp4_status fa4fp4_fwd_fp8pv(const void* q_codes, const void* q_scales, const void* k_codes,
                                          const void* k_scales, const void* v8_codes, const void* v8_scales,
                                          int B, int Hq, int Hkv, int N, int d, float softmax_scale, int causal,
                                          void* o, int out_dtype, float* lse, void* stream);

/* NVFP4 block quantization along d (technical summary, Methodology 1
 * "Format Selection": NVFP4 for Q and K, for its fine-grained scaling; the
 * public NVFP4 layout).  x_bf16 is [B][H][N][d] bf16.  Writes codes
 * [B][H][N][d/2] (E2M1, element 2i in the low nibble), scales [B][H][N][d/16]
 * (unsigned E4M3, one per 16 elements) and *ts, the tensor's FP32 scale, in
 * device memory.  Every step is an FP32 operation rounded to nearest: ts =
 * amax/2688 (1 for an all-zero tensor), block scale E4M3(amax_b / (6 ts)),
 * element E2M1(x / (block scale * ts)), saturating, sign kept; a block whose
 * scale rounds to zero gets signed zeros.  Three launches on `stream` (tensor
 * amax, tensor scale, blocks); *ts is also their scratch word. */
FA4FP4_API fa4fp4_status fa4fp4_quantize_nvfp4(const void* x_bf16, int B, int H, int N, int d, void* codes,
                                               void* scales, float* ts, void* stream);

/* The forward with NVFP4 Q and K (from fa4fp4_quantize_nvfp4): q_ts and k_ts
 * point to their device tensor scales.  S = Q K^T runs as tcgen05 kind::mxf4nvf4
 * (UE4M3 scales per 16); the two tensor scales fold into the softmax scale,
 * fl32(fl32(softmax_scale * q_ts) * k_ts), which also enters the LSE.  fp8pv
 * selects the P/V path: 0 = Direct-P with V^T as MXFP4 (fa4fp4_fwd), 1 = the
 * FP8 P/V route with V^T as MXFP8 (fa4fp4_fwd_fp8pv).  Other arguments and
 * errors as fa4fp4_fwd. */
FA4FP4_API fa4fp4_status fa4fp4_fwd_nvfp4(const void* q_codes, const void* q_scales, const float* q_ts,
                                          const void* k_codes, const void* k_scales, const float* k_ts,
                                          const void* vt_codes, const void* vt_scales, int B, int Hq, int Hkv,
                                          int N, int d, float softmax_scale, int causal, int fp8pv, void* o,
                                          int out_dtype, float* lse, void* stream);

/* Direct-P forward (or the FP8 P/V route, fp8pv = 1) with Q in bf16: Q is
 * quantized to MXFP4 (E8M0 per 32 along d, the fa4fp4_quantize rule) inside
 * the forward's prologue, so an inference step reads Q once and needs no
 * separate pass over it (technical summary, Methodology 2 "Gradient Formats":
 * quantization happens where the operands are produced, not as a pass of its
 * own).  q: bf16 [B][Hq][N][d]; k, vt as in fa4fp4_fwd (vt MXFP8 along N when
 * fp8pv = 1).  Results are identical, bit for bit, to fa4fp4_quantize of Q
 * followed by fa4fp4_fwd (fa4fp4_fwd_fp8pv).  Errors as fa4fp4_fwd. */
FA4FP4_API fa4fp4_status fa4fp4_fwd_qbf16(const void* q, const void* k_codes, const void* k_scales,
                               const void* vt_codes, const void* vt_scales, int B, int Hq, int Hkv,
                               int N, int d, float softmax_scale, int causal, int fp8pv, void* o,
                               int out_dtype, float* lse, void* stream);

/* K (MXFP4 along d) and V (MXFP4 along N, transposed) in one launch: the
 * operands fa4fp4_fwd_qbf16 takes quantized.  Byte-identical to two
 * fa4fp4_quantize calls.  k, v: bf16 [B][Hkv][N][d]; outputs in the layouts
 * of fa4fp4_qtensor_bytes. */
FA4FP4_API fa4fp4_status fa4fp4_quantize_kv(const void* k, const void* v, int B, int Hkv, int N, int d,
                                 void* k_codes, void* k_scales, void* vt_codes, void* vt_scales,
                                 void* stream);

/* Bytes of caller-provided workspace fa4fp4_bwd needs. */
FA4FP4_API size_t fa4fp4_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d);

/* Quantized causal backward (technical summary, Methodology 2 "Quantized
 * Causal Backward": P recomputed from the forward's FP4 Q/K and its LSE;
 * FP8 copies of Q, K and V blocked along each product's contraction axis;
 * abstract: FP8 gradient operands).
 *   q4, k4: the forward's MXFP4 Q/K (along d);
 *   q8c, k8c: MXFP8 Q/K blocked along N ([B][H][d][Np] transposed views);
 *   v8r: MXFP8 V blocked along d ([B][Hkv][N][d]);
 *   o: forward output [B][Hq][N][d] (f32 or bf16 per o_dtype);
 *   dout: upstream gradient, bf16 [B][Hq][N][d];  lse: f32 [B][Hq][N].
 * Computes P = 2^x with x = fl32(s' c), s' = S + fl32(-fl32(lse*log2 e) / c)
 * accumulated by the tensor core (S the FP4 product, c = scale*log2 e; within
 * a few units in the last place of fmaf(S, c, -fl32(lse*log2 e))),
 * D = rowsum(dO*O), the MXFP8
 * views of dO (blocks along d and blocks of 32 queries), dP = dO V^T, dS =
 * P*(dP-D), and, with P and dS quantized to MXFP8 (P and dS in blocks of 32
 * queries for dV/dK, dS in blocks of 32 keys for dQ; P's blocks take the
 * least X with amax <= 448 * 2^X, dS's the OCP MX exponent):
 *   dV = P^T dO, dK = scale * dS^T Q, dQ = scale * dS K
 * summed over the query heads of each kv head.  dq [B][Hq][N][d], dk/dv
 * [B][Hkv][N][d], all f32, fully overwritten.  `workspace` must hold
 * fa4fp4_bwd_workspace_bytes(...) bytes (FA4FP4_ERR_WORKSPACE otherwise); it
 * receives the MXFP8 views of dO and, per query row, -fl32(lse*log2 e) / c and
 * -D as bf16 parts (16 bytes), and must not be shared with another
 * call in flight.  d = 64 or 128. */
FA4FP4_API fa4fp4_status fa4fp4_bwd(const void* q4_codes, const void* q4_scales, const void* k4_codes,
                         const void* k4_scales, const void* q8c_codes, const void* q8c_scales,
                         const void* k8c_codes, const void* k8c_scales, const void* v8r_codes,
                         const void* v8r_scales, const void* o, int o_dtype, const void* dout,
                         const float* lse, int B, int Hq, int Hkv, int N, int d,
                         float softmax_scale, int causal, float* dq, float* dk, float* dv,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Size of the fixed device scratch array used by fa4fp4_bwd_noalloc. */
#define FA4FP4_BWD_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* fa4fp4_bwd for callers that cannot allocate device memory (plugins whose
 * host framework owns every device allocation, runtimes that forbid
 * allocation after start-up, code whose device memory is budgeted up front).
 * The paper has no counterpart: this is a deployment variant of fa4fp4_bwd.
 * Same arguments and results as fa4fp4_bwd without the workspace, and the
 * same status for a bad argument; the scratch is a fixed
 * FA4FP4_BWD_NOALLOC_SCRATCH_BYTES device array inside this library (held by
 * every GPU that loads it until exit).  Returns FA4FP4_ERR_WORKSPACE when
 * fa4fp4_bwd_workspace_bytes(...) exceeds that size.  Allocates nothing.
 * The first call on a device looks up the array's device address on that
 * device; make that first call before any stream capture.  All calls share
 * the array: calls that overlap on the GPU (other streams or host threads)
 * race on it. */
FA4FP4_API fa4fp4_status fa4fp4_bwd_noalloc(
    const void* q4_codes, const void* q4_scales, const void* k4_codes, const void* k4_scales,
    const void* q8c_codes, const void* q8c_scales, const void* k8c_codes, const void* k8c_scales,
    const void* v8r_codes, const void* v8r_scales, const void* o, int o_dtype, const void* dout,
    const float* lse, int B, int Hq, int Hkv, int N, int d, float softmax_scale, int causal,
    float* dq, float* dk, float* dv, void* stream);

/* BF16 FlashAttention forward, the speedup reference for fa4fp4_fwd
 * (technical summary, Results: the BF16 kernel its speedups are measured
 * against).  q [B][Hq][N][d], k/v
 * [B][Hkv][N][d] bf16; exact online softmax with P rounded to bf16 for the
 * P V product.  o as in fa4fp4_fwd; lse (nullable) = natural-log LSE. */
FA4FP4_API fa4fp4_status fa4bf16_fwd(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                          int N, int d, float softmax_scale, int causal, void* o, int out_dtype,
                          float* lse, void* stream);

/* Direct-P code map on its own, with the device routines fa4fp4_fwd uses
 * (technical summary, Methodology 1 "Direct Mapping", which allows hardware
 * exponentials for part of the classification).
 * For every score: codes[i] = #{k : fmaf(s[i], c, -fl32(m*c)) >= T_k}.
 * native_exp = 0 computes it with the threshold count; native_exp = 1 with
 * the forward's route: e = ex2(x), codes of 6e(1-2^-18) and 6e(1+2^-18), the
 * threshold count only where those two differ.  Both give identical codes.
 * s: n FP32 scores, codes: n bytes (device arrays). */
FA4FP4_API fa4fp4_status fa4fp4_directp_codes(const float* s, int64_t n, float m, float c,
                                              int native_exp, uint8_t* codes, void* stream);

/* Watchdog self-test: launches one CTA whose pipeline wait can never be
 * satisfied, bounded by limit_ns (0 < limit_ns <= 2e9).  The wait expires,
 * the kernel returns, and the next fa4fp4_sync_status reports
 * FA4FP4_ERR_DEVICE_TIMEOUT; the context stays usable.  Exercises the same
 * bounded-wait routine every kernel of the library uses (2 s limit). */
FA4FP4_API fa4fp4_status fa4fp4_watchdog_selftest(int64_t limit_ns, void* stream);

/* Synchronizes `stream`, then returns FA4FP4_ERR_CUDA for a pending CUDA error
 * or FA4FP4_ERR_DEVICE_TIMEOUT if any kernel's bounded wait expired since the
 * last call (the flag is cleared), else FA4FP4_OK. */
FA4FP4_API fa4fp4_status fa4fp4_sync_status(void* stream);

/* Static description of a status code. */
FA4FP4_API const char* fa4fp4_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA4FP4_H */
