// internal.h -- host-side declarations shared by the library's translation
// units (kernel launchers and their parameter blocks).  Not part of the ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa4 {

struct Thresh { float v[7]; };

// Round N up to the padded key length of the along-N layouts.
inline int padded_n(int N) { return (N + 127) / 128 * 128; }

// ---------------------------------------------------------------- quantize
// Q, K (MXFP4 along d) and V (MXFP4 along N) in one launch.
struct QkvParams {
  const uint4* q;
  const uint4* k;
  const void* v;               // bf16
  uint8_t *qc, *qs, *kc, *ks, *vc, *vs;
  int N, Np;
  long long nbq, nbk;          // 32-element blocks of Q and K
  long long nq_cta, nk_cta;    // CTAs of 512 row blocks
  long long nvw;               // 32-token V blocks (one warp each)
  long long nv;                // V CTAs (8 blocks each)
  long long period;            // every period-th CTA (of the first nv) is a V tile
};
cudaError_t launch_quantize_qkv(const void* q, const void* k, const void* v, long long BHq, long long BHkv,
                                int N, int d, void* qc, void* qs, void* kc, void* ks, void* vc, void* vs,
                                cudaStream_t st);
// NVFP4 along d of n bf16 values (n a multiple of 16): codes, E4M3 scales per
// 16, the FP32 tensor scale into *ts (device).
cudaError_t launch_quantize_nvfp4(const void* x, long long n, void* codes, void* scales, float* ts,
                                  cudaStream_t st);
cudaError_t launch_quantize(const void* x, long long rows, int d, int N, long long BH, int fmt,
                            int axis, void* codes, void* scales, cudaStream_t st);

// ---------------------------------------------------------------- FP4 fwd
struct FwdFp4Params {
  CUtensorMap tm_q, tm_k, tm_v;     // MXFP4 codes of Q, K (along d); V^T (along N): MXFP4,
                                    // or MXFP8 for the FP8 P/V route
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  void* o;
  float* lse;
  unsigned* err;
  int B, Hq, Hkv, N, d, Np, causal, out_bf16;
  int o_align32;                    // O 32-byte aligned: the epilogue writes 32-byte words
  int fp8pv;                        // 0: Direct-P (E2M1 P); 1: FP8 P/V route (E4M3 P and V)
  const float* ts_q;                // NVFP4 Q/K: device tensor scales; nullptr for MXFP4 Q/K
  const float* ts_k;
  const void* q_bf16;               // bf16 Q quantized in the kernel's prologue (tm_q unused), or nullptr
  float scale, c;                   // softmax scale, fl32(scale*log2 e)
  float T[7];                       // Direct-P thresholds
};
cudaError_t launch_fwd_fp4(const FwdFp4Params& p, cudaStream_t st);
cudaError_t launch_directp_codes(const float* s, long long n, float m, float c, const float* T,
                                 int native, uint8_t* codes, cudaStream_t st);

cudaError_t launch_watchdog_selftest(unsigned* err, unsigned long long limit_ns, cudaStream_t st);

// ---------------------------------------------------------------- BF16 fwd
struct FwdBf16Params {
  CUtensorMap tm_q, tm_k, tm_v;     // bf16 Q, K, V
  void* o;
  float* lse;
  unsigned* err;
  int B, Hq, Hkv, N, d, causal, out_bf16;
  float scale, c;
};
cudaError_t launch_fwd_bf16(const FwdBf16Params& p, cudaStream_t st);

// ---------------------------------------------------------------- bwd
struct BwdParams {
  CUtensorMap tm_q4, tm_k4;          // MXFP4 codes (along d)
  CUtensorMap tm_q8c, tm_k8c;        // MXFP8 column views [bh][d][Np]
  CUtensorMap tm_v8r;                // MXFP8 row view of V [bh][N][d]
  CUtensorMap tm_do_r, tm_do_c;      // MXFP8 views of dO (workspace)
  CUtensorMap tm_dq;                 // dq fp32 [bh][N][d], for bulk reductions
  CUtensorMap tm_fold;               // [bh][N] x 16 B: bf16 parts of -LSE log2 e / c and -D (workspace)
  const uint8_t *q4_s, *k4_s, *q8c_s, *k8c_s, *v8r_s, *do_r_s, *do_c_s;
  float *dq, *dk, *dv;
  unsigned* err;
  int B, Hq, Hkv, N, d, Np, causal;
  float scale, c, l2e;
};
struct BwdPrepParams {
  const void* o;
  const void* dout;
  int o_bf16;
  int B, Hq, N, d, Np;
  uint8_t *do_r, *do_r_s, *do_c, *do_c_s;
  const float* lse;
  float c, l2e;
  uint4* fold;                       // per row: bf16 parts of -LSE log2 e / c and of -D
  float* dq;
};
cudaError_t launch_bwd_prep(const BwdPrepParams& p, cudaStream_t st);
cudaError_t launch_bwd_main(const BwdParams& p, cudaStream_t st);

}  // namespace fa4
