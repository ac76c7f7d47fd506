// api.cu -- the C ABI declared in include/fa4fp4.h: argument validation,
// TMA tensor-map encoding, the Direct-P threshold constants, kernel launches
// and the device watchdog word.
#include <cmath>
#include <cstring>
#include <mutex>
#include "../../include/fa4fp4.h"
#include "internal.h"

using namespace fa4;

// Device error word: bounded waits that expire OR a flag in here.
__device__ unsigned g_fa4fp4_err;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};

unsigned* err_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fa4fp4_err) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned*>(ptr);
  }
  return g_err_ptr[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D tiled map over a [d2][d1][d0] tensor of `elem` bytes per element.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int elem, const void* base, uint64_t d0,
              uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * elem, d0 * d1 * elem};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Direct-P thresholds: T_k is the smallest FP32 x for which 6*2^x rounds
// (nearest, ties to even) to at least the k-th E2M1 magnitude.  The rounding
// switches at the midpoint mu_k below magnitude k; a value exactly on mu_k
// rounds up only when magnitude k has an even code (1.0, 2.0, 4.0).
const float* directp_thresholds() {
  static float T[7];
  static std::once_flag once;
  std::call_once(once, [] {
    const double mu[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};
    for (int k = 1; k <= 7; ++k) {
      auto reaches = [&](float x) {
        double v = 6.0 * std::exp2((double)x);
        return v > mu[k - 1] || (v == mu[k - 1] && (k % 2) == 0);
      };
      float x = (float)std::log2(mu[k - 1] / 6.0);
      while (reaches(std::nextafter(x, -INFINITY))) x = std::nextafter(x, -INFINITY);
      while (!reaches(x)) x = std::nextafter(x, INFINITY);
      T[k - 1] = x;
    }
  });
  return T;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

float default_scale(float s, int d) { return s > 0.f ? s : (float)(1.0 / std::sqrt((double)d)); }

fa4fp4_status launch_status(cudaError_t e) { return e == cudaSuccess ? FA4FP4_OK : FA4FP4_ERR_CUDA; }

fa4fp4_status check_dims(int B, int Hq, int Hkv, int N, int d) {
  if (B < 0 || Hq < 0 || Hkv < 0 || N < 1) return FA4FP4_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA4FP4_ERR_UNSUPPORTED;
  if (Hkv == 0 ? Hq != 0 : (Hq % Hkv) != 0) return FA4FP4_ERR_UNSUPPORTED;
  if ((long long)B * Hq * N * d > (1LL << 40)) return FA4FP4_ERR_UNSUPPORTED;
  return FA4FP4_OK;
}

}  // namespace

extern "C" {

const char* fa4fp4_status_string(int s) {
  switch (s) {
    case FA4FP4_OK: return "ok";
    case FA4FP4_ERR_INVALID_ARG: return "invalid argument";
    case FA4FP4_ERR_UNSUPPORTED: return "unsupported shape or option";
    case FA4FP4_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case FA4FP4_ERR_CUDA: return "CUDA error";
    case FA4FP4_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case FA4FP4_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

size_t fa4fp4_qtensor_bytes(int B, int H, int N, int d, int fmt, int axis, size_t* scale_bytes) {
  if (B < 0 || H < 0 || N < 1 || (d != 64 && d != 128) || (fmt != 0 && fmt != 1) ||
      (axis != 0 && axis != 1)) {
    if (scale_bytes) *scale_bytes = 0;
    return 0;
  }
  size_t L = axis == 0 ? (size_t)d : (size_t)padded_n(N);
  size_t R = axis == 0 ? (size_t)N : (size_t)d;
  size_t per = fmt == 0 ? L / 2 : L;
  if (scale_bytes) *scale_bytes = (size_t)B * H * R * (L / 32);
  return (size_t)B * H * R * per;
}

fa4fp4_status fa4fp4_quantize(const void* x, int B, int H, int N, int d, int fmt, int axis,
                              void* codes, void* scales, void* stream) {
  if ((fmt != 0 && fmt != 1) || (axis != 0 && axis != 1)) return FA4FP4_ERR_INVALID_ARG;
  fa4fp4_status s = check_dims(B, H, H, N, d);
  if (s != FA4FP4_OK) return s;
  if (B == 0 || H == 0) return FA4FP4_OK;
  if (!x || !codes || !scales) return FA4FP4_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return FA4FP4_ERR_ALIGNMENT;
  long long BH = (long long)B * H;
  return launch_status(launch_quantize(x, BH * N, d, N, BH, fmt, axis, codes, scales,
                                       static_cast<cudaStream_t>(stream)));
}

fa4fp4_status fa4fp4_quantize_qkv(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                                  int N, int d, void* q_codes, void* q_scales, void* k_codes, void* k_scales,
                                  void* vt_codes, void* vt_scales, void* stream) {
  fa4fp4_status s = check_dims(B, Hq, Hkv, N, d);
  if (s != FA4FP4_OK) return s;
  if (B == 0 || Hq == 0) return FA4FP4_OK;
  const void* ptrs[] = {q, k, v, q_codes, q_scales, k_codes, k_scales, vt_codes, vt_scales};
  for (const void* ptr : ptrs)
    if (!ptr) return FA4FP4_ERR_INVALID_ARG;
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FA4FP4_ERR_ALIGNMENT;
  return launch_status(launch_quantize_qkv(q, k, v, (long long)B * Hq, (long long)B * Hkv, N, d, q_codes,
                                           q_scales, k_codes, k_scales, vt_codes, vt_scales,
                                           static_cast<cudaStream_t>(stream)));
}

// Shared by the Direct-P forward (fp8pv = 0, V^T MXFP4) and the FP8 P/V
// route (fp8pv = 1, V^T MXFP8).
// q_bf16 non-null: Q is bf16 [B][Hq][N][d], quantized to MXFP4 by the
// kernel's prologue (qc, qs unused).
static fa4fp4_status fwd_common(const void* qc, const void* qs, const void* kc, const void* ks,
                                const void* vc, const void* vs, int B, int Hq, int Hkv, int N, int d,
                                float softmax_scale, int causal, void* o, int out_dtype, float* lse,
                                int fp8pv, const float* ts_q, const float* ts_k, void* stream,
                                const void* q_bf16 = nullptr) {
  if (out_dtype != FA4FP4_OUT_F32 && out_dtype != FA4FP4_OUT_BF16) return FA4FP4_ERR_INVALID_ARG;
  fa4fp4_status s = check_dims(B, Hq, Hkv, N, d);
  if (s != FA4FP4_OK) return s;
  if (B == 0 || Hq == 0) return FA4FP4_OK;
  if (q_bf16) {
    qc = qs = q_bf16;     // validated below like the code and scale pointers
  }
  if (!qc || !qs || !kc || !ks || !vc || !vs || !o) return FA4FP4_ERR_INVALID_ARG;
  if ((ts_q == nullptr) != (ts_k == nullptr)) return FA4FP4_ERR_INVALID_ARG;
  if ((ts_q && (reinterpret_cast<uintptr_t>(ts_q) & 3)) || (ts_k && (reinterpret_cast<uintptr_t>(ts_k) & 3)))
    return FA4FP4_ERR_ALIGNMENT;
  const void* ptrs[] = {qc, qs, kc, ks, vc, vs, o};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FA4FP4_ERR_ALIGNMENT;
  if (lse && !aligned16(lse)) return FA4FP4_ERR_ALIGNMENT;
  FwdFp4Params p;
  memset(&p, 0, sizeof(p));
  const int Np = padded_n(N);
  const CUtensorMapSwizzle qsw = d == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  // V^T rows of 128 keys: 64 bytes of E2M1 (64-byte swizzle) or 128 bytes of
  // E4M3 (128-byte swizzle)
  const int vrow = fp8pv ? 128 : 64;
  if ((!q_bf16 && !make_map(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qc, d / 2, N, (uint64_t)B * Hq, d / 2, 128, qsw)) ||
      !make_map(&p.tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kc, d / 2, N, (uint64_t)B * Hkv, d / 2, 128, qsw) ||
      !make_map(&p.tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, vc, fp8pv ? Np : Np / 2, d, (uint64_t)B * Hkv, vrow, d,
                fp8pv ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
    return FA4FP4_ERR_CUDA;
  p.q_scales = static_cast<const uint8_t*>(qs);
  p.k_scales = static_cast<const uint8_t*>(ks);
  p.v_scales = static_cast<const uint8_t*>(vs);
  p.o = o;
  p.lse = lse;
  p.err = err_word();
  if (!p.err) return FA4FP4_ERR_CUDA;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d; p.Np = Np;
  p.causal = causal ? 1 : 0;
  p.out_bf16 = out_dtype == FA4FP4_OUT_BF16;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31) == 0;   // rows are 128 or 256 bytes (bf16) or more
  p.fp8pv = fp8pv;
  p.ts_q = ts_q;
  p.ts_k = ts_k;
  p.q_bf16 = q_bf16;
  p.scale = default_scale(softmax_scale, d);
  p.c = (float)((double)p.scale * 1.4426950408889634);
  const float* T = directp_thresholds();
  for (int k = 0; k < 7; ++k) p.T[k] = T[k];
  return launch_status(launch_fwd_fp4(p, static_cast<cudaStream_t>(stream)));
}

fa4fp4_status fa4fp4_fwd(const void* qc, const void* qs, const void* kc, const void* ks,
                         const void* vc, const void* vs, int B, int Hq, int Hkv, int N, int d,
                         float softmax_scale, int causal, void* o, int out_dtype, float* lse,
                         void* stream) {
  return fwd_common(qc, qs, kc, ks, vc, vs, B, Hq, Hkv, N, d, softmax_scale, causal, o, out_dtype, lse,
                    0, nullptr, nullptr, stream);
}

fa4fp4_status fa4fp4_fwd_fp8pv(const void* qc, const void* qs, const void* kc, const void* ks,
                               const void* v8c, const void* v8s, int B, int Hq, int Hkv, int N, int d,
                               float softmax_scale, int causal, void* o, int out_dtype, float* lse,
                               void* stream) {
  return fwd_common(qc, qs, kc, ks, v8c, v8s, B, Hq, Hkv, N, d, softmax_scale, causal, o, out_dtype, lse,
                    1, nullptr, nullptr, stream);
}

fa4fp4_status fa4fp4_fwd_qbf16(const void* q, const void* kc, const void* ks, const void* vc, const void* vs,
                               int B, int Hq, int Hkv, int N, int d, float softmax_scale, int causal, int fp8pv,
                               void* o, int out_dtype, float* lse, void* stream) {
  if (fp8pv != 0 && fp8pv != 1) return FA4FP4_ERR_INVALID_ARG;
  if (!q && !(B == 0 || Hq == 0)) return FA4FP4_ERR_INVALID_ARG;
  return fwd_common(nullptr, nullptr, kc, ks, vc, vs, B, Hq, Hkv, N, d, softmax_scale, causal, o, out_dtype, lse,
                    fp8pv, nullptr, nullptr, stream, q);
}

fa4fp4_status fa4fp4_quantize_kv(const void* k, const void* v, int B, int Hkv, int N, int d, void* k_codes,
                                 void* k_scales, void* vt_codes, void* vt_scales, void* stream) {
  fa4fp4_status s = check_dims(B, Hkv, Hkv, N, d);
  if (s != FA4FP4_OK) return s;
  if (B == 0 || Hkv == 0) return FA4FP4_OK;
  const void* ptrs[] = {k, v, k_codes, k_scales, vt_codes, vt_scales};
  for (const void* ptr : ptrs)
    if (!ptr) return FA4FP4_ERR_INVALID_ARG;
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FA4FP4_ERR_ALIGNMENT;
  // the Q/K/V launch with no Q rows: its row CTAs all take K
  return launch_status(launch_quantize_qkv(nullptr, k, v, 0, (long long)B * Hkv, N, d, nullptr, nullptr, k_codes,
                                           k_scales, vt_codes, vt_scales, static_cast<cudaStream_t>(stream)));
}

fa4fp4_status fa4fp4_fwd_nvfp4(const void* qc, const void* qs, const float* q_ts, const void* kc,
                               const void* ks, const float* k_ts, const void* vc, const void* vs, int B,
                               int Hq, int Hkv, int N, int d, float softmax_scale, int causal, int fp8pv,
                               void* o, int out_dtype, float* lse, void* stream) {
  if (fp8pv != 0 && fp8pv != 1) return FA4FP4_ERR_INVALID_ARG;
  const bool empty = B == 0 || Hq == 0;
  if (!empty && (!q_ts || !k_ts)) return FA4FP4_ERR_INVALID_ARG;
  return fwd_common(qc, qs, kc, ks, vc, vs, B, Hq, Hkv, N, d, softmax_scale, causal, o, out_dtype, lse,
                    fp8pv, q_ts, k_ts, stream);
}

fa4fp4_status fa4fp4_quantize_nvfp4(const void* x, int B, int H, int N, int d, void* codes, void* scales,
                                    float* ts, void* stream) {
  fa4fp4_status s = check_dims(B, H, H, N, d);
  if (s != FA4FP4_OK) return s;
  if (B == 0 || H == 0) return FA4FP4_OK;
  if (!x || !codes || !scales || !ts) return FA4FP4_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || (reinterpret_cast<uintptr_t>(ts) & 3))
    return FA4FP4_ERR_ALIGNMENT;
  return launch_status(launch_quantize_nvfp4(x, (long long)B * H * N * d, codes, scales, ts,
                                             static_cast<cudaStream_t>(stream)));
}

fa4fp4_status fa4fp4_directp_codes(const float* s, int64_t n, float m, float c, int native_exp,
                                   uint8_t* codes, void* stream) {
  if (!s || !codes || n < 0 || (native_exp != 0 && native_exp != 1)) return FA4FP4_ERR_INVALID_ARG;
  if (n == 0) return FA4FP4_OK;
  return launch_status(launch_directp_codes(s, n, m, c, directp_thresholds(), native_exp, codes,
                                            static_cast<cudaStream_t>(stream)));
}

size_t fa4fp4_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
  if (check_dims(B, Hq, Hkv, N, d) != FA4FP4_OK) return 0;
  const size_t rows = (size_t)B * Hq * N;
  const size_t Np = (size_t)padded_n(N);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  // dO row view (codes + scales), dO column view (codes + scales), 16 bytes
  // per row for the initial values of S^T and dP^T
  return up(rows * d) + up(rows * d / 32) + up((size_t)B * Hq * d * Np) +
         up((size_t)B * Hq * d * Np / 32) + up(rows * 16);
}

fa4fp4_status fa4fp4_bwd(const void* q4c, const void* q4s, const void* k4c, const void* k4s,
                         const void* q8c, const void* q8s, const void* k8c, const void* k8s,
                         const void* v8c, const void* v8s, const void* o, int o_dtype,
                         const void* dout, const float* lse, int B, int Hq, int Hkv, int N, int d,
                         float softmax_scale, int causal, float* dq, float* dk, float* dv,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (o_dtype != FA4FP4_OUT_F32 && o_dtype != FA4FP4_OUT_BF16) return FA4FP4_ERR_INVALID_ARG;
  fa4fp4_status s = check_dims(B, Hq, Hkv, N, d);
  if (s != FA4FP4_OK) return s;
  if (B == 0 || Hq == 0) return FA4FP4_OK;
  const void* ptrs[] = {q4c, q4s, k4c, k4s, q8c, q8s, k8c, k8s, v8c, v8s, o, dout, lse, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr) return FA4FP4_ERR_INVALID_ARG;
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FA4FP4_ERR_ALIGNMENT;
  const size_t need = fa4fp4_bwd_workspace_bytes(B, Hq, Hkv, N, d);
  if (!workspace || workspace_bytes < need) return FA4FP4_ERR_WORKSPACE;
  if (!aligned16(workspace)) return FA4FP4_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int Np = padded_n(N);
  const size_t rows = (size_t)B * Hq * N;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* w = static_cast<uint8_t*>(workspace);
  uint8_t* do_r = w;           w += up(rows * d);
  uint8_t* do_r_s = w;         w += up(rows * d / 32);
  uint8_t* do_c = w;           w += up((size_t)B * Hq * d * Np);
  uint8_t* do_c_s = w;         w += up((size_t)B * Hq * d * Np / 32);
  uint8_t* fold = w;
  const float scale = default_scale(softmax_scale, d);
  const float c = (float)((double)scale * 1.4426950408889634);
  const float l2e = (float)1.4426950408889634;

  BwdPrepParams pp;
  pp.o = o; pp.dout = dout; pp.o_bf16 = o_dtype == FA4FP4_OUT_BF16;
  pp.B = B; pp.Hq = Hq; pp.N = N; pp.d = d; pp.Np = Np;
  pp.do_r = do_r; pp.do_r_s = do_r_s; pp.do_c = do_c; pp.do_c_s = do_c_s; pp.dq = dq;
  pp.lse = lse; pp.c = c; pp.l2e = l2e; pp.fold = reinterpret_cast<uint4*>(fold);
  cudaError_t e = launch_bwd_prep(pp, st);
  if (e != cudaSuccess) return FA4FP4_ERR_CUDA;

  BwdParams p;
  memset(&p, 0, sizeof(p));
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint64_t BHq = (uint64_t)B * Hq, BHk = (uint64_t)B * Hkv;
  // rows along d: d/2 bytes of E2M1 (64- or 32-byte swizzle), d bytes of E4M3
  // (128- or 64-byte swizzle); rows along N: 128 or 64 bytes
  const CUtensorMapSwizzle sw4 = d == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  const CUtensorMapSwizzle sw8 = d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (!make_map(&p.tm_k4, u8, 1, k4c, d / 2, N, BHk, d / 2, 128, sw4) ||
      !make_map(&p.tm_v8r, u8, 1, v8c, d, N, BHk, d, 128, sw8) ||
      !make_map(&p.tm_k8c, u8, 1, k8c, Np, d, BHk, 128, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&p.tm_q4, u8, 1, q4c, d / 2, N, BHq, d / 2, 64, sw4) ||
      !make_map(&p.tm_do_r, u8, 1, do_r, d, N, BHq, d, 64, sw8) ||
      !make_map(&p.tm_q8c, u8, 1, q8c, Np, d, BHq, 64, d, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&p.tm_do_c, u8, 1, do_c, Np, d, BHq, 64, d, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&p.tm_dq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dq, d, N, BHq, d, 32, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&p.tm_fold, u8, 1, fold, 16, N, BHq, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE))
    return FA4FP4_ERR_CUDA;
  p.q4_s = static_cast<const uint8_t*>(q4s);
  p.k4_s = static_cast<const uint8_t*>(k4s);
  p.q8c_s = static_cast<const uint8_t*>(q8s);
  p.k8c_s = static_cast<const uint8_t*>(k8s);
  p.v8r_s = static_cast<const uint8_t*>(v8s);
  p.do_r_s = do_r_s;
  p.do_c_s = do_c_s;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.err = err_word();
  if (!p.err) return FA4FP4_ERR_CUDA;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d; p.Np = Np;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.c = c;
  p.l2e = l2e;
  return launch_status(launch_bwd_main(p, st));
}

fa4fp4_status fa4bf16_fwd(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                          int N, int d, float softmax_scale, int causal, void* o, int out_dtype,
                          float* lse, void* stream) {
  if (out_dtype != FA4FP4_OUT_F32 && out_dtype != FA4FP4_OUT_BF16) return FA4FP4_ERR_INVALID_ARG;
  fa4fp4_status s = check_dims(B, Hq, Hkv, N, d);
  if (s != FA4FP4_OK) return s;
  if (B == 0 || Hq == 0) return FA4FP4_OK;
  if (!q || !k || !v || !o) return FA4FP4_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
    return FA4FP4_ERR_ALIGNMENT;
  FwdBf16Params p;
  memset(&p, 0, sizeof(p));
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&p.tm_q, bf, 2, q, d, N, (uint64_t)B * Hq, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&p.tm_k, bf, 2, k, d, N, (uint64_t)B * Hkv, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&p.tm_v, bf, 2, v, d, N, (uint64_t)B * Hkv, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return FA4FP4_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.err = err_word();
  if (!p.err) return FA4FP4_ERR_CUDA;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d;
  p.causal = causal ? 1 : 0;
  p.out_bf16 = out_dtype == FA4FP4_OUT_BF16;
  p.scale = default_scale(softmax_scale, d);
  p.c = (float)((double)p.scale * 1.4426950408889634);
  return launch_status(launch_fwd_bf16(p, static_cast<cudaStream_t>(stream)));
}

fa4fp4_status fa4fp4_watchdog_selftest(int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 2000000000LL) return FA4FP4_ERR_INVALID_ARG;
  unsigned* w = err_word();
  if (!w) return FA4FP4_ERR_CUDA;
  return launch_status(launch_watchdog_selftest(w, (unsigned long long)limit_ns,
                                                static_cast<cudaStream_t>(stream)));
}

fa4fp4_status fa4fp4_sync_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return FA4FP4_ERR_CUDA;
  unsigned* w = err_word();
  if (!w) return FA4FP4_ERR_CUDA;
  unsigned host = 0;
  if (cudaMemcpy(&host, w, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return FA4FP4_ERR_CUDA;
  if (host) {
    unsigned zero = 0;
    cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    return FA4FP4_ERR_DEVICE_TIMEOUT;
  }
  return FA4FP4_OK;
}

}  // extern "C"
