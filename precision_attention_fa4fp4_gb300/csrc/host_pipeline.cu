// host_pipeline.cu -- the end-to-end inference call on host buffers:
// fa4fp4_fwd_host copies bf16 Q, K, V in from host memory, quantizes them to
// MXFP4, runs the Direct-P forward and copies O (and LSE) back out, all in
// one call.  The work is cut into chunks of (batch, range of kv heads) with
// their query heads; chunk k's inputs are copied in on one internal stream
// while chunk k-1 is quantized and attended on the caller's stream and chunk
// k-2's output is copied out on a second internal stream, so the host link
// and the GPU stay busy together.  Staging buffers (two sets) live in a
// workspace the caller allocates; events order every reuse.
#include <mutex>
#include "../../include/fa4fp4.h"
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kTargetChunks = 8;   // pipeline depth the chunking aims for
constexpr size_t kAlign = 256;

struct DeviceResources {
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
  std::mutex mu;   // one call's enqueue at a time per device
};

DeviceResources g_res[kMaxDevices];
std::mutex g_init_mu;

// The internal streams and events of the current device, created on its
// first call and kept for the life of the process.
DeviceResources* resources() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_init_mu);
  DeviceResources& r = g_res[dev];
  if (!r.ready) {
    const unsigned ef = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&r.s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&r.s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&r.ev_start, ef) == cudaSuccess;
    for (int b = 0; ok && b < 2; ++b)
      ok = cudaEventCreateWithFlags(&r.ev_in[b], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&r.ev_comp[b], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&r.ev_out[b], ef) == cudaSuccess;
    if (!ok) return nullptr;
    r.ready = true;
  }
  return &r;
}

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Chunking: every batch element's Hkv kv heads are cut into `per_b` ranges of
// at most hc heads, so that there are about kTargetChunks chunks in all.
struct Plan {
  int hc = 0;      // kv heads per full chunk
  int per_b = 0;   // chunks per batch element
  int g = 1;       // query heads per kv head
};

Plan make_plan(int B, int Hq, int Hkv) {
  Plan p;
  p.g = Hq / Hkv;
  int want = (kTargetChunks + B - 1) / B;          // chunks per batch element
  if (want < 1) want = 1;
  if (want > Hkv) want = Hkv;
  p.hc = (Hkv + want - 1) / want;
  p.per_b = (Hkv + p.hc - 1) / p.hc;
  return p;
}

// Byte offsets of the workspace pieces for one plan (sized for a full chunk,
// O sized for f32).
struct Layout {
  size_t q, k, v, o, l;               // bytes of one buffer of each staging set
  size_t q4c, q4s, k4c, k4s, vtc, vts;
  size_t off_in[2], off_out[2], off_quant, total;
};

Layout make_layout(const Plan& p, int N, int d) {
  Layout L;
  const size_t hq = (size_t)p.hc * p.g, hk = (size_t)p.hc;
  L.q = up(hq * N * d * 2);
  L.k = up(hk * N * d * 2);
  L.v = L.k;
  L.o = up(hq * N * d * 4);
  L.l = up(hq * N * 4);
  size_t s = 0;
  L.q4c = up(fa4fp4_qtensor_bytes(1, (int)hq, N, d, 0, 0, &s)); L.q4s = up(s);
  L.k4c = up(fa4fp4_qtensor_bytes(1, (int)hk, N, d, 0, 0, &s)); L.k4s = up(s);
  L.vtc = up(fa4fp4_qtensor_bytes(1, (int)hk, N, d, 0, 1, &s)); L.vts = up(s);
  size_t off = 0;
  for (int b = 0; b < 2; ++b) { L.off_in[b] = off; off += L.q + L.k + L.v; }
  for (int b = 0; b < 2; ++b) { L.off_out[b] = off; off += L.o + L.l; }
  L.off_quant = off;
  off += L.q4c + L.q4s + L.k4c + L.k4s + L.vtc + L.vts;
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

size_t fa4fp4_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
  if (B < 0 || Hq < 0 || Hkv < 0 || N < 1 || (d != 64 && d != 128)) return 0;
  if (Hkv == 0 ? Hq != 0 : (Hq % Hkv) != 0) return 0;
  if (B == 0 || Hq == 0) return 0;
  return make_layout(make_plan(B, Hq, Hkv), N, d).total;
}

fa4fp4_status fa4fp4_fwd_host(const void* q_host, const void* k_host, const void* v_host, int B, int Hq,
                              int Hkv, int N, int d, float softmax_scale, int causal, void* o_host,
                              int out_dtype, float* lse_host, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || N < 1) return FA4FP4_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA4FP4_ERR_UNSUPPORTED;
  if (Hkv == 0 ? Hq != 0 : (Hq % Hkv) != 0) return FA4FP4_ERR_UNSUPPORTED;
  if ((long long)B * Hq * N * d > (1LL << 40)) return FA4FP4_ERR_UNSUPPORTED;
  if (out_dtype != FA4FP4_OUT_F32 && out_dtype != FA4FP4_OUT_BF16) return FA4FP4_ERR_INVALID_ARG;
  if (B == 0 || Hq == 0) return FA4FP4_OK;
  if (!q_host || !k_host || !v_host || !o_host) return FA4FP4_ERR_INVALID_ARG;
  if (!aligned16(q_host) || !aligned16(k_host) || !aligned16(v_host) || !aligned16(o_host) ||
      (lse_host && (reinterpret_cast<uintptr_t>(lse_host) & 3u)))
    return FA4FP4_ERR_ALIGNMENT;
  const Plan P = make_plan(B, Hq, Hkv);
  const Layout L = make_layout(P, N, d);
  if (!workspace || workspace_bytes < L.total) return FA4FP4_ERR_WORKSPACE;
  if (!aligned16(workspace)) return FA4FP4_ERR_ALIGNMENT;
  DeviceResources* R = resources();
  if (!R) return FA4FP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(R->mu);

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const size_t oel = out_dtype == FA4FP4_OUT_BF16 ? 2 : 4;
  char* qx = ws + L.off_quant;
  void *q4c = qx, *q4s = qx + L.q4c, *k4c = qx + L.q4c + L.q4s, *k4s = qx + L.q4c + L.q4s + L.k4c;
  void *vtc = qx + L.q4c + L.q4s + L.k4c + L.k4s, *vts = qx + L.q4c + L.q4s + L.k4c + L.k4s + L.vtc;

#define FA4_CK(x) do { if ((x) != cudaSuccess) return FA4FP4_ERR_CUDA; } while (0)
  // everything earlier on the caller's stream comes first
  FA4_CK(cudaEventRecord(R->ev_start, cs));
  FA4_CK(cudaStreamWaitEvent(R->s_in, R->ev_start, 0));
  FA4_CK(cudaStreamWaitEvent(R->s_out, R->ev_start, 0));
  int k = 0;
  for (int b = 0; b < B; ++b) {
    for (int c = 0; c < P.per_b; ++c, ++k) {
      const int h0 = c * P.hc;
      const int hk = Hkv - h0 < P.hc ? Hkv - h0 : P.hc;   // kv heads of this chunk
      const int hq = hk * P.g;
      const int buf = k & 1;
      const size_t nd = (size_t)N * d;
      const size_t qoff = ((size_t)b * Hq + (size_t)h0 * P.g) * nd;   // elements
      const size_t koff = ((size_t)b * Hkv + h0) * nd;
      char* in = ws + L.off_in[buf];
      char* qd = in;
      char* kd = in + L.q;
      char* vd = in + L.q + L.k;
      char* od = ws + L.off_out[buf];
      float* ld = reinterpret_cast<float*>(od + L.o);
      // copy in, once the compute of chunk k-2 has read this staging set
      if (k >= 2) FA4_CK(cudaStreamWaitEvent(R->s_in, R->ev_comp[buf], 0));
      FA4_CK(cudaMemcpyAsync(qd, static_cast<const char*>(q_host) + qoff * 2, (size_t)hq * nd * 2,
                             cudaMemcpyHostToDevice, R->s_in));
      FA4_CK(cudaMemcpyAsync(kd, static_cast<const char*>(k_host) + koff * 2, (size_t)hk * nd * 2,
                             cudaMemcpyHostToDevice, R->s_in));
      FA4_CK(cudaMemcpyAsync(vd, static_cast<const char*>(v_host) + koff * 2, (size_t)hk * nd * 2,
                             cudaMemcpyHostToDevice, R->s_in));
      FA4_CK(cudaEventRecord(R->ev_in[buf], R->s_in));
      // quantize and attend on the caller's stream, once the inputs are in and
      // chunk k-2's output has left this output set
      FA4_CK(cudaStreamWaitEvent(cs, R->ev_in[buf], 0));
      if (k >= 2) FA4_CK(cudaStreamWaitEvent(cs, R->ev_out[buf], 0));
      fa4fp4_status s = fa4fp4_quantize_qkv(qd, kd, vd, 1, hq, hk, N, d, q4c, q4s, k4c, k4s, vtc, vts, cs);
      if (s != FA4FP4_OK) return s;
      s = fa4fp4_fwd(q4c, q4s, k4c, k4s, vtc, vts, 1, hq, hk, N, d, softmax_scale, causal, od, out_dtype,
                     lse_host ? ld : nullptr, cs);
      if (s != FA4FP4_OK) return s;
      FA4_CK(cudaEventRecord(R->ev_comp[buf], cs));
      // copy out
      FA4_CK(cudaStreamWaitEvent(R->s_out, R->ev_comp[buf], 0));
      FA4_CK(cudaMemcpyAsync(static_cast<char*>(o_host) + qoff * oel, od, (size_t)hq * nd * oel,
                             cudaMemcpyDeviceToHost, R->s_out));
      if (lse_host)
        FA4_CK(cudaMemcpyAsync(lse_host + ((size_t)b * Hq + (size_t)h0 * P.g) * N, ld, (size_t)hq * N * 4,
                               cudaMemcpyDeviceToHost, R->s_out));
      FA4_CK(cudaEventRecord(R->ev_out[buf], R->s_out));
    }
  }
  // the call completes on the caller's stream with its last copies out
  FA4_CK(cudaStreamWaitEvent(cs, R->ev_out[(k - 1) & 1], 0));
  if (k >= 2) FA4_CK(cudaStreamWaitEvent(cs, R->ev_out[k & 1], 0));
#undef FA4_CK
  return FA4FP4_OK;
}

}  // extern "C"
