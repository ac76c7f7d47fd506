// host_pipeline.cu -- the end-to-end inference call on host buffers:
// fa4fp4_fwd_host copies bf16 Q, K, V in from host memory, quantizes them to
// MXFP4, runs the Direct-P forward and copies O (and LSE) back out, all in
// one call.  The work is cut into chunks of consecutive (batch, kv head)
// units with their query heads (contiguous in every tensor); chunk k's inputs
// are copied in on one internal stream while earlier chunks are quantized and
// attended, alternately on the caller's stream and a second internal stream,
// and copied out on a third, so the host link and the GPU stay busy together.
// The last chunk holds one unit, so that the work left after the last copy
// in is short.  Staging buffers (two sets) live in a workspace the caller
// allocates; events order every reuse.
#include <mutex>
#include "../../include/fa4fp4.h"
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kTargetChunks = 8;   // pipeline depth the chunking aims for
constexpr size_t kAlign = 256;

struct DeviceResources {
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr, s_c = nullptr;
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
              cudaStreamCreateWithFlags(&r.s_c, cudaStreamNonBlocking) == cudaSuccess &&
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

// Chunking over the U = B * Hkv (batch, kv head) units in order: chunks of
// hc units (about kTargetChunks of them, at most kMaxChunkBytes of bf16
// inputs unless one unit is larger), the last one cut so that the final
// chunk is a single unit.
constexpr size_t kMaxChunkBytes = (size_t)64 << 20;

struct Plan {
  int hc = 0;      // units per full chunk
  int g = 1;       // query heads per kv head
  long long U = 0;
};

Plan make_plan(int B, int Hq, int Hkv, int N, int d) {
  Plan p;
  p.g = Hq / Hkv;
  p.U = (long long)B * Hkv;
  long long hc = (p.U + kTargetChunks - 1) / kTargetChunks;
  const long long cap = (long long)(kMaxChunkBytes / ((size_t)(p.g + 2) * N * d * 2));
  if (hc > cap) hc = cap;
  p.hc = (int)(hc < 1 ? 1 : hc);
  return p;
}

// units of chunk starting at unit u0
int chunk_units(const Plan& p, long long u0) {
  long long n = p.U - u0 < p.hc ? p.U - u0 : p.hc;
  if (n > 1 && u0 + n == p.U) n -= 1;    // split the final unit off
  return (int)n;
}

// Byte offsets of the workspace pieces for one plan (sized for a full chunk,
// O sized for f32).
struct Layout {
  size_t q, k, v, o, l;               // bytes of one buffer of each staging set
  size_t q4c, q4s, k4c, k4s, vtc, vts;
  size_t off_in[2], off_out[2], off_quant[2], total;
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
  for (int b = 0; b < 2; ++b) { L.off_quant[b] = off; off += L.q4c + L.q4s + L.k4c + L.k4s + L.vtc + L.vts; }
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
  return make_layout(make_plan(B, Hq, Hkv, N, d), N, d).total;
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
  const Plan P = make_plan(B, Hq, Hkv, N, d);
  const Layout L = make_layout(P, N, d);
  if (!workspace || workspace_bytes < L.total) return FA4FP4_ERR_WORKSPACE;
  if (!aligned16(workspace)) return FA4FP4_ERR_ALIGNMENT;
  DeviceResources* R = resources();
  if (!R) return FA4FP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(R->mu);

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const size_t oel = out_dtype == FA4FP4_OUT_BF16 ? 2 : 4;

#define FA4_CK(x) do { if ((x) != cudaSuccess) return FA4FP4_ERR_CUDA; } while (0)
  // everything earlier on the caller's stream comes first
  FA4_CK(cudaEventRecord(R->ev_start, cs));
  FA4_CK(cudaStreamWaitEvent(R->s_in, R->ev_start, 0));
  FA4_CK(cudaStreamWaitEvent(R->s_out, R->ev_start, 0));
  FA4_CK(cudaStreamWaitEvent(R->s_c, R->ev_start, 0));
  const size_t nd = (size_t)N * d;
  int k = 0;
  for (long long u0 = 0; u0 < P.U; ++k) {
    const int nu = chunk_units(P, u0);     // kv heads (units) of this chunk
    const int hq = nu * P.g;
    const int buf = k & 1;
    cudaStream_t sc = buf ? R->s_c : cs;   // chunks alternate between two compute streams
    const size_t qoff = (size_t)u0 * P.g * nd;   // elements
    const size_t koff = (size_t)u0 * nd;
    char* in = ws + L.off_in[buf];
    char* qd = in;
    char* kd = in + L.q;
    char* vd = in + L.q + L.k;
    char* od = ws + L.off_out[buf];
    float* ld = reinterpret_cast<float*>(od + L.o);
    char* qx = ws + L.off_quant[buf];
    void *q4c = qx, *q4s = qx + L.q4c, *k4c = qx + L.q4c + L.q4s, *k4s = qx + L.q4c + L.q4s + L.k4c;
    void *vtc = qx + L.q4c + L.q4s + L.k4c + L.k4s, *vts = qx + L.q4c + L.q4s + L.k4c + L.k4s + L.vtc;
    // copy in, once the compute of chunk k-2 has read this staging set
    if (k >= 2) FA4_CK(cudaStreamWaitEvent(R->s_in, R->ev_comp[buf], 0));
    FA4_CK(cudaMemcpyAsync(qd, static_cast<const char*>(q_host) + qoff * 2, (size_t)hq * nd * 2,
                           cudaMemcpyHostToDevice, R->s_in));
    FA4_CK(cudaMemcpyAsync(kd, static_cast<const char*>(k_host) + koff * 2, (size_t)nu * nd * 2,
                           cudaMemcpyHostToDevice, R->s_in));
    FA4_CK(cudaMemcpyAsync(vd, static_cast<const char*>(v_host) + koff * 2, (size_t)nu * nd * 2,
                           cudaMemcpyHostToDevice, R->s_in));
    FA4_CK(cudaEventRecord(R->ev_in[buf], R->s_in));
    // quantize and attend once the inputs are in and chunk k-2's output has
    // left this output set (chunk k-2 ran on the same compute stream, so its
    // MXFP4 set is free)
    FA4_CK(cudaStreamWaitEvent(sc, R->ev_in[buf], 0));
    if (k >= 2) FA4_CK(cudaStreamWaitEvent(sc, R->ev_out[buf], 0));
    fa4fp4_status s = fa4fp4_quantize_qkv(qd, kd, vd, 1, hq, nu, N, d, q4c, q4s, k4c, k4s, vtc, vts, sc);
    if (s != FA4FP4_OK) return s;
    s = fa4fp4_fwd(q4c, q4s, k4c, k4s, vtc, vts, 1, hq, nu, N, d, softmax_scale, causal, od, out_dtype,
                   lse_host ? ld : nullptr, sc);
    if (s != FA4FP4_OK) return s;
    FA4_CK(cudaEventRecord(R->ev_comp[buf], sc));
    // copy out
    FA4_CK(cudaStreamWaitEvent(R->s_out, R->ev_comp[buf], 0));
    FA4_CK(cudaMemcpyAsync(static_cast<char*>(o_host) + qoff * oel, od, (size_t)hq * nd * oel,
                           cudaMemcpyDeviceToHost, R->s_out));
    if (lse_host)
      FA4_CK(cudaMemcpyAsync(lse_host + (size_t)u0 * P.g * N, ld, (size_t)hq * N * 4, cudaMemcpyDeviceToHost,
                             R->s_out));
    FA4_CK(cudaEventRecord(R->ev_out[buf], R->s_out));
    u0 += nu;
  }
  // the call completes on the caller's stream with its last copies out
  FA4_CK(cudaStreamWaitEvent(cs, R->ev_out[(k - 1) & 1], 0));
  if (k >= 2) FA4_CK(cudaStreamWaitEvent(cs, R->ev_out[k & 1], 0));
#undef FA4_CK
  return FA4FP4_OK;
}

}  // extern "C"
