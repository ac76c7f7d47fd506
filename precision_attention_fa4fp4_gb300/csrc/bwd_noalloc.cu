// bwd_noalloc.cu -- fa4fp4_bwd for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: plugins whose host framework owns every
// device allocation, runtimes that forbid allocation after start-up, or code
// whose device memory is budgeted once up front.  For them this file provides
// fa4fp4_bwd_noalloc, which runs the same backward as
// fa4fp4_bwd but takes its scratch (the MXFP8 views of dO and the per-row
// initial values of S^T and dP^T)
// from a fixed array in device memory instead of a caller workspace.
//
// The array is a file-scope __device__ variable of FA4FP4_BWD_NOALLOC_SCRATCH_BYTES
// bytes: every GPU that loads this library holds it until the process exits.
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, once per device, with that
// device current, on the first call made on that device.
// Every call shares the array and leaves the last call's contents in it; the
// backward rewrites all of it before reading it, so nothing has to be cleared,
// but two calls that overlap on the GPU (different streams, or different host
// threads) race on it.
#include <mutex>
#include "../../include/fa4fp4.h"

namespace {

constexpr size_t kScratchBytes = FA4FP4_BWD_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (looked up once).
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" fa4fp4_status fa4fp4_bwd_noalloc(
    const void* q4_codes, const void* q4_scales, const void* k4_codes, const void* k4_scales,
    const void* q8c_codes, const void* q8c_scales, const void* k8c_codes, const void* k8c_scales,
    const void* v8r_codes, const void* v8r_scales, const void* o, int o_dtype, const void* dout,
    const float* lse, int B, int Hq, int Hkv, int N, int d, float softmax_scale, int causal,
    float* dq, float* dk, float* dv, void* stream) {
  // The arguments are checked first, by fa4fp4_bwd itself: given no
  // workspace it validates every argument, launches nothing, and returns
  // FA4FP4_ERR_WORKSPACE for a well-formed non-empty problem.  So a bad
  // argument gets the same status from both entry points, and the scratch
  // address is looked up only for a call that will run.
  const fa4fp4_status s =
      fa4fp4_bwd(q4_codes, q4_scales, k4_codes, k4_scales, q8c_codes, q8c_scales, k8c_codes, k8c_scales,
                 v8r_codes, v8r_scales, o, o_dtype, dout, lse, B, Hq, Hkv, N, d, softmax_scale, causal, dq,
                 dk, dv, nullptr, 0, stream);
  if (s != FA4FP4_ERR_WORKSPACE) return s;   // an argument error, or an empty problem (OK)
  if (fa4fp4_bwd_workspace_bytes(B, Hq, Hkv, N, d) > kScratchBytes) return FA4FP4_ERR_WORKSPACE;
  void* scratch = scratch_address();
  if (!scratch) return FA4FP4_ERR_CUDA;
  return fa4fp4_bwd(q4_codes, q4_scales, k4_codes, k4_scales, q8c_codes, q8c_scales, k8c_codes,
                    k8c_scales, v8r_codes, v8r_scales, o, o_dtype, dout, lse, B, Hq, Hkv, N, d,
                    softmax_scale, causal, dq, dk, dv, scratch, kScratchBytes, stream);
}
