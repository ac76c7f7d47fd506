// quantize.cu -- MXFP4 / MXFP8 block quantization (OCP MX rule).
//
// "Hardware-Aware FP4 FlashAttention-4", technical summary, Methodology 1
// ("Format Selection": MXFP4, one scale that is a power of two for every 32
// consecutive elements)
// and Methodology 2 ("Gradient Formats": FP8 copies blocked along rows or
// along columns).
//
// Per block of 32 values: amax, E8M0 exponent X = E(amax) - 127 - emax
// (emax = 2 for E2M1, 8 for E4M3; clamped to [-127,127]), elements x*2^-X
// converted with round-to-nearest-even and saturation by the hardware
// converters.  The kernels are HBM-bound: 16-byte coalesced loads and one
// thread per block for blocks along d; for blocks along N one warp per
// 32-token block, each lane holding a pair of channels of every token row in
// registers (no shared-memory transpose).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "common.cuh"
#include "internal.h"

namespace fa4 {
namespace {

FA4_DEV float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
FA4_DEV float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// exponent of the block: returns X, writes 2^-X to *inv
template <int FMT>
FA4_DEV int block_exp(float amax, float* inv) {
  constexpr int emax = FMT == 0 ? 2 : 8;
  int E = (int)((__float_as_uint(amax) >> 23) & 0xff);
  int X = E - 127 - emax;
  X = X < -127 ? -127 : (X > 127 ? 127 : X);
  *inv = __uint_as_float((uint32_t)(127 - X) << 23);
  return X;
}

// blocks along d: one thread per 32-element block b, given its 64 bf16 bytes.
template <int FMT>
FA4_DEV void quant_row_block_v(const uint4 (&v)[4], long long b, uint8_t* __restrict__ codes,
                               uint8_t* __restrict__ scales) {
  if constexpr (FMT == 0) {
    uint4 o;
    scales[b] = (uint8_t)mxfp4_block32_bf16(v, o);
    reinterpret_cast<uint4*>(codes)[b] = o;
    return;
  }
  float f[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[i * 8 + 2 * j] = bf_lo(w[j]);
      f[i * 8 + 2 * j + 1] = bf_hi(w[j]);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  float inv;
  int X = block_exp<FMT>(amax, &inv);
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] *= inv;
  scales[b] = (uint8_t)(X + 127);
  if (FMT == 0) {
    uint4 o;
    o.x = pack_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
    o.y = pack_e2m1x8(f[8], f[9], f[10], f[11], f[12], f[13], f[14], f[15]);
    o.z = pack_e2m1x8(f[16], f[17], f[18], f[19], f[20], f[21], f[22], f[23]);
    o.w = pack_e2m1x8(f[24], f[25], f[26], f[27], f[28], f[29], f[30], f[31]);
    reinterpret_cast<uint4*>(codes)[b] = o;
  } else {
    uint4 o0, o1;
    o0.x = pack_e4m3x4(f[0], f[1], f[2], f[3]);
    o0.y = pack_e4m3x4(f[4], f[5], f[6], f[7]);
    o0.z = pack_e4m3x4(f[8], f[9], f[10], f[11]);
    o0.w = pack_e4m3x4(f[12], f[13], f[14], f[15]);
    o1.x = pack_e4m3x4(f[16], f[17], f[18], f[19]);
    o1.y = pack_e4m3x4(f[20], f[21], f[22], f[23]);
    o1.z = pack_e4m3x4(f[24], f[25], f[26], f[27]);
    o1.w = pack_e4m3x4(f[28], f[29], f[30], f[31]);
    reinterpret_cast<uint4*>(codes)[2 * b] = o0;
    reinterpret_cast<uint4*>(codes)[2 * b + 1] = o1;
  }
}

template <int FMT>
FA4_DEV void quant_row_block(const uint4* __restrict__ x, long long b, uint8_t* __restrict__ codes,
                             uint8_t* __restrict__ scales) {
  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __ldg(x + b * 4 + i);
  quant_row_block_v<FMT>(v, b, codes, scales);
}

template <int FMT>
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint4* __restrict__ x,
                                                          long long nblocks,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblocks;
       b += (long long)gridDim.x * blockDim.x)
    quant_row_block<FMT>(x, b, codes, scales);
}

// blocks along N, output transposed [bh][d][Np]: one warp per 32-token
// block kb of one (b,h), no shared memory.  Each lane owns a pair of
// channels per pass (two passes at d = 128): its 4-byte loads of the pair
// from the block's 32 token rows give the warp 128 contiguous bytes of every
// row, and the 32 values of each of its channels end up in its registers, so
// the block maximum, the scale and the conversion are thread-local.  Tokens
// at or past N load as zero (codes +0, scale byte 0 for an all-zero block).
template <int FMT, int D>
FA4_DEV void quant_col_block_warp(const __nv_bfloat16* __restrict__ x, long long bh, int kb, int N, int Np,
                                  uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int lane) {
  const int t0 = kb * 32;
  const int valid = min(32, N - t0);
  const uint32_t* src = reinterpret_cast<const uint32_t*>(x) + ((bh * N + t0) * (long long)D) / 2;
  constexpr int BYTES = FMT == 0 ? 16 : 32;    // code bytes per 32-token block
#pragma unroll
  for (int pass = 0; pass < D / 64; ++pass) {
    const int c0 = pass * 64 + 2 * lane;
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = i < valid ? __ldg(src + (i * D + c0) / 2) : 0u;
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      float f[32];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        f[i] = hc ? bf_hi(w[i]) : bf_lo(w[i]);
        amax = fmaxf(amax, fabsf(f[i]));
      }
      float inv;
      const int X = block_exp<FMT>(amax, &inv);
      const long long row = bh * D + c0 + hc;
      scales[row * (Np / 32) + kb] = (uint8_t)(X + 127);
      uint8_t* dst = codes + row * (long long)(Np * BYTES / 32) + kb * BYTES;
#pragma unroll
      for (int i = 0; i < 32; ++i) f[i] *= inv;
      if (FMT == 0) {
        uint4 o;
        o.x = pack_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
        o.y = pack_e2m1x8(f[8], f[9], f[10], f[11], f[12], f[13], f[14], f[15]);
        o.z = pack_e2m1x8(f[16], f[17], f[18], f[19], f[20], f[21], f[22], f[23]);
        o.w = pack_e2m1x8(f[24], f[25], f[26], f[27], f[28], f[29], f[30], f[31]);
        *reinterpret_cast<uint4*>(dst) = o;
      } else {
        uint4 o0, o1;
        o0.x = pack_e4m3x4(f[0], f[1], f[2], f[3]);
        o0.y = pack_e4m3x4(f[4], f[5], f[6], f[7]);
        o0.z = pack_e4m3x4(f[8], f[9], f[10], f[11]);
        o0.w = pack_e4m3x4(f[12], f[13], f[14], f[15]);
        o1.x = pack_e4m3x4(f[16], f[17], f[18], f[19]);
        o1.y = pack_e4m3x4(f[20], f[21], f[22], f[23]);
        o1.z = pack_e4m3x4(f[24], f[25], f[26], f[27]);
        o1.w = pack_e4m3x4(f[28], f[29], f[30], f[31]);
        reinterpret_cast<uint4*>(dst)[0] = o0;
        reinterpret_cast<uint4*>(dst)[1] = o1;
      }
    }
  }
}

// one warp per (b,h, 32-token block); nwarps = BH * Np / 32
template <int FMT, int D>
__global__ void __launch_bounds__(256) quant_cols_kernel(const __nv_bfloat16* __restrict__ x, int N, int Np,
                                                          long long nwarps, uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
  const long long wg = blockIdx.x * 8LL + threadIdx.x / 32;
  if (wg >= nwarps) return;
  const int nkb = Np / 32;
  quant_col_block_warp<FMT, D>(x, wg / nkb, (int)(wg % nkb), N, Np, codes, scales, threadIdx.x % 32);
}

// Q and K (blocks along d) and V (blocks along N) in one grid.  CTA i is a V
// CTA (eight 32-token blocks) when i is a multiple of `period` (the first nv
// of them), else a CTA of 512 row blocks of Q, then of K: the V blocks are
// spread among the row streams instead of running after them.
template <int D>
__global__ void __launch_bounds__(256) quant_qkv_kernel(const QkvParams p) {
  const long long i = blockIdx.x;
  const long long P = p.period;
  if (i % P == 0 && i / P < p.nv) {
    // a V CTA: 8 warps, each one 32-token block of one (b, kv head)
    const long long wg = (i / P) * 8 + threadIdx.x / 32;
    const int nkb = p.Np / 32;
    if (wg < p.nvw)
      quant_col_block_warp<0, D>(static_cast<const __nv_bfloat16*>(p.v), wg / nkb, (int)(wg % nkb), p.N, p.Np,
                                 p.vc, p.vs, threadIdx.x % 32);
    return;
  }
  const long long before = (i + P - 1) / P;
  const long long r = i - (before < p.nv ? before : p.nv);   // index among the row CTAs
  // a row CTA takes 512 blocks: each thread loads two blocks before converting
  // either, for more bytes in flight
  const bool isq = r < p.nq_cta;
  const uint4* x = isq ? p.q : p.k;
  const long long nb = isq ? p.nbq : p.nbk;
  const long long b0 = (isq ? r : r - p.nq_cta) * 512 + threadIdx.x, b1 = b0 + 256;
  uint4 va[4], vb[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    va[t] = b0 < nb ? __ldg(x + b0 * 4 + t) : make_uint4(0, 0, 0, 0);
    vb[t] = b1 < nb ? __ldg(x + b1 * 4 + t) : make_uint4(0, 0, 0, 0);
  }
  uint8_t* codes = isq ? p.qc : p.kc;
  uint8_t* scales = isq ? p.qs : p.ks;
  if (b0 < nb) quant_row_block_v<0>(va, b0, codes, scales);
  if (b1 < nb) quant_row_block_v<0>(vb, b1, codes, scales);
}

// ---------------------------------------------------------------- NVFP4
// E2M1 elements, one unsigned E4M3 scale per 16 consecutive elements along d,
// one FP32 scale per tensor ("Format Selection": NVFP4 for Q and K).  Every
// step is an FP32 operation rounded to nearest: ts = amax_t / 2688, block
// scale sb = E4M3(amax_b / (6 ts)), element code E2M1(x / (sb ts)); a block
// whose scale rounds to zero gets signed-zero codes.

// max |x| of the tensor into *amax_bits (non-negative floats order as their
// bit patterns); the caller zeroes it first
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const uint4* __restrict__ x, long long nvec,
                                                         unsigned* __restrict__ amax_bits) {
  float m = 0.f;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nvec;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(x + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmax3(m, fabsf(bf_lo(w[j])), fabsf(bf_hi(w[j])));
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(amax_bits, __float_as_uint(m));
}

// the tensor's amax (bits, in place) -> its scale
__global__ void nvfp4_tensor_scale_kernel(float* ts) {
  const float amax = __uint_as_float(*reinterpret_cast<unsigned*>(ts));
  *ts = amax > 0.f ? amax / 2688.0f : 1.0f;
}

FA4_DEV float e4m3_byte_value(uint32_t b) {
  uint32_t h;
  asm("{\n .reg .b16 t;\n mov.b16 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n" : "=r"(h) : "h"((unsigned short)b));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

// one thread per 16-element block
__global__ void __launch_bounds__(256) quant_nvfp4_kernel(const uint4* __restrict__ x, long long nblocks,
                                                          const float* __restrict__ tsp,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
  const float ts = *tsp;
  const float six_ts = 6.0f * ts;
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblocks;
       b += (long long)gridDim.x * blockDim.x) {
    const uint4 v0 = __ldg(x + 2 * b), v1 = __ldg(x + 2 * b + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f[2 * j] = bf_lo(w[j]);
      f[2 * j + 1] = bf_hi(w[j]);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    const float sbf = __fdiv_rn(amax, six_ts);
    const uint32_t sbc = pack_e4m3x4(sbf, 0.f, 0.f, 0.f) & 0xffu;
    scales[b] = (uint8_t)sbc;
    const float den = __fmul_rn(e4m3_byte_value(sbc), ts);
    uint2 o;
    if (den == 0.f) {
      // signed zeros
      uint32_t c[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 16; ++i) c[i / 8] |= (__float_as_uint(f[i]) >> 31) << (4 * (i % 8) + 3);
      o = make_uint2(c[0], c[1]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = __fdiv_rn(f[i], den);
      o.x = pack_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
      o.y = pack_e2m1x8(f[8], f[9], f[10], f[11], f[12], f[13], f[14], f[15]);
    }
    reinterpret_cast<uint2*>(codes)[b] = o;
  }
}

int grid_for(long long work, int per_cta) {
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long need = (work + per_cta - 1) / per_cta;
  long long cap = (long long)sms * 8;
  return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

// One CTA waits, with a bounded wait, on an mbarrier that nothing arrives at:
// the wait must expire, flag the device error word and return.
__global__ void watchdog_selftest_kernel(unsigned* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  mbar_wait_ns(&bar, 0, &abort_flag, err, limit_ns);
}

}  // namespace

cudaError_t launch_quantize_qkv(const void* q, const void* k, const void* v, long long BHq, long long BHkv,
                                int N, int d, void* qc, void* qs, void* kc, void* ks, void* vc, void* vs,
                                cudaStream_t st) {
  QkvParams p;
  p.q = (const uint4*)q;
  p.k = (const uint4*)k;
  p.v = v;
  p.qc = (uint8_t*)qc; p.qs = (uint8_t*)qs;
  p.kc = (uint8_t*)kc; p.ks = (uint8_t*)ks;
  p.vc = (uint8_t*)vc; p.vs = (uint8_t*)vs;
  p.N = N;
  p.Np = padded_n(N);
  p.nbq = BHq * N * (d / 32);
  p.nbk = BHkv * N * (d / 32);
  p.nq_cta = (p.nbq + 511) / 512;
  p.nk_cta = (p.nbk + 511) / 512;
  p.nvw = (long long)(p.Np / 32) * BHkv;     // 32-token V blocks, one warp each
  p.nv = (p.nvw + 7) / 8;                    // V CTAs of 8 warps
  const long long total = p.nv + p.nq_cta + p.nk_cta;
  p.period = total / p.nv;
  if (total > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (d == 128) quant_qkv_kernel<128><<<(unsigned)total, 256, 0, st>>>(p);
  else quant_qkv_kernel<64><<<(unsigned)total, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize_nvfp4(const void* x, long long n, void* codes, void* scales, float* ts,
                                  cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ts, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  nvfp4_amax_kernel<<<grid_for(n / 8, 256), 256, 0, st>>>((const uint4*)x, n / 8, reinterpret_cast<unsigned*>(ts));
  nvfp4_tensor_scale_kernel<<<1, 1, 0, st>>>(ts);
  const long long nblocks = n / 16;
  quant_nvfp4_kernel<<<grid_for(nblocks, 256), 256, 0, st>>>((const uint4*)x, nblocks, ts, (uint8_t*)codes,
                                                            (uint8_t*)scales);
  return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(unsigned* err, unsigned long long limit_ns, cudaStream_t st) {
  watchdog_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void* x, long long rows, int d, int N, long long BH, int fmt,
                            int axis, void* codes, void* scales, cudaStream_t st) {
  if (axis == 0) {
    long long nblocks = rows * (d / 32);
    int grid = grid_for(nblocks, 256);
    if (fmt == 0)
      quant_rows_kernel<0><<<grid, 256, 0, st>>>((const uint4*)x, nblocks, (uint8_t*)codes,
                                                 (uint8_t*)scales);
    else
      quant_rows_kernel<1><<<grid, 256, 0, st>>>((const uint4*)x, nblocks, (uint8_t*)codes,
                                                 (uint8_t*)scales);
  } else {
    const int Np = padded_n(N);
    const long long nwarps = BH * (Np / 32);
    const unsigned grid = (unsigned)((nwarps + 7) / 8);
    const __nv_bfloat16* xb = (const __nv_bfloat16*)x;
    if (d == 128) {
      if (fmt == 0) quant_cols_kernel<0, 128><<<grid, 256, 0, st>>>(xb, N, Np, nwarps, (uint8_t*)codes, (uint8_t*)scales);
      else quant_cols_kernel<1, 128><<<grid, 256, 0, st>>>(xb, N, Np, nwarps, (uint8_t*)codes, (uint8_t*)scales);
    } else {
      if (fmt == 0) quant_cols_kernel<0, 64><<<grid, 256, 0, st>>>(xb, N, Np, nwarps, (uint8_t*)codes, (uint8_t*)scales);
      else quant_cols_kernel<1, 64><<<grid, 256, 0, st>>>(xb, N, Np, nwarps, (uint8_t*)codes, (uint8_t*)scales);
    }
  }
  return cudaGetLastError();
}

}  // namespace fa4
