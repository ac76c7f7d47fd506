// fwd_bf16.cu -- BF16 FlashAttention forward for sm_103a, the reference the
// FP4 Direct-P forward is measured against ("Hardware-Aware FP4
// FlashAttention-4", technical summary, Results: speedups are quoted over a
// BF16 FlashAttention-4 baseline).
//
// Same CTA organisation as the FP4 kernel: one CTA per (batch*head,
// 128-query tile); warp 0 TMA producer, warp 1 TMEM owner + tcgen05.mma
// (kind::f16, BF16 x BF16 -> FP32) issuer, warps 2-17 softmax: thread (row r,
// column group g) owns S[r][32g, 32g+32), the row max is exchanged through
// shared memory.  Exact online softmax: P = 2^(c*s - c*m) (MUFU ex2), the
// normalizer summed from FP32 P (per-thread partial sums, combined at the
// end), P rounded to BF16 for the P V product, O rescaled in TMEM whenever the
// running max grows.
// Q, K and P are K-major with the 128-byte swizzle (64-element chunks); V is
// consumed MN-major straight from its row-major [keys][d] layout.
#include <cuda_bf16.h>
#include "common.cuh"
#include "internal.h"

namespace fa4 {
namespace {

constexpr int BM = 128, BN = 128;
constexpr int NSOFT = 16;
constexpr int NTHREADS = 32 * (2 + NSOFT);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;

template <int D>
struct SmemB {
  static constexpr int STAGES = D == 128 ? 2 : 4;
  static constexpr int CH = 128 * 128;              // one [128 rows][128 B] chunk
  static constexpr int QB = (D / 64) * CH;          // Q tile
  static constexpr int KB = (D / 64) * CH;          // K tile
  static constexpr int VB = (D / 64) * CH;          // V tile [128 keys][D]
  static constexpr int PB = 2 * CH;                 // P tile [128][128] bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB;
  static constexpr int OFF_V = OFF_K + STAGES * KB;
  static constexpr int OFF_P = OFF_V + STAGES * VB;
  static constexpr int OFF_RED = OFF_P + PB;                // float [2][4][128]
  static constexpr int OFF_BAR = OFF_RED + 2 * 4 * 128 * 4;
  static constexpr int NBAR = 1 + 4 * STAGES + 2 + 2 + 1 + 1 + 1 + 8;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int BYTES = OFF_MISC + 64 + 1024;
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) fwd_bf16_kernel(const __grid_constant__ FwdBf16Params p) {
  using L = SmemB<D>;
  constexpr int STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + STAGES;
  uint64_t* v_full = k_empty + STAGES;
  uint64_t* v_empty = v_full + STAGES;
  uint64_t* s_full = v_empty + STAGES;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* mma_done = o_done + 1;
  uint64_t* red_bar = mma_done + 1;          // [2 parities][4 quadrants]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  float* red = reinterpret_cast<float*>(smem + L::OFF_RED);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nq = (p.N + BM - 1) / BM;
  // causal: x runs over (batch, head), y over query tiles, longest first
  const int qt = p.causal ? (nq - 1 - (int)blockIdx.y) : (int)blockIdx.x;
  const int bh = p.causal ? (int)blockIdx.x : (int)blockIdx.y;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int q0 = qt * BM;
  const int nk_all = (p.N + BN - 1) / BN;
  const int nt = p.causal ? min(nk_all, qt + 1) : nk_all;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) { mbar_init(&s_full[s], 1); mbar_init(&s_free[s], NSOFT); }
    mbar_init(p_full, NSOFT);
    mbar_init(o_done, 1);
    mbar_init(mma_done, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&red_bar[i], 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(q_full, L::QB);
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + L::OFF_Q + c * L::CH, &p.tm_q, q_full, 64 * c, q0, bh);
      // K_j is released by QK_j, V_j only by P_j V_j: two rings, K loaded
      // one tile ahead of V so that a slow V slot never holds back K
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j <= nt; ++j) {
        if (j < nt) {
          const int st = j % STAGES;
          if (j >= STAGES && !mbar_wait(&k_empty[st], ((j / STAGES) - 1) & 1, abort_flag, p.err)) break;
          mbar_arrive_expect_tx(&k_full[st], L::KB);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + L::OFF_K + st * L::KB + c * L::CH, &p.tm_k, &k_full[st], 64 * c, j * BN, bkv);
          issued_k = j + 1;
        }
        if (j >= 1) {
          const int t = j - 1, st = t % STAGES;
          if (t >= STAGES && !mbar_wait(&v_empty[st], ((t / STAGES) - 1) & 1, abort_flag, p.err)) break;
          mbar_arrive_expect_tx(&v_full[st], L::VB);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + L::OFF_V + st * L::VB + c * L::CH, &p.tm_v, &v_full[st], 64 * c, t * BN, bkv);
          issued_v = t + 1;
        }
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int j = max(0, issued_k - STAGES); j < issued_k; ++j)
          mbar_wait(&k_full[j % STAGES], (j / STAGES) & 1, &no_abort, p.err);
        for (int j = max(0, issued_v - STAGES); j < issued_v; ++j)
          mbar_wait(&v_full[j % STAGES], (j / STAGES) & 1, &no_abort, p.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc_s = idesc_f16(BM, BN, true, false, false);
      const uint32_t idesc_o = idesc_f16(BM, D, true, false, true);
      const uint32_t sq = smem_u32(smem + L::OFF_Q);
      const uint32_t sp = smem_u32(smem + L::OFF_P);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.err);
      tc_fence_after();
      auto issue_pv = [&](int t) -> bool {
        const int st = t % STAGES;
        if (!mbar_wait(&v_full[st], (t / STAGES) & 1, abort_flag, p.err)) return false;
        if (!mbar_wait(p_full, t & 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t sv = smem_u32(smem + L::OFF_V + st * L::VB);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          uint64_t ad = make_sdesc(sp + (k / 4) * L::CH + (k % 4) * 32, 16, 1024, SW_128B);
          uint64_t bd = make_sdesc(sv + k * 16 * 128, L::CH, 1024, SW_128B);
          mma_f16(tbase + COL_O, ad, bd, idesc_o, t > 0 || k > 0);
        }
        mma_commit(o_done);
        mma_commit(&v_empty[st]);
        return true;
      };
      for (int j = 0; ok && j < nt; ++j) {
        const int st = j % STAGES;
        if (!mbar_wait(&k_full[st], (j / STAGES) & 1, abort_flag, p.err)) { ok = false; break; }
        const int sb = j & 1;
        if (j >= 2 && !mbar_wait(&s_free[sb], ((j >> 1) - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sk = smem_u32(smem + L::OFF_K + st * L::KB);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          uint32_t off = (k / 4) * L::CH + (k % 4) * 32;
          mma_f16(tbase + (sb ? COL_S1 : COL_S0), make_sdesc(sq + off, 16, 1024, SW_128B),
                  make_sdesc(sk + off, 16, 1024, SW_128B), idesc_s, k > 0);
        }
        mma_commit(&s_full[sb]);
        mma_commit(&k_empty[st]);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && nt > 0) issue_pv(nt - 1);
      mma_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, &no_abort, p.err);
    }
    __syncwarp();
  } else {
    const int quad = warp & 3;
    const int g = (warp - 2) >> 2;            // column group 0..3
    const int r = quad * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lane_base = tbase + ((uint32_t)(quad * 32) << 16);
    const float c = p.c;
    float m = -INFINITY, l = 0.f;             // l: this thread's partial sum
    bool ok = true;
    // P row r: keys 64*(g/2) .. in chunk g/2; this thread's 4 16-byte pieces
    uint8_t* prow = smem + L::OFF_P + (g >> 1) * L::CH + r * 128;
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      float s[32];
      {
        uint32_t v[32];
        tmem_ld32(lane_base + (sb ? COL_S1 : COL_S0) + 32 * g, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(v[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);
      const int kbase = j * BN + 32 * g;
      if (j * BN + BN > p.N || (p.causal && j * BN + BN - 1 > q0)) {
        const int lim = p.causal ? min(p.N - 1, qi) : p.N - 1;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (kbase + i > lim) s[i] = -INFINITY;
      }
      float pm = fmax3(s[0], s[1], s[2]);
#pragma unroll
      for (int i = 3; i + 1 < 32; i += 2) pm = fmax3(pm, s[i], s[i + 1]);
      pm = fmaxf(pm, s[31]);
      float* rslot = red + (sb * 4) * 128;
      rslot[g * 128 + r] = pm;
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_bar[sb * 4 + quad]);
      if (!mbar_wait(&red_bar[sb * 4 + quad], (j >> 1) & 1, abort_flag, p.err)) { ok = false; break; }
      const float tmax = fmaxf(fmaxf(rslot[r], rslot[128 + r]), fmaxf(rslot[256 + r], rslot[384 + r]));
      const float m_new = fmaxf(m, tmax);
      const float mc = m_new * c;
      uint32_t pk[16];
      float2 ls2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 x = ffma2(make_float2(s[2 * i], s[2 * i + 1]), make_float2(c, c), make_float2(-mc, -mc));
        const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        ls2 = fadd2(ls2, pp);
        __nv_bfloat162 t = __floats2bfloat162_rn(pp.x, pp.y);
        pk[i] = *reinterpret_cast<uint32_t*>(&t);
      }
      const float lsum = ls2.x + ls2.y;
      const float alpha = (m == -INFINITY) ? 1.f : ex2_approx(fmaf(m, c, -mc));
      if (j > 0) {
        if (!mbar_wait(o_done, (j - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f) && 32 * g < D) {
          uint32_t v[32];
          tmem_ld32(lane_base + COL_O + 32 * g, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float2 t = fmul2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                             make_float2(alpha, alpha));
            v[i] = __float_as_uint(t.x);
            v[i + 1] = __float_as_uint(t.y);
          }
          tmem_st32(lane_base + COL_O + 32 * g, v);
          tmem_st_wait();
        }
      }
      l = alpha * l + lsum;
      m = m_new;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int sub = (g & 1) * 4 + k;
        *reinterpret_cast<uint4*>(prow + ((sub ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // combine the four partial normalizers of each row (all used the same m)
    const int pe = nt & 1;                    // slot parity not used by the last tile
    float* lslot = red + (pe * 4) * 128;
    if (ok) {
      lslot[g * 128 + r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_bar[pe * 4 + quad]);
      ok = mbar_wait(&red_bar[pe * 4 + quad], (nt >> 1) & 1, abort_flag, p.err);
    }
    if (ok && nt > 0 && mbar_wait(o_done, (nt - 1) & 1, abort_flag, p.err)) {
      tc_fence_after();
      const float lt = (lslot[r] + lslot[128 + r]) + (lslot[256 + r] + lslot[384 + r]);
      const float inv_l = 1.f / lt;
      const bool valid = qi < p.N;
      const long long orow = ((long long)bh * p.N + qi) * D + 32 * g;
      if (32 * g < D) {
        uint32_t v[32];
        tmem_ld32(lane_base + COL_O + 32 * g, v);
        tmem_ld_wait();
        if (valid) {
          if (p.out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + orow);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(v[q * 8 + 2 * e]) * inv_l,
                                                         __uint_as_float(v[q * 8 + 2 * e + 1]) * inv_l);
                w[e] = *reinterpret_cast<uint32_t*>(&t);
              }
              dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) + orow);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(v[4 * q]) * inv_l, __uint_as_float(v[4 * q + 1]) * inv_l,
                                   __uint_as_float(v[4 * q + 2]) * inv_l, __uint_as_float(v[4 * q + 3]) * inv_l);
          }
        }
      }
      if (g == 0 && valid && p.lse) p.lse[(long long)bh * p.N + qi] = p.scale * m + logf(lt);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, TMEM_COLS);
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdBf16Params& p, cudaStream_t st) {
  const int nq = (p.N + BM - 1) / BM;
  const dim3 grid = p.causal ? dim3(p.B * p.Hq, nq) : dim3(nq, p.B * p.Hq);
  if (p.d == 128) {
    auto k = fwd_bf16_kernel<128>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemB<128>::BYTES);
    k<<<grid, NTHREADS, SmemB<128>::BYTES, st>>>(p);
  } else {
    auto k = fwd_bf16_kernel<64>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemB<64>::BYTES);
    k<<<grid, NTHREADS, SmemB<64>::BYTES, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace fa4
