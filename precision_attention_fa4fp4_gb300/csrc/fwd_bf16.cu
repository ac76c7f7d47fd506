// fwd_bf16.cu -- BF16 FlashAttention forward for sm_103a, the reference the
// FP4 Direct-P forward is measured against ("Hardware-Aware FP4
// FlashAttention-4", technical summary, Results: speedups are quoted over a
// BF16 FlashAttention-4 baseline).
//
// One CTA per (batch*head, pair of 128-query tiles A and B), 12 warps in
// three warpgroups (setmaxnreg gives the two softmax warpgroups most of the
// registers):
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: one thread per
//               query row (TMEM lane quadrant = warp mod 4).  Exact online
//               softmax: row max, P = 2^(c*s - c*m) (MUFU ex2), the normalizer
//               summed from FP32 P, P rounded to bf16 into tensor memory, O
//               rescaled in TMEM whenever the running max grows.
//   warp 8      producer: TMA loads of Q_A, Q_B once, then K_j and V_j (two
//               rings) shared by both tiles.
//   warp 9      TMEM allocation; one elected lane issues tcgen05.mma kind::f16
//               (BF16 x BF16 -> FP32): S_X = Q_X K_j^T into the tile's own S
//               buffer, and O_X += P_X V_j with P_X read from tensor memory
//               (the softmax warps write it as bf16 over the first half of
//               S_X), V_j MN-major straight from its row-major [keys][d] tile.
//   warps 10-11 idle.
// TMEM: S_A, S_B, O_A, O_B (512 columns at d = 128).  The next QK^T of a tile
// is issued after its P V, so the in-order tensor pipe has read P_X before it
// overwrites S_X; while one tile's warps work on their scores the tensor core
// runs the other tile's products.
#include <cuda_bf16.h>
#include "common.cuh"
#include "internal.h"

namespace fa4 {
namespace {

constexpr int BM = 128, BN = 128;
constexpr int NTHREADS = 384;
constexpr int W_PROD = 8, W_MMA = 9;
// registers per thread after setmaxnreg (3 warpgroups x 128 threads share the
// CTA's 65536): 2 x 208 + 88 = 504 of 512
constexpr int REG_SOFT = 208, REG_MISC = 88;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S0 = 0;             // S_X at 128 X, O_X at 256 + d X

template <int D>
struct SmemB {
  static constexpr int STAGES = D == 128 ? 2 : 4;   // K and V ring depth
  static constexpr int CH = 128 * 128;              // one [128 rows][128 B] chunk (64 bf16)
  static constexpr int QB = (D / 64) * CH;          // a Q tile
  static constexpr int KB = (D / 64) * CH;          // a K tile
  static constexpr int VB = (D / 64) * CH;          // a V tile [128 keys][D]
  static constexpr int OFF_Q = 0;                   // Q_A, Q_B
  static constexpr int OFF_K = OFF_Q + 2 * QB;
  static constexpr int OFF_V = OFF_K + STAGES * KB;
  static constexpr int OFF_BAR = OFF_V + STAGES * VB;
  static constexpr int NBAR = 1 + 4 * STAGES + 2 + 2 + 2 + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int BYTES = OFF_MISC + 64 + 1024;
  static constexpr uint32_t COL_O0 = 256;
  static_assert(COL_O0 + 2 * D <= TMEM_COLS, "TMEM budget");
  static_assert(BYTES <= 227 * 1024, "shared memory budget");
};

// Maximum of 128 values by a tree of fmax3 (short dependency chains).
FA4_DEV float rowmax128(const float (&s)[4][32]) {
  float a[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) a[i] = fmax3(s[0][i], s[1][i], fmaxf(s[2][i], s[3][i]));
#pragma unroll
  for (int n = 32; n > 1; n /= 2)
#pragma unroll
    for (int i = 0; i < n / 2; ++i) a[i] = fmaxf(a[i], a[i + n / 2]);
  return a[0];
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) fwd_bf16_kernel(const __grid_constant__ FwdBf16Params p) {
  using L = SmemB<D>;
  constexpr int STAGES = L::STAGES;
  constexpr uint32_t COL_O0 = L::COL_O0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + STAGES;
  uint64_t* v_full = k_empty + STAGES;
  uint64_t* v_empty = v_full + STAGES;
  uint64_t* s_full = v_empty + STAGES;       // [X]: S_X holds Q_X K_j^T
  uint64_t* p_full = s_full + 2;             // [X]: P_X in TMEM, O_X rescaled
  uint64_t* o_done = p_full + 2;             // [X]: P_X V of the last tile done
  uint64_t* mma_done = o_done + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nq = (p.N + BM - 1) / BM;
  const int npair = (nq + 1) / 2;
  // causal: x runs over (batch, head), y over query-tile pairs, longest first
  const int pair = p.causal ? (npair - 1 - (int)blockIdx.y) : (int)blockIdx.x;
  const int bh = p.causal ? (int)blockIdx.x : (int)blockIdx.y;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int q0 = pair * 2 * BM;              // first row of tile A; tile B follows
  const int nk_all = (p.N + BN - 1) / BN;
  // key tiles of the pair (tile A takes the last one fully masked when
  // causal: its P is 0 there, adding exact zeros to O_A and l_A)
  const int nt = p.causal ? min(nk_all, 2 * pair + 2) : nk_all;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 4);
      mbar_init(&o_done[x], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == W_MMA) tmem_alloc(tmem_holder, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  // Roles by warpgroup; each sets its register budget first, inside its own
  // branch so the compiler allocates each role's code within that budget.
  if (warp >= W_PROD) {
    setmaxnreg_dec<REG_MISC>();
  if (warp == W_PROD) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(q_full, 2 * L::QB);
      for (int x = 0; x < 2; ++x)
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::OFF_Q + x * L::QB + c * L::CH, &p.tm_q, q_full, 64 * c, q0 + x * BM, bh);
      // K_j is released by the two QK_j, V_j only by the two P_j V_j: two
      // rings, K loaded one tile ahead of V so a slow V slot never holds K
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
        mbar_wait(q_full, 0, &no_abort, p.err);
        for (int j = max(0, issued_k - STAGES); j < issued_k; ++j)
          mbar_wait(&k_full[j % STAGES], (j / STAGES) & 1, &no_abort, p.err);
        for (int j = max(0, issued_v - STAGES); j < issued_v; ++j)
          mbar_wait(&v_full[j % STAGES], (j / STAGES) & 1, &no_abort, p.err);
      }
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule in uniform control flow; one elected
    // lane issues each tcgen05 instruction.
    const bool leader = elect_one();
    const uint32_t idesc_s = idesc_f16(BM, BN, true, false, false);
    const uint32_t idesc_o = idesc_f16(BM, D, true, false, true);   // A from TMEM, V MN-major
    const uint32_t sq = smem_u32(smem + L::OFF_Q);
    bool ok = mbar_wait(q_full, 0, abort_flag, p.err);
    tc_fence_after();
    // S_X = Q_X K_t^T
    auto issue_qk = [&](int x, int t) -> bool {
      const int st = t % STAGES;
      if (x == 0 && !mbar_wait(&k_full[st], (t / STAGES) & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      const uint32_t sqx = sq + x * L::QB;
      const uint32_t sk = smem_u32(smem + L::OFF_K + st * L::KB);
      if (leader) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * L::CH + (k % 4) * 32;
          mma_f16(tbase + COL_S0 + 128 * x, make_sdesc(sqx + off, 16, 1024, SW_128B),
                  make_sdesc(sk + off, 16, 1024, SW_128B), idesc_s, k > 0);
        }
        mma_commit(&s_full[x]);
        if (x == 1) mma_commit(&k_empty[st]);
      }
      __syncwarp();
      return true;
    };
    // O_X += P_X V_t (P_X: bf16 pairs in the first 64 columns of S_X)
    auto issue_pv = [&](int x, int t) -> bool {
      const int st = t % STAGES;
      if (x == 0 && !mbar_wait(&v_full[st], (t / STAGES) & 1, abort_flag, p.err)) return false;
      if (!mbar_wait(&p_full[x], t & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      const uint32_t sv = smem_u32(smem + L::OFF_V + st * L::VB);
      if (leader) {
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_f16_tmem_a(tbase + COL_O0 + D * x, tbase + COL_S0 + 128 * x + 8 * k,
                         make_sdesc(sv + k * 16 * 128, L::CH, 1024, SW_128B), idesc_o, t > 0 || k > 0);
        mma_commit(&o_done[x]);
        if (x == 1) mma_commit(&v_empty[st]);
      }
      __syncwarp();
      return true;
    };
    // Each tile's next QK^T follows its own P V, so the pipe reads P_X
    // before it overwrites S_X.
    if (ok && nt > 0) ok = issue_qk(0, 0) && issue_qk(1, 0);
    for (int j = 0; ok && j < nt; ++j) {
      if (!issue_pv(0, j)) { ok = false; break; }
      if (j + 1 < nt && !issue_qk(0, j + 1)) { ok = false; break; }
      if (!issue_pv(1, j)) { ok = false; break; }
      if (j + 1 < nt && !issue_qk(1, j + 1)) { ok = false; break; }
    }
    if (leader) mma_commit(mma_done);
    __syncwarp();
    volatile int no_abort = 0;
    mbar_wait(mma_done, 0, &no_abort, p.err);
    __syncwarp();
  }
  } else {
    setmaxnreg_inc<REG_SOFT>();
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;                  // query tile 0 (A) or 1 (B)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;           // row within the tile
    const int qi = q0 + x * BM + r;
    const uint32_t lane_base = tbase + ((uint32_t)(quad * 32) << 16);
    const uint32_t col_s = COL_S0 + 128 * x, col_o = COL_O0 + D * x;
    const float c = p.c;
    const int lim = p.causal ? min(p.N - 1, qi) : p.N - 1;   // last key of the row
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      if (!mbar_wait(&s_full[x], j & 1, abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      float s[4][32];
      {
        uint32_t v[4][32];
#pragma unroll
        for (int g = 0; g < 4; ++g) tmem_ld32(lane_base + col_s + 32 * g, v[g]);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          reg_fence32(v[g]);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[g][i] = __uint_as_float(v[g][i]);
        }
      }
      if (j * BN + BN - 1 > lim) {
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (j * BN + 32 * g + i > lim) s[g][i] = -INFINITY;
      }
      const float m_new = fmaxf(m, rowmax128(s));
      const float mc = m_new * c;
      // P = 2^(c s - c m), the normalizer from FP32 P, P to bf16 over S_X
      float2 ls = make_float2(0.f, 0.f);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 xx = ffma2(make_float2(s[g][2 * i], s[g][2 * i + 1]), make_float2(c, c), make_float2(-mc, -mc));
          const float2 pp = make_float2(ex2_approx(xx.x), ex2_approx(xx.y));
          ls = fadd2(ls, pp);
          __nv_bfloat162 t = __floats2bfloat162_rn(pp.x, pp.y);   // key 2i in the low half
          pk[i] = *reinterpret_cast<uint32_t*>(&t);
        }
        tmem_st16(lane_base + col_s + 16 * g, pk);
      }
      const float alpha = (j == 0 || m_new == m) ? 1.f : ex2_approx(fmaf(m, c, -mc));
      if (j > 0) {
        // rescale O_X to the new max once P_X V of tile j-1 is in
        if (!mbar_wait(&o_done[x], (j - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          uint32_t ov[D / 32][32];
#pragma unroll
          for (int g = 0; g < D / 32; ++g) tmem_ld32(lane_base + col_o + 32 * g, ov[g]);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < D / 32; ++g) {
            reg_fence32(ov[g]);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 t = fmul2(make_float2(__uint_as_float(ov[g][i]), __uint_as_float(ov[g][i + 1])),
                                     make_float2(alpha, alpha));
              ov[g][i] = __float_as_uint(t.x);
              ov[g][i + 1] = __float_as_uint(t.y);
            }
            tmem_st32(lane_base + col_o + 32 * g, ov[g]);
          }
        }
      }
      l = alpha * l + (ls.x + ls.y);
      m = m_new;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x]);
    }
    if (ok && nt > 0 && mbar_wait(&o_done[x], (nt - 1) & 1, abort_flag, p.err)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool valid = qi < p.N;
      const long long orow = ((long long)bh * p.N + qi) * D;
#pragma unroll 1
      for (int g = 0; g < D / 32; ++g) {
        uint32_t v[32];
        tmem_ld32(lane_base + col_o + 32 * g, v);
        tmem_ld_wait();
        reg_fence32(v);
        if (valid && p.out_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + orow + 32 * g);
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
        } else if (valid) {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) + orow + 32 * g);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]) * inv_l, __uint_as_float(v[4 * q + 1]) * inv_l,
                                 __uint_as_float(v[4 * q + 2]) * inv_l, __uint_as_float(v[4 * q + 3]) * inv_l);
        }
      }
      if (valid && p.lse) p.lse[(long long)bh * p.N + qi] = p.scale * m + logf(l);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) tmem_dealloc(tbase, TMEM_COLS);
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdBf16Params& p, cudaStream_t st) {
  const int nq = (p.N + BM - 1) / BM;
  const int npair = (nq + 1) / 2;
  const dim3 grid = p.causal ? dim3(p.B * p.Hq, npair) : dim3(npair, p.B * p.Hq);
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
