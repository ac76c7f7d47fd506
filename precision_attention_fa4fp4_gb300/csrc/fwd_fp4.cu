// fwd_fp4.cu -- Direct-P FP4 attention forward for sm_103a.
//
// "Hardware-Aware FP4 FlashAttention-4" (arXiv:2609.04105), technical
// summary, Methodology 1: S = Q K^T on FP4 tensor cores; each score's offset
// from the running row max classified straight into an E2M1 probability code
// (Direct Mapping: a classifier, with hardware exponentials allowed for part
// of the work); the normalizer accumulated from the same codes the P V
// product consumes (Consistent Normalization); MXFP4 for P and V (Format
// Selection).  Q and K are MXFP4 as well.
//
// One CTA per (batch*head, pair of 128-query tiles A and B), 10 warps:
//   warp 0      producer: TMA loads of Q_A, Q_B, K_j, V^T_j codes into swizzled
//               shared memory; their E8M0 scales rearranged into the 32x16-byte
//               chunks the scale-factor TMEM copy expects.  K_j and V_j are
//               loaded once for both query tiles.
//   warp 1      TMEM allocation; one elected lane issues tcgen05.cp (scale
//               factors) and tcgen05.mma kind::mxf4 block_scale: S = Q_X K_j^T
//               into one S buffer that the two query tiles take in turn, and
//               [O_X | l_X] += P_X [V_j | 1]: the V^T operand carries 16 extra
//               rows of E2M1 ones under unit scales, so the same MMA (N = d +
//               16) sums the normalizer from exactly the codes P V consumes.
//   warps 2-5   softmax of tile A, warps 6-9 softmax of tile B: one thread per
//               query row (TMEM lane quadrant = warp mod 4), holding the row's
//               128 scores of the key tile.  Row max, Direct-P codes (native
//               exponentials bracketed to the exact threshold map, threshold
//               count where the bracket is ambiguous), the row's 64-byte P
//               chunk, eager rescale of the row of O_X and l_X.
// While one tile's warps build codes, the other tile's S is computed and its
// P V runs, so the latency of each hand-off hides behind the other tile's work.
#include <cuda_bf16.h>
#include "common.cuh"
#include "internal.h"

namespace fa4 {
namespace {

constexpr int BM = 128;         // queries per tile; a CTA holds two tiles
constexpr int BN = 128;         // keys per tile
constexpr int NSOFT = 8;        // softmax warps: 4 per query tile
constexpr int NTHREADS = 32 * (2 + NSOFT);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O0 = 128;   // [O_X | l_X] at 128 + (d + 16) X

// Shared-memory and TMEM layout of one CTA.  P8: the FP8 P/V route (E4M3 P
// and V^T, one E8M0 scale per 32 keys), else Direct-P (E2M1 P and V^T).
// NV: NVFP4 Q and K (one UE4M3 scale per 16 along d: d/64 scale chunks per
// tile, one per K=64 MMA step), else MXFP4 (one E8M0 scale per 32: one chunk).
template <int D, bool P8, bool NV>
struct Layout {
  static constexpr int QSB = NV ? D / 16 : D / 32;   // scale bytes per Q/K row
  static constexpr int NSC = NV ? D / 64 : 1;        // scale chunks per Q/K tile
  static constexpr int STAGES = P8 ? 4 : ((NV && D == 128) ? 4 : 6);   // K/V pipeline depth
  static constexpr int NO = D + 16;           // columns of [O_X | l_X]: d of O, 16 copies of l
  static constexpr int QB = BM * D / 2;       // bytes of a Q or K code tile
  static constexpr int KB = BN * D / 2;
  static constexpr int PROW = P8 ? BN : BN / 2;   // bytes of a P (or V^T) row of 128 keys
  static constexpr int VD = D * PROW;         // V^T: d channel rows of 128 keys (the TMA box)
  static constexpr int VB = NO * PROW;        // a V stage: the d rows, then 16 rows of ones
  static constexpr int PB = BM * PROW;
  static constexpr int OFF_Q = 0;                          // Q_A, Q_B
  static constexpr int OFF_K = OFF_Q + 2 * QB;
  static constexpr int OFF_V = OFF_K + STAGES * KB;
  static constexpr int OFF_P = OFF_V + STAGES * VB;        // [tile X][2 buffers]
  static constexpr int OFF_SF = OFF_P + 4 * PB;           // 512-byte scale chunks
  static constexpr int SF_Q = OFF_SF;                     // [X][NSC]
  static constexpr int SF_1 = SF_Q + 2 * NSC * 512;       // unit scales (ones rows of V^T; Direct-P P)
  static constexpr int SF_P = SF_1 + 512;                 // P8: [X][step parity]
  static constexpr int SF_K = SF_P + (P8 ? 4 * 512 : 0);  // [stage][NSC]
  static constexpr int SF_V = SF_K + 512 * NSC * STAGES;
  static constexpr int OFF_BAR = SF_V + 512 * STAGES;
  static constexpr int NBAR = 1 + 4 * STAGES + 2 + 2 + 2 + 2 + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int BYTES = OFF_MISC + 64 + 1024;    // + alignment slack
  // TMEM scale-factor columns (4 per chunk): Q_X, unit, P_X (P8), K and V
  // rings.  A V stage's scales cover its d + 16 rows (row r in column r/32):
  // at d = 64 the ones rows 64..79 fall in the chunk's third column, at
  // d = 128 rows 128..143 need a fifth column, so the stage takes 8 columns,
  // the upper four holding unit scales.
  static constexpr uint32_t SFVS = D == 128 ? 8 : 4;
  static constexpr uint32_t COL_SFQ0 = 416, COL_SF1 = COL_SFQ0 + 8 * NSC, COL_SFP0 = COL_SF1 + 4,
                            COL_SFK = COL_SFP0 + (P8 ? 8 : 0), COL_SFV = COL_SFK + 4 * NSC * STAGES;
  static_assert(COL_O0 + 2 * NO <= COL_SFQ0, "TMEM budget: S, O_A, O_B");
  static_assert(COL_SFV + SFVS * STAGES <= TMEM_COLS, "TMEM budget");
  static_assert(BYTES <= 227 * 1024, "shared memory budget");
};

// Direct-P code of one scaled offset x: #{k : x >= T_k}.
FA4_DEV uint32_t directp_code(float x, const float (&T)[7]) {
  uint32_t c = 0;
#pragma unroll
  for (int k = 0; k < 7; ++k) c += (x >= T[k]) ? 1u : 0u;
  return c;
}

// Codes of 32 consecutive scores, packed 8 per word (element e of word w in
// nibble e).  Native-exponential route made exact.  The method's offset is
// x = fmaf(s, c, -mc); the lane instead forms x' = fmaf(s, c, klo) with
// klo = (log2 6 - eps) - mc, so ylo = ex2(x') is 6 2^x 2^-eps up to the
// rounding of klo and x' and the error of ex2, and yhi = ylo R.  With
// eps = 2^-19 + 2u and R = 1 + 2^-18 + 3u (u = ulp(mc)), ylo < 6 2^x < yhi:
// where 6 2^x is near an E2M1 midpoint (|x| < 8) those roundings move x' by
// at most 2^-20 + u, and ex2 is within 2^-22 relative.  Rounding to E2M1 is
// monotone, so where the codes of ylo and yhi agree that code is the exact
// one; the lanes where they do not (scores within about 2^-18 of a midpoint)
// redo their scores with the threshold count.  Folding the factor 6 and the
// lower bracket into x' leaves one product per score (yhi).  Returns the
// packed codes in pw.
constexpr float LOG2_6 = 0x1.4ae00ep+1f;   // fl32(log2 6), within 2^-23.2 of it

FA4_DEV void directp_codes32(const float (&s)[32], float c, float mc, const float (&T)[7],
                             uint32_t (&pw)[4]) {
  const float u = __uint_as_float(__float_as_uint(mc) & 0x7f800000u) * 0x1p-23f;   // ulp(mc), normal mc
  const float klo = (LOG2_6 - fmaf(2.f, u, 0x1p-19f)) - mc;
  const float R = 1.f + fmaf(3.f, u, 0x1p-18f);
  bool ambiguous = false;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float ylo[8], yhi[8];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float2 x = ffma2(make_float2(s[8 * w + e], s[8 * w + e + 1]), make_float2(c, c),
                             make_float2(klo, klo));
      const float2 a = make_float2(ex2_approx(x.x), ex2_approx(x.y));
      const float2 b = fmul2(a, make_float2(R, R));
      ylo[e] = a.x; ylo[e + 1] = a.y;
      yhi[e] = b.x; yhi[e + 1] = b.y;
    }
    const uint32_t lo = pack_e2m1x8(ylo[0], ylo[1], ylo[2], ylo[3], ylo[4], ylo[5], ylo[6], ylo[7]);
    const uint32_t hi = pack_e2m1x8(yhi[0], yhi[1], yhi[2], yhi[3], yhi[4], yhi[5], yhi[6], yhi[7]);
    pw[w] = lo;
    ambiguous |= lo != hi;
  }
  if (__any_sync(0xffffffffu, ambiguous) && ambiguous) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) word |= directp_code(fmaf(s[8 * w + e], c, -mc), T) << (4 * e);
      pw[w] = word;
    }
  }
}

// Maximum of 128 values by a tree of fmax3 (short dependency chains).
FA4_DEV float max128(const float (&s)[4][32]) {
  float a[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) a[i] = fmax3(s[0][i], s[1][i], fmaxf(s[2][i], s[3][i]));
#pragma unroll
  for (int n = 32; n > 1; n /= 2)
#pragma unroll
    for (int i = 0; i < n / 2; ++i) a[i] = fmaxf(a[i], a[i + n / 2]);
  return a[0];
}

// Rearrange 128 rows of per-row scale words into the scale-factor chunk:
// chunk byte (r%32)*16 + (r/32)*4 + kblock.  The word of row r is the 4 (or,
// for 2-byte rows, 2) scale bytes at byte `off` of the row.  Called by a full
// warp.
FA4_DEV void stage_sf_rows(uint8_t* chunk, const uint8_t* src, int row0, int nrows_valid,
                           int bytes_per_row, int lane, int off = 0) {
  uint32_t w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    int r = lane + 32 * c;
    uint32_t v = 0;
    if (r < nrows_valid) {
      const uint8_t* p = src + (long long)(row0 + r) * bytes_per_row + off;
      v = bytes_per_row >= 4 ? *reinterpret_cast<const uint32_t*>(p)
                             : (uint32_t)*reinterpret_cast<const uint16_t*>(p);
    }
    w[c] = v;
  }
  *reinterpret_cast<uint4*>(chunk + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

// QBF: Q arrives as bf16 and the softmax warps quantize it to MXFP4 in the
// kernel's prologue (one thread per query row, straight into the swizzled Q
// tiles and their scale chunks), so an inference step needs no separate pass
// over Q; K and V^T arrive quantized.
template <int D, bool P8, bool NV, bool QBF>
__global__ void __launch_bounds__(NTHREADS, 1) fwd_fp4_kernel(const __grid_constant__ FwdFp4Params p) {
  using L = Layout<D, P8, NV>;
  constexpr int NSC = L::NSC, QSB = L::QSB;
  constexpr int STAGES = L::STAGES;
  constexpr uint32_t COL_SFQ0 = L::COL_SFQ0, COL_SF1 = L::COL_SF1, COL_SFP0 = L::COL_SFP0,
                     COL_SFK = L::COL_SFK, COL_SFV = L::COL_SFV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + STAGES;
  uint64_t* v_full = k_empty + STAGES;
  uint64_t* v_empty = v_full + STAGES;
  uint64_t* s_full = v_empty + STAGES;       // [X]: S holds Q_X K_j^T
  uint64_t* s_free = s_full + 2;             // [X]: tile X's warps hold their S
  uint64_t* p_full = s_free + 2;             // [X]: P_X written, O_X rescaled
  uint64_t* o_done = p_full + 2;             // [X]: P_X V of the last tile done
  uint64_t* mma_done = o_done + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nq = (p.N + BM - 1) / BM;
  const int npair = (nq + 1) / 2;
  // causal: the grid's x runs over (batch, head) and its y over query-tile
  // pairs, the pair with the most key tiles first, so that the block scheduler
  // starts the longest CTAs of every head before any shorter one
  const int pair = p.causal ? (npair - 1 - (int)blockIdx.y) : (int)blockIdx.x;
  const int bh = p.causal ? (int)blockIdx.x : (int)blockIdx.y;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int q0 = pair * 2 * BM;              // first row of tile A; tile B follows
  const int nk_all = (p.N + BN - 1) / BN;
  // key tiles of the pair (tile A takes the last one fully masked when causal:
  // its codes are all 0, so it adds exact zeros to O_A and l_A)
  const int nt = p.causal ? min(nk_all, 2 * pair + 2) : nk_all;

  if (threadIdx.x == 0) {
    mbar_init(q_full, QBF ? NSOFT : 1);   // bf16 Q: one arrival per softmax warp
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&s_free[x], 4);
      mbar_init(&p_full[x], 4);
      mbar_init(&o_done[x], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    // unit E8M0 scales (byte 127) for the ones rows (and every Direct-P P
    // block); the 16 ones rows after the d channel rows of every V stage hold
    // 1.0 in every element: E2M1 code 2 per nibble or E4M3 code 0x38 per byte
    reinterpret_cast<uint4*>(smem + L::SF_1)[lane] = make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
    const uint32_t one = P8 ? 0x38383838u : 0x22222222u;
    for (int st = 0; st < STAGES; ++st)
      for (int i = lane; i < L::PROW; i += 32)    // 16 rows x PROW bytes = PROW 16-byte words
        reinterpret_cast<uint4*>(smem + L::OFF_V + st * L::VB + L::VD)[i] = make_uint4(one, one, one, one);
    if constexpr (D == 64) {
      // V scale chunks: rows 64..79 (column 2, lanes 0..15) unit, rows 80..127
      // zero; the producer refreshes rows 0..63 for every key tile
      for (int st = 0; st < STAGES; ++st) {
        uint32_t* w = reinterpret_cast<uint32_t*>(smem + L::SF_V + 512 * st) + lane * 4;
        w[2] = lane < 16 ? 0x7f7f7f7fu : 0u;
        w[3] = 0u;
      }
    }
    fence_proxy_async_smem();
    tmem_alloc(tmem_holder, TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
    }
    // Q_A, Q_B scales: 4-byte words by cp.async, completing on q_full with the
    // tiles, so that the tile loads are not held behind them; the 2-byte
    // words of d = 64 by plain loads
    const uint8_t* qs = p.q_scales + (long long)bh * p.N * QSB;
    if constexpr (QBF) {
      // Q is quantized by the softmax warps
    } else if constexpr (QSB >= 4) {
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int k = 0; k < NSC; ++k)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int row = q0 + x * BM + lane + 32 * c;
            const bool in = row < p.N;
            cp_async4(smem + L::SF_Q + (x * NSC + k) * 512 + lane * 16 + 4 * c,
                      qs + (long long)(in ? row : 0) * QSB + 4 * k, in ? 4u : 0u);
          }
      cp_async_mbar_arrive(q_full);
    } else {
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int k = 0; k < NSC; ++k)
          stage_sf_rows(smem + L::SF_Q + (x * NSC + k) * 512, qs, q0 + x * BM, min(BM, p.N - q0 - x * BM), QSB,
                        lane, 4 * k);
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (!QBF && lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * L::QB);
      tma_load_3d(smem + L::OFF_Q, &p.tm_q, q_full, 0, q0, bh);
      tma_load_3d(smem + L::OFF_Q + L::QB, &p.tm_q, q_full, 0, q0 + BM, bh);
    }
    const uint8_t* ks = p.k_scales + (long long)bkv * p.N * QSB;
    const uint8_t* vs = p.v_scales + (long long)bkv * D * (p.Np / 32);
    int issued = 0;
    for (int j = 0; j < nt; ++j) {
      const int st = j % STAGES;
      const int ph = ((j / STAGES) - 1) & 1;
      // K_j: codes by TMA, scales rearranged into the chunk (cp.async for
      // 4-byte scale words, plain loads for the 2-byte words of d = 64)
      if (j >= STAGES && !mbar_wait(&k_empty[st], ph, abort_flag, p.err)) break;
      uint8_t* kchunk = smem + L::SF_K + 512 * NSC * st;
      if (QSB >= 4) {
#pragma unroll
        for (int k = 0; k < NSC; ++k)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int r = lane + 32 * c;
            const bool in = j * BN + r < p.N;
            cp_async4(kchunk + 512 * k + lane * 16 + 4 * c, ks + (long long)(j * BN + (in ? r : 0)) * QSB + 4 * k,
                      in ? 4u : 0u);
          }
        cp_async_mbar_arrive(&k_full[st]);
      } else {
        stage_sf_rows(kchunk, ks, j * BN, min(BN, p.N - j * BN), QSB, lane);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&k_full[st], L::KB);
        tma_load_3d(smem + L::OFF_K + st * L::KB, &p.tm_k, &k_full[st], 0, j * BN, bkv);
      }
      // V^T_j: channel rows, the 4 key blocks of tile j
      if (j >= STAGES && !mbar_wait(&v_empty[st], ph, abort_flag, p.err)) break;
      uint8_t* vchunk = smem + L::SF_V + 512 * st;
#pragma unroll
      for (int c = 0; c < D / 32; ++c)   // the d channel rows (the ones rows' scales are fixed)
        cp_async4(vchunk + lane * 16 + 4 * c, vs + (long long)(lane + 32 * c) * (p.Np / 32) + 4 * j, 4u);
      cp_async_mbar_arrive(&v_full[st]);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&v_full[st], L::VD);
        tma_load_3d(smem + L::OFF_V + st * L::VB, &p.tm_v, &v_full[st], j * L::PROW, 0, bkv);
      }
      issued = j + 1;
    }
    if (*abort_flag && lane == 0) {
      volatile int no_abort = 0;
      mbar_wait(q_full, 0, &no_abort, p.err);
      for (int j = max(0, issued - STAGES); j < issued; ++j) {
        mbar_wait(&k_full[j % STAGES], (j / STAGES) & 1, &no_abort, p.err);
        mbar_wait(&v_full[j % STAGES], (j / STAGES) & 1, &no_abort, p.err);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule (waits, descriptor arithmetic) in
    // uniform control flow; one elected lane issues each tcgen05 instruction.
    const bool leader = elect_one();
    constexpr int KSTEPS = D / 64;   // K = 64 per mxf4 MMA
    const uint32_t idesc_s = idesc_bs(BM, BN, 1, 1, false, false, 0, 0);
    // [O | l] += P [V | 1]: E2M1 (kind::mxf4 code 1) or E4M3 (kind::mxf8f6f4 code 0), N = d + 16
    const uint32_t idesc_o = idesc_bs(BM, L::NO, P8 ? 0 : 1, P8 ? 0 : 1, false, false, 0, 0);
    constexpr Swizzle QSW = D == 128 ? SW_64B : SW_32B;
    constexpr uint32_t QSBO = D == 128 ? 512 : 256;
    const uint32_t sq = smem_u32(smem + L::OFF_Q);
    bool ok = mbar_wait(q_full, 0, abort_flag, p.err);
    fence_proxy_async_smem();   // Q scale words written by cp.async
    tc_fence_after();
    if (ok && leader) {
#pragma unroll
      for (int i = 0; i < 2 * NSC; ++i) tmem_cp_sf(tbase + COL_SFQ0 + 4 * i, smem + L::SF_Q + 512 * i);
      tmem_cp_sf(tbase + COL_SF1, smem + L::SF_1);
      if constexpr (D == 128) {
        // unit scales of the ones rows 128..143 of every V stage (fifth column)
#pragma unroll
        for (int st = 0; st < STAGES; ++st) tmem_cp_sf(tbase + COL_SFV + L::SFVS * st + 4, smem + L::SF_1);
      }
    }
    __syncwarp();
    // S = Q_X K_t^T once the other tile's warps hold their S (first = no wait)
    auto issue_qk = [&](int x, int t, bool first) -> bool {
      const int st = t % STAGES;
      if (x == 0) {
        if (!mbar_wait(&k_full[st], (t / STAGES) & 1, abort_flag, p.err)) return false;
        fence_proxy_async_smem();
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int k = 0; k < NSC; ++k)
            tmem_cp_sf(tbase + COL_SFK + 4 * (NSC * st + k), smem + L::SF_K + 512 * (NSC * st + k));
        }
        __syncwarp();
      }
      // the S buffer's last reader: tile B of t-1 (for A), tile A of t (for B)
      if (!first && !mbar_wait(&s_free[x ^ 1], (x == 0 ? t - 1 : t) & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      const uint32_t sqx = sq + x * L::QB;
      const uint32_t sk = smem_u32(smem + L::OFF_K + st * L::KB);
      if (leader) {
#pragma unroll
        for (int k = 0; k < KSTEPS; ++k) {
          uint64_t ad = make_sdesc(sqx + 32 * k, 16, QSBO, QSW);
          uint64_t bd = make_sdesc(sk + 32 * k, 16, QSBO, QSW);
          if constexpr (NV) {
            // UE4M3 scales (descriptor bit 23 clear), chunk k holds the 4
            // scales of this K=64 step
            mma_nvf4(tbase + COL_S, ad, bd, idesc_s & ~(1u << 23), tbase + COL_SFQ0 + 4 * (x * NSC + k),
                     tbase + COL_SFK + 4 * (NSC * st + k), k > 0);
          } else {
            uint32_t id = idesc_s | ((uint32_t)(2 * k) << 29) | ((uint32_t)(2 * k) << 4);
            mma_mxf4(tbase + COL_S, ad, bd, id, tbase + COL_SFQ0 + 4 * x, tbase + COL_SFK + 4 * st, k > 0);
          }
        }
        mma_commit(&s_full[x]);
        if (x == 1) mma_commit(&k_empty[st]);
      }
      __syncwarp();
      return true;
    };
    // [O_X | l_X] += P_X [V_t | 1]
    auto issue_pv = [&](int x, int t) -> bool {
      const int st = t % STAGES;
      if (x == 0) {
        if (!mbar_wait(&v_full[st], (t / STAGES) & 1, abort_flag, p.err)) return false;
        fence_proxy_async_smem();
        if (leader) tmem_cp_sf(tbase + COL_SFV + L::SFVS * st, smem + L::SF_V + 512 * st);
        __syncwarp();
      }
      if (!mbar_wait(&p_full[x], t & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      const uint32_t sp = smem_u32(smem + L::OFF_P + (2 * x + (t & 1)) * L::PB);
      const uint32_t sv = smem_u32(smem + L::OFF_V + st * L::VB);
      if (leader) {
        if constexpr (P8) {
          // E4M3 P with its per-32-key scales (this tile, this step)
          tmem_cp_sf(tbase + COL_SFP0 + 4 * x, smem + L::SF_P + (2 * x + (t & 1)) * 512);
#pragma unroll
          for (int k = 0; k < 4; ++k) {   // 128 keys = 4 x K32
            const uint64_t ad = make_sdesc(sp + 32 * k, 16, 1024, SW_128B);
            const uint32_t sf = ((uint32_t)k << 29) | ((uint32_t)k << 4);
            mma_mxf8(tbase + COL_O0 + L::NO * x, ad, make_sdesc(sv + 32 * k, 16, 1024, SW_128B), idesc_o | sf,
                     tbase + COL_SFP0 + 4 * x, tbase + COL_SFV + L::SFVS * st, t > 0 || k > 0);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 2; ++k) {   // 128 keys = 2 x K64
            const uint64_t ad = make_sdesc(sp + 32 * k, 16, 512, SW_64B);
            const uint32_t sf = ((uint32_t)(2 * k) << 29) | ((uint32_t)(2 * k) << 4);
            mma_mxf4(tbase + COL_O0 + L::NO * x, ad, make_sdesc(sv + 32 * k, 16, 512, SW_64B), idesc_o | sf,
                     tbase + COL_SF1, tbase + COL_SFV + L::SFVS * st, t > 0 || k > 0);
          }
        }
        mma_commit(&o_done[x]);
        if (x == 1) mma_commit(&v_empty[st]);
      }
      __syncwarp();
      return true;
    };
    // Issue order follows the order the hand-offs arrive in: tile A finishes
    // tile j-1 (P_A V_{j-1}), then loads S_j (so S_j of tile B is computed);
    // tile B finishes j-1 (P_B V_{j-1}), then loads S_j (S_{j+1} of tile A).
    // P V goes first so the rescale in the tile's next step finds it done; the
    // other tile needs its S only half a step later.
    if (ok && nt > 0) ok = issue_qk(0, 0, true);
    for (int j = 0; ok && j < nt; ++j) {
      if (j > 0 && !issue_pv(0, j - 1)) { ok = false; break; }
      if (!issue_qk(1, j, false)) { ok = false; break; }
      if (j > 0 && !issue_pv(1, j - 1)) { ok = false; break; }
      if (j + 1 < nt && !issue_qk(0, j + 1, false)) { ok = false; break; }
    }
    if (ok && nt > 0) ok = issue_pv(0, nt - 1) && issue_pv(1, nt - 1);
    if (leader) mma_commit(mma_done);
    __syncwarp();
    volatile int no_abort = 0;
    mbar_wait(mma_done, 0, &no_abort, p.err);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int x = (warp - 2) >> 2;            // query tile 0 (A) or 1 (B)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;           // row within the tile
    const int qi = q0 + x * BM + r;
    const uint32_t lane_base = tbase + ((uint32_t)(quad * 32) << 16);
    // NVFP4 Q/K: the MMA's scores lack the two tensor scales, which fold into
    // the softmax scale: fl32(fl32(scale * ts_q) * ts_k)
    float c = p.c, sm_scale = p.scale;
    if constexpr (NV) {
      sm_scale = (p.scale * *p.ts_q) * *p.ts_k;
      c = (float)((double)sm_scale * 1.4426950408889634);
    }
    const float (&T)[7] = p.T;                // read from the parameter space
    const int lim = p.causal ? min(p.N - 1, qi) : p.N - 1;   // last key of the row
    // swizzle phase of row r: 64-byte rows (E2M1) or 128-byte rows (E4M3)
    const int sw = P8 ? (r & 7) : ((r >> 1) & 3);
    uint8_t* prow = smem + L::OFF_P + 2 * x * L::PB + r * L::PROW;
    if constexpr (QBF) {
      // prologue: this thread's bf16 Q row to MXFP4 (blocks of 32 along d),
      // the codes into the swizzled row of the Q tile (64-byte rows with the
      // 64-byte swizzle at d = 128, 32-byte rows with the 32-byte swizzle at
      // d = 64), the d/32 scale bytes into the tile's scale chunk; rows past
      // N hold zeros, as the tile load would give them
      uint8_t* qrow = smem + L::OFF_Q + x * L::QB + r * (D / 2);
      uint32_t sword = 0;
      uint4 code[D / 32];
      if (qi < p.N) {
        const uint4* src = reinterpret_cast<const uint4*>(p.q_bf16) + ((long long)bh * p.N + qi) * (D / 8);
        uint4 v[D / 32][4];
#pragma unroll
        for (int kb = 0; kb < D / 32; ++kb)
#pragma unroll
          for (int i = 0; i < 4; ++i) v[kb][i] = __ldg(src + 4 * kb + i);
#pragma unroll
        for (int kb = 0; kb < D / 32; ++kb) sword |= mxfp4_block32_bf16(v[kb], code[kb]) << (8 * kb);
      } else {
#pragma unroll
        for (int kb = 0; kb < D / 32; ++kb) code[kb] = make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int kb = 0; kb < D / 32; ++kb) {
        const int cs = D == 128 ? (kb ^ ((r >> 1) & 3)) : (kb ^ ((r >> 2) & 1));
        *reinterpret_cast<uint4*>(qrow + 16 * cs) = code[kb];
      }
      *reinterpret_cast<uint32_t*>(smem + L::SF_Q + x * 512 + (r % 32) * 16 + (r / 32) * 4) = sword;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    float m = -INFINITY;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      if (!mbar_wait(&s_full[x], j & 1, abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      float s[4][32];
      {
        uint32_t v[4][32];
#pragma unroll
        for (int g = 0; g < 4; ++g) tmem_ld32(lane_base + COL_S + 32 * g, v[g]);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          reg_fence32(v[g]);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[g][i] = __uint_as_float(v[g][i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[x]);
      if (j * BN + BN - 1 > lim) {
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (j * BN + 32 * g + i > lim) s[g][i] = -INFINITY;
      }
      const float m_new = fmaxf(m, max128(s));
      const float mc = m_new * c;
      uint8_t* pb = prow + (j & 1) * L::PB;
      if constexpr (P8) {
        // p = 2^x with x = fl32(fl32(s - m) * c) (exact difference near the
        // max: the row max gets p = 1 exactly), then E4M3 with one E8M0 scale
        // per 32 keys (the least X with amax <= 448 * 2^X); the row's four
        // scale bytes go to the scale-factor chunk of this tile and step
        uint32_t sfw = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 xx = fmul2(fadd2(make_float2(s[g][i], s[g][i + 1]), make_float2(-m_new, -m_new)),
                                    make_float2(c, c));
            s[g][i] = ex2_approx(xx.x);
            s[g][i + 1] = ex2_approx(xx.y);
            amax = fmax3(amax, s[g][i], s[g][i + 1]);
          }
          const int X = e4m3_p_block_exp(amax);
          const float inv = __uint_as_float((uint32_t)(127 - X) << 23);
          sfw |= (uint32_t)(X + 127) << (8 * g);
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 a = fmul2(make_float2(s[g][4 * e], s[g][4 * e + 1]), make_float2(inv, inv));
            const float2 b = fmul2(make_float2(s[g][4 * e + 2], s[g][4 * e + 3]), make_float2(inv, inv));
            w[e] = pack_e4m3x4(a.x, a.y, b.x, b.y);
          }
          *reinterpret_cast<uint4*>(pb + (((2 * g) ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(pb + (((2 * g + 1) ^ sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        *reinterpret_cast<uint32_t*>(smem + L::SF_P + (2 * x + (j & 1)) * 512 + (r % 32) * 16 + (r / 32) * 4) = sfw;
      } else {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t pw[4];
          directp_codes32(s[g], c, mc, T, pw);
          *reinterpret_cast<uint4*>(pb + ((g ^ sw) << 4)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
      }
      fence_proxy_async_smem();
      if (j > 0) {
        // rescale O_X and l_X to the new max once P_X V of tile j-1 is in
        if (!mbar_wait(&o_done[x], (j - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        const float alpha = (m_new == m) ? 1.f : ex2_approx(fmaf(m, c, -mc));
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          // the row of O_X and l_X in one TMEM round trip
          uint32_t ov[D / 32][32];
#pragma unroll
          for (int g = 0; g < D / 32; ++g) tmem_ld32(lane_base + COL_O0 + L::NO * x + 32 * g, ov[g]);
          uint32_t lv = tmem_ld1(lane_base + COL_O0 + L::NO * x + D);
          tmem_ld_wait_regs(ov[0], lv);
#pragma unroll
          for (int g = 0; g < D / 32; ++g) {
            reg_fence32(ov[g]);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float2 t = fmul2(make_float2(__uint_as_float(ov[g][i]), __uint_as_float(ov[g][i + 1])),
                               make_float2(alpha, alpha));
              ov[g][i] = __float_as_uint(t.x);
              ov[g][i + 1] = __float_as_uint(t.y);
            }
            tmem_st32(lane_base + COL_O0 + L::NO * x + 32 * g, ov[g]);
          }
          tmem_st1(lane_base + COL_O0 + L::NO * x + D, __float_as_uint(__uint_as_float(lv) * alpha));
          tmem_st_wait();
        }
      }
      m = m_new;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x]);
    }
    if (ok && nt > 0 && mbar_wait(&o_done[x], (nt - 1) & 1, abort_flag, p.err)) {
      tc_fence_after();
      const float l = __uint_as_float(tmem_ld1(lane_base + COL_O0 + L::NO * x + D));
      tmem_ld_wait();
      const float inv_l = 1.f / l;
      const bool valid = qi < p.N;
      const long long orow = ((long long)bh * p.N + qi) * D;
#pragma unroll
      for (int g = 0; g < D / 32; ++g) {
        uint32_t v[32];
        tmem_ld32(lane_base + COL_O0 + L::NO * x + 32 * g, v);
        tmem_ld_wait();
        reg_fence32(v);
        // each thread writes its own row: 32-byte stores where O is 32-byte
        // aligned (every row then is), else 16-byte ones
        if (valid && p.out_bf16) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 t = fmul2(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])),
                                   make_float2(inv_l, inv_l));
            __nv_bfloat162 b2 = __floats2bfloat162_rn(t.x, t.y);
            w[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
          __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.o) + orow + 32 * g;
          if (p.o_align32) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
              st_global_v8(dst + 16 * h, w + 8 * h);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        } else if (valid) {
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 t = fmul2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                   make_float2(inv_l, inv_l));
            w[e] = __float_as_uint(t.x);
            w[e + 1] = __float_as_uint(t.y);
          }
          float* dst = reinterpret_cast<float*>(p.o) + orow + 32 * g;
          if (p.o_align32) {
#pragma unroll
            for (int h = 0; h < 4; ++h)
              st_global_v8(dst + 8 * h, w + 8 * h);
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
      }
      // LSE: Direct-P codes carry the factor 6 of 6*2^x, the FP8 route does not
      if (valid && p.lse) p.lse[(long long)bh * p.N + qi] = sm_scale * m + logf(P8 ? l : l * (1.f / 6.f));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, TMEM_COLS);
}

// Elementwise Direct-P codes with the forward's routines: NATIVE = the
// bracketed native-exponential classifier (32 scores per thread), else the
// threshold count.
template <bool NATIVE>
__global__ void directp_codes_kernel(const float* __restrict__ s, long long n, float m, float c,
                                     Thresh T, uint8_t* __restrict__ out) {
  float t[7];
#pragma unroll
  for (int k = 0; k < 7; ++k) t[k] = T.v[k];
  const float mc = m * c;
  const long long nchunks = (n + 31) / 32;
  for (long long ch = blockIdx.x * (long long)blockDim.x + threadIdx.x; ch - threadIdx.x < nchunks;
       ch += (long long)gridDim.x * blockDim.x) {
    // whole warps stay converged for the warp vote inside the classifier
    const bool live = ch < nchunks;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const long long idx = ch * 32 + i;
      v[i] = (live && idx < n) ? s[idx] : -INFINITY;
    }
    uint32_t pw[4];
    if (NATIVE) {
      directp_codes32(v, c, mc, t, pw);
    } else {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) word |= directp_code(fmaf(v[8 * w + e], c, -mc), t) << (4 * e);
        pw[w] = word;
      }
    }
    if (live) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const long long idx = ch * 32 + i;
        if (idx < n) out[idx] = (uint8_t)((pw[i / 8] >> (4 * (i % 8))) & 0xfu);
      }
    }
  }
}

}  // namespace

template <int D, bool P8, bool NV, bool QBF = false>
static cudaError_t launch_fwd_t(const FwdFp4Params& p, cudaStream_t st) {
  using L = Layout<D, P8, NV>;
  const int nq = (p.N + BM - 1) / BM;
  const dim3 grid = p.causal ? dim3(p.B * p.Hq, (nq + 1) / 2) : dim3((nq + 1) / 2, p.B * p.Hq);
  auto k = fwd_fp4_kernel<D, P8, NV, QBF>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
  k<<<grid, NTHREADS, L::BYTES, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp4(const FwdFp4Params& p, cudaStream_t st) {
  const bool nv = p.ts_q != nullptr;
  if (p.q_bf16) {   // MXFP4 Q quantized in the forward's prologue
    if (p.fp8pv) return p.d == 128 ? launch_fwd_t<128, true, false, true>(p, st) : launch_fwd_t<64, true, false, true>(p, st);
    return p.d == 128 ? launch_fwd_t<128, false, false, true>(p, st) : launch_fwd_t<64, false, false, true>(p, st);
  }
  if (p.fp8pv) {
    if (nv) return p.d == 128 ? launch_fwd_t<128, true, true>(p, st) : launch_fwd_t<64, true, true>(p, st);
    return p.d == 128 ? launch_fwd_t<128, true, false>(p, st) : launch_fwd_t<64, true, false>(p, st);
  }
  if (nv) return p.d == 128 ? launch_fwd_t<128, false, true>(p, st) : launch_fwd_t<64, false, true>(p, st);
  return p.d == 128 ? launch_fwd_t<128, false, false>(p, st) : launch_fwd_t<64, false, false>(p, st);
}

cudaError_t launch_directp_codes(const float* s, long long n, float m, float c, const float* T,
                                 int native, uint8_t* codes, cudaStream_t st) {
  Thresh t;
  for (int k = 0; k < 7; ++k) t.v[k] = T[k];
  long long blocks = ((n + 31) / 32 + 255) / 256;
  int grid = (int)(blocks < 152 * 16 ? (blocks > 0 ? blocks : 1) : 152 * 16);
  if (native) directp_codes_kernel<true><<<grid, 256, 0, st>>>(s, n, m, c, t, codes);
  else directp_codes_kernel<false><<<grid, 256, 0, st>>>(s, n, m, c, t, codes);
  return cudaGetLastError();
}

}  // namespace fa4
