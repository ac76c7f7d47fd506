// bwd.cu -- quantized attention backward for sm_103a.
//
// "Hardware-Aware FP4 FlashAttention-4" (arXiv:2609.04105), technical
// summary, Methodology 2 ("Quantized Causal Backward"): the forward keeps
// the FP4 codes and block scales of Q and K and the log-sum-exp; the backward
// recomputes P from those instead of a BF16 score path ("Reconstruction"), and the gradient
// products read FP8 copies of Q, K and V blocked along whichever axis each
// product contracts ("Gradient Formats"); the abstract adds FP8 gradient
// operands for P, dS and dO.
//
// bwd_prep_kernel: D_i = sum_t dO_it O_it, each query row's 16-byte row of
//   initial values (-fl32(LSE_i log2 e) / c and -D_i, each as three bf16
//   parts that sum to it exactly), and zeroes dq (the main kernel adds into dq
//   with bulk tensor reductions).  The MXFP8 views of dO come from the
//   quantize kernels.
// bwd_kernel: one CTA per (batch, kv head, 128-key tile); loop over the query
//   heads of the GQA group x 64-query tiles (causal: from the diagonal on).
//   warp 0       producer (TMA of the step's tiles and initial-value rows,
//                scale-chunk staging)
//   warp 1       TMEM owner + tcgen05 issuer:
//                  S^T  = -LSE log2 e / c + K4 Q4^T
//                                          kind::f16 (ones x initial-value
//                                          rows, K = 16) then kind::mxf4,
//                                          M=128 keys, N=64
//                  dP^T = -D + V8r dOr^T   kind::f16 then kind::mxf8f6f4
//                  dV  += Pq^T dOc         M=128 keys, N=d, K=64 queries
//                  dK  += dSc^T Q8c        M=128 keys, N=d
//                  dQ^T = K8c^T dSr        M=d, N=64 queries, K=128 keys
//                                          (B operand MN-major)
//   warps 2-9    one key row x 32 queries per thread: P = 2^(c s'), s' the
//                accumulator S - LSE log2 e / c, dS = P (dP - D) with dP - D
//                read from its accumulator, quantized to MXFP8:
//                P and dS in blocks of 32 queries (thread-local), dS in
//                blocks of 32 keys (warp-wide max with redux.sync).
//   warps 10-13  dQ^T from TMEM, times softmax_scale, added into dq in two
//                halves of 32 queries, each staged in shared memory and added
//                by its own bulk tensor reduction (staging one half overlaps
//                the reduction still reading the other).
//   After the loop: dV and dK * softmax_scale written by warps 2-9.
// Starting the accumulators at the per-query offsets (an MMA of a constant
// ones operand with the step's initial-value rows) takes the LSE and D
// operands off the P/dS warps (no per-query shared-memory loads, one multiply
// per score instead of an FMA and a subtraction) and off the producer (the
// rows arrive by TMA with the step's tiles).  The exponent is formed as
// fl32(fl32(S + t) c) instead of fmaf(S, c, -fl32(LSE log2 e)): both round
// once at the magnitude of S or of LSE log2 e / c, so they differ by a few
// units in the last place of x.
// d = 64 or 128 (template D).  Block-scaled MMAs have M = 128, so at d = 64
// the A operand of dQ^T (K8c^T, d rows) is padded to 128 rows with zeros in
// shared memory and the extra 64 TMEM lanes of dQ^T are not read.
// The P/dS warps release S^T and dP^T as soon as they hold them in registers,
// so S^T and dP^T of step t+1 run on the tensor core while step t's P and dS
// are built; P, dS and their scale chunks are double-buffered by step parity.
#include <cuda_bf16.h>
#include "common.cuh"
#include "internal.h"

namespace fa4 {
namespace {

constexpr int BK = 128;          // keys per CTA
constexpr int BQ = 64;           // queries per step
constexpr int NST = 3;           // input stages (Q4, dOr, Q8, dOc and initial-value rows of a step)
constexpr int BWD_GROUP = 4;     // causal CTA order: kv heads per group
constexpr int NTHREADS = 14 * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_ST = 0, COL_DPT = 64, COL_DQT = 128, COL_DV = 192, COL_DK = 320,
                   SF_K4 = 448, SF_V8 = 452, SF_K8 = 456, SF_P = 460, SF_DSC = 464, SF_DSR = 468,
                   SF_Q4 = 472, SF_DOR = 480, SF_Q8 = 488, SF_DOC = 496;   // last four: [2 stages]
static_assert(SF_DOC + 8 <= TMEM_COLS, "TMEM budget");

template <int D>
struct BL {   // shared-memory layout (bytes)
  static constexpr int K4 = 0;                       // 128 keys x d/2 B (E2M1)
  static constexpr int V8 = K4 + BK * D / 2;         // 128 keys x d B (E4M3)
  static constexpr int K8 = V8 + BK * D;             // d rows x 128 keys (E4M3), zero rows up to 128
  static constexpr int STG = K8 + 128 * BK;          // stages
  static constexpr int Q4 = 0, DOR = Q4 + BQ * D / 2, Q8 = DOR + BQ * D, DOC = Q8 + D * BQ;
  static constexpr int STAGE_BYTES = DOC + D * BQ;   // 28 KB at d = 128, 14 KB at d = 64
  static constexpr int PQ = STG + NST * STAGE_BYTES; // [2] x 128 keys x 64 B
  static constexpr int DSC = PQ + 2 * BK * BQ;       // [2]
  static constexpr int DSR = DSC + 2 * BK * BQ;      // [2]
  static constexpr int SFC = DSR + 2 * BK * BQ;      // scale chunks, 512 B each
  // chunk ids: 0 K4, 1 V8, 2 K8, 3-4 P, 5-6 dSc, 7-8 dSr (by step parity),
  // 9 + 4 * stage + {0 Q4, 1 dOr, 2 Q8, 3 dOc}
  // [NST] x 64 query rows x 16 B: bf16 parts of -LSE log2 e / c and of -D
  // (the B operand of the accumulator-initialising MMAs)
  static constexpr int FOLD = SFC + (9 + 4 * NST) * 512;
  static constexpr int ONES = FOLD + NST * BQ * 16;       // A operands: [rows 1,1,1,0..][0,0,0,1,1,1,0,0][zeros]
  static constexpr int DQS = ONES + 384;                  // dQ tile [64 q][128 d] fp32
  static constexpr int OKS = DQS + BQ * D * 4;             // int [4]: dQ writers' status
  static constexpr int BAR = OKS + 16;
  static constexpr int NBAR = 1 + NST + NST + 1 + 1 + 2 + 1 + 1 + 1 + 1;
  static constexpr int MISC = BAR + 8 * NBAR;
  static constexpr int BYTES = MISC + 64 + 1024;
};

FA4_DEV int e4m3_block_exp(float amax, float* inv) {
  int E = (int)((__float_as_uint(amax) >> 23) & 0xff);
  int X = E - 127 - 8;
  X = X < -127 ? -127 : (X > 127 ? 127 : X);
  *inv = __uint_as_float((uint32_t)(127 - X) << 23);
  return X;
}

// scale words of `nrows` rows, `bpr` bytes each (<= 4), into a chunk
// The loads of stage_chunk alone: this lane's 16-byte word of the chunk.
FA4_DEV uint4 load_chunk(const uint8_t* __restrict__ src, long long stride, int nvalid, int bpr, int lane) {
  uint32_t w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    int r = lane + 32 * c;
    uint32_t v = 0;
    if (r < nvalid) {
      const uint8_t* p = src + r * stride;
      v = bpr == 4 ? __ldg(reinterpret_cast<const uint32_t*>(p)) : (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(p));
    }
    w[c] = v;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

FA4_DEV void stage_chunk(uint8_t* chunk, const uint8_t* src, long long stride, int nvalid,
                         int bpr, int lane) {
  *reinterpret_cast<uint4*>(chunk + lane * 16) = load_chunk(src, stride, nvalid, bpr, lane);
}

// One 16-byte row of the initialising MMAs' B operand: a and b each as three
// bf16 parts, then two zeros.  Round-to-nearest splitting: each part takes
// the next 8 significant bits of the remainder, and each remainder is exact in
// FP32, so the three parts sum exactly to any float of magnitude >= 2^-110
// (below that the last part loses bits to bf16 subnormals).
FA4_DEV uint4 fold_row(float a, float b) {
  uint16_t h[8];
  const float v[2] = {a, b};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float r = v[j];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const __nv_bfloat16 t = __float2bfloat16_rn(r);
      h[3 * j + k] = __bfloat16_as_ushort(t);
      r -= __bfloat162float(t);
    }
  }
  h[6] = h[7] = 0;
  return make_uint4(h[0] | (uint32_t)h[1] << 16, h[2] | (uint32_t)h[3] << 16, h[4] | (uint32_t)h[5] << 16,
                    h[6] | (uint32_t)h[7] << 16);
}

// 32 floats * inv -> 32 E4M3 codes as two uint4 (element 0 in byte 0)
FA4_DEV void e4m3x32(const float* v, float inv, uint4& lo, uint4& hi) {
  uint32_t w[8];
  const float2 f = make_float2(inv, inv);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 a = fmul2(make_float2(v[4 * i], v[4 * i + 1]), f);
    const float2 b = fmul2(make_float2(v[4 * i + 2], v[4 * i + 3]), f);
    w[i] = pack_e4m3x4(a.x, a.y, b.x, b.y);
  }
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
}

// max |v| over the 32 lanes of the warp
FA4_DEV float warp_max_abs(float v) {
  float r;
  asm volatile("redux.sync.max.abs.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// two 16-byte chunks 2g, 2g+1 of row r of a [rows][64 B] SW64 tile
FA4_DEV void st_row_sw64(uint8_t* tile, int r, int g, uint4 lo, uint4 hi) {
  const int x = (r >> 1) & 3;
  uint8_t* row = tile + r * 64;
  *reinterpret_cast<uint4*>(row + (((2 * g) ^ x) << 4)) = lo;
  *reinterpret_cast<uint4*>(row + (((2 * g + 1) ^ x) << 4)) = hi;
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) bwd_kernel(const __grid_constant__ BwdParams p) {
  using BL = fa4::BL<D>;
  // operand tiles with d-byte (E4M3) or d/2-byte (E2M1) rows along d
  constexpr Swizzle SW4 = D == 128 ? SW_64B : SW_32B;     // Q4, K4
  constexpr uint32_t SBO4 = D == 128 ? 512 : 256;
  constexpr Swizzle SW8 = D == 128 ? SW_128B : SW_64B;    // V8r, dOr
  constexpr uint32_t SBO8 = D == 128 ? 1024 : 512;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BL::BAR);
  uint64_t* fix_full = bars;
  uint64_t* in_full = bars + 1;               // [NST]
  uint64_t* in_empty = in_full + NST;         // [NST]
  uint64_t* s_full = in_empty + NST;
  uint64_t* st_free = s_full + 1;             // the P/dS warps hold S^T, dP^T
  uint64_t* p_full = st_free + 1;             // [2]: P, dS of a step written
  uint64_t* dq_full = p_full + 2;
  uint64_t* dq_free = dq_full + 1;
  uint64_t* acc_done = dq_free + 1;
  uint64_t* mma_done = acc_done + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + BL::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + BL::MISC + 4);
  uint8_t* sfc = smem + BL::SFC;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // CTA order: groups of G (batch, kv head) pairs, key tile major inside a
  // group.  Causal (G = BWD_GROUP): key tile 0 has the most query steps, so
  // the block scheduler starts the longest CTAs of a group first, while only
  // a few heads' dq rows are being accumulated in L2 at a time.  G = 1 (all
  // key tiles of one head, then the next) when every CTA has the same work.
  const int nkt = (p.N + BK - 1) / BK;
  const int nbkv = p.B * p.Hkv;
  const int G = p.causal ? min(BWD_GROUP, nbkv) : 1;
  const int lin = (int)blockIdx.x;
  const int gbase = (lin / (G * nkt)) * G;
  const int gsz = min(G, nbkv - gbase);
  const int rem = lin - gbase * nkt;
  const int kt = rem / gsz;
  const int bkv = gbase + rem % gsz;
  const int b = bkv / p.Hkv, hk = bkv % p.Hkv;
  const int group = p.Hq / p.Hkv;
  const int k0 = kt * BK;
  const int nqt = (p.N + BQ - 1) / BQ;
  const int i0 = p.causal ? k0 / BQ : 0;
  const int per_head = nqt - i0;
  const int nsteps = group * per_head;

  if (threadIdx.x == 0) {
    // fix_full, in_full: the producer's two arrivals, one with the tile bytes
    // before the TMA loads and one after its own shared-memory writes
    mbar_init(fix_full, 2);
    for (int s = 0; s < NST; ++s) { mbar_init(&in_full[s], 2); mbar_init(&in_empty[s], 1); }
    mbar_init(s_full, 1);
    mbar_init(st_free, 8);
    mbar_init(&p_full[0], 8);
    mbar_init(&p_full[1], 8);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);
    mbar_init(acc_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, TMEM_COLS);
  if (warp >= 2) {
    if (D < 128) {
      // zero rows d..127 of the K8c^T operand (the TMA fills rows 0..d-1)
      uint4* z = reinterpret_cast<uint4*>(smem + BL::K8 + D * BK);
      for (int i = threadIdx.x - 64; i < (128 - D) * BK / 16; i += NTHREADS - 64) z[i] = make_uint4(0, 0, 0, 0);
    }
    // the constant A operands of the initialising MMAs: one 8-row core matrix
    // each (every row group reads it), bf16 ones in K columns 0-2 or 3-5,
    // then a zero core matrix for K columns 8-15
    const int i = threadIdx.x - 64;
    if (i < 24) {
      const uint32_t one = 0x3f80u;
      const uint4 v = i < 8 ? make_uint4(one | one << 16, one, 0, 0)
                            : (i < 16 ? make_uint4(0, one << 16, one | one << 16, 0) : make_uint4(0, 0, 0, 0));
      reinterpret_cast<uint4*>(smem + BL::ONES)[i] = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The key tile's loads go first; its scale chunks (plain loads by the
    // warp) are fetched while they are in flight.
    const int nk_valid = min(BK, p.N - k0);
    if (lane == 0) {
      mbar_arrive_expect_tx(fix_full, BK * D / 2 + BK * D + D * BK);
      tma_load_3d(smem + BL::K4, &p.tm_k4, fix_full, 0, k0, bkv);
      tma_load_3d(smem + BL::V8, &p.tm_v8r, fix_full, 0, k0, bkv);
      tma_load_3d(smem + BL::K8, &p.tm_k8c, fix_full, k0, 0, bkv);
    }
    stage_chunk(sfc + 0 * 512, p.k4_s + ((long long)bkv * p.N + k0) * (D / 32), D / 32, nk_valid, D / 32, lane);
    stage_chunk(sfc + 1 * 512, p.v8r_s + ((long long)bkv * p.N + k0) * (D / 32), D / 32, nk_valid, D / 32, lane);
    stage_chunk(sfc + 2 * 512, p.k8c_s + (long long)bkv * D * (p.Np / 32) + k0 / 32, p.Np / 32, D, 4, lane);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(fix_full);
    int issued = 0;
    // The scale-chunk words of a step are loaded into registers before the
    // producer waits for that step's stage to be released, so their latency
    // overlaps the wait; the tile loads are issued as soon as it is free.
    uint4 c0, c1, c2, c3;
    auto load_chunks = [&](int t) {
      const int bh = b * p.Hq + hk * group + t / per_head;
      const int q0 = (i0 + t % per_head) * BQ;
      const int nq_valid = min(BQ, p.N - q0);
      c0 = load_chunk(p.q4_s + ((long long)bh * p.N + q0) * (D / 32), D / 32, nq_valid, D / 32, lane);
      c1 = load_chunk(p.do_r_s + ((long long)bh * p.N + q0) * (D / 32), D / 32, nq_valid, D / 32, lane);
      c2 = load_chunk(p.q8c_s + (long long)bh * D * (p.Np / 32) + q0 / 32, p.Np / 32, D, 2, lane);
      c3 = load_chunk(p.do_c_s + (long long)bh * D * (p.Np / 32) + q0 / 32, p.Np / 32, D, 2, lane);
    };
    if (nsteps > 0) load_chunks(0);
    for (int t = 0; t < nsteps; ++t) {
      const int st = t % NST;
      const int h = hk * group + t / per_head;
      const int q0 = (i0 + t % per_head) * BQ;
      const int bh = b * p.Hq + h;
      if (t >= NST && !mbar_wait(&in_empty[st], ((t / NST) - 1) & 1, abort_flag, p.err)) break;
      if (lane == 0) {
        uint8_t* sb = smem + BL::STG + st * BL::STAGE_BYTES;
        mbar_arrive_expect_tx(&in_full[st], BL::STAGE_BYTES + BQ * 16);
        tma_load_3d(sb + BL::Q4, &p.tm_q4, &in_full[st], 0, q0, bh);
        tma_load_3d(sb + BL::DOR, &p.tm_do_r, &in_full[st], 0, q0, bh);
        tma_load_3d(sb + BL::Q8, &p.tm_q8c, &in_full[st], q0, 0, bh);
        tma_load_3d(sb + BL::DOC, &p.tm_do_c, &in_full[st], q0, 0, bh);
        tma_load_3d(smem + BL::FOLD + st * BQ * 16, &p.tm_fold, &in_full[st], 0, q0, bh);
      }
      uint8_t* sc = sfc + (9 + 4 * st) * 512;
      reinterpret_cast<uint4*>(sc)[lane] = c0;
      reinterpret_cast<uint4*>(sc + 512)[lane] = c1;
      reinterpret_cast<uint4*>(sc + 1024)[lane] = c2;
      reinterpret_cast<uint4*>(sc + 1536)[lane] = c3;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&in_full[st]);
      issued = t + 1;
      if (t + 1 < nsteps) load_chunks(t + 1);
    }
    if (*abort_flag && lane == 0) {
      volatile int no_abort = 0;
      mbar_wait(fix_full, 0, &no_abort, p.err);
      for (int t = max(0, issued - NST); t < issued; ++t) mbar_wait(&in_full[t % NST], (t / NST) & 1, &no_abort, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule in uniform control flow; one elected
    // lane issues each tcgen05 instruction.
    const bool leader = elect_one();
    const uint32_t id_st = idesc_bs(128, BQ, 1, 1, false, false, 0, 0);      // mxf4
    const uint32_t id_dp = idesc_bs(128, BQ, 0, 0, false, false, 0, 0);      // mxf8 e4m3
    const uint32_t id_acc = idesc_bs(128, D, 0, 0, false, false, 0, 0);   // N = d
    const uint32_t id_dq = idesc_bs(128, BQ, 0, 0, false, true, 0, 0);
    const uint32_t id_fold = idesc_f16(128, BQ, true, false, false);      // bf16, K = 16
    const uint32_t s_k4 = smem_u32(smem + BL::K4), s_v8 = smem_u32(smem + BL::V8),
                   s_k8 = smem_u32(smem + BL::K8), s_pq = smem_u32(smem + BL::PQ),
                   s_dsc = smem_u32(smem + BL::DSC), s_dsr = smem_u32(smem + BL::DSR),
                   s_fold = smem_u32(smem + BL::FOLD), s_ones = smem_u32(smem + BL::ONES);
    bool ok = mbar_wait(fix_full, 0, abort_flag, p.err);
    tc_fence_after();
    if (ok && leader) {
      tmem_cp_sf(tbase + SF_K4, sfc + 0 * 512);
      tmem_cp_sf(tbase + SF_V8, sfc + 1 * 512);
      tmem_cp_sf(tbase + SF_K8, sfc + 2 * 512);
    }
    __syncwarp();
    // S^T(t) = K4 Q4^T and dP^T(t) = V8r dOr^T, into TMEM the P/dS warps have
    // released (first = nothing to wait for)
    auto issue_sdp = [&](int t, bool first) -> bool {
      const int st = t % NST, sp = t & 1;     // input stage; TMEM scale slot
      if (!mbar_wait(&in_full[st], (t / NST) & 1, abort_flag, p.err)) return false;
      if (!first && !mbar_wait(st_free, (t - 1) & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      const uint32_t sb = smem_u32(smem + BL::STG + st * BL::STAGE_BYTES);
      if (leader) {
        const uint8_t* sc = sfc + (9 + 4 * st) * 512;
        tmem_cp_sf(tbase + SF_Q4 + 4 * sp, sc);
        tmem_cp_sf(tbase + SF_DOR + 4 * sp, sc + 512);
        tmem_cp_sf(tbase + SF_Q8 + 4 * sp, sc + 1024);
        tmem_cp_sf(tbase + SF_DOC + 4 * sp, sc + 1536);
        // S^T starts at -LSE log2 e / c and dP^T at -D of each query column:
        // ones (128 x 16, K columns 0-2 or 3-5) times the stage's bf16 parts
        // (64 x 16; the descriptor's K offset 0 repeats columns 0-7 as 8-15,
        // which meet the zero half of A)
        const uint64_t fb = make_sdesc(s_fold + st * BQ * 16, 0, 128, SW_NONE);
        mma_f16(tbase + COL_ST, make_sdesc(s_ones, 256, 0, SW_NONE), fb, id_fold, false);
        mma_f16(tbase + COL_DPT, make_sdesc(s_ones + 128, 128, 0, SW_NONE), fb, id_fold, false);
#pragma unroll
        for (int k = 0; k < D / 64; ++k) {     // K = d: K64 steps
          const uint32_t sf = ((uint32_t)(2 * k) << 29) | ((uint32_t)(2 * k) << 4);
          mma_mxf4(tbase + COL_ST, make_sdesc(s_k4 + 32 * k, 16, SBO4, SW4),
                   make_sdesc(sb + BL::Q4 + 32 * k, 16, SBO4, SW4), id_st | sf, tbase + SF_K4,
                   tbase + SF_Q4 + 4 * sp, true);
        }
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {     // K = d: K32 steps
          const uint32_t sf = ((uint32_t)k << 29) | ((uint32_t)k << 4);
          mma_mxf8(tbase + COL_DPT, make_sdesc(s_v8 + 32 * k, 16, SBO8, SW8),
                   make_sdesc(sb + BL::DOR + 32 * k, 16, SBO8, SW8), id_dp | sf, tbase + SF_V8,
                   tbase + SF_DOR + 4 * sp, true);
        }
        mma_commit(s_full);
      }
      __syncwarp();
      return true;
    };
    if (ok && nsteps > 0) ok = issue_sdp(0, true);
    for (int t = 0; ok && t < nsteps; ++t) {
      const int st = t % NST, sp = t & 1;
      if (t + 1 < nsteps && !issue_sdp(t + 1, false)) { ok = false; break; }
      if (!mbar_wait(&p_full[sp], (t >> 1) & 1, abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      if (t >= 1 && !mbar_wait(dq_free, (t - 1) & 1, abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sb = smem_u32(smem + BL::STG + st * BL::STAGE_BYTES);
      if (leader) {
        tmem_cp_sf(tbase + SF_P, sfc + (3 + sp) * 512);
        tmem_cp_sf(tbase + SF_DSC, sfc + (5 + sp) * 512);
        tmem_cp_sf(tbase + SF_DSR, sfc + (7 + sp) * 512);
        // dV += Pq^T dOc, dK += dSc^T Q8c (K = 64 queries: 2 x K32)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t sf = ((uint32_t)k << 29) | ((uint32_t)k << 4);
          mma_mxf8(tbase + COL_DV, make_sdesc(s_pq + sp * BK * BQ + 32 * k, 16, 512, SW_64B),
                   make_sdesc(sb + BL::DOC + 32 * k, 16, 512, SW_64B), id_acc | sf, tbase + SF_P,
                   tbase + SF_DOC + 4 * sp, t > 0 || k > 0);
          mma_mxf8(tbase + COL_DK, make_sdesc(s_dsc + sp * BK * BQ + 32 * k, 16, 512, SW_64B),
                   make_sdesc(sb + BL::Q8 + 32 * k, 16, 512, SW_64B), id_acc | sf, tbase + SF_DSC,
                   tbase + SF_Q8 + 4 * sp, t > 0 || k > 0);
        }
        // dQ^T = K8c^T dSr (K = 128 keys: 4 x K32; dSr stored [keys][64 q], MN-major;
        // A has 128 rows: d rows of K8c^T, then zeros)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t sf = ((uint32_t)k << 29) | ((uint32_t)k << 4);
          mma_mxf8(tbase + COL_DQT, make_sdesc(s_k8 + 32 * k, 16, 1024, SW_128B),
                   make_sdesc(s_dsr + sp * BK * BQ + 2048 * k, 8192, 512, SW_64B), id_dq | sf,
                   tbase + SF_K8, tbase + SF_DSR, k > 0);
        }
        mma_commit(dq_full);
        mma_commit(&in_empty[st]);
      }
      __syncwarp();
    }
    if (leader) {
      mma_commit(acc_done);
      mma_commit(mma_done);
    }
    __syncwarp();
    volatile int no_abort = 0;
    mbar_wait(mma_done, 0, &no_abort, p.err);
    __syncwarp();
  } else if (warp < 10) {
    // ------------------------------------------------------------ P / dS
    const int quad = warp & 3;
    const int g = (warp - 2) >> 2;            // query group 0..1 (32 queries each)
    const int r = quad * 32 + lane;           // key row
    const int key = k0 + r;
    const uint32_t lane_base = tbase + ((uint32_t)(quad * 32) << 16);
    const float c = p.c;
    bool ok = true;
    uint8_t* const pq0 = smem + BL::PQ;
    uint8_t* const dsc0 = smem + BL::DSC;
    uint8_t* const dsr0 = smem + BL::DSR;
    for (int t = 0; t < nsteps; ++t) {
      const int st = t % NST, sp = t & 1;     // input stage; P/dS buffer
      const int q0 = (i0 + t % per_head) * BQ;
      uint8_t* pq = pq0 + sp * BK * BQ;
      uint8_t* dsc = dsc0 + sp * BK * BQ;
      uint8_t* dsr = dsr0 + sp * BK * BQ;
      // S^T and dP^T of step t.  The MMAs that wrote them waited for the
      // step's input stage, so that stage is always complete here; at d = 64
      // the warps wait for it all the same (measured 3.6 % faster at d = 64
      // with the wait and 2.8 % faster at d = 128 without it)
      if (!mbar_wait(s_full, t & 1, abort_flag, p.err)) { ok = false; break; }
      if constexpr (D == 64) {
        if (!mbar_wait(&in_full[st], (t / NST) & 1, abort_flag, p.err)) { ok = false; break; }
      }
      tc_fence_after();
      float s[32], dp[32];
      {
        uint32_t v[32], w[32];
        tmem_ld32(lane_base + COL_ST + 32 * g, v);
        tmem_ld32(lane_base + COL_DPT + 32 * g, w);
        tmem_ld_wait();
        reg_fence32(v);
        reg_fence32(w);
#pragma unroll
        for (int i = 0; i < 32; ++i) { s[i] = __uint_as_float(v[i]); dp[i] = __uint_as_float(w[i]); }
      }
      // S^T and dP^T are in registers: the tensor core may overwrite them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(st_free);
      const int qbase = q0 + 32 * g;
      float pmax = 0.f, dsmax = 0.f;
      // every (key, query) of this warp's block in range and unmasked: the
      // same arithmetic without the per-element validity test
      const bool full = k0 + BK <= p.N && qbase + 32 <= p.N && (!p.causal || k0 + BK - 1 <= qbase);
      // s holds S - LSE log2 e / c and dp holds dP - D (the accumulators
      // started there)
      if (full) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = fmul2(make_float2(s[i], s[i + 1]), make_float2(c, c));
          const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          const float2 ds = fmul2(pv, make_float2(dp[i], dp[i + 1]));
          s[i] = pv.x; s[i + 1] = pv.y;
          dp[i] = ds.x; dp[i + 1] = ds.y;
          pmax = fmax3(pmax, pv.x, pv.y);
          dsmax = fmax3(dsmax, fabsf(ds.x), fabsf(ds.y));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int q = qbase + i;
          const bool valid = key < p.N && q < p.N && (!p.causal || key <= q);
          const float pv = valid ? ex2_approx(s[i] * c) : 0.f;
          const float ds = pv * dp[i];
          s[i] = pv;
          dp[i] = ds;
          pmax = fmaxf(pmax, pv);
          dsmax = fmaxf(dsmax, fabsf(ds));
        }
      }
      // P and dS in blocks of 32 queries (this thread's columns); P under the
      // probability blocks' exponent, dS under the OCP one
      float inv;
      uint4 lo, hi;
      const int xp = e4m3_p_block_exp(pmax);
      e4m3x32(s, __uint_as_float((uint32_t)(127 - xp) << 23), lo, hi);
      st_row_sw64(pq, r, g, lo, hi);
      const int xc = e4m3_block_exp(dsmax, &inv);
      e4m3x32(dp, inv, lo, hi);
      st_row_sw64(dsc, r, g, lo, hi);
      sfc[(3 + sp) * 512 + lane * 16 + quad * 4 + g] = (uint8_t)(xp + 127);
      sfc[(5 + sp) * 512 + lane * 16 + quad * 4 + g] = (uint8_t)(xc + 127);
      // dS in blocks of 32 keys (the 32 lanes of this warp) per query column.
      // The block exponent rule of e4m3_block_exp, from the biased exponent E
      // of the column's amax (sign bit clear): X = max(E - 135, -127), so the
      // factor 2^-X has exponent field min(262 - E, 254) and the scale byte is
      // X + 127 = max(E, 8) - 8.
      // The column maxima are warp-uniform: their exponent bytes are packed
      // four to a word, and each lane picks its own column's at the end.
      uint32_t ew[8];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        uint32_t eb[4];
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
          const uint32_t a0 = __float_as_uint(warp_max_abs(dp[i + u]));
          const uint32_t a1 = __float_as_uint(warp_max_abs(dp[i + u + 1]));
          const float2 f = make_float2(__uint_as_float(min(0x83000000u - (a0 & 0x7f800000u), 0x7f000000u)),
                                       __uint_as_float(min(0x83000000u - (a1 & 0x7f800000u), 0x7f000000u)));
          const float2 qv = fmul2(make_float2(dp[i + u], dp[i + u + 1]), f);
          dp[i + u] = qv.x;
          dp[i + u + 1] = qv.y;
          eb[u] = a0 << 1;          // E in byte 3
          eb[u + 1] = a1 << 1;
        }
        ew[i / 4] = __byte_perm(__byte_perm(eb[0], eb[1], 0x0073), __byte_perm(eb[2], eb[3], 0x0073), 0x5410);
      }
      {
        uint32_t pair_lo, pair_hi;   // words 2k, 2k+1 with k = lane / 8
        const uint32_t l0 = (lane & 8) ? ew[2] : ew[0], h0 = (lane & 8) ? ew[3] : ew[1];
        const uint32_t l1 = (lane & 8) ? ew[6] : ew[4], h1 = (lane & 8) ? ew[7] : ew[5];
        pair_lo = (lane & 16) ? l1 : l0;
        pair_hi = (lane & 16) ? h1 : h0;
        const uint32_t my_e = __byte_perm(pair_lo, pair_hi, (uint32_t)(lane & 7)) & 0xffu;
        sfc[(7 + sp) * 512 + lane * 16 + g * 4 + quad] = (uint8_t)(max(my_e, 8u) - 8u);
      }
      {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = pack_e4m3x4(dp[4 * i], dp[4 * i + 1], dp[4 * i + 2], dp[4 * i + 3]);
        st_row_sw64(dsr, r, g, make_uint4(w[0], w[1], w[2], w[3]), make_uint4(w[4], w[5], w[6], w[7]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sp]);
    }
    // dV, dK out
    if (ok && mbar_wait(acc_done, 0, abort_flag, p.err)) {
      tc_fence_after();
      const bool valid = key < p.N;
      const long long orow = ((long long)bkv * p.N + key) * D;
#pragma unroll 1
      for (int cc = (D / 64) * g; cc < (D / 64) * (g + 1); ++cc) {    // d/32 x 32 columns, half per group
        uint32_t v[32];
        tmem_ld32(lane_base + COL_DV + 32 * cc, v);
        tmem_ld_wait();
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(p.dv + orow + 32 * cc);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
        tmem_ld32(lane_base + COL_DK + 32 * cc, v);
        tmem_ld_wait();
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(p.dk + orow + 32 * cc);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]) * p.scale, __uint_as_float(v[4 * q + 1]) * p.scale,
                                 __uint_as_float(v[4 * q + 2]) * p.scale, __uint_as_float(v[4 * q + 3]) * p.scale);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ writer
    // dQ^T from TMEM, times softmax_scale, staged as a [64 q][128 d] fp32 tile
    // in shared memory and added into dq by one bulk tensor reduction per step.
    const int quad = warp & 3;
    const int drow = quad * 32 + lane;
    const uint32_t lane_base = tbase + ((uint32_t)(quad * 32) << 16);
    float* stage = reinterpret_cast<float*>(smem + BL::DQS);
    int* okw = reinterpret_cast<int*>(smem + BL::OKS);
    const bool issuer = warp == 10 && lane == 0;
    bool prev_b = false;
    for (int t = 0; t < nsteps; ++t) {
      const int h = hk * group + t / per_head;
      const int q0 = (i0 + t % per_head) * BQ;
      // the four writer warps leave together: each publishes its status
      // before the barrier and all read the four after it
      const bool wok = mbar_wait(dq_full, t & 1, abort_flag, p.err);
      uint32_t v0[32], v1[32];
      if (wok) {
        tc_fence_after();
        tmem_ld32(lane_base + COL_DQT, v0);
        tmem_ld32(lane_base + COL_DQT + 32, v1);
        tmem_ld_wait();
        reg_fence32(v0);
        reg_fence32(v1);
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0 && wok) mbar_arrive(dq_free);
      // the staging tile is two halves of 32 queries, each added into dq by
      // its own bulk reduction: half A of this step is written once the
      // previous step's half A has been read (its half B may still be read),
      // and half B once the previous half B has been read (a step whose
      // second half lies past N issues no reduction for it)
      if (issuer) {
        if (prev_b) bulk_wait_read1();
        else bulk_wait_read0();
      }
      const bool all_ok = __all_sync(0xffffffffu, wok);
      if (lane == 0) okw[warp - 10] = all_ok ? 1 : 0;
      named_bar(1, 128);
      if (!(okw[0] & okw[1] & okw[2] & okw[3])) break;
      if (drow < D) {     // TMEM lanes d..127 hold the zero rows of the padded operand
#pragma unroll
        for (int i = 0; i < 32; ++i) stage[i * D + drow] = __uint_as_float(v0[i]) * p.scale;
      }
      fence_proxy_async_smem();
      named_bar(1, 128);
      if (issuer) {
        tma_reduce_add_3d(&p.tm_dq, stage, 0, q0, b * p.Hq + h);
        bulk_commit();
        bulk_wait_read1();
      }
      named_bar(1, 128);
      if (drow < D) {
#pragma unroll
        for (int i = 0; i < 32; ++i) stage[(32 + i) * D + drow] = __uint_as_float(v1[i]) * p.scale;
      }
      fence_proxy_async_smem();
      named_bar(1, 128);
      prev_b = q0 + 32 < p.N;
      if (issuer && prev_b) {
        tma_reduce_add_3d(&p.tm_dq, stage + 32 * D, 0, q0 + 32, b * p.Hq + h);
        bulk_commit();
      }
    }
    if (issuer) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, TMEM_COLS);
}

// D_i = sum_t dO_it * O_it (one warp per row), the row's initial values
// -fl32(LSE_i log2 e) / c and -D_i as bf16 parts, and dq = 0.
template <int D, bool O_BF16>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const void* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        const float* __restrict__ lse, float c, float l2e,
                                                        long long rows, uint4* __restrict__ fold,
                                                        float* __restrict__ dq) {
  const int lane = threadIdx.x % 32;
  const long long wpb = blockDim.x / 32;
  constexpr int E = D / 32;     // elements per lane: 4 (d = 128) or 2 (d = 64)
  for (long long row = blockIdx.x * wpb + threadIdx.x / 32; row < rows; row += (long long)gridDim.x * wpb) {
    const long long base = row * D + lane * E;
    uint32_t dw[E / 2];
    float dof[E], of[E];
    if constexpr (E == 4) {
      const uint2 t = *reinterpret_cast<const uint2*>(dout + base);
      dw[0] = t.x; dw[1] = t.y;
    } else {
      dw[0] = *reinterpret_cast<const uint32_t*>(dout + base);
    }
#pragma unroll
    for (int u = 0; u < E / 2; ++u) {
      dof[2 * u] = __uint_as_float(dw[u] << 16);
      dof[2 * u + 1] = __uint_as_float(dw[u] & 0xffff0000u);
    }
    if constexpr (O_BF16) {
      uint32_t ow[E / 2];
      const __nv_bfloat16* ob = reinterpret_cast<const __nv_bfloat16*>(o) + base;
      if constexpr (E == 4) {
        const uint2 t = *reinterpret_cast<const uint2*>(ob);
        ow[0] = t.x; ow[1] = t.y;
      } else {
        ow[0] = *reinterpret_cast<const uint32_t*>(ob);
      }
#pragma unroll
      for (int u = 0; u < E / 2; ++u) {
        of[2 * u] = __uint_as_float(ow[u] << 16);
        of[2 * u + 1] = __uint_as_float(ow[u] & 0xffff0000u);
      }
    } else {
      const float* of32 = reinterpret_cast<const float*>(o) + base;
      if constexpr (E == 4) {
        const float4 t = *reinterpret_cast<const float4*>(of32);
        of[0] = t.x; of[1] = t.y; of[2] = t.z; of[3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(of32);
        of[0] = t.x; of[1] = t.y;
      }
    }
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < E; ++u) acc += dof[u] * of[u];
#pragma unroll
    for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) fold[row] = fold_row(-(lse[row] * l2e) / c, -acc);
    if constexpr (E == 4) *reinterpret_cast<float4*>(dq + base) = make_float4(0.f, 0.f, 0.f, 0.f);
    else *reinterpret_cast<float2*>(dq + base) = make_float2(0.f, 0.f);
  }
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdPrepParams& p, cudaStream_t st) {
  const long long rows = (long long)p.B * p.Hq * p.N;
  cudaError_t e;
  if ((e = launch_quantize(p.dout, rows, p.d, p.N, (long long)p.B * p.Hq, 1, 0, p.do_r, p.do_r_s, st)) != cudaSuccess) return e;
  if ((e = launch_quantize(p.dout, rows, p.d, p.N, (long long)p.B * p.Hq, 1, 1, p.do_c, p.do_c_s, st)) != cudaSuccess) return e;
  long long blocks = (rows + 7) / 8;
  int grid = (int)(blocks < 152 * 16 ? blocks : 152 * 16);
  const __nv_bfloat16* dout = (const __nv_bfloat16*)p.dout;
  if (p.d == 128) {
    if (p.o_bf16) bwd_prep_kernel<128, true><<<grid, 256, 0, st>>>(p.o, dout, p.lse, p.c, p.l2e, rows, p.fold, p.dq);
    else bwd_prep_kernel<128, false><<<grid, 256, 0, st>>>(p.o, dout, p.lse, p.c, p.l2e, rows, p.fold, p.dq);
  } else {
    if (p.o_bf16) bwd_prep_kernel<64, true><<<grid, 256, 0, st>>>(p.o, dout, p.lse, p.c, p.l2e, rows, p.fold, p.dq);
    else bwd_prep_kernel<64, false><<<grid, 256, 0, st>>>(p.o, dout, p.lse, p.c, p.l2e, rows, p.fold, p.dq);
  }
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_bwd_main_t(const BwdParams& p, cudaStream_t st) {
  const dim3 grid((unsigned)((p.N + BK - 1) / BK) * (unsigned)(p.B * p.Hkv));
  auto k = bwd_kernel<D>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, BL<D>::BYTES);
  k<<<grid, NTHREADS, BL<D>::BYTES, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdParams& p, cudaStream_t st) {
  return p.d == 128 ? launch_bwd_main_t<128>(p, st) : launch_bwd_main_t<64>(p, st);
}

}  // namespace fa4
