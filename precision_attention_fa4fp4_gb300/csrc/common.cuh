// common.cuh -- inline-PTX building blocks for the sm_103a kernels:
// mbarriers with bounded waits, TMA tile loads, tcgen05 (TMEM allocation,
// MMA issue, commit, TMEM load/store, shared->TMEM scale copies) and the
// shared-memory matrix descriptors the MMAs consume.
//
// Every wait is bounded: after FA4_WAIT_NS nanoseconds a wait records an
// error code in the library's device error word, raises the CTA's abort flag
// and returns false, so a broken pipeline ends the kernel instead of hanging
// the GPU.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#define FA4_DEV __device__ __forceinline__

#ifndef FA4_WAIT_NS
#define FA4_WAIT_NS 2000000000ull   // 2 s
#endif

// error codes written to the device error word (bit flags)
enum : unsigned {
  FA4_DEVERR_TIMEOUT = 1u,
};

namespace fa4 {

FA4_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

FA4_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

FA4_DEV bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
FA4_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

FA4_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

FA4_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

FA4_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

FA4_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// (after flagging the error and the CTA abort word) once limit_ns have passed,
// or when another role of the CTA already aborted.
FA4_DEV bool mbar_wait_ns(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                          unsigned* err, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(err, FA4_DEVERR_TIMEOUT);
      return false;
    }
  }
}

FA4_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                       unsigned* err) {
  return mbar_wait_ns(bar, parity, abort_flag, err, FA4_WAIT_NS);
}

// ----------------------------------------------------------------------------
// fences
// ----------------------------------------------------------------------------
FA4_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
FA4_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FA4_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ----------------------------------------------------------------------------
// TMA (tiled tensor loads into shared memory, completion on an mbarrier)
// ----------------------------------------------------------------------------
FA4_DEV void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                         int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Element-wise add of a shared-memory tile into global memory (bulk tensor
// reduction; out-of-range rows of the box are not written).  Completion is
// tracked by the issuing thread's bulk async groups.
FA4_DEV void tma_reduce_add_3d(const CUtensorMap* map, const void* src_smem, int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src_smem)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
FA4_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// One 32-byte global store of w[0..7] (the address must be 32-byte aligned).
FA4_DEV void st_global_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
// the issuing thread's bulk groups have finished reading shared memory
FA4_DEV void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... all but the most recent one have
FA4_DEV void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// ... and have completed
FA4_DEV void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

FA4_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory
// ----------------------------------------------------------------------------
// Allocate `ncols` TMEM columns (power of two >= 32); whole warp executes.
FA4_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
FA4_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns: thread i of the warp gets lane
// (quadrant base + i), columns [col, col+32).
FA4_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
      "14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
FA4_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Ties 32 registers to this point in the instruction stream: placed after a
// tcgen05.wait::ld, arithmetic on registers loaded before the wait cannot be
// scheduled ahead of it.
FA4_DEV void reg_fence32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}
// The same wait, with the loaded registers as operands: arithmetic on them
// cannot be scheduled ahead of the wait when other work sits between the
// load and its first use.
FA4_DEV void tmem_ld_wait_regs(uint32_t (&r)[32], uint32_t& x) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]), "+r"(x)
               :
               : "memory");
}

FA4_DEV void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%"
      "13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 32 bit, 16 consecutive columns.
FA4_DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%"
      "16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
FA4_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------------------
// shared-memory matrix descriptors (tcgen05 format)
// ----------------------------------------------------------------------------
enum Swizzle : uint32_t { SW_NONE = 0, SW_128B = 2, SW_64B = 4, SW_32B = 6 };

// start address, leading-dimension byte offset, stride-dimension byte offset,
// swizzle mode; bits 46-48 carry the fixed descriptor version 0b001.
FA4_DEV uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, Swizzle sw) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)sw << 61;
  return d;
}

// ----------------------------------------------------------------------------
// instruction descriptors
// ----------------------------------------------------------------------------
// kind::f16 with FP32 accumulate: a/b type 1 = BF16; a_mn/b_mn = 1 for an
// MN-major operand.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn,
                                                 bool b_mn) {
  return (1u << 4)                                   // D = F32
         | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10)
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Block-scaled kinds (UE8M0 scales).  fmt: element format code of the kind
// (kind::mxf4: E2M1 = 1; kind::mxf8f6f4: E4M3 = 0).  The scale-factor ids
// select which byte of each 32-bit TMEM scale column the MMA reads first.
__host__ __device__ constexpr uint32_t idesc_bs(int M, int N, uint32_t afmt, uint32_t bfmt,
                                                bool a_mn, bool b_mn, uint32_t a_sf_id,
                                                uint32_t b_sf_id) {
  return (b_sf_id << 4) | (afmt << 7) | (bfmt << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | (1u << 23)  // UE8M0
         | ((uint32_t)(M >> 4) << 24) | (a_sf_id << 29);
}

// ----------------------------------------------------------------------------
// tcgen05 MMA issue (single thread) and commit
// ----------------------------------------------------------------------------
FA4_DEV void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                     bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// kind::f16 with the A operand in tensor memory (M lanes, K/2 32-bit columns
// of packed bf16 pairs, lower K index in the low half) and B in shared memory.
FA4_DEV void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                            bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

FA4_DEV void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"((uint32_t)accumulate)
      : "memory");
}

// kind::mxf4nvf4 with one UE4M3 scale per 16 elements of K (4 per K=64 MMA);
// the instruction descriptor's scale-format bit (23) is 0 for UE4M3.
FA4_DEV void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"((uint32_t)accumulate)
      : "memory");
}

FA4_DEV void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05 operations of this
// thread have completed.
FA4_DEV void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Copy a 32-row x 128-bit block of scale factors from shared memory into TMEM,
// replicated to all four lane quadrants (row r of the block lands in lanes r,
// 32+r, 64+r, 96+r; its four 32-bit words in columns taddr..taddr+3).
FA4_DEV void tmem_cp_sf(uint32_t taddr, const void* src_smem) {
  uint64_t desc = make_sdesc(smem_u32(src_smem), 16, 128, SW_NONE);
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}

// ----------------------------------------------------------------------------
// numeric helpers
// ----------------------------------------------------------------------------
FA4_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

FA4_DEV float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Pack eight floats into eight E2M1 codes (RNE, satfinite); element 0 in the
// low nibble.
FA4_DEV uint32_t pack_e2m1x8(float x0, float x1, float x2, float x3, float x4, float x5,
                             float x6, float x7) {
  uint32_t out;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}\n"
      : "=r"(out)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(x4), "f"(x5), "f"(x6), "f"(x7));
  return out;
}

// Pack four floats into four E4M3 codes (RNE, satfinite); element 0 in byte 0.
FA4_DEV uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t out;
  asm("{\n .reg .b16 lo, hi;\n"
      " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
      " mov.b32 %0, {lo, hi};\n}\n"
      : "=r"(out)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return out;
}

// E8M0 exponent of a block of probabilities rounded to E4M3: the least X with
// amax <= 448 * 2^X, clamped to [-127, 127].  From the FP32 fields of amax
// (sign clear): the OCP exponent E - 135, plus one where the significand is
// above 1.75 (448 = 1.75 * 2^8), so no element saturates and a probability 1
// computed an ulp low scales to 256 - 2^-16 -> 256, as 1 itself does.  Adding
// 0x1fffff to the bits carries into the exponent field exactly when the
// significand field exceeds 0x600000; E + 1 - 135 <= 121 needs no upper clamp.
FA4_DEV int e4m3_p_block_exp(float amax) {
  const int X = (int)((__float_as_uint(amax) + 0x1fffffu) >> 23) - 135;
  return X < -127 ? -127 : X;
}

// One MXFP4 block (OCP MX rule) of 32 bf16 values given as four 16-byte words
// (element 2i in the low half of word i/2): amax, exponent X = E(amax) - 127 -
// 2 clamped to [-127, 127], elements x * 2^-X (exact) rounded to E2M1 (nearest
// even, saturating).  Returns the scale byte X + 127; the 32 codes go to
// `codes` (element 2i in the low nibble of byte i).  The one routine behind
// every MXFP4 quantization along d (the quantize kernels and the forward's
// bf16-Q prologue), so both give identical bytes.
FA4_DEV uint32_t mxfp4_block32_bf16(const uint4 (&v)[4], uint4& codes) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[i * 8 + 2 * j] = __uint_as_float(w[j] << 16);
      f[i * 8 + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  int X = (int)((__float_as_uint(amax) >> 23) & 0xff) - 127 - 2;
  X = X < -127 ? -127 : (X > 127 ? 127 : X);
  const float inv = __uint_as_float((uint32_t)(127 - X) << 23);
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] *= inv;
  codes.x = pack_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
  codes.y = pack_e2m1x8(f[8], f[9], f[10], f[11], f[12], f[13], f[14], f[15]);
  codes.z = pack_e2m1x8(f[16], f[17], f[18], f[19], f[20], f[21], f[22], f[23]);
  codes.w = pack_e2m1x8(f[24], f[25], f[26], f[27], f[28], f[29], f[30], f[31]);
  return (uint32_t)(X + 127);
}

// 2^e as a float for integer e in [-126, 127].
FA4_DEV float exp2i(int e) { return __int_as_float((e + 127) << 23); }

}  // namespace fa4

namespace fa4 {

// 1 column x 32 lanes TMEM load / store.
FA4_DEV uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
  return r;
}
FA4_DEV void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// Per-warpgroup register budget (every warp of the warpgroup executes it;
// counts are multiples of 8 in [24, 256]).
template <int N>
FA4_DEV void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
FA4_DEV void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// Named barrier over `nthreads` threads (whole warps).
FA4_DEV void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Packed FP32x2 fused multiply-add (two lanes per instruction).
FA4_DEV float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
FA4_DEV float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Two floats -> one byte of two E2M1 codes (RNE, satfinite); a in the low nibble.
FA4_DEV uint32_t cvt_e2m1x2(float a, float b) {
  uint32_t out;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n cvt.u32.u8 %0, t;\n}\n"
      : "=r"(out)
      : "f"(a), "f"(b));
  return out;
}

}  // namespace fa4

namespace fa4 {

// 4-byte asynchronous global->shared copy; src_bytes = 0 writes zeros.
FA4_DEV void cp_async4(void* dst_smem, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst_smem)), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// The mbarrier phase cannot complete before this thread's earlier cp.async
// copies have landed (pending count +1 now, arrive when they complete).
FA4_DEV void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

}  // namespace fa4

namespace fa4 {

FA4_DEV float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

}  // namespace fa4
