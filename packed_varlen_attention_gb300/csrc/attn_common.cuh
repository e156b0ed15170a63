// attn_common.cuh -- device helpers shared by the attention kernels (forward
// and backward): block classification, TMEM loads/stores, grouped
// tcgen05.mma issue, bounded waits, packed arithmetic.  Internal header: each
// kernel translation unit gets its own copy (anonymous namespace).
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "fm_device.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

// kClsP: partially masked through the column intervals (element mask from the
// four vectors); kClsPC: partially masked only through causality and the
// sample bound (the diagonal block of a causal mask).  Both count as
// partially masked.
enum : int { kClsF = 0, kClsP = 1, kClsU = 2, kClsPC = 3 };

__device__ __forceinline__ int clamp_tok(int x, int T) { return x < 0 ? 0 : (x > T ? T : x); }

// Block class from the eight statistics of the key tile (FlashMask article,
// section 3.2; rows [r0, r1) half-open, the diagonal counts as lower).
__device__ __forceinline__ int classify_block(int r0, int r1, int c0, int c1, const int* st,
                                              bool has_mask, bool causal) {
  bool lt_full = false, lt_touch = false, ut_full = false, ut_touch = false;
  if (has_mask) {
    lt_full = r0 >= st[1] && r1 <= st[2];
    lt_touch = r0 < st[3] && r1 > st[0];
    ut_full = r0 >= st[5] && r1 <= st[6];
    ut_touch = r0 < st[7] && r1 > st[4];
  }
  if (causal) ut_full = ut_touch = true;
  if (r1 - 1 < c0) return ut_full ? kClsF : (ut_touch ? kClsP : kClsU);
  if (r0 >= c1 - 1) return lt_full ? kClsF : (lt_touch ? kClsP : kClsU);
  if (lt_full && ut_full) return kClsF;
  if (lt_touch || (!causal && ut_touch)) return kClsP;
  if (causal) return kClsPC;  // only the diagonal (and no interval) masks it
  return kClsU;
}

// ---------------------------------------------------------------------------
// TMEM helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// 16 consecutive 32-bit columns per lane, with the wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 64 consecutive 32-bit columns per lane, one wait for all of them.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// 128 consecutive 32-bit columns per lane, one wait for all of them.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}

// The whole S row of one thread (BN columns) with one wait.
template <int BN>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&r)[BN]);
template <>
__device__ __forceinline__ void tmem_ld_row<64>(uint32_t taddr, uint32_t (&r)[64]) {
  tmem_ld64(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_row<128>(uint32_t taddr, uint32_t (&r)[128]) {
  tmem_ld128(taddr, r);
}

// Bits of the columns [a, b) that fall in 32-column word w (empty if b <= a).
__device__ __forceinline__ uint32_t range_bits(int a, int b, int w) {
  const int lo = min(max(a - 32 * w, 0), 32);
  const int hi = min(max(b - 32 * w, 0), 32);
  return static_cast<uint32_t>((1ull << hi) - 1ull) & ~static_cast<uint32_t>((1ull << lo) - 1ull);
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Groups of MMAs issued from one asm block by the converged warp: every lane
// runs the block and elect.sync picks the one that issues.  Issue from a
// warp-uniform stream costs far fewer issue cycles than the same MMAs issued
// by lane 0 inside a divergent branch, and keeps up with the tensor pipe
// when softmax warps share the issuer's SMSP.  Between consecutive MMAs the
// issuing lane only adds two descriptor offsets.  The first step accumulates
// iff acc0 != 0, the later ones always accumulate.
// SS: A and B from shared memory, step k adds OA_k / OB_k to the descriptors'
// start-address fields.  TS: A from TMEM (8 columns per K=16 step), B from
// shared memory advanced by OB per step.
template <int OA1, int OB1, int OA2, int OB2, int OA3, int OB3>
__device__ __forceinline__ void umma_ss_group4(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t acc0) {
  asm volatile("{\n\t.reg .pred p, q, e;\n\t.reg .b32 el;\n\t"
               ".reg .b64 a, b;\n\t"
               "elect.sync el|e, 0xffffffff;\n\t"
               "setp.ne.b32 p, %4, 0;\n\t"
               "setp.eq.u32 q, 0, 0;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               "add.s64 a, %1, %5;\n\tadd.s64 b, %2, %6;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "add.s64 a, %1, %7;\n\tadd.s64 b, %2, %8;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "add.s64 a, %1, %9;\n\tadd.s64 b, %2, %10;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "}"
               :: "r"(d_tmem),
                  "l"(a_desc),
                  "l"(b_desc),
                  "r"(idesc),
                  "r"(acc0),
                  "n"(OA1),
                  "n"(OB1),
                  "n"(OA2),
                  "n"(OB2),
                  "n"(OA3),
                  "n"(OB3)
               : "memory");
}

template <int OA1, int OB1, int OA2, int OB2, int OA3, int OB3, int OA4, int OB4, int OA5, int OB5, int OA6, int OB6, int OA7, int OB7>
__device__ __forceinline__ void umma_ss_group8(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t acc0) {
  asm volatile("{\n\t.reg .pred p, q, e;\n\t.reg .b32 el;\n\t"
               ".reg .b64 a, b;\n\t"
               "elect.sync el|e, 0xffffffff;\n\t"
               "setp.ne.b32 p, %4, 0;\n\t"
               "setp.eq.u32 q, 0, 0;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               "add.s64 a, %1, %5;\n\tadd.s64 b, %2, %6;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "add.s64 a, %1, %7;\n\tadd.s64 b, %2, %8;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "add.s64 a, %1, %9;\n\tadd.s64 b, %2, %10;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "add.s64 a, %1, %11;\n\tadd.s64 b, %2, %12;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "add.s64 a, %1, %13;\n\tadd.s64 b, %2, %14;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "add.s64 a, %1, %15;\n\tadd.s64 b, %2, %16;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "add.s64 a, %1, %17;\n\tadd.s64 b, %2, %18;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
               "}"
               :: "r"(d_tmem),
                  "l"(a_desc),
                  "l"(b_desc),
                  "r"(idesc),
                  "r"(acc0),
                  "n"(OA1),
                  "n"(OB1),
                  "n"(OA2),
                  "n"(OB2),
                  "n"(OA3),
                  "n"(OB3),
                  "n"(OA4),
                  "n"(OB4),
                  "n"(OA5),
                  "n"(OB5),
                  "n"(OA6),
                  "n"(OB6),
                  "n"(OA7),
                  "n"(OB7)
               : "memory");
}

template <int OB>
__device__ __forceinline__ void umma_ts_group4(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t acc0) {
  asm volatile("{\n\t.reg .pred p, q, e;\n\t.reg .b32 el;\n\t"
               ".reg .b64 b;\n\t.reg .b32 a;\n\t"
               "elect.sync el|e, 0xffffffff;\n\t"
               "setp.ne.b32 p, %4, 0;\n\t"
               "setp.eq.u32 q, 0, 0;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
               "add.u32 a, %1, 8;\n\tadd.s64 b, %2, %5;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 16;\n\tadd.s64 b, %2, %6;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 24;\n\tadd.s64 b, %2, %7;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "}"
               :: "r"(d_tmem),
                  "r"(a_tmem),
                  "l"(b_desc),
                  "r"(idesc),
                  "r"(acc0),
                  "n"(1 * OB),
                  "n"(2 * OB),
                  "n"(3 * OB)
               : "memory");
}

template <int OB>
__device__ __forceinline__ void umma_ts_group8(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t acc0) {
  asm volatile("{\n\t.reg .pred p, q, e;\n\t.reg .b32 el;\n\t"
               ".reg .b64 b;\n\t.reg .b32 a;\n\t"
               "elect.sync el|e, 0xffffffff;\n\t"
               "setp.ne.b32 p, %4, 0;\n\t"
               "setp.eq.u32 q, 0, 0;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
               "add.u32 a, %1, 8;\n\tadd.s64 b, %2, %5;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 16;\n\tadd.s64 b, %2, %6;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 24;\n\tadd.s64 b, %2, %7;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 32;\n\tadd.s64 b, %2, %8;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 40;\n\tadd.s64 b, %2, %9;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 48;\n\tadd.s64 b, %2, %10;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 56;\n\tadd.s64 b, %2, %11;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "}"
               :: "r"(d_tmem),
                  "r"(a_tmem),
                  "l"(b_desc),
                  "r"(idesc),
                  "r"(acc0),
                  "n"(1 * OB),
                  "n"(2 * OB),
                  "n"(3 * OB),
                  "n"(4 * OB),
                  "n"(5 * OB),
                  "n"(6 * OB),
                  "n"(7 * OB)
               : "memory");
}

// Bounded waits shared by every role; on expiry the CTA is told to stop and
// FM_DEVERR_TIMEOUT is recorded.

// tcgen05.commit from the lane elect.sync picks (the lane that issued the
// MMAs: the whole warp is converged at every call, so the same lane is
// elected each time).
__device__ __forceinline__ void umma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 el;\n\t"
      "elect.sync el|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}


__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}

__device__ __forceinline__ float sum_f32x2(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}

// (lo * s, hi * s) rounded to bf16x2 (lo in the low half) with one packed
// multiply; s2 holds s in both halves.  Bitwise the same as two scalar
// round-to-nearest multiplies followed by the conversion.
__device__ __forceinline__ uint32_t scale_pack_bf16x2(uint32_t lo, uint32_t hi, uint64_t s2) {
  uint32_t packed;
  asm("{\n\t.reg .b64 x, y;\n\t.reg .f32 y0, y1;\n\t"
      "mov.b64 x, {%1, %2};\n\t"
      "mul.rn.f32x2 y, x, %3;\n\t"
      "mov.b64 {y0, y1}, y;\n\t"
      "cvt.rn.bf16x2.f32 %0, y1, y0;\n\t}"
      : "=r"(packed)
      : "r"(lo), "r"(hi), "l"(s2));
  return packed;
}

// Two softmax numerators at once: p_k = 2^(s_k * scale + base) with one
// packed FMA and two ex2; (p0, p1) is added to the packed partial sums and
// returned as bf16x2 (p0 in the low half).
__device__ __forceinline__ uint32_t exp2_pair_bf16(uint32_t s0, uint32_t s1, uint64_t scale2,
                                                   uint64_t base2, uint64_t& sum2) {
  uint32_t packed;
  asm("{\n\t.reg .b64 x, y, p;\n\t.reg .f32 y0, y1, p0, p1;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "fma.rn.f32x2 y, x, %4, %5;\n\t"
      "mov.b64 {y0, y1}, y;\n\t"
      "ex2.approx.ftz.f32 p0, y0;\n\t"
      "ex2.approx.ftz.f32 p1, y1;\n\t"
      "mov.b64 p, {p0, p1};\n\t"
      "add.f32x2 %1, %1, p;\n\t"
      "cvt.rn.bf16x2.f32 %0, p1, p0;\n\t}"
      : "=r"(packed), "+l"(sum2)
      : "r"(s0), "r"(s1), "l"(scale2), "l"(base2));
  return packed;
}

// Sets the CTA's stop flag and the error bit.  The first wait in the grid to
// expire (not one that gave up because another had already failed) also
// records where it was: barrier index, parity, block and warp.  Kept out of
// line: it only runs on the failure path.
__device__ __noinline__ void sync_fail(volatile int* abort, int* err, int bar, uint32_t parity) {
  if (*abort == 0 && atomicCAS(err + 1, 0, 1) == 0) {
    err[2] = bar;
    err[3] = static_cast<int>(parity);
    err[4] = static_cast<int>((blockIdx.x << 8) | (threadIdx.x >> 5));
  }
  *abort = 1;
  atomicOr(err, static_cast<int>(FM_DEVERR_TIMEOUT));
}

struct Sync {
  uint64_t* bars;
  volatile int* abort;
  uint64_t tmo;
  int* err;  // device error word; the four ints after it record the first expiry
  int lane;
  __device__ __forceinline__ void fail(int bar, uint32_t parity) const {
    sync_fail(abort, err, bar, parity);
  }
  // single-thread wait
  __device__ __forceinline__ bool lone(int bar, uint32_t parity) const {
    if (mbar_wait_bounded(&bars[bar], parity, tmo, abort)) return true;
    fail(bar, parity);
    return false;
  }
  // every lane waits; the warp proceeds only if all lanes saw the phase.
  // A phase that has already completed costs one test and one vote.
  __device__ __forceinline__ bool warp(int bar, uint32_t parity) const {
    if (__all_sync(0xffffffffu, mbar_test_wait(&bars[bar], parity))) return true;
    const bool ok = mbar_wait_bounded(&bars[bar], parity, tmo, abort);
    const bool all = __all_sync(0xffffffffu, ok);
    if (!all && lane == 0) fail(bar, parity);
    return all;
  }
};

}  // namespace
}  // namespace fm
