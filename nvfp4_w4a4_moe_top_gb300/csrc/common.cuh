// Device helpers shared by the kernels of libmoe_nvfp4.so (sm_103a only).
//
// Codecs here are bit-level encoders of the NVFP4 element/scale formats
// (E2M1 elements, E4M3 block scales: miniTE Technical Report section 2.2 and
// section 5.1 equation).  They are written for the GPU from the format
// definitions and share nothing with the CPU oracle; parity tests compare the
// two over every float input.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <stdint.h>

#include "../../include/moe_nvfp4.h"

namespace moe {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// scalar helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// FP32 -> BF16 bits, round to nearest even (hardware cvt.rn.bf16.f32).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// Two FP32 -> packed BF16x2 (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
}

// E2M1 encoder, round to nearest with ties to the even code, saturating at 6.
// The code of |q| is the number of decision boundaries it has crossed; at
// 0.25, 1.25, 2.5 and 5 the tie stays on the lower (even) code, at 0.75,
// 1.75 and 3.5 it moves up to the even code.  Sign bit = sign bit of q.
__device__ __forceinline__ uint32_t e2m1_encode(float q) {
  const float a = fabsf(q);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) +
               (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
  return c | ((__float_as_uint(q) >> 28) & 8u);
}

// E4M3 (OCP "FN") decoder for a non-negative scale byte 0x00..0x7E.
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  if (e == 0) return (float)m * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// E4M3 encoder for t >= 0: round to nearest even, saturate at 448 (0x7E).
// Below 2^-6 the grid is m * 2^-9 (m = 0..8), so the code is rint(t * 512);
// above it, rounding the float's exponent+mantissa field to 3 mantissa bits
// with an integer round-half-even carries into the exponent as needed, and
// the biased exponents differ by 127 - 7.
__device__ __forceinline__ uint32_t e4m3_encode(float t) {
  if (!(t < 448.0f)) return 0x7Eu;  // also +inf (NaN is flagged by callers)
  if (t < 0.015625f) return (uint32_t)__float2int_rn(t * 512.0f);
  const uint32_t u = __float_as_uint(t);
  const uint32_t r = (u + 0x7FFFFu + ((u >> 20) & 1u)) >> 20;
  return r - (120u << 3);
}

// The hardware E4M3 conversion (round to nearest even, saturating; equal to
// e4m3_encode on every non-negative finite float, checked exhaustively by the
// tests) of two values at once: lo's code in bits 0-7, hi's in bits 8-15.
__device__ __forceinline__ uint32_t e4m3x2_hw(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(lo), "f"(hi));
  return r;
}
// The hardware E4M3 decode of a code (0..0x7E), through half precision
// (exact: every E4M3 value is a half).
__device__ __forceinline__ float e4m3_decode_hw(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)code));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}
// Reciprocal of a row's block-scale divisor den = 6 g for block_scale_code:
// RN(1/den), or 0 where den < 2^-120 (the exact division serves).
__device__ __forceinline__ float block_scale_rden(float den) {
  return den >= 7.52316384526264e-37f ? __frcp_rn(den) : 0.0f;
}
// E4M3 block scale s = E4M3(RN(a_b / den)) from the block's amax a_b >= 0.
// With rden = RN(1/den), q = RN(a_b * rden) is within 2 * 2^-24 of a_b/den,
// so the products RN(q (1 -+ 2^-21)) bracket RN(a_b / den); the encoder is
// monotone, so when their codes agree that is the code (values too small
// for a nonzero code, or large enough to saturate, agree on both sides).
// Otherwise (a quotient within about 2^-21 of an E4M3 rounding boundary)
// the code is taken from the correctly rounded division.
__device__ __forceinline__ uint32_t block_scale_code(float ab, float den, float rden) {
  if (rden != 0.0f) {
    const float q = __fmul_rn(ab, rden);
    const uint32_t c2 = e4m3x2_hw(__fmul_rn(q, 0.99999952316284180f), __fmul_rn(q, 1.00000047683715820f));
    if ((c2 & 0xFFu) == (c2 >> 8)) return c2 & 0xFFu;
  }
  return e4m3x2_hw(__fdiv_rn(ab, den), 0.0f) & 0xFFu;
}

// Byte offset of logical block scale (row, col) of a [rows][K/16] matrix in
// the 128x4 tile layout (tiles row-group-major, 512 bytes each).
__device__ __forceinline__ int64_t sf_tile_offset(int64_t row, int col, int kgroups) {
  return ((row >> 7) * kgroups + (col >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (col & 3);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ void set_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ bool is_finite_f32(float v) { return (__float_as_uint(v) & 0x7F800000u) != 0x7F800000u; }
__device__ __forceinline__ bool bf16x2_finite(uint32_t p) {
  return ((p & 0x7F80u) != 0x7F80u) && ((p & 0x7F800000u) != 0x7F800000u);
}

// Largest magnitude among 16 BF16 values (two uint4), as the BF16 bit
// pattern with the sign cleared.  For finite values and +inf the integer
// order of these patterns is the order of the magnitudes, and any NaN
// compares above +inf (0x7F80), so a result >= 0x7F80 means a non-finite
// value is present.
__device__ __forceinline__ uint32_t absmax_bits16(const uint4 p0, const uint4 p1) {
  uint32_t m = __vmaxu2(p0.x & 0x7FFF7FFFu, p0.y & 0x7FFF7FFFu);
  m = __vmaxu2(m, __vmaxu2(p0.z & 0x7FFF7FFFu, p0.w & 0x7FFF7FFFu));
  m = __vmaxu2(m, __vmaxu2(p1.x & 0x7FFF7FFFu, p1.y & 0x7FFF7FFFu));
  m = __vmaxu2(m, __vmaxu2(p1.z & 0x7FFF7FFFu, p1.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}

// Largest magnitude among a lane's BF16 values with NaNs left out (the
// maximum fmaxf would give), as magnitude bits.
template <int NG>
__device__ __forceinline__ uint32_t absmax_bits_no_nan(const uint4 (&v)[NG][4]) {
  uint32_t fm = 0;
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w[4] = {v[g][q].x, v[g][q].y, v[g][q].z, v[g][q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0x7FFFu, hi = (w[i] >> 16) & 0x7FFFu;
        if (lo <= 0x7F80u) fm = max(fm, lo);
        if (hi <= 0x7F80u) fm = max(fm, hi);
      }
    }
  return fm;
}

// Eight FP32 -> eight E2M1 codes with the hardware conversion (nearest
// even, saturating; element 0 in the low nibble).  Its equality with
// e2m1_encode over every float is part of the codec parity test.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Two FP32 values in one 64-bit register (first argument in the low half),
// the operand form of the packed f32x2 arithmetic.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// Element-wise product of two FP32 pairs, each rounded to nearest even: the
// same two results as two __fmul_rn, in one instruction.
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// e2m1x8 of four FP32 pairs (pair i holds elements 2i, 2i+1).
__device__ __forceinline__ uint32_t e2m1x8_pairs(const uint64_t (&p)[4]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .f32 x0, x1, x2, x3, x4, x5, x6, x7;\n\t"
      "mov.b64 {x0, x1}, %1;\n\t"
      "mov.b64 {x2, x3}, %2;\n\t"
      "mov.b64 {x4, x5}, %3;\n\t"
      "mov.b64 {x6, x7}, %4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, x1, x0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, x3, x2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, x5, x4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, x7, x6;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "l"(p[0]), "l"(p[1]), "l"(p[2]), "l"(p[3]));
  return r;
}

// Element-wise fused multiply-add of two FP32 pairs, a * b + c rounded once
// to nearest even per element: the same two results as two fmaf.
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Exact E2M1 codes with no fallback path: RN(v / S) by Markstein's
// correctly rounded division (P. W. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34,
// 1990; in FMA form also in Cornea, Harrison and Tang, "Scientific
// Computing on Itanium-based Systems", 2002):
//   y  = RN(1/S)                     the IEEE reciprocal, once per block
//   q0 = RN(v y)                     within 1.5 ulp of v/S
//   q1 = RN(q0 + RN(v - S q0) y)     within 0.5 ulp + 2^-45 relative: faithful
//   q2 = RN(q1 + (v - S q1) y)       Markstein: with y the correctly rounded
//                                    reciprocal and q1 faithful, the residual
//                                    is exact and q2 = RN(v / S).
// Domain: 2^-96 <= S <= 2^120 and |v| <= 16 S.  The residual of a quotient
// of at least 2^-3 is then a multiple of 2^-145 or coarser, so it stays
// exact; smaller quotients encode to zero whatever their last bits.  y is
// normal and no step overflows.  The quantisers meet |v| <= 16 S by
// construction: a block's scale is E4M3(RN(a_b / (6 g))) of the block's own
// largest magnitude a_b, at most a factor 1.5 below a_b / (6 g) (the E4M3
// subnormal step), so |v| / S <= 9.  The sign of v is ORed into the quotient,
// which keeps the sign of a zero v.
//
// S lies in the domain through a power-of-two factor f per row: v and S are
// both multiplied by f, which leaves v / S unchanged.  For a row with outer
// scale g > 0 every block scale is RN(g s_b) with s_b a nonzero E4M3 value
// (2^-9 .. 448); f = 2^64 below g = 2^-87, 2^-64 above g = 2^111, else 1,
// puts g f in [2^-87, 2^111] and so S f in [2^-96, 2^120].  S f is exact;
// v f is exact except, for f = 2^-64, below |v| = 2^-62, where in such a row
// the quotient is under 2^-164 and encodes to zero (with v's sign) either
// way.
__device__ __forceinline__ float e2m1_row_factor(float g) {
  return g < 0x1p-87f ? 0x1p64f : (g > 0x1p111f ? 0x1p-64f : 1.0f);
}
struct E2m1Div {
  uint64_t f, nS, y;  // (f, f), (-S f, -S f) and (RN(1/(S f)), RN(1/(S f)))
};
__device__ __forceinline__ E2m1Div e2m1_div(float S, float f) {
  E2m1Div d;
  const float Sf = S * f;
  const float y = __frcp_rn(Sf);
  d.f = f32x2_pack(f, f);
  d.nS = f32x2_pack(-Sf, -Sf);
  d.y = f32x2_pack(y, y);
  return d;
}
// SCALED false: the caller guarantees f = 1 (the row scale within
// [2^-87, 2^111], e2m1_div_row_scale_ok), and the multiply by f is left out.
template <bool SCALED = true>
__device__ __forceinline__ uint32_t e2m1_codes8_div(const uint32_t (&w)[4], const E2m1Div& d) {
  uint64_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t v0 = f32x2_pack(bf16_lo(w[i]), bf16_hi(w[i]));
    const uint64_t v = SCALED ? mul_f32x2(v0, d.f) : v0;
    const uint64_t q0 = mul_f32x2(v, d.y);
    const uint64_t q1 = fma_f32x2(fma_f32x2(d.nS, q0, v), d.y, q0);
    const uint64_t q2 = fma_f32x2(fma_f32x2(d.nS, q1, v), d.y, q1);
    const uint64_t sign = ((uint64_t)(w[i] & 0x80000000u) << 32) | (uint64_t)((w[i] & 0x8000u) << 16);
    q[i] = q2 | sign;
  }
  return e2m1x8_pairs(q);
}
// Codes of 16 BF16 values (two groups of 4 packed words) for a block scale
// S > 0 of a row with factor f = e2m1_row_factor(g): Q_E2M1(RN(v / S)).
// SCALED as e2m1_codes8_div.
template <bool SCALED = true>
__device__ __forceinline__ uint2 e2m1_codes16_div(const uint32_t (&w0)[4], const uint32_t (&w1)[4], float S, float f) {
  const E2m1Div d = e2m1_div(S, f);
  return make_uint2(e2m1_codes8_div<SCALED>(w0, d), e2m1_codes8_div<SCALED>(w1, d));
}
// The row scales whose row factor is 1: g in [2^-87, 2^111].
__device__ __forceinline__ bool e2m1_div_row_scale_ok(float g) { return g >= 0x1p-87f && g <= 0x1p111f; }

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, TMA, tcgen05
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Wait for the phase of the given parity, suspending the thread for up to
// 65536 ns (it resumes as soon as the phase completes); false if the time
// limit passed first.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(65536u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// 2D tiled TMA load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Four rows y0..y3 of a 2-D tensor (the map's box is one row high) into
// four consecutive rows of shared memory, swizzled as rows of one box.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0, int y1, int y2, int y3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
      : "memory");
}
// L2 cache policy for data other threads read again soon (evict last).
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// L2 cache policy for data no thread reads again soon (evict first).
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 16-byte global store with an L2 cache policy.
__device__ __forceinline__ void st_global_hint(void* p, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(policy)
               : "memory");
}
// Drops the 128-byte L2 line holding p without writing it back (its data
// becomes undefined): for scratch that will be rewritten before it is read.
__device__ __forceinline__ void discard_l2_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}
// Contiguous bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// 16-byte asynchronous copy global -> shared (zero-filled when !valid: src
// is then not read), and its group commit / wait.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Shared -> global tensor store of one box, in this thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The same with an L2 cache policy for the written lines.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src, int x, int y, uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src), "l"(policy)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's bulk stores: their shared-memory sources read (read0), or
// complete (wait0).
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic shared-memory writes before later async-proxy
// (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand staged by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;             // leading byte offset (unused when swizzled), 16 B
  d |= (uint64_t)(1024u >> 4) << 32;   // stride byte offset: next 8-row group
  d |= (uint64_t)1u << 46;             // descriptor version for tcgen05
  d |= (uint64_t)2u << 61;             // 128-byte swizzle
  return d;
}
// Descriptor of a 32-row x 16-byte block-scale tile (no swizzle, rows
// contiguous, 8-row groups 128 bytes apart) for tcgen05.cp 32x128b.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  return d;
}

}  // namespace moe
