// SwiGLU of the FC1 epilogue, correctly rounded: h = RN_bf16(silu(g) * up)
// with silu(g) = g / (1 + e^-g), g and up BF16 values (the casts of the
// execution specification: u = BF16(FC1 output), h = BF16(SwiGLU), one
// rounding).  Three tiers, each exact where it answers:
//
//   1. Bracket (every element).  e^-g = 2^(g C1) * 2^(g C2), where C1 + C2 =
//      -log2 e and C1 carries 16 significant bits, so that g C1 is exact
//      for a BF16 g; 2^(g C1) comes from the hardware ex2 and the small
//      second factor from its first-order term, 1 + g C2 ln 2.  Then
//      p = RN(RN(g * rcp(1 + E)) * up) with the hardware reciprocal, in
//      packed f32x2 arithmetic.  Wherever the intermediates stay normal, p
//      has a relative error below kSwigluEps - 2^-24 (the hardware terms of
//      the bound are measured exhaustively by the tests), so the BF16
//      roundings of p * (1 - eps) and p * (1 + eps) bracket RN_bf16 of the
//      exact value: when they agree, that is the answer.  Where E overflows
//      or the reciprocal underflows (g < -87) p is zero; zero and results
//      below 2^-100 in magnitude (where a subnormal product would escape the
//      relative bound) go to the next tier; the caller handles all-zero
//      rows (pad rows) itself, whose h is zero.
//   2. Double-float (elements the bracket leaves open, about one in 2000).
//      e^-g by Tang's table-driven method (P. T. P. Tang, ACM TOMS 15(2),
//      1989: g = k ln2/64 + r, e^r by its Taylor polynomial, 2^(j/64) from a
//      table) carried in pairs of floats with Dekker's error-free sums and
//      products (T. J. Dekker, Numer. Math. 18, 1971); the quotient
//      g up / (1 + e^-g) to about 2^-42 relative.  Only a quotient within
//      2^-40 of a BF16 rounding midpoint is left open.
//   3. FP64 (what tier 2 leaves open, and |g| > 64 or extreme products):
//      g / (1 + exp(-g)) * up in double, rounded to BF16 through
//      round-to-odd single precision (which keeps the one rounding exact).
//
// Error bound of tier 1 (relative): ex2 of the exact argument (2^-22.7,
// its maximum measured over every input it sees); the first-order factor
// drops (g C2 ln 2)^2 / 2 <= 9.4e-8 (|g| <= 88.7, beyond which E is
// infinite) and rounds once (2^-24); these errors reach 1 + E scaled by
// E / (1 + E) <= 1.  The reciprocal adds 2^-23.3 (measured), the roundings
// of 1 + E, of g * r and of p three times 2^-24, and the bracket products'
// own rounding 2^-24: 6.35e-7 in all, under kSwigluEps = 7.15e-7.
#pragma once

#include "common.cuh"
#include "exp_table.cuh"

namespace moe {

// -log2 e = kNegLog2eHi + C2 with kNegLog2eHi = -47274 / 2^15 (16
// significant bits); kNegLog2eLoLn2 = RN(C2 ln 2)
constexpr float kNegLog2eHi = -0x1.7154p+0f;
constexpr float kNegLog2eLoLn2 = -0x1.480fb6p-18f;
// tier-1 half-width of the bracket: the error bound of p (see above) plus
// 2^-24 for the rounding of the bracket products, a multiple of 2^-23 so
// that 1 -+ eps are exact floats
constexpr float kSwigluEps = 0x1.8p-21f;              // 6 * 2^-23 = 7.15e-7
constexpr uint32_t kSwigluTinyBits = 0x0D80u;         // BF16 pattern of 2^-100

__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint64_t f32x2_bits(float lo, float hi) { return f32x2_pack(lo, hi); }
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Packed BF16x2 of a pair (first element in the low half), nearest even.
__device__ __forceinline__ uint32_t bf16x2_of(uint64_t v) {
  float lo, hi;
  f32x2_unpack(v, lo, hi);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// Tier 1 for one packed pair of gate values and one of up values: the BF16
// pair of p and a nonzero `open` when the bracket leaves a half undecided.
__device__ __forceinline__ uint32_t swiglu_pair_fast(uint32_t gw, uint32_t uw, uint32_t& open) {
  const uint64_t z = f32x2_bits(bf16_lo(gw), bf16_hi(gw));
  float t0, t1;
  f32x2_unpack(mul_f32x2(z, f32x2_bits(kNegLog2eHi, kNegLog2eHi)), t0, t1);  // exact
  const uint64_t dl = mul_f32x2(z, f32x2_bits(kNegLog2eLoLn2, kNegLog2eLoLn2));
  uint64_t E = f32x2_bits(ex2_ftz(t0), ex2_ftz(t1));
  E = fma_f32x2(E, dl, E);  // E (1 + g C2 ln 2)
  float d0, d1;
  f32x2_unpack(add_f32x2(E, f32x2_bits(1.0f, 1.0f)), d0, d1);
  const uint64_t s = mul_f32x2(z, f32x2_bits(rcp_ftz(d0), rcp_ftz(d1)));
  const uint64_t p = mul_f32x2(s, f32x2_bits(bf16_lo(uw), bf16_hi(uw)));
  const uint32_t lo = bf16x2_of(mul_f32x2(p, f32x2_bits(1.0f - kSwigluEps, 1.0f - kSwigluEps)));
  const uint32_t hi = bf16x2_of(mul_f32x2(p, f32x2_bits(1.0f + kSwigluEps, 1.0f + kSwigluEps)));
  open = lo ^ hi;
  return lo;
}

// ---- tier 3 ----
__device__ __noinline__ uint32_t swiglu_bf16_f64(float g, float up) {
  const double gd = (double)g;
  const double p = gd / (1.0 + exp(-gd)) * (double)up;
  float f = __double2float_rz(p);
  if ((double)f != p) f = __uint_as_float(__float_as_uint(f) | 1u);  // round to odd
  return f32_to_bf16_bits(f);
}

// ---- tier 2 ----
// Error-free transformations (Dekker): s + e == a + b exactly.
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {  // |a| >= |b|
  s = __fadd_rn(a, b);
  e = __fadd_rn(b, -__fadd_rn(s, -a));
}
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fadd_rn(s, -a);
  e = __fadd_rn(__fadd_rn(a, -__fadd_rn(s, -bb)), __fadd_rn(b, -bb));
}

// RN_bf16(g * up / (1 + e^-g)) for finite BF16 values g, up.
__device__ __noinline__ uint32_t swiglu_bf16_exact(float g, float up) {
  const float Z = __fmul_rn(g, up);  // exact: two 8-bit significands
  const float aZ = fabsf(Z);
  if (!(fabsf(g) <= 64.0f) || !(aZ >= 0x1p-100f) || !(aZ <= 0x1p100f)) return swiglu_bf16_f64(g, up);
  // e^x with x = -g = k ln2/64 + r: k = rint(x 64/ln2) (|k| < 2^13), r in
  // pairs of floats; k * kLn2_64_1 is exact (11 + 13 bits), and so is r1
  const float x = -g;
  const float kf = rintf(__fmul_rn(x, kInvLn2_64));
  const int k = (int)kf;
  const int j = k & 63, m = k >> 6;  // k = 64 m + j
  const float r1 = __fmaf_rn(-kf, kLn2_64_1, x);
  const float c2h = __fmul_rn(kf, kLn2_64_2);
  const float c2l = __fmaf_rn(kf, kLn2_64_2, -c2h);
  float rh, re;
  two_sum(r1, -c2h, rh, re);
  const float rl = __fadd_rn(__fadd_rn(re, -c2l), __fmul_rn(-kf, kLn2_64_3));
  // e^r = 1 + r + r^2/2 + r^3/6 + r^4/24 + r^5/120 for |r| <= 0.0055 (the
  // next term is below 2^-54); r^2 exactly as sq_h + sq_l
  const float sq_h = __fmul_rn(rh, rh);
  const float sq_l = __fmaf_rn(rh, rh, -sq_h);
  float c = __fmaf_rn(rh, 1.0f / 120.0f, 1.0f / 24.0f);
  c = __fmaf_rn(rh, c, 1.0f / 6.0f);
  const float P = __fmul_rn(c, __fmul_rn(sq_h, rh));
  const float R = __fadd_rn(__fadd_rn(__fmaf_rn(rh, rl, rl), __fmul_rn(sq_l, 0.5f)), P);
  float ah, al, bh, bl, Sh, Sl;
  fast_two_sum(1.0f, rh, ah, al);
  fast_two_sum(ah, __fmul_rn(sq_h, 0.5f), bh, bl);
  fast_two_sum(bh, __fadd_rn(__fadd_rn(al, bl), R), Sh, Sl);
  // E = 2^m * 2^(j/64) * e^r
  const float Th = kExp2Tab[j][0], Tl = kExp2Tab[j][1];
  const float Ph = __fmul_rn(Th, Sh);
  const float Pl = __fadd_rn(__fmaf_rn(Th, Sh, -Ph), __fmaf_rn(Th, Sl, __fmul_rn(Tl, Sh)));
  const float sc = __uint_as_float((uint32_t)(127 + m) << 23);  // 2^m, |m| <= 93
  const float Eh = __fmul_rn(Ph, sc), El = __fmul_rn(Pl, sc);
  // D = 1 + E, Q = Z / D
  float Dh, De;
  two_sum(1.0f, Eh, Dh, De);
  const float Dl = __fadd_rn(De, El);
  const float rD = rcp_ftz(Dh);
  const float qh = __fmul_rn(Z, rD);
  if (!(fabsf(qh) >= 0x1p-110f)) return swiglu_bf16_f64(g, up);
  const float e1 = __fmaf_rn(-qh, Dh, Z);
  const float e2 = __fmaf_rn(-qh, Dl, e1);
  const float ql = __fmul_rn(e2, rD);
  float Qh, Ql;
  fast_two_sum(qh, ql, Qh, Ql);
  const uint32_t qb = __float_as_uint(Qh);
  // Q lies within half a float ulp (+ 2^-42 Q) of Qh; only when Qh is itself
  // a BF16 midpoint does the sign of the remainder decide
  if ((qb & 0xFFFFu) != 0x8000u) return f32_to_bf16_bits(Qh);
  if (!(fabsf(Ql) > fabsf(Qh) * 0x1p-40f)) return swiglu_bf16_f64(g, up);
  const bool away = (Ql > 0.0f) == (Qh > 0.0f);
  return ((qb >> 16) + (away ? 1u : 0u)) & 0xFFFFu;
}

// True when the bracket cannot decide half `sh` (0 or 16) of a pair: open,
// or a result below 2^-100 in magnitude (zero included).
__device__ __forceinline__ bool swiglu_half_open(uint32_t lo, uint32_t open, int sh) {
  return ((open >> sh) & 0xFFFFu) != 0u || ((lo >> sh) & 0x7FFFu) < kSwigluTinyBits;
}

// The exact pair: each half from the bracket where it decides, else from
// tier 2.
__device__ __forceinline__ uint32_t swiglu_pair_fix(uint32_t gw, uint32_t uw) {
  uint32_t open;
  const uint32_t lo = swiglu_pair_fast(gw, uw, open);
  uint32_t r0 = lo & 0xFFFFu, r1 = lo >> 16;
  if (swiglu_half_open(lo, open, 0)) r0 = swiglu_bf16_exact(bf16_lo(gw), bf16_lo(uw));
  if (swiglu_half_open(lo, open, 16)) r1 = swiglu_bf16_exact(bf16_hi(gw), bf16_hi(uw));
  return r0 | (r1 << 16);
}

// The exact pair, out of line: for rare fixes made away from the hot loop.
__device__ __noinline__ uint32_t swiglu_pair_exact(uint32_t gw, uint32_t uw) { return swiglu_pair_fix(gw, uw); }

// The 16 inputs of a group and its 8 result words, passed by value so that
// the rare path below takes its arguments in registers.
struct Swiglu16In {
  uint32_t g[8], u[8];
};
struct Swiglu16Out {
  uint32_t h[8];
};

// Rare path of swiglu16, out of line (its code and register needs stay out
// of the caller's loop): the pairs whose bit is set in `mask` are recomputed
// exactly.
__device__ __noinline__ Swiglu16Out swiglu16_rare(const Swiglu16In in, Swiglu16Out out, uint32_t mask) {
#pragma unroll
  for (int w = 0; w < 8; ++w)
    if (mask & (1u << w)) out.h[w] = swiglu_pair_fix(in.g[w], in.u[w]);
  return out;
}

// Bit of the swiglu16_fast mask that sends every pair of the group to the
// exact path (a result below 2^-100, or zero, somewhere in it).
constexpr uint32_t kSwigluAll = 0x100u;

// Tier 1 of 16 elements (8 packed gate words, 8 packed up words): h[w] is
// the bracket's BF16 pair, exact unless bit w of the returned mask is set
// (kSwigluAll: no pair may be trusted); hmax gets the largest |h| as packed
// magnitude bits.
__device__ __forceinline__ uint32_t swiglu16_fast(const uint32_t (&gw)[8], const uint32_t (&uw)[8], uint32_t (&h)[8],
                                                  uint32_t& hmax) {
  uint32_t mask = 0, hmin = 0x7FFF7FFFu;
  hmax = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t open;
    h[w] = swiglu_pair_fast(gw[w], uw[w], open);
    mask |= (open != 0u ? 1u : 0u) << w;
    const uint32_t m = h[w] & 0x7FFF7FFFu;
    hmax = __vmaxu2(hmax, m);
    hmin = __vminu2(hmin, m);
  }
  if (min(hmin & 0xFFFFu, hmin >> 16) < kSwigluTinyBits) mask = kSwigluAll | 0xFFu;
  return mask;
}

// The pairs of `mask` (bits 0-7) recomputed exactly, and hmax updated.
__device__ __forceinline__ void swiglu16_fix(const uint32_t (&gw)[8], const uint32_t (&uw)[8], uint32_t (&h)[8],
                                             uint32_t mask, uint32_t& hmax) {
  Swiglu16In in;
  Swiglu16Out o;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    in.g[w] = gw[w];
    in.u[w] = uw[w];
    o.h[w] = h[w];
  }
  o = swiglu16_rare(in, o, mask & 0xFFu);
  hmax = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    h[w] = o.h[w];
    hmax = __vmaxu2(hmax, h[w] & 0x7FFF7FFFu);
  }
}

// h of 16 elements into 8 packed BF16 words, exact; returns the largest |h|
// of the 16 as packed magnitude bits (the larger of its two halves is the
// maximum).
__device__ __forceinline__ uint32_t swiglu16(const uint32_t (&gw)[8], const uint32_t (&uw)[8], uint32_t (&h)[8]) {
  uint32_t hmax;
  const uint32_t mask = swiglu16_fast(gw, uw, h, hmax);
  if (mask) swiglu16_fix(gw, uw, h, mask, hmax);
  return hmax;
}

}  // namespace moe
