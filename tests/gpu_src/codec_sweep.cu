// Test-only sweep of the library's device codecs over every float input.
// Builds into tests/_build/libcodec_sweep.so; the parity test compares the
// results with the CPU oracle.
#include "../../nvfp4_w4a4_moe_top_gb300/csrc/common.cuh"

// For every non-negative finite bit pattern p: the code of p, checked for
// monotonicity against p - 1, and the first pattern of each code.
__global__ void e4m3_sweep(unsigned int* first, unsigned long long* viol) {
  const unsigned int stride = gridDim.x * blockDim.x;
  unsigned long long bad = 0;
  for (unsigned int p = 1u + blockIdx.x * blockDim.x + threadIdx.x; p < 0x7F800000u; p += stride) {
    const unsigned int c = moe::e4m3_encode(__uint_as_float(p));
    const unsigned int c0 = moe::e4m3_encode(__uint_as_float(p - 1u));
    if (c < c0 || c > 0x7Eu) ++bad;
    if (c != c0) atomicMin(&first[c & 0x7F], p);
  }
  if (bad) atomicAdd(viol, bad);
}

// Same for the E2M1 magnitude codes, plus the sign rule code(-q) = code(q) | 8.
__global__ void e2m1_sweep(unsigned int* first, unsigned long long* viol, unsigned long long* sign_viol) {
  const unsigned int stride = gridDim.x * blockDim.x;
  unsigned long long bad = 0, sbad = 0;
  for (unsigned int p = 1u + blockIdx.x * blockDim.x + threadIdx.x; p < 0x7F800000u; p += stride) {
    const unsigned int c = moe::e2m1_encode(__uint_as_float(p));
    const unsigned int c0 = moe::e2m1_encode(__uint_as_float(p - 1u));
    if (c < c0 || c > 7u) ++bad;
    if (c != c0) atomicMin(&first[c & 7], p);
    if (moe::e2m1_encode(__uint_as_float(p | 0x80000000u)) != (c | 8u)) ++sbad;
  }
  if (bad) atomicAdd(viol, bad);
  if (sbad) atomicAdd(sign_viol, sbad);
}

// The hardware conversion used by the quantisers against the reference
// encoder, over every finite float of either sign.
__global__ void e2m1_cvt_sweep(unsigned long long* viol) {
  const unsigned int stride = gridDim.x * blockDim.x;
  unsigned long long bad = 0;
  for (unsigned int p = blockIdx.x * blockDim.x + threadIdx.x; p < 0x7F800000u; p += stride) {
    for (unsigned int sgn = 0; sgn < 2; ++sgn) {
      const float v = __uint_as_float(p | (sgn << 31));
      const float eight[8] = {v, v, v, v, v, v, v, v};
      const unsigned int c = moe::e2m1_encode(v);
      if (moe::e2m1x8(eight) != c * 0x11111111u) ++bad;
    }
  }
  if (bad) atomicAdd(viol, bad);
}

__global__ void e4m3_decode_all(float* out) {
  const int c = threadIdx.x;
  if (c < 0x7F) out[c] = moe::e4m3_decode(c);
}

extern "C" int run_cvt_sweep(unsigned long long* viol) {
  unsigned long long* d_v;
  if (cudaMalloc(&d_v, 8)) return -1;
  cudaMemset(d_v, 0, 8);
  e2m1_cvt_sweep<<<152 * 8, 256>>>(d_v);
  const int rc = cudaMemcpy(viol, d_v, 8, cudaMemcpyDeviceToHost) ? -2 : 0;
  cudaFree(d_v);
  return rc;
}

extern "C" int run_codec_sweeps(unsigned int* e4m3_first, unsigned long long* e4m3_viol, unsigned int* e2m1_first,
                                unsigned long long* e2m1_viol, unsigned long long* e2m1_sign_viol, float* e4m3_values) {
  unsigned int *d_f4, *d_f2;
  unsigned long long* d_v;
  float* d_val;
  if (cudaMalloc(&d_f4, 128 * 4) || cudaMalloc(&d_f2, 8 * 4) || cudaMalloc(&d_v, 3 * 8) || cudaMalloc(&d_val, 128 * 4))
    return -1;
  cudaMemset(d_f4, 0xFF, 128 * 4);
  cudaMemset(d_f2, 0xFF, 8 * 4);
  cudaMemset(d_v, 0, 3 * 8);
  e4m3_sweep<<<152 * 8, 256>>>(d_f4, d_v);
  e2m1_sweep<<<152 * 8, 256>>>(d_f2, d_v + 1, d_v + 2);
  e4m3_decode_all<<<1, 128>>>(d_val);
  unsigned long long v[3];
  int rc = 0;
  if (cudaMemcpy(e4m3_first, d_f4, 128 * 4, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(e2m1_first, d_f2, 8 * 4, cudaMemcpyDeviceToHost) || cudaMemcpy(v, d_v, 3 * 8, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(e4m3_values, d_val, 127 * 4, cudaMemcpyDeviceToHost))
    rc = -2;
  *e4m3_viol = v[0];
  *e2m1_viol = v[1];
  *e2m1_sign_viol = v[2];
  cudaFree(d_f4); cudaFree(d_f2); cudaFree(d_v); cudaFree(d_val);
  return rc;
}

// ---- the quantisers' fast paths against their exact definitions ----

// The hardware E4M3 conversion of two values at once against e4m3_encode on
// every non-negative finite float (in either position), and the hardware
// decode against e4m3_decode on every code.
__global__ void e4m3_hw_sweep(unsigned long long* viol) {
  const unsigned int stride = gridDim.x * blockDim.x;
  unsigned long long bad = 0;
  for (unsigned int p = blockIdx.x * blockDim.x + threadIdx.x; p < 0x7F800000u; p += stride) {
    const float t = __uint_as_float(p);
    const unsigned int c = moe::e4m3_encode(t);
    if (moe::e4m3x2_hw(t, 0.0f) != c || moe::e4m3x2_hw(0.0f, t) != (c << 8)) ++bad;
  }
  if (blockIdx.x == 0 && threadIdx.x < 0x7F)
    if (__float_as_uint(moe::e4m3_decode_hw(threadIdx.x)) != __float_as_uint(moe::e4m3_decode(threadIdx.x))) ++bad;
  if (bad) atomicAdd(viol, bad);
}

// A positive float spread over [2^-126, 2^126) in exponent, from an index.
__device__ __forceinline__ float spread(unsigned int i) {
  const unsigned int e = 1u + (i % 252u);                    // biased exponents 1 .. 252
  const unsigned int m = (i * 2654435761u) & 0x007FFFFFu;    // mixed mantissa
  return __uint_as_float((e << 23) | m);
}

// block_scale_code against the exact definition E4M3(RN(a / den)) for every
// finite non-negative BF16 amax a and 65536 divisors den spread over the
// float range (including den below 2^-120, where the exact path serves).
__global__ void block_scale_sweep(unsigned long long* viol) {
  const float den = spread(blockIdx.x * blockDim.x + threadIdx.x);
  const float rden = moe::block_scale_rden(den);
  unsigned long long bad = 0;
  for (unsigned int b = 0; b < 0x7F80u; ++b) {
    const float a = __uint_as_float(b << 16);
    if (moe::block_scale_code(a, den, rden) != moe::e4m3_encode(__fdiv_rn(a, den))) ++bad;
  }
  if (bad) atomicAdd(viol, bad);
}

// The quantisers' E2M1 encoder (e2m1_codes16_div with the row factor of
// e2m1_row_factor) against the exact definition Q(RN(v / S)) for every
// finite BF16 v (either sign) with |v| <= 16 S (other v are replaced by
// zero; the quantisers never exceed 9 S) and 65536 scales S spread over the
// whole float range, each as the block scale of rows with outer scale
// g = S / s_b for s_b = 256, 1 and 2^-9 (the factor follows g).
__global__ void e2m1_row_sweep(unsigned long long* viol) {
  const float S = spread(blockIdx.x * blockDim.x + threadIdx.x);
  unsigned long long bad = 0;
  for (int k = 0; k < 3; ++k) {
    const float g = S * (k == 0 ? 0x1p-8f : (k == 1 ? 1.0f : 0x1p9f));
    const float f = moe::e2m1_row_factor(g);
    for (unsigned int b0 = 0; b0 < 0x10000u; b0 += 16) {
      uint32_t w[2][4];
      float q[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t lo = b0 + 8 * h + 2 * i, hi = lo + 1;
          if ((lo & 0x7F80u) == 0x7F80u || fabsf(__uint_as_float(lo << 16)) > 16.0f * S) lo = 0;
          if ((hi & 0x7F80u) == 0x7F80u || fabsf(__uint_as_float(hi << 16)) > 16.0f * S) hi = 0;
          w[h][i] = lo | (hi << 16);
          q[h][2 * i] = __fdiv_rn(moe::bf16_lo(w[h][i]), S);
          q[h][2 * i + 1] = __fdiv_rn(moe::bf16_hi(w[h][i]), S);
        }
      const uint2 c = moe::e2m1_codes16_div(w[0], w[1], S, f);
      if (c.x != moe::e2m1x8(q[0]) || c.y != moe::e2m1x8(q[1])) ++bad;
    }
  }
  if (bad) atomicAdd(viol, bad);
}

// The E2M1 codes of 8 values through Markstein's division (e2m1_codes8_div)
// against the exact definition Q(RN(v / S)) for every finite BF16 v (either
// sign) within the division's domain |v| <= 16 S, over scales S in
// [2^-96, 2^120]: threads 0 .. 215 take S with an all-ones significand at
// each exponent of that range, the others S spread over it.  `checked`
// counts the (v, S) pairs compared.
__device__ __forceinline__ float spread_div_domain(unsigned int i) {
  if (i < 216u) return __uint_as_float(((31u + i) << 23) | 0x007FFFFFu);  // biased exponents 31 .. 246
  const unsigned int e = 31u + (i % 216u);
  const unsigned int m = (i * 2654435761u) & 0x007FFFFFu;
  return __uint_as_float((e << 23) | m);
}
__global__ void e2m1_div_sweep(unsigned long long* viol, unsigned long long* checked) {
  const float S = spread_div_domain(blockIdx.x * blockDim.x + threadIdx.x);
  const moe::E2m1Div dv = moe::e2m1_div(S, 1.0f);
  const bool in = S >= 0x1p-96f && S <= 0x1p120f;
  const float lim = 16.0f * S;
  unsigned long long bad = 0, n = 0;
  for (unsigned int b0 = 0; b0 < 0x10000u; b0 += 8) {
    uint32_t w[4];
    float q[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo = b0 + 2 * i, hi = b0 + 2 * i + 1;
      // non-finite patterns and values outside the domain: zero instead
      if ((lo & 0x7F80u) == 0x7F80u || fabsf(__uint_as_float(lo << 16)) > lim) lo = 0;
      else ++n;
      if ((hi & 0x7F80u) == 0x7F80u || fabsf(__uint_as_float(hi << 16)) > lim) hi = 0;
      else ++n;
      w[i] = lo | (hi << 16);
      q[2 * i] = __fdiv_rn(moe::bf16_lo(w[i]), S);
      q[2 * i + 1] = __fdiv_rn(moe::bf16_hi(w[i]), S);
    }
    if (!in || moe::e2m1_codes8_div(w, dv) != moe::e2m1x8(q)) ++bad;
  }
  if (bad) atomicAdd(viol, bad);
  atomicAdd(checked, n);
}

extern "C" int run_div_sweep(unsigned long long* viol, unsigned long long* checked) {
  unsigned long long* d_v;
  if (cudaMalloc(&d_v, 2 * 8)) return -1;
  cudaMemset(d_v, 0, 2 * 8);
  e2m1_div_sweep<<<256, 256>>>(d_v, d_v + 1);
  unsigned long long v[2];
  const int rc = cudaMemcpy(v, d_v, 2 * 8, cudaMemcpyDeviceToHost) ? -2 : 0;
  *viol = v[0];
  *checked = v[1];
  cudaFree(d_v);
  return rc;
}

extern "C" int run_fast_path_sweeps(unsigned long long* viol_e4m3, unsigned long long* viol_scale,
                                    unsigned long long* viol_e2m1) {
  unsigned long long* d_v;
  if (cudaMalloc(&d_v, 3 * 8)) return -1;
  cudaMemset(d_v, 0, 3 * 8);
  e4m3_hw_sweep<<<152 * 8, 256>>>(d_v);
  block_scale_sweep<<<256, 256>>>(d_v + 1);
  e2m1_row_sweep<<<256, 256>>>(d_v + 2);
  unsigned long long v[3];
  const int rc = cudaMemcpy(v, d_v, 3 * 8, cudaMemcpyDeviceToHost) ? -2 : 0;
  *viol_e4m3 = v[0];
  *viol_scale = v[1];
  *viol_e2m1 = v[2];
  cudaFree(d_v);
  return rc;
}
