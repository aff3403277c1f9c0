// Test-only sweeps of the library's SwiGLU (swiglu.cuh).  Builds into
// tests/_build/libswiglu_sweep.so; the tests compare it with the CPU oracle
// and with its own FP64 tier.
#include "../../nvfp4_w4a4_moe_top_gb300/csrc/swiglu.cuh"

namespace {

__device__ __forceinline__ bool finite_bf16(uint32_t b) { return (b & 0x7F80u) != 0x7F80u; }

// Largest relative error of ex2.approx.ftz over every float t with
// 2^-30 <= |t| <= 128 and a normal result (below 2^-30 the result is 1 or
// its neighbour, within 2^-30 of 2^t), and of rcp.approx.ftz over every float
// in [1, 2^126) (float bits of the maxima: non-negative floats order like
// their bits).  The bracket's exponent argument g * kNegLog2eHi of any
// finite BF16 g, and its 1 + E, lie in these ranges wherever the result is
// not flagged for the exact tiers.
__global__ void hw_bounds(unsigned int* out) {
  const unsigned int stride = gridDim.x * blockDim.x;
  const unsigned int i0 = blockIdx.x * blockDim.x + threadIdx.x;
  float e_ex2 = 0.0f, e_rcp = 0.0f;
  for (unsigned int b = 0x30800000u + i0; b <= 0x43000000u; b += stride)
    for (unsigned int s = 0; s < 2; ++s) {
      const float t = __uint_as_float(b | (s << 31));
      if (t < -126.0f) continue;
      const float y = moe::ex2_ftz(t);
      if (isinf(y)) continue;  // an infinite E makes p zero, which the exact tiers take
      const double r = exp2((double)t);
      e_ex2 = fmaxf(e_ex2, (float)(fabs((double)y - r) / r));
    }
  for (unsigned int b = 0x3F800000u + i0; b < 0x7E800000u; b += stride) {
    const float D = __uint_as_float(b);
    const double r = 1.0 / (double)D;
    e_rcp = fmaxf(e_rcp, (float)(fabs((double)moe::rcp_ftz(D) - r) / r));
  }
  atomicMax(out + 0, __float_as_uint(e_ex2));
  atomicMax(out + 1, __float_as_uint(e_rcp));
}

// Every pair of finite BF16 values (g, up): h from swiglu16 (16 up values
// per call, one g) against the FP64 tier; counts mismatches, and how many
// halves the bracket left open (|h| >= 2^-100 only).
__global__ void sweep_all(unsigned long long* out) {
  unsigned long long bad = 0, open_n = 0, tested = 0;
  const uint32_t gb = blockIdx.x;  // 65536 blocks: one g each
  if (!finite_bf16(gb)) return;
  const float g = moe::bf16_bits_to_f32(gb);
  for (uint32_t u0 = threadIdx.x * 16u; u0 < 65536u; u0 += blockDim.x * 16u) {
    uint32_t gw[8], uw[8], h[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      gw[w] = gb | (gb << 16);
      uw[w] = (u0 + 2 * w) | ((u0 + 2 * w + 1) << 16);
    }
    (void)moe::swiglu16(gw, uw, h);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      uint32_t open;
      const uint32_t lo = moe::swiglu_pair_fast(gw[w], uw[w], open);
      for (int hf = 0; hf < 2; ++hf) {
        const uint32_t ub = (uw[w] >> (16 * hf)) & 0xFFFFu;
        if (!finite_bf16(ub)) continue;
        ++tested;
        const uint32_t ref = moe::swiglu_bf16_f64(g, moe::bf16_bits_to_f32(ub));
        if (((h[w] >> (16 * hf)) & 0xFFFFu) != ref) ++bad;
        if (((open >> (16 * hf)) & 0xFFFFu) && ((lo >> (16 * hf)) & 0x7FFFu) >= 0x0D80u) ++open_n;
      }
    }
  }
  atomicAdd(out + 0, bad);
  atomicAdd(out + 1, open_n);
  atomicAdd(out + 2, tested);
}

// Tier 2 alone on every pair of finite BF16 values against the FP64 tier.
__global__ void sweep_tier2(unsigned long long* out) {
  unsigned long long bad = 0;
  const uint32_t gb = blockIdx.x;
  if (!finite_bf16(gb)) return;
  const float g = moe::bf16_bits_to_f32(gb);
  for (uint32_t ub = threadIdx.x; ub < 65536u; ub += blockDim.x) {
    if (!finite_bf16(ub)) continue;
    const float up = moe::bf16_bits_to_f32(ub);
    if (moe::swiglu_bf16_exact(g, up) != moe::swiglu_bf16_f64(g, up)) ++bad;
  }
  atomicAdd(out, bad);
}

// h of n (g, up) pairs, 16 at a time (n % 16 == 0).
__global__ void eval_pairs(const uint16_t* g, const uint16_t* up, uint16_t* h, int n) {
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) * 16;
  if (i >= n) return;
  uint32_t gw[8], uw[8], hw[8];
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    gw[w] = g[i + 2 * w] | ((uint32_t)g[i + 2 * w + 1] << 16);
    uw[w] = up[i + 2 * w] | ((uint32_t)up[i + 2 * w + 1] << 16);
  }
  (void)moe::swiglu16(gw, uw, hw);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    h[i + 2 * w] = (uint16_t)(hw[w] & 0xFFFFu);
    h[i + 2 * w + 1] = (uint16_t)(hw[w] >> 16);
  }
}

}  // namespace

extern "C" float swiglu_eps() { return moe::kSwigluEps; }
extern "C" float swiglu_c1() { return moe::kNegLog2eHi; }
extern "C" float swiglu_c2ln2() { return moe::kNegLog2eLoLn2; }

extern "C" int run_hw_bounds(float* e_ex2, float* e_rcp) {
  unsigned int* d;
  if (cudaMalloc(&d, 8)) return -1;
  cudaMemset(d, 0, 8);
  hw_bounds<<<152 * 8, 256>>>(d);
  unsigned int h[2];
  const int rc = cudaMemcpy(h, d, 8, cudaMemcpyDeviceToHost) ? -2 : 0;
  cudaFree(d);
  memcpy(e_ex2, &h[0], 4);
  memcpy(e_rcp, &h[1], 4);
  return rc;
}

extern "C" int run_sweep_all(unsigned long long* bad, unsigned long long* open_n, unsigned long long* tested,
                             unsigned long long* bad_tier2) {
  unsigned long long* d;
  if (cudaMalloc(&d, 32)) return -1;
  cudaMemset(d, 0, 32);
  sweep_all<<<65536, 256>>>(d);
  sweep_tier2<<<65536, 256>>>(d + 3);
  unsigned long long h[4];
  const int rc = cudaMemcpy(h, d, 32, cudaMemcpyDeviceToHost) ? -2 : 0;
  cudaFree(d);
  *bad = h[0];
  *open_n = h[1];
  *tested = h[2];
  *bad_tier2 = h[3];
  return rc;
}

extern "C" int run_eval_pairs(const uint16_t* g, const uint16_t* up, uint16_t* h, int n) {
  if (n % 16) return -3;
  uint16_t *dg, *du, *dh;
  const size_t bytes = (size_t)n * 2;
  if (cudaMalloc(&dg, bytes) || cudaMalloc(&du, bytes) || cudaMalloc(&dh, bytes)) return -1;
  cudaMemcpy(dg, g, bytes, cudaMemcpyHostToDevice);
  cudaMemcpy(du, up, bytes, cudaMemcpyHostToDevice);
  const int threads = n / 16;
  eval_pairs<<<(threads + 127) / 128, 128>>>(dg, du, dh, n);
  const int rc = cudaMemcpy(h, dh, bytes, cudaMemcpyDeviceToHost) ? -2 : 0;
  cudaFree(dg);
  cudaFree(du);
  cudaFree(dh);
  return rc;
}
