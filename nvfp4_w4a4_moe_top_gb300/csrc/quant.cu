// NVFP4 row quantiser: one warp per destination row, the row held in
// registers (128-bit loads), warp-shuffle amax, per-row outer scale
// g = amax/(6*448), E4M3 block scales and E2M1 codes written straight into
// the GEMM's operand buffers (miniTE Technical Report section 5.1 equation;
// AI summary "Methodology in Plain English": the quantiser writes packed
// codes, block scales and outer-scale metadata into the contiguous buffers
// the GEMM consumes).
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// Byte offset of the 4-byte word holding block scales (row, 4*c4 .. 4*c4+3).
__device__ __forceinline__ int64_t sf_word_offset(int64_t row, int c4, int kgroups) {
  return ((row >> 7) * kgroups + c4) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

template <int MAXCH>
__global__ void __launch_bounds__(256) quantize_rows_kernel(
    const uint16_t* __restrict__ src, int64_t src_rows, int K, const int32_t* __restrict__ row_map,
    const float* __restrict__ amax, int64_t amax_rows, int64_t dst_rows, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ sf, float* __restrict__ gout, int* status, int nonfinite_bit) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= dst_rows) return;
  const int kg = K / 64;
  int64_t s = row_map ? (int64_t)row_map[r] : r;
  if (s >= src_rows) {  // invalid map entry: write a zero row and flag it
    if (lane == 0) set_status(status, MOE_STATUS_BAD_ROUTING);
    s = -1;
  }
  uint8_t* crow = codes + r * (K / 2);
  if (s < 0) {
    for (int i = lane; i < K / 8; i += 32) reinterpret_cast<uint32_t*>(crow)[i] = 0u;
    for (int c4 = lane; c4 < kg; c4 += 32) *reinterpret_cast<uint32_t*>(sf + sf_word_offset(r, c4, kg)) = 0u;
    if (lane == 0) gout[r] = 0.0f;
    return;
  }
  const uint4* srow = reinterpret_cast<const uint4*>(src + s * (int64_t)K);
  const int n8 = K / 8;  // 8-element groups in the row
  uint4 v[MAXCH];
  float a = 0.0f;
  bool fin = true;
#pragma unroll
  for (int i = 0; i < MAXCH; ++i) {
    const int e8 = i * 32 + lane;
    v[i] = make_uint4(0u, 0u, 0u, 0u);
    if (e8 < n8) {
      v[i] = __ldg(srow + e8);
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        fin = fin && bf16x2_finite(w[q]);
        a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[q])), fabsf(bf16_hi(w[q]))));
      }
    }
  }
  if (!__all_sync(0xFFFFFFFFu, fin) && lane == 0) set_status(status, nonfinite_bit);
  a = amax ? amax[s / amax_rows] : warp_max(a);
  const float g = __fdiv_rn(a, 2688.0f);
  const float den = __fmul_rn(6.0f, g);
#pragma unroll
  for (int i = 0; i < MAXCH; ++i) {
    if (i * 32 < n8) {  // warp-uniform
      const int e8 = i * 32 + lane;
      uint32_t sb;
      const uint32_t packed = quant_half_block(v[i], g, den, &sb);
      const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
      const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sb, 4);
      const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sb, 6);
      if (e8 < n8) {
        reinterpret_cast<uint32_t*>(crow)[e8] = packed;
        if ((lane & 7) == 0)
          *reinterpret_cast<uint32_t*>(sf + sf_word_offset(r, e8 >> 3, kg)) = sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
      }
    }
  }
  if (lane == 0) gout[r] = g;
}

int launch_quantize_rows(const uint16_t* src, int64_t src_rows, int K, const int32_t* row_map,
                         const float* amax, int64_t amax_rows, int64_t dst_rows, uint8_t* codes, uint8_t* sf,
                         float* g, int* status, int nonfinite_bit, cudaStream_t stream) {
  if (dst_rows <= 0) return 0;
  const int nch = (K / 8 + 31) / 32;
  const dim3 grid((unsigned)((dst_rows + 7) / 8));
  if (nch <= 4)
    quantize_rows_kernel<4><<<grid, 256, 0, stream>>>(src, src_rows, K, row_map, amax, amax_rows, dst_rows, codes, sf,
                                                      g, status, nonfinite_bit);
  else if (nch <= 8)
    quantize_rows_kernel<8><<<grid, 256, 0, stream>>>(src, src_rows, K, row_map, amax, amax_rows, dst_rows, codes, sf,
                                                      g, status, nonfinite_bit);
  else
    quantize_rows_kernel<16><<<grid, 256, 0, stream>>>(src, src_rows, K, row_map, amax, amax_rows, dst_rows, codes,
                                                       sf, g, status, nonfinite_bit);
  return 0;
}

// max |W_e| of each expert tensor (one outer scale per expert weight tensor:
// miniTE Technical Report section 4.3 table, "miniTE CUTLASS" column).
// blockIdx.y is the expert; the blocks of one expert stride over its N*K
// values with 128-bit loads, reduce in shared memory and fold their maximum
// into amax_e[e] with one integer atomicMax on the float's bits (valid
// because every candidate is >= +0, and amax_e starts at +0).  NaNs do not
// win a maximum; the quantiser flags them.
__global__ void __launch_bounds__(256) expert_amax_kernel(const uint16_t* __restrict__ W, int64_t per_expert,
                                                          float* __restrict__ amax_e) {
  const uint4* src = reinterpret_cast<const uint4*>(W + (int64_t)blockIdx.y * per_expert);
  const int64_t n8 = per_expert / 8;
  const int64_t stride = (int64_t)gridDim.x * 256;
  float a = 0.0f;
  int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[q])), fabsf(bf16_hi(w[q]))));
    }
  }
  for (; i < n8; i += stride) {
    const uint4 v = __ldg(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[q])), fabsf(bf16_hi(w[q]))));
  }
  a = warp_max(a);
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x < 32) {
    a = threadIdx.x < 8 ? red[threadIdx.x] : 0.0f;
    a = warp_max(a);
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(amax_e + blockIdx.y), __float_as_uint(a));
  }
}

int launch_quantize_weights_per_expert(const uint16_t* W, int E, int N, int K, uint8_t* codes, uint8_t* sf, float* g,
                                       float* amax_e, int* status, cudaStream_t stream) {
  if (cudaMemsetAsync(amax_e, 0, (size_t)E * sizeof(float), stream) != cudaSuccess) return -1;
  const int64_t per_expert = (int64_t)N * K;
  // about eight resident 256-thread blocks per SM over all experts, and no
  // block without work
  const int64_t want = (8 * 152 + E - 1) / E;
  const int64_t most = (per_expert / 8 + 255) / 256;
  const unsigned gx = (unsigned)(want < most ? want : most);
  expert_amax_kernel<<<dim3(gx, (unsigned)E), 256, 0, stream>>>(W, per_expert, amax_e);
  return launch_quantize_rows(W, (int64_t)E * N, K, nullptr, amax_e, N, (int64_t)E * N, codes, sf, g, status,
                              MOE_STATUS_NONFINITE_WEIGHT, stream);
}

}  // namespace moe
