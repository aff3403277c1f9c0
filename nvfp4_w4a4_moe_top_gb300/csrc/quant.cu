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

// One warp per destination row.  Lane L holds, for each group of 1024
// columns, the 32 consecutive columns from 32*L: two whole 16-element blocks,
// so every block's scale is computed once, its codes leave as one 16-byte
// store and lanes L, L ^ 1 form one 32-bit scale word.  The blocks' largest
// magnitudes, taken as BF16 bit patterns, give the block amax, the row amax
// and the non-finite check at once.  A row holding a NaN takes its amax over
// the other values, as fmaxf does; its codes are unspecified and the status
// bit reports it.

// The row (K BF16 values) into the warp's registers.
template <int NG>
__device__ __forceinline__ void load_row(const uint16_t* __restrict__ src_row, int K, int lane, uint4 (&v)[NG][4]) {
  const uint4* srow = reinterpret_cast<const uint4*>(src_row);
  const int n8 = K / 8;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int e8 = g * 128 + 4 * lane;
#pragma unroll
    for (int q = 0; q < 4; ++q) v[g][q] = e8 < n8 ? __ldg(srow + e8 + q) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Largest magnitude of the row as BF16 magnitude bits, NaNs left out (warp
// reduction); sets `nonfinite_bit` in status when the row holds a NaN or Inf.
template <int NG>
__device__ __forceinline__ uint32_t row_amax_bits(const uint4 (&v)[NG][4], uint32_t (&bm)[NG][2], int lane, int* status,
                                                  int nonfinite_bit) {
  uint32_t lm = 0;
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      bm[g][b] = absmax_bits16(v[g][2 * b], v[g][2 * b + 1]);
      lm = max(lm, bm[g][b]);
    }
  const uint32_t rm = __reduce_max_sync(0xFFFFFFFFu, lm);
  if (rm >= 0x7F80u && lane == 0) set_status(status, nonfinite_bit);
  // a NaN in the row (warp-uniform, rare): the largest other magnitude
  return rm <= 0x7F80u ? rm : __reduce_max_sync(0xFFFFFFFFu, absmax_bits_no_nan(v));
}

// Codes, block scales and g of destination row r from the row in registers
// (bm: its blocks' magnitude maxima) and the row's outer scale gs.  SCALED
// false: gs passes e2m1_div_row_scale_ok, so the row factor is 1.
template <int NG, bool SCALED>
__device__ __forceinline__ void encode_row(const uint4 (&v)[NG][4], const uint32_t (&bm)[NG][2], float gs, int64_t r,
                                           int K, int lane, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                           float* __restrict__ gout) {
  const int kg = K / 64;
  const int n8 = K / 8;
  uint4* crow = reinterpret_cast<uint4*>(codes + r * (K / 2));
  const int64_t sf_row = (r >> 7) * kg * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
  const float den = __fmul_rn(6.0f, gs);
  const float rden = block_scale_rden(den);
  const float f = SCALED ? e2m1_row_factor(gs) : 1.0f;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int e8 = g * 128 + 4 * lane;
    if (g * 128 >= n8) break;  // warp-uniform
    uint32_t c[4] = {0u, 0u, 0u, 0u}, sb2 = 0u;
    if (e8 < n8 && gs != 0.0f) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {  // the lane's two blocks of 16
        const uint4 p0 = v[g][2 * b], p1 = v[g][2 * b + 1];
        const uint32_t w0[4] = {p0.x, p0.y, p0.z, p0.w}, w1[4] = {p1.x, p1.y, p1.z, p1.w};
        const uint32_t sb = block_scale_code(__uint_as_float(bm[g][b] << 16), den, rden);
        const float S = __fmul_rn(gs, e4m3_decode_hw(sb));
        if (S != 0.0f) {
          const uint2 cc = e2m1_codes16_div<SCALED>(w0, w1, S, f);
          c[2 * b] = cc.x;
          c[2 * b + 1] = cc.y;
        }
        sb2 |= sb << (8 * b);
      }
    }
    const uint32_t sfw = sb2 | (__shfl_xor_sync(0xFFFFFFFFu, sb2, 1) << 16);
    if (e8 < n8) {
      crow[e8 >> 2] = make_uint4(c[0], c[1], c[2], c[3]);
      if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(sf + sf_row + (int64_t)(e8 >> 3) * 512) = sfw;
    }
  }
  if (lane == 0) gout[r] = gs;
}

template <int NG>
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
  if (s < 0) {
    uint4* crow = reinterpret_cast<uint4*>(codes + r * (K / 2));
    const int64_t sf_row = (r >> 7) * kg * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
    for (int i = lane; i < K / 32; i += 32) crow[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int c4 = lane; c4 < kg; c4 += 32) *reinterpret_cast<uint32_t*>(sf + sf_row + c4 * 512) = 0u;
    if (lane == 0) gout[r] = 0.0f;
    return;
  }
  uint4 v[NG][4];
  load_row<NG>(src + s * (int64_t)K, K, lane, v);
  uint32_t bm[NG][2];
  const uint32_t ab = row_amax_bits<NG>(v, bm, lane, status, nonfinite_bit);
  const float a = amax ? amax[s / amax_rows] : __uint_as_float(ab << 16);
  const float gs = __fdiv_rn(a, 2688.0f);
  if (gs != 0.0f && !e2m1_div_row_scale_ok(gs)) {  // warp-uniform and rare: left to the fix-up pass
    if (lane == 0) gout[r] = gs;
    return;
  }
  encode_row<NG, false>(v, bm, gs, r, K, lane, codes, sf, gout);
}

// Fix-up pass after quantize_rows_kernel: the rows it left, whose outer
// scale g (already in gout) is nonzero and outside [2^-87, 2^111], encoded
// with the E2M1 division's row factor.  Such rows are rare (row maxima
// below about 1.7e-23 or above 7e36), so the main pass carries a single
// copy of the encoder, without the factor; here each warp reads the g of
// 32 rows at a time and takes the flagged ones one by one.
template <int NG>
__global__ void __launch_bounds__(256) quantize_rows_fixup_kernel(
    const uint16_t* __restrict__ src, int K, const int32_t* __restrict__ row_map, int64_t dst_rows,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ gout) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * 8;
  for (int64_t r0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * 32; r0 < dst_rows; r0 += nw * 32) {
    const float gl = r0 + lane < dst_rows ? gout[r0 + lane] : 0.0f;
    unsigned need = __ballot_sync(0xFFFFFFFFu, gl != 0.0f && !e2m1_div_row_scale_ok(gl));
    while (need) {
      const int i = __ffs(need) - 1;
      need &= need - 1;
      const int64_t r = r0 + i;
      const float gs = __shfl_sync(0xFFFFFFFFu, gl, i);
      // the main pass zeroed the rows of invalid map entries (g = 0), so s is valid
      const int64_t s = row_map ? (int64_t)row_map[r] : r;
      uint4 v[NG][4];
      load_row<NG>(src + s * (int64_t)K, K, lane, v);
      uint32_t bm[NG][2];
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int b = 0; b < 2; ++b) bm[g][b] = absmax_bits16(v[g][2 * b], v[g][2 * b + 1]);
      encode_row<NG, true>(v, bm, gs, r, K, lane, codes, sf, gout);
    }
  }
}

int launch_quantize_rows(const uint16_t* src, int64_t src_rows, int K, const int32_t* row_map,
                         const float* amax, int64_t amax_rows, int64_t dst_rows, uint8_t* codes, uint8_t* sf,
                         float* g, int* status, int nonfinite_bit, cudaStream_t stream) {
  if (dst_rows <= 0) return 0;
  const int ng = (K + 1023) / 1024;
  const dim3 grid((unsigned)((dst_rows + 7) / 8));
  // fix-up pass: 256 rows per block and iteration, at most four blocks per SM
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    sms = 152;
  const int64_t fix_all = (dst_rows + 255) / 256;
  const dim3 fix_grid((unsigned)(fix_all < 4 * sms ? fix_all : 4 * sms));
#define MOE_QR(N)                                                                                            \
  quantize_rows_kernel<N><<<grid, 256, 0, stream>>>(src, src_rows, K, row_map, amax, amax_rows, dst_rows, codes, \
                                                    sf, g, status, nonfinite_bit);                                \
  quantize_rows_fixup_kernel<N><<<fix_grid, 256, 0, stream>>>(src, K, row_map, dst_rows, codes, sf, g)
  if (ng <= 1) { MOE_QR(1); }
  else if (ng <= 2) { MOE_QR(2); }
  else { MOE_QR(4); }
#undef MOE_QR
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
