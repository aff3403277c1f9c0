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
