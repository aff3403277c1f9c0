// Host-side launch functions of the kernels (internal to libmoe_nvfp4.so).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kRouteChunk = 64;  // tokens per routing chunk (one CTA); a multiple of 32

// amax (optional) holds one entry per amax_rows consecutive source rows.
// Two launches: the row quantiser, then its fix-up pass for the rows whose
// outer scale lies outside [2^-87, 2^111] (encoded with the E2M1 division's
// row factor).
int launch_quantize_rows(const uint16_t* src, int64_t src_rows, int K, const int32_t* row_map,
                         const float* amax, int64_t amax_rows, int64_t dst_rows, uint8_t* codes, uint8_t* sf,
                         float* g, int* status, int nonfinite_bit, cudaStream_t stream);

// Per-expert max |W| into amax_e[E], then the row quantiser with that amax
// for all N rows of each expert.  Returns -1 if the memset fails to enqueue.
int launch_quantize_weights_per_expert(const uint16_t* W, int E, int N, int K, uint8_t* codes, uint8_t* sf, float* g,
                                       float* amax_e, int* status, cudaStream_t stream);

// Routing: top-k, weights, in-chunk ranks (into token_slot_row) and chunk
// histograms hist[C][E].
int launch_route(const float* logits, const int32_t* ext_ids, const float* ext_w, int T, int E, int k,
                 int32_t* topk_ids, float* topk_w, int32_t* token_slot_row, int32_t* hist, int* status,
                 cudaStream_t stream);

// Chunk histograms -> exclusive chunk bases (in place) and counts; the
// padded offsets come from launch_pad_rows, which runs next.
int launch_scan(int32_t* hist, int C, int E, int32_t* counts, cudaStream_t stream);

// Final rows of the slots, row_to_token, and (when x != NULL) per-token amax
// gathered in the same pass.
int launch_permute_amax(const int32_t* topk_ids, int32_t* token_slot_row, const int32_t* hist, const int32_t* offsets,
                        int T, int E, int k, const uint16_t* x, int d, int32_t* row_to_token, float* amax_tok,
                        float* amax_row, int* status, cudaStream_t stream);

// Padded offsets [E+1] from the counts, then the pad rows of every group
// (and rows >= M_pad up to m_cap): row_to_token = -1, amax_row = 0, and when
// codes != NULL zero codes / block scales / g.
int launch_pad_rows(int32_t* offsets, const int32_t* counts, int E, int64_t m_cap, int32_t* row_to_token,
                    float* amax_row, uint8_t* codes, int K, uint8_t* sf, float* g, cudaStream_t stream);

// Fused permute + amax + quantise of the forward: x read once, codes written
// into the k destination rows of each token.
// tok_codes: NULL, or token-ordered codes [T + 1][d/2] (row T zeroed here)
// written instead of the k row copies of `codes`.
int launch_permute_quant(const int32_t* topk_ids, int32_t* token_slot_row, const int32_t* hist, const int32_t* offsets,
                         int T, int E, int k, const uint16_t* x, int d, int32_t* row_to_token, float* amax_tok,
                         uint8_t* codes, uint8_t* tok_codes, uint8_t* sf, float* g, int* status, cudaStream_t stream);

// out[t] = BF16(sum_j FP32(z[token_slot_row[t][j]])), j ascending.
int launch_unpermute_reduce(const uint16_t* z, const int32_t* token_slot_row, int T, int k, int d, uint16_t* out,
                            cudaStream_t stream);

struct Fc1Args {
  CUtensorMap tmap_a, tmap_b;
  const uint8_t* a_sf;
  const float* a_g;
  const uint8_t* w_sf;
  const float* w_g;
  const int32_t* offsets;
  int E, d, d_ff;
  uint8_t* h_codes;
  uint8_t* h_sf;
  float* h_g;
  float* dbg_u;
  uint16_t* dbg_h;
  uint16_t* save_u;  // BF16 u [rows][2 d_ff] for the backward, or NULL
  // Gather-on-load A: tmap_a then maps token-ordered codes [zero_row + 1]
  // rows with 1-row boxes; row r of a unit is token a_rows[r] (zero_row when
  // negative).  NULL: tmap_a maps the permuted rows (128-row boxes).
  const int32_t* a_rows;
  int zero_row;
  uint16_t* scratch;
  int* status;
  int rings, na, nb, resident;  // pipeline plan, set by launch_fc1
};
constexpr int kMaxGemmCtas = 256;
constexpr int kFc1EpiThreads = 512;  // FC1 epilogue threads per CTA
constexpr int kFc1DeferSlots = 16;   // deferred exact-SwiGLU fixes per epilogue thread and unit
// FC1 workspace: h staging, two 128 x d_ff BF16 buffers per CTA, then
// kFc1DeferSlots 16-byte slots per epilogue thread for the SwiGLU pairs
// whose exact evaluation waits until the end of the unit.
__host__ __device__ inline size_t fc1_staging_bytes(int d_ff) { return (size_t)kMaxGemmCtas * 2 * 128 * d_ff * 2; }
inline size_t fc1_workspace_bytes(int d_ff) {
  return fc1_staging_bytes(d_ff) + (size_t)kMaxGemmCtas * kFc1EpiThreads * kFc1DeferSlots * 16;
}
struct Fc2Args {
  CUtensorMap tmap_a, tmap_b;
  CUtensorMap tmap_out;  // output rows [m_cap][d] BF16 (z, or dy2 in MODE 2): boxes 64 x 32, 128-byte swizzle
  const uint8_t* a_sf;
  const float* a_g;
  const uint8_t* w_sf;
  const float* w_g;
  const int32_t* offsets;
  int E, d_ff, d, k;
  const int32_t* row_to_token;
  const int32_t* token_slot_row;
  const float* topk_w;
  float* dbg_y;
  // backward recomputation (dw set): dY bf16 [T][d] in, dw f32 [T][k] out,
  // and tmap_out maps dy2 bf16 [m_cap][d] instead of the z rows
  const uint16_t* dY;
  float* dw;
  int* status;
  int rings, na, nb, resident;  // pipeline plan, set by launch_fc2
};

// BF16 grouped GEMMs of the backward (bwd.cu).
enum { BWD_DGRAD_SWIGLU = 0, BWD_DGRAD = 1, BWD_WGRAD = 2 };
struct BwdGemmArgs {
  CUtensorMap tmap_a, tmap_b;  // A: K-major box 64 x 128 (dgrad) or MN-major 64 x 64 (wgrad); B: MN-major 64 x 64
  CUtensorMap tmap_out;        // DGRAD / WGRAD: FP32 `out`, boxes of 32 x 32, 128-byte swizzle
  int mode, a_mn;
  int E;
  const int32_t* offsets;
  int N;        // output columns
  int K;        // dgrad: contraction length (rows of B per expert)
  int Mo;       // wgrad: output rows per expert
  int F;        // DGRAD_SWIGLU: d_ff
  const uint16_t* u;  // DGRAD_SWIGLU: saved u [rows][2F]
  uint16_t* du;       // DGRAD_SWIGLU: out [rows][2F]
  float* out;         // DGRAD: [rows][N]; WGRAD: [E][Mo][N]
  int* status;
  int bn, stages;     // set by launch_bwd_gemm
};
int launch_bwd_gemm(BwdGemmArgs& a, int max_row_tiles, cudaStream_t stream);
int launch_bwd_xrows(const uint16_t* x, const int32_t* row_to_token, const int32_t* offsets, int E, int T, int d,
                     int64_t m_rows, uint16_t* xp, int blocks, cudaStream_t stream);
int launch_bwd_logits(const float* dw, const float* topk_w, const int32_t* topk_ids, int T, int E, int k,
                      float* dlogits, cudaStream_t stream);
int launch_bwd_dx(const float* dxr, const int32_t* token_slot_row, int T, int k, int d, float* dx, cudaStream_t stream);

int gemm_num_ctas();  // persistent grid size on the current device
int launch_fc1(Fc1Args& a, int64_t m_cap, cudaStream_t stream);
int launch_fc2(Fc2Args& a, int64_t m_cap, cudaStream_t stream);

}  // namespace moe
