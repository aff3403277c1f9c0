/*
 * MOE-NVFP4-SPEC-1 oracle: a plain, slow CPU restatement of the native NVFP4
 * W4A4 MoE expert forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  It shares
 * no code, header, table or constant with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Sources (page title, section):
 *   [TR 2.2]   "miniTE Technical Report: Stable and Efficient Reinforcement
 *              Learning with Native NVFP4", section 2.2 (E2M1 element, E4M3
 *              block scale per 16 elements, FP32 outer scale; decode is the
 *              product of the three).
 *   [TR 2.3]   same report, section 2.3 (per-token amax restricts the scale
 *              domain to the row).
 *   [TR 4.3]   same report, section 4.3 table ("miniTE per-token": one outer
 *              scale per token for activations, one per row of the flattened
 *              expert weights).
 *   [TR 5.1]   same report, section 5.1 equation: block scale
 *              d = Q_E4M3(amax(b)/(6 s)), decode x^ = s d Q_E2M1(x/(s d)).
 *   [SUM-M]    "miniTE: Diagnosing and Bridging the Execution Gap in Native
 *              NVFP4 Reinforcement Learning" AI summary, "Methodology in Plain
 *              English" (per-row activation outer scale, FP32 epilogue after
 *              the block-scaled multiply, BF16 cast at the end, RHT and
 *              stochastic rounding off, amax gathered during permutation).
 *   [RB-P]     paper.rainbus.top summary, prerequisites: NVFP4 format
 *              (s_b = E4M3(a_b/(6g)), x^ = g s_b c) and MoE grouped GEMM
 *              (router top-k, FC1-SwiGLU-FC2, permutation, padding, expert
 *              offsets, uneven and empty groups).
 *   [RB-C]     same summary, core method (U_e = MMA_NVFP4(X_e, W_e^T), then
 *              the FP32 epilogue broadcasts g_x g_w and casts to BF16).
 *   [RB-S]     same summary, method steps 4-6 (g_x = max_k |X| / (6*448),
 *              g_w per row likewise, 16-element E4M3 blocks, E2M1 codes,
 *              Hadamard and stochastic rounding off; sort fused with amax,
 *              padding carries the statistics, device-side offsets).
 *
 * Where the pages are silent, the reading taken is stated at each function
 * below.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_*.py.
 */
#ifndef MOE_NVFP4_ORACLE_H
#define MOE_NVFP4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar codecs ---- */
float    orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);          /* round to nearest even */
uint16_t orc_f64_to_bf16(double x);         /* one rounding, nearest even */
float    orc_e2m1_value(uint8_t code);      /* 4-bit code -> value */
uint8_t  orc_e2m1_encode(float q);          /* nearest, ties to even code, saturate at 6 */
float    orc_e4m3_value(uint8_t code);      /* OCP E4M3 (FN) byte -> value */
uint8_t  orc_e4m3_encode(float t);          /* t >= 0: nearest, ties even, saturate at 448 */

/* ---- block-scale storage layout ---- */
int64_t orc_sf_offset(int64_t row, int64_t col, int64_t K);
int64_t orc_sf_bytes(int64_t rows, int64_t K);
int64_t orc_m_cap(int64_t T, int64_t E, int64_t k);
void    orc_unswizzle_sf(const uint8_t* sf_swz, int64_t rows, int K, uint8_t* logical);

/* ---- quantisation ---- */
void orc_quantize_row(const float* v, int K, float amax,
                      uint8_t* codes, uint8_t* sf_logical, float* g);
void orc_amax_rows_bf16(const uint16_t* x, int64_t rows, int K, float* amax);
void orc_quantize_rows_bf16(const uint16_t* src, int64_t src_rows, int K,
                            const int32_t* row_map, const float* amax,
                            int64_t dst_rows, uint8_t* codes, uint8_t* sf_swz,
                            float* g);
void orc_dequantize_rows(const uint8_t* codes, const uint8_t* sf_swz,
                         const float* g, int64_t rows, int K, double* out);

/* ---- routing and permutation ---- */
int  orc_route(const float* logits, int64_t T, int E, int k,
               int32_t* ids, float* w);
int  orc_permute(const int32_t* ids, int64_t T, int E, int k, int64_t m_cap,
                 int32_t* counts, int32_t* offsets, int32_t* row_to_token,
                 int32_t* token_slot_row);

/* ---- grouped GEMM and epilogues ---- */
void orc_grouped_gemm(const uint8_t* a_codes, const uint8_t* a_sf_swz,
                      const float* a_g, const int32_t* offsets, int E,
                      int64_t M, int K, int N, const uint8_t* w_codes,
                      const uint8_t* w_sf_swz, const float* w_g, float* y);
void orc_swiglu(const float* y, int64_t M, int F, uint16_t* u, uint16_t* h);
void orc_combine(const float* y2, const int32_t* row_to_token,
                 const int32_t* token_slot_row, const float* topk_w,
                 int64_t T, int k, int64_t M, int d, uint16_t* slots);
void orc_reduce(const uint16_t* slots, int64_t T, int k, int d, uint16_t* out);

/* ---- self checks used by the pins ---- */
int64_t orc_e4m3_first_input_of_code(uint8_t code);
int64_t orc_e2m1_first_input_of_code(uint8_t code);
int     orc_num_threads(void);
void    orc_set_num_threads(int n);

/* ---- contrast recipes (not the hot path's recipe) ---- */

/* Random Hadamard transform along K in blocks of 16, a contrast reference
 * for the recipe the pages switch off ([SUM-M]: Hadamard transforms off, so
 * a token's codes do not depend on the other tokens of its batch):
 *   y[16b + i] = RN_f32( (1/4) * sum_j H[i][j] * s[j] * x[16b + j] ),
 * H the 16x16 Sylvester Hadamard matrix (H[i][j] = (-1)^popcount(i & j)),
 * s a +-1 sign vector of length 16; evaluated in FP64, rounded once. */
void orc_rht16_rows(const float* x, int64_t rows, int K, const int8_t* signs16, float* y);

/* Per-tensor NVFP4 quantisation of FP32 rows: one outer scale
 * g = amax(all rows) / 2688 shared by every row ([RB-P]: the outer scale's
 * granularity, per-tensor / per-row / per-token, is a recipe choice), block
 * scales and codes as orc_quantize_row.  g_out[r] = g for every row. */
void orc_quantize_tensor(const float* x, int64_t rows, int K, uint8_t* codes, uint8_t* sf_swz, float* g_out);

/* Weights with one outer scale per expert tensor ("miniTE CUTLASS" column of
 * [TR 4.3]'s table): for expert e, g_e = max |W_e| / 2688 over its N x K
 * entries; every row of the expert is quantised with that amax.
 * g[e][n] = g_e for all n. */
void orc_quantize_weights_per_expert(const uint16_t* W, int E, int N, int K, uint8_t* codes, uint8_t* sf_swz,
                                     float* g);

/* ---- backward (straight-through, BF16 GEMM operands) ----
 *
 * [SUM-M] and the main paper's contributions list: the backward is a
 * straight-through estimator on the saved original BF16 activations and
 * weights, with no backward quantisation; [RB-S] step 5: BF16 GEMMs on the
 * saved BF16 operands.  [TR 4.3] (text below the table): the layer bypass
 * saves the original BF16 operands and skips backward quantisation.
 * Readings: the quantisers pass gradients unchanged; the saved values are
 * the forward's own u = BF16(FC1 output), h = BF16(SwiGLU output) and the
 * FP32 expert output y2; the BF16 GEMM operands are dy2 = BF16(w * dY)
 * (router coefficient in FP32, then the cast, as in the forward) and
 * du = BF16(SwiGLU backward); everything else is evaluated in FP64 here. */

/* Router gradients from the saved expert outputs:
 *   dw[t][j]  = sum_n dY[t][n] * y2[row(t,j)][n]
 *   dlogits[t][ids[t][j]] = w_j * (dw_j - sum_i w_i dw_i), 0 elsewhere
 * (the weights are a softmax over the selected logits; top-k selection is
 * piecewise constant).  FP64, rounded once to FP32. */
void orc_bwd_router(const uint16_t* dY, const float* y2, const float* w, const int32_t* ids,
                    const int32_t* token_slot_row, int64_t T, int k, int d, int E, float* dw, float* dlogits);

/* dy2[row(t,j)][n] = BF16(RN_f32(w[t][j] * dY[t][n])); pad rows (every row
 * not named by token_slot_row) are zero.  dy2 is [M][d]. */
void orc_bwd_dy2(const uint16_t* dY, const float* w, const int32_t* token_slot_row, int64_t T, int k, int d,
                 int64_t M, uint16_t* dy2);

/* One expert over n of its rows (dy2, u, h, xr hold those rows; xr[i] is the
 * BF16 input row of the row's token, zero on pad rows):
 *   dh[r][f]  = sum_n dy2[r][n] W2[n][f]                        (FP64)
 *   s = 1/(1+exp(-g)), g = u[r][f], v = u[r][F+f]
 *   du[r][f]   = BF16(dh * v * s * (1 + g (1 - s)))             (gate half)
 *   du[r][F+f] = BF16(dh * g * s)                                (up half)
 *   dxr[r][i] = sum_j du[r][j] W1[j][i]                         (FP64 out)
 *   dW2[n][f] = sum_r dy2[r][n] h[r][f],  dW1[j][i] = sum_r du[r][j] xr[r][i]
 * (FP64, rounded once to FP32).  W1 is [2F][d], W2 is [d][F]. */
void orc_bwd_expert(const uint16_t* dy2, const uint16_t* u, const uint16_t* h, const uint16_t* xr, int64_t n,
                    int d, int F, const uint16_t* W1, const uint16_t* W2, uint16_t* du, double* dxr, float* dW1,
                    float* dW2);

#ifdef __cplusplus
}
#endif
#endif
