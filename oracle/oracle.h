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
 * Readings where the pages are silent are listed in the design doc and restated at
 * each function below.
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

#ifdef __cplusplus
}
#endif
#endif
