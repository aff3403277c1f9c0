/*
 * moe_nvfp4.h -- C ABI of libmoe_nvfp4.so: the native NVFP4 W4A4
 * Mixture-of-Experts expert forward on one NVIDIA GB300 (sm_103a).
 *
 * The operation and its sources (page title, section):
 *   - NVFP4 format: E2M1 elements, one E4M3 block scale per 16 elements, an
 *     FP32 outer scale; decode x^ = g * s_b * c.  "miniTE Technical Report:
 *     Stable and Efficient Reinforcement Learning with Native NVFP4", section
 *     2.2, and the paper.rainbus.top summary, prerequisites ("NVFP4 format").
 *   - Block scale s_b = Q_E4M3(a_b / (6 g)), element code Q_E2M1(x / (g s_b)):
 *     Technical Report section 5.1, equation.
 *   - Outer scale g = amax / (6*448), per token for activations and per output
 *     row for weights: Technical Report section 4.3 table ("miniTE
 *     per-token"), rainbus summary, method step 4.
 *   - Quantiser writes packed codes, block scales and outer scales straight
 *     into the contiguous buffers the grouped GEMM consumes; per-token amax is
 *     gathered during permutation; expert offsets live on the device: AI
 *     summary ("miniTE: Diagnosing and Bridging the Execution Gap in Native
 *     NVFP4 Reinforcement Learning"), "Methodology in Plain English" and "Key
 *     Contributions" item 4; rainbus summary, method step 6.
 *   - Grouped GEMM U_e = MMA_NVFP4(X_e, W_e^T) with the FP32 epilogue that
 *     multiplies by g_x g_w and casts to BF16: rainbus summary, core method.
 *   - Router top-k and the FC1 -> SwiGLU -> FC2 expert, uneven and empty
 *     groups: rainbus summary, prerequisites ("MoE and grouped GEMM").
 *
 * Execution specification (MOE-NVFP4-SPEC-1), fixed here:
 *   route: top-k by (FP32 logit desc, expert id asc); slot j = j-th selected
 *     expert in ascending id; weights = softmax over the selected logits.
 *   permute: groups padded to 128 rows; rows of a group in ascending token
 *     order; pad rows are all-zero rows.
 *   quantise: g = amax/2688; s_b = E4M3_RNE_satfinite(a_b/(6g));
 *     S_b = g*s_b; c = E2M1_RNE_satfinite(v/S_b) (true division); amax = 0
 *     gives g = 0 and zero codes; codes two per byte, even element in the low
 *     nibble; sign of a zero code = sign of the quotient.
 *   FC1: y = acc*(g_x*g_w) in FP32, u = BF16(y); gate = columns [0,d_ff),
 *     up = [d_ff, 2 d_ff); h = BF16(silu(gate)*up); h requantised per row.
 *   FC2: y2 = acc*(g_h*g_w2) in FP32; z = BF16(w_{t,e}*y2) stored as slot
 *     (t, j), which lives at row token_slot_row[t][j] of the z rows;
 *     out[t] = BF16(sum_j FP32(z_j)) in ascending j.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller, 16-byte aligned
 *     (TMA and 128-bit accesses).  The library never allocates, frees or
 *     synchronises; every call is enqueued on `stream` (a cudaStream_t passed
 *     as void*, NULL = legacy default stream) and returns before the GPU work
 *     completes.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Return value: MOE_OK or a negative MOE_ERR_* code, detected on the host
 *     before anything is enqueued (except MOE_ERR_CUDA, reported from
 *     cudaGetLastError after the launches).
 *   - `status` (optional device int*, may be NULL) receives MOE_STATUS_* bits
 *     OR-ed in by the kernels when they see data faults (non-finite inputs,
 *     invalid routing replay) or give up a bounded wait.  The kernels finish
 *     in all cases; nothing traps.  The caller zeroes it.
 *   - Results are deterministic bit for bit for given inputs.
 *   - Block-scale buffers ("sf") use the 128x4 tile layout: logical byte
 *     (r, c) of a [rows][K/16] matrix lives at
 *     ((r/128)*(K/64) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4,
 *     nvfp4_sf_bytes(rows, K) bytes in total.
 *
 * Shape limits: 1 <= k <= min(E, 32), E <= 1024, T >= 0 (T = 0 is a no-op),
 * d % 128 == 0, d_ff % 128 == 0, 128 <= d, d_ff <= 4096; row counts < 2^31.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_NVFP4_ABI_VERSION 1

/* return codes */
#define MOE_OK              0
#define MOE_ERR_POINTER    -1   /* required pointer NULL or not 16-byte aligned */
#define MOE_ERR_SHAPE      -2   /* shape outside the limits above */
#define MOE_ERR_WORKSPACE  -3   /* workspace smaller than the *_workspace_bytes helper */
#define MOE_ERR_CUDA       -4   /* CUDA runtime or launch error */
#define MOE_ERR_DEVICE     -5   /* current device is not compute capability 10.3 */

/* device status bits */
#define MOE_STATUS_NONFINITE_X       0x01  /* NaN/Inf in activations (x or h) */
#define MOE_STATUS_NONFINITE_LOGITS  0x02  /* NaN/Inf in router logits */
#define MOE_STATUS_NONFINITE_WEIGHT  0x04  /* NaN/Inf in weights being quantised */
#define MOE_STATUS_BAD_ROUTING       0x08  /* replayed ids out of range or not strictly ascending */
#define MOE_STATUS_TIMEOUT           0x10  /* a GEMM gave up a bounded wait; its outputs are invalid */

/* ---------------------------------------------------------------------- */
/* Helpers (host only, no CUDA calls).                                      */
/* ---------------------------------------------------------------------- */
int         moe_abi_version(void);
const char* moe_status_string(int code);

/* Rows of the padded routed-row buffers: T*k + 127*min(E, T*k), rounded up to
 * a multiple of 128.  Every per-row buffer below has this many rows. */
int64_t moe_m_cap(int T, int E, int k);

/* Bytes of a block-scale buffer for `rows` rows of K elements (K % 64 == 0). */
size_t nvfp4_sf_bytes(int64_t rows, int K);

/* Workspace of moe_permute_amax (chunk histograms). */
size_t moe_permute_workspace_bytes(int T, int E);

/* Workspace of nvfp4_grouped_gemm_fc1_swiglu: h staging, two 128 x d_ff
 * BF16 buffers per CTA (a unit is staged while the previous one is
 * requantised), then sixteen 16-byte slots per epilogue thread (512 per
 * CTA) for the SwiGLU pairs whose exact evaluation is deferred to the end of
 * the unit. */
size_t nvfp4_fc1_workspace_bytes(int d_ff);

/* Workspace of moe_expert_forward (all intermediates of one forward). */
size_t moe_expert_forward_workspace_bytes(int T, int E, int k, int d, int d_ff);

/* Workspace of moe_expert_backward: dy2 and the permuted x (BF16 [M_cap][d]
 * each), du (BF16 [M_cap][2 d_ff]) and the per-row dgrad dxr (FP32
 * [M_cap][d]), in that order. */
size_t moe_expert_backward_workspace_bytes(int T, int E, int k, int d, int d_ff);

/* Byte offsets of the intermediates inside moe_expert_forward's workspace,
 * for inspection after a call (index order: 0 topk_ids i32[T][k],
 * 1 topk_w f32[T][k], 2 token_slot_row i32[T][k], 3 counts i32[E],
 * 4 offsets i32[E+1], 5 row_to_token i32[M_cap], 6 amax_tok f32[T],
 * 7 x_codes u8[M_cap][d/2], 8 x_sf, 9 x_g f32[M_cap], 10 h_codes
 * u8[M_cap][d_ff/2], 11 h_sf, 12 h_g f32[M_cap], 13 z rows bf16[M_cap][d]
 * (slot (t, j) at row token_slot_row[t][j]), 14 chunk histograms, 15 FC1
 * workspace: h staging and deferred SwiGLU slots).  Writes 16 entries; returns 0. */
int moe_expert_forward_workspace_layout(int T, int E, int k, int d, int d_ff,
                                        size_t offsets_out[16]);

/* ---------------------------------------------------------------------- */
/* Entry points.                                                            */
/* ---------------------------------------------------------------------- */

/* Per-output-row NVFP4 quantisation of expert weights (Technical Report
 * section 4.3 table: one outer scale per row of the flattened expert
 * weights; section 5.1 equation for the block scales and codes).
 *   W      bf16 [E][N][K], row-major.
 *   codes  u8   [E][N][K/2]       (out)
 *   sf     u8   nvfp4_sf_bytes(E*N, K), the E*N rows as one matrix (out)
 *   g      f32  [E][N]            (out)
 * Needs N % 128 == 0, K % 64 == 0, 64 <= K <= 4096.  Called for W1
 * (N = 2 d_ff, K = d) and W2 (N = d, K = d_ff).  Two launches on `stream`:
 * the row quantiser, then a fix-up pass that encodes the rare rows whose
 * outer scale lies outside [2^-87, 2^111] (row maxima below about 1.7e-23
 * or above about 7e36), which the first leaves. */
int moe_nvfp4_quantize_weights(const uint16_t* W, int E, int N, int K,
                               uint8_t* codes, uint8_t* sf, float* g,
                               int* status, void* stream);

/* NVFP4 quantisation of expert weights with ONE outer scale per expert
 * weight tensor (Technical Report section 4.3 table, "miniTE CUTLASS"
 * column, recipe nvfp4_cursor2_cutlass_v2; the per-row variant above is the
 * "miniTE per-token" column).  g_e = max|W_e| / (6 * 448); block scales and
 * codes follow the section 5.1 equation with that g_e for every row of
 * expert e.  g_e is written replicated into g[e][0..N-1], so the grouped
 * GEMMs consume the result unchanged (their epilogue multiplies by
 * g_x * g_w of the row).
 *   W, codes, sf, g, shapes   as moe_nvfp4_quantize_weights
 *   amax_e f32 [E]  (out) max |W_e| of each expert; also the accumulator of
 *                   the reduction, so it must not alias W, codes, sf or g
 * Three launches and one memset on `stream`: zero amax_e, per-expert
 * maximum (integer atomicMax on the bits of non-negative floats), then the
 * row quantiser and its fix-up pass (as moe_nvfp4_quantize_weights).  NaN/Inf weights set MOE_STATUS_NONFINITE_WEIGHT; NaNs do not
 * enter the maximum.  Errors as moe_nvfp4_quantize_weights, plus
 * MOE_ERR_CUDA if the memset cannot be enqueued. */
int moe_nvfp4_quantize_weights_per_expert(const uint16_t* W, int E, int N,
                                          int K, uint8_t* codes, uint8_t* sf,
                                          float* g, float* amax_e, int* status,
                                          void* stream);

/* Route, permute, pad, expert offsets, and per-token amax gathered in the
 * same pass (rainbus summary, method step 6: sort fused with the amax scan,
 * padding carries the statistics; AI summary methodology: no separate amax
 * scan).
 *   logits        f32 [T][E], or NULL to replay routing from ext_ids/ext_w
 *   ext_ids/ext_w i32/f32 [T][k]: replayed routing (ids strictly ascending per
 *                 token), used only when logits == NULL
 *   x             bf16 [T][d], or NULL to skip amax (then d is ignored and
 *                 amax_tok/amax_row may be NULL)
 *   topk_ids      i32 [T][k] (out) ascending expert ids = slot order
 *   topk_w        f32 [T][k] (out) renormalised router weights
 *   counts        i32 [E]    (out) routed rows per expert
 *   offsets       i32 [E+1]  (out) padded exclusive prefix; offsets[E] = M_pad
 *   row_to_token  i32 [M_cap](out) token of each row, -1 on pad rows and on
 *                 rows >= M_pad
 *   token_slot_row i32 [T][k](out) row of slot (t, j)
 *   amax_tok      f32 [T]    (out) max |x_t|
 *   amax_row      f32 [M_cap](out) amax_tok of the row's token, 0 on pad rows
 *   ws            device scratch of moe_permute_workspace_bytes(T, E) bytes */
int moe_permute_amax(const float* logits, const int32_t* ext_ids,
                     const float* ext_w, const uint16_t* x, int T, int E,
                     int k, int d, int32_t* topk_ids, float* topk_w,
                     int32_t* counts, int32_t* offsets, int32_t* row_to_token,
                     int32_t* token_slot_row, float* amax_tok, float* amax_row,
                     void* ws, size_t ws_bytes, int* status, void* stream);

/* moe_permute_amax without a workspace argument, for callers that cannot
 * allocate device memory: a plugin of another runtime that owns all device
 * memory and passes in only its buffers and a stream, or a serving loop that
 * must not call cudaMalloc (which can synchronise the device) on its hot
 * path.  The paper has no counterpart of this entry point: it is a library
 * convenience.
 *
 * Arguments and results are those of moe_permute_amax.  The chunk-histogram
 * scratch lives in a fixed MOE_PERMUTE_NOALLOC_SCRATCH_BYTES array inside
 * the library, held on every GPU that loads the library until the process
 * exits; nothing is allocated or freed.  Shapes whose scratch,
 * moe_permute_workspace_bytes(T, E), exceeds that size return
 * MOE_ERR_WORKSPACE before any CUDA call (with 4 MiB: T up to 524288 tokens
 * at E = 128, 65536 at E = 1024).
 *
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress); no address is kept between calls, so a
 * cudaDeviceReset in the process, after which the array may sit elsewhere,
 * does not leave a stale pointer.  The first call on a device may load the
 * library's device code there: make it before any stream capture.  All
 * calls share the one array, so calls whose GPU work overlaps (other streams
 * or host threads at the same time) race and give wrong results: serialise
 * them.  The array needs no clearing between calls. */
#define MOE_PERMUTE_NOALLOC_SCRATCH_BYTES (1 << 22)
int moe_permute_amax_noalloc(const float* logits, const int32_t* ext_ids,
                             const float* ext_w, const uint16_t* x, int T,
                             int E, int k, int d, int32_t* topk_ids,
                             float* topk_w, int32_t* counts, int32_t* offsets,
                             int32_t* row_to_token, int32_t* token_slot_row,
                             float* amax_tok, float* amax_row, int* status,
                             void* stream);

/* Quantise rows into the GEMM's buffers (Technical Report section 5.1
 * equation; AI summary methodology: codes, block scales and outer scales are
 * written straight into the contiguous buffers the GEMM consumes).
 *   src      bf16 [src_rows][K]
 *   row_map  i32 [dst_rows]: destination row r takes source row row_map[r];
 *            a negative entry writes an all-zero row; NULL = identity
 *   amax     f32 [src_rows] outer-scale arguments, NULL = computed per row
 *   codes    u8 [dst_rows][K/2], sf nvfp4_sf_bytes(dst_rows, K), g f32
 *            [dst_rows] (out)
 * Needs K % 64 == 0, 64 <= K <= 4096.  Two launches on `stream` (the row
 * quantiser and its fix-up pass, as moe_nvfp4_quantize_weights). */
int nvfp4_quantize_rows(const uint16_t* src, int src_rows, int K,
                        const int32_t* row_map, const float* amax,
                        int dst_rows, uint8_t* codes, uint8_t* sf, float* g,
                        int* status, void* stream);

/* Grouped FC1 with fused SwiGLU and requantisation (rainbus summary, core
 * method: native block-scaled MMA, FP32 epilogue broadcast of g_x g_w, BF16
 * cast; prerequisites: FC1 -> SwiGLU -> FC2).  Groups are the 128-row
 * aligned ranges [offsets[e], offsets[e+1]) read on the device; empty groups
 * are skipped.
 *   a_codes/a_sf/a_g  quantised activations, M_cap rows of K = d
 *   w1_codes/w1_sf/w1_g  from moe_nvfp4_quantize_weights(W1, E, 2 d_ff, d)
 *   h_codes/h_sf/h_g  quantised h, M_cap rows of K = d_ff (out; rows >=
 *                     offsets[E] untouched)
 *   dbg_u_f32  f32 [M_cap][2 d_ff] pre-cast FC1 outputs, or NULL
 *   dbg_h      bf16 [M_cap][d_ff] h before requantisation, or NULL
 *   ws         nvfp4_fc1_workspace_bytes(d_ff) bytes of device scratch
 * Launch: where A fits resident beside the pipeline (d <= 2048), the kernel
 * runs on pairs of CTAs (clusters of two, cta_group::2 MMAs covering two
 * 128-row tiles and a chunk's gate and up columns); elsewhere on single
 * CTAs.  Both give the same bits.  The environment variable
 * MOE_FC1_CTA_PAIRS=0, read at each launch, selects single CTAs throughout
 * (this entry point and the forwards). */
int nvfp4_grouped_gemm_fc1_swiglu(
    const uint8_t* a_codes, const uint8_t* a_sf, const float* a_g,
    const int32_t* offsets, int E, int64_t M_cap, int d, int d_ff,
    const uint8_t* w1_codes, const uint8_t* w1_sf, const float* w1_g,
    uint8_t* h_codes, uint8_t* h_sf, float* h_g, float* dbg_u_f32,
    uint16_t* dbg_h, void* ws, size_t ws_bytes, int* status, void* stream);

/* Grouped FC2 with the router-weighted epilogue, then the unpermute reduce
 * (two launches).  z = BF16(topk_w[t][j] * (acc * (g_h * g_w2))) of routed
 * row r = token_slot_row[t][j] goes to row r of `slots` (the slot (t, j) of
 * the combine, kept in routed-row order so that each 128-row tile leaves
 * the GEMM with whole-tile tensor stores), then out[t] = BF16(sum_j
 * FP32(slots[token_slot_row[t][j]])) in ascending j (= ascending expert
 * id).
 *   h_codes/h_sf/h_g  M_cap rows of K = d_ff
 *   w2_codes/w2_sf/w2_g from moe_nvfp4_quantize_weights(W2, E, d, d_ff)
 *   row_to_token, token_slot_row, topk_w from moe_permute_amax
 *   slots      bf16 [M_cap][d] (workspace, also an output): z by routed
 *              row; pad rows are written as zeros
 *   out        bf16 [T][d] (out)
 *   dbg_y_f32  f32 [M_cap][d] pre-weighting expert outputs y2, or NULL
 * Launch: where d is a multiple of 256 the GEMM runs on pairs of CTAs
 * (clusters of two, cta_group::2 MMAs covering two 128-row tiles and 256
 * output columns); elsewhere on single CTAs.  Both give the same bits.  The
 * environment variable MOE_FC2_CTA_PAIRS=0, read at each launch, selects
 * single CTAs throughout (this entry point, the forwards and the backward's
 * recomputation of FC2, whose dw then sums its columns in another grouping:
 * equal within FP32 reassociation, dy2 bit for bit). */
int nvfp4_grouped_gemm_fc2_unpermute(
    const uint8_t* h_codes, const uint8_t* h_sf, const float* h_g,
    const int32_t* offsets, int E, int64_t M_cap, int d_ff, int d,
    const uint8_t* w2_codes, const uint8_t* w2_sf, const float* w2_g,
    const int32_t* row_to_token, const int32_t* token_slot_row,
    const float* topk_w, int T, int k, uint16_t* slots, uint16_t* out,
    float* dbg_y_f32, int* status, void* stream);

/* The whole expert forward: route, permute + amax + quantise (x read once),
 * FC1 + SwiGLU + requantise, FC2 + router-weighted scatter, unpermute
 * reduce.  Seven launches on `stream` (route, chunk scan, pad rows, permute +
 * quantise, FC1, FC2, reduce), no host synchronisation (capturable in a CUDA
 * graph).
 *   x       bf16 [T][d];  logits f32 [T][E]
 *   w1_*, w2_* quantised weights as above
 *   out     bf16 [T][d] (out)
 *   ws      moe_expert_forward_workspace_bytes(...) bytes of device scratch;
 *           the intermediates stay there (see ..._workspace_layout) */
int moe_expert_forward(const uint16_t* x, const float* logits, int T, int E,
                       int k, int d, int d_ff, const uint8_t* w1_codes,
                       const uint8_t* w1_sf, const float* w1_g,
                       const uint8_t* w2_codes, const uint8_t* w2_sf,
                       const float* w2_g, uint16_t* out, void* ws,
                       size_t ws_bytes, int* status, void* stream);

/* moe_expert_forward that also records eight caller-owned CUDA events on
 * `stream` (cudaEvent_t handles passed as void*, created by the caller with
 * timing enabled): events[0] before the first launch and events[i] after the
 * i-th of the seven launches (route, chunk scan, pad rows, permute +
 * quantise, FC1, FC2, reduce), so that the caller can time each kernel on the
 * launching stream.  Same kernels, arguments, workspace and results as
 * moe_expert_forward (the pages have no counterpart: it serves measurement).
 * MOE_ERR_POINTER if events or one of its eight entries is NULL. */
int moe_expert_forward_timed(const uint16_t* x, const float* logits, int T,
                             int E, int k, int d, int d_ff,
                             const uint8_t* w1_codes, const uint8_t* w1_sf,
                             const float* w1_g, const uint8_t* w2_codes,
                             const uint8_t* w2_sf, const float* w2_g,
                             uint16_t* out, void* ws, size_t ws_bytes,
                             int* status, void* stream, void* const* events);

/* moe_expert_forward with gather-on-load FC1, a step toward the single-pass
 * fusion the pages name as future work (AI summary, "Future Directions":
 * fuse amax, quantisation and GEMM; main paper, section 5.6 "Exploring
 * Single-Pass Fusion", title only).  Each token is quantised ONCE: its codes
 * go to token row t of the x_codes workspace entry (rows 0..T-1, row T all
 * zero) instead of k row copies, and FC1's producer fetches the A rows of
 * each 128-row tile by row_to_token with TMA tile::gather4 (pad rows read
 * the zero row).  Block scales and g stay one copy per routed row (x_sf,
 * x_g), as in moe_expert_forward.  Same arguments, workspace and results
 * (bit for bit) as moe_expert_forward; only the content of the x_codes
 * workspace entry differs.  Needs d >= 256 (a code row must span the
 * 128-byte gather box), else MOE_ERR_SHAPE. */
int moe_expert_forward_gather(const uint16_t* x, const float* logits, int T,
                              int E, int k, int d, int d_ff,
                              const uint8_t* w1_codes, const uint8_t* w1_sf,
                              const float* w1_g, const uint8_t* w2_codes,
                              const uint8_t* w2_sf, const float* w2_g,
                              uint16_t* out, void* ws, size_t ws_bytes,
                              int* status, void* stream);

/* moe_expert_forward that also keeps what the straight-through backward
 * needs (main paper, contributions list: BF16 backward on saved operands;
 * Technical Report section 4.3, text below the table: the layer bypass saves
 * the original BF16 operands).  The forward's own results are identical.
 *   save_u   bf16 [M_cap][2 d_ff] (out) u = BF16(FC1 output), gate half first
 *   save_h   bf16 [M_cap][d_ff]   (out) h = BF16(silu(u_gate) u_up) before
 *            requantisation
 * Rows below offsets[E] are written (pad rows: u = h = 0); rows at or past
 * offsets[E] are untouched.  The routing, the permutation and the
 * requantised h that the backward needs stay in `ws`
 * (moe_expert_forward_workspace_layout entries 0, 1, 2, 4, 5, 10, 11, 12).
 * M_cap = moe_m_cap(T, E, k).  Errors as moe_expert_forward, plus
 * MOE_ERR_POINTER for a missing save buffer. */
int moe_expert_forward_train(const uint16_t* x, const float* logits, int T,
                             int E, int k, int d, int d_ff,
                             const uint8_t* w1_codes, const uint8_t* w1_sf,
                             const float* w1_g, const uint8_t* w2_codes,
                             const uint8_t* w2_sf, const float* w2_g,
                             uint16_t* out, void* ws, size_t ws_bytes,
                             uint16_t* save_u, uint16_t* save_h, int* status,
                             void* stream);

/* Straight-through BF16 backward of the expert layer (main paper,
 * contributions list; AI summary, "Methodology in Plain English": a
 * straight-through estimator on the saved BF16 activations and weights, no
 * backward quantisation; rainbus summary, method step 5: BF16 GEMMs on the
 * saved BF16 operands).  With u, h from moe_expert_forward_train, y2 the
 * forward's FP32 expert outputs and w = topk_w:
 *   dw[t][j]    = sum_n dY[t][n] y2[row(t,j)][n]                      (FP32)
 *   dlogits[t][ids[t][j]] = w_j (dw_j - sum_i w_i dw_i), 0 elsewhere   (FP32)
 *   dy2[row]    = BF16(RN_f32(w_tj dY[t]))                (BF16 GEMM operand)
 *   dh          = dy2 . W2_e                              (FP32 accumulate)
 *   du[gate]    = BF16(dh up s (1 + g (1 - s))), du[up] = BF16(dh g s),
 *                 g = u[gate], up = u[up], s = sigmoid(g) (BF16 GEMM operand)
 *   dW2_e       = dy2_e^T . h_e,   dW1_e = du_e^T . x_e   (FP32 out)
 *   dx[t]       = sum_j (du . W1_e)[row(t,j)], ascending j (FP32 out)
 * y2 is not stored by the forward: the backward recomputes it with the
 * forward's own FC2 kernel from the requantised h and the quantised W2
 * (bit-identical), taking the dot products with dY in that kernel's
 * epilogue.
 *   dY        bf16 [T][d];  x bf16 [T][d] (the forward's input)
 *   W1, W2    bf16 [E][2 d_ff][d], [E][d][d_ff]: the ORIGINAL weights
 *   w2_codes, w2_sf, w2_g   the quantised W2 the forward used
 *   topk_ids, topk_w, offsets, row_to_token, token_slot_row, h_codes, h_sf,
 *   h_g       the forward's routing, permutation and requantised h
 *             (moe_expert_forward_workspace_layout entries 0, 1, 4, 5, 2,
 *             10, 11, 12 of the training forward's workspace)
 *   u, h      the forward's saved values
 *   dx f32 [T][d], dW1 f32 [E][2 d_ff][d], dW2 f32 [E][d][d_ff],
 *   dw f32 [T][k] (out); dlogits f32 [T][E] (out, or NULL to skip)
 *   ws        moe_expert_backward_workspace_bytes(...) bytes
 * Eight launches (FC2 recomputation with dw and dy2, x rows, logits, four
 * tcgen05 BF16 grouped GEMMs, dx reduce), no host synchronisation.  All run
 * on `stream` but the x-row copy, which runs on a second stream the library
 * owns (one per host thread and device, created on first use), forked from
 * `stream` after the FC2 recomputation and joined back before the dW1 GEMM
 * by events, so that it overlaps the GEMMs before it; MOE_BWD_SIDE_STREAM=0
 * in the environment keeps it on `stream` (same results bit for bit).  The
 * call is complete, for `stream`, when its last launch is.  Experts without
 * rows get zero weight gradients.
 * Errors: MOE_ERR_SHAPE as moe_expert_forward, MOE_ERR_POINTER,
 * MOE_ERR_WORKSPACE, MOE_ERR_DEVICE, MOE_ERR_CUDA; a wait that runs out sets
 * MOE_STATUS_TIMEOUT. */
int moe_expert_backward(const uint16_t* dY, const uint16_t* x, int T, int E,
                        int k, int d, int d_ff, const uint16_t* W1,
                        const uint16_t* W2, const uint8_t* w2_codes,
                        const uint8_t* w2_sf, const float* w2_g,
                        const int32_t* topk_ids, const float* topk_w,
                        const int32_t* offsets, const int32_t* row_to_token,
                        const int32_t* token_slot_row, const uint16_t* u,
                        const uint16_t* h, const uint8_t* h_codes,
                        const uint8_t* h_sf, const float* h_g, float* dx,
                        float* dW1, float* dW2, float* dlogits, float* dw,
                        void* ws, size_t ws_bytes, int* status, void* stream);

/* ---------------------------------------------------------------------- */
/* Pipelined forward on host-resident batches (a runtime around the         */
/* entry points; the pages have no counterpart: it serves callers whose     */
/* token batches live in host memory).                                      */
/* ---------------------------------------------------------------------- */
#define MOE_PIPELINE_MAX_DEPTH 4

typedef struct moe_pipeline moe_pipeline;  /* opaque, owned by the library */

/* Device bytes moe_pipeline_create needs: `depth` slots of x (bf16 [T][d]),
 * logits (f32 [T][E]) and out (bf16 [T][d]), then one
 * moe_expert_forward_workspace_bytes workspace.  0 for an unsupported shape
 * (as moe_expert_forward, plus T >= 1 and 1 <= depth <=
 * MOE_PIPELINE_MAX_DEPTH). */
size_t moe_pipeline_device_bytes(int T, int E, int k, int d, int d_ff, int depth);

/* Create a pipeline on the current device over the caller's device buffer
 * (1024-byte aligned, at least moe_pipeline_device_bytes; owned by the
 * caller, who keeps it until moe_pipeline_destroy).  Creates three
 * non-blocking streams (copy-in, compute, copy-out) and three events per
 * slot; allocates no device memory.  Errors: MOE_ERR_POINTER (null `out` or
 * buffer, misaligned buffer), MOE_ERR_SHAPE, MOE_ERR_WORKSPACE,
 * MOE_ERR_CUDA. */
int moe_pipeline_create(int T, int E, int k, int d, int d_ff, int depth,
                        void* device_buffer, size_t bytes, moe_pipeline** out);

/* Enqueue one step and return: copy host_x (bf16 [T][d]) and host_logits
 * (f32 [T][E]) to the step's slot, run moe_expert_forward with the given
 * quantised weights (device pointers), copy the output to host_out (bf16
 * [T][d]).  Step i uses slot i % depth; its copy-in overlaps the forward of
 * step i - 1 and its copy-out the forward of step i + 1.  The host buffers
 * must stay untouched until moe_pipeline_synchronize returns (pinned memory
 * makes the copies asynchronous).  Must be called with the creating device
 * current (else MOE_ERR_DEVICE).  Errors as moe_expert_forward. */
int moe_pipeline_submit(moe_pipeline* p, const uint16_t* host_x,
                        const float* host_logits, uint16_t* host_out,
                        const uint8_t* w1_codes, const uint8_t* w1_sf,
                        const float* w1_g, const uint8_t* w2_codes,
                        const uint8_t* w2_sf, const float* w2_g, int* status);

/* Block until every submitted step, copies included, has finished. */
int moe_pipeline_synchronize(moe_pipeline* p);

/* Synchronize, then release the streams and events (not the buffer). */
int moe_pipeline_destroy(moe_pipeline* p);

#ifdef __cplusplus
}
#endif
#endif /* MOE_NVFP4_H */
