/*
 * MOE-NVFP4-SPEC-1 oracle (C++17, CPU).  TEST INFRASTRUCTURE ONLY: it is
 * loaded by tests/, by __graft_entry__.smoke() and by the CPU legs of
 * bench.py, never by the CUDA library.  Build flags: -O2 -ffp-contract=off
 * -fno-fast-math, no flush-to-zero, so every float operation below is one
 * IEEE binary32 operation rounded to nearest even.
 *
 * The method is an encoding followed by an approximate GEMM, so this file
 * restates its steps in the order the pages give them, one loop per step,
 * with no blocking or fusion.  Citation tags are defined in oracle.h.
 */
#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

float f32_from_bits(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
uint32_t bits_from_f32(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }

/* Value of a non-negative BF16 magnitude pattern, with the pattern just past
 * the largest finite value read as 2^128 (the value IEEE rounding compares
 * against when it decides between the largest finite number and infinity). */
double bf16_mag_value(uint32_t mag) {
    if (mag >= 0x7F80u) return std::ldexp(1.0, 128);
    return (double)f32_from_bits(mag << 16);
}

/* Nearest of the BF16 magnitudes {c-1, c, c+1} to a >= 0, ties to the even
 * pattern.  The caller guarantees the answer is among them. */
uint32_t bf16_nearest_mag(double a, uint32_t c) {
    uint32_t best = c;
    double best_d = std::fabs(bf16_mag_value(c) - a);
    const uint32_t cand[2] = {c + 1u, c == 0 ? c : c - 1u};
    for (uint32_t m : cand) {
        double dd = std::fabs(bf16_mag_value(m) - a);
        if (dd < best_d || (dd == best_d && (m & 1u) == 0u && (best & 1u) == 1u)) {
            best = m;
            best_d = dd;
        }
    }
    return best;
}

/* E2M1 magnitude from its three low bits: two exponent bits with bias 1 and
 * one mantissa bit; exponent 0 is subnormal (m * 0.5). */
double e2m1_mag(uint8_t code3) {
    const int e = (code3 >> 1) & 3;
    const int m = code3 & 1;
    if (e == 0) return 0.5 * m;
    return std::ldexp(1.0 + 0.5 * m, e - 1);
}

/* OCP E4M3 ("FN") magnitude from the seven low bits: four exponent bits with
 * bias 7, three mantissa bits, exponent 0 subnormal (m * 2^-9); the pattern
 * 0x7F is NaN and there is no infinity, so the largest finite value is
 * 0x7E = 1.75 * 2^8 = 448. */
double e4m3_mag(uint8_t code7) {
    const int e = (code7 >> 3) & 15;
    const int m = code7 & 7;
    if (e == 15 && m == 7) return std::nan("");
    if (e == 0) return std::ldexp((double)m, -9);
    return std::ldexp(1.0 + m / 8.0, e - 7);
}

}  // namespace

extern "C" {

float orc_bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

uint16_t orc_f32_to_bf16(float f) { return orc_f64_to_bf16((double)f); }

uint16_t orc_f64_to_bf16(double x) {
    if (std::isnan(x)) return 0x7FC0;
    const uint32_t sign = std::signbit(x) ? 0x8000u : 0u;
    const double a = std::fabs(x);
    if (std::isinf(a)) return (uint16_t)(sign | 0x7F80u);
    /* Bracket a: the float nearest to a truncated to its top 16 bits is
     * within one BF16 step of the answer. */
    const float f = (float)a;
    const uint32_t c = std::isinf(f) ? 0x7F7Fu : (bits_from_f32(f) >> 16);
    return (uint16_t)(sign | bf16_nearest_mag(a, c));
}

float orc_e2m1_value(uint8_t code) {
    const double m = e2m1_mag(code & 7);
    return (float)((code & 8) ? -m : m);
}

/* E2M1 round-to-nearest-even with saturation: the code whose value is
 * nearest to |q|, exact ties to the even code, |q| >= 6 gives 6; the sign bit
 * is the sign bit of q, so -0 and small negatives give 0x8 ([TR 5.1] Q_E2M1;
 * RNE from the execution specification; the sign of a zero code is a
 * reading: the pages leave it open). */
uint8_t orc_e2m1_encode(float q) {
    if (std::isnan(q)) return 0;  /* out of contract; the GPU flags it */
    const double a = std::fabs((double)q);
    uint8_t best = 7;
    if (a < 6.0) {
        double best_d = INFINITY;
        for (uint8_t c = 0; c < 8; ++c) {
            const double dd = std::fabs(e2m1_mag(c) - a);
            if (dd < best_d || (dd == best_d && (c & 1) == 0)) {
                best = c;
                best_d = dd;
            }
        }
    }
    return (uint8_t)(best | (std::signbit(q) ? 8 : 0));
}

float orc_e4m3_value(uint8_t code) {
    const double m = e4m3_mag(code & 0x7F);
    return (float)((code & 0x80) ? -m : m);
}

/* E4M3 round-to-nearest-even with saturation to the largest finite value,
 * for a non-negative block-scale argument t ([TR 5.1] Q_E4M3; subnormal
 * scales are kept).  Returns 0x7F (NaN) only for a NaN argument, which is out
 * of contract. */
uint8_t orc_e4m3_encode(float t) {
    if (std::isnan(t)) return 0x7F;
    const double a = (double)t;
    if (a >= 448.0) return 0x7E;
    uint8_t best = 0;
    double best_d = INFINITY;
    for (uint8_t c = 0; c <= 0x7E; ++c) {
        const double dd = std::fabs(e4m3_mag(c) - a);
        if (dd < best_d || (dd == best_d && (c & 1) == 0)) {
            best = c;
            best_d = dd;
        }
    }
    return best;
}

/* Block-scale storage: logical [row][K/16] bytes stored as 512-byte tiles of
 * 128 rows x 4 scale columns, tiles in row-group-major then K-group order;
 * inside a tile the byte of (r, c) sits at (r%32)*16 + ((r/32)%4)*4 + c%4.
 * This is the 1-D block-scale layout of the public tcgen05/cuBLAS
 * documentation; the pages only say the scales are written straight into the
 * buffers the GEMM consumes ([SUM-M]). */
int64_t orc_sf_offset(int64_t row, int64_t col, int64_t K) {
    const int64_t kgroups = K / 64;
    const int64_t tile = (row / 128) * kgroups + col / 4;
    return tile * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4 + (col % 4);
}

int64_t orc_sf_bytes(int64_t rows, int64_t K) {
    return ((rows + 127) / 128) * (K / 64) * 512;
}

void orc_unswizzle_sf(const uint8_t* sf_swz, int64_t rows, int K, uint8_t* logical) {
    for (int64_t r = 0; r < rows; ++r)
        for (int c = 0; c < K / 16; ++c)
            logical[r * (K / 16) + c] = sf_swz[orc_sf_offset(r, c, K)];
}

/* Largest padded row count the permutation can produce: every non-empty
 * expert adds fewer than 128 pad rows. */
int64_t orc_m_cap(int64_t T, int64_t E, int64_t k) {
    const int64_t routed = T * k;
    const int64_t nonempty = std::min<int64_t>(E, routed);
    const int64_t m = routed + 127 * nonempty;
    return ((m + 127) / 128) * 128;
}

/* Quantise one row v[0..K) with outer-scale argument amax ([TR 5.1] equation,
 * [RB-P] NVFP4 format, [RB-S] step 4):
 *   g   = amax / (6*448)
 *   s_b = Q_E4M3(a_b / (6 g))           a_b = max |v| over the 16-block
 *   S_b = g * s_b
 *   c_j = Q_E2M1(v_j / S_b)
 * Readings: amax == 0 gives g = 0, scales 0, codes +0; S_b == 0 gives codes
 * +0; the quotient is a true division (the equation divides by s_i d_ij).
 * Codes pack two per byte, even element in the low nibble. */
void orc_quantize_row(const float* v, int K, float amax, uint8_t* codes,
                      uint8_t* sf_logical, float* g_out) {
    const float g = amax / 2688.0f;
    *g_out = g;
    std::memset(codes, 0, (size_t)K / 2);
    std::memset(sf_logical, 0, (size_t)K / 16);
    if (amax == 0.0f) { *g_out = 0.0f; return; }
    const float den = 6.0f * g;
    for (int b = 0; b < K / 16; ++b) {
        float ab = 0.0f;
        for (int j = 0; j < 16; ++j) ab = std::max(ab, std::fabs(v[b * 16 + j]));
        const float tb = ab / den;
        const uint8_t sb = orc_e4m3_encode(tb);
        sf_logical[b] = sb;
        const float Sb = g * orc_e4m3_value(sb);
        if (Sb == 0.0f) continue;
        for (int j = 0; j < 16; ++j) {
            const int idx = b * 16 + j;
            const float q = v[idx] / Sb;
            const uint8_t c = orc_e2m1_encode(q);
            codes[idx / 2] |= (uint8_t)((idx % 2 == 0) ? c : (c << 4));
        }
    }
}

/* Per-row amax of BF16 rows (an exact maximum of magnitudes) ([TR 2.3],
 * [RB-S] step 4: g_x = max_k |X_{e,t,k}| / (6*448)). */
void orc_amax_rows_bf16(const uint16_t* x, int64_t rows, int K, float* amax) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float a = 0.0f;
        for (int j = 0; j < K; ++j)
            a = std::max(a, std::fabs(orc_bf16_to_f32(x[r * K + j])));
        amax[r] = a;
    }
}

/* Quantise dst_rows rows into the GEMM's buffers: destination row r takes
 * source row row_map[r] (identity when row_map is NULL); a negative map entry
 * is a pad row and comes out all zero ([SUM-M]: the quantiser writes codes,
 * block scales and outer scales straight into the contiguous GEMM buffers).
 * amax, when given, is per source row (gathered during permutation, [SUM-M]);
 * otherwise it is computed from the row.  sf_swz must hold
 * orc_sf_bytes(dst_rows, K) bytes; only bytes of rows < dst_rows are written. */
void orc_quantize_rows_bf16(const uint16_t* src, int64_t src_rows, int K,
                            const int32_t* row_map, const float* amax,
                            int64_t dst_rows, uint8_t* codes, uint8_t* sf_swz,
                            float* g) {
    (void)src_rows;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < dst_rows; ++r) {
        const int64_t s = row_map ? (int64_t)row_map[r] : r;
        std::vector<float> v((size_t)K, 0.0f);
        std::vector<uint8_t> sf((size_t)K / 16, 0);
        float gr = 0.0f;
        if (s >= 0) {
            float a = 0.0f;
            for (int j = 0; j < K; ++j) {
                v[j] = orc_bf16_to_f32(src[s * K + j]);
                a = std::max(a, std::fabs(v[j]));
            }
            if (amax) a = amax[s];
            orc_quantize_row(v.data(), K, a, codes + r * (K / 2), sf.data(), &gr);
        } else {
            std::memset(codes + r * (K / 2), 0, (size_t)K / 2);
        }
        g[r] = gr;
        for (int c = 0; c < K / 16; ++c) sf_swz[orc_sf_offset(r, c, K)] = sf[c];
    }
}

/* Reconstruction x^ = g * s_b * c in FP64 ([TR 2.2], [RB-P]). */
void orc_dequantize_rows(const uint8_t* codes, const uint8_t* sf_swz,
                         const float* g, int64_t rows, int K, double* out) {
    for (int64_t r = 0; r < rows; ++r)
        for (int j = 0; j < K; ++j) {
            const uint8_t byte = codes[r * (K / 2) + j / 2];
            const uint8_t c = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
            const uint8_t s = sf_swz[orc_sf_offset(r, j / 16, K)];
            out[r * K + j] = (double)g[r] * (double)orc_e4m3_value(s) *
                             (double)orc_e2m1_value(c);
        }
}

/* Router ([RB-P] MoE prerequisite: the router picks the top-k experts per
 * token; softmax over the selected logits).  Readings: ranking by (logit
 * descending, expert id ascending), so the lower id wins a tie; the k
 * selected ids are stored in ascending id order (the slot order j); the
 * weights are a softmax over the selected logits, evaluated in FP64 and
 * rounded once to FP32.  Returns -1 on a non-finite logit. */
int orc_route(const float* logits, int64_t T, int E, int k, int32_t* ids,
              float* w) {
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        std::vector<int32_t> order((size_t)E);
        std::iota(order.begin(), order.end(), 0);
        for (int e = 0; e < E; ++e)
            if (!std::isfinite(l[e])) bad = 1;
        std::stable_sort(order.begin(), order.end(),
                         [l](int32_t a, int32_t b) { return l[a] > l[b]; });
        std::vector<int32_t> sel(order.begin(), order.begin() + k);
        std::sort(sel.begin(), sel.end());
        const double m = (double)l[order[0]];
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += std::exp((double)l[sel[j]] - m);
        for (int j = 0; j < k; ++j) {
            ids[t * k + j] = sel[j];
            w[t * k + j] = (float)(std::exp((double)l[sel[j]] - m) / den);
        }
    }
    return bad ? -1 : 0;
}

/* Permutation, padding and expert offsets ([RB-P]: grouped GEMM needs
 * permutation, padding and expert offsets, groups may be uneven or empty;
 * [RB-S] step 6: device-side expert offsets).  Readings: each group is padded
 * to a multiple of 128 rows; inside a group rows follow ascending token order
 * (a stable counting sort).  row_to_token is -1 on pad rows and on rows from
 * the padded total up to m_cap.  Returns the padded total M_pad, or -1 if an
 * id is out of range or m_cap is too small. */
int orc_permute(const int32_t* ids, int64_t T, int E, int k, int64_t m_cap,
                int32_t* counts, int32_t* offsets, int32_t* row_to_token,
                int32_t* token_slot_row) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t i = 0; i < T * k; ++i) {
        if (ids[i] < 0 || ids[i] >= E) return -1;
        counts[ids[i]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + ((counts[e] + 127) / 128) * 128;
    if ((int64_t)offsets[E] > m_cap) return -1;
    for (int64_t r = 0; r < m_cap; ++r) row_to_token[r] = -1;
    std::vector<int32_t> next(offsets, offsets + E);
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            const int32_t e = ids[t * k + j];
            const int32_t r = next[e]++;
            row_to_token[r] = (int32_t)t;
            token_slot_row[t * k + j] = r;
        }
    return offsets[E];
}

/* Grouped block-scaled GEMM with the FP32 epilogue ([RB-C]: U_e =
 * MMA_NVFP4(X_e, W_e^T), then the epilogue multiplies by g_x g_w in FP32;
 * [SUM-M]: outer factors applied after the native block-scaled multiply, no
 * decoded BF16 operand).  For every row r of group e and column n:
 *   acc = +0; for k ascending: acc = acc + (c_a s_a)(c_w s_w)   (FP32)
 *   y[r][n] = acc * (g_a[r] * g_w[e][n])                          (FP32)
 * Every product of decoded codes and block scales is exact in FP32 (at most
 * 12 significant bits, magnitude in [2^-20, 2688^2]), so only the additions
 * round, in fixed k order.  Rows outside every group are left untouched. */
void orc_grouped_gemm(const uint8_t* a_codes, const uint8_t* a_sf_swz,
                      const float* a_g, const int32_t* offsets, int E,
                      int64_t M, int K, int N, const uint8_t* w_codes,
                      const uint8_t* w_sf_swz, const float* w_g, float* y) {
    (void)M;
    for (int e = 0; e < E; ++e) {
        const int64_t r0 = offsets[e], r1 = offsets[e + 1];
        if (r1 <= r0) continue;
        /* decoded weights of expert e: c_w * s_w per element */
        std::vector<float> wdec((size_t)N * K);
#pragma omp parallel for schedule(static)
        for (int n = 0; n < N; ++n) {
            const int64_t wr = (int64_t)e * N + n;
            for (int j = 0; j < K; ++j) {
                const uint8_t byte = w_codes[wr * (K / 2) + j / 2];
                const uint8_t c = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
                const uint8_t s = w_sf_swz[orc_sf_offset(wr, j / 16, K)];
                wdec[(size_t)n * K + j] = orc_e2m1_value(c) * orc_e4m3_value(s);
            }
        }
#pragma omp parallel for schedule(static)
        for (int64_t r = r0; r < r1; ++r) {
            std::vector<float> adec((size_t)K);
            for (int j = 0; j < K; ++j) {
                const uint8_t byte = a_codes[r * (K / 2) + j / 2];
                const uint8_t c = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
                const uint8_t s = a_sf_swz[orc_sf_offset(r, j / 16, K)];
                adec[j] = orc_e2m1_value(c) * orc_e4m3_value(s);
            }
            for (int n = 0; n < N; ++n) {
                const float* wv = &wdec[(size_t)n * K];
                float acc = 0.0f;
                for (int j = 0; j < K; ++j) acc = acc + adec[j] * wv[j];
                const float scale = a_g[r] * w_g[(int64_t)e * N + n];
                y[r * N + n] = acc * scale;
            }
        }
    }
}

/* FC1 output cast and SwiGLU ([RB-P]: expert FFN is FC1 -> SwiGLU -> FC2;
 * [SUM-M]: cast to BF16 at the end of the GEMM).  Readings: u = BF16(y);
 * gate = columns [0, F), up = columns [F, 2F);
 * h = BF16(silu(u_gate) * u_up) with silu(z) = z / (1 + e^-z), evaluated in
 * FP64 and rounded once.  u may be NULL. */
void orc_swiglu(const float* y, int64_t M, int F, uint16_t* u, uint16_t* h) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < M; ++r) {
        for (int j = 0; j < F; ++j) {
            const uint16_t ug = orc_f32_to_bf16(y[r * 2 * F + j]);
            const uint16_t uu = orc_f32_to_bf16(y[r * 2 * F + F + j]);
            if (u) {
                u[r * 2 * F + j] = ug;
                u[r * 2 * F + F + j] = uu;
            }
            const double zg = (double)orc_bf16_to_f32(ug);
            const double zu = (double)orc_bf16_to_f32(uu);
            const double s = zg / (1.0 + std::exp(-zg));
            h[r * F + j] = orc_f64_to_bf16(s * zu);
        }
    }
}

/* Router-weighted scatter after FC2 (execution-specification freedom named
 * on the pages: router coefficient placement and output cast; fixed here as
 * z = BF16(w_{t,e} * y2) in FP32, stored at slot (t, j)). */
void orc_combine(const float* y2, const int32_t* row_to_token,
                 const int32_t* token_slot_row, const float* topk_w,
                 int64_t T, int k, int64_t M, int d, uint16_t* slots) {
    (void)row_to_token;
    (void)M;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            const int64_t r = token_slot_row[t * k + j];
            const float w = topk_w[t * k + j];
            for (int n = 0; n < d; ++n)
                slots[(t * k + j) * d + n] = orc_f32_to_bf16(w * y2[r * d + n]);
        }
}

/* Unpermute and reduce: out[t] = BF16(sum over slots in ascending expert id
 * order, FP32, starting from the first slot). */
void orc_reduce(const uint16_t* slots, int64_t T, int k, int d, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int n = 0; n < d; ++n) {
            float s = orc_bf16_to_f32(slots[(t * k) * d + n]);
            for (int j = 1; j < k; ++j)
                s = s + orc_bf16_to_f32(slots[(t * k + j) * d + n]);
            out[t * d + n] = orc_f32_to_bf16(s);
        }
}

/* Smallest non-negative float bit pattern that encodes to `code` (binary
 * search over the monotone encoder), or -1 if the code is never produced. */
int64_t orc_e4m3_first_input_of_code(uint8_t code) {
    int64_t lo = 0, hi = 0x7F800000LL;  /* [0, +inf) */
    if (orc_e4m3_encode(f32_from_bits(0x7F7FFFFFu)) < code) return -1;
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (orc_e4m3_encode(f32_from_bits((uint32_t)mid)) >= code) hi = mid;
        else lo = mid + 1;
    }
    return orc_e4m3_encode(f32_from_bits((uint32_t)lo)) == code ? lo : -1;
}

int64_t orc_e2m1_first_input_of_code(uint8_t code) {
    if (code > 7) return -1;
    int64_t lo = 0, hi = 0x7F800000LL;
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (orc_e2m1_encode(f32_from_bits((uint32_t)mid)) >= code) hi = mid;
        else lo = mid + 1;
    }
    return orc_e2m1_encode(f32_from_bits((uint32_t)lo)) == code ? lo : -1;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops from now on (n >= 1); the results do not
   depend on it (each output is summed in a fixed order by one thread). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

}  // extern "C"

/* ---- contrast recipes ---- */

/* Blockwise 16-point random Hadamard transform ([SUM-M] contrast). */
void orc_rht16_rows(const float* x, int64_t rows, int K, const int8_t* signs16, float* y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int b = 0; b < K / 16; ++b) {
            const float* xb = x + r * K + 16 * b;
            float* yb = y + r * K + 16 * b;
            for (int i = 0; i < 16; ++i) {
                double acc = 0.0;
                for (int j = 0; j < 16; ++j) {
                    const int hij = (__builtin_popcount((unsigned)(i & j)) & 1) ? -1 : 1;
                    acc += (double)(hij * signs16[j]) * (double)xb[j];
                }
                yb[i] = (float)(acc * 0.25);
            }
        }
    }
}

/* One outer scale for the whole tensor ([RB-P] scale-granularity choice). */
void orc_quantize_tensor(const float* x, int64_t rows, int K, uint8_t* codes, uint8_t* sf_swz, float* g_out) {
    float a = 0.0f;
    for (int64_t i = 0; i < rows * (int64_t)K; ++i) a = std::max(a, std::fabs(x[i]));
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        std::vector<uint8_t> sf((size_t)K / 16, 0);
        float gr = 0.0f;
        orc_quantize_row(x + r * K, K, a, codes + r * (K / 2), sf.data(), &gr);
        g_out[r] = gr;
        for (int c = 0; c < K / 16; ++c) sf_swz[orc_sf_offset(r, c, K)] = sf[c];
    }
}

/* Per-expert weight outer scale ("miniTE CUTLASS", [TR 4.3] table). */
void orc_quantize_weights_per_expert(const uint16_t* W, int E, int N, int K, uint8_t* codes, uint8_t* sf_swz,
                                     float* g) {
    for (int e = 0; e < E; ++e) {
        float a = 0.0f;
        const uint16_t* we = W + (int64_t)e * N * K;
        for (int64_t i = 0; i < (int64_t)N * K; ++i) a = std::max(a, std::fabs(orc_bf16_to_f32(we[i])));
#pragma omp parallel for schedule(static)
        for (int n = 0; n < N; ++n) {
            const int64_t r = (int64_t)e * N + n;
            std::vector<float> v((size_t)K);
            std::vector<uint8_t> sf((size_t)K / 16, 0);
            for (int j = 0; j < K; ++j) v[j] = orc_bf16_to_f32(we[(int64_t)n * K + j]);
            float gr = 0.0f;
            orc_quantize_row(v.data(), K, a, codes + r * (K / 2), sf.data(), &gr);
            g[r] = gr;
            for (int c = 0; c < K / 16; ++c) sf_swz[orc_sf_offset(r, c, K)] = sf[c];
        }
    }
}

/* ---- backward ---- */

void orc_bwd_router(const uint16_t* dY, const float* y2, const float* w, const int32_t* ids,
                    const int32_t* token_slot_row, int64_t T, int k, int d, int E, float* dw, float* dlogits) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        std::vector<double> g((size_t)k);
        for (int j = 0; j < k; ++j) {
            const int64_t r = token_slot_row[t * k + j];
            double s = 0.0;
            for (int n = 0; n < d; ++n) s += (double)orc_bf16_to_f32(dY[t * d + n]) * (double)y2[r * d + n];
            g[j] = s;
            dw[t * k + j] = (float)s;
        }
        double mean = 0.0;
        for (int j = 0; j < k; ++j) mean += (double)w[t * k + j] * g[j];
        for (int e = 0; e < E; ++e) dlogits[t * E + e] = 0.0f;
        for (int j = 0; j < k; ++j) dlogits[t * E + ids[t * k + j]] = (float)((double)w[t * k + j] * (g[j] - mean));
    }
}

void orc_bwd_dy2(const uint16_t* dY, const float* w, const int32_t* token_slot_row, int64_t T, int k, int d,
                 int64_t M, uint16_t* dy2) {
    for (int64_t i = 0; i < M * d; ++i) dy2[i] = 0;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            const int64_t r = token_slot_row[t * k + j];
            const float wj = w[t * k + j];
            for (int n = 0; n < d; ++n) {
                const float p = wj * orc_bf16_to_f32(dY[t * d + n]);  // one FP32 rounding
                dy2[r * d + n] = orc_f32_to_bf16(p);
            }
        }
}

void orc_bwd_expert(const uint16_t* dy2, const uint16_t* u, const uint16_t* h, const uint16_t* xr, int64_t n,
                    int d, int F, const uint16_t* W1, const uint16_t* W2, uint16_t* du, double* dxr, float* dW1,
                    float* dW2) {
    const int F2 = 2 * F;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        std::vector<double> dh((size_t)F, 0.0);
        for (int m = 0; m < d; ++m) {
            const double a = orc_bf16_to_f32(dy2[r * d + m]);
            if (a == 0.0) continue;
            for (int f = 0; f < F; ++f) dh[f] += a * (double)orc_bf16_to_f32(W2[(int64_t)m * F + f]);
        }
        for (int f = 0; f < F; ++f) {
            const double g = orc_bf16_to_f32(u[r * F2 + f]);
            const double v = orc_bf16_to_f32(u[r * F2 + F + f]);
            const double s = 1.0 / (1.0 + std::exp(-g));
            du[r * F2 + f] = orc_f64_to_bf16(dh[f] * v * s * (1.0 + g * (1.0 - s)));
            du[r * F2 + F + f] = orc_f64_to_bf16(dh[f] * g * s);
        }
        for (int i = 0; i < d; ++i) dxr[r * d + i] = 0.0;
        for (int j = 0; j < F2; ++j) {
            const double a = orc_bf16_to_f32(du[r * F2 + j]);
            if (a == 0.0) continue;
            for (int i = 0; i < d; ++i) dxr[r * d + i] += a * (double)orc_bf16_to_f32(W1[(int64_t)j * d + i]);
        }
    }
#pragma omp parallel for schedule(static)
    for (int m = 0; m < d; ++m) {
        std::vector<double> acc((size_t)F, 0.0);
        for (int64_t r = 0; r < n; ++r) {
            const double a = orc_bf16_to_f32(dy2[r * d + m]);
            if (a == 0.0) continue;
            for (int f = 0; f < F; ++f) acc[f] += a * (double)orc_bf16_to_f32(h[r * F + f]);
        }
        for (int f = 0; f < F; ++f) dW2[(int64_t)m * F + f] = (float)acc[f];
    }
#pragma omp parallel for schedule(static)
    for (int j = 0; j < F2; ++j) {
        std::vector<double> acc((size_t)d, 0.0);
        for (int64_t r = 0; r < n; ++r) {
            const double a = orc_bf16_to_f32(du[r * F2 + j]);
            if (a == 0.0) continue;
            for (int i = 0; i < d; ++i) acc[i] += a * (double)orc_bf16_to_f32(xr[r * d + i]);
        }
        for (int i = 0; i < d; ++i) dW1[(int64_t)j * d + i] = (float)acc[i];
    }
}
