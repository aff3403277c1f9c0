// Routing, permutation, padding and expert offsets with per-token amax
// gathered in the same pass (rainbus summary, prerequisites "MoE and grouped
// GEMM": router top-k, permutation, padding, expert offsets, uneven and empty
// groups; method step 6: sort fused with the amax scan, padding carries the
// statistics, device-side expert offsets).
//
// The permutation is a deterministic stable counting sort with no
// arrival-order atomics: per 64-token chunk, a bitmask per expert records
// which tokens chose it (atomicOr is order-independent), a token's rank in
// its expert is a popcount of the lower bits, chunk histograms are scanned
// once, and a row is offsets[e] + chunk base + rank.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kChunk = kRouteChunk;

// Order-preserving map of a float (finite or -inf, with -0 taken as +0) to
// an unsigned key: a > b as floats iff key(a) > key(b).
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// One CTA per chunk of kChunk tokens, kChunk / 8 warps (8 tokens each), one
// warp per token at a time.  Small chunks spread the tokens evenly over the
// SMs (1024 CTAs for 64k tokens).
constexpr int kRouteThreads = kChunk * 4;
template <int NPL>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const float* __restrict__ logits,
                                                   const int32_t* __restrict__ ext_ids,
                                                   const float* __restrict__ ext_w, int T, int E, int k,
                                                   int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
                                                   int32_t* __restrict__ rank_out, int32_t* __restrict__ hist,
                                                   int* status) {
  extern __shared__ uint32_t mask[];  // [E][kChunk/32]
  constexpr int W = kChunk / 32;
  const int c = blockIdx.x;
  const int t0 = c * kChunk;
  for (int i = threadIdx.x; i < E * W; i += blockDim.x) mask[i] = 0u;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float NEG_INF = __uint_as_float(0xFF800000u);
  const int tstep = blockDim.x / 32;
  // the warp's next token's logits are loaded while it routes the current one
  float nxt[NPL];
  auto load_logits = [&](int t) {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      nxt[i] = e < E ? __ldg(logits + (int64_t)t * E + e) : NEG_INF;
    }
  };
  if (logits && t0 + warp < T) load_logits(t0 + warp);
  for (int tl = warp; tl < kChunk; tl += tstep) {
    const int t = t0 + tl;
    if (t >= T) break;
    int my_id = 0x7FFFFFFF;
    float my_w = 0.0f;
    if (logits) {
      float v[NPL];
      bool fin = true;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const float x = nxt[i];
        v[i] = NEG_INF;
        if (i * 32 + lane < E) {
          if (is_finite_f32(x)) v[i] = x; else fin = false;
        }
      }
      if (tl + tstep < kChunk && t + tstep < T) load_logits(t + tstep);
      if (!__all_sync(0xFFFFFFFFu, fin) && lane == 0) set_status(status, MOE_STATUS_NONFINITE_LOGITS);
      // k rounds: the lane's best untaken logit (its ids ascend with i, so
      // the first of equal keys has the smaller id), then the warp's largest
      // key and, among lanes holding it, the smallest id -- two redux.sync
      // maxima (logit descending, id ascending).
      uint32_t key[NPL];
#pragma unroll
      for (int i = 0; i < NPL; ++i) key[i] = (i * 32 + lane < E) ? order_key(v[i]) : 0u;
      float my_v = NEG_INF, vmax = NEG_INF;
      if constexpr (NPL <= 4) {
        // The lane's keys sorted once, largest first and, among equal keys,
        // smaller id first (ids differ, so the order is total); absent
        // experts carry key 0, below every logit, and sort last.  Each round
        // the heads compete and the winning lane pops its head, so a lane's
        // head is always its best untaken key, as the rescan below finds it.
        uint32_t sk[NPL];
        int si[NPL];
#pragma unroll
        for (int i = 0; i < NPL; ++i) { sk[i] = key[i]; si[i] = i; }
        auto order = [&](int a, int b) {  // (sk[a], si[a]) before (sk[b], si[b])
          if (sk[b] > sk[a] || (sk[b] == sk[a] && si[b] < si[a])) {
            const uint32_t tk = sk[a]; sk[a] = sk[b]; sk[b] = tk;
            const int ti = si[a]; si[a] = si[b]; si[b] = ti;
          }
        };
        if constexpr (NPL == 2) order(0, 1);
        if constexpr (NPL == 4) { order(0, 1); order(2, 3); order(0, 2); order(1, 3); order(1, 2); }
        for (int j = 0; j < k; ++j) {
          const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, sk[0]);  // a present expert's key: E >= k
          const uint32_t hid = (uint32_t)(si[0] * 32 + lane);
          const uint32_t my_inv = sk[0] == mk ? 0xFFFFFFFFu - hid : 0u;
          const int be = (int)(0xFFFFFFFFu - __reduce_max_sync(0xFFFFFFFFu, my_inv));
          if (sk[0] == mk && (int)hid == be) {
#pragma unroll
            for (int i = 0; i + 1 < NPL; ++i) { sk[i] = sk[i + 1]; si[i] = si[i + 1]; }
            sk[NPL - 1] = 0u;
          }
          const float bv = key_value(mk);
          if (lane == j) { my_id = be; my_v = bv; }
          if (j == 0) vmax = bv;
        }
      } else {
        uint32_t taken = 0u;
        for (int j = 0; j < k; ++j) {
          uint32_t bk = 0u;
          int bi = -1;
#pragma unroll
          for (int i = 0; i < NPL; ++i)
            if (!((taken >> i) & 1u) && (bi < 0 || key[i] > bk) && i * 32 + lane < E) { bk = key[i]; bi = i; }
          const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, bi >= 0 ? bk : 0u);
          const uint32_t my_inv = (bi >= 0 && bk == mk) ? 0xFFFFFFFFu - (uint32_t)(bi * 32 + lane) : 0u;
          const int be = (int)(0xFFFFFFFFu - __reduce_max_sync(0xFFFFFFFFu, my_inv));
          if (bi >= 0 && bi * 32 + lane == be) taken |= 1u << bi;
          const float bv = key_value(mk);
          if (lane == j) { my_id = be; my_v = bv; }
          if (j == 0) vmax = bv;
        }
      }
      // softmax over the selected logits (FP32)
      float ex = (lane < k) ? expf(my_v - vmax) : 0.0f;
      float den = ex;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, o);
      my_w = (lane < k) ? __fdiv_rn(ex, den) : 0.0f;
    } else {
      // routing replay: ids must lie in [0, E) and be strictly ascending
      if (lane < k) {
        my_id = ext_ids[(int64_t)t * k + lane];
        my_w = ext_w[(int64_t)t * k + lane];
      }
      const int prev = __shfl_up_sync(0xFFFFFFFFu, my_id, 1);
      const bool bad = lane < k && (my_id < 0 || my_id >= E || (lane > 0 && prev >= my_id));
      if (__any_sync(0xFFFFFFFFu, bad)) {
        if (lane == 0) set_status(status, MOE_STATUS_BAD_ROUTING);
        if (lane < k) my_id = min(max(my_id, 0), E - 1);  // stay in bounds
      }
    }
    // slot order = ascending expert id
    int pos = 0;
    for (int i = 0; i < k; ++i) pos += (__shfl_sync(0xFFFFFFFFu, my_id, i) < my_id) ? 1 : 0;
    if (lane < k) {
      topk_ids[(int64_t)t * k + pos] = my_id;
      topk_w[(int64_t)t * k + pos] = my_w;
      atomicOr(&mask[my_id * W + (tl >> 5)], 1u << (tl & 31));
    }
  }
  __syncthreads();
  // in-chunk rank of each (token, slot): tokens of the chunk that chose the
  // same expert and come earlier
  for (int tl = threadIdx.x; tl < kChunk; tl += blockDim.x) {
    const int t = t0 + tl;
    if (t >= T) break;
    for (int j = 0; j < k; ++j) {
      const int e = topk_ids[(int64_t)t * k + j];
      int rank = __popc(mask[e * W + (tl >> 5)] & ((1u << (tl & 31)) - 1u));
      for (int w = 0; w < (tl >> 5); ++w) rank += __popc(mask[e * W + w]);
      rank_out[(int64_t)t * k + j] = rank;
    }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int h = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) h += __popc(mask[e * W + w]);
    hist[(int64_t)c * E + e] = h;
  }
}

int launch_route(const float* logits, const int32_t* ext_ids, const float* ext_w, int T, int E, int k,
                 int32_t* topk_ids, float* topk_w, int32_t* token_slot_row, int32_t* hist, int* status,
                 cudaStream_t stream) {
  const int C = (T + kChunk - 1) / kChunk;
  if (C == 0) return 0;
  const size_t smem = (size_t)E * (kChunk / 32) * sizeof(uint32_t);
  const int npl = (E + 31) / 32;
#define MOE_ROUTE(N)                                                                                 \
  route_kernel<N><<<C, kRouteThreads, smem, stream>>>(logits, ext_ids, ext_w, T, E, k, topk_ids, topk_w, \
                                           token_slot_row, hist, status)
  if (npl <= 1) MOE_ROUTE(1);
  else if (npl <= 2) MOE_ROUTE(2);
  else if (npl <= 4) MOE_ROUTE(4);
  else if (npl <= 8) MOE_ROUTE(8);
  else if (npl <= 16) MOE_ROUTE(16);
  else MOE_ROUTE(32);
#undef MOE_ROUTE
  return 0;
}

// One CTA of 256 threads per expert e: the exclusive scan of the expert's
// chunk counts over the chunks (written back in place as chunk bases) and
// the expert's total (counts[e]).  The padded offsets follow in
// pad_rows_kernel, which needs them first.
__global__ void __launch_bounds__(256) scan_kernel(int32_t* __restrict__ hist, int C, int E,
                                                   int32_t* __restrict__ counts) {
  __shared__ int warp_sum[8];
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int run = 0;
  // rounds of 1024 chunks: thread i takes chunks 4i .. 4i+3 of the round,
  // whose four loads go out together
  for (int base = 0; base < C; base += 1024) {
    const int c0 = base + 4 * threadIdx.x;
    int v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = c0 + q < C ? hist[(int64_t)(c0 + q) * E + e] : 0;
    const int own = v[0] + v[1] + v[2] + v[3];
    // inclusive scan of the threads' sums within the warp, then across the 8 warps
    int x = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sum[wid] = x;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int ws = warp_sum[w];
      before += w < wid ? ws : 0;
      total += ws;
    }
    int ex = run + before + x - own;  // exclusive prefix of chunk c0
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (c0 + q < C) hist[(int64_t)(c0 + q) * E + e] = ex;
      ex += v[q];
    }
    run += total;
    __syncthreads();  // warp_sum is rewritten by the next round
  }
  if (threadIdx.x == 0) counts[e] = run;
}

int launch_scan(int32_t* hist, int C, int E, int32_t* counts, cudaStream_t stream) {
  if (E < 1) return 0;
  scan_kernel<<<E, 256, 0, stream>>>(hist, C, E, counts);
  return 0;
}

__device__ __forceinline__ int slot_row(int e, int t, int rank, const int32_t* __restrict__ hist,
                                        const int32_t* __restrict__ offsets, int E) {
  return offsets[e] + hist[(int64_t)(t / kChunk) * E + e] + rank;
}

// One warp per token: final rows of its slots, and per-token amax of x read
// with 128-bit loads and a warp-shuffle max.
__global__ void __launch_bounds__(256) permute_amax_kernel(
    const int32_t* __restrict__ topk_ids, int32_t* __restrict__ tsr, const int32_t* __restrict__ hist,
    const int32_t* __restrict__ offsets, int T, int E, int k, const uint16_t* __restrict__ x, int d,
    int32_t* __restrict__ row_to_token, float* __restrict__ amax_tok, float* __restrict__ amax_row, int* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  int row = -1;
  if (lane < k) {
    const int64_t i = (int64_t)t * k + lane;
    row = slot_row(topk_ids[i], t, tsr[i], hist, offsets, E);
    tsr[i] = row;
    row_to_token[row] = t;
  }
  if (x) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)t * d);
    float a = 0.0f;
    bool fin = true;
    for (int i = lane; i < d / 8; i += 32) {
      const uint4 v = __ldg(xr + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        fin = fin && bf16x2_finite(w[q]);
        a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[q])), fabsf(bf16_hi(w[q]))));
      }
    }
    if (!__all_sync(0xFFFFFFFFu, fin) && lane == 0) set_status(status, MOE_STATUS_NONFINITE_X);
    a = warp_max(a);
    if (lane == 0 && amax_tok) amax_tok[t] = a;
    if (lane < k && amax_row) amax_row[row] = a;
  }
}

int launch_permute_amax(const int32_t* topk_ids, int32_t* token_slot_row, const int32_t* hist, const int32_t* offsets,
                        int T, int E, int k, const uint16_t* x, int d, int32_t* row_to_token, float* amax_tok,
                        float* amax_row, int* status, cudaStream_t stream) {
  if (T == 0) return 0;
  permute_amax_kernel<<<(T + 7) / 8, 256, 0, stream>>>(topk_ids, token_slot_row, hist, offsets, T, E, k, x, d,
                                                      row_to_token, amax_tok, amax_row, status);
  return 0;
}

// First the padded offsets, which every block computes for itself from the
// counts: off_e = sum over e' < e of ceil(count_e' / 128) * 128 (block e
// writes offsets[e + 1], block 0 also offsets[0] = 0).  Then blocks [0, E):
// the pad rows of group e (fewer than 128); blocks >= E: rows from the
// padded total up to m_cap (maps only; the GEMMs never read them).
__global__ void __launch_bounds__(128) pad_rows_kernel(int32_t* __restrict__ offsets,
                                                       const int32_t* __restrict__ counts, int E, int64_t m_cap,
                                                       int32_t* __restrict__ row_to_token, float* __restrict__ amax_row,
                                                       uint8_t* __restrict__ codes, int K, uint8_t* __restrict__ sf,
                                                       float* __restrict__ g) {
  __shared__ int part_before[4], part_all[4];
  const int me = (int)blockIdx.x < E ? (int)blockIdx.x : E;  // the group whose start this block needs
  int before = 0, all = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    const int pc = (counts[i] + 127) & ~127;
    all += pc;
    if (i < me) before += pc;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xFFFFFFFFu, before, o);
    all += __shfl_xor_sync(0xFFFFFFFFu, all, o);
  }
  if ((threadIdx.x & 31) == 0) {
    part_before[threadIdx.x >> 5] = before;
    part_all[threadIdx.x >> 5] = all;
  }
  __syncthreads();
  const int64_t off_me = (int64_t)part_before[0] + part_before[1] + part_before[2] + part_before[3];
  const int64_t total = (int64_t)part_all[0] + part_all[1] + part_all[2] + part_all[3];
  if ((int)blockIdx.x < E) {
    const int e = blockIdx.x;
    const int cnt = counts[e];
    const int64_t end = off_me + ((cnt + 127) & ~127);
    if (threadIdx.x == 0) {
      offsets[e + 1] = (int32_t)end;
      if (e == 0) offsets[0] = 0;
    }
    // the group's pad rows [p0, end) are contiguous: their codes are zeroed
    // by the whole block with coalesced 16-byte stores, their scale words
    // (one per 64 columns, scattered over the 128 x 4 tiles) spread over
    // the threads
    const int64_t p0 = off_me + cnt;
    const int np = (int)(end - p0);
    if (threadIdx.x < np) {
      const int64_t r = p0 + threadIdx.x;
      row_to_token[r] = -1;
      if (amax_row) amax_row[r] = 0.0f;
      if (sf) g[r] = 0.0f;
    }
    if (codes && np > 0) {
      uint4* cr = reinterpret_cast<uint4*>(codes + p0 * (K / 2));
      const int n16 = np * (K / 32);
      for (int i = threadIdx.x; i < n16; i += blockDim.x) cr[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (sf && np > 0) {
      const int kg = K / 64;
      for (int i = threadIdx.x; i < np * kg; i += blockDim.x) {
        const int64_t r = p0 + i / kg;
        const int c4 = i % kg;
        *reinterpret_cast<uint32_t*>(sf + ((r >> 7) * kg + c4) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4) = 0u;
      }
    }
  } else {
    for (int64_t r = total + (int64_t)(blockIdx.x - E) * blockDim.x + threadIdx.x; r < m_cap;
         r += (int64_t)(gridDim.x - E) * blockDim.x) {
      row_to_token[r] = -1;
      if (amax_row) amax_row[r] = 0.0f;
    }
  }
}

int launch_pad_rows(int32_t* offsets, const int32_t* counts, int E, int64_t m_cap, int32_t* row_to_token,
                    float* amax_row, uint8_t* codes, int K, uint8_t* sf, float* g, cudaStream_t stream) {
  pad_rows_kernel<<<E + 64, 128, 0, stream>>>(offsets, counts, E, m_cap, row_to_token, amax_row, codes, K, sf, g);
  return 0;
}

// One warp per token: rows of its k slots, amax of x (read once into
// registers), quantisation, and the same codes / block scales / outer scale
// written into each of the k destination rows.  With tok_codes set, the
// codes go once to token row t of tok_codes instead (the grouped GEMM then
// gathers them by row_to_token); scales and g still go to the k rows.  Lane L holds, for each group
// of 1024 columns, the 32 consecutive columns from 32*L (two whole 16-element
// blocks), so a block never spans lanes, its codes go out as one 16-byte
// store per row, and lanes L, L ^ 1 together form one 32-bit scale word.
// Codes (cw, one 16-byte word per group of 32 columns) and block-scale
// words (sfw, the lane pair's four scales) of a token's row held in
// registers, from its blocks' magnitude maxima bm and outer scale gs.
template <int NG>
__device__ __forceinline__ void encode_token(const uint4 (&v)[NG][4], const uint32_t (&bm)[NG][2], float gs,
                                             uint4 (&cw)[NG], uint32_t (&sfw)[NG]) {
  const float den = __fmul_rn(6.0f, gs);
  const float rden = block_scale_rden(den);
  const float f = e2m1_row_factor(gs);
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    uint32_t c[4] = {0u, 0u, 0u, 0u}, sb2 = 0u;
#pragma unroll
    for (int b = 0; b < 2; ++b) {  // the lane's two blocks of 16
      const uint4 p0 = v[g][2 * b], p1 = v[g][2 * b + 1];
      const uint32_t w0[4] = {p0.x, p0.y, p0.z, p0.w}, w1[4] = {p1.x, p1.y, p1.z, p1.w};
      const float ab = __uint_as_float(bm[g][b] << 16);
      uint32_t sb = 0;
      if (gs != 0.0f) {
        sb = block_scale_code(ab, den, rden);
        const float S = __fmul_rn(gs, e4m3_decode_hw(sb));
        if (S != 0.0f) {
          const uint2 cc = e2m1_codes16_div(w0, w1, S, f);
          c[2 * b] = cc.x;
          c[2 * b + 1] = cc.y;
        }
      }
      sb2 |= sb << (8 * b);
    }
    cw[g] = make_uint4(c[0], c[1], c[2], c[3]);
    sfw[g] = sb2 | (__shfl_xor_sync(0xFFFFFFFFu, sb2, 1) << 16);
  }
}

template <int NG>
__global__ void __launch_bounds__(256) permute_quant_kernel(
    const int32_t* __restrict__ topk_ids, int32_t* __restrict__ tsr, const int32_t* __restrict__ hist,
    const int32_t* __restrict__ offsets, int T, int E, int k, const uint16_t* __restrict__ x, int d,
    int32_t* __restrict__ row_to_token, float* __restrict__ amax_tok, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ tok_codes, uint8_t* __restrict__ sf, float* __restrict__ gout, int* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  // the row's loads go out first, so their latency overlaps the dependent
  // loads that place the token's k rows
  const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)t * d);
  const int n8 = d / 8;  // 8-column vectors of the row
  uint4 v[NG][4];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int e8 = g * 128 + 4 * lane;
#pragma unroll
    for (int q = 0; q < 4; ++q) v[g][q] = e8 < n8 ? __ldg(xr + e8 + q) : make_uint4(0u, 0u, 0u, 0u);
  }
  int row = -1;
  if (lane < k) {
    const int64_t i = (int64_t)t * k + lane;
    row = slot_row(topk_ids[i], t, tsr[i], hist, offsets, E);
    tsr[i] = row;
    row_to_token[row] = t;
  }
  uint32_t bm[NG][2];  // magnitude bits of each block's largest |x|
  uint32_t lm = 0;
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      bm[g][b] = absmax_bits16(v[g][2 * b], v[g][2 * b + 1]);
      lm = max(lm, bm[g][b]);
    }
  const uint32_t rm = __reduce_max_sync(0xFFFFFFFFu, lm);
  if (rm >= 0x7F80u && lane == 0) set_status(status, MOE_STATUS_NONFINITE_X);
  // a NaN in the row (warp-uniform, rare): the largest other magnitude
  const float a =
      __uint_as_float((rm <= 0x7F80u ? rm : __reduce_max_sync(0xFFFFFFFFu, absmax_bits_no_nan(v))) << 16);
  if (lane == 0 && amax_tok) amax_tok[t] = a;
  const float gs = __fdiv_rn(a, 2688.0f);
  const int kg = d / 64;
  uint4 cw[NG];
  uint32_t sfw[NG];
  encode_token<NG>(v, bm, gs, cw, sfw);
  if (tok_codes) {
    uint4* crow = reinterpret_cast<uint4*>(tok_codes + (int64_t)t * (d / 2));
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int e8 = g * 128 + 4 * lane;
      if (e8 < n8) crow[e8 >> 2] = cw[g];
    }
  }
  for (int j = 0; j < k; ++j) {
    const int64_t r = __shfl_sync(0xFFFFFFFFu, row, j);
    uint4* crow = tok_codes ? nullptr : reinterpret_cast<uint4*>(codes + r * (d / 2));
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int e8 = g * 128 + 4 * lane;
      if (e8 < n8) {
        if (crow) crow[e8 >> 2] = cw[g];
        if ((lane & 1) == 0)
          *reinterpret_cast<uint32_t*>(sf + ((r >> 7) * kg + (e8 >> 3)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4) =
              sfw[g];
      }
    }
    if (lane == 0) gout[r] = gs;
  }
}

int launch_permute_quant(const int32_t* topk_ids, int32_t* token_slot_row, const int32_t* hist, const int32_t* offsets,
                         int T, int E, int k, const uint16_t* x, int d, int32_t* row_to_token, float* amax_tok,
                         uint8_t* codes, uint8_t* tok_codes, uint8_t* sf, float* g, int* status, cudaStream_t stream) {
  if (T == 0) return 0;
  const int ng = (d + 1023) / 1024;
  const dim3 grid((T + 7) / 8);
  // row T of the token-ordered codes is the all-zero row the pad rows gather
  if (tok_codes && cudaMemsetAsync(tok_codes + (int64_t)T * (d / 2), 0, (size_t)d / 2, stream) != cudaSuccess) return -1;
#define MOE_PQ(N)                                                                                       \
  permute_quant_kernel<N><<<grid, 256, 0, stream>>>(topk_ids, token_slot_row, hist, offsets, T, E, k, x, d, \
                                                    row_to_token, amax_tok, codes, tok_codes, sf, g, status)
  if (ng <= 1) MOE_PQ(1);
  else if (ng <= 2) MOE_PQ(2);
  else MOE_PQ(4);
#undef MOE_PQ
  return 0;
}

// out[t] = BF16(sum_j FP32(z[token_slot_row[t][j]])), j ascending (the
// ascending expert ids of the token's slots); 8 columns per thread.
// KMAX >= k: all k row loads are issued before the ordered sum.
template <int KMAX>
__global__ void __launch_bounds__(256) unpermute_reduce_kernel(const uint16_t* __restrict__ z,
                                                               const int32_t* __restrict__ token_slot_row, int T,
                                                               int k, int d, uint16_t* __restrict__ out) {
  const int c8n = d / 8;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)T * c8n) return;
  const int64_t t = idx / c8n;
  const int c8 = (int)(idx - t * c8n);
  const int32_t* ts = token_slot_row + t * k;
  uint4 v[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (j < k) v[j] = __ldg(reinterpret_cast<const uint4*>(z + (int64_t)__ldg(ts + j) * d) + c8);
  float s[8];
  {
    const uint32_t w[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) { s[2 * q] = bf16_lo(w[q]); s[2 * q + 1] = bf16_hi(w[q]); }
  }
#pragma unroll
  for (int j = 1; j < KMAX; ++j) {
    if (j < k) {
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        s[2 * q] = __fadd_rn(s[2 * q], bf16_lo(w[q]));
        s[2 * q + 1] = __fadd_rn(s[2 * q + 1], bf16_hi(w[q]));
      }
    }
  }
  uint4 o;
  o.x = pack_bf16x2(s[0], s[1]);
  o.y = pack_bf16x2(s[2], s[3]);
  o.z = pack_bf16x2(s[4], s[5]);
  o.w = pack_bf16x2(s[6], s[7]);
  reinterpret_cast<uint4*>(out + t * (int64_t)d)[c8] = o;
}

int launch_unpermute_reduce(const uint16_t* z, const int32_t* token_slot_row, int T, int k, int d, uint16_t* out,
                            cudaStream_t stream) {
  const int64_t n = (int64_t)T * (d / 8);
  if (n == 0) return 0;
  const unsigned grid = (unsigned)((n + 255) / 256);
  if (k <= 4) unpermute_reduce_kernel<4><<<grid, 256, 0, stream>>>(z, token_slot_row, T, k, d, out);
  else if (k <= 8) unpermute_reduce_kernel<8><<<grid, 256, 0, stream>>>(z, token_slot_row, T, k, d, out);
  else if (k <= 16) unpermute_reduce_kernel<16><<<grid, 256, 0, stream>>>(z, token_slot_row, T, k, d, out);
  else unpermute_reduce_kernel<32><<<grid, 256, 0, stream>>>(z, token_slot_row, T, k, d, out);
  return 0;
}

}  // namespace moe
