// Straight-through BF16 backward of the MoE expert layer (main paper,
// contributions list, and the AI summary's "Methodology in Plain English":
// a straight-through estimator on the saved original BF16 activations and
// weights, no backward quantisation; rainbus summary, method step 5: BF16
// GEMMs on the saved BF16 operands; Technical Report section 4.3, text below
// the table: the layer bypass saves the original BF16 operands).
//
// Launch sequence of moe_expert_backward:
//   FC2 in MODE 2 (gemm.cu: fc2_pair_kernel<2> on CTA pairs, else
//                       fc2_scatter_kernel<2>) recomputes the forward's
//                       expert outputs y2 from the saved FP4 operands
//                       (bit-identical) and, per permuted row r of token t,
//                       slot j:
//                         dw[t][j] = <dY[t], y2[r]>            (FP32)
//                         dy2[r] = BF16(RN_f32(w_tj * dY[t]))  (GEMM operand)
//                       with dy2 zero on pad rows.
//   bwd_xrows_kernel    xp[r] = x[t] (GEMM operand), zero on pad rows; on a
//                       second stream, beside the next three GEMMs.
//   bwd_logits_kernel   dlogits[t][e_j] = w_j (dw_j - sum_i w_i dw_i).
//   bwd_gemm (DGRAD_SWIGLU)  dh = dy2 . W2_e (FP32 in tensor memory), then
//                       SwiGLU backward in the epilogue against the saved u:
//                         du[gate] = BF16(dh * up * s (1 + g (1 - s)))
//                         du[up]   = BF16(dh * g * s),  s = sigmoid(g).
//   bwd_gemm (WGRAD)    dW2_e = dy2_e^T . h_e       (FP32 out)
//   bwd_gemm (DGRAD)    dxr = du . W1_e             (FP32 per row)
//   bwd_gemm (WGRAD)    dW1_e = du_e^T . xp_e       (FP32 out)
//   bwd_dx_kernel       dx[t] = sum_j dxr[row(t,j)], ascending j, FP32.
//
// bwd_gemm is one persistent kernel (one CTA per SM, 10 warps) running
// tcgen05.mma kind::f16 (BF16 x BF16 -> FP32, K = 16 per instruction) from
// 128-byte-swizzled TMA tiles: on CTA pairs (cta_group::2, M = 256, N = 256)
// where N and, for the wgrads, the output rows per expert are multiples of
// 256, else on single CTAs (M = 128, N = 128 or 256):
//   warp 8   TMA producer: per 64-deep k-step one A tile (128 rows) and one B
//            tile (N columns) into a ring of stages;
//   warp 9   MMA issuer: four MMAs per k-step into one of two accumulators
//            (tensor memory columns [0, N) and [N, 2N));
//   warps 0-7  epilogue: warp w reads lanes 32 (w % 4).. and half w / 4 of
//            the accumulator's columns.
// Operand majorness: dgrad reads A (dy2 or du, rows of the permuted tokens)
// K-major and B (the expert's weights, stored [K][N]) MN-major; wgrad reads
// both operands MN-major (the contraction runs over the expert's rows).  An
// MN-major tile is stored as 64-column chunks of 64 rows x 128 bytes, one TMA
// box each; the descriptor's leading offset is the chunk stride and its
// stride offset the 8-row group stride (1024 bytes).
//
// Every wait is bounded; on expiry the kernel raises MOE_STATUS_TIMEOUT,
// lets its own copies and MMAs land, frees tensor memory and returns.
#include <cstdlib>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BK = 64;                 // BK BF16 elements = one 128-byte row
constexpr int A_TILE = BM * BK * 2;              // 16 KB
constexpr int CHUNK = 64 * 128;                  // one MN-major 64 x 64 box: 8 KB
constexpr int NEPI = 8;                          // epilogue warps
constexpr int PROD_WARP = 8, MMA_WARP = 9;
constexpr int THREADS = 320;
constexpr int MAX_STAGES = 8;
constexpr int TMEM_COLS = 512;
constexpr int STAGE_TILE = 32 * 128;             // FP32 output staging per epilogue warp

// Staging tiles per epilogue warp: two for the SwiGLU backward (saved u in
// and du out, double-buffered), one otherwise.
__host__ __device__ constexpr int stage_tiles(int mode) { return mode == BWD_DGRAD_SWIGLU ? 2 : 1; }
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

struct BTail {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
#pragma unroll 1
  for (int i = 0; i < 256; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
      *abort_flag = 1;
      set_status(status, MOE_STATUS_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ bool bwarp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = bwait(bar, parity, abort_flag, status);
  ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  if (ok) (void)mbar_try_wait(bar, parity);
  return ok;
}

// Descriptor of an MN-major operand: 64-column chunks `chunk` bytes apart
// (leading byte offset), 8-row groups of 1024 bytes (stride byte offset).
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t chunk) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((chunk >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

__device__ __forceinline__ void bf16_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void bcommit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ uint32_t pack2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// Expert owning 128-row tile mt of the permuted rows.
__device__ __forceinline__ int expert_of_tile(const int32_t* off, int E, int mt) {
  const int row0 = mt * BM;
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(off + mid) <= row0) lo = mid + 1; else hi = mid;
  }
  return lo - 1;
}

struct Unit {
  int e, mt, nt;  // expert, 128-row output tile, N tile
  int k0, nk;     // first contraction row (wgrad) and number of 64-deep k-steps
  bool ghost;     // CTA pairs: a repeated tile that stores nothing
};

struct Plan {
  int units, ntn;
  __device__ Unit unit(const BwdGemmArgs& a, int u) const {
    Unit U;
    if (a.mode != BWD_WGRAD) {
      U.mt = u / ntn;
      U.nt = u - U.mt * ntn;
      U.e = expert_of_tile(a.offsets, a.E, U.mt);
      U.k0 = 0;
      U.nk = a.K / BK;
    } else {
      const int per_e = (a.Mo / BM) * ntn;
      U.e = u / per_e;
      const int rem = u - U.e * per_e;
      U.mt = rem / ntn;
      U.nt = rem - U.mt * ntn;
      U.k0 = __ldg(a.offsets + U.e);
      U.nk = (__ldg(a.offsets + U.e + 1) - U.k0) / BK;
    }
    U.ghost = false;
    return U;
  }
};

// CTA pairs (cta_group::2 MMAs of M = 256, N = 256): a unit is a pair of
// 128-row output tiles and one 256-column N tile; rank r of the pair takes
// row tile r of the pair and loads N columns 128 r .. of the tile's B.
// dgrad: the pairs are consecutive row tiles of one expert, numbered expert
// by expert (an expert with n tiles owns ceil(n / 2) pairs; when n is odd,
// rank 1's tile of the last pair repeats tile 0's rows and stores nothing);
// wgrad: the expert's Mo / 128 output row tiles in pairs (Mo % 256 == 0).
// The cursor walks the experts forward, so successive calls of one CTA
// (increasing u) continue where the previous one stopped.
struct PairCursor {
  int e = 0, p0 = 0;
};
__device__ __forceinline__ bool pair_unit(const BwdGemmArgs& a, int ntn, int u, int rank, PairCursor& cur, Unit& U) {
  const int p = u / ntn;
  U.nt = u - p * ntn;
  U.ghost = false;
  if (a.mode == BWD_WGRAD) {
    const int per_e = a.Mo / (2 * BM);
    U.e = p / per_e;
    if (U.e >= a.E) return false;
    U.mt = 2 * (p - U.e * per_e) + rank;
    U.k0 = __ldg(a.offsets + U.e);
    U.nk = (__ldg(a.offsets + U.e + 1) - U.k0) / BK;
    return true;
  }
  while (cur.e < a.E) {
    const int t0 = __ldg(a.offsets + cur.e) / BM, t1 = __ldg(a.offsets + cur.e + 1) / BM;
    const int np = (t1 - t0 + 1) >> 1;
    if (p < cur.p0 + np) {
      U.e = cur.e;
      U.mt = t0 + 2 * (p - cur.p0) + rank;
      if (U.mt >= t1) {
        U.ghost = true;
        U.mt -= 1;
      }
      U.k0 = 0;
      U.nk = a.K / BK;
      return true;
    }
    cur.p0 += np;
    ++cur.e;
  }
  return false;
}

// The CTA's units in order: single CTAs take u = blockIdx.x, + gridDim.x,
// ...; pairs take pair units u = cluster, + clusters, ...
template <bool PAIR>
struct UnitWalk {
  const BwdGemmArgs& a;
  const Plan& P;
  int u, step, rank;
  PairCursor cur;
  __device__ UnitWalk(const BwdGemmArgs& a_, const Plan& P_, int start, int step_, int rank_)
      : a(a_), P(P_), u(start), step(step_), rank(rank_) {}
  __device__ bool next(Unit& U) {
    if constexpr (PAIR) {
      const bool ok = pair_unit(a, P.ntn, u, rank, cur, U);
      u += step;
      return ok;
    } else {
      if (u >= P.units) return false;
      U = P.unit(a, u);
      u += step;
      return true;
    }
  }
};

__device__ __forceinline__ uint32_t b_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t b_cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t b_cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t b_map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// 2D tiled TMA load whose completion is signalled on a barrier of either CTA
// of the pair (rank 1's loads complete on rank 0's barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bf16_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void bcommit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void b_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void b_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ Plan make_plan(const BwdGemmArgs& a) {
  Plan p;
  p.ntn = a.N / a.bn;
  if (a.mode != BWD_WGRAD)
    p.units = (__ldg(a.offsets + a.E) / BM) * p.ntn;
  else
    p.units = a.E * (a.Mo / BM) * p.ntn;
  return p;
}

// PAIR: each CTA loads its A tile and its 128 columns of B; rank 0's
// full[s] counts both CTAs' bytes (rank 1's loads complete on it), and each
// CTA waits for its own empty[s], which the MMAs' commits reach in both.
template <bool PAIR>
__device__ void producer(const BwdGemmArgs& a, const Plan& P, uint32_t ring, BTail* tl, volatile int* abort_flag,
                         UnitWalk<PAIR> walk, uint32_t rank) {
  const int bcols = PAIR ? a.bn / 2 : a.bn;  // B columns this CTA loads per stage
  const uint32_t stage_bytes = A_TILE + bcols * 128;
  const uint32_t tx = PAIR ? 2 * stage_bytes : stage_bytes;
  // stage s and use count of the CTA's running k-step, advanced by increments
  uint32_t s = 0, use = 0;
  uint32_t last_use[MAX_STAGES];
  for (int i = 0; i < MAX_STAGES; ++i) last_use[i] = 0xFFFFFFFFu;
  bool aborted = false;
  Unit U;
  while (!aborted && walk.next(U)) {
    const int brow0 = a.mode == BWD_WGRAD ? U.k0 : U.e * a.K;
    const int bcol0 = U.nt * a.bn + (PAIR ? (int)rank * bcols : 0);
    for (int ks = 0; ks < U.nk; ++ks) {
      if (!bwait(smem_u32(&tl->empty[s]), (use & 1u) ^ 1u, abort_flag, a.status)) { aborted = true; break; }
      const uint32_t st = ring + s * stage_bytes;
      const uint32_t fb_own = smem_u32(&tl->full[s]);
      const uint32_t fb = PAIR ? b_map_to_rank(fb_own, 0) : fb_own;
      if (!PAIR || rank == 0) mbar_arrive_expect_tx(fb_own, tx);
      auto load = [&](uint32_t dst, const CUtensorMap* map, int x, int y) {
        if (PAIR)
          tma_load_2d_pair(dst, map, x, y, fb);
        else
          tma_load_2d(dst, map, x, y, fb);
      };
      if (a.a_mn) {
        load(st, &a.tmap_a, U.mt * BM, U.k0 + ks * BK);
        load(st + CHUNK, &a.tmap_a, U.mt * BM + 64, U.k0 + ks * BK);
      } else {
        load(st, &a.tmap_a, ks * BK, U.mt * BM);
      }
      for (int c = 0; c < bcols / 64; ++c) load(st + A_TILE + c * CHUNK, &a.tmap_b, bcol0 + c * 64, brow0 + ks * BK);
      last_use[s] = use;
      if (++s == (uint32_t)a.stages) {
        s = 0;
        ++use;
      }
    }
  }
  if (aborted) {
    // let the copies this thread issued land before the CTA can exit (a
    // pair's rank 1 waits on its own barrier's phase too: its copies have
    // landed once rank 0's phase completed, which the cluster barrier at
    // exit covers)
    for (int s2 = 0; s2 < MAX_STAGES; ++s2)
      if (last_use[s2] != 0xFFFFFFFFu && (!PAIR || rank == 0)) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&tl->full[s2]), last_use[s2] & 1u) && global_timer_ns() - t0 < WAIT_LIMIT_NS) {
        }
      }
  }
}

// PAIR: run by rank 0 alone; cta_group::2 MMAs of M = 256 (each CTA's 128
// rows from its A tile) and N = 256 (each CTA's 128 columns of B), commits
// reaching both CTAs.
template <bool PAIR>
__device__ void mma_issuer(const BwdGemmArgs& a, const Plan& P, uint32_t ring, BTail* tl, uint32_t tmem,
                           volatile int* abort_flag, UnitWalk<PAIR> walk) {
  const int bcols = PAIR ? a.bn / 2 : a.bn;
  const uint32_t stage_bytes = A_TILE + bcols * 128;
  const uint32_t m = PAIR ? 2 * BM : BM;
  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((a.a_mn ? 1u : 0u) << 15) | (1u << 16) |
                         ((uint32_t)(a.bn >> 3) << 17) | ((m >> 4) << 24);
  // The single issuing thread's per-k-step work is what the tensor pipe
  // waits on: descriptors and barrier addresses are formed once, and the
  // stage position advances by increments.  K = 16 per instruction: 32
  // bytes (2 descriptor units) along a K-major row, or two 8-row groups
  // (2048 bytes, 128 units) down an MN-major tile.
  const uint32_t full0 = smem_u32(&tl->full[0]), empty0 = smem_u32(&tl->empty[0]);
  const uint32_t stage_desc = stage_bytes >> 4;
  const uint64_t adesc0 = a.a_mn ? sdesc_mn_sw128(ring, CHUNK) : sdesc_k_sw128(ring);
  const uint64_t bdesc0 = sdesc_mn_sw128(ring + A_TILE, CHUNK);
  const uint32_t astep = a.a_mn ? 128u : 2u;
  auto mma = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t acc) {
    if constexpr (PAIR)
      bf16_mma_pair(d, ad, bd, idesc, acc);
    else
      bf16_mma(d, ad, bd, idesc, acc);
  };
  auto commit = [&](uint32_t bar) {
    if constexpr (PAIR)
      bcommit_pair(bar);
    else
      bcommit(bar);
  };
  uint32_t s = 0, use = 0, it = 0;
  bool aborted = false;
  Unit U;
  while (!aborted && walk.next(U)) {
    if (U.nk == 0) continue;
    const uint32_t acc = it & 1u, ause = it >> 1;
    if (!bwait(smem_u32(&tl->tempty[acc]), (ause & 1u) ^ 1u, abort_flag, a.status)) { aborted = true; break; }
    tc_fence_after();
    const uint32_t d = tmem + acc * (uint32_t)a.bn;
    for (int ks = 0; ks < U.nk; ++ks) {
      if (!bwait(full0 + 8u * s, use & 1u, abort_flag, a.status)) { aborted = true; break; }
      tc_fence_after();
      const uint64_t ad = adesc0 + s * stage_desc, bd = bdesc0 + s * stage_desc;
      mma(d, ad, bd, ks != 0 ? 1u : 0u);
      mma(d, ad + astep, bd + 128u, 1u);
      mma(d, ad + 2u * astep, bd + 256u, 1u);
      mma(d, ad + 3u * astep, bd + 384u, 1u);
      commit(empty0 + 8u * s);
      if (++s == (uint32_t)a.stages) {
        s = 0;
        ++use;
      }
    }
    if (aborted) break;
    commit(smem_u32(&tl->tfull[acc]));
    ++it;
  }
  commit(smem_u32(&tl->done));
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(smem_u32(&tl->done), 0u) && global_timer_ns() - t0 < WAIT_LIMIT_NS) {
  }
}

// SwiGLU backward of 32 columns f0.. of one row (FP32 dh in v).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

// SwiGLU backward of the 32 columns f0.. of a warp's 32 rows (FP32 dh of the
// lane's row in v).  The rows' gate and up segments (64 bytes each) pass
// through one of the warp's two staging tiles both ways: gate of row r at
// tile + 64 r, up at tile + 2048 + 64 r, 16-byte chunk j at chunk
// j ^ ((r / 2) % 4) (eight consecutive rows cover all eight 16-byte bank
// groups).  Copies and stores go four lanes per row, eight rows per
// instruction, instead of one row per lane.  The segments of the next chunk
// are copied in (cp.async, one group per chunk) while this one is computed.
__device__ __forceinline__ void swiglu_u_fetch(const uint16_t* u_row0, int F, int f0, uint32_t tile, int lane) {
  const int64_t ld = 2 * (int64_t)F;  // elements per row of u
  const int cj = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rr = i * 8 + (lane >> 2);
    const uint32_t off = rr * 64 + ((cj ^ ((rr >> 1) & 3)) << 4);
    cp_async16(tile + off, reinterpret_cast<const uint4*>(u_row0 + rr * ld + f0) + cj, true);
    cp_async16(tile + 2048 + off, reinterpret_cast<const uint4*>(u_row0 + rr * ld + F + f0) + cj, true);
  }
  cp_async_commit();
}

// PENDING: copy groups issued after this chunk's (0 or 1).
template <int PENDING>
__device__ __forceinline__ void swiglu_bwd32(const uint32_t (&v)[32], uint16_t* du_row0, int F, int f0, uint32_t tile,
                                             int lane) {
  const int64_t ld = 2 * (int64_t)F;  // elements per row of du
  const int cj = lane & 3;
  asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t off = lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4);
    const uint4 g4 = lds128(tile + off), u4 = lds128(tile + 2048 + off);
    const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, uw[4] = {u4.x, u4.y, u4.z, u4.w};
    uint32_t og[4], ou[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      float rg[2], ru[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float g = h ? bf16_hi(gw[p]) : bf16_lo(gw[p]);
        const float x = h ? bf16_hi(uw[p]) : bf16_lo(uw[p]);
        const float dh = __uint_as_float(v[q * 8 + p * 2 + h]);
        const float s = 1.0f / (1.0f + __expf(-g));
        rg[h] = dh * x * (s * (1.0f + g * (1.0f - s)));
        ru[h] = dh * (g * s);
      }
      og[p] = pack2_rn(rg[0], rg[1]);
      ou[p] = pack2_rn(ru[0], ru[1]);
    }
    sts128(tile + off, og[0], og[1], og[2], og[3]);
    sts128(tile + 2048 + off, ou[0], ou[1], ou[2], ou[3]);
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rr = i * 8 + (lane >> 2);
    const uint32_t off = rr * 64 + ((cj ^ ((rr >> 1) & 3)) << 4);
    reinterpret_cast<uint4*>(du_row0 + rr * ld + f0)[cj] = lds128(tile + off);
    reinterpret_cast<uint4*>(du_row0 + rr * ld + F + f0)[cj] = lds128(tile + 2048 + off);
  }
  __syncwarp();
}

// FP32 outputs leave through a per-warp staging tile (32 rows x 128 bytes,
// 16-byte chunk j of row r at chunk j ^ (r % 8), the 128-byte swizzle of the
// output tensor map) and one TMA store per 32 x 32 chunk, instead of each
// lane writing its own row.
// PAIR: each CTA drains its own 128 rows (all a.bn columns of the pair's
// accumulator) and releases the accumulator to rank 0's barrier; a ghost
// tile stores nothing.
template <bool PAIR>
__device__ void epilogue(const BwdGemmArgs& a, const Plan& P, BTail* tl, uint32_t tmem, uint32_t staging,
                         volatile int* abort_flag, UnitWalk<PAIR> walk) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q4 = warp & 3, part = warp >> 2;
  const int rl = q4 * 32 + lane;
  const int half = a.bn / 2;
  const bool sw = a.mode == BWD_DGRAD_SWIGLU;
  const uint32_t stg = staging + (uint32_t)warp * (uint32_t)stage_tiles(a.mode) * STAGE_TILE;
  bool pending = false;  // lane 0: a store from stg may still be reading it
  uint32_t it = 0;
  const uint32_t tempty0 = PAIR ? b_map_to_rank(smem_u32(&tl->tempty[0]), 0) : smem_u32(&tl->tempty[0]);
  Unit U;
  while (walk.next(U)) {
    const int c0 = U.nt * a.bn + part * half;  // first output column of this thread
    if (U.nk == 0) {  // wgrad of an expert without rows: zero gradient
      float4* o = reinterpret_cast<float4*>(a.out + ((int64_t)U.e * a.Mo + U.mt * BM + rl) * a.N + c0);
      for (int i = 0; i < half / 4; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      continue;
    }
    const uint32_t acc = it & 1u, ause = it >> 1;
    ++it;
    const int64_t row0 = (int64_t)U.mt * BM + q4 * 32;  // DGRAD_SWIGLU: the warp's first row
    // DGRAD_SWIGLU: the first chunk's saved u is copied in before the wait
    if (sw && !U.ghost) swiglu_u_fetch(a.u + row0 * 2 * a.F, a.F, c0, stg, lane);
    if (!bwarp_wait(smem_u32(&tl->tfull[acc]), ause & 1u, abort_flag, a.status)) break;
    tc_fence_after();
    const uint32_t tbase = tmem + ((uint32_t)(q4 * 32) << 16) + acc * (uint32_t)a.bn + part * half;
    for (int c = 0; c < half && !U.ghost; c += 32) {
      uint32_t v[32];
      tld32(tbase + c, v);
      if (sw) {
        const uint32_t tile = stg + (uint32_t)((c >> 5) & 1) * STAGE_TILE;
        if (c + 32 < half) {
          swiglu_u_fetch(a.u + row0 * 2 * a.F, a.F, c0 + c + 32, stg + (uint32_t)(((c >> 5) + 1) & 1) * STAGE_TILE,
                         lane);
          swiglu_bwd32<1>(v, a.du + row0 * 2 * a.F, a.F, c0 + c, tile, lane);
        } else {
          swiglu_bwd32<0>(v, a.du + row0 * 2 * a.F, a.F, c0 + c, tile, lane);
        }
      } else {
        const int orow0 = a.mode == BWD_WGRAD ? U.e * a.Mo + U.mt * BM + q4 * 32 : U.mt * BM + q4 * 32;
        if (lane == 0 && pending) bulk_wait_read0();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          sts128(stg + lane * 128 + ((j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&a.tmap_out, stg, c0 + c, orow0);
          pending = true;
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if constexpr (PAIR)
        b_arrive_cluster(tempty0 + 8u * acc);
      else
        mbar_arrive(tempty0 + 8u * acc);
    }
  }
  if (sw) cp_async_wait_all();  // no copy into shared memory outlives the CTA
  if (lane == 0 && pending) bulk_wait0();  // the last stores complete before the CTA exits
  __syncwarp();
}

}  // namespace

// PAIR: clusters of two CTAs (cta_group::2 MMAs issued by rank 0); the
// barriers rank 0's MMA thread waits on count both CTAs (full: both CTAs'
// bytes; tempty: both CTAs' epilogue warps); the cluster barrier at entry
// orders the barrier initialisation before any remote arrival, and the one
// at exit holds both CTAs until rank 0 has seen all MMAs complete.
template <bool PAIR>
__global__ void __launch_bounds__(THREADS, 1) bwd_gemm_kernel(const __grid_constant__ BwdGemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int bcols = PAIR ? a.bn / 2 : a.bn;
  const uint32_t stage_bytes = A_TILE + bcols * 128;
  uint8_t* staging = smem + (size_t)a.stages * stage_bytes;
  BTail* tl = reinterpret_cast<BTail*>(staging + NEPI * stage_tiles(a.mode) * STAGE_TILE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? b_cluster_rank() : 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(smem_u32(&tl->full[s]), 1);
      mbar_init(smem_u32(&tl->empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&tl->tfull[s]), 1);
      mbar_init(smem_u32(&tl->tempty[s]), PAIR ? 2 * NEPI : NEPI);
    }
    mbar_init(smem_u32(&tl->done), 1);
    tl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    if constexpr (PAIR) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tl->tmem_base)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tl->tmem_base)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    b_cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  const Plan P = make_plan(a);
  volatile int* abort_flag = &tl->abort_flag;
  const uint32_t ring = smem_u32(smem);
  const int start = PAIR ? (int)b_cluster_id() : (int)blockIdx.x;
  const int step = PAIR ? (int)b_cluster_count() : (int)gridDim.x;
  const UnitWalk<PAIR> walk(a, P, start, step, (int)rank);
  if (warp == PROD_WARP) {
    if (lane == 0) {
      prefetch_tmap(&a.tmap_a);
      prefetch_tmap(&a.tmap_b);
      if (a.mode != BWD_DGRAD_SWIGLU) prefetch_tmap(&a.tmap_out);
      producer<PAIR>(a, P, ring, tl, abort_flag, walk, rank);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (lane == 0 && (!PAIR || rank == 0)) mma_issuer<PAIR>(a, P, ring, tl, tl->tmem_base, abort_flag, walk);
    __syncwarp();
  } else {
    epilogue<PAIR>(a, P, tl, tl->tmem_base, smem_u32(staging), abort_flag, walk);
  }
  tc_fence_before();
  if constexpr (PAIR)
    b_cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP) {
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tl->tmem_base), "r"(TMEM_COLS)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tl->tmem_base), "r"(TMEM_COLS)
                   : "memory");
  }
}

int bwd_gemm_smem_bytes(int mode, int bn, int stages) {
  return 1024 + stages * (A_TILE + bn * 128) + NEPI * stage_tiles(mode) * STAGE_TILE + (int)sizeof(BTail);
}

// The most stages, up to `most`, whose shared memory fits one CTA (B tiles of
// `bcols` columns).
static int fit_stages(int mode, int bcols, int most) {
  int s = most;
  while (s > 2 && bwd_gemm_smem_bytes(mode, bcols, s) > 232448) --s;
  return s;
}

// max_row_tiles: for dgrad, an upper bound of offsets[E] / 128 (the number
// of units is read on the device); ignored for wgrad.
// The GEMMs with N % 256 == 0 (and, for wgrad, Mo % 256 == 0) run on CTA
// pairs, six 32 KB stages per CTA; the rest on single CTAs with four 48 KB
// (N tile 256) or six 32 KB (N tile 128) stages.  The SwiGLU backward's
// second staging tile per warp takes one stage's room where they do not all
// fit.  MOE_BWD_CTA_PAIRS=0 in the environment selects single CTAs
// throughout.
int launch_bwd_gemm(BwdGemmArgs& a, int max_row_tiles, cudaStream_t stream) {
  a.bn = a.N % 256 == 0 ? 256 : 128;
  const int ntn = a.N / a.bn;
  const char* env = std::getenv("MOE_BWD_CTA_PAIRS");
  const bool pairs = !(env && env[0] == '0') && a.bn == 256 && (a.mode != BWD_WGRAD || a.Mo % 256 == 0);
  int sms = gemm_num_ctas();
  if (sms <= 0) return -1;
  if (pairs) {
    a.stages = fit_stages(a.mode, a.bn / 2, 6);
    const int smem = bwd_gemm_smem_bytes(a.mode, a.bn / 2, a.stages);
    if (cudaFuncSetAttribute(bwd_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, bwd_gemm_kernel<true>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      clusters = 0;
    }
    if (clusters > sms / 2) clusters = sms / 2;
    const int64_t max_units = a.mode == BWD_WGRAD ? (int64_t)a.E * (a.Mo / (2 * BM)) * ntn
                                                  : ((int64_t)max_row_tiles / 2 + a.E) * ntn;
    if (max_units < clusters) clusters = (int)max_units;
    if (clusters >= 1) {
      cfg.gridDim = dim3((unsigned)(2 * clusters));
      return cudaLaunchKernelEx(&cfg, bwd_gemm_kernel<true>, a) == cudaSuccess ? 0 : -1;
    }
  }
  a.stages = fit_stages(a.mode, a.bn, a.bn == 256 ? 4 : 6);
  const int64_t max_units = a.mode == BWD_WGRAD ? (int64_t)a.E * (a.Mo / BM) * ntn : (int64_t)max_row_tiles * ntn;
  const int smem = bwd_gemm_smem_bytes(a.mode, a.bn, a.stages);
  if (cudaFuncSetAttribute(bwd_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  int grid = sms;
  if (max_units < grid) grid = (int)max_units;
  if (grid < 1) return 0;
  bwd_gemm_kernel<false><<<grid, THREADS, smem, stream>>>(a);
  return 0;
}

// ---------------------------------------------------------------------------
// Row, logit and dx kernels (HBM-bound, one warp per row or token)
// ---------------------------------------------------------------------------
// xp[r] = x[row_to_token[r]] (the wgrad operand of FC1), zero on pad rows;
// rows at or past offsets[E] are left alone.  d % 8 == 0.  One warp per row,
// the warps of the grid striding over the rows.
__global__ void __launch_bounds__(256) bwd_xrows_kernel(const uint16_t* __restrict__ x,
                                                        const int32_t* __restrict__ row_to_token,
                                                        const int32_t* __restrict__ offsets, int E, int T, int d,
                                                        int64_t m_rows, uint16_t* __restrict__ xp) {
  const int lane = threadIdx.x & 31;
  const int64_t end = min(m_rows, (int64_t)__ldg(offsets + E));  // past the padded rows: never read
  const int n8 = d / 8;
  for (int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < end; r += (int64_t)gridDim.x * 8) {
    uint4* xrow = reinterpret_cast<uint4*>(xp + r * d);
    const int t = __ldg(row_to_token + r);
    if (t < 0 || t >= T) {
      for (int i = lane; i < n8; i += 32) xrow[i] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const uint4* xsrc = reinterpret_cast<const uint4*>(x + (int64_t)t * d);
    for (int i = lane; i < n8; i += 32) xrow[i] = __ldg(xsrc + i);
  }
}

// dlogits[t][:] = 0, then w_j (dw_j - sum_i w_i dw_i) at the selected ids.
__global__ void __launch_bounds__(256) bwd_logits_kernel(const float* __restrict__ dw, const float* __restrict__ topk_w,
                                                         const int32_t* __restrict__ topk_ids, int T, int E, int k,
                                                         float* __restrict__ dlogits) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  float mean = 0.0f;
  for (int j = 0; j < k; ++j) mean = fmaf(__ldg(topk_w + t * k + j), __ldg(dw + t * k + j), mean);
  for (int e = lane; e < E; e += 32) dlogits[t * E + e] = 0.0f;
  __syncwarp();
  for (int j = lane; j < k; j += 32) {
    const int e = __ldg(topk_ids + t * k + j);
    if (e >= 0 && e < E) dlogits[t * E + e] = __ldg(topk_w + t * k + j) * (__ldg(dw + t * k + j) - mean);
  }
}

// dx[t] = sum_j dxr[token_slot_row[t][j]] (FP32, ascending j).  d % 4 == 0.
// KMAX >= k: the k row loads of a column group are issued before the sum.
template <int KMAX>
__global__ void __launch_bounds__(256) bwd_dx_kernel(const float* __restrict__ dxr,
                                                     const int32_t* __restrict__ token_slot_row, int T, int k, int d,
                                                     float* __restrict__ dx) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int n4 = d / 4;
  int rows[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) rows[j] = j < k ? __ldg(token_slot_row + t * k + j) : 0;
  for (int i = lane; i < n4; i += 32) {
    float4 v[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) v[j] = __ldg(reinterpret_cast<const float4*>(dxr + (int64_t)rows[j] * d) + i);
    float4 s = v[0];
#pragma unroll
    for (int j = 1; j < KMAX; ++j) {
      if (j < k) {
        s.x += v[j].x; s.y += v[j].y; s.z += v[j].z; s.w += v[j].w;
      }
    }
    reinterpret_cast<float4*>(dx + t * d)[i] = s;
  }
}

// blocks > 0: that many blocks stride over the rows (a grid small enough to
// run beside a persistent GEMM); else one block per eight rows.
int launch_bwd_xrows(const uint16_t* x, const int32_t* row_to_token, const int32_t* offsets, int E, int T, int d,
                     int64_t m_rows, uint16_t* xp, int blocks, cudaStream_t stream) {
  if (m_rows <= 0) return 0;
  const int64_t all = (m_rows + 7) / 8;
  const unsigned grid = (unsigned)(blocks > 0 && blocks < all ? blocks : all);
  bwd_xrows_kernel<<<grid, 256, 0, stream>>>(x, row_to_token, offsets, E, T, d, m_rows, xp);
  return 0;
}

int launch_bwd_logits(const float* dw, const float* topk_w, const int32_t* topk_ids, int T, int E, int k,
                      float* dlogits, cudaStream_t stream) {
  if (T <= 0) return 0;
  bwd_logits_kernel<<<(unsigned)((T + 7) / 8), 256, 0, stream>>>(dw, topk_w, topk_ids, T, E, k, dlogits);
  return 0;
}

int launch_bwd_dx(const float* dxr, const int32_t* token_slot_row, int T, int k, int d, float* dx, cudaStream_t stream) {
  if (T <= 0) return 0;
  const unsigned grid = (unsigned)((T + 7) / 8);
  if (k <= 4) bwd_dx_kernel<4><<<grid, 256, 0, stream>>>(dxr, token_slot_row, T, k, d, dx);
  else if (k <= 8) bwd_dx_kernel<8><<<grid, 256, 0, stream>>>(dxr, token_slot_row, T, k, d, dx);
  else if (k <= 16) bwd_dx_kernel<16><<<grid, 256, 0, stream>>>(dxr, token_slot_row, T, k, d, dx);
  else bwd_dx_kernel<32><<<grid, 256, 0, stream>>>(dxr, token_slot_row, T, k, d, dx);
  return 0;
}

}  // namespace moe
