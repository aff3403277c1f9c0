// Grouped block-scaled NVFP4 GEMMs of the MoE expert: U_e = MMA_NVFP4(X_e,
// W_e^T) on the 5th-generation tensor cores, then the FP32 epilogue that
// multiplies by g_x * g_w and casts to BF16 (rainbus summary, core method;
// AI summary methodology: outer factors applied in FP32 after the native
// block-scaled multiply, no decoded BF16 operand).
//
// Design (one persistent CTA per SM; NE epilogue warps, NE = 16 in FC1 and in
// FC2 on CTA pairs, 8 in FC2 on single CTAs, then 4 scale writers, 3
// producers and the MMA issuer):
//   warps NE+4 .. NE+6  TMA producers.  A work unit is one 128-row tile of
//            the routed rows (one expert).  Its A operand (128 rows x K FP4,
//            128-byte swizzle) is loaded once into resident shared memory, one
//            slice per 256 elements of K; the B operand (128 weight rows x 256
//            elements of K) and the block-scale tiles of both operands stream
//            through three or four rings of one or two stages, the k-steps
//            dealt round-robin over the rings; producer warp p feeds the rings
//            r with r % 3 == p, each ring from one warp in order.  When K does
//            not fit, A streams through the stages too.
//   warps NE .. NE+3  block-scale writers, one per tensor-memory lane
//            quadrant.  For each stage they move the scale tiles from shared
//            to tensor memory with tcgen05.st: the B scales replicated in
//            every quadrant (each quadrant of the tensor core reads all of
//            them), the A scales only on the diagonal (row r is read from lane
//            r, column base + r/32), and signal the stage's scales as ready.
//   warp NE+7  MMA issuer: tcgen05.mma kind::mxf4nvf4 block_scale.scale_vec::4X
//            (M=128, N=128, K=64, UE4M3 scale per 16 elements) into one of
//            the 128-column FP32 accumulators (three for FC1, two for FC2);
//            nothing else goes through the tensor pipe.  Tensor memory after
//            the accumulators holds one 32-column scale buffer per stage.
//   warps 0 .. NE-1  epilogue: warp w reads TMEM lanes 32*(w%4).. (its 32
//            rows) and part w/4 of the accumulator's columns, releases the
//            accumulator, then does the FP32 epilogue from registers.  The
//            expert's per-column outer scales are staged in shared memory per
//            unit.
//
//   FC1: the items of a unit are, per 128-column chunk c of h, a gate tile
//        (W1 rows c*128..) then an up tile (rows d_ff + c*128..).  The
//        epilogue forms u = BF16(acc * (g_x * g_w)), h = BF16(silu(gate) * up),
//        stages h in a per-CTA scratch (L2-resident) and keeps each row's
//        running amax; after the last chunk it requantises the row
//        (g_h = amax/2688, E4M3 block scales, E2M1 codes).
//   FC2: the items of a unit are the d/128 output tiles; the epilogue forms
//        y2 = acc * (g_h * g_w2), z = BF16(w_{t,e} * y2) and writes it to the
//        row's own row of the z rows (slot (t, j) of the combine lives at row
//        token_slot_row[t][j]): each warp stages its 32 x 64 tile, swizzled
//        like the destination's tensor map, and sends it with one TMA tensor
//        store.
//
// FC1 on CTA pairs (where its plan fits): clusters of two CTAs, a unit being
// two 128-row tiles of one expert.  Rank 0's MMA thread issues
// tcgen05.mma.cta_group::2 of M = 256 (each CTA's 128 rows from its own
// resident A) and N = 256 (a chunk's gate from rank 0's B tile, its up from
// rank 1's), K = 64, into one 256-column accumulator per CTA; every commit
// arrives in both CTAs.  Both CTAs' scale writers and epilogue warps arrive
// on rank 0's sf_full / tempty barriers.  Each CTA runs the epilogue of its
// own rows, and releases the accumulator once u is formed, before the SwiGLU.
//
// FC2 on CTA pairs (where d is a multiple of 256): the same pair units; an
// item is 256 output columns, W2 rows nt*256.. in rank 0's B tile and the
// next 128 in rank 1's, one 256-column accumulator per CTA, 16 epilogue
// warps of 64 columns.  The backward's recomputation of FC2 (dw, dy2) runs
// on the same kernel.
//
// The 24-warp kernels (FC1, FC2 on pairs) launch at 80 registers a thread and
// move registers to the epilogue with setmaxnreg (96 for the epilogue, 56 for
// the scale writers, 40 for the producers and the MMA issuer).
//
// Every wait is bounded (a few seconds of wall clock); on expiry the kernel
// raises MOE_STATUS_TIMEOUT, drains its own copies and MMAs, frees tensor
// memory and returns.
#include <cstdlib>

#include "common.cuh"
#include "kernels.cuh"
#include "swiglu.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BN = 128, BK_BYTES = 128;
constexpr int A_SLICE = BM * BK_BYTES;                 // 16 KB
constexpr int B_BYTES = BN * BK_BYTES;                 // 16 KB
constexpr int SF_STAGE = 4 * 512;                      // 2 KB per operand
constexpr int B_STAGE = B_BYTES + 2 * SF_STAGE;        // 20 KB: B, SFB, SFA
// CTA pairs (FC1): one MMA covers 256 rows (128 per CTA) and 256 columns,
// a chunk's gate (columns 0-127, rank 0's B tile) and up (128-255, rank 1's
// B tile) together, into one 256-column accumulator.  A stage holds the
// CTA's B tile, the scale tiles of both B tiles and the CTA's A scales; the
// scale buffers in tensor memory form a ring of their own, decoupled from
// the stages.
constexpr int PAIR_STAGE = B_BYTES + 3 * SF_STAGE;     // 22 KB: B, SFB gate, SFB up, SFA
constexpr int PAIR_RINGS_MAX = 4;                      // rings of one stage (3 when 4 do not fit)
constexpr int PAIR_SFBUF = 4;                          // tensor-memory scale buffers
constexpr int PAIR_ACC_COLS = 2 * BN;                  // the 256-column accumulator
constexpr int PAIR_SF_COLS = 64;                       // per buffer: [A scales 16 | B scales 32 | unused 16]
constexpr int MAX_A_SLOTS = 16;
constexpr int MAX_STAGES = 8;                          // over all rings (one TMEM scale buffer each)
constexpr int NPROD_WARPS = 3;                         // producer warps: warp p feeds rings r with r % 3 == p
constexpr int NSLOT_MAX = 3;                           // accumulators
constexpr int FC1_NSLOT = 3;                           // FC1 pairs gate and up tiles: three
constexpr int FC2_NSLOT = 2;                           // FC2: double buffering
// Epilogue warps per kernel: warp w serves TMEM lane quadrant w % 4 and
// column part w / 4 of each accumulator.  FC1's SwiGLU/requantisation is
// latency-bound and gains from four warps per scheduler (16 warps, 32
// columns each); FC2 on pairs drains 64 columns per warp of its 256-column
// accumulator with 16 warps; FC2 on single CTAs keeps 8 warps of 64 columns
// at 128 registers.
constexpr int FC1_NE = 16, FC2_NE = 8;
constexpr int FC2P_NE = 16;
// Register split of the 24-warp kernels (launched at 80 per thread)
constexpr int REG_EPI = 96, REG_SFW = 56, REG_PROD = 40;
static_assert(4 * REG_EPI + REG_SFW + REG_PROD == 6 * 80, "register split");  // FC2 on CTA pairs: 4 column parts of 64 of the 256-column accumulator
static_assert(FC1_NE * 32 <= kFc1EpiThreads, "FC1 epilogue threads");
constexpr int FC1_PARTS = FC1_NE / 4, FC1_PART_COLS = BN / FC1_PARTS;  // column parts of a chunk, one per warp
// h is staged and requantised in 32-column sub-parts (two 16-element blocks,
// half of a scale word); a thread's part holds FC1_SUB of them and
// FC1_HALVES 16-column halves.
constexpr int FC1_VPARTS = 4, FC1_SUB = FC1_VPARTS / FC1_PARTS, FC1_HALVES = FC1_PART_COLS / 16;
constexpr int FC2_PARTS = FC2_NE / 4, FC2_PART_COLS = BN / FC2_PARTS;  // 2 parts of 64 columns
constexpr int FC2_STAGE_ROW = FC2_PART_COLS * 2;       // FC2 output staging: one part's BF16 columns per row
constexpr int FC2_STAGING_BYTES = FC2_NE * 32 * FC2_STAGE_ROW;  // 32 rows per epilogue warp
constexpr int TMEM_COLS = 512;
constexpr int SF_COLS = 32;                            // per stage: [A scales 16 | B scales 16]
// Warp roles for NE epilogue warps: epilogue 0..NE-1, scale writers
// NE..NE+3, producers NE+4..NE+6, MMA issuer NE+7.
template <int NE>
struct Roles {
  static constexpr int EPI_THREADS = NE * 32;
  static constexpr int SFW = NE;
  static constexpr int PROD = NE + 4;
  static constexpr int MMA = PROD + NPROD_WARPS;
  static constexpr int THREADS = (MMA + 1) * 32;
};
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int SMEM_LIMIT = 232448;  // opt-in shared memory per CTA

// Instruction descriptor: E2M1 x E2M1, UE4M3 scales, both operands K-major,
// N = 128 (bits 17-22 hold N/8), M = 128 (bits 24-28 hold M/16).
constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
// The same for a CTA pair: M = 256 (rows 0-127 from the issuing CTA's A,
// 128-255 from the peer's), N = 256 (columns 0-127 from the issuing CTA's B
// tile, 128-255 from the peer's).
constexpr uint32_t IDESC_PAIR =
    (1u << 7) | (1u << 10) | ((uint32_t)PAIR_ACC_COLS >> 3 << 17) | ((uint32_t)((2 * BM) >> 4) << 24);

struct Tail {
  uint64_t a_full[MAX_A_SLOTS];
  uint64_t a_empty[MAX_A_SLOTS];
  uint64_t b_full[MAX_STAGES];
  uint64_t b_empty[MAX_STAGES];
  uint64_t sf_full[MAX_STAGES];
  uint64_t sf_empty[PAIR_SFBUF];  // CTA pairs: scale buffer free again
  uint64_t tfull[NSLOT_MAX];
  uint64_t tempty[NSLOT_MAX];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
  float rowmax[4][BM];  // per column part (FC1)
};

constexpr size_t TAIL_BYTES = (sizeof(Tail) + 1023) / 1024 * 1024;

// The CTA's abort flag (in shared memory), held as its 32-bit shared
// address: a wait raises it on timeout, and every role checks it.
struct AbortFlag {
  uint32_t addr;
  __device__ __forceinline__ bool raised() const {
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v != 0u;
  }
  __device__ __forceinline__ void raise() const {
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(addr), "r"(1u) : "memory");
  }
};

// Poll the barrier; the abort flag and the wall clock are consulted only
// every 256 failed polls, so a short wait costs nothing but the polls.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, AbortFlag abort_flag, int* status) {
#pragma unroll 1
  for (int i = 0; i < 256; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag.raised()) return false;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
      abort_flag.raise();
      set_status(status, MOE_STATUS_TIMEOUT);
      return false;
    }
  }
}

// Warp-wide wait: lane 0 polls, the other lanes wait at the warp barrier
// and then take their own (immediately satisfied) look at the completed
// phase, so a waiting warp costs the barrier unit one poller, not 32.  All
// 32 lanes call it; the result is the same in every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, AbortFlag abort_flag, int* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_bounded(bar, parity, abort_flag, status);
  ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  if (ok) (void)mbar_try_wait(bar, parity);
  return ok;
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// CTA pairs: the commit arrives on the barrier at the same offset in both
// CTAs of the cluster.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(IDESC_PAIR), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on a barrier of another CTA of the cluster (or this one, by its
// cluster address).  What the arrival orders is tensor-memory and tensor-core
// work, which the tcgen05 fences around the wait and the arrival order; the
// release/acquire forms at cluster scope cost FC1 a millisecond on the 64k
// layer and are not needed for it.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(IDESC), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
template <int NE>
__device__ __forceinline__ void epi_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(Roles<NE>::EPI_THREADS) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// Expert owning 128-row tile mt: the last e with offsets[e] <= mt*128.
__device__ __forceinline__ int expert_of(const int32_t* off, int E, int mt) {
  const int row0 = mt * BM;
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(off + mid) <= row0) lo = mid + 1; else hi = mid;
  }
  return lo - 1;
}

struct Geometry {
  int num_mt;      // 128-row tiles
  bool pair;       // CTA pairs: units of two tiles, half of B per CTA
  uint32_t rank;   // rank in the pair (0 issues the MMAs)
  int cluster, nclusters;
  int b_bytes;     // B bytes per stage
  int sfb_tiles;   // B scale tiles per stage: 1, or 2 in a pair (gate and up)
  int acc_cols;    // TMEM columns per accumulator: BN, or PAIR_ACC_COLS in a pair
  int sf_cols;     // TMEM columns per scale buffer: SF_COLS, or PAIR_SF_COLS in a pair
  int items;       // accumulator tiles per unit
  int nk;          // k-steps of 256 elements
  int kgroups;     // K / 64 (block-scale 4-column groups)
  int rings;       // rings of stages, 3 or 4; ring r is fed by producer warp r % 3
  int log2_stages; // stages per ring = 1 << log2_stages
  int stage_bytes; // [A slice when streamed][B][SFB][SFA]
  int nslot;       // accumulators (128 TMEM columns each)
  bool resident;   // A slices loaded once per unit into their own slots
  __device__ uint32_t b_off() const { return resident ? 0u : (uint32_t)A_SLICE; }
  // first TMEM column of the scale buffers (after the accumulators; one per
  // stage, or a ring of PAIR_SFBUF in a pair)
  __device__ uint32_t sf_col() const { return (uint32_t)(nslot * acc_cols); }
  // CTA pairs keep a separate ring of scale buffers (released by sf_empty)
  // unless the stage ring has as many stages as there are buffers: then
  // buffer and stage coincide, and a stage's refill (after the commit of its
  // previous MMAs) already says the buffer is free.
  __device__ bool sf_ring() const { return pair && (rings << log2_stages) != PAIR_SFBUF; }
  // scale buffer of CTA-local k-step kc (stage slot `slot`) and its use count
  __device__ void sfbuf_of(uint32_t kc, uint32_t slot, uint32_t use, uint32_t& buf, uint32_t& buse) const {
    if (sf_ring()) {
      buf = kc & (PAIR_SFBUF - 1);
      buse = kc / PAIR_SFBUF;
    } else {
      buf = slot;
      buse = use;
    }
  }
  // ring of CTA-local k-step kc and its position in the ring
  __device__ void ring_of(uint32_t kc, uint32_t& r, uint32_t& pos) const {
    if (rings == 4) {
      r = kc & 3u;
      pos = kc >> 2;
    } else {
      pos = kc / 3u;
      r = kc - 3u * pos;
    }
  }
  // ring slot of CTA-local k-step kc and the use count of that slot
  __device__ void slot_of(uint32_t kc, uint32_t& slot, uint32_t& use) const {
    uint32_t r, pos;
    ring_of(kc, r, pos);
    slot = (r << log2_stages) + (pos & ((1u << log2_stages) - 1u));
    use = pos >> log2_stages;
  }
};

// The CTA's work units, in order (index iu = 0, 1, ...).  Single CTAs: a
// unit is one 128-row tile; CTA i takes tiles i, i + gridDim.x, ...  CTA
// pairs: a unit is two consecutive 128-row tiles of one expert; cluster c
// takes pair units c, c + clusters, ... (numbered expert by expert, an
// expert with n tiles owning ceil(n / 2)), and rank r of the pair owns the
// unit's tile r.  When an expert's tile count is odd its last unit has no
// second tile: rank 1 then repeats tile 0's operands (the MMA needs its half
// of B all the same) and writes nothing (`ghost`).  The cursor walks the
// experts forward, so each call continues where the previous one stopped.
struct UnitCursor {
  int e = 0, p0 = 0;  // expert under the cursor, its first pair-unit index
};
__device__ __forceinline__ bool unit_at(const Geometry& G, const int32_t* off, int E, int iu, UnitCursor& cur,
                                        int& tile, int& e, bool& ghost) {
  if (!G.pair) {
    const int u = (int)blockIdx.x + iu * (int)gridDim.x;
    if (u >= G.num_mt) return false;
    tile = u;
    e = expert_of(off, E, u);
    ghost = false;
    return true;
  }
  const int p = G.cluster + iu * G.nclusters;
  while (cur.e < E) {
    const int t0 = __ldg(off + cur.e) / BM, t1 = __ldg(off + cur.e + 1) / BM;
    const int np = (t1 - t0 + 1) >> 1;
    if (p < cur.p0 + np) {
      e = cur.e;
      tile = t0 + 2 * (p - cur.p0) + (int)G.rank;
      ghost = tile >= t1;
      if (ghost) tile -= 1;
      return true;
    }
    cur.p0 += np;
    ++cur.e;
  }
  return false;
}

// Weight row of item q of a unit of expert e.
struct ItemRows {
  bool fc1;
  int N, d_ff;
  __device__ int operator()(int e, int q) const {
    if (fc1) return e * N + (q & 1) * d_ff + (q >> 1) * BN;
    return e * N + q * BN;
  }
};

// A slice (128 rows x 128 bytes) of unit u at byte column x: one 128-row box
// (GATHER false, issued by the one producer lane), or, gathered, lane i's
// four-row copy of rows 4i..4i+3 (their tokens; negative -> zero_row), all
// 32 lanes of the producer warp issuing together.
template <bool GATHER>
__device__ __forceinline__ void load_a_slice(uint32_t dst, const CUtensorMap* tmap_a, int x, int u,
                                             const int32_t* a_rows, int zero_row, uint32_t bar, int lane) {
  if (!GATHER) {
    tma_load_2d(dst, tmap_a, x, u * BM, bar);
    return;
  }
  const int4 r = __ldg(reinterpret_cast<const int4*>(a_rows + (int64_t)u * BM) + lane);
  tma_gather4(dst + lane * 4 * BK_BYTES, tmap_a, x, r.x < 0 ? zero_row : r.x, r.y < 0 ? zero_row : r.y,
              r.z < 0 ? zero_row : r.z, r.w < 0 ? zero_row : r.w, bar);
}

// Barrier wait of a producer: the single producer lane polls alone; with
// GATHER the whole warp takes part (lane 0 polls).
template <bool GATHER>
__device__ __forceinline__ bool producer_wait(uint32_t bar, uint32_t parity, AbortFlag abort_flag, int* status) {
  return GATHER ? warp_wait(bar, parity, abort_flag, status) : wait_bounded(bar, parity, abort_flag, status);
}

// Producer r of R: lane 0 of warp PROD + r alone, or, with GATHER, all 32
// lanes (lane 0 polls the barriers and issues the box and bulk copies, every
// lane its share of a gathered A slice; the extra lanes cost the epilogue
// warps issue slots, so the box path keeps one lane).  The CTA's k-steps (over units, items, K) are numbered
// kc = 0, 1, ...; k-step kc travels through ring kc % R, position kc / R.
// Each ring has one producer and is consumed in order, so every barrier sees
// its phases in order.  A producer runs at most R*S k-steps ahead of the
// MMAs; the plan keeps that below the reach that would let a resident A
// slot's a_empty wait (at the first item of a unit, by whichever producer
// owns that k-step) alias an older phase.
template <bool GATHER>
__device__ void producer_loop(int r, const CUtensorMap* tmap_a, const CUtensorMap* tmap_b, const uint8_t* a_sf,
                              const uint8_t* b_sf, const Geometry& G, const ItemRows& rows, const int32_t* off, int E,
                              uint32_t a_base, uint32_t ring_base, Tail* tl, AbortFlag abort_flag, int* status,
                              const int32_t* a_rows, int zero_row) {
  const uint32_t b_off = G.b_off();
  const int lane = threadIdx.x & 31;
  uint32_t kc = 0;
  uint32_t last_stage_use[MAX_STAGES], last_a_use[MAX_A_SLOTS];
  for (int i = 0; i < MAX_STAGES; ++i) last_stage_use[i] = 0xFFFFFFFFu;
  for (int i = 0; i < MAX_A_SLOTS; ++i) last_a_use[i] = 0xFFFFFFFFu;
  bool aborted = false;
  UnitCursor cur;
  int u, e;
  bool ghost;
  for (int iu = 0; !aborted && unit_at(G, off, E, iu, cur, u, e, ghost); ++iu) {
    const uint32_t unit_use = (uint32_t)iu;
    const int64_t sfa_row = (int64_t)u * G.kgroups;
    for (int q = 0; q < G.items && !aborted; ++q) {
      // a pair's item is chunk q: rank 0 loads its gate rows, rank 1 its up
      // rows, and both load the scales of both
      const int br = G.pair ? rows(e, 2 * q) : rows(e, q);
      const int b_row = G.pair ? rows(e, 2 * q + (int)G.rank) : br;
      const int64_t sfb_row = (int64_t)(br / BM) * G.kgroups;
      const int64_t sfb_row2 = G.pair ? (int64_t)(rows(e, 2 * q + 1) / BM) * G.kgroups : 0;
      for (int ks = 0; ks < G.nk; ++ks, ++kc) {
        uint32_t ring, pos;
        G.ring_of(kc, ring, pos);
        if (ring % (uint32_t)NPROD_WARPS != (uint32_t)r) continue;
        uint32_t slot, use;
        G.slot_of(kc, slot, use);
        if (!producer_wait<GATHER>(smem_u32(&tl->b_empty[slot]), (use & 1u) ^ 1u, abort_flag, status)) {
          aborted = true;
          break;
        }
        const int nsf = min(4, G.kgroups - 4 * ks);
        const uint32_t st = ring_base + slot * G.stage_bytes;
        const uint32_t fb = smem_u32(&tl->b_full[slot]);
        if (G.resident && q == 0) {
          if (!producer_wait<GATHER>(smem_u32(&tl->a_empty[ks]), (unit_use & 1u) ^ 1u, abort_flag, status)) {
            aborted = true;
            break;
          }
          const uint32_t ab = smem_u32(&tl->a_full[ks]);
          if (lane == 0) mbar_arrive_expect_tx(ab, A_SLICE);
          if (GATHER) __syncwarp();
          load_a_slice<GATHER>(a_base + ks * A_SLICE, tmap_a, ks * BK_BYTES, u, a_rows, zero_row, ab, lane);
          last_a_use[ks] = unit_use;
        }
        if (lane == 0) mbar_arrive_expect_tx(fb, G.b_bytes + (G.sfb_tiles + 1) * nsf * 512 + b_off);
        if (GATHER) __syncwarp();
        if (!G.resident) load_a_slice<GATHER>(st, tmap_a, ks * BK_BYTES, u, a_rows, zero_row, fb, lane);
        if (lane == 0) {
          tma_load_2d(st + b_off, tmap_b, ks * BK_BYTES, b_row, fb);
          bulk_load(st + b_off + G.b_bytes, b_sf + (sfb_row + 4 * ks) * 512, nsf * 512, fb);
          if (G.pair) bulk_load(st + b_off + G.b_bytes + SF_STAGE, b_sf + (sfb_row2 + 4 * ks) * 512, nsf * 512, fb);
          bulk_load(st + b_off + G.b_bytes + G.sfb_tiles * SF_STAGE, a_sf + (sfa_row + 4 * ks) * 512, nsf * 512, fb);
        }
        last_stage_use[slot] = use;
      }
    }
  }
  if (aborted) {
    // let the copies this thread issued land before the CTA can exit
    for (int s = 0; s < MAX_STAGES; ++s)
      if (last_stage_use[s] != 0xFFFFFFFFu) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&tl->b_full[s]), last_stage_use[s] & 1u) && global_timer_ns() - t0 < WAIT_LIMIT_NS) {
        }
      }
    for (int ks = 0; ks < MAX_A_SLOTS; ++ks)
      if (last_a_use[ks] != 0xFFFFFFFFu) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&tl->a_full[ks]), last_a_use[ks] & 1u) && global_timer_ns() - t0 < WAIT_LIMIT_NS) {
        }
      }
  }
}

// Scale writer for lane quadrant qd (warp 8 + qd).  Per k-step, once the
// stage has landed: lane l (row or weight row 32*qd + l) stores
//   - the B scales of the four 64-wide K groups, replicated: columns
//     B0 + 4i + j hold bytes [16*l + 4j, +4) of B-scale tile i, exactly as
//     a 32x128b.warpx4 copy of the tile would place them in every quadrant;
//   - the A scales on the diagonal only: column A0 + 4i + qd holds the four
//     scale bytes of row 32*qd + l in A-scale tile i (bytes 16*l + 4*qd).
// Single CTAs: the stage's buffer is rewritten only after its next use has
// landed, which the producer issues only after the MMAs of the previous use
// completed.  CTA pairs with as many stages as scale buffers: the same.
// Otherwise the buffers form a ring of their own, and a buffer is rewritten
// once the commit of its previous MMAs (sf_empty, arriving in both CTAs)
// says they completed.
// The writers also wait for the resident A slice of the k-step (first item of
// a unit), so the MMA thread waits on sf_full alone: its completion implies
// that the stage's operands and the A slice have landed (in a pair, in both
// CTAs: all eight writer warps arrive on rank 0's barrier).
__device__ void sf_writer_loop(int qd, const Geometry& G, const int32_t* off, int E, uint32_t ring_base, Tail* tl,
                               uint32_t tmem, AbortFlag abort_flag, int* status) {
  const int lane = threadIdx.x & 31;
  const uint32_t b_off = G.b_off();
  const uint32_t tq = tmem + ((uint32_t)(qd * 32) << 16);
  uint32_t kc = 0;
  bool aborted = false;
  UnitCursor cur;
  int u, e;
  bool ghost;
  for (int iu = 0; !aborted && unit_at(G, off, E, iu, cur, u, e, ghost); ++iu) {
    const uint32_t unit_use = (uint32_t)iu;
    for (int q = 0; q < G.items && !aborted; ++q) {
      for (int ks = 0; ks < G.nk; ++ks, ++kc) {
        uint32_t slot, use, buf, buse;
        G.slot_of(kc, slot, use);
        G.sfbuf_of(kc, slot, use, buf, buse);
        bool ok = warp_wait(smem_u32(&tl->b_full[slot]), use & 1u, abort_flag, status);
        if (ok && G.resident && q == 0) ok = warp_wait(smem_u32(&tl->a_full[ks]), unit_use & 1u, abort_flag, status);
        if (ok && G.sf_ring()) ok = warp_wait(smem_u32(&tl->sf_empty[buf]), (buse & 1u) ^ 1u, abort_flag, status);
        if (!ok) { aborted = true; break; }
        tc_fence_after();
        const int nsf = min(4, G.kgroups - 4 * ks);
        const uint32_t sfb_s = ring_base + slot * G.stage_bytes + b_off + G.b_bytes;
        const uint32_t sfa_s = sfb_s + G.sfb_tiles * SF_STAGE;
        const uint32_t col = tq + G.sf_col() + buf * G.sf_cols;
        uint32_t wa[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) wa[i] = i < nsf ? lds32(sfa_s + 512 * i + 16 * lane + 4 * qd) : 0u;
        if (G.pair) {
          // N = 256: the B scales of MMA i take 8 columns, B rows 0-127 (the
          // gate tile) in the first 4 and rows 128-255 (the up tile) in the next
          uint32_t wb[32];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const uint4 v = i < nsf ? lds128(sfb_s + t * SF_STAGE + 512 * i + 16 * lane) : make_uint4(0u, 0u, 0u, 0u);
              wb[8 * i + 4 * t] = v.x; wb[8 * i + 4 * t + 1] = v.y; wb[8 * i + 4 * t + 2] = v.z; wb[8 * i + 4 * t + 3] = v.w;
            }
          tmem_st32(col + 16, wb);
        } else {
          uint32_t wb[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = i < nsf ? lds128(sfb_s + 512 * i + 16 * lane) : make_uint4(0u, 0u, 0u, 0u);
            wb[4 * i] = v.x; wb[4 * i + 1] = v.y; wb[4 * i + 2] = v.z; wb[4 * i + 3] = v.w;
          }
          tmem_st16(col + 16, wb);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) tmem_st1(col + 4 * i + qd, wa[i]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (G.pair)
            mbar_arrive_cluster(map_to_rank(smem_u32(&tl->sf_full[buf]), 0));
          else
            mbar_arrive(smem_u32(&tl->sf_full[buf]));
        }
      }
    }
  }
}

// PAIR: issued by rank 0 of the pair alone, as cta_group::2 MMAs over both
// CTAs' operands; every commit arrives in both CTAs.  Its waits (sf_full,
// tempty) also count arrivals from the peer's threads.
template <bool PAIR>
__device__ void mma_loop(const Geometry& G, const int32_t* off, int E, uint32_t a_base, uint32_t ring_base, Tail* tl,
                         uint32_t tmem, AbortFlag abort_flag, int* status) {
  // The per-k-step work of this single thread is the latency the tensor
  // pipe waits on, so everything that does not change per k-step is
  // computed here, and the ring position advances by increments: k-step kc
  // sits in ring r = kc % rings at position pos = kc / rings, in stage slot
  // r * S + pos % S, used for the (pos / S)-th time.
  const uint32_t R = (uint32_t)G.rings, lgS = (uint32_t)G.log2_stages, Smask = (1u << lgS) - 1u;
  const bool sf_ring = G.sf_ring();
  const uint32_t sf_full0 = smem_u32(&tl->sf_full[0]), b_empty0 = smem_u32(&tl->b_empty[0]);
  const uint32_t a_empty0 = smem_u32(&tl->a_empty[0]), sf_empty0 = smem_u32(&tl->sf_empty[0]);
  const uint32_t tempty0 = smem_u32(&tl->tempty[0]), tfull0 = smem_u32(&tl->tfull[0]);
  const uint32_t stage_desc = (uint32_t)G.stage_bytes >> 4;  // descriptor units (16 B) per stage
  const uint64_t bdesc0 = sdesc_k_sw128(ring_base + G.b_off());
  const uint64_t adesc0 = sdesc_k_sw128(G.resident ? a_base : ring_base);
  const uint32_t adesc_step = G.resident ? (uint32_t)(A_SLICE >> 4) : 0u;
  const uint32_t sf0 = tmem + G.sf_col();
  uint32_t kc = 0, it = 0, r = 0, pos = 0;
  bool aborted = false;
  UnitCursor cur;
  int u, e;
  bool ghost;
  for (int iu = 0; !aborted && unit_at(G, off, E, iu, cur, u, e, ghost); ++iu) {
    for (int q = 0; q < G.items && !aborted; ++q, ++it) {
      const uint32_t acc_slot = PAIR ? 0u : it % (uint32_t)G.nslot, suse = PAIR ? it : it / (uint32_t)G.nslot;
      if (!wait_bounded(tempty0 + 8u * acc_slot, (suse & 1u) ^ 1u, abort_flag, status)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t dacc = tmem + acc_slot * (uint32_t)G.acc_cols;
      const bool last_item = G.resident && q == G.items - 1;
      for (int ks = 0; ks < G.nk; ++ks, ++kc) {
        const uint32_t slot = (r << lgS) | (pos & Smask), use = pos >> lgS;
        const uint32_t buf = sf_ring ? (kc & (PAIR_SFBUF - 1)) : slot;
        const uint32_t buse = sf_ring ? kc / PAIR_SFBUF : use;
        if (++r == R) {
          r = 0;
          ++pos;
        }
        if (!wait_bounded(sf_full0 + 8u * buf, buse & 1u, abort_flag, status)) { aborted = true; break; }
        tc_fence_after();
        const int nmma = min(4, G.kgroups - 4 * ks);
        const uint32_t sf_a = sf0 + buf * (uint32_t)G.sf_cols;
        const uint64_t bdesc = bdesc0 + slot * stage_desc;
        const uint64_t adesc = adesc0 + (G.resident ? (uint32_t)ks * adesc_step : slot * stage_desc);
        if constexpr (PAIR) {
          const uint32_t sf_b = sf_a + 16;
          if (nmma == 4) {
            const uint32_t acc0 = ks != 0 ? 1u : 0u;
            tc_mma_pair(dacc, adesc, bdesc, sf_a, sf_b, acc0);
            tc_mma_pair(dacc, adesc + 2, bdesc + 2, sf_a + 4, sf_b + 8, 1u);
            tc_mma_pair(dacc, adesc + 4, bdesc + 4, sf_a + 8, sf_b + 16, 1u);
            tc_mma_pair(dacc, adesc + 6, bdesc + 6, sf_a + 12, sf_b + 24, 1u);
          } else {
            for (int i = 0; i < nmma; ++i)
              tc_mma_pair(dacc, adesc + 2 * i, bdesc + 2 * i, sf_a + 4 * i, sf_b + 8 * i, (ks | i) != 0 ? 1u : 0u);
          }
          tc_commit_pair(b_empty0 + 8u * slot);
          if (sf_ring) tc_commit_pair(sf_empty0 + 8u * buf);
          if (last_item) tc_commit_pair(a_empty0 + 8u * (uint32_t)ks);
        } else {
          const uint32_t sf_b = sf_a + 16;
          if (nmma == 4) {
            const uint32_t acc0 = ks != 0 ? 1u : 0u;
            tc_mma(dacc, adesc, bdesc, sf_a, sf_b, acc0);
            tc_mma(dacc, adesc + 2, bdesc + 2, sf_a + 4, sf_b + 4, 1u);
            tc_mma(dacc, adesc + 4, bdesc + 4, sf_a + 8, sf_b + 8, 1u);
            tc_mma(dacc, adesc + 6, bdesc + 6, sf_a + 12, sf_b + 12, 1u);
          } else {
            for (int i = 0; i < nmma; ++i)
              tc_mma(dacc, adesc + 2 * i, bdesc + 2 * i, sf_a + 4 * i, sf_b + 4 * i, (ks | i) != 0 ? 1u : 0u);
          }
          tc_commit(b_empty0 + 8u * slot);
          if (last_item) tc_commit(a_empty0 + 8u * (uint32_t)ks);
        }
      }
      if (!aborted) {
        if constexpr (PAIR)
          tc_commit_pair(tfull0 + 8u * acc_slot);
        else
          tc_commit(tfull0 + 8u * acc_slot);
      }
    }
  }
  // all MMAs of this CTA (pair) have completed once `done` fires
  if constexpr (PAIR)
    tc_commit_pair(smem_u32(&tl->done));
  else
    tc_commit(smem_u32(&tl->done));
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(smem_u32(&tl->done), 0u) && global_timer_ns() - t0 < WAIT_LIMIT_NS) {
  }
}

// Prologue: barriers and tensor memory.  PAIR: sf_full collects the writers
// of both CTAs and tempty the epilogue warps of both; the tensor memory is
// allocated for the pair (one warp in each CTA), and the cluster barrier
// makes both CTAs' barriers initialised before any arrival from the peer.
template <int NE, bool PAIR = false>
__device__ __forceinline__ Tail* setup(uint8_t* tail_ptr) {
  Tail* tl = reinterpret_cast<Tail*>(tail_ptr);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < MAX_A_SLOTS; ++s) {
      mbar_init(smem_u32(&tl->a_full[s]), 1);
      mbar_init(smem_u32(&tl->a_empty[s]), 1);
    }
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(smem_u32(&tl->b_full[s]), 1);
      mbar_init(smem_u32(&tl->b_empty[s]), 1);
      mbar_init(smem_u32(&tl->sf_full[s]), PAIR ? 8 : 4);
    }
    for (int s = 0; s < PAIR_SFBUF; ++s) mbar_init(smem_u32(&tl->sf_empty[s]), 1);
    for (int s = 0; s < NSLOT_MAX; ++s) {
      mbar_init(smem_u32(&tl->tfull[s]), 1);
      mbar_init(smem_u32(&tl->tempty[s]), PAIR ? 2 * NE : NE);
    }
    mbar_init(smem_u32(&tl->done), 1);
    tl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == Roles<NE>::MMA) {
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
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after();
  return tl;
}

// PAIR: the cluster barrier holds both CTAs (their shared and tensor
// memory, which the pair's MMAs read and write) until rank 0's MMA thread
// has seen all MMAs complete.
template <int NE, bool PAIR = false>
__device__ __forceinline__ void teardown(Tail* tl) {
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == Roles<NE>::MMA) {
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tl->tmem_base), "r"(TMEM_COLS)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tl->tmem_base), "r"(TMEM_COLS)
                   : "memory");
  }
}

// One 32-byte global store (address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Two FP32 -> BF16x2 (lo = first argument), round to nearest even.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// Codes of 16 BF16 values (8 packed words) for block scale S > 0 of a row
// with factor f = e2m1_row_factor(g).
__device__ __forceinline__ uint2 e2m1_block16(const uint32_t (&w)[8], float S, float f) {
  const uint32_t w0[4] = {w[0], w[1], w[2], w[3]}, w1[4] = {w[4], w[5], w[6], w[7]};
  return e2m1_codes16_div(w0, w1, S, f);
}

// Largest BF16 magnitude of 16 values (8 packed words), as a float.
__device__ __forceinline__ float amax16_bf16(const uint32_t (&w)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
  return __uint_as_float(__vmaxu2(m, m >> 16) << 16);
}

// Stage n floats (n % 4 == 0) from global into shared memory with the
// epilogue threads.
template <int NE>
__device__ __forceinline__ void stage_scales(float* dst, const float* src, int n, int tid) {
  for (int i = tid; i < n / 4; i += Roles<NE>::EPI_THREADS)
    reinterpret_cast<float4*>(dst)[i] = __ldg(reinterpret_cast<const float4*>(src) + i);
}

// FC1 requantisation of one thread's 32 columns (sub-part vp of chunk c,
// two blocks of 16) of row `row`, read back from the scratch vectors this
// thread staged: per block the E4M3 scale s_b = E4M3(a_b / (6 g)) and the
// E2M1 codes of h / (g s_b).  The two scale bytes are bytes 2*(vp % 2)
// and +1 of scale word 2c + vp/2.  Called by all 32 lanes of the warp: the
// scratch lines it has read are then dropped from L2 without a write-back
// (the buffer is rewritten before it is read again).
__device__ __forceinline__ void requant_chunk(const uint4* scr, int c, int vp, int rl, int64_t row, float g,
                                              float den, uint8_t* h_codes, uint8_t* h_sf, int d_ff) {
  uint4 cur[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) cur[v] = scr[(size_t)((c * FC1_VPARTS + vp) * 4 + v) * BM + rl];
  uint32_t sb2 = 0;
  uint32_t cw[4];
  const float rden = block_scale_rden(den);
  const float f = e2m1_row_factor(g);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t wb[8] = {cur[2 * b].x, cur[2 * b].y, cur[2 * b].z, cur[2 * b].w,
                            cur[2 * b + 1].x, cur[2 * b + 1].y, cur[2 * b + 1].z, cur[2 * b + 1].w};
    uint32_t sb = 0;
    uint2 p = make_uint2(0u, 0u);
    if (g != 0.0f) {
      sb = block_scale_code(amax16_bf16(wb), den, rden);
      const float S = __fmul_rn(g, e4m3_decode_hw(sb));
      if (S != 0.0f) p = e2m1_block16(wb, S, f);
    }
    cw[2 * b] = p.x;
    cw[2 * b + 1] = p.y;
    sb2 |= sb << (8 * b);
  }
  *reinterpret_cast<uint4*>(h_codes + row * (d_ff / 2) + (c * BN + vp * 32) / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  const int kgh = d_ff / 64;
  *reinterpret_cast<uint16_t*>(h_sf + ((row >> 7) * kgh + 2 * c + (vp >> 1)) * 512 + (row & 31) * 16 +
                               ((row >> 5) & 3) * 4 + 2 * (vp & 1)) = (uint16_t)sb2;
  // each 128-byte line holds 8 rows' 16 bytes: discarded once all 32 lanes
  // have used what they read
  __syncwarp();
  if ((rl & 7) == 0) {
#pragma unroll
    for (int v = 0; v < 4; ++v) discard_l2_line(scr + (size_t)((c * FC1_VPARTS + vp) * 4 + v) * BM + rl);
  }
}

// Shared roles of both GEMMs.  Returns true for the epilogue warps, which
// the caller then runs.  PAIR: rank 1's MMA warp has nothing to issue.
template <int NE, bool PAIR = false>
__device__ __forceinline__ bool run_pipeline_roles(const CUtensorMap* tmap_a, const CUtensorMap* tmap_b,
                                                   const uint8_t* a_sf, const uint8_t* b_sf, const Geometry& G,
                                                   const ItemRows& rows, const int32_t* off, int E, uint32_t a_base,
                                                   uint32_t ring_base, Tail* tl, int* status,
                                                   const int32_t* a_rows = nullptr, int zero_row = 0) {
  const AbortFlag abort_flag{smem_u32(&tl->abort_flag)};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  using RL = Roles<NE>;
  // 24 warps (16 epilogue) launch at 80 registers a thread; the epilogue's
  // four warpgroups take registers from the scale writers' group and from
  // the producers' and MMA issuer's group (sums: 4 x 96 + 56 + 40 = 6 x 80)
  constexpr bool SPLIT = NE == 16;
  if (warp >= RL::PROD && warp < RL::MMA) {
    if constexpr (SPLIT) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_PROD));
    if (lane == 0) {
      prefetch_tmap(tmap_a);
      prefetch_tmap(tmap_b);
    }
    if (a_rows)
      producer_loop<true>(warp - RL::PROD, tmap_a, tmap_b, a_sf, b_sf, G, rows, off, E, a_base, ring_base, tl,
                          abort_flag, status, a_rows, zero_row);
    else if (lane == 0)
      producer_loop<false>(warp - RL::PROD, tmap_a, tmap_b, a_sf, b_sf, G, rows, off, E, a_base, ring_base, tl,
                           abort_flag, status, nullptr, 0);
    __syncwarp();
    return false;
  }
  if (warp == RL::MMA) {
    if constexpr (SPLIT) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_PROD));
    if (lane == 0 && (!PAIR || G.rank == 0))
      mma_loop<PAIR>(G, off, E, a_base, ring_base, tl, tl->tmem_base, abort_flag, status);
    __syncwarp();
    return false;
  }
  if (warp >= RL::SFW && warp < RL::SFW + 4) {
    if constexpr (SPLIT) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_SFW));
    sf_writer_loop(warp - RL::SFW, G, off, E, ring_base, tl, tl->tmem_base, abort_flag, status);
    return false;
  }
  if constexpr (SPLIT) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REG_EPI));
  return true;
}

}  // namespace

// ---------------------------------------------------------------------------
// FC1 + SwiGLU + requantisation
// ---------------------------------------------------------------------------
// DBG: also write the debug outputs (pre-cast FP32 u, h before
// requantisation) when their pointers are set; the production launch uses
// the instantiation without them.  PAIR: launched in clusters of two CTAs
// that compute 256-row units with cta_group::2 MMAs of N = 256 (A resident;
// an item is one chunk, gate and up in one 256-column accumulator; rank 0
// holds the gate rows of B, rank 1 the up rows); each CTA runs the epilogue
// of its own 128 rows.
template <bool DBG, bool PAIR>
__global__ void __launch_bounds__(Roles<FC1_NE>::THREADS, 1) fc1_swiglu_kernel(const __grid_constant__ Fc1Args args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int d_ff = args.d_ff, nch = d_ff / BN;
  Geometry G;
  G.num_mt = __ldg(args.offsets + args.E) / BM;
  G.pair = PAIR;
  G.rank = PAIR ? cluster_rank() : 0u;
  G.cluster = PAIR ? (int)cluster_id_x() : 0;
  G.nclusters = PAIR ? (int)cluster_count_x() : 1;
  G.b_bytes = B_BYTES;
  G.sfb_tiles = PAIR ? 2 : 1;
  G.acc_cols = PAIR ? PAIR_ACC_COLS : BN;
  G.sf_cols = PAIR ? PAIR_SF_COLS : SF_COLS;
  G.items = PAIR ? nch : 2 * nch;
  G.nk = (args.d + 255) / 256;
  G.kgroups = args.d / 64;
  G.rings = args.rings;
  G.log2_stages = args.nb == 2 ? 1 : 0;
  G.nslot = PAIR ? 1 : FC1_NSLOT;
  G.resident = args.resident != 0;
  G.stage_bytes = (G.resident ? 0 : A_SLICE) + G.b_bytes + (G.sfb_tiles + 1) * SF_STAGE;
  const uint32_t a_base = smem_u32(smem);
  const size_t a_bytes = G.resident ? (size_t)G.nk * A_SLICE : 0;
  const size_t ring_bytes = (size_t)G.rings * (1 << G.log2_stages) * G.stage_bytes;
  const uint32_t ring_base = a_base + (uint32_t)a_bytes;
  Tail* tl = setup<FC1_NE, PAIR>(smem + a_bytes + ring_bytes);
  float* gw_s = reinterpret_cast<float*>(smem + a_bytes + ring_bytes + TAIL_BYTES);
  const AbortFlag abort_flag{smem_u32(&tl->abort_flag)};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ItemRows rows{true, 2 * d_ff, d_ff};
  // the accumulator release goes to rank 0's barrier, which counts both CTAs
  const uint32_t tempty0 = PAIR ? map_to_rank(smem_u32(&tl->tempty[0]), 0) : smem_u32(&tl->tempty[0]);

  if (run_pipeline_roles<FC1_NE, PAIR>(&args.tmap_a, &args.tmap_b, args.a_sf, args.w_sf, G, rows, args.offsets,
                                       args.E, a_base, ring_base, tl, args.status, args.a_rows, args.zero_row)) {
    // ---------------- epilogue warps ----------------
    const int q4 = warp & 3, part = warp >> 2;  // part: columns FC1_PART_COLS*part.. of each chunk
    const int rl = q4 * 32 + lane;              // row within the tile = TMEM lane
    // DBG: the saved u and h take 256-bit stores when 32-byte aligned
    const bool al32 = DBG && ((reinterpret_cast<uintptr_t>(args.save_u) | reinterpret_cast<uintptr_t>(args.dbg_h)) & 31u) == 0;
    const uint32_t tmem = tl->tmem_base + ((uint32_t)(q4 * 32) << 16) + part * FC1_PART_COLS;
    // Two scratch buffers per CTA: unit i stages h in buffer i % 2 while the
    // thread requantises its own row half of unit i - 1 from the other,
    // one chunk after each chunk of unit i (the thread reads back only what
    // it wrote, so program order is the only ordering needed).
    // (Pointers that live across the unit loop are recomputed where they are
    // used, from the kernel parameters: fewer registers held in the loop.)
    auto scratch_buf = [&](uint32_t parity) {
      return reinterpret_cast<uint4*>(args.scratch) + ((size_t)blockIdx.x * 2 + parity) * (size_t)(d_ff / 8) * BM;
    };
    // This thread's slots for SwiGLU pairs the bracket left open: their exact
    // values are computed at the end of the unit, so that the rare slow path
    // runs once per unit and not inside the item that met it (the next
    // accumulator release would wait for it).  Each slot: gate word, up word,
    // position (chunk << 5 | half << 3 | word).
    auto defer_slots = [&]() {
      return reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(args.scratch) + fc1_staging_bytes(d_ff)) +
             ((size_t)blockIdx.x * kFc1EpiThreads + threadIdx.x) * kFc1DeferSlots;
    };
    int ndefer = 0;
    bool have_prev = false, ghost_prev = false;
    int u_prev = 0;  // the previous unit's tile, staged in scratch_buf((uc - 1) & 1)
    float g_prev = 0.0f;  // its outer scale (the block-scale divisor is 6 g_prev)
    uint32_t it = 0, uc = 0;
    UnitCursor cur;
    int u, e;
    bool ghost;
    for (int iu = 0; unit_at(G, args.offsets, args.E, iu, cur, u, e, ghost); ++iu, ++uc) {
      const int64_t row = (int64_t)u * BM + rl;
      const bool out = !PAIR || !ghost;  // a ghost tile computes but writes nothing
      const float ga = args.a_g[row];
      // one buffer: every read of the previous unit's scales precedes the
      // end-of-unit barrier, which precedes this staging
      float* gws = gw_s;
      stage_scales<FC1_NE>(gws, args.w_g + (int64_t)e * 2 * d_ff, 2 * d_ff, threadIdx.x);
      epi_barrier<FC1_NE>();
      uint32_t amax2 = 0;  // packed BF16 magnitudes
      for (int c = 0; c < nch; ++c, it += PAIR ? 1 : 2) {
        // gate and up accumulators: two of the three slots, or the two halves
        // of the pair's 256-column accumulator
        const uint32_t sg = PAIR ? 0u : it % FC1_NSLOT, su = PAIR ? 0u : (it + 1) % FC1_NSLOT;
        const uint32_t gcol = PAIR ? 0u : sg * BN, ucol = PAIR ? (uint32_t)BN : su * BN;
        const int n0 = c * BN + part * FC1_PART_COLS;  // first h column of this thread
        bool ok = __all_sync(0xFFFFFFFFu, !abort_flag.raised());
        if (ok) ok = warp_wait(smem_u32(&tl->tfull[sg]), (PAIR ? it : it / FC1_NSLOT) & 1u, abort_flag, args.status);
        if (ok && !PAIR) ok = warp_wait(smem_u32(&tl->tfull[su]), ((it + 1) / FC1_NSLOT) & 1u, abort_flag, args.status);
        // Drain: halves of 16 columns, gate and up of a half in one
        // tensor-memory round trip; the accumulators are released as soon as
        // the last round trip has landed (before its scaling), so the next
        // MMAs wait for the round trips only.  u = BF16(acc * (g_x * g_w)) is
        // kept as packed pairs; the SwiGLU then runs from the registers: h =
        // BF16(silu(u_gate) * u_up), staged, with the row amax.
        uint32_t ugw[FC1_HALVES][8], uuw[FC1_HALVES][8];
        auto release = [&]() {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (PAIR) {
              mbar_arrive_cluster(tempty0);
            } else {
              mbar_arrive(tempty0 + sg * 8u);
              mbar_arrive(tempty0 + su * 8u);
            }
          }
        };
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int hh = 0; hh < FC1_HALVES; ++hh) {
            const int nh = n0 + hh * 16;
            uint32_t V[2][16];
            tmem_ld16(tmem + gcol + hh * 16, V[0]);
            tmem_ld16(tmem + ucol + hh * 16, V[1]);
            tmem_wait_ld();
            if (hh == FC1_HALVES - 1) release();
#pragma unroll
            for (int gu = 0; gu < 2; ++gu) {
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const float4 fs = *reinterpret_cast<const float4*>(gws + gu * d_ff + nh + i);
                const float ss[4] = {fs.x, fs.y, fs.z, fs.w};
#pragma unroll
                for (int jj = 0; jj < 4; jj += 2) {
                  const int m = i + jj;
                  const float y0 = __fmul_rn(__uint_as_float(V[gu][m]), __fmul_rn(ga, ss[jj]));
                  const float y1 = __fmul_rn(__uint_as_float(V[gu][m + 1]), __fmul_rn(ga, ss[jj + 1]));
                  if (gu) uuw[hh][m >> 1] = bf16x2_rn(y0, y1); else ugw[hh][m >> 1] = bf16x2_rn(y0, y1);
                  if (DBG && out && args.dbg_u) {
                    float* du = args.dbg_u + row * 2 * d_ff + gu * d_ff;
                    du[nh + m] = y0; du[nh + m + 1] = y1;
                  }
                }
              }
            }
          }
        } else {
          release();
        }
        if (ok) {
#pragma unroll
          for (int hh = 0; hh < FC1_HALVES; ++hh) {
            const int nh = n0 + hh * 16;
            // h = BF16(silu(u_gate) * u_up), rounded once; a row with g_x = 0
            // (all-zero activations, pad rows) has u = +0 and so h = +0
            uint32_t hp[8];
            if (ga != 0.0f) {
              uint32_t hmax;
              const uint32_t open = swiglu16_fast(ugw[hh], uuw[hh], hp, hmax);
              if (open) {
                // open pairs wait for the end of the unit in the slots (more
                // than fit: computed here); where the whole group is open
                // its bracket values may exceed the exact ones, so none of
                // them enters the amax (the exact values do, later)
                if (open & kSwigluAll) hmax = 0;
                uint4* defer = defer_slots();
#pragma unroll
                for (int w = 0; w < 8; ++w)
                  if (open & (1u << w)) {
                    if (ndefer < kFc1DeferSlots) {
                      defer[ndefer++] = make_uint4(ugw[hh][w], uuw[hh][w], (uint32_t)(c << 5 | hh << 3 | w), 0u);
                    } else {
                      hp[w] = swiglu_pair_exact(ugw[hh][w], uuw[hh][w]);
                      hmax = __vmaxu2(hmax, hp[w] & 0x7FFF7FFFu);
                    }
                  }
              }
              amax2 = __vmaxu2(amax2, hmax);
            } else {
#pragma unroll
              for (int w = 0; w < 8; ++w) hp[w] = 0u;
            }
            // the saved u and h (training forward): each lane writes its own
            // row's 32-byte segments, one 256-bit store each where the
            // buffers are 32-byte aligned (half the store transactions of
            // two 16-byte stores: training forward 3.39 -> 2.94 ms on the
            // 64k layer)
            if (DBG && out && args.save_u) {  // gate, then up
              uint16_t* su = args.save_u + row * 2 * d_ff + nh;
              if (al32) {
                st_global_v8(su, ugw[hh]);
                st_global_v8(su + d_ff, uuw[hh]);
              } else {
                uint4* sg4 = reinterpret_cast<uint4*>(su);
                uint4* su4 = reinterpret_cast<uint4*>(su + d_ff);
                sg4[0] = make_uint4(ugw[hh][0], ugw[hh][1], ugw[hh][2], ugw[hh][3]);
                sg4[1] = make_uint4(ugw[hh][4], ugw[hh][5], ugw[hh][6], ugw[hh][7]);
                su4[0] = make_uint4(uuw[hh][0], uuw[hh][1], uuw[hh][2], uuw[hh][3]);
                su4[1] = make_uint4(uuw[hh][4], uuw[hh][5], uuw[hh][6], uuw[hh][7]);
              }
            }
            if (DBG && out && args.dbg_h) {
              uint16_t* dh = args.dbg_h + row * d_ff + nh;
              if (al32) {
                st_global_v8(dh, hp);
              } else {
                uint4* dh4 = reinterpret_cast<uint4*>(dh);
                dh4[0] = make_uint4(hp[0], hp[1], hp[2], hp[3]);
                dh4[1] = make_uint4(hp[4], hp[5], hp[6], hp[7]);
              }
            }
            // staged h stays in L2 until it is requantised (evict last)
            uint4* sv = scratch_buf(uc & 1) + (size_t)((c * FC1_VPARTS + part * FC1_SUB) * 4 + 2 * hh) * BM + rl;
            const uint64_t pol = l2_evict_last();
            st_global_hint(sv, make_uint4(hp[0], hp[1], hp[2], hp[3]), pol);
            st_global_hint(sv + BM, make_uint4(hp[4], hp[5], hp[6], hp[7]), pol);
          }
        }
        if (__all_sync(0xFFFFFFFFu, have_prev && !ghost_prev && !abort_flag.raised()))
#pragma unroll
          for (int sp = 0; sp < FC1_SUB; ++sp)
            requant_chunk(scratch_buf((uc - 1) & 1), c, part * FC1_SUB + sp, rl, (int64_t)u_prev * BM + rl, g_prev,
                          __fmul_rn(6.0f, g_prev), args.h_codes, args.h_sf, d_ff);
      }
      // deferred pairs: exact values over the bracket's in the staged h (and
      // the debug copy), and into the row amax
      for (int i = 0; i < ndefer; ++i) {
        const uint4 en = defer_slots()[i];
        const uint32_t hw = swiglu_pair_exact(en.x, en.y);
        const int c = (int)(en.z >> 5), hh = (int)(en.z >> 3) & 3, w = (int)en.z & 7;
        reinterpret_cast<uint32_t*>(scratch_buf(uc & 1) +
                                    (size_t)((c * FC1_VPARTS + part * FC1_SUB) * 4 + 2 * hh + (w >> 2)) * BM + rl)[w & 3] =
            hw;
        amax2 = __vmaxu2(amax2, hw & 0x7FFF7FFFu);
        if (DBG && out && args.dbg_h)
          reinterpret_cast<uint32_t*>(args.dbg_h + row * d_ff + c * BN + part * FC1_PART_COLS + hh * 16)[w] = hw;
      }
      ndefer = 0;
      // ---- outer scale of the unit's rows: amax over the full d_ff row ----
      tl->rowmax[part][rl] = __uint_as_float(__vmaxu2(amax2, amax2 >> 16) << 16);
      epi_barrier<FC1_NE>();
      float a = tl->rowmax[0][rl];
#pragma unroll
      for (int p2 = 1; p2 < FC1_PARTS; ++p2) a = fmaxf(a, tl->rowmax[p2][rl]);
      if (have_prev && !ghost_prev && part == 0) args.h_g[(int64_t)u_prev * BM + rl] = g_prev;
      if (out && !abort_flag.raised() && !is_finite_f32(a)) set_status(args.status, MOE_STATUS_NONFINITE_X);
      have_prev = true;
      ghost_prev = !out;
      u_prev = u;
      g_prev = __fdiv_rn(a, 2688.0f);
    }
    // the last unit
    if (have_prev && !ghost_prev) {
      if (__all_sync(0xFFFFFFFFu, !abort_flag.raised()))
        for (int c = 0; c < nch; ++c)
          for (int sp = 0; sp < FC1_SUB; ++sp)
            requant_chunk(scratch_buf((uc - 1) & 1), c, part * FC1_SUB + sp, rl, (int64_t)u_prev * BM + rl, g_prev,
                          __fmul_rn(6.0f, g_prev), args.h_codes, args.h_sf, d_ff);
      if (part == 0) args.h_g[(int64_t)u_prev * BM + rl] = g_prev;
    }
  }
  teardown<FC1_NE, PAIR>(tl);
}

// ---------------------------------------------------------------------------
// FC2 + router-weighted scatter
// ---------------------------------------------------------------------------
// MODE 0: the forward (z rows).  MODE 1: also the debug output (pre-weighting
// FP32 y2).  MODE 2: the straight-through backward's recomputation of the
// same y2 (same code, same results) against the output gradient: dw[t][j] =
// sum_n dY[t][n] y2[row][n] (FP32) and the BF16 dgrad operand dy2[row] =
// BF16(w_tj dY[t]) written in place of the z rows (zero on pad rows).  The
// output rows (z or dy2, [m_cap][d] BF16) leave through args.tmap_out; pad
// rows come out as zeros (their h and router weight are zero).
template <int MODE>
__global__ void __launch_bounds__(Roles<FC2_NE>::THREADS, 1) fc2_scatter_kernel(const __grid_constant__ Fc2Args args) {
  constexpr bool DBG = MODE == 1, DW = MODE == 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int d = args.d, k = args.k;
  Geometry G;
  G.num_mt = __ldg(args.offsets + args.E) / BM;
  G.pair = false;
  G.rank = 0u;
  G.cluster = 0;
  G.nclusters = 1;
  G.b_bytes = B_BYTES;
  G.sfb_tiles = 1;
  G.acc_cols = BN;
  G.sf_cols = SF_COLS;
  G.items = d / BN;
  G.nk = (args.d_ff + 255) / 256;
  G.kgroups = args.d_ff / 64;
  G.rings = args.rings;
  G.log2_stages = args.nb == 2 ? 1 : 0;
  G.nslot = FC2_NSLOT;
  G.resident = args.resident != 0;
  G.stage_bytes = (G.resident ? 0 : A_SLICE) + G.b_bytes + 2 * SF_STAGE;
  const uint32_t a_base = smem_u32(smem);
  const size_t a_bytes = G.resident ? (size_t)G.nk * A_SLICE : 0;
  const size_t ring_bytes = (size_t)G.rings * (1 << G.log2_stages) * G.stage_bytes;
  const uint32_t ring_base = a_base + (uint32_t)a_bytes;
  Tail* tl = setup<FC2_NE>(smem + a_bytes + ring_bytes);
  float* gw_s = reinterpret_cast<float*>(smem + a_bytes + ring_bytes + TAIL_BYTES);
  const AbortFlag abort_flag{smem_u32(&tl->abort_flag)};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ItemRows rows{false, d, args.d_ff};
  // per epilogue warp: 32 rows x 64 BF16 columns, 16-byte chunks XOR-swizzled by row
  const uint32_t stg = smem_u32(smem + a_bytes + ring_bytes + TAIL_BYTES + (size_t)2 * d * 4) +
                       (uint32_t)(warp < FC2_NE ? warp : 0) * 32 * FC2_STAGE_ROW;
  // DW: a second tile per warp, after all output tiles, for the copied-in
  // output gradient
  const uint32_t dyb = stg + FC2_STAGING_BYTES;

  if (run_pipeline_roles<FC2_NE>(&args.tmap_a, &args.tmap_b, args.a_sf, args.w_sf, G, rows, args.offsets, args.E, a_base,
                         ring_base, tl, args.status)) {
    const int q4 = warp & 3, part = warp >> 2;
    const int rl = q4 * 32 + lane;
    const uint32_t tmem = tl->tmem_base + ((uint32_t)(q4 * 32) << 16) + part * 64;
    uint32_t it = 0, uc = 0;
    bool stores = false;  // lane 0: a tensor store of this warp may be in flight
    if (lane == 0) prefetch_tmap(&args.tmap_out);
    for (int u = blockIdx.x; u < G.num_mt; u += gridDim.x, ++uc) {
      const int e = expert_of(args.offsets, args.E, u);
      const int64_t row = (int64_t)u * BM + rl;
      const int t = args.row_to_token[row];
      int j = 0;
      float w = 0.0f;
      if (t >= 0) {
        // slot of this row among the token's k (loads issued eight at a time)
        const int32_t* ts = args.token_slot_row + (int64_t)t * k;
        for (int j0 = 0; j0 < k; j0 += 8) {
          int v8[8];
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) v8[q8] = j0 + q8 < k ? ts[j0 + q8] : -1;
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8)
            if (v8[q8] == (int)row) j = j0 + q8;
        }
        w = args.topk_w[(int64_t)t * k + j];
      }
      const float gh = args.a_g[row];
      float* gws = gw_s + (uc & 1) * d;
      stage_scales<FC2_NE>(gws, args.w_g + (int64_t)e * d, d, threadIdx.x);
      epi_barrier<FC2_NE>();
      const uint16_t* dy_row = DW ? args.dY + (int64_t)(t < 0 ? 0 : t) * d : nullptr;
      float dot = 0.0f;
      // DW: an item's 32 output-gradient row segments (64 columns each) are
      // copied asynchronously into the warp's input tile (8 lanes per row, 4
      // rows per instruction) while the item before is processed
      auto issue_dy = [&](int nt) {
        const unsigned long long my_src =
            t >= 0 ? reinterpret_cast<unsigned long long>(dy_row + nt * BN + part * 64) : 0ull;
        const int sub = lane >> 3, ch = lane & 7;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = i * 4 + sub;
          const unsigned long long sp = __shfl_sync(0xFFFFFFFFu, my_src, rr);
          cp_async16(dyb + rr * FC2_STAGE_ROW + 16 * (ch ^ (rr & 7)),
                     sp ? reinterpret_cast<const uint4*>(sp) + ch : reinterpret_cast<const uint4*>(args.dY), sp != 0);
        }
        cp_async_commit();
      };
      if (DW) {
        __syncwarp();  // every lane is done with the previous unit's input tile
        issue_dy(0);
      }
      for (int nt = 0; nt < G.items; ++nt, ++it) {
        const uint32_t slot = it % FC2_NSLOT;
        bool ok = __all_sync(0xFFFFFFFFu, !abort_flag.raised());
        if (ok) ok = warp_wait(smem_u32(&tl->tfull[slot]), (it / FC2_NSLOT) & 1u, abort_flag, args.status);
        // Drain the accumulator (this thread's 64 columns) into registers,
        // release it to the MMA warp, then scale, weight and store.
        uint32_t R[4][16];
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int hf = 0; hf < 4; ++hf) tmem_ld16(tmem + slot * BN + hf * 16, R[hf]);
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tl->tempty[slot]));
        if (ok) {
          // the staging tile is free once the previous store has read it
          if (lane == 0 && stores) bulk_wait_read0();
          __syncwarp();
          if (DW) {  // this item's output-gradient segments have landed
            cp_async_wait_all();
            __syncwarp();
          }
          // scale and weight into the staging tile (the 128-byte-swizzled
          // layout of the destination tensor map), then one TMA store of the
          // warp's 32 rows x 64 columns
#pragma unroll
          for (int hf = 0; hf < 4; ++hf) {
            const int n0 = nt * BN + part * 64 + hf * 16;
            uint32_t zp[8];
            float yv[16];
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 f4 = *reinterpret_cast<const float4*>(gws + n0 + i);
              const float f[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
              for (int jj = 0; jj < 4; jj += 2) {
                const int m = i + jj;
                const float y0 = __fmul_rn(__uint_as_float(R[hf][m]), __fmul_rn(gh, f[jj]));
                const float y1 = __fmul_rn(__uint_as_float(R[hf][m + 1]), __fmul_rn(gh, f[jj + 1]));
                if (!DW) zp[m >> 1] = bf16x2_rn(__fmul_rn(w, y0), __fmul_rn(w, y1));
                yv[m] = y0;
                yv[m + 1] = y1;
              }
            }
            if (DW) {  // this row's 16 output-gradient columns, from the staging tile
              const uint4 g0 = lds128(dyb + lane * FC2_STAGE_ROW + 16 * ((2 * hf) ^ (lane & 7)));
              const uint4 g1 = lds128(dyb + lane * FC2_STAGE_ROW + 16 * ((2 * hf + 1) ^ (lane & 7)));
              const uint32_t gw4[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float d0 = bf16_lo(gw4[q]), d1 = bf16_hi(gw4[q]);
                dot = fmaf(d0, yv[2 * q], dot);
                dot = fmaf(d1, yv[2 * q + 1], dot);
                zp[q] = bf16x2_rn(__fmul_rn(w, d0), __fmul_rn(w, d1));
              }
            }
            if (DBG && args.dbg_y && t >= 0) {  // two 32-byte sectors
              float4* y4 = reinterpret_cast<float4*>(args.dbg_y + row * d + n0);
#pragma unroll
              for (int q = 0; q < 4; ++q) y4[q] = make_float4(yv[4 * q], yv[4 * q + 1], yv[4 * q + 2], yv[4 * q + 3]);
            }
            sts128(stg + lane * FC2_STAGE_ROW + 16 * ((2 * hf) ^ (lane & 7)), zp[0], zp[1], zp[2], zp[3]);
            sts128(stg + lane * FC2_STAGE_ROW + 16 * ((2 * hf + 1) ^ (lane & 7)), zp[4], zp[5], zp[6], zp[7]);
          }
          if (DW && nt + 1 < G.items) {  // the input tile is free again
            __syncwarp();
            issue_dy(nt + 1);
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&args.tmap_out, stg, nt * BN + part * 64, u * BM + q4 * 32);
            stores = true;
          }
        }
      }
      if (DW) {  // dw of the row: the two column parts' sums, part 0 + part 1
        tl->rowmax[part][rl] = dot;
        epi_barrier<FC2_NE>();
        if (part == 0 && t >= 0) args.dw[(int64_t)t * k + j] = dot + tl->rowmax[1][rl];
      }
    }
    if (DW) cp_async_wait_all();  // no copy into shared memory outlives the CTA
    if (lane == 0 && stores) bulk_wait0();  // the stores complete before the CTA exits
    __syncwarp();
  }
  teardown<FC2_NE>(tl);
}


// FC2 on CTA pairs (MODE as fc2_scatter_kernel's): clusters of two CTAs, a
// unit being two 128-row tiles of one expert, walked as FC1's pair units
// (ghost tile included).  An item is 256 output columns: rank 0's B tile
// holds W2 rows nt*256 .. +127, rank 1's the next 128; one cta_group::2 MMA
// of M = 256, N = 256, K = 64 per 64-deep K group into one 256-column
// accumulator per CTA.  16 epilogue warps: warp w drains TMEM lane quadrant
// w % 4 and accumulator columns 64 (w / 4) .., in two round trips of 32
// columns; the accumulator is released (to rank 0's barrier) once the
// second round trip has landed; z = BF16(w * acc * (g_h * g_w2)) goes
// through the warp's swizzled 32 x 64 staging tile to one TMA tensor store,
// as in the single-CTA kernel.  A ghost tile computes but stores nothing.
// MODE 2: the staging tile first receives the item's output-gradient
// segments (cp.async, issued before the accumulator wait); each row's dY
// values are read back for dw and replaced by dy2 = BF16(w dY) in place,
// which then leaves by the tile's TMA store.  dw of a row: the four column
// parts' sums, ((p0 + p1) + p2) + p3.
template <int MODE>
__global__ void __launch_bounds__(Roles<FC2P_NE>::THREADS, 1) fc2_pair_kernel(const __grid_constant__ Fc2Args args) {
  constexpr bool DBG = MODE == 1, DW = MODE == 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int d = args.d, k = args.k;
  Geometry G;
  G.num_mt = __ldg(args.offsets + args.E) / BM;
  G.pair = true;
  G.rank = cluster_rank();
  G.cluster = (int)cluster_id_x();
  G.nclusters = (int)cluster_count_x();
  G.b_bytes = B_BYTES;
  G.sfb_tiles = 2;
  G.acc_cols = PAIR_ACC_COLS;
  G.sf_cols = PAIR_SF_COLS;
  G.items = d / (2 * BN);
  G.nk = (args.d_ff + 255) / 256;
  G.kgroups = args.d_ff / 64;
  G.rings = args.rings;
  G.log2_stages = 0;
  G.nslot = 1;
  G.resident = true;
  G.stage_bytes = G.b_bytes + 3 * SF_STAGE;
  const uint32_t a_base = smem_u32(smem);
  const size_t a_bytes = (size_t)G.nk * A_SLICE;
  const size_t ring_bytes = (size_t)G.rings * G.stage_bytes;
  const uint32_t ring_base = a_base + (uint32_t)a_bytes;
  Tail* tl = setup<FC2P_NE, true>(smem + a_bytes + ring_bytes);
  float* gw_s = reinterpret_cast<float*>(smem + a_bytes + ring_bytes + TAIL_BYTES);
  const AbortFlag abort_flag{smem_u32(&tl->abort_flag)};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ItemRows rows{false, d, args.d_ff};
  const uint32_t stg = smem_u32(smem + a_bytes + ring_bytes + TAIL_BYTES + (size_t)2 * d * 4) +
                       (uint32_t)(warp < FC2P_NE ? warp : 0) * 32 * FC2_STAGE_ROW;
  const uint32_t tempty0 = map_to_rank(smem_u32(&tl->tempty[0]), 0);

  if (run_pipeline_roles<FC2P_NE, true>(&args.tmap_a, &args.tmap_b, args.a_sf, args.w_sf, G, rows, args.offsets,
                                        args.E, a_base, ring_base, tl, args.status)) {
    const int q4 = warp & 3, part = warp >> 2;  // part: accumulator columns 64*part ..
    const int rl = q4 * 32 + lane;
    const uint32_t tmem = tl->tmem_base + ((uint32_t)(q4 * 32) << 16) + part * 64;
    uint32_t it = 0, uc = 0;
    bool stores = false;  // lane 0: a tensor store of this warp may be in flight
    if (lane == 0) prefetch_tmap(&args.tmap_out);
    UnitCursor cur;
    int u, e;
    bool ghost;
    for (int iu = 0; unit_at(G, args.offsets, args.E, iu, cur, u, e, ghost); ++iu, ++uc) {
      const int64_t row = (int64_t)u * BM + rl;
      const int t = args.row_to_token[row];
      float w = 0.0f;
      int j = 0;
      if (t >= 0) {
        // slot of this row among the token's k (loads issued eight at a time)
        const int32_t* ts = args.token_slot_row + (int64_t)t * k;
        for (int j0 = 0; j0 < k; j0 += 8) {
          int v8[8];
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) v8[q8] = j0 + q8 < k ? ts[j0 + q8] : -1;
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8)
            if (v8[q8] == (int)row) j = j0 + q8;
        }
        w = args.topk_w[(int64_t)t * k + j];
      }
      const float gh = args.a_g[row];
      float* gws = gw_s + (uc & 1) * d;
      stage_scales<FC2P_NE>(gws, args.w_g + (int64_t)e * d, d, threadIdx.x);
      epi_barrier<FC2P_NE>();
      // DW: the row's output gradient, and its partial dot product with y2
      const uint16_t* dy_row = DW ? args.dY + (int64_t)(t < 0 ? 0 : t) * d : nullptr;
      float dot = 0.0f;
      for (int nt = 0; nt < G.items; ++nt, ++it) {
        if (DW && !ghost) {
          // the staging tile receives this item's 32 output-gradient row
          // segments (64 columns each; 8 lanes per row, 4 rows per
          // instruction, zeros for pad rows) once the previous store has
          // read it
          if (lane == 0 && stores) bulk_wait_read0();
          __syncwarp();
          const unsigned long long my_src =
              t >= 0 ? reinterpret_cast<unsigned long long>(dy_row + nt * 2 * BN + part * 64) : 0ull;
          const int sub = lane >> 3, ch = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = i * 4 + sub;
            const unsigned long long sp = __shfl_sync(0xFFFFFFFFu, my_src, rr);
            cp_async16(stg + rr * FC2_STAGE_ROW + 16 * (ch ^ (rr & 7)),
                       sp ? reinterpret_cast<const uint4*>(sp) + ch : reinterpret_cast<const uint4*>(args.dY), sp != 0);
          }
          cp_async_commit();
        }
        bool ok = __all_sync(0xFFFFFFFFu, !abort_flag.raised());
        if (ok) ok = warp_wait(smem_u32(&tl->tfull[0]), it & 1u, abort_flag, args.status);
        auto release = [&]() {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty0);
        };
        uint32_t zp[32];  // the row's 64 z (DW: dy2) values, packed pairs
        if (ok) {
          tc_fence_after();
          if (DW && !ghost) {  // this item's output-gradient segments have landed
            cp_async_wait_all();
            __syncwarp();
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t R[2][16];
            tmem_ld16(tmem + hh * 32, R[0]);
            tmem_ld16(tmem + hh * 32 + 16, R[1]);
            tmem_wait_ld();
            if (hh == 1) release();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int c0 = hh * 32 + hf * 16;  // column within the warp's 64
              const int n0 = nt * 2 * BN + part * 64 + c0;
              float yv[16];
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const float4 f4 = *reinterpret_cast<const float4*>(gws + n0 + i);
                const float f[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                for (int jj = 0; jj < 4; jj += 2) {
                  const int m = i + jj;
                  const float y0 = __fmul_rn(__uint_as_float(R[hf][m]), __fmul_rn(gh, f[jj]));
                  const float y1 = __fmul_rn(__uint_as_float(R[hf][m + 1]), __fmul_rn(gh, f[jj + 1]));
                  if (!DW) zp[(c0 + m) >> 1] = bf16x2_rn(__fmul_rn(w, y0), __fmul_rn(w, y1));
                  yv[m] = y0;
                  yv[m + 1] = y1;
                }
              }
              if (DW && !ghost) {  // this row's 16 output-gradient columns, from the staging tile
                const int c8 = c0 >> 3;  // 16-byte chunk of the row
                const uint4 g0 = lds128(stg + lane * FC2_STAGE_ROW + 16 * (c8 ^ (lane & 7)));
                const uint4 g1 = lds128(stg + lane * FC2_STAGE_ROW + 16 * ((c8 + 1) ^ (lane & 7)));
                const uint32_t gw4[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const float d0 = bf16_lo(gw4[q]), d1 = bf16_hi(gw4[q]);
                  dot = fmaf(d0, yv[2 * q], dot);
                  dot = fmaf(d1, yv[2 * q + 1], dot);
                  zp[(c0 >> 1) + q] = bf16x2_rn(__fmul_rn(w, d0), __fmul_rn(w, d1));
                }
              }
              if (DBG && args.dbg_y && t >= 0 && !ghost) {
                float4* y4 = reinterpret_cast<float4*>(args.dbg_y + row * d + n0);
#pragma unroll
                for (int q = 0; q < 4; ++q) y4[q] = make_float4(yv[4 * q], yv[4 * q + 1], yv[4 * q + 2], yv[4 * q + 3]);
              }
            }
          }
        } else {
          release();
        }
        if (ok && !ghost) {
          // the staging tile is free once the previous store has read it
          // (DW: that was waited for before the output gradient came in, and
          // each lane overwrites only its own row, which it has read)
          if (!DW && lane == 0 && stores) bulk_wait_read0();
          __syncwarp();
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            sts128(stg + lane * FC2_STAGE_ROW + 16 * (ch ^ (lane & 7)), zp[4 * ch], zp[4 * ch + 1], zp[4 * ch + 2],
                   zp[4 * ch + 3]);
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            // evict-first: the 2.15 GB of z rows pass through L2 once, and
            // should not push out the W2 tiles other clusters still read
            // (DW: dy2, which the next GEMM reads, keeps the default policy)
            if (DW)
              tma_store_2d(&args.tmap_out, stg, nt * 2 * BN + part * 64, u * BM + q4 * 32);
            else
              tma_store_2d_hint(&args.tmap_out, stg, nt * 2 * BN + part * 64, u * BM + q4 * 32, l2_evict_first());
            stores = true;
          }
        }
      }
      if (DW) {  // dw of the row: the four column parts' sums in a fixed order
        tl->rowmax[part][rl] = dot;
        epi_barrier<FC2P_NE>();
        if (part == 0 && t >= 0 && !ghost)
          args.dw[(int64_t)t * k + j] = ((dot + tl->rowmax[1][rl]) + tl->rowmax[2][rl]) + tl->rowmax[3][rl];
      }
      // every read of this unit's scale buffer precedes the barrier that
      // precedes the staging of the unit after next into it
    }
    if (DW) cp_async_wait_all();  // no copy into shared memory outlives the CTA
    if (lane == 0 && stores) bulk_wait0();  // the stores complete before the CTA exits
    __syncwarp();
  }
  teardown<FC2P_NE, true>(tl);
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
int gemm_num_ctas() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms < kMaxGemmCtas ? sms : kMaxGemmCtas;
}

// Pipeline plan for reduction length K, `items` accumulator tiles per unit,
// `scale_bytes` of per-column scales staged per unit and `extra`
// bytes of epilogue staging.  The tensor memory after the accumulators holds
// one scale buffer per stage; rings are 3 or 4, stages per ring 1 or 2, and
// the plan takes the most stages that fit.  A is resident (loaded once per
// unit) when its slices fit beside the rings and a unit spans enough
// k-steps: a producer runs up to rings*S k-steps ahead of the MMAs, and
// (items + 1) * nk >= rings*S keeps it from reaching the A slots of unit m
// before the slots of unit m-2 are released, so the parity of every a_empty
// wait is unambiguous.  Otherwise A streams through the stages with B.
static bool plan(int K, int items, size_t scale_bytes, int nslot, size_t extra, int* rings, int* na, int* nb,
                 int* resident, size_t* smem) {
  const int nk = (K + 255) / 256;
  const size_t fixed = 1024 /* alignment */ + TAIL_BYTES + scale_bytes + extra;
  if (fixed >= (size_t)SMEM_LIMIT) return false;
  const size_t avail = SMEM_LIMIT - fixed;
  static const int cand[4][2] = {{4, 2}, {3, 2}, {4, 1}, {3, 1}};  // (rings, stages per ring), most stages first
  for (int pass = 0; pass < 2; ++pass) {  // pass 0: A resident, pass 1: A streamed
    for (const auto& c : cand) {
      const int R = c[0], S = c[1];
      if (nslot * BN + R * S * SF_COLS > TMEM_COLS) continue;
      size_t need;
      if (pass == 0) {
        if (nk > MAX_A_SLOTS || (int64_t)(items + 1) * nk < (int64_t)R * S) continue;
        need = (size_t)nk * A_SLICE + (size_t)R * S * B_STAGE;
      } else {
        need = (size_t)R * S * (A_SLICE + B_STAGE);
      }
      if (need > avail) continue;
      *rings = R;
      *nb = S;
      *resident = pass == 0 ? 1 : 0;
      *na = pass == 0 ? nk : 0;
      *smem = fixed + need;
      return true;
    }
  }
  return false;
}

static int set_smem(const void* kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess ? 0 : -1;
}

// Persistent grid: one CTA per SM, but no more CTAs than the m_cap / 128
// row tiles the launch can have (the actual count is read on the device).
static int fc_grid(int64_t m_cap) {
  int grid = gemm_num_ctas();
  if (grid <= 0) return -1;
  const int64_t tiles = m_cap / BM;
  if (tiles < grid) grid = tiles < 1 ? 1 : (int)tiles;
  return grid;
}

// CTA-pair plan: A resident, PAIR_RINGS_MAX (or one fewer) rings of one
// PAIR_STAGE stage each, PAIR_SFBUF scale buffers after the accumulator.
// The a_empty reach rule is the single-CTA plan's.
static bool plan_pair(int K, int items, size_t scale_bytes, size_t extra, int* rings, size_t* smem) {
  const int nk = (K + 255) / 256;
  if (PAIR_ACC_COLS + PAIR_SFBUF * PAIR_SF_COLS > TMEM_COLS) return false;
  for (int R = PAIR_RINGS_MAX; R >= PAIR_RINGS_MAX - 1; --R) {
    if (nk > MAX_A_SLOTS || (int64_t)(items + 1) * nk < R) continue;
    const size_t need = 1024 + TAIL_BYTES + scale_bytes + extra + (size_t)nk * A_SLICE + (size_t)R * PAIR_STAGE;
    if (need > (size_t)SMEM_LIMIT) continue;
    *rings = R;
    *smem = need;
    return true;
  }
  return false;
}

// Clusters of two that can be resident at once with `smem` bytes per CTA of
// `threads` threads (the occupancy query is cached per host thread, keyed by
// device, kernel and shared-memory size).
template <class Args>
static int pair_clusters(void (*kern)(const Args), size_t smem, int threads) {
  thread_local void (*cached_kern)(const Args) = nullptr;
  thread_local size_t cached_smem = 0;
  thread_local int cached_dev = -1, cached = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (kern == cached_kern && smem == cached_smem && dev == cached_dev) return cached;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cached_kern = kern;
  cached_smem = smem;
  cached_dev = dev;
  cached = n;
  return n;
}

// FC1 runs on CTA pairs (clusters of two, cta_group::2 MMAs) when the pair
// plan fits and the device can hold clusters of two (A rows loaded as boxes
// or gathered alike: each CTA loads its own tile's rows);
// MOE_FC1_CTA_PAIRS=0 in the environment selects single CTAs throughout.
int launch_fc1(Fc1Args& a, int64_t m_cap, cudaStream_t stream) {
  const bool dbg = a.dbg_u != nullptr || a.dbg_h != nullptr || a.save_u != nullptr;
  const char* env = std::getenv("MOE_FC1_CTA_PAIRS");
  const bool allow_pairs = !(env && env[0] == '0');
  size_t smem;
  int pair_rings = 0;
  if (allow_pairs && plan_pair(a.d, a.d_ff / BN, (size_t)2 * a.d_ff * 4, 0, &pair_rings, &smem)) {
    void (*kern)(const Fc1Args) = dbg ? fc1_swiglu_kernel<true, true> : fc1_swiglu_kernel<false, true>;
    if (set_smem((const void*)kern, smem) != 0) return -1;
    int clusters = pair_clusters(kern, smem, Roles<FC1_NE>::THREADS);
    const int sms = gemm_num_ctas();
    if (sms > 0 && clusters > sms / 2) clusters = sms / 2;
    // every pair unit holds at least one of the m_cap / 128 tiles (the device
    // walks the actual units)
    const int64_t pair_units = m_cap / BM;
    if (pair_units < clusters) clusters = (int)pair_units;
    if (clusters >= 1) {
      a.rings = pair_rings;
      a.nb = 1;
      a.resident = 1;
      a.na = (a.d + 255) / 256;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(2 * clusters));
      cfg.blockDim = dim3(Roles<FC1_NE>::THREADS);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess ? 0 : -1;
    }
  }
  if (!plan(a.d, 2 * (a.d_ff / BN), (size_t)2 * a.d_ff * 4, FC1_NSLOT, 0, &a.rings, &a.na, &a.nb, &a.resident, &smem))
    return -1;
  void (*kern)(const Fc1Args) = dbg ? fc1_swiglu_kernel<true, false> : fc1_swiglu_kernel<false, false>;
  if (set_smem((const void*)kern, smem) != 0) return -1;
  const int grid = fc_grid(m_cap);
  if (grid <= 0) return -1;
  kern<<<grid, Roles<FC1_NE>::THREADS, smem, stream>>>(a);
  return 0;
}

// FC2 runs on CTA pairs (clusters of two) where the pair plan fits, d is a
// multiple of 256 and clusters of two can be resident, the forward and the
// backward's recomputation (dw set) alike; elsewhere on single CTAs.
// MOE_FC2_CTA_PAIRS=0 in the environment selects single CTAs throughout.
int launch_fc2(Fc2Args& a, int64_t m_cap, cudaStream_t stream) {
  size_t smem;
  const char* env = std::getenv("MOE_FC2_CTA_PAIRS");
  const bool allow_pairs = !(env && env[0] == '0') && a.d % (2 * BN) == 0;
  int pair_rings = 0;
  if (allow_pairs && plan_pair(a.d_ff, a.d / (2 * BN), (size_t)2 * a.d * 4, (size_t)FC2P_NE * 32 * FC2_STAGE_ROW,
                               &pair_rings, &smem)) {
    void (*kern)(const Fc2Args) = a.dw != nullptr      ? fc2_pair_kernel<2>
                                   : a.dbg_y != nullptr ? fc2_pair_kernel<1>
                                                        : fc2_pair_kernel<0>;
    if (set_smem((const void*)kern, smem) != 0) return -1;
    int clusters = pair_clusters(kern, smem, Roles<FC2P_NE>::THREADS);
    const int sms = gemm_num_ctas();
    if (sms > 0 && clusters > sms / 2) clusters = sms / 2;
    const int64_t pair_units = m_cap / BM;
    if (pair_units < clusters) clusters = (int)pair_units;
    if (clusters >= 1) {
      a.rings = pair_rings;
      a.nb = 1;
      a.resident = 1;
      a.na = (a.d_ff + 255) / 256;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(2 * clusters));
      cfg.blockDim = dim3(Roles<FC2P_NE>::THREADS);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess ? 0 : -1;
    }
  }
  const size_t staging = (a.dw != nullptr ? 2 : 1) * (size_t)FC2_STAGING_BYTES;
  if (!plan(a.d_ff, a.d / BN, (size_t)2 * a.d * 4, FC2_NSLOT, staging, &a.rings, &a.na, &a.nb, &a.resident,
            &smem))
    return -1;
  void (*kern)(const Fc2Args) = a.dw != nullptr      ? fc2_scatter_kernel<2>
                                 : a.dbg_y != nullptr ? fc2_scatter_kernel<1>
                                                      : fc2_scatter_kernel<0>;
  if (set_smem((const void*)kern, smem) != 0) return -1;
  const int grid = fc_grid(m_cap);
  if (grid <= 0) return -1;
  kern<<<grid, Roles<FC2_NE>::THREADS, smem, stream>>>(a);
  return 0;
}

}  // namespace moe
