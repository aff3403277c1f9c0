// Grouped block-scaled NVFP4 GEMMs of the MoE expert: U_e = MMA_NVFP4(X_e,
// W_e^T) on the 5th-generation tensor cores, then the FP32 epilogue that
// multiplies by g_x * g_w and casts to BF16 (rainbus summary, core method;
// AI summary methodology: outer factors applied in FP32 after the native
// block-scaled multiply, no decoded BF16 operand).
//
// Design (one persistent CTA per SM, 10 warps):
//   warp 8   TMA producer: A and B tiles (128 rows x 128 bytes = 256 FP4 of
//            K, 128-byte swizzle) by cp.async.bulk.tensor, their block-scale
//            tiles (4 x 512 bytes) by cp.async.bulk, into a 5-stage ring.
//   warp 9   MMA issuer: copies block scales to tensor memory (tcgen05.cp
//            32x128b.warpx4) and issues tcgen05.mma kind::mxf4nvf4
//            block_scale.scale_vec::4X (M=128, N=128, K=64, UE4M3 scale per
//            16 elements) into one of three 128-column FP32 accumulators.
//   warps 0-7 epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//            32*(w%4).. and half (w/4) of the columns).
// Group boundaries are the device-side offsets (multiples of 128 rows), so
// every 128-row tile belongs to one expert; empty experts own no tile.
//
//   FC1: a work unit is one 128-row tile of the routed activations; it runs
//        over d_ff/128 chunks, each a gate tile (W1 rows c*128..) and an up
//        tile (rows d_ff + c*128..).  The epilogue forms u = BF16(y),
//        h = BF16(silu(gate) * up), stages h in a per-CTA scratch and keeps
//        each row's running amax; after the last chunk it requantises the
//        row (g_h = amax/2688, E4M3 block scales, E2M1 codes) into the FC2
//        operand buffers.
//   FC2: a work unit is one 128 x 128 output tile; the epilogue forms
//        y2 = acc * (g_h * g_w2), z = BF16(w_{t,e} * y2) and writes it to
//        slot (t, j) of the token.
//
// Every wait is bounded (a few seconds of wall clock); on expiry the kernel
// raises MOE_STATUS_TIMEOUT, drains its own copies and MMAs, frees tensor
// memory and returns.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BN = 128, BK_BYTES = 128;
constexpr int NST = 5;
constexpr int A_BYTES = BM * BK_BYTES;
constexpr int B_BYTES = BN * BK_BYTES;
constexpr int SF_STAGE = 4 * 512;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + 2 * SF_STAGE;  // 36 KB, a multiple of 1024
constexpr int NSLOT = 3;
constexpr int TMEM_COLS = 512;
constexpr int SF_TMEM_COL = NSLOT * BN;  // two 32-column buffers: [SFA 16 | SFB 16]
constexpr int NEPI_WARPS = 8;
constexpr int PRODUCER_WARP = 8, MMA_WARP = 9;
constexpr int NTHREADS = 320;
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;

// Instruction descriptor: E2M1 x E2M1, UE4M3 scales, both operands K-major,
// N = 128 (bits 17-22 hold N/8), M = 128 (bits 24-28 hold M/16).
constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct Tail {
  uint64_t full[NST];
  uint64_t empty[NST];
  uint64_t tfull[NSLOT];
  uint64_t tempty[NSLOT];
  uint64_t sffree[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
  float rowmax[2][BM];
  int offsets[1025];
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)NST * STAGE_BYTES + sizeof(Tail);

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
      *abort_flag = 1;
      set_status(status, MOE_STATUS_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(IDESC), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Expert owning 128-row tile mt: the last e with offsets[e] <= mt*128.
__device__ __forceinline__ int expert_of(const int* off, int E, int mt) {
  const int row0 = mt * BM;
  int lo = 0, hi = E;  // first e' in [0, E] with off[e'] > row0, minus one
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= row0) lo = mid + 1; else hi = mid;
  }
  return lo - 1;
}

struct Mainloop {
  const CUtensorMap* tmap_a;
  const CUtensorMap* tmap_b;
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  int kgroups;  // K / 64
  int nk;       // k-steps of 256 elements
};

// Sequence of accumulator tiles of this CTA.  FC1: per 128-row unit, chunks
// c = 0..nch-1, each a gate item then an up item.  FC2: one item per
// (m-tile, n-tile) unit.
struct Schedule {
  bool fc1;
  int E, num_mt, nch, ntn, N, d_ff;
  __device__ int units() const { return fc1 ? num_mt : num_mt * ntn; }
  __device__ int items(int) const { return fc1 ? 2 * nch : 1; }
  __device__ int mtile(int u) const { return fc1 ? u : u / ntn; }
  __device__ int brow(int u, int e, int q) const {
    if (fc1) return e * N + (q & 1) * d_ff + (q >> 1) * BN;
    return e * N + (u % ntn) * BN;
  }
};

__device__ void producer_loop(const Mainloop& ml, const Schedule& sc, const int* off, uint8_t* stages, Tail* tl,
                              volatile int* abort_flag, int* status) {
  const uint32_t base = smem_u32(stages);
  uint32_t kc = 0;
  uint32_t issued_use[NST];
  for (int s = 0; s < NST; ++s) issued_use[s] = 0xFFFFFFFFu;
  bool aborted = false;
  for (int u = blockIdx.x; u < sc.units() && !aborted; u += gridDim.x) {
    const int mt = sc.mtile(u);
    const int e = expert_of(off, sc.E, mt);
    const int nq = sc.items(u);
    for (int q = 0; q < nq && !aborted; ++q) {
      const int br = sc.brow(u, e, q);
      for (int ks = 0; ks < ml.nk; ++ks, ++kc) {
        const uint32_t s = kc % NST, use = kc / NST;
        if (!wait_bounded(smem_u32(&tl->empty[s]), (use & 1u) ^ 1u, abort_flag, status)) { aborted = true; break; }
        const int nsf = min(4, ml.kgroups - 4 * ks);
        const uint32_t st = base + s * STAGE_BYTES;
        const uint32_t fb = smem_u32(&tl->full[s]);
        mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES + 2 * nsf * 512);
        tma_load_2d(st, ml.tmap_a, ks * BK_BYTES, mt * BM, fb);
        tma_load_2d(st + A_BYTES, ml.tmap_b, ks * BK_BYTES, br, fb);
        bulk_load(st + A_BYTES + B_BYTES, ml.a_sf + ((int64_t)mt * ml.kgroups + 4 * ks) * 512, nsf * 512, fb);
        bulk_load(st + A_BYTES + B_BYTES + SF_STAGE, ml.b_sf + ((int64_t)(br / BM) * ml.kgroups + 4 * ks) * 512,
                  nsf * 512, fb);
        issued_use[s] = use;
      }
    }
  }
  if (aborted) {
    // let the copies already issued land before the CTA can exit
    for (int s = 0; s < NST; ++s)
      if (issued_use[s] != 0xFFFFFFFFu) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&tl->full[s]), issued_use[s] & 1u) && global_timer_ns() - t0 < WAIT_LIMIT_NS) {
        }
      }
  }
}

__device__ void mma_loop(const Mainloop& ml, const Schedule& sc, const int* off, uint8_t* stages, Tail* tl,
                         uint32_t tmem, volatile int* abort_flag, int* status) {
  const uint32_t base = smem_u32(stages);
  uint32_t kc = 0, it = 0;
  bool aborted = false;
  for (int u = blockIdx.x; u < sc.units() && !aborted; u += gridDim.x) {
    const int nq = sc.items(u);
    for (int q = 0; q < nq && !aborted; ++q, ++it) {
      const uint32_t slot = it % NSLOT, suse = it / NSLOT;
      if (!wait_bounded(smem_u32(&tl->tempty[slot]), (suse & 1u) ^ 1u, abort_flag, status)) { aborted = true; break; }
      tc_fence_after();
      const uint32_t dacc = tmem + slot * BN;
      for (int ks = 0; ks < ml.nk; ++ks, ++kc) {
        const uint32_t s = kc % NST, use = kc / NST;
        if (!wait_bounded(smem_u32(&tl->full[s]), use & 1u, abort_flag, status)) { aborted = true; break; }
        const uint32_t sfb = kc & 1u;
        if (kc >= 2 && !wait_bounded(smem_u32(&tl->sffree[sfb]), ((kc >> 1) - 1u) & 1u, abort_flag, status)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const int nmma = min(4, ml.kgroups - 4 * ks);
        const uint32_t st = base + s * STAGE_BYTES;
        const uint32_t sf_a = tmem + SF_TMEM_COL + sfb * 32;
        const uint32_t sf_b = sf_a + 16;
        for (int i = 0; i < nmma; ++i) {
          tc_cp_sf(sf_a + 4 * i, sdesc_sf(st + A_BYTES + B_BYTES + 512 * i));
          tc_cp_sf(sf_b + 4 * i, sdesc_sf(st + A_BYTES + B_BYTES + SF_STAGE + 512 * i));
        }
        const uint64_t adesc = sdesc_k_sw128(st);
        const uint64_t bdesc = sdesc_k_sw128(st + A_BYTES);
        for (int i = 0; i < nmma; ++i)
          tc_mma(dacc, adesc + 2 * i, bdesc + 2 * i, sf_a + 4 * i, sf_b + 4 * i, (ks | i) != 0 ? 1u : 0u);
        tc_commit(smem_u32(&tl->empty[s]));
        tc_commit(smem_u32(&tl->sffree[sfb]));
      }
      if (!aborted) tc_commit(smem_u32(&tl->tfull[slot]));
    }
  }
  // all MMAs and scale copies of this CTA have completed once `done` fires
  tc_commit(smem_u32(&tl->done));
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(smem_u32(&tl->done), 0u) && global_timer_ns() - t0 < WAIT_LIMIT_NS) {
  }
}

// Quantise 16 BF16 values held by one thread (one block): packed codes in
// 8 bytes (even element in the low nibble) and the block-scale byte.
__device__ __forceinline__ uint2 quant_block16(const uint32_t (&w)[8], float g, float den, uint32_t* sb_out) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  uint32_t sb = 0;
  uint2 p = make_uint2(0u, 0u);
  if (g != 0.0f) {
    sb = e4m3_encode(__fdiv_rn(a, den));
    const float S = __fmul_rn(g, e4m3_decode(sb));
    if (S != 0.0f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t c0 = e2m1_encode(__fdiv_rn(bf16_lo(w[i]), S));
        const uint32_t c1 = e2m1_encode(__fdiv_rn(bf16_hi(w[i]), S));
        const uint32_t byte = c0 | (c1 << 4);
        if (i < 4) p.x |= byte << (8 * i); else p.y |= byte << (8 * (i - 4));
      }
    }
  }
  *sb_out = sb;
  return p;
}

// Common prologue: barriers, tensor memory, offsets.  Returns the base of
// the 1024-aligned stage ring.
__device__ __forceinline__ uint8_t* setup(uint8_t* smem_raw, Tail*& tl, const int32_t* offsets, int E) {
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  tl = reinterpret_cast<Tail*>(stages + (size_t)NST * STAGE_BYTES);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&tl->full[s]), 1);
      mbar_init(smem_u32(&tl->empty[s]), 1);
    }
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(smem_u32(&tl->tfull[s]), 1);
      mbar_init(smem_u32(&tl->tempty[s]), NEPI_WARPS);
    }
    mbar_init(smem_u32(&tl->sffree[0]), 1);
    mbar_init(smem_u32(&tl->sffree[1]), 1);
    mbar_init(smem_u32(&tl->done), 1);
    tl->abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i <= E; i += blockDim.x) tl->offsets[i] = offsets[i];
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tl->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return stages;
}

__device__ __forceinline__ void teardown(Tail* tl) {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == MMA_WARP) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tl->tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// FC1 + SwiGLU + requantisation
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NTHREADS, 1) fc1_swiglu_kernel(const __grid_constant__ Fc1Args args) {
  extern __shared__ uint8_t smem_raw[];
  Tail* tl;
  uint8_t* stages = setup(smem_raw, tl, args.offsets, args.E);
  volatile int* abort_flag = &tl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* off = tl->offsets;
  const int d_ff = args.d_ff;
  Schedule sc;
  sc.fc1 = true;
  sc.E = args.E;
  sc.num_mt = off[args.E] / BM;
  sc.nch = d_ff / BN;
  sc.ntn = 1;
  sc.N = 2 * d_ff;
  sc.d_ff = d_ff;
  Mainloop ml{&args.tmap_a, &args.tmap_b, args.a_sf, args.w_sf, args.d / 64, (args.d + 255) / 256};

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      prefetch_tmap(&args.tmap_a);
      prefetch_tmap(&args.tmap_b);
      producer_loop(ml, sc, off, stages, tl, abort_flag, args.status);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (lane == 0) mma_loop(ml, sc, off, stages, tl, tl->tmem_base, abort_flag, args.status);
    __syncwarp();
  } else {
    // ---------------- epilogue warps ----------------
    const int q = warp & 3, hh = warp >> 2;
    const int rl = q * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t tmem = tl->tmem_base + ((uint32_t)(q * 32) << 16);
    uint4* scratch = reinterpret_cast<uint4*>(args.scratch) + (size_t)blockIdx.x * (size_t)(d_ff / 8) * BM;
    const int kgh = d_ff / 64;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < sc.num_mt; u += gridDim.x) {
      const int e = expert_of(off, args.E, u);
      const int64_t row = (int64_t)u * BM + rl;
      const float ga = args.a_g[row];
      const float* wg = args.w_g + (int64_t)e * 2 * d_ff;
      float rowmax = 0.0f;
      for (int c = 0; c < sc.nch; ++c, it += 2) {
        const uint32_t sg = it % NSLOT, su = (it + 1) % NSLOT;
        bool ok = !*abort_flag;
        if (ok) ok = wait_bounded(smem_u32(&tl->tfull[sg]), (it / NSLOT) & 1u, abort_flag, args.status);
        if (ok) ok = wait_bounded(smem_u32(&tl->tfull[su]), ((it + 1) / NSLOT) & 1u, abort_flag, args.status);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) {
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            const int col = hh * 64 + cc * 32;  // column within the 128-wide chunk
            uint32_t G[32], U[32];
            tmem_ld32(tmem + sg * BN + col, G);
            tmem_ld32(tmem + su * BN + col, U);
            const int n0 = c * BN + col;  // h column
            uint32_t hp[16];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float sgt = __fmul_rn(ga, __ldg(wg + n0 + i));
              const float sup = __fmul_rn(ga, __ldg(wg + d_ff + n0 + i));
              const float yg = __fmul_rn(__uint_as_float(G[i]), sgt);
              const float yu = __fmul_rn(__uint_as_float(U[i]), sup);
              const float ug = bf16_bits_to_f32(f32_to_bf16_bits(yg));
              const float uu = bf16_bits_to_f32(f32_to_bf16_bits(yu));
              const float sl = __fdividef(ug, 1.0f + __expf(-ug));
              const uint32_t hb = f32_to_bf16_bits(__fmul_rn(sl, uu));
              rowmax = fmaxf(rowmax, fabsf(bf16_bits_to_f32(hb)));
              if (i & 1) hp[i >> 1] |= hb << 16; else hp[i >> 1] = hb;
              if (args.dbg_u) {
                args.dbg_u[row * 2 * d_ff + n0 + i] = yg;
                args.dbg_u[row * 2 * d_ff + d_ff + n0 + i] = yu;
              }
            }
            if (args.dbg_h) {
              uint4* dh = reinterpret_cast<uint4*>(args.dbg_h + row * d_ff + n0);
#pragma unroll
              for (int v = 0; v < 4; ++v) dh[v] = make_uint4(hp[4 * v], hp[4 * v + 1], hp[4 * v + 2], hp[4 * v + 3]);
            }
            const int grp = ((c * 2 + hh) * 2 + cc) * 4;  // 16-byte column group index
#pragma unroll
            for (int v = 0; v < 4; ++v)
              scratch[(size_t)(grp + v) * BM + rl] = make_uint4(hp[4 * v], hp[4 * v + 1], hp[4 * v + 2], hp[4 * v + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&tl->tempty[sg]));
          mbar_arrive(smem_u32(&tl->tempty[su]));
        }
      }
      // ---- requantise the tile's rows: amax over the full d_ff row ----
      tl->rowmax[hh][rl] = rowmax;
      epi_barrier();
      const float a = fmaxf(tl->rowmax[0][rl], tl->rowmax[1][rl]);
      if (!*abort_flag) {
        if (!is_finite_f32(a)) set_status(args.status, MOE_STATUS_NONFINITE_X);
        const float g = __fdiv_rn(a, 2688.0f);
        const float den = __fmul_rn(6.0f, g);
        for (int c = 0; c < sc.nch; ++c) {
          uint32_t sfword = 0;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int grp = ((c * 2 + hh) * 2 + cc) * 4;
            uint32_t w[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 x = scratch[(size_t)(grp + v) * BM + rl];
              w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
            }
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              uint32_t wb[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) wb[i] = w[8 * b + i];
              uint32_t sb;
              const uint2 p = quant_block16(wb, g, den, &sb);
              const int n = c * BN + hh * 64 + cc * 32 + b * 16;  // first column of the block
              *reinterpret_cast<uint2*>(args.h_codes + row * (d_ff / 2) + n / 2) = p;
              sfword |= sb << (8 * (cc * 2 + b));
            }
          }
          const int c4 = 2 * c + hh;  // block-scale column group of columns c*128 + hh*64 .. +64
          *reinterpret_cast<uint32_t*>(args.h_sf + ((row >> 7) * kgh + c4) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4) =
              sfword;
        }
        if (hh == 0) args.h_g[row] = g;
      }
      epi_barrier();
    }
  }
  teardown(tl);
}

// ---------------------------------------------------------------------------
// FC2 + router-weighted scatter
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NTHREADS, 1) fc2_scatter_kernel(const __grid_constant__ Fc2Args args) {
  extern __shared__ uint8_t smem_raw[];
  Tail* tl;
  uint8_t* stages = setup(smem_raw, tl, args.offsets, args.E);
  volatile int* abort_flag = &tl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* off = tl->offsets;
  const int d = args.d, k = args.k;
  Schedule sc;
  sc.fc1 = false;
  sc.E = args.E;
  sc.num_mt = off[args.E] / BM;
  sc.nch = 1;
  sc.ntn = d / BN;
  sc.N = d;
  sc.d_ff = args.d_ff;
  Mainloop ml{&args.tmap_a, &args.tmap_b, args.a_sf, args.w_sf, args.d_ff / 64, (args.d_ff + 255) / 256};

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      prefetch_tmap(&args.tmap_a);
      prefetch_tmap(&args.tmap_b);
      producer_loop(ml, sc, off, stages, tl, abort_flag, args.status);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (lane == 0) mma_loop(ml, sc, off, stages, tl, tl->tmem_base, abort_flag, args.status);
    __syncwarp();
  } else {
    const int q = warp & 3, hh = warp >> 2;
    const int rl = q * 32 + lane;
    const uint32_t tmem = tl->tmem_base + ((uint32_t)(q * 32) << 16);
    uint32_t it = 0;
    for (int u = blockIdx.x; u < sc.units(); u += gridDim.x, ++it) {
      const int mt = u / sc.ntn, nt = u % sc.ntn;
      const int e = expert_of(off, args.E, mt);
      const int64_t row = (int64_t)mt * BM + rl;
      const int t = args.row_to_token[row];
      int j = 0;
      float w = 0.0f;
      if (t >= 0) {
        for (int jj = 0; jj < k; ++jj)
          if (args.token_slot_row[(int64_t)t * k + jj] == (int)row) j = jj;
        w = args.topk_w[(int64_t)t * k + j];
      }
      const float gh = args.a_g[row];
      const float* wg = args.w_g + (int64_t)e * d;
      const uint32_t slot = it % NSLOT;
      bool ok = !*abort_flag;
      if (ok) ok = wait_bounded(smem_u32(&tl->tfull[slot]), (it / NSLOT) & 1u, abort_flag, args.status);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          const int col = hh * 64 + cc * 32;
          uint32_t R[32];
          tmem_ld32(tmem + slot * BN + col, R);
          const int n0 = nt * BN + col;
          if (t >= 0) {
            uint32_t zp[16];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float sc2 = __fmul_rn(gh, __ldg(wg + n0 + i));
              const float y2 = __fmul_rn(__uint_as_float(R[i]), sc2);
              const uint32_t zb = f32_to_bf16_bits(__fmul_rn(w, y2));
              if (i & 1) zp[i >> 1] |= zb << 16; else zp[i >> 1] = zb;
              if (args.dbg_y) args.dbg_y[row * d + n0 + i] = y2;
            }
            uint4* dst = reinterpret_cast<uint4*>(args.slots + ((int64_t)t * k + j) * d + n0);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(zp[4 * v], zp[4 * v + 1], zp[4 * v + 2], zp[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tl->tempty[slot]));
    }
  }
  teardown(tl);
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

static bool g_attr_set[2][64];

template <typename K>
static int prepare(K kernel, int which) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev < 64 && !g_attr_set[which][dev]) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES) != cudaSuccess)
      return -1;
    g_attr_set[which][dev] = true;
  }
  return 0;
}

int launch_fc1(const Fc1Args& a, cudaStream_t stream) {
  if (prepare(fc1_swiglu_kernel, 0) != 0) return -1;
  const int grid = gemm_num_ctas();
  if (grid <= 0) return -1;
  fc1_swiglu_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(a);
  return 0;
}

int launch_fc2(const Fc2Args& a, cudaStream_t stream) {
  if (prepare(fc2_scatter_kernel, 1) != 0) return -1;
  const int grid = gemm_num_ctas();
  if (grid <= 0) return -1;
  fc2_scatter_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(a);
  return 0;
}

}  // namespace moe
