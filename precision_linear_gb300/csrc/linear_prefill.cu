// tcgen05 NVFP4 + LoRA linear for large M (log-prob recompute, prefill), sm_103a.
//
// Computes the forward map of "QeRL: When Quantized Weights Help Reinforcement
// Learning, and Where the Evidence Stops", section 2.1 (y = W_hat h + lambda B (A h)),
// on the section 3.1 NVFP4 backbone (w_hat = s_g s_b q), with h the section 5.1
// RMSNorm-AQN of x.  Three kernels, chained by programmatic dependent launch:
//
//   k_act (linear_tc.cu)  per token row: hq = f16(h / rowscale) with rowscale a power of
//                         two (max |hq| in [2^13, 2^14)); A -> f16; split counters := 0.
//   k_lora_down           T[m, :] = (lambda / s_g) sum_k A[:, k] hq[m, k]: each CTA one K
//                         split of 128 tokens (tcgen05.mma, 128 x r, K = 16 steps, from
//                         TMA-staged hq and f16 A tiles, FP32 accumulator in tensor memory)
//                         into its partial; the last split of a token tile to finish adds
//                         the partials up in split order (deterministic) and writes
//                         Tq = bf16(T) [M][64] (zero beyond r).  The LoRA up-projection is
//                         then 64 more K columns of the contraction: since t = A h = rowscale
//                         A hq, s_g rowscale[m] sum_j B[o, j] Tq[m, j] = lambda sum_j B[o, j]
//                         t[m, j], with B (bf16, as stored) the A operand of that step.
//   k_gemm_nvfp4          the dense contraction on CTA pairs (clusters of two, the
//                         tcgen05 cta_group::2 form), persistent over 256 (weight rows) x
//                         TN (tokens; 192 or 160 by the rounds they need, 128 when 192 leaves
//                         pairs idle) tiles,
//                         o-tiles fastest so that concurrent pairs share their hq tiles in
//                         L2.  Each CTA of a pair owns 128 of the weight rows and half of
//                         the tokens:
//     warp 0      TMA: per 64-wide K step this CTA's half of the hq tile (TN/2 x 64 f16,
//                 128-byte swizzle) and the packed codes of its rows (128 x 32 B); every
//                 4th step the E4M3 scales of the next 256 K (128 x 16 B); one more step
//                 per tile with the Tq rows of its tokens; per tile the row scales of
//                 all TN tokens;
//     warps 2-9   dequantise each K step into a 32-column tensor-memory slot (E2M1 -> f16
//                 conversion times the f16 block scale: exact), one weight row and half
//                 of the step per thread; the LoRA step gets the B rows (bf16) instead;
//                 the odd CTA's warps signal the even CTA's barrier;
//     warp 1      in the even CTA: tcgen05.mma.cta_group::2 kind::f16, M = 256, N = TN,
//                 K = 16: D (each CTA's 128 rows in its own tensor memory, two buffers of
//                 TN columns) += W_hat / s_g x hq^T (f16) + B x Tq^T (bf16), the A rows from both
//                 CTAs' tensor memory and the B rows from both CTAs' shared memory, so
//                 each SM stages and reads only half of the token tile;
//     warps 10-13 epilogue of the previous tile while the next one accumulates:
//                 y[m, o] = s_g rowscale[m] D[o, m], stored as BF16 or FP32.
//
// Every mbarrier wait is bounded (200 ms); a wait that gives up sets the status word,
// the CTA stops issuing work, drains its copies, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace pl {

__device__ uint32_t g_pf_status = 0;

// Per-CTA wait accounting for development builds (-DPL_TIMELINE); compiled out otherwise.
#ifdef PL_TIMELINE
__device__ unsigned long long g_pf_wait[1024][12];
#define PF_T0() const uint64_t pf_t0_ = globaltimer_ns()
#define PF_ACC(slot) do { if (blockIdx.x < 1024) atomicAdd(&g_pf_wait[blockIdx.x][slot], globaltimer_ns() - pf_t0_); } while (0)
#else
#define PF_T0() do { } while (0)
#define PF_ACC(slot) do { } while (0)
#endif

namespace {

constexpr int kTO = 128;  // weight rows per tile
constexpr int kTN = 192;  // tokens per pair tile, at most (the GEMM is instantiated for 128 and 192)
constexpr int kKS = 64;   // K per pipeline step (one 128-byte row of f16)
constexpr int kMaxStages = 10;
constexpr int kMaxASlots = 8;
// Tensor-memory weight slots (32 columns: one 64-wide K step of 128 rows) beside the two
// accumulator buffers of TN columns: 4 at TN = 192, 6 at 160, 8 at 128.
__host__ __device__ constexpr int a_slots_of(int tn) { return (512 - 2 * tn) / 32 < kMaxASlots ? (512 - 2 * tn) / 32 : kMaxASlots; }
constexpr uint32_t kCodeBytes = kTO * kKS / 2;  // 4 KB
// one pipeline stage of a CTA: its half of the tile's tokens (tn / 2 rows of hq) and its codes
__host__ __device__ constexpr uint32_t stage_bytes_of(int tn) { return static_cast<uint32_t>(tn / 2) * kKS * 2 + kCodeBytes; }
constexpr uint32_t kScaleBytes = kTO * 16;      // scales of 256 K
// Scale slots: the group of step 4G is loaded once the stage of step 4G - stages is free, so
// the dequant warps may still read groups down to (4G - stages + 1) / 4: ceil((stages - 1) / 4)
// of them besides G.
constexpr int kScaleSlots = 4;
static_assert(kMaxStages <= 4 * (kScaleSlots - 1) + 1, "scale slots too few for the stage count");
constexpr int kDeqWarps = 8;  // two per tensor-memory lane quarter: each dequantises half of a K step
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kDeqWarps + kEpiWarps) * 32;  // 448
constexpr uint32_t kTmemCols = 512;

constexpr int kMaxR = 32;
constexpr int kLoraK = 64;  // K columns the LoRA step adds (r <= 32 of them nonzero)

// One projection of a launch (a group shares the input): its pairs of weight tiles are
// [ot0, ot0 + n_ot) of the launch's; its tiles (n_ot pairs x the token tiles) are
// [t0, t0 + n_ot x token tiles) of the launch's, member after member, so that one member's
// weights stay in L2 across its token tiles.
struct GMember {
  int64_t d_o;
  int r, ot0, n_ot, t0;
  const float* s_g;
  const __nv_bfloat16* B;  // [d_o][r], as stored: the A operand of the LoRA step
  void* y;                 // [M][d_o]
};

struct GParams {
  int64_t M, d_i;
  int n_ot, n_tiles, n_ks, stages, n_g;
  const float* rowscale;  // [M_pad]
  int y_f32;
  uint32_t off_scales, off_t, t_slot_bytes, off_ctrl;
  GMember g[kMaxPrefillGroup];
};

struct GMaps {
  CUtensorMap hq;
  CUtensorMap codes[kMaxPrefillGroup], scales[kMaxPrefillGroup], tq[kMaxPrefillGroup];
};

// Tile -> (member, token tile, the member's pair of weight tiles): members one after
// another, within a member the weight pairs fastest (concurrent pairs share their token tile).
struct TileAt {
  int gi, mt, otl;
};
__device__ __forceinline__ TileAt tile_at(const GParams& p, int tile) {
  int gi = 0;
#pragma unroll
  for (int q = 1; q < kMaxPrefillGroup; ++q)
    if (q < p.n_g && tile >= p.g[q].t0) gi = q;
  const int local = tile - p.g[gi].t0;
  return TileAt{gi, local / p.g[gi].n_ot, local % p.g[gi].n_ot};
}

// One commit per K step (main or LoRA) to sdone[step mod kSDone]: it releases that step's stage
// (both CTAs' dequant warps read its codes before the MMAs could start, the MMAs read its
// token rows) and its tensor-memory slot, so one tensor-core instruction serves both.
constexpr int kSDone = 16;
static_assert(kMaxStages <= kSDone && kMaxASlots <= kSDone, "a waiter is never two phases behind");
struct GCtrl {
  uint64_t full[kMaxStages], sdone[kSDone];
  uint64_t afull[kMaxASlots];
  uint64_t dfull[2], dempty[2];
  uint64_t tfull[2], tempty[2];
  uint64_t mma_done;  // every MMA this CTA issued has completed
  uint32_t tmem_base;
  int abort_flag;
  float s_g[kMaxPrefillGroup];
};

__device__ __noinline__ bool wait_p_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return wait_or_abort_status(bar, parity, abort_flag, &g_pf_status);
}
// Bounded wait: the common case (already complete) inline, the polling loop out of line.
PL_DEVINL bool wait_p(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_try_wait(bar, parity) || wait_p_slow(bar, parity, abort_flag);
}
// Position and phase of a ring of n barriers (no division on the issue paths).
struct Ring {
  int i = 0;
  uint32_t ph = 0;
  PL_DEVINL void next(int n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};
PL_DEVINL void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// ---- CTA-pair (cta_group::2) forms: the even CTA of a cluster of two issues M = 256 MMAs
// whose A rows 0-127 / 128-255 come from the even / odd CTA's tensor memory, whose B rows
// [0, N/2) / [N/2, N) come from the even / odd CTA's shared memory (same offsets), and
// whose D rows 0-127 / 128-255 land in the even / odd CTA's tensor memory.
PL_DEVINL void tmem_alloc2(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst), "r"(ncols) : "memory");
}
PL_DEVINL void tmem_relinquish2() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory"); }
PL_DEVINL void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
PL_DEVINL void mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accum) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
               :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accum) : "memory");
}
// Arrival on the barrier at this offset in both CTAs of the pair once every MMA issued so far
// has completed.
PL_DEVINL void tc_commit2(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               :: "r"(bar), "h"(static_cast<uint16_t>(3)) : "memory");
}
PL_DEVINL uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Arrival on the barrier at this offset in the even CTA (default semantics: the data it
// orders is tensor memory, ordered by the tcgen05 fences around the arrival and the wait;
// a cluster-scope release would cost about a microsecond per arrival).
PL_DEVINL void mbar_arrive_leader(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" :: "r"(mapa_shared(bar, 0)) : "memory");
}
// ------------------------------------------------------------------ main contraction
// A cluster of two CTAs (a pair) per 256 (weight rows) x TN (tokens) tile: each CTA
// dequantises its own 128 weight rows into its tensor memory and stages its own half of the
// tile's tokens in shared memory; the even CTA issues the M = 256 MMAs for both.
template <int TN>
__global__ void __launch_bounds__(kThreads, 1) k_gemm_nvfp4(const __grid_constant__ GMaps maps, const GParams p) {
  constexpr int kTH = TN / 2;  // token rows of the B operand this CTA stages
  constexpr int kASlots = a_slots_of(TN);
  constexpr uint32_t kColD0 = 32u * kASlots;  // D buffer b at columns [kColD0 + TN b, kColD0 + TN (b + 1))
  constexpr uint32_t kHBytesT = kTH * kKS * 2, kStageBytes = stage_bytes_of(TN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GCtrl& C = *reinterpret_cast<GCtrl*>(smem + p.off_ctrl);
  volatile int* abort_flag = &C.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const int nst = p.stages, n_ks = p.n_ks;
  const int rank = static_cast<int>(cta_rank());  // 0: issues the MMAs of the pair
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
#ifdef PL_TIMELINE
    if (blockIdx.x < 1024) g_pf_wait[blockIdx.x][10] = globaltimer_ns();
#endif
    pdl_launch_dependents();
    for (int s = 0; s < nst; ++s) mbar_init(smem_u32(&C.full[s]), 1);
    for (int s = 0; s < kSDone; ++s) mbar_init(smem_u32(&C.sdone[s]), 1);  // the pair's MMA commit
    for (int a = 0; a < kASlots; ++a)
      mbar_init(smem_u32(&C.afull[a]), 2 * kDeqWarps);  // both CTAs' dequant warps (waited on in the even one)
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&C.dfull[b]), 1);
      mbar_init(smem_u32(&C.dempty[b]), 2 * kEpiWarps);  // both CTAs' epilogue warps (waited on in the even one)
      mbar_init(smem_u32(&C.tfull[b]), 1);
      mbar_init(smem_u32(&C.tempty[b]), kEpiWarps);
    }
    mbar_init(smem_u32(&C.mma_done), 1);
    C.abort_flag = 0;
    for (int q = 0; q < p.n_g; ++q) {
      C.s_g[q] = *p.g[q].s_g;  // weight inputs: not written by the preceding kernel
      tma_prefetch_desc(&maps.codes[q]);
      tma_prefetch_desc(&maps.scales[q]);
    }
    fence_mbar_init();
    tma_prefetch_desc(&maps.hq);
  }
  if (warp == 1) {
    tmem_alloc2(smem_u32(&C.tmem_base), kTmemCols);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and tensor memory exist before either touches the other's
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      pdl_wait();  // hq, row scales and Tq come from the preceding kernels
      const uint32_t tbytes = static_cast<uint32_t>(TN) * 4;
      bool ok = true;
      int64_t gs = 0;
      Ring rs;            // stage ring
      uint32_t grp = ~0u;  // scale groups loaded so far - 1
      int it = 0, t_issued = 0;
      for (int tile = pair; tile < p.n_tiles && ok; tile += npairs, ++it) {
        const TileAt at = tile_at(p, tile);
        const int gi = at.gi, mt = at.mt;
        const int n_steps = n_ks + (p.g[gi].r > 0 ? 1 : 0);  // K steps of this tile, the LoRA step last
        const int32_t m0 = mt * TN, o0 = at.otl * 2 * kTO + rank * kTO, mh = m0 + rank * kTH;
        {  // the row scales of this tile's tokens (all TN: this CTA's accumulator spans them)
          const int tb = it & 1;
          {
            PF_T0();
            if (it >= 2) ok = wait_p(smem_u32(&C.tempty[tb]), ((it >> 1) - 1) & 1, abort_flag);
            PF_ACC(1);
          }
          if (!ok) break;
          const uint32_t tb_bar = smem_u32(&C.tfull[tb]);
          const uint32_t dst = sbase + p.off_t + tb * p.t_slot_bytes;
          mbar_arrive_expect_tx(tb_bar, tbytes);
          bulk_g2s(dst, p.rowscale + m0, TN * 4, tb_bar);
          ++t_issued;
        }
        for (int s = 0; s < n_steps && ok; ++s, ++gs, rs.next(nst)) {
          const int st = rs.i;
          {
            PF_T0();
            const int64_t gd = gs - nst;  // the step that last used stage st
            if (gs >= nst) ok = wait_p(smem_u32(&C.sdone[gd % kSDone]), static_cast<uint32_t>(gd / kSDone) & 1u, abort_flag);
            PF_ACC(0);
          }
          if (!ok) break;
          const uint32_t fb = smem_u32(&C.full[st]);
          if (s == n_ks) {  // the LoRA step: Tq rows of this CTA's half of the tokens
            mbar_arrive_expect_tx(fb, kHBytesT);
            tma_load_2d(sbase + st * kStageBytes, &maps.tq[gi], 0, mh, fb);
            continue;
          }
          const bool scl = (s & 3) == 0;
          mbar_arrive_expect_tx(fb, kStageBytes + (scl ? kScaleBytes : 0));
          const uint32_t stage = sbase + st * kStageBytes;
          tma_load_2d(stage, &maps.hq, s * kKS, mh, fb);
          // weights and hq both stay in L2: every weight tile is read once per token tile
          tma_load_2d(stage + kHBytesT, &maps.codes[gi], s * (kKS / 2), o0, fb);
          if (scl) {
            ++grp;
            tma_load_2d(sbase + p.off_scales + (grp % kScaleSlots) * kScaleBytes, &maps.scales[gi],
                        s * (kKS / 16), o0, fb);
          }
        }
      }
      if (*abort_flag) {  // every issued copy lands before this CTA exits
        for (int64_t d = gs - nst > 0 ? gs - nst : 0; d < gs; ++d)
          drain(smem_u32(&C.full[d % nst]), static_cast<uint32_t>(d / nst) & 1);
        for (int d = t_issued - 2 > 0 ? t_issued - 2 : 0; d < t_issued; ++d)
          drain(smem_u32(&C.tfull[d & 1]), (d >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_f16(2 * kTO, TN, 0);
      const uint32_t idesc_l = idesc_f16(2 * kTO, TN, 1);  // the LoRA step: bf16 B and T
      bool ok = true;
      Ring rs, ra;  // stage and slot rings
      const uint64_t hdesc0 = smem_desc_sw128(sbase, 1024);
      int it = 0;
      int64_t gstep = 0;  // K steps issued, main and LoRA
      for (int tile = pair; tile < p.n_tiles && ok; tile += npairs, ++it) {
        const int b = it & 1;
        const int r_t = p.g[tile_at(p, tile).gi].r;  // this tile's adapter rank
        const bool lora = r_t > 0;
        const int l_sub = (r_t + 15) / 16;  // the LoRA step's K sub-steps of 16
        {
          PF_T0();
          if (it >= 2) ok = wait_p(smem_u32(&C.dempty[b]), ((it >> 1) - 1) & 1, abort_flag);
          PF_ACC(2);
        }
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + (kColD0 + static_cast<uint32_t>(TN) * b);
        // main K steps (the first one starts the accumulator), then the LoRA step: kept out
        // of the loop, whose single issuing thread bounds the kernel
        for (int s = 0; s < n_ks && ok; ++s) {
          const int st = rs.i, a = ra.i;
          {
            // both CTAs' slot a is dequantised; each dequant warp waited for its CTA's stage
            // st first, so both halves of the token tile have landed too
            PF_T0();
            ok = wait_p(smem_u32(&C.afull[a]), ra.ph, abort_flag);
            PF_ACC(4);
          }
          if (!ok) break;
          tc_fence_after();
          const uint64_t hdesc = hdesc0 + static_cast<uint64_t>(static_cast<uint32_t>(st) * (kStageBytes >> 4));
          const uint32_t acol = tmem + 32u * a;
          mma2_ts(d, acol, hdesc, idesc, s > 0 ? 1u : 0u);
          mma2_ts(d, acol + 8u, hdesc + 2u, idesc, 1u);
          mma2_ts(d, acol + 16u, hdesc + 4u, idesc, 1u);
          mma2_ts(d, acol + 24u, hdesc + 6u, idesc, 1u);
          tc_commit2(smem_u32(&C.sdone[gstep % kSDone]));
          ++gstep;
          rs.next(nst);
          ra.next(kASlots);
        }
        if (lora && ok) {
          const int st = rs.i, a = ra.i;
          ok = wait_p(smem_u32(&C.afull[a]), ra.ph, abort_flag);
          if (ok) {
            tc_fence_after();
            const uint64_t hdesc = hdesc0 + static_cast<uint64_t>(static_cast<uint32_t>(st) * (kStageBytes >> 4));
            const uint32_t acol = tmem + 32u * a;
            for (int kk = 0; kk < l_sub; ++kk) mma2_ts(d, acol + 8u * kk, hdesc + 2u * kk, idesc_l, 1u);
            tc_commit2(smem_u32(&C.sdone[gstep % kSDone]));
            ++gstep;
            rs.next(nst);
            ra.next(kASlots);
          }
        }
        tc_commit2(smem_u32(&C.dfull[b]));
      }
      tc_commit2(smem_u32(&C.mma_done));
      drain(smem_u32(&C.mma_done), 0);  // tensor memory is freed only after the last MMA
    }
  } else if (warp < 2 + kDeqWarps) {
    // ---------------------------------------------------------------- dequant
    const int quarter = warp & 3, row = quarter * 32 + lane, g = (warp - 2) >> 2;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;

    bool ok = true;
    int64_t gs = 0;
    Ring rs, ra;         // stage and slot rings
    uint32_t grp = ~0u;  // scale groups used so far - 1
    int it = 0;
    for (int tile = pair; tile < p.n_tiles && ok; tile += npairs, ++it) {
      const TileAt at = tile_at(p, tile);
      const GMember& G = p.g[at.gi];
      const int r = G.r;
      const bool lora = r > 0;
      const int n_steps = n_ks + (lora ? 1 : 0);
      const int64_t o = static_cast<int64_t>(at.otl) * 2 * kTO + rank * kTO + row;
      // this thread's half of the LoRA step's 64 K columns of its row: B[o][32 g .. 32 g + 32),
      // bf16 as stored, zero beyond r (r <= 32: the g = 1 half is all zero)
      uint4 bq[4] = {};
      if (lora && g == 0 && o < G.d_o) {
        if ((r & 7) == 0) {
          const uint4* src = reinterpret_cast<const uint4*>(G.B + o * r);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (8 * q < r) bq[q] = src[q];
        } else {
          const uint16_t* src = reinterpret_cast<const uint16_t*>(G.B + o * r);
          uint32_t w[16];
#pragma unroll
          for (int j2 = 0; j2 < 16; ++j2) {
            const uint32_t lo = 2 * j2 < r ? src[2 * j2] : 0u, hi = 2 * j2 + 1 < r ? src[2 * j2 + 1] : 0u;
            w[j2] = lo | (hi << 16);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) bq[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      for (int s = 0; s < n_steps && ok; ++s, ++gs, rs.next(nst), ra.next(kASlots)) {
        const int st = rs.i, a = ra.i;
        {
          PF_T0();
          ok = wait_p(smem_u32(&C.full[st]), rs.ph, abort_flag);
          if (lane == 0 && warp == 2) PF_ACC(5);
        }
        {
          PF_T0();
          const int64_t gd = gs - kASlots;  // the step that last used slot a
          ok = ok && (gs < kASlots || wait_p(smem_u32(&C.sdone[gd % kSDone]), static_cast<uint32_t>(gd / kSDone) & 1u, abort_flag));
          if (lane == 0 && warp == 2) PF_ACC(6);
        }
        if (!ok) break;
        uint32_t v[16];
        if (s == n_ks) {
          const uint32_t w16[16] = {bq[0].x, bq[0].y, bq[0].z, bq[0].w, bq[1].x, bq[1].y, bq[1].z, bq[1].w,
                                    bq[2].x, bq[2].y, bq[2].z, bq[2].w, bq[3].x, bq[3].y, bq[3].z, bq[3].w};
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = w16[i];
        } else {
          const uint8_t* stage = smem + st * kStageBytes;
          const uint4 cw = *reinterpret_cast<const uint4*>(stage + kHBytesT + row * 32 + g * 16);  // 32 codes
          if ((s & 3) == 0) ++grp;
          const uint32_t sw = *reinterpret_cast<const uint16_t*>(smem + p.off_scales + (grp % kScaleSlots) * kScaleBytes +
                                                                  row * 16 + (s & 3) * 4 + g * 2);
          const uint32_t s01 = cvt_e4m3x2_to_f16x2(sw);
          const uint32_t sa = prmt(s01, s01, 0x1010u), sb = prmt(s01, s01, 0x3232u);
          e2m1x8_to_f16x8(cw.x, v[0], v[1], v[2], v[3]);
          e2m1x8_to_f16x8(cw.y, v[4], v[5], v[6], v[7]);
          e2m1x8_to_f16x8(cw.z, v[8], v[9], v[10], v[11]);
          e2m1x8_to_f16x8(cw.w, v[12], v[13], v[14], v[15]);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = hmul2_u32(v[i], sa);
#pragma unroll
          for (int i = 8; i < 16; ++i) v[i] = hmul2_u32(v[i], sb);
        }
        tmem_st16(tmem + lane_addr + 32u * a + 16u * g, v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(smem_u32(&C.afull[a]));
          else mbar_arrive_leader(smem_u32(&C.afull[a]));
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    int it = 0;
    for (int tile = pair; tile < p.n_tiles && ok; tile += npairs, ++it) {
      const TileAt at = tile_at(p, tile);
      const int mt = at.mt, gi = at.gi;
      const int b = it & 1;
      const GMember& G = p.g[gi];
      const float s_g = C.s_g[gi];
      const int64_t o = static_cast<int64_t>(at.otl) * 2 * kTO + rank * kTO + row;
      {
        PF_T0();
        ok = wait_p(smem_u32(&C.dfull[b]), (it >> 1) & 1, abort_flag) &&
             wait_p(smem_u32(&C.tfull[b]), (it >> 1) & 1, abort_flag);
        if (lane == 0 && warp == 10) PF_ACC(7);
      }
      if (!ok) break;
      tc_fence_after();
      const float* rsc = reinterpret_cast<const float*>(smem + p.off_t + b * p.t_slot_bytes);
      for (int cb = 0; cb < TN / 16; ++cb) {
        const int col = cb * 16;  // token columns [col, col + 16) of the tile
        uint32_t dv[16];
        tmem_ld16(tmem + lane_addr + (kColD0 + static_cast<uint32_t>(TN) * b) + col, dv);
        tmem_ld_wait();
        if (o < G.d_o) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int64_t m = static_cast<int64_t>(mt) * TN + col + i;
            const float v = s_g * rsc[col + i] * __uint_as_float(dv[i]);
            if (m < p.M) {
              if (p.y_f32) static_cast<float*>(G.y)[m * G.d_o + o] = v;
              else static_cast<__nv_bfloat16*>(G.y)[m * G.d_o + o] = __float2bfloat16_rn(v);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(smem_u32(&C.dempty[b]));
        else mbar_arrive_leader(smem_u32(&C.dempty[b]));
        mbar_arrive(smem_u32(&C.tempty[b]));
      }
    }
  }
  // both CTAs are done (the even CTA's last MMA has completed) before either frees its
  // tensor memory or leaves while the other may still signal it
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem, kTmemCols);
  }
#ifdef PL_TIMELINE
  if (threadIdx.x == 0 && blockIdx.x < 1024) g_pf_wait[blockIdx.x][11] = globaltimer_ns();
#endif
}

// ------------------------------------------------------------------ LoRA down-projection
constexpr int kLdStages = 8;
constexpr int kLdThreads = 6 * 32;  // TMA, MMA, 4 epilogue warps
constexpr uint32_t kLdH = 128 * kKS * 2;  // 16 KB

// One adapter of a down-projection launch: its r rows of A16 (and columns of the MMA's N)
// start at col0; the launch writes its Tq.
struct LMember {
  int r, col0;
  float lambda;
  const float* s_g;
  __nv_bfloat16* Tq;       // [Mp][64]: bf16(T), T = (lambda / s_g) A hq, zero beyond r
  float* t;                // or, when not null, t[m][j] = c_m (A hq)[m][j] = (A h)[m][j] in FP32
  int t_ld;
};
struct LParams {
  int64_t M, d_i, Mp;
  const float* rowscale;   // [M]: c_m (read in the t form only)
  int rb, n_ks, splits, stages;  // rb: every member's rows, each rounded up to 16 (the MMA's N)
  float* t_part;           // [splits][Mp][rb]
  int* counters;           // [token tiles]; zero on entry
  int mtiles, n_m;
  LMember m[kMaxPrefillGroup];
};
struct LMaps {
  CUtensorMap hq, a16;
};
struct LCtrl {
  uint64_t full[kLdStages], empty[kLdStages], dfull;
  uint32_t tmem_base;
  int abort_flag;
  int last;  // this CTA is the last split of its token tile to finish
};

__global__ void __launch_bounds__(kLdThreads, 1) k_lora_down(const __grid_constant__ LMaps maps, const LParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t abytes = static_cast<uint32_t>(p.rb) * kKS * 2;
  const uint32_t stage_bytes = kLdH + abytes;
  const int nst = p.stages;
  LCtrl& C = *reinterpret_cast<LCtrl*>(smem + nst * stage_bytes);
  volatile int* abort_flag = &C.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const int mtile = blockIdx.x / p.splits, sp = blockIdx.x % p.splits;
  const int s0 = (sp * p.n_ks) / p.splits, s1 = ((sp + 1) * p.n_ks) / p.splits;
  const int32_t m0 = mtile * 128;
  if (threadIdx.x == 0) {
    pdl_launch_dependents();
    for (int s = 0; s < nst; ++s) {
      mbar_init(smem_u32(&C.full[s]), 1);
      mbar_init(smem_u32(&C.empty[s]), 1);
    }
    mbar_init(smem_u32(&C.dfull), 1);
    C.abort_flag = 0;
    fence_mbar_init();
  }
  const uint32_t tcols = p.rb <= 32 ? 32u : (p.rb <= 64 ? 64u : 128u);
  if (warp == 1) {
    tmem_alloc(smem_u32(&C.tmem_base), tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;
  if (warp == 0) {
    if (lane == 0) {
      pdl_wait();  // hq and A16 come from the row prologue
      bool ok = true;
      int i = 0;
      for (int s = s0; s < s1 && ok; ++s, ++i) {
        const int st = i % nst;
        if (i >= nst) ok = wait_p(smem_u32(&C.empty[st]), ((i / nst) - 1) & 1, abort_flag);
        if (!ok) break;
        const uint32_t fb = smem_u32(&C.full[st]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        tma_load_2d(sbase + st * stage_bytes, &maps.hq, s * kKS, m0, fb);
        tma_load_2d(sbase + st * stage_bytes + kLdH, &maps.a16, s * kKS, 0, fb);
      }
      if (*abort_flag)
        for (int d = i - nst > 0 ? i - nst : 0; d < i; ++d) drain(smem_u32(&C.full[d % nst]), (d / nst) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, p.rb, 0);
      bool ok = true;
      int i = 0;
      for (int s = s0; s < s1 && ok; ++s, ++i) {
        const int st = i % nst;
        ok = wait_p(smem_u32(&C.full[st]), (i / nst) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint64_t hd = smem_desc_sw128(sbase + st * stage_bytes, 1024);
        const uint64_t ad = smem_desc_sw128(sbase + st * stage_bytes + kLdH, 1024);
#pragma unroll
        for (int kk = 0; kk < kKS / 16; ++kk) mma_ss(tmem, hd + 2u * kk, ad + 2u * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(smem_u32(&C.empty[st]));
      }
      tc_commit(smem_u32(&C.dfull));
    }
  } else {
    const int quarter = warp & 3;
    const int64_t m = static_cast<int64_t>(m0) + quarter * 32 + lane;  // < Mp
    const bool ok = wait_p(smem_u32(&C.dfull), 0, abort_flag) && !*abort_flag && s1 > s0;
    tc_fence_after();
    float* part = p.t_part + (static_cast<int64_t>(sp) * p.Mp + m) * p.rb;
    uint32_t v[16];
    for (int jb = 0; jb < p.rb; jb += 16) {
      tmem_ld16(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + jb, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) part[jb + j] = (ok && m < p.M) ? __uint_as_float(v[j]) : 0.f;
    }
    __threadfence();
    named_bar(1, 128);
    if (threadIdx.x == 64) C.last = atomicAdd(&p.counters[mtile], 1) == p.splits - 1;
    named_bar(1, 128);
    for (int mi = 0; C.last && mi < p.n_m; ++mi) {
      // every split of this token tile is in memory: add member mi's columns up in split order
      __threadfence();
      const LMember& L = p.m[mi];
      const float f = L.t != nullptr ? 1.f : L.lambda / *L.s_g;  // the t form has no s_g
      const int R4 = (L.r + 3) / 4 * 4;
      float acc[kMaxR];
#pragma unroll
      for (int j = 0; j < kMaxR; ++j) acc[j] = 0.f;
      for (int q = 0; q < p.splits; ++q) {  // all loads of one split issued together
        const float4* src =
            reinterpret_cast<const float4*>(p.t_part + (static_cast<int64_t>(q) * p.Mp + m) * p.rb + L.col0);
        float4 v[kMaxR / 4];
#pragma unroll
        for (int j4 = 0; j4 < kMaxR / 4; ++j4) v[j4] = 4 * j4 < R4 ? __ldcg(src + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j4 = 0; j4 < kMaxR / 4; ++j4) {
          acc[4 * j4] += v[j4].x;
          acc[4 * j4 + 1] += v[j4].y;
          acc[4 * j4 + 2] += v[j4].z;
          acc[4 * j4 + 3] += v[j4].w;
        }
      }
      if (L.t != nullptr) {  // FP32 t = c_m A hq (the W8A8 form's adapter input)
        if (m < p.M) {
          const float c = p.rowscale[m];
#pragma unroll
          for (int j = 0; j < kMaxR; ++j)
            if (j < L.r) L.t[m * L.t_ld + j] = c * acc[j];
        }
        continue;
      }
      // the LoRA step's B operand row: 64 bf16, T in the first r, zero beyond
      uint4* dst = reinterpret_cast<uint4*>(L.Tq + m * kLoraK);
#pragma unroll
      for (int q = 0; q < kLoraK / 8; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int j = 8 * q + 2 * h;
          const float lo = j < L.r && j < kMaxR ? f * acc[j < kMaxR ? j : 0] : 0.f;
          const float hi = j + 1 < L.r && j + 1 < kMaxR ? f * acc[j + 1 < kMaxR ? j + 1 : 0] : 0.f;
          w[h] = f32x2_to_bf16x2(lo, hi);
        }
        dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}


// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* base, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of the per-token arrays (row scales, Tq): a multiple of every token tile (128, 160
// or 192 for the GEMM, 128 for the down-projection), so that whole tiles can be read and
// written.
int64_t m_pad(int64_t M) { return (M + 1919) / 1920 * 1920; }

constexpr int kMaxLdSplits = 8;

// Workspace of one launch: the shared f16 rows and row scales; the f16 adapters of every
// member with one, side by side (each member's rows rounded up to 16, the padding zero); the
// down-projection's split partials and counters; per member its Tq.
int r16(int r) { return (r + 15) / 16 * 16; }

struct PfWs {
  __half* hq;
  float* rowscale;
  __half* A16;            // [rb][d_i], rb = sum of the members' r16(r)
  float* t_part;          // [kMaxLdSplits][Mp][rb]
  int* counters;          // [token tiles of the down-projection]
  __nv_bfloat16* Tq[kMaxPrefillGroup];  // [Mp][64]: bf16(T), zero beyond r
  size_t bytes;
};

PfWs carve(void* ws, int64_t M, int64_t d_i, const int* r, int n) {
  PfWs w{};
  const uintptr_t b = reinterpret_cast<uintptr_t>(ws);
  size_t off = 0;
  const int64_t Mp = m_pad(M);
  int rb = 0;
  for (int i = 0; i < n; ++i) rb += r16(r[i]);
  w.hq = reinterpret_cast<__half*>(b + off);
  off += align_up(static_cast<size_t>(M) * d_i * 2, 256);
  w.rowscale = reinterpret_cast<float*>(b + off);
  off += align_up(static_cast<size_t>(Mp) * 4, 256);
  if (rb > 0) {
    w.A16 = reinterpret_cast<__half*>(b + off);
    off += align_up(static_cast<size_t>(rb) * d_i * 2, 256);
    w.t_part = reinterpret_cast<float*>(b + off);
    off += align_up(static_cast<size_t>(kMaxLdSplits) * Mp * rb * 4, 256);
    w.counters = reinterpret_cast<int*>(b + off);
    off += align_up(static_cast<size_t>((M + 127) / 128 + 6) * 4, 256);
  }
  for (int i = 0; i < n; ++i) {
    if (r[i] == 0) continue;
    w.Tq[i] = reinterpret_cast<__nv_bfloat16*>(b + off);
    off += align_up(static_cast<size_t>(Mp) * kLoraK * 2, 256);
  }
  w.bytes = off;
  return w;
}

struct GPlan {
  int stages;
  uint32_t off_scales, off_t, t_slot_bytes, off_ctrl;
  size_t smem;
};

GPlan gplan(int r, int tn) {
  GPlan g{};
  const uint32_t kStageBytes = stage_bytes_of(tn);
  g.t_slot_bytes = static_cast<uint32_t>(align_up(static_cast<size_t>(tn) * 4, 128));  // row scales of a tile
  const size_t fixed = kScaleSlots * kScaleBytes + 2 * static_cast<size_t>(g.t_slot_bytes) + sizeof(GCtrl) + 128 + 1024;
  int st = static_cast<int>((227 * 1024 - fixed) / kStageBytes);
  g.stages = st > kMaxStages ? kMaxStages : st;
  g.off_scales = g.stages * kStageBytes;
  g.off_t = g.off_scales + kScaleSlots * kScaleBytes;
  g.off_ctrl = static_cast<uint32_t>(align_up(g.off_t + 2 * static_cast<size_t>(g.t_slot_bytes), 128));
  g.smem = g.off_ctrl + sizeof(GCtrl) + 1024;
  return g;
}

cudaError_t set_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(k_gemm_nvfp4<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_gemm_nvfp4<160>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_gemm_nvfp4<192>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_lora_down, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  return err;
}

}  // namespace

bool prefill_supported(int64_t M, int64_t d_i, int64_t d_o, int r) {
  return M > 64 && d_i >= 256 && d_i % 256 == 0 && d_i <= 32768 && d_o >= 1 && r >= 0 && r <= kMaxR &&
         gplan(r, kTN).stages >= 3;
}

bool prefill_group_supported(int64_t M, int64_t d_i, const TcProj* projs, int n) {
  if (n < 1 || n > kMaxPrefillGroup) return false;
  for (int i = 0; i < n; ++i)
    if (!prefill_supported(M, d_i, projs[i].d_o, projs[i].r)) return false;
  return true;
}

size_t prefill_group_workspace_bytes(int64_t M, int64_t d_i, const TcProj* projs, int n) {
  int r[kMaxPrefillGroup] = {0};
  for (int i = 0; i < n && i < kMaxPrefillGroup; ++i) r[i] = projs[i].r;
  return carve(nullptr, M, d_i, r, n < kMaxPrefillGroup ? n : kMaxPrefillGroup).bytes;
}

size_t prefill_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r) {
  const TcProj one{d_o, nullptr, nullptr, nullptr, nullptr, nullptr, r, 0.f, nullptr, 0};
  return prefill_group_workspace_bytes(M, d_i, &one, 1);
}

cudaError_t launch_linear_prefill_group(const LinearArgs& in, const TcProj* projs, int n, cudaStream_t stream) {
  cudaError_t e = set_attributes();
  if (e != cudaSuccess) return e;
  if (n < 1 || n > kMaxPrefillGroup) return cudaErrorInvalidValue;
  int r[kMaxPrefillGroup] = {0};
  for (int i = 0; i < n; ++i) r[i] = projs[i].A != nullptr && projs[i].B != nullptr ? projs[i].r : 0;
  const PfWs w = carve(in.ws, in.M, in.d_i, r, n);
  const int64_t Mp = m_pad(in.M);
  const int mtiles = static_cast<int>((in.M + 127) / 128);  // token tiles of the LoRA down-projection

  // 1. one row pass for the group; every adapter to f16 (side by side, padding rows zeroed),
  //    the down-projection's counters zeroed
  ActConv conv{};
  int rb = 0, col0[kMaxPrefillGroup] = {0};
  for (int i = 0; i < n; ++i) {
    col0[i] = rb;
    rb += r16(r[i]);
  }
  if (rb > 0) {
    conv.zero[conv.n_zero_ranges] = reinterpret_cast<float*>(w.counters);
    conv.n_zero[conv.n_zero_ranges++] = (mtiles + 3) / 4 * 4;
  }
  for (int i = 0; i < n; ++i) {
    if (r[i] == 0) continue;
    conv.A[conv.n] = projs[i].A;
    conv.A16[conv.n] = w.A16 + static_cast<int64_t>(col0[i]) * in.d_i;
    conv.r[conv.n] = r[i];
    ++conv.n;
    if (r16(r[i]) > r[i]) {  // padding rows: (r16 - r) d_i halves = (r16 - r) d_i / 2 floats
      conv.zero[conv.n_zero_ranges] = reinterpret_cast<float*>(w.A16 + static_cast<int64_t>(col0[i] + r[i]) * in.d_i);
      conv.n_zero[conv.n_zero_ranges++] = static_cast<int64_t>(r16(r[i]) - r[i]) * in.d_i / 2;
    }
  }
  e = launch_act_prologue(in, w.hq, w.rowscale, conv, stream);
  if (e != cudaSuccess) return e;

  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  const int n_ks = static_cast<int>(in.d_i / kKS);
  const int sms = sm_count();

  // 2. the adapters' down-projection, every member at once (the MMA's N = rb):
  //    Tq_i = bf16((lambda_i / s_g_i) A_i hq)
  if (rb > 0) {
    LMaps lm;
    bool ok = encode_2d(&lm.hq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.hq, in.d_i, in.M, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_2d(&lm.a16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.A16, in.d_i, rb, 64, rb,
                        CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;
    LParams lp{};
    lp.M = in.M;
    lp.d_i = in.d_i;
    lp.Mp = Mp;
    lp.rb = rb;
    lp.n_ks = n_ks;
    int splits = sms / mtiles;  // one wave: every split of every token tile resident at once
    splits = splits > kMaxLdSplits ? kMaxLdSplits : splits;
    splits = splits > n_ks ? n_ks : (splits < 1 ? 1 : splits);  // every split has at least one K step
    lp.splits = splits;
    const size_t stage_bytes = kLdH + static_cast<size_t>(rb) * kKS * 2;
    int st = static_cast<int>((227 * 1024 - sizeof(LCtrl) - 1024) / stage_bytes);
    lp.stages = st > kLdStages ? kLdStages : st;
    lp.t_part = w.t_part;
    lp.counters = w.counters;
    lp.mtiles = mtiles;
    for (int i = 0; i < n; ++i) {
      if (r[i] == 0) continue;
      lp.m[lp.n_m++] = LMember{r[i], col0[i], projs[i].lambda, projs[i].s_g, w.Tq[i], nullptr, 0};
    }
    cudaLaunchConfig_t c{};
    c.gridDim = dim3(static_cast<unsigned>(mtiles * splits));
    c.blockDim = dim3(kLdThreads);
    c.dynamicSmemBytes = lp.stages * stage_bytes + sizeof(LCtrl) + 1024;
    c.stream = stream;
    c.attrs = pdl;
    c.numAttrs = 1;
    e = cudaLaunchKernelEx(&c, k_lora_down, lm, lp);
    if (e != cudaSuccess) return e;
  }

  // 3. one contraction over every member's pairs of weight tiles (o fastest).  Token tiles
  // of 128 when 192 leaves pairs idle; else 192 (the widest MMA the two accumulator buffers
  // allow) or 160, whichever needs fewer rounds of the pairs, a round of 160-token tiles
  // costing 0.966 of one of 192 (measured)
  const int pairs = sms / 2;
  int64_t n_ot64 = 0;
  for (int i = 0; i < n; ++i) n_ot64 += (projs[i].d_o + 2 * kTO - 1) / (2 * kTO);
  auto rounds = [&](int t) { return (n_ot64 * ((in.M + t - 1) / t) + pairs - 1) / pairs; };
  int tn = kTN;
  if (n_ot64 * ((in.M + tn - 1) / tn) < pairs) tn = 128;
  else if (0.966 * static_cast<double>(rounds(160)) < static_cast<double>(rounds(192))) tn = 160;
  GMaps gm;
  memset(&gm, 0, sizeof(gm));
  bool ok = encode_2d(&gm.hq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.hq, in.d_i, in.M, 64, tn / 2,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  for (int i = 0; i < n && ok; ++i) {
    ok = encode_2d(&gm.codes[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, projs[i].codes, in.d_i / 2, projs[i].d_o, kKS / 2,
                   kTO, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode_2d(&gm.scales[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, projs[i].scales, in.d_i / 16, projs[i].d_o, 16,
                   kTO, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (ok && r[i] > 0)
      ok = encode_2d(&gm.tq[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.Tq[i], kLoraK, Mp, 64, tn / 2,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    else
      gm.tq[i] = gm.hq;  // unused
  }
  if (!ok) return cudaErrorInvalidValue;
  int rmax = 0;
  for (int i = 0; i < n; ++i) rmax = r[i] > rmax ? r[i] : rmax;
  const GPlan g = gplan(rmax, tn);
  GParams p{};
  p.M = in.M;
  p.d_i = in.d_i;
  p.n_ot = static_cast<int>(n_ot64);
  p.n_tiles = static_cast<int>(p.n_ot * ((in.M + tn - 1) / tn));
  p.n_ks = n_ks;
  p.stages = g.stages;
  p.n_g = n;
  p.rowscale = w.rowscale;
  p.y_f32 = in.y_f32 ? 1 : 0;
  p.off_scales = g.off_scales;
  p.off_t = g.off_t;
  p.t_slot_bytes = g.t_slot_bytes;
  p.off_ctrl = g.off_ctrl;
  const int mtiles_g = static_cast<int>((in.M + tn - 1) / tn);
  for (int i = 0, ot0 = 0, t0 = 0; i < n; ++i) {
    const int n_ot_i = static_cast<int>((projs[i].d_o + 2 * kTO - 1) / (2 * kTO));
    p.g[i].d_o = projs[i].d_o;
    p.g[i].r = r[i];
    p.g[i].ot0 = ot0;
    p.g[i].n_ot = n_ot_i;
    p.g[i].t0 = t0;
    t0 += n_ot_i * mtiles_g;
    p.g[i].s_g = projs[i].s_g;
    p.g[i].B = r[i] > 0 ? static_cast<const __nv_bfloat16*>(projs[i].B) : nullptr;
    p.g[i].y = projs[i].y;
    ot0 += static_cast<int>((projs[i].d_o + 2 * kTO - 1) / (2 * kTO));
  }
  cudaLaunchAttribute gattrs[2];
  gattrs[0] = pdl[0];
  gattrs[1].id = cudaLaunchAttributeClusterDimension;
  gattrs[1].val.clusterDim.x = 2;
  gattrs[1].val.clusterDim.y = 1;
  gattrs[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t c{};
  c.gridDim = dim3(static_cast<unsigned>(2 * (p.n_tiles < pairs ? p.n_tiles : pairs)));
  c.blockDim = dim3(kThreads);
  c.dynamicSmemBytes = g.smem;
  c.stream = stream;
  c.attrs = gattrs;
  c.numAttrs = 2;
  if (tn == 128) return cudaLaunchKernelEx(&c, k_gemm_nvfp4<128>, gm, p);
  if (tn == 160) return cudaLaunchKernelEx(&c, k_gemm_nvfp4<160>, gm, p);
  return cudaLaunchKernelEx(&c, k_gemm_nvfp4<192>, gm, p);
}

size_t lora_down_t_scratch_bytes(int64_t M, int r) {
  const int64_t Mp = (M + 127) / 128 * 128;
  return align_up(static_cast<size_t>(kMaxLdSplits) * Mp * r16(r) * 4, 256);
}

cudaError_t launch_lora_down_t(const __half* hq, int64_t M, int64_t d_i, const __half* A16, int r,
                               const float* rowscale, float* t, int t_ld, float* t_part, int* counters,
                               cudaStream_t stream) {
  cudaError_t e = set_attributes();
  if (e != cudaSuccess) return e;
  const int rb = r16(r);
  const int mtiles = static_cast<int>((M + 127) / 128);
  const int n_ks = static_cast<int>(d_i / kKS);
  LMaps lm;
  if (!encode_2d(&lm.hq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hq, d_i, M, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&lm.a16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A16, d_i, rb, 64, rb, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  LParams lp{};
  lp.M = M;
  lp.d_i = d_i;
  lp.Mp = (M + 127) / 128 * 128;
  lp.rowscale = rowscale;
  lp.rb = rb;
  lp.n_ks = n_ks;
  int splits = sm_count() / mtiles;
  splits = splits > kMaxLdSplits ? kMaxLdSplits : splits;
  lp.splits = splits > n_ks ? n_ks : (splits < 1 ? 1 : splits);
  const size_t stage_bytes = kLdH + static_cast<size_t>(rb) * kKS * 2;
  const int st = static_cast<int>((227 * 1024 - sizeof(LCtrl) - 1024) / stage_bytes);
  lp.stages = st > kLdStages ? kLdStages : st;
  lp.t_part = t_part;
  lp.counters = counters;
  lp.mtiles = mtiles;
  lp.n_m = 1;
  lp.m[0] = LMember{r, 0, 0.f, nullptr, nullptr, t, t_ld};
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c{};
  c.gridDim = dim3(static_cast<unsigned>(mtiles * lp.splits));
  c.blockDim = dim3(kLdThreads);
  c.dynamicSmemBytes = lp.stages * stage_bytes + sizeof(LCtrl) + 1024;
  c.stream = stream;
  c.attrs = pdl;
  c.numAttrs = 1;
  return cudaLaunchKernelEx(&c, k_lora_down, lm, lp);
}

cudaError_t launch_linear_prefill(const LinearArgs& a, cudaStream_t stream) {
  const TcProj one{a.d_o, a.codes, a.scales, a.s_g, a.r > 0 ? a.A : nullptr, a.r > 0 ? a.B : nullptr, a.r, a.lambda,
                   a.y, 0};
  return launch_linear_prefill_group(a, &one, 1, stream);
}

#ifdef PL_TIMELINE
extern "C" int pl_debug_read_prefill_waits(unsigned long long* out) {
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  if (cudaMemcpyFromSymbol(out, g_pf_wait, sizeof(g_pf_wait)) != cudaSuccess) return 2;
  static unsigned long long zero[1024][12];
  return cudaMemcpyToSymbol(g_pf_wait, zero, sizeof(zero)) != cudaSuccess ? 3 : 0;
}
#endif

uint32_t prefill_read_and_clear_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_pf_status, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_pf_status, &zero, sizeof(zero));
  return v;
}

}  // namespace pl
