// tcgen05 tensor-core NVFP4 + LoRA linear (decode, M <= 64), sm_103a.
//
// Computes the forward map of "QeRL: When Quantized Weights Help Reinforcement
// Learning, and Where the Evidence Stops", section 2.1 (y = W_hat h + lambda B (A h))
// on the section 3.1 NVFP4 backbone (w_hat = s_g s_b q) with the section 5.1
// RMSNorm-AQN input h = u (.) (w_norm + z).
//
// Two kernels per call, chained by programmatic dependent launch:
//
// k_act (a group of warps per token row): h = x / rms (.) (w_norm + z) in FP32, a power-of-two
//   c_m with max|h| / c_m in [2^13, 2^14), and the f16 activations h / c_m (11-bit
//   significand, no overflow) into the workspace; a few more CTAs copy the LoRA matrix
//   A into the workspace as f16.
//
// k_tc_decode (a cluster of S CTAs per 128 weight rows; CTA s takes the s-th slice of
//   the K = d_i axis in chunks of 256):
//   * warp 0 TMA-loads, per chunk, the packed codes (128 rows x 128 B, 128-byte
//     swizzle) and E4M3 scales (128 x 16 B) -- issued before the wait on k_act, they
//     do not depend on it -- the f16 activations (N rows x 256, 128-byte swizzle:
//     the canonical K-major layout) and the chunk of the f16 copy of A (r x 256);
//   * warps 2..9 dequantise: each thread owns one weight row and half the chunk, turns
//     8 codes per 32-bit word into 4 f16x2 words with the hardware E2M1 conversion,
//     multiplies by the block scale (q * s_b is exact in f16) and stores them into
//     tensor memory, where they are the MMA's A operand;
//   * four warps issue tcgen05.mma kind::f16 (K = 16 each; one thread issues one only
//     every few tens of ns, so the work is shared): weights (tensor memory) x
//     activations^T into accumulator D1, and A (shared memory, 128-row operand whose
//     rows >= r are don't-care) x activations^T into accumulator Dt, whose lanes < r are
//     this CTA's K slice of t = A h -- each of D1 and Dt as two partial sums over the two
//     halves of every chunk's K steps;
//   * epilogue (warps 2..9): every CTA adds the partial sums and puts s_g c_m D1 and its
//     Dt slice in shared memory; after a cluster barrier CTA s sums, over DSMEM and in split order
//     (deterministic), the t slices of all S CTAs into t, and the D1 partials of its
//     share of the 128 rows; it adds the LoRA up-projection lambda B t on CUDA cores
//     and writes y.
//
// Every mbarrier wait is bounded (200 ms); a wait that gives up sets the device
// status word, the CTA drains its own copies and MMAs (again bounded), frees its
// tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace pl {

__device__ uint32_t g_tc_status = 0;

// Phase timestamps for development builds (-DPL_TIMELINE); compiled out otherwise.
#ifdef PL_TIMELINE
__device__ unsigned long long g_tl_main[1024][16];
__device__ unsigned long long g_tl_pro[256][8];
__device__ unsigned long long g_tl_chunk[1024][4][32];  // per chunk: W issued, MMA ready, A ready, dequant start
#define PL_TLC(kind, c) do { if (blockIdx.x < 1024 && (c) < 32) g_tl_chunk[blockIdx.x][kind][c] = globaltimer_ns(); } while (0)
#define PL_TL(slot) do { if (blockIdx.x < 1024) g_tl_main[blockIdx.x][slot] = globaltimer_ns(); } while (0)
#define PL_TLP(slot) do { const unsigned b_ = blockIdx.x + gridDim.x * blockIdx.y; \
                          if (b_ < 256) g_tl_pro[b_][slot] = globaltimer_ns(); } while (0)
#else
#define PL_TL(slot) do { } while (0)
#define PL_TLP(slot) do { } while (0)
#define PL_TLC(kind, c) do { } while (0)
#endif

namespace {

constexpr int kTileO = 128;
constexpr int kChunkK = 256;
constexpr int kCodesBytes = kTileO * kChunkK / 2;   // 16 KB
constexpr int kScaleBytes = kTileO * kChunkK / 16;  // 2 KB
constexpr int kDeqWarps = 8;
constexpr int kIssuers = 4;        // MMA-issuing warps: D1 and Dt, each in two K halves
constexpr int kThreads = (2 + kDeqWarps + kIssuers - 1) * 32;  // producer, issuer 0, dequant/epilogue, issuers 1..3
constexpr int kEpiThreads = kDeqWarps * 32;
constexpr int kMaxStages = 8;
constexpr int kMaxSplit = 8;
constexpr int kMaxLa = 3;  // slots of the shared-memory ring of A chunks
constexpr int kMaxN = 64;
constexpr int kMaxR = 64;
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: kAbuf weight (MMA A operand) buffers of 128 columns from 0, then
// the accumulators of the four issuers, N <= 64 columns each: D1 over the first and the
// second half of every chunk's K steps, and Dt likewise
constexpr int kAbuf = 2;
constexpr uint32_t kColA0 = 0;
constexpr uint32_t kColAcc = 256;  // issuer q accumulates at kColAcc + 64 q
static_assert(kAbuf * 128 <= kColAcc && kColAcc + kIssuers * kMaxN <= kTmemCols, "TMEM columns");
constexpr int kTStride = kMaxR + 4;  // floats per token row of the t buffers (16-byte rows, spread banks)

struct TcParams {
  int64_t M, d_i, d_o;
  int N, r, rb, tiles, splits, kc, stages, la;
  uint32_t stage_bytes;
  float lambda;
  const float* s_g;
  const float* rowscale;
  const __nv_bfloat16* Blora;
  void* y;
  int y_f32;
};

struct TcMaps {
  CUtensorMap codes, scales, hq, alora;
};

struct Smem {
  uint64_t wfull[kMaxStages], hfull[kMaxStages], empty[kMaxStages];
  uint64_t a_full[kAbuf], a_empty[kAbuf];
  uint64_t lfull[kMaxLa], lempty[kMaxLa];  // shared-memory ring of A chunks
  uint64_t d_full;
  uint32_t tmem_base;
  int abort_flag;
  float s_g;
  float rowscale[kMaxN];
};

// Wait that also gives up when another role of the CTA has already given up.
PL_DEVINL bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return wait_or_abort_status(bar, parity, abort_flag, &g_tc_status);
}

// Test probe of the bounded-wait path: waits on a barrier that nothing completes,
// gives up after `limit_ns`, records the time-out in the status word and returns.
__global__ void k_wait_timeout_probe(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    const uint64_t t0 = globaltimer_ns();
    bool done = false;
    while (!done && globaltimer_ns() - t0 < limit_ns) done = mbar_try_wait(smem_u32(&bar), 0);
    if (!done) atomicOr(&g_tc_status, kStatusTimeout);
  }
}

// ------------------------------------------------------------------ activation prologue
constexpr int kActThreads = 256;
constexpr int kActWarps = kActThreads / 32;  // token rows in flight per CTA
constexpr int kActPieces = 16;               // 16-byte pieces of x per thread, held in registers
constexpr int kActUnroll = 4;                // loads per thread in flight in the copy loops

// CTAs 0 .. n_row_ctas-1: token rows, a group of wpr warps per row (kActWarps / wpr rows
// per CTA, rows strided over the CTAs).  w + z of the whole row sits in shared memory
// (FP32); the group holds its row of x in registers while sum(x^2) and max |x (w + z)|
// are reduced, then writes hq = f16(x (w + z) inv / c_m) and c_m.
// CTAs n_row_ctas and up: the f16 copy of A (r x d_i), 8 elements per thread and slot, and
// zeros into `zero` (n_zero floats, a multiple of 4; the accumulator of the large-M
// LoRA down-projection), 4 per thread and slot.
// kRowZ: z holds one noise vector per token row (z_ld floats apart), added to w_norm as
// each row is taken; otherwise w_norm + z is formed once, in shared memory.
template <bool kRowZ>
__global__ void __launch_bounds__(kActThreads, 2) k_act(const __nv_bfloat16* __restrict__ x, int64_t M, int64_t d_i,
                                                     const float* __restrict__ w_norm,
                                                     const float* __restrict__ z, int64_t z_ld, float eps,
                                                     __half* __restrict__ hq, float* __restrict__ rowscale,
                                                     const __nv_bfloat16* __restrict__ A, int r,
                                                     __half* __restrict__ A16, float* __restrict__ zero,
                                                     int64_t n_zero, int n_row_ctas, int wpr) {
  extern __shared__ float4 g4[];  // [d_i / 4]: w_norm + z of the whole row (1 without the norm)
  __shared__ float red_s[kActWarps], red_m[kActWarps];
  if (threadIdx.x == 0) {
    PL_TLP(0);
    pdl_launch_dependents();
  }
  pdl_wait();  // x may come from the preceding kernel, which may also still read the workspace
  if (threadIdx.x == 0) PL_TLP(1);
  if (static_cast<int>(blockIdx.x) >= n_row_ctas) {
    const int64_t nslot = static_cast<int64_t>(r) * d_i / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x - n_row_ctas) * kActThreads;
    // kActUnroll slots per thread and round, every load of the round in flight before the stores
    for (int64_t s0 = (blockIdx.x - n_row_ctas) * kActThreads + threadIdx.x; s0 < nslot; s0 += kActUnroll * stride) {
      uint4 v[kActUnroll];
#pragma unroll
      for (int u = 0; u < kActUnroll; ++u) {
        const int64_t sl = s0 + u * stride;
        if (sl < nslot) v[u] = reinterpret_cast<const uint4*>(A)[sl];
      }
#pragma unroll
      for (int u = 0; u < kActUnroll; ++u) {
        const int64_t sl = s0 + u * stride;
        if (sl < nslot)
          reinterpret_cast<uint4*>(A16)[sl] =
              make_uint4(f32x2_to_f16x2(bf16lo_to_f32(v[u].x), bf16hi_to_f32(v[u].x)),
                         f32x2_to_f16x2(bf16lo_to_f32(v[u].y), bf16hi_to_f32(v[u].y)),
                         f32x2_to_f16x2(bf16lo_to_f32(v[u].z), bf16hi_to_f32(v[u].z)),
                         f32x2_to_f16x2(bf16lo_to_f32(v[u].w), bf16hi_to_f32(v[u].w)));
      }
    }
    for (int64_t sl = (blockIdx.x - n_row_ctas) * kActThreads + threadIdx.x; sl < n_zero / 4; sl += stride)
      reinterpret_cast<float4*>(zero)[sl] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const bool norm = w_norm != nullptr, noise = !kRowZ && norm && z != nullptr;
  // one noise vector per token row: added row by row below, w_norm alone in g4
  const float* zrows = (kRowZ && norm) ? z : nullptr;
  const int64_t n4 = d_i / 4;
  for (int64_t i0 = threadIdx.x; i0 < n4; i0 += kActUnroll * kActThreads) {
    float4 g[kActUnroll], zz[kActUnroll];
#pragma unroll
    for (int u = 0; u < kActUnroll; ++u) {  // every load of the round in flight
      const int64_t i = i0 + u * kActThreads;
      g[u] = make_float4(1.f, 1.f, 1.f, 1.f);
      zz[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < n4) {
        if (norm) g[u] = reinterpret_cast<const float4*>(w_norm)[i];
        if (noise) zz[u] = reinterpret_cast<const float4*>(z)[i];
      }
    }
#pragma unroll
    for (int u = 0; u < kActUnroll; ++u) {
      const int64_t i = i0 + u * kActThreads;
      if (i < n4) g4[i] = make_float4(g[u].x + zz[u].x, g[u].y + zz[u].y, g[u].z + zz[u].z, g[u].w + zz[u].w);
    }
  }
  __syncthreads();
  // a group of wpr warps per token row (wpr = 1 for rows up to 8 KB): thread t of the group
  // holds the 16-byte pieces t, t + 32 wpr, ... of x in registers (at most kActPieces: the
  // host picks wpr so), for the row statistics and then the scaled f16 row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_cta = kActWarps / wpr, grp = warp / wpr, gt = (warp % wpr) * 32 + lane, gstride = 32 * wpr;
  const int64_t nv8 = d_i / 8;
  const int64_t per_round = static_cast<int64_t>(n_row_ctas) * rows_cta;
  const int64_t rounds = (M + per_round - 1) / per_round;
  for (int64_t rd = 0; rd < rounds; ++rd) {
    const int64_t m = rd * per_round + static_cast<int64_t>(blockIdx.x) * rows_cta + grp;
    const bool live = m < M;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (live ? m : 0) * d_i);
    const float4* zr = kRowZ && zrows != nullptr ? reinterpret_cast<const float4*>(zrows + (live ? m : 0) * z_ld)
                                                  : nullptr;
    // w_norm + z of this row for piece q (8 channels)
    auto gpiece = [&](int64_t q, float (&g8)[8]) {
      float4 ga = g4[2 * q], gb = g4[2 * q + 1];
      if (kRowZ && zr != nullptr) {
        const float4 za = zr[2 * q], zb = zr[2 * q + 1];
        ga.x += za.x; ga.y += za.y; ga.z += za.z; ga.w += za.w;
        gb.x += zb.x; gb.y += zb.y; gb.z += zb.z; gb.w += zb.w;
      }
      g8[0] = ga.x; g8[1] = ga.y; g8[2] = ga.z; g8[3] = ga.w;
      g8[4] = gb.x; g8[5] = gb.y; g8[6] = gb.z; g8[7] = gb.w;
    };
    uint4 xv[kActPieces];
#pragma unroll
    for (int i = 0; i < kActPieces; ++i) {
      const int64_t q = gt + static_cast<int64_t>(i) * gstride;
      xv[i] = live && q < nv8 ? xr[q] : make_uint4(0u, 0u, 0u, 0u);  // every load of the row in flight
    }
    float ss = 0.f, mx = 0.f;
#pragma unroll
    for (int i = 0; i < kActPieces; ++i) {
      const int64_t q = gt + static_cast<int64_t>(i) * gstride;
      if (q < nv8) {
        float g8[8];
        gpiece(q, g8);
        const uint32_t w4[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a0 = bf16lo_to_f32(w4[j]), a1 = bf16hi_to_f32(w4[j]);
          ss = fmaf(a0, a0, fmaf(a1, a1, ss));
          mx = fmaxf(mx, fmaxf(fabsf(a0 * g8[2 * j]), fabsf(a1 * g8[2 * j + 1])));
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
    if (wpr > 1) {  // the group's warps add up through shared memory
      if (lane == 0) {
        red_s[warp] = ss;
        red_m[warp] = mx;
      }
      __syncthreads();
      ss = 0.f;
      mx = 0.f;
      for (int w = grp * wpr; w < (grp + 1) * wpr; ++w) {
        ss += red_s[w];
        mx = fmaxf(mx, red_m[w]);
      }
      __syncthreads();
    }
    if (!live) continue;
    const float inv = norm ? 1.0f / sqrtf(ss / static_cast<float>(d_i) + eps) : 1.0f;
    const float hmax = inv * mx;
    int e = hmax > 0.f ? ilogbf(hmax) - 13 : 0;  // max |h| / c_m in [2^13, 2^14)
    e = e < -100 ? -100 : (e > 100 ? 100 : e);
    const float f = inv * ldexpf(1.0f, -e);
    if (gt == 0) rowscale[m] = ldexpf(1.0f, e);
    uint4* hr = reinterpret_cast<uint4*>(hq + m * d_i);
#pragma unroll
    for (int i = 0; i < kActPieces; ++i) {
      const int64_t q = gt + static_cast<int64_t>(i) * gstride;
      if (q < nv8) {
        const uint4 v = xv[i];
        float g8[8];
        gpiece(q, g8);
        hr[q] = make_uint4(f32x2_to_f16x2(bf16lo_to_f32(v.x) * g8[0] * f, bf16hi_to_f32(v.x) * g8[1] * f),
                           f32x2_to_f16x2(bf16lo_to_f32(v.y) * g8[2] * f, bf16hi_to_f32(v.y) * g8[3] * f),
                           f32x2_to_f16x2(bf16lo_to_f32(v.z) * g8[4] * f, bf16hi_to_f32(v.z) * g8[5] * f),
                           f32x2_to_f16x2(bf16lo_to_f32(v.w) * g8[6] * f, bf16hi_to_f32(v.w) * g8[7] * f));
      }
    }
  }
  if (threadIdx.x == 0) PL_TLP(5);
}

// ------------------------------------------------------------------ main kernel
__global__ void __launch_bounds__(kThreads, 1) k_tc_decode(const __grid_constant__ TcMaps maps,
                                                           const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int N = p.N, stages = p.stages, la = p.la;
  const uint32_t h_bytes = static_cast<uint32_t>(N) * 512u;
  const uint32_t l_bytes = static_cast<uint32_t>(p.rb) * 512u;  // one A chunk (rb rows x 256 bf16)
  uint8_t* lring = smem + static_cast<size_t>(stages) * p.stage_bytes;           // la A chunks
  __nv_bfloat16* sBt = reinterpret_cast<__nv_bfloat16*>(lring + la * l_bytes);  // [kMaxR][128]: B^T of the tile
  Smem& S = *reinterpret_cast<Smem*>(reinterpret_cast<uint8_t*>(sBt) + kTileO * kMaxR * 2);
  volatile int* abort_flag = &S.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  const int c0 = static_cast<int>((static_cast<int64_t>(split) * p.kc) / p.splits);
  const int c1 = static_cast<int>((static_cast<int64_t>(split + 1) * p.kc) / p.splits);
  const int nch = c1 - c0;
  const bool lora = p.r > 0;
  const int n_iss = lora ? kIssuers : 2;  // the Dt issuers idle without an adapter
  bool go = false;  // epilogue threads: this CTA's accumulators are valid

  const uint64_t pol_w = policy_evict_first();  // weights are streamed once
  const int pre = nch < stages ? nch : stages;
  const int32_t row0 = tile * kTileO;
  if (threadIdx.x == 0) {
    PL_TL(0);
    pdl_launch_dependents();
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&S.wfull[s]), 1);
      mbar_init(smem_u32(&S.hfull[s]), 1);
      mbar_init(smem_u32(&S.empty[s]), kDeqWarps + n_iss);
    }
    for (int b = 0; b < kAbuf; ++b) {
      mbar_init(smem_u32(&S.a_full[b]), kDeqWarps);
      mbar_init(smem_u32(&S.a_empty[b]), 2);
    }
    for (int b = 0; b < la; ++b) {
      mbar_init(smem_u32(&S.lfull[b]), 1);
      mbar_init(smem_u32(&S.lempty[b]), 2);
    }
    mbar_init(smem_u32(&S.d_full), n_iss);
    S.abort_flag = 0;
    fence_mbar_init();
    // the first stages of weights do not depend on the prologue: issue them at once
    for (int c = 0; c < pre; ++c) {
      uint8_t* st = smem + static_cast<size_t>(c) * p.stage_bytes;
      const uint32_t wb = smem_u32(&S.wfull[c]);
      mbar_arrive_expect_tx(wb, kCodesBytes + kScaleBytes);
      const int kc = c0 + c;
      PL_TLC(0, c);
      tma_load_2d_hint(smem_u32(st), &maps.codes, kc * (kChunkK / 2), row0, wb, pol_w);
      tma_load_2d_hint(smem_u32(st + kCodesBytes + h_bytes), &maps.scales, kc * (kChunkK / 16), row0, wb, pol_w);
    }
    tma_prefetch_desc(&maps.hq);
    if (lora) tma_prefetch_desc(&maps.alora);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  if (threadIdx.x == 0) PL_TL(1);

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const int lpre = lora ? (nch < la ? nch : la) : 0;
      PL_TL(2);
      pdl_wait();  // activations and the f16 copy of A come from the prologue
      PL_TL(3);
      for (int c = 0; c < pre; ++c) {
        uint8_t* st = smem + static_cast<size_t>(c) * p.stage_bytes;
        const uint32_t hb = smem_u32(&S.hfull[c]);
        mbar_arrive_expect_tx(hb, h_bytes);
        for (int q = 0; q < 4; ++q)
          tma_load_2d(smem_u32(st + kCodesBytes + q * N * 128), &maps.hq, (c0 + c) * kChunkK + 64 * q, 0, hb);
      }
      for (int c = 0; c < lpre; ++c) {
        const uint32_t lb = smem_u32(&S.lfull[c]);
        mbar_arrive_expect_tx(lb, l_bytes);
        for (int q = 0; q < 4; ++q)
          tma_load_2d(smem_u32(lring + c * l_bytes + q * p.rb * 128), &maps.alora, (c0 + c) * kChunkK + 64 * q, 0,
                      lb);
      }
      int c = pre, lc = lpre;
      bool ok = true;
      while (ok && (c < nch || lc < (lora ? nch : 0))) {
        // Issue in the order the MMA frees the buffers: A chunk lc reuses the ring slot of
        // chunk lc - la, weight chunk c the stage of chunk c - stages.  (Taking A first
        // whenever it is behind would wait on the MMA of the chunk just issued and leave
        // the weight stream one chunk deep.)
        if (lora && lc < nch && (c >= nch || lc - la <= c - stages)) {
          const int b = lc % la;
          ok = wait_or_abort(smem_u32(&S.lempty[b]), ((lc / la) - 1) & 1, abort_flag);
          if (!ok) break;
          const uint32_t lb = smem_u32(&S.lfull[b]);
          mbar_arrive_expect_tx(lb, l_bytes);
          for (int q = 0; q < 4; ++q)
            tma_load_2d(smem_u32(lring + b * l_bytes + q * p.rb * 128), &maps.alora, (c0 + lc) * kChunkK + 64 * q,
                        0, lb);
          ++lc;
          continue;
        }
        if (c >= nch) break;
        const int s = c % stages;
        ok = wait_or_abort(smem_u32(&S.empty[s]), ((c / stages) - 1) & 1, abort_flag);
        if (!ok) break;
        uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
        const uint32_t wb = smem_u32(&S.wfull[s]), hb = smem_u32(&S.hfull[s]);
        const int kc = c0 + c;
        PL_TLC(0, c);
        mbar_arrive_expect_tx(wb, kCodesBytes + kScaleBytes);
        tma_load_2d_hint(smem_u32(st), &maps.codes, kc * (kChunkK / 2), row0, wb, pol_w);
        tma_load_2d_hint(smem_u32(st + kCodesBytes + h_bytes), &maps.scales, kc * (kChunkK / 16), row0, wb, pol_w);
        mbar_arrive_expect_tx(hb, h_bytes);
        for (int q = 0; q < 4; ++q)
          tma_load_2d(smem_u32(st + kCodesBytes + q * N * 128), &maps.hq, kc * kChunkK + 64 * q, 0, hb);
        ++c;
      }
      if (*abort_flag) {  // every issued copy must land before this CTA exits
        for (int d = (c - stages > 0 ? c - stages : 0); d < c; ++d) {
          drain(smem_u32(&S.wfull[d % stages]), (d / stages) & 1);
          drain(smem_u32(&S.hfull[d % stages]), (d / stages) & 1);
        }
        for (int d = (lc - la > 0 ? lc - la : 0); d < lc; ++d) drain(smem_u32(&S.lfull[d % la]), (d / la) & 1);
      }
    }
  } else if (warp == 1 || warp >= 2 + kDeqWarps) {
    // ---------------------------------------------------------------- MMA issuers
    // One thread can issue a tcgen05.mma only every few tens of ns, so four warps share the
    // work: issuer q takes K steps [8 (q & 1), 8 (q & 1) + 8) of every chunk, q < 2 the
    // weights (tensor memory) x activations^T into D1 half q, q >= 2 the adapter A (shared
    // memory, a 128-row operand whose rows >= r are don't-care) x activations^T into Dt
    // half q - 2.  Each accumulator is a partial sum; the epilogue adds the two halves.
    const int q = warp == 1 ? 0 : warp - (1 + kDeqWarps);
    if (lane == 0 && q < n_iss) {
      const uint32_t idesc = idesc_f16(kTileO, N, 0);
      const uint32_t dcol = tmem + kColAcc + 64u * static_cast<uint32_t>(q);
      const int k0 = 8 * (q & 1);
      const bool wq = q < 2;
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        const int s = c % stages, b = c % kAbuf, lb = c % la;
        ok = (wq ? wait_or_abort(smem_u32(&S.a_full[b]), (c / kAbuf) & 1, abort_flag)
                 : wait_or_abort(smem_u32(&S.lfull[lb]), (c / la) & 1, abort_flag)) &&
             wait_or_abort(smem_u32(&S.hfull[s]), (c / stages) & 1, abort_flag);
        if (!ok) break;
        PL_TLC(wq ? 1 : 2, c);
        tc_fence_after();
        const uint32_t hbase = smem_u32(smem + static_cast<size_t>(s) * p.stage_bytes + kCodesBytes);
        if (wq) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int kk = k0 + i;
            const uint64_t bdesc = smem_desc_sw128(hbase + (kk >> 2) * N * 128 + (kk & 3) * 32, 1024);
            mma_ts(dcol, tmem + kColA0 + 128u * b + kk * 8, bdesc, idesc, (c > 0 || i > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&S.a_empty[b]));
        } else {
          // rows >= rb of the A operand read bytes that follow the chunk (still inside this
          // CTA's allocation) and only feed accumulator lanes >= r, which are never used
          const uint32_t abase = smem_u32(lring + lb * l_bytes);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int kk = k0 + i;
            const uint64_t adesc = smem_desc_sw128(abase + (kk >> 2) * p.rb * 128 + (kk & 3) * 32, 1024);
            const uint64_t bdesc = smem_desc_sw128(hbase + (kk >> 2) * N * 128 + (kk & 3) * 32, 1024);
            mma_ss(dcol, adesc, bdesc, idesc, (c > 0 || i > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&S.lempty[lb]));
        }
        tc_commit(smem_u32(&S.empty[s]));
      }
      tc_commit(smem_u32(&S.d_full));  // also reached on abort: tracks every MMA issued
      if (q == 0) PL_TL(6);
    }
  } else {
    // ---------------------------------------------------------------- dequant + epilogue
    const int dw = warp - 2;              // 0..7
    const int quarter = warp & 3;         // tensor-memory lane quarter of this warp
    const int g = dw >> 2;                // K half of each chunk
    const int row = quarter * 32 + lane;  // weight row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    if (threadIdx.x == 64) S.s_g = *p.s_g;  // weight inputs: never written by the preceding kernel
    if (lora) {
      // B rows of this tile, transposed into sBt[j][row] (bf16, zero past r and past d_o);
      // the tile's rows are one contiguous block of 128 r elements of B
      const int et0 = threadIdx.x - 64;
      const int64_t o0 = static_cast<int64_t>(tile) * kTileO;
      const int rows = static_cast<int>(p.d_o - o0 < kTileO ? p.d_o - o0 : kTileO);
      for (int i = et0; i < kTileO * kMaxR; i += kEpiThreads) sBt[i] = __float2bfloat16_rn(0.f);
      named_bar(1, kEpiThreads);
      const int n8 = rows * p.r / 8;  // 16-byte pieces (r % 8 == 0) or element-wise otherwise
      if ((p.r & 7) == 0) {
        const uint4* src = reinterpret_cast<const uint4*>(p.Blora + o0 * p.r);
        for (int i = et0; i < n8; i += kEpiThreads) {
          const uint4 v = src[i];
          const uint16_t* e8 = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int flat = 8 * i + q, rr = flat / p.r, j = flat % p.r;
            sBt[j * kTileO + rr] = __ushort_as_bfloat16(e8[q]);
          }
        }
      } else {
        for (int i = et0; i < rows * p.r; i += kEpiThreads) {
          const int rr = i / p.r, j = i % p.r;
          sBt[j * kTileO + rr] = p.Blora[(o0 + rr) * p.r + j];
        }
      }
    }
    for (int c = 0; c < nch; ++c) {
      const int s = c % stages, b = c % kAbuf;
      ok = wait_or_abort(smem_u32(&S.wfull[s]), (c / stages) & 1, abort_flag) &&
           (c < kAbuf || wait_or_abort(smem_u32(&S.a_empty[b]), ((c / kAbuf) - 1) & 1, abort_flag));
      if (!ok) break;
      if (c == 0 && threadIdx.x == 64) PL_TL(4);
      if (threadIdx.x == 64) PL_TLC(3, c);
      const uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
      const uint8_t* crow = st + row * 128;
      const uint2 sc8 = *reinterpret_cast<const uint2*>(st + kCodesBytes + h_bytes + row * 16 + g * 8);
      const uint32_t sc_words[2] = {sc8.x, sc8.y};
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = 4 * g + jj;  // 16-byte chunk of the row (32 codes, 2 scale blocks)
        const uint4 cw = *reinterpret_cast<const uint4*>(crow + ((j ^ (row & 7)) << 4));
        const uint32_t sbytes = (sc_words[jj >> 1] >> (16 * (jj & 1))) & 0xFFFFu;
        const uint32_t s2 = cvt_e4m3x2_to_f16x2(sbytes);
        const uint32_t sa = prmt(s2, s2, 0x1010u), sb = prmt(s2, s2, 0x3232u);
        uint32_t v[16];
        e2m1x8_to_f16x8(cw.x, v[0], v[1], v[2], v[3]);
        e2m1x8_to_f16x8(cw.y, v[4], v[5], v[6], v[7]);
        e2m1x8_to_f16x8(cw.z, v[8], v[9], v[10], v[11]);
        e2m1x8_to_f16x8(cw.w, v[12], v[13], v[14], v[15]);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = hmul2_u32(v[i], sa);
#pragma unroll
        for (int i = 8; i < 16; ++i) v[i] = hmul2_u32(v[i], sb);
        tmem_st16(tmem + lane_addr + kColA0 + 128u * b + j * 16, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&S.a_full[b]));
        mbar_arrive(smem_u32(&S.empty[s]));
      }
    }
    if (threadIdx.x == 64) PL_TL(5);
    // ---------------------------------------------------------------- epilogue, part 1
    ok = wait_or_abort(smem_u32(&S.d_full), 0, abort_flag) && ok;
    tc_fence_after();
    if (threadIdx.x == 64) PL_TL(7);
    pdl_wait();  // the row scales belong to this call's prologue
    const int et = threadIdx.x - 64;  // 0 .. 255
    if (et < N) S.rowscale[et] = et < p.M ? p.rowscale[et] : 0.f;
    go = named_bar_and(1, kEpiThreads, ok && !*abort_flag);  // one decision, publishes the row scales
    if (threadIdx.x == 64) PL_TL(8);
    if (go) {
      float* red = reinterpret_cast<float*>(smem);  // [N][128]    s_g c_n D1, reuses the stages
      float* tred = red + N * kTileO;                // [N][kTStride]  c_n Dt: this CTA's slice of t
      const float s_g = S.s_g;
      const int half = N / 2;  // 8, 16, 24 or 32 tokens per thread
      const int n0 = g * half;
      const bool trow = lora && quarter < 2;  // lanes 0..63 hold rows of t
      const uint32_t acc = tmem + lane_addr + kColAcc + static_cast<uint32_t>(n0);
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        if (cb * 8 < half) {  // 8 tokens at a time: the two halves of D1 (and of Dt)
          uint32_t da[8], db[8], ta[8], tb[8];
          tmem_ld8(acc + cb * 8, da);
          tmem_ld8(acc + 64 + cb * 8, db);
          if (trow) {
            tmem_ld8(acc + 128 + cb * 8, ta);
            tmem_ld8(acc + 192 + cb * 8, tb);
          }
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int n = n0 + cb * 8 + i;
            red[n * kTileO + row] = s_g * S.rowscale[n] * (__uint_as_float(da[i]) + __uint_as_float(db[i]));
            if (trow) tred[n * kTStride + row] = S.rowscale[n] * (__uint_as_float(ta[i]) + __uint_as_float(tb[i]));
          }
        }
      }
    }
  }
  if (threadIdx.x == 64) PL_TL(9);
  tc_fence_before();
  __syncthreads();
  // ------------------------------------------------------------------ epilogue, part 2
  // After a cluster barrier every CTA sums the t slices of all S CTAs (split order) into
  // lambda t, then the D1 partials of its row groups (4 rows each, groups
  // [32 split / S, 32 (split+1) / S)), adds B (lambda t) and writes y.
  cluster_sync();
  if (threadIdx.x == 0) PL_TL(10);
  if (threadIdx.x >= 64 && threadIdx.x < 64 + kEpiThreads && go) {
    const int et = threadIdx.x - 64;
    float* red = reinterpret_cast<float*>(smem);
    float* tred = red + N * kTileO;
    float* tful = tred + N * kTStride;  // [N][kTStride]: lambda t
    const uint32_t red_addr = smem_u32(red), tred_addr = smem_u32(tred);
    const int mt = static_cast<int>(p.M < N ? p.M : N);
    if (lora) {
      const int rq = (p.r + 3) / 4;  // groups of 4 adapter rows
      for (int e = et; e < mt * rq; e += kEpiThreads) {
        const int n = e / rq, jj = 4 * (e % rq);
        const uint32_t addr = tred_addr + static_cast<uint32_t>((n * kTStride + jj) * 4);
        float4 part[kMaxSplit];
#pragma unroll
        for (int sp = 0; sp < kMaxSplit; ++sp)
          if (sp < p.splits) part[sp] = ld_dsmem_f32x4(mapa_shared(addr, sp));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int sp = 0; sp < kMaxSplit; ++sp)
          if (sp < p.splits) {
            acc.x += part[sp].x;
            acc.y += part[sp].y;
            acc.z += part[sp].z;
            acc.w += part[sp].w;
          }
        // adapter rows past r (accumulator lanes that hold don't-care sums) become zeros
        reinterpret_cast<float4*>(tful + n * kTStride + jj)[0] =
            make_float4(jj < p.r ? p.lambda * acc.x : 0.f, jj + 1 < p.r ? p.lambda * acc.y : 0.f,
                        jj + 2 < p.r ? p.lambda * acc.z : 0.f, jj + 3 < p.r ? p.lambda * acc.w : 0.f);
      }
      named_bar(1, kEpiThreads);
    }
    // This CTA's share of the tile's rows: groups of 4 rows [g0, g1) of 32.  Thread et takes
    // row r0 + et % nrows and every ngrp-th token from et / nrows; it holds the row of B in
    // registers, sums the D1 partials of the S CTAs (split order) and adds B (lambda t).
    const int g0 = (split * (kTileO / 4)) / p.splits, g1 = ((split + 1) * (kTileO / 4)) / p.splits;
    const int r0 = 4 * g0, nrows = 4 * (g1 - g0);
    const int ngrp = kEpiThreads / nrows;  // >= 2: a share has at most 128 rows
    const int rl = et % nrows, tg = et / nrows;
    if (tg < ngrp) {
      const int rr = r0 + rl;
      const int64_t oo = static_cast<int64_t>(tile) * kTileO + rr;
      const int r4 = lora ? (p.r + 3) / 4 : 0;
      // y[n][rr] = (sum over splits of the D1 partials) + lora, stored as FP32 or BF16
      auto finish = [&](int n, float lora_sum) {
        float d = 0.f;
        if (p.splits == 1) {
          d = red[n * kTileO + rr];
        } else {
          const uint32_t addr = red_addr + static_cast<uint32_t>((n * kTileO + rr) * 4);
          float part[kMaxSplit];
#pragma unroll
          for (int sp = 0; sp < kMaxSplit; ++sp)
            if (sp < p.splits) part[sp] = ld_dsmem_f32(mapa_shared(addr, sp));
#pragma unroll
          for (int sp = 0; sp < kMaxSplit; ++sp)
            if (sp < p.splits) d += part[sp];
        }
        const float v = d + lora_sum;
        if (oo < p.d_o) {
          if (p.y_f32) static_cast<float*>(p.y)[n * p.d_o + oo] = v;
          else static_cast<__nv_bfloat16*>(p.y)[n * p.d_o + oo] = __float2bfloat16_rn(v);
        }
      };
      // four tokens per round (n + i ngrp): independent FMA chains in flight; B[rr][j] comes
      // from sBt[j][rr] (zeros past r), 32 neighbouring rows of one row of sBt per warp
      constexpr int kTok = 4;
      for (int n = tg; n < mt; n += kTok * ngrp) {
        float acc[kTok] = {0.f, 0.f, 0.f, 0.f};
        const float4* tn[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i) {
          const int ni = n + i * ngrp;
          tn[i] = reinterpret_cast<const float4*>(tful + (ni < mt ? ni : n) * kTStride);
        }
        for (int j4 = 0; j4 < r4; ++j4) {
          const float w0 = __bfloat162float(sBt[(4 * j4) * kTileO + rr]);
          const float w1 = __bfloat162float(sBt[(4 * j4 + 1) * kTileO + rr]);
          const float w2 = __bfloat162float(sBt[(4 * j4 + 2) * kTileO + rr]);
          const float w3 = __bfloat162float(sBt[(4 * j4 + 3) * kTileO + rr]);
#pragma unroll
          for (int i = 0; i < kTok; ++i) {
            const float4 t4 = tn[i][j4];  // the same address across the warp: a broadcast
            acc[i] = fmaf(w0, t4.x, fmaf(w1, t4.y, fmaf(w2, t4.z, fmaf(w3, t4.w, acc[i]))));
          }
        }
#pragma unroll
        for (int i = 0; i < kTok; ++i)
          if (n + i * ngrp < mt) finish(n + i * ngrp, acc[i]);
      }
    }
  }
  if (threadIdx.x == 64) PL_TL(11);
  cluster_sync();  // peers keep their shared memory until every reader is done
  if (threadIdx.x == 0) PL_TL(12);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
    if (lane == 0) PL_TL(13);
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

struct Plan {
  int N, rb, tiles, kc, splits, stages, la;
  uint32_t stage_bytes;
  size_t smem, act_smem;
};

uint32_t stage_bytes_for(int N) { return kCodesBytes + kScaleBytes + static_cast<uint32_t>(N) * 512u; }

// Shared memory: `stages` stages, the ring of `la` A chunks (rb rows x 512 B each), the
// B rows of the tile, the control block and 1 KB of alignment slack.  The ring has a
// third slot when that costs no weight stage.  The epilogue reuses the stage region for
// its partials ([N][128] + 2 x [N][68] FP32 < 1.1 KB x N), which two stages always cover.
void stage_plan(int N, int rb, int& stages, int& la, uint32_t& sb, size_t& total) {
  sb = stage_bytes_for(N);
  const size_t limit = 227 * 1024;
  auto fit = [&](int l, size_t& fixed) {
    fixed = 1024 + static_cast<size_t>(l) * rb * 512 + kTileO * kMaxR * 2 + sizeof(Smem);
    int st = static_cast<int>((limit - fixed) / sb);
    st = st > kMaxStages ? kMaxStages : st;
    return st < 2 ? 2 : st;
  };
  size_t fixed2, fixed3;
  const int st2 = fit(2, fixed2), st3 = fit(kMaxLa, fixed3);
  la = st3 >= st2 && fixed3 + static_cast<size_t>(st3) * sb <= limit ? kMaxLa : 2;
  stages = la == kMaxLa ? st3 : st2;
  total = (la == kMaxLa ? fixed3 : fixed2) + static_cast<size_t>(stages) * sb;
}

cudaError_t set_kernel_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(k_tc_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_act<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_act<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  });
  return err;
}

// Clusters of `cs` decode CTAs that can be resident at once (cached per N and A rows).
int max_active_clusters(int N, int rb, int cs) {
  static int cache[kMaxN / 16 + 1][kMaxR / 8 + 1][kMaxSplit + 1];
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  int& c = cache[N / 16][rb / 8][cs];
  if (c == 0) {
    int st, la;
    uint32_t sb;
    size_t total;
    stage_plan(N, rb, st, la, sb, total);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(cs * 64));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = total;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(cs);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_tc_decode, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = sm_count() / cs;
    }
    c = n < 1 ? 1 : n;
  }
  return c;
}

// Split count: minimise (waves) x (chunks per CTA + fixed per-CTA cost), the fixed
// cost counted as 1.5 chunks; ties go to fewer splits.
int choose_splits(int N, int rb, int tiles, int kc) {
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= kMaxSplit && s <= kc; ++s) {
    const int clusters = max_active_clusters(N, rb, s);
    const int waves = (tiles + clusters - 1) / clusters;
    const double cost = waves * (static_cast<double>((kc + s - 1) / s) + 1.5);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

Plan make_plan(int64_t M, int64_t d_i, int64_t d_o, int r) {
  Plan pl{};
  pl.N = static_cast<int>((M + 15) / 16 * 16);
  pl.rb = r > 0 ? (r + 7) / 8 * 8 : 8;
  pl.tiles = static_cast<int>((d_o + kTileO - 1) / kTileO);
  pl.kc = static_cast<int>(d_i / kChunkK);
  pl.splits = choose_splits(pl.N, pl.rb, pl.tiles, pl.kc);
  stage_plan(pl.N, pl.rb, pl.stages, pl.la, pl.stage_bytes, pl.smem);
  pl.act_smem = static_cast<size_t>(d_i) * 4;
  return pl;
}

struct TcWs {
  __half* hq;
  float* rowscale;
  __half* A16;
  size_t bytes;
};

TcWs carve(void* ws, int64_t M, int64_t d_i, int r) {
  TcWs w{};
  const uintptr_t b = reinterpret_cast<uintptr_t>(ws);
  size_t off = 0;
  w.hq = reinterpret_cast<__half*>(b + off);
  off += align_up(static_cast<size_t>(M) * d_i * 2, 256);
  w.rowscale = reinterpret_cast<float*>(b + off);
  off += align_up(static_cast<size_t>(M) * 4, 256);
  w.A16 = reinterpret_cast<__half*>(b + off);
  off += align_up(static_cast<size_t>(r) * d_i * 2, 256);
  w.bytes = off;
  return w;
}

}  // namespace

bool tc_supported(int64_t M, int64_t d_i, int64_t, int r) {
  // k_act holds a token row of at most 32768 elements in the registers of one CTA
  return M >= 1 && M <= kMaxN && d_i >= kChunkK && d_i % kChunkK == 0 && d_i <= 32768 && r >= 0 && r <= kMaxR;
}

size_t tc_workspace_bytes(int64_t M, int64_t d_i, int64_t, int r) { return carve(nullptr, M, d_i, r).bytes; }

cudaError_t launch_linear_tc(const LinearArgs& a, cudaStream_t stream) {
  cudaError_t e = set_kernel_attributes();
  if (e != cudaSuccess) return e;
  const Plan pl = make_plan(a.M, a.d_i, a.d_o, a.r);
  const TcWs w = carve(a.ws, a.M, a.d_i, a.r);
  TcMaps maps;
  bool ok = encode_2d(&maps.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, a.d_i / 2, a.d_o, 128, kTileO,
                      CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&maps.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.scales, a.d_i / 16, a.d_o, 16, kTileO,
                      CU_TENSOR_MAP_SWIZZLE_NONE) &&
            encode_2d(&maps.hq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.hq, a.d_i, a.M, 64, pl.N,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok && a.r > 0)
    ok = encode_2d(&maps.alora, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.A16, a.d_i, a.r, 64, pl.rb,
                   CU_TENSOR_MAP_SWIZZLE_128B);
  else
    maps.alora = maps.hq;  // unused
  if (!ok) return cudaErrorInvalidValue;

  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = static_cast<unsigned>(pl.splits);
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;

  e = launch_act_prologue(a, w.hq, w.rowscale, w.A16, nullptr, 0, stream);
  if (e != cudaSuccess) return e;

  TcParams p{};
  p.M = a.M;
  p.d_i = a.d_i;
  p.d_o = a.d_o;
  p.N = pl.N;
  p.r = a.r;
  p.rb = pl.rb;
  p.tiles = pl.tiles;
  p.splits = pl.splits;
  p.kc = pl.kc;
  p.stages = pl.stages;
  p.la = pl.la;
  p.stage_bytes = pl.stage_bytes;
  p.lambda = a.lambda;
  p.s_g = a.s_g;
  p.rowscale = w.rowscale;
  p.Blora = static_cast<const __nv_bfloat16*>(a.B);
  p.y = a.y;
  p.y_f32 = a.y_f32 ? 1 : 0;

  cudaLaunchConfig_t c2{};
  c2.gridDim = dim3(static_cast<unsigned>(pl.tiles * pl.splits));
  c2.blockDim = dim3(kThreads);
  c2.dynamicSmemBytes = pl.smem;
  c2.stream = stream;
  c2.attrs = attrs;
  c2.numAttrs = 2;
  return cudaLaunchKernelEx(&c2, k_tc_decode, maps, p);
}

cudaError_t launch_act_prologue(const LinearArgs& a, __half* hq, float* rowscale, __half* A16, float* zero,
                                int64_t n_zero, cudaStream_t stream) {
  cudaError_t e = set_kernel_attributes();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const int64_t a_slots = static_cast<int64_t>(a.r) * a.d_i / 8 + n_zero / 4;
  int nconv = static_cast<int>((a_slots + kActThreads * 4 - 1) / (kActThreads * 4));
  nconv = a_slots > 0 ? (nconv < 1 ? 1 : (nconv > 64 ? 64 : nconv)) : 0;
  // row CTAs, at most two per SM (each holds w_norm + z): a group of wpr warps per row,
  // wpr the power of two that gives each thread at most kActPieces pieces of 16 bytes
  const int64_t nv8 = a.d_i / 8;
  int wpr = 1;
  while (wpr < kActWarps && nv8 > kActPieces * 32 * wpr) wpr *= 2;
  if (nv8 > static_cast<int64_t>(kActPieces) * 32 * wpr) return cudaErrorInvalidValue;  // d_i > 32768
  const int rows_cta = kActWarps / wpr;
  const int64_t want = (a.M + rows_cta - 1) / rows_cta;
  const int n_row_ctas = static_cast<int>(want < 2 * sm_count() ? want : 2 * sm_count());
  cudaLaunchConfig_t c{};
  c.gridDim = dim3(static_cast<unsigned>(n_row_ctas + nconv));
  c.blockDim = dim3(kActThreads);
  c.dynamicSmemBytes = static_cast<size_t>(a.d_i) * 4;
  c.stream = stream;
  c.attrs = attr;
  c.numAttrs = 1;
  auto* kern = (a.z != nullptr && a.z_ld != 0) ? k_act<true> : k_act<false>;
  return cudaLaunchKernelEx(&c, kern, static_cast<const __nv_bfloat16*>(a.x), a.M, a.d_i, a.w_norm, a.z, a.z_ld,
                            a.eps, hq,
                            rowscale, static_cast<const __nv_bfloat16*>(a.A), a.r, A16, zero, n_zero, n_row_ctas,
                            wpr);
}

cudaError_t launch_wait_timeout_probe(cudaStream_t stream) {
  k_wait_timeout_probe<<<1, 32, 0, stream>>>(2ull * 1000 * 1000);  // 2 ms
  return cudaGetLastError();
}

#ifdef PL_TIMELINE
extern "C" int pl_debug_read_timeline(unsigned long long* main_out, unsigned long long* pro_out) {
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  if (cudaMemcpyFromSymbol(main_out, g_tl_main, sizeof(g_tl_main)) != cudaSuccess) return 2;
  if (cudaMemcpyFromSymbol(pro_out, g_tl_pro, sizeof(g_tl_pro)) != cudaSuccess) return 3;
  return 0;
}

extern "C" int pl_debug_read_timeline_chunks(unsigned long long* out) {
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  return cudaMemcpyFromSymbol(out, g_tl_chunk, sizeof(g_tl_chunk)) == cudaSuccess ? 0 : 2;
}
#endif

uint32_t tc_read_and_clear_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(zero));
  return v;
}

}  // namespace pl
