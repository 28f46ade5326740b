// tcgen05 tensor-core NVFP4 + LoRA linear (decode, M <= 64), sm_103a.
//
// Computes the forward map of "QeRL: When Quantized Weights Help Reinforcement
// Learning, and Where the Evidence Stops", section 2.1 (y = W_hat h + lambda B (A h))
// on the section 3.1 NVFP4 backbone (w_hat = s_g s_b q) with the section 5.1
// RMSNorm-AQN input h = u (.) (w_norm + z), for one projection or for a group of
// projections that read the same input (the projections behind one RMSNorm of a layer:
// q, k and v, or gate and up).
//
// Two kernels per call, chained by programmatic dependent launch:
//
// k_pro_rows (rows up to 8192 long; one CTA per input, group of R <= 4 token rows and group
//   of 8 adapter rows): u = x (.) (w_norm + z) in FP32 for the whole rows, per row the sum of x^2 and max
//   |u|, rs = 1 / sqrt(mean x^2 + eps) and the power of two c_m with max |h| / c_m in
//   [2^13, 2^14); the CTA of adapter group 0 writes the f16 activations h / c_m (11-bit
//   significand, no overflow) and c_m, every CTA t = rs A_p u (FP32, CUDA cores) for its
//   adapter rows.  The adapter's down-projection is thereby done once per call, not once per
//   weight tile, and no CTA waits on another.  Longer rows take k_pro_dec: clusters of 8 CTAs
//   over 1, 2 or 4 token rows, CTA c the c-th slice of K, one exchange of the row statistics
//   and of the adapter sums over distributed shared memory.
//
// k_tc_decode (a cluster of S CTAs per 128 weight rows of one projection; CTA s takes the
//   s-th slice of K in chunks of 256):
//   * warp 0 TMA-loads, per chunk, the packed codes (128 rows x 128 B, 128-byte
//     swizzle) and E4M3 scales (128 x 16 B) -- issued before the wait on the prologue,
//     they do not depend on it -- and the f16 activations (N rows x 256, 128-byte swizzle:
//     the canonical K-major layout);
//   * warps 2..9 dequantise: each thread owns one weight row and half the chunk, turns
//     8 codes per 32-bit word into 4 f16x2 words with the hardware E2M1 conversion,
//     multiplies by the block scale (q * s_b is exact in f16) and stores them into
//     tensor memory, where they are the MMA's A operand;
//   * two warps issue tcgen05.mma kind::f16 (K = 16 each; one thread issues one only
//     every few tens of ns, so each takes half of every chunk's K steps): weights (tensor
//     memory) x activations^T into two partial accumulators;
//   * epilogue (warps 2..9): every CTA adds its two partials and puts s_g c_m D1 in
//     shared memory; after a cluster barrier CTA s sums, over DSMEM and in split order
//     (deterministic), the partials of its share of the 128 rows, adds lambda B t on CUDA
//     cores (t from the prologue) and writes y.
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
__device__ unsigned long long g_tl_chunk[1024][6][32];  // per chunk: W issued, MMA ready, dequant end, dequant start, weights landed, issuer saw A
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
constexpr int kIssuers = 2;  // MMA-issuing warps: the two K halves of every chunk
// warps: weight producer, issuer 0, dequant/epilogue, issuer 1, activation producer
constexpr int kThreads = (2 + kDeqWarps + kIssuers) * 32;
constexpr int kIssuer1Warp = 2 + kDeqWarps;
constexpr int kHWarp = 3 + kDeqWarps;
constexpr int kEpiThreads = kDeqWarps * 32;
constexpr int kMaxStages = 10;   // weight stages (codes + scales of one chunk)
constexpr int kMaxHStages = 4;   // activation stages (the N token rows of one chunk)
constexpr uint32_t kWStage = kCodesBytes + kScaleBytes;  // 18 KB
constexpr int kMaxSplit = 8;
constexpr int kMaxN = 64;
constexpr int kMaxR = 64;        // adapter rank of one projection
constexpr int kMaxProj = 8;      // members (projections) of one launch
constexpr int kMaxSets = 8;      // distinct inputs (x, M, norm, noise) of one launch
constexpr int kMaxAdapt = 4;     // members reading one input
constexpr int kMaxRTot = 128;    // adapter rows over the members reading one input
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: kAbuf weight (MMA A operand) buffers of 128 columns from 0, then
// the two accumulators, N <= 64 columns each: D1 over the first and the second half of
// every chunk's K steps
constexpr int kAbuf = 3;
constexpr uint32_t kColA0 = 0;
constexpr uint32_t kColAcc = 384;  // issuer q accumulates at kColAcc + 64 q
static_assert(kAbuf * 128 <= kColAcc && kColAcc + kIssuers * kMaxN <= kTmemCols, "TMEM columns");
// Activation stages for N token rows: as many as 64 KB hold, 2 to kMaxHStages (the rows come
// from L2, written by the prologue).
__host__ __device__ constexpr int h_stages_for(int N) {
  return 65536 / (N * 512) < 2 ? 2 : (65536 / (N * 512) > kMaxHStages ? kMaxHStages : 65536 / (N * 512));
}

// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, bytes a multiple of 16).  Only a
// hint: L2 is the point of coherence, so a line fetched before its producer finished is
// refreshed by that producer's writes and later loads see them.
__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(ptr), "r"(bytes) : "memory");
}

// Orders this thread's generic shared-memory writes before later tensor-core (async-proxy) reads.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory operands of the adapter's up-projection (128-byte swizzled, K-major, bf16,
// zero past r): the B rows of the tile [128][64] and lambda t of the tokens [N][64], N the
// largest of the launch.
constexpr uint32_t kBaBytes = kTileO * 128;

// One projection of a group, as the main kernel sees it.
struct TcProjDev {
  int64_t d_o;
  const float* s_g;
  const __nv_bfloat16* B;  // [d_o][r] or null
  void* y;                 // [M][d_o]
  int r, toff, tile0;      // adapter rank, its first column of t, its first weight tile
  float lambda;
  int set;                 // the input it reads
};

// One input of a launch, as the main kernel sees it.
struct TcSetDev {
  int64_t M;
  int N;                   // M rounded up to 16: the MMA's N
  const float* rowscale;   // [M]: c_m
  const float* t;          // [M][t_ld]: t = rs A_p u of every member reading this input, at column toff_p
  int t_ld;
};

struct TcParams {
  int64_t d_i;
  int splits, kc, n_proj;
  uint32_t stage_region;   // shared-memory bytes for the weight ring; each CTA fits as many
                           // stages of its own N as the region holds (at most kMaxStages)
  uint32_t tq_region;      // bytes of the lambda t operand: the launch's largest N x 128
  int y_f32;
  TcProjDev proj[kMaxProj];
  TcSetDev set[kMaxSets];
};

struct TcMaps {
  CUtensorMap hq[kMaxSets];
  CUtensorMap codes[kMaxProj], scales[kMaxProj];
};

struct Smem {
  uint64_t wfull[kMaxStages], empty[kMaxStages], hfull[kMaxHStages], hempty[kMaxHStages];
  uint64_t a_full[kAbuf], a_empty[kAbuf];
  uint64_t d_full, tq_full;
  uint32_t tmem_base;
  int abort_flag;
  float s_g;
  float rowscale[kMaxN];
};

// One input of the prologue (cluster prologue: its clusters start at cl0; row prologue: its
// CTAs start at cta0).
struct ProSet {
  const __nv_bfloat16* x;
  int64_t M, d_i;
  const float* w_norm;  // [d_i] or null (no norm)
  const float* z;       // null, [d_i] (z_ld == 0) or rows z_ld apart
  int64_t z_ld;
  float eps;
  __half* hq;           // [M][d_i] (f16 mode)
  float* rowscale;      // [M]: c_m (f16 mode), s_x (FP8 mode)
  uint8_t* qx;          // [M][d_i] E4M3 codes (FP8 mode)
  float* t;             // [M][t_ld]
  int t_ld;
  int R;                // token rows per cluster (cluster prologue) or per CTA (row prologue)
  int C, cl0;           // cluster prologue: CTAs per cluster, first cluster
  int H, JG, cta0;      // row prologue: adapter groups, adapter rows per group (4 or 8), first CTA
  int n_proj, rtot;
  const __nv_bfloat16* A[kMaxAdapt];  // [r_p][d_i]
  int r[kMaxAdapt], toff[kMaxAdapt];
};
// Arguments of the prologue: its inputs, one cluster or CTA range each.
struct ProParams {
  int n_sets;
  ProSet set[kMaxSets];
};
constexpr int kProThreads = 256;
constexpr int kProWarps = kProThreads / 32;
constexpr int kProMaxR = 4;  // token rows per cluster or per CTA
constexpr int kProMaxC = 8;  // CTAs per cluster (cluster prologue)
constexpr int64_t kRowsMaxDi = 8192;  // the row prologue takes rows up to this long

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
                                                     uint8_t* __restrict__ qx, float* __restrict__ s_x,
                                                     const __grid_constant__ ActConv conv, int n_row_ctas, int wpr) {
  extern __shared__ float4 g4[];  // [d_i / 4]: w_norm + z of the whole row (1 without the norm)
  __shared__ float red_s[kActWarps], red_m[kActWarps];
  if (threadIdx.x == 0) {
    PL_TLP(0);
    pdl_launch_dependents();
  }
  pdl_wait();  // x may come from the preceding kernel, which may also still read the workspace
  if (threadIdx.x == 0) PL_TLP(1);
  if (static_cast<int>(blockIdx.x) >= n_row_ctas) {
    // the adapters to f16 (one segment per projection) and the counters to zero
    const int64_t stride = static_cast<int64_t>(gridDim.x - n_row_ctas) * kActThreads;
    for (int zr = 0; zr < conv.n_zero_ranges; ++zr)
      for (int64_t sl = (blockIdx.x - n_row_ctas) * kActThreads + threadIdx.x; sl < conv.n_zero[zr] / 4; sl += stride)
        reinterpret_cast<float4*>(conv.zero[zr])[sl] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sg = 0; sg < conv.n; ++sg) {
      const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(conv.A[sg]);
      __half* A16 = conv.A16[sg];
      const int64_t nslot = static_cast<int64_t>(conv.r[sg]) * d_i / 8;
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
    }
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
    if (qx != nullptr) {
      // the W8A8 form's activations, as the cluster prologue computes them: s_x = max |h| / 448,
      // q_x = E4M3(h / s_x) (round to nearest even, saturating, +0 for values rounding to zero)
      const float sx = hmax > 0.f ? __fdiv_rn(hmax, 448.0f) : 1.0f;
      if (gt == 0) s_x[m] = sx;
      uint2* qr = reinterpret_cast<uint2*>(qx + m * d_i);
#pragma unroll
      for (int i = 0; i < kActPieces; ++i) {
        const int64_t q = gt + static_cast<int64_t>(i) * gstride;
        if (q < nv8) {
          const uint4 v = xv[i];
          float g8[8];
          gpiece(q, g8);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
          uint32_t c[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t c4 = 0;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint32_t w = w4[2 * hh + j];
              const float h0 = bf16lo_to_f32(w) * g8[4 * hh + 2 * j] * inv;
              const float h1 = bf16hi_to_f32(w) * g8[4 * hh + 2 * j + 1] * inv;
              uint32_t c2 = cvt_e4m3x2(__fdiv_rn(h1, sx), __fdiv_rn(h0, sx));
              if ((c2 & 0x7Fu) == 0) c2 &= 0xFF00u;
              if ((c2 & 0x7F00u) == 0) c2 &= 0x00FFu;
              c4 |= c2 << (16 * j);
            }
            c[hh] = c4;
          }
          qr[q] = make_uint2(c[0], c[1]);
        }
      }
    }
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


// ------------------------------------------------------------------ cluster prologue
// A cluster of C CTAs per R token rows (rows m0 .. m0 + R - 1); CTA c of the cluster takes
// the pieces [c n8 / C, (c + 1) n8 / C) of 8 elements along K.  See the file comment.
// kFp8: instead of the f16 rows, the per-token FP8 quantisation of h for the W8A8 linear:
// s_x = fp32(max |h| / 448) (1 for a zero row), codes E4M3(fp32(h / s_x)), round to
// nearest even, saturating, +0 for values that round to zero.
template <bool kFp8>
// At most 64 registers a thread: four CTAs per SM, so that a batch's clusters fit in one wave.
__global__ void __launch_bounds__(kProThreads, 4) k_pro_dec(const __grid_constant__ ProParams pr) {
  // the input this cluster works on: the last one whose first cluster is <= this one
  int si = 0;
#pragma unroll
  for (int q = 1; q < kMaxSets; ++q)
    if (q < pr.n_sets && static_cast<int>(blockIdx.x) / pr.set[0].C >= pr.set[q].cl0) si = q;
  const ProSet& p = pr.set[si];
  extern __shared__ float4 pro_smem4[];
  float* u = reinterpret_cast<float*>(pro_smem4);  // [R][Lmax]: u = x (.) (w_norm + z), this CTA's slice
  __shared__ float red[kProWarps][kProMaxR][2];
  // read by the peers: per row the slice's sum of x^2 and max |u|, then the adapter sums [R][J]
  __shared__ __align__(16) float xch[2 * kProMaxR + kProMaxR * kMaxRTot];
  __shared__ float s_inv[kProMaxR], s_f[kProMaxR];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = p.C, R = p.R, J = p.rtot;
  uint32_t rank_u;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank_u));
  const int rank = static_cast<int>(rank_u);
  const int64_t m0 = static_cast<int64_t>(blockIdx.x / C - p.cl0) * R;
  const int64_t n8 = p.d_i / 8;
  const int64_t q0 = rank * n8 / C, q1 = (rank + 1) * n8 / C;
  const int L8 = static_cast<int>(q1 - q0);
  const int Lmax = static_cast<int>((n8 + C - 1) / C) * 8;
  const bool norm = p.w_norm != nullptr;
  const bool zshared = norm && p.z != nullptr && p.z_ld == 0, zrows = norm && p.z != nullptr && p.z_ld != 0;
  if (tid == 0) {
    PL_TLP(0);
    pdl_launch_dependents();
  }
  // While the preceding kernel finishes: bring this CTA's slices of the rows, the norm
  // scale, the noise and the adapters into L2 (one bulk prefetch per row slice).
  {
    const uint32_t xb = static_cast<uint32_t>(L8) * 16u, fb = static_cast<uint32_t>(L8) * 32u;
    if (tid < R && m0 + tid < p.M) {
      prefetch_l2(p.x + (m0 + tid) * p.d_i + q0 * 8, xb);
      if (zrows) prefetch_l2(p.z + (m0 + tid) * p.z_ld + q0 * 8, fb);
    } else if (tid == kProMaxR && norm) {
      prefetch_l2(p.w_norm + q0 * 8, fb);
    } else if (tid == kProMaxR + 1 && zshared) {
      prefetch_l2(p.z + q0 * 8, fb);
    } else if (tid >= 32 && tid - 32 < J) {
      const int jj = tid - 32;
      for (int pp = 0; pp < p.n_proj; ++pp)
        if (jj >= p.toff[pp] && jj < p.toff[pp] + p.r[pp])
          prefetch_l2(p.A[pp] + static_cast<int64_t>(jj - p.toff[pp]) * p.d_i + q0 * 8, xb);
    }
  }
  pdl_wait();  // x, w_norm and z may come from the preceding kernel, which may also still read the workspace
  if (tid == 0) PL_TLP(1);

  // 1. u of this CTA's rows and slice; per row the sum of x^2 and max |u|
  float ss[kProMaxR], mx[kProMaxR];
#pragma unroll
  for (int m = 0; m < kProMaxR; ++m) {
    ss[m] = 0.f;
    mx[m] = 0.f;
  }
  for (int qi = tid; qi < L8; qi += kProThreads) {
    const int64_t q = q0 + qi;
    float g[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = 1.f;
    if (norm) {
      const float4 a = reinterpret_cast<const float4*>(p.w_norm)[2 * q], b = reinterpret_cast<const float4*>(p.w_norm)[2 * q + 1];
      g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w; g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
      if (zshared) {
        const float4 za = reinterpret_cast<const float4*>(p.z)[2 * q], zb = reinterpret_cast<const float4*>(p.z)[2 * q + 1];
        g[0] += za.x; g[1] += za.y; g[2] += za.z; g[3] += za.w; g[4] += zb.x; g[5] += zb.y; g[6] += zb.z; g[7] += zb.w;
      }
    }
    uint4 xr[kProMaxR];  // the rows' pieces, all loads issued before any use
#pragma unroll
    for (int m = 0; m < kProMaxR; ++m)
      xr[m] = m < R && m0 + m < p.M ? __ldg(reinterpret_cast<const uint4*>(p.x + (m0 + m) * p.d_i) + q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int m = 0; m < kProMaxR; ++m) {
      if (m < R) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
        const int64_t row = m0 + m;
        if (row < p.M) {
          const uint4 xv = xr[m];
          float gz[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) gz[i] = g[i];
          if (zrows) {
            const float4* zr = reinterpret_cast<const float4*>(p.z + row * p.z_ld) + 2 * q;
            const float4 za = zr[0], zb = zr[1];
            gz[0] += za.x; gz[1] += za.y; gz[2] += za.z; gz[3] += za.w;
            gz[4] += zb.x; gz[5] += zb.y; gz[6] += zb.z; gz[7] += zb.w;
          }
          const uint32_t w4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float a0 = bf16lo_to_f32(w4[j]), a1 = bf16hi_to_f32(w4[j]);
            ss[m] = fmaf(a0, a0, fmaf(a1, a1, ss[m]));
            v[2 * j] = a0 * gz[2 * j];
            v[2 * j + 1] = a1 * gz[2 * j + 1];
            mx[m] = fmaxf(mx[m], fmaxf(fabsf(v[2 * j]), fabsf(v[2 * j + 1])));
          }
        }
        float4* ud = reinterpret_cast<float4*>(u + m * Lmax + qi * 8);
        ud[0] = make_float4(v[0], v[1], v[2], v[3]);
        ud[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kProMaxR; ++m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss[m] += __shfl_xor_sync(0xFFFFFFFFu, ss[m], o);
      mx[m] = fmaxf(mx[m], __shfl_xor_sync(0xFFFFFFFFu, mx[m], o));
    }
    if (lane == 0) {
      red[warp][m][0] = ss[m];
      red[warp][m][1] = mx[m];
    }
  }
  __syncthreads();
  if (tid < R) {
    float s = 0.f, x = 0.f;
#pragma unroll
    for (int w = 0; w < kProWarps; ++w) {
      s += red[w][tid][0];
      x = fmaxf(x, red[w][tid][1]);
    }
    xch[2 * tid] = s;
    xch[2 * tid + 1] = x;
  }

  // 2. this slice's adapter sums P[m][jj] = sum_k A[jj][k] u[m][k] over every projection of
  //    the group (adapter rows jj = toff_p + j): warp w takes rows 4w .. 4w + 3, then
  //    4w + 32 ..; the lanes split the pieces, a fixed shuffle tree adds them up
  for (int jb = 4 * warp; jb < J; jb += 4 * kProWarps) {
    const __nv_bfloat16* arow[4];
#pragma unroll
    for (int jr = 0; jr < 4; ++jr) {
      arow[jr] = nullptr;
      const int jj = jb + jr;
      for (int pp = 0; pp < p.n_proj; ++pp)
        if (jj >= p.toff[pp] && jj < p.toff[pp] + p.r[pp]) arow[jr] = p.A[pp] + (jj - p.toff[pp]) * p.d_i;
    }
    float acc[4][kProMaxR];
#pragma unroll
    for (int jr = 0; jr < 4; ++jr)
#pragma unroll
      for (int m = 0; m < kProMaxR; ++m) acc[jr][m] = 0.f;
    for (int qi = lane; qi < L8; qi += 32) {
      uint4 av[4];
#pragma unroll
      for (int jr = 0; jr < 4; ++jr)
        av[jr] = arow[jr] != nullptr ? __ldg(reinterpret_cast<const uint4*>(arow[jr]) + q0 + qi) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int m = 0; m < kProMaxR; ++m) {
        if (m < R) {
          const float4* us = reinterpret_cast<const float4*>(u + m * Lmax + qi * 8);
          const float4 ua = us[0], ub = us[1];
          const float uv[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
          for (int jr = 0; jr < 4; ++jr) {
            const uint32_t w4[4] = {av[jr].x, av[jr].y, av[jr].z, av[jr].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              acc[jr][m] = fmaf(bf16lo_to_f32(w4[j]), uv[2 * j], acc[jr][m]);
              acc[jr][m] = fmaf(bf16hi_to_f32(w4[j]), uv[2 * j + 1], acc[jr][m]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int jr = 0; jr < 4; ++jr)
#pragma unroll
      for (int m = 0; m < kProMaxR; ++m) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[jr][m] += __shfl_xor_sync(0xFFFFFFFFu, acc[jr][m], o);
        if (lane == 0 && m < R && jb + jr < J) xch[2 * kProMaxR + m * J + jb + jr] = acc[jr][m];
      }
  }
  if (tid == 0) PL_TLP(2);

  // 3. exchange: the row statistics of the whole row, then this CTA's f16 activations and
  //    its share of t (entries e = rank mod C of [R][J]), the slices added in slice order
  cluster_sync();
  if (tid < R) {
    float s = 0.f, x = 0.f, sv[kProMaxC], xv[kProMaxC];
#pragma unroll
    for (int c = 0; c < kProMaxC; ++c)  // all loads first: they are in flight together
      if (c < C) {
        sv[c] = ld_dsmem_f32(mapa_shared(smem_u32(&xch[2 * tid]), static_cast<uint32_t>(c)));
        xv[c] = ld_dsmem_f32(mapa_shared(smem_u32(&xch[2 * tid + 1]), static_cast<uint32_t>(c)));
      }
#pragma unroll
    for (int c = 0; c < kProMaxC; ++c)
      if (c < C) {
        s += sv[c];
        x = fmaxf(x, xv[c]);
      }
    const float inv = norm ? 1.0f / sqrtf(s / static_cast<float>(p.d_i) + p.eps) : 1.0f;
    const float hmax = inv * x;  // max |h|: rounding is monotone, so this is max |fl(u inv)|
    s_inv[tid] = inv;
    if (kFp8) {
      const float sx = hmax > 0.f ? __fdiv_rn(hmax, 448.0f) : 1.0f;
      s_f[tid] = sx;
      if (rank == 0 && m0 + tid < p.M) p.rowscale[m0 + tid] = sx;
    } else {
      int e = hmax > 0.f ? ilogbf(hmax) - 13 : 0;  // max |h| / c_m in [2^13, 2^14)
      e = e < -100 ? -100 : (e > 100 ? 100 : e);
      s_f[tid] = inv * ldexpf(1.0f, -e);
      if (rank == 0 && m0 + tid < p.M) p.rowscale[m0 + tid] = ldexpf(1.0f, e);
    }
  }
  __syncthreads();
  for (int qi = tid; qi < L8; qi += kProThreads) {
#pragma unroll
    for (int m = 0; m < kProMaxR; ++m) {
      const int64_t row = m0 + m;
      if (m < R && row < p.M) {
        const float4* us = reinterpret_cast<const float4*>(u + m * Lmax + qi * 8);
        const float4 a = us[0], b = us[1];
        const float f = s_f[m];
        if (kFp8) {
          const float inv = s_inv[m];
          const float hv[8] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv, b.x * inv, b.y * inv, b.z * inv, b.w * inv};
          uint32_t w[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t c4 = 0;
#pragma unroll
            for (int i = 0; i < 4; i += 2) {
              // two codes per conversion; a value that rounds to zero keeps no sign
              uint32_t c2 = cvt_e4m3x2(__fdiv_rn(hv[4 * hh + i + 1], f), __fdiv_rn(hv[4 * hh + i], f));
              if ((c2 & 0x7Fu) == 0) c2 &= 0xFF00u;
              if ((c2 & 0x7F00u) == 0) c2 &= 0x00FFu;
              c4 |= c2 << (8 * i);
            }
            w[hh] = c4;
          }
          reinterpret_cast<uint2*>(p.qx + row * p.d_i)[q0 + qi] = make_uint2(w[0], w[1]);
        } else {
          reinterpret_cast<uint4*>(p.hq + row * p.d_i)[q0 + qi] =
              make_uint4(f32x2_to_f16x2(a.x * f, a.y * f), f32x2_to_f16x2(a.z * f, a.w * f),
                         f32x2_to_f16x2(b.x * f, b.y * f), f32x2_to_f16x2(b.z * f, b.w * f));
        }
      }
    }
  }
  for (int e = rank + C * tid; e < R * J; e += C * kProThreads) {
    const int m = e / J, jj = e % J;
    if (m0 + m < p.M) {
      const uint32_t a = smem_u32(&xch[2 * kProMaxR + m * J + jj]);
      float s = 0.f, sv[kProMaxC];
#pragma unroll
      for (int c = 0; c < kProMaxC; ++c)  // all loads first: they are in flight together
        if (c < C) sv[c] = ld_dsmem_f32(mapa_shared(a, static_cast<uint32_t>(c)));
#pragma unroll
      for (int c = 0; c < kProMaxC; ++c)
        if (c < C) s += sv[c];
      p.t[(m0 + m) * p.t_ld + jj] = s_inv[m] * s;
    }
  }
  if (tid == 0) PL_TLP(3);
  cluster_sync();  // the peers read this CTA's shared memory until here
}

// ------------------------------------------------------------------ row prologue
// One CTA per (input, group of R token rows, group of JG adapter rows).  Every CTA of a row
// group reads its R rows whole: u = x (.) (w_norm + z) in FP32 into shared memory and, per
// row, the sum of x^2 and max |u| (a fixed shuffle tree, then the warps in order), so
// rs = 1 / sqrt(mean x^2 + eps) and the power of two c_m need no exchange between CTAs.  The
// CTA of adapter group 0 writes the f16 rows h / c_m (max |h| / c_m in [2^13, 2^14)) and c_m;
// every CTA writes t = rs A_p u for its adapter rows: warp w takes four adapter rows and one
// slice of K (JG / 4 row groups x 8 / (JG / 4) slices), the lanes split the slice in pieces
// of 8, a fixed shuffle tree and then the slices in order add them up (deterministic).
// kFp8: instead of the f16 rows, the per-token FP8 quantisation of h for the W8A8 linear:
// s_x = fp32(max |h| / 448) (1 for a zero row), codes E4M3(fp32(h / s_x)), round to
// nearest even, saturating, +0 for values that round to zero.
template <bool kFp8>
__global__ void __launch_bounds__(kProThreads, 1) k_pro_rows(const __grid_constant__ ProParams pr) {
  // the input of this CTA: the last one whose first CTA is <= this one
  int si = 0;
#pragma unroll
  for (int q = 1; q < kMaxSets; ++q)
    if (q < pr.n_sets && static_cast<int>(blockIdx.x) >= pr.set[q].cta0) si = q;
  const ProSet& p = pr.set[si];
  extern __shared__ float4 pro_smem4[];
  float* u = reinterpret_cast<float*>(pro_smem4);  // [R][d_i]
  __shared__ float red[kProWarps][kProMaxR][2];
  __shared__ float part[kProWarps][4][kProMaxR];   // adapter sums per K slice
  __shared__ float s_inv[kProMaxR], s_f[kProMaxR];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int local = static_cast<int>(blockIdx.x) - p.cta0;
  const int grp = local / p.H, hg = local - grp * p.H;  // row group, adapter group
  const int64_t m0 = static_cast<int64_t>(grp) * p.R;
  const int rows = static_cast<int>(p.M - m0 < p.R ? p.M - m0 : p.R);
  const int J = p.rtot, JG = p.JG;
  const int j0 = hg * JG, j1 = j0 + JG < J ? j0 + JG : J;
  const int64_t n8 = p.d_i / 8;
  const bool norm = p.w_norm != nullptr;
  const bool zshared = norm && p.z != nullptr && p.z_ld == 0, zrows = norm && p.z != nullptr && p.z_ld != 0;
  // the member and row of adapter row jj of this input (null past J)
  auto arow_of = [&](int jj) -> const __nv_bfloat16* {
    const __nv_bfloat16* a = nullptr;
    for (int pp = 0; pp < p.n_proj; ++pp)
      if (jj < j1 && jj >= p.toff[pp] && jj < p.toff[pp] + p.r[pp]) a = p.A[pp] + static_cast<int64_t>(jj - p.toff[pp]) * p.d_i;
    return a;
  };
  if (tid == 0) {
    PL_TLP(0);
    pdl_launch_dependents();
  }
  // While the preceding kernel finishes: bring this CTA's rows, its adapter rows, the norm
  // scale and the noise into L2.
  {
    const uint32_t rb = static_cast<uint32_t>(p.d_i) * 2u, fb = static_cast<uint32_t>(p.d_i) * 4u;
    if (tid < rows) {
      prefetch_l2(p.x + (m0 + tid) * p.d_i, rb);
      if (zrows) prefetch_l2(p.z + (m0 + tid) * p.z_ld, fb);
    } else if (tid == kProMaxR && norm) {
      prefetch_l2(p.w_norm, fb);
    } else if (tid == kProMaxR + 1 && zshared) {
      prefetch_l2(p.z, fb);
    } else if (tid >= 32 && tid - 32 < j1 - j0) {
      const __nv_bfloat16* a = arow_of(j0 + tid - 32);
      if (a != nullptr) prefetch_l2(a, rb);
    }
  }
  pdl_wait();  // x, w_norm and z may come from the preceding kernel, which may also still read the workspace
  if (tid == 0) PL_TLP(1);

  // 1. u of the rows; per row the sum of x^2 and max |u|
  float ss[kProMaxR], mx[kProMaxR];
#pragma unroll
  for (int m = 0; m < kProMaxR; ++m) {
    ss[m] = 0.f;
    mx[m] = 0.f;
  }
  for (int64_t q = tid; q < n8; q += kProThreads) {
    uint4 xr[kProMaxR];  // the rows' pieces, all loads issued before any use
#pragma unroll
    for (int m = 0; m < kProMaxR; ++m)
      xr[m] = m < rows ? __ldg(reinterpret_cast<const uint4*>(p.x + (m0 + m) * p.d_i) + q) : make_uint4(0u, 0u, 0u, 0u);
    float g[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = 1.f;
    if (norm) {
      const float4 a = reinterpret_cast<const float4*>(p.w_norm)[2 * q], b = reinterpret_cast<const float4*>(p.w_norm)[2 * q + 1];
      g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w; g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
      if (zshared) {
        const float4 za = reinterpret_cast<const float4*>(p.z)[2 * q], zb = reinterpret_cast<const float4*>(p.z)[2 * q + 1];
        g[0] += za.x; g[1] += za.y; g[2] += za.z; g[3] += za.w; g[4] += zb.x; g[5] += zb.y; g[6] += zb.z; g[7] += zb.w;
      }
    }
#pragma unroll
    for (int m = 0; m < kProMaxR; ++m) {
      if (m < rows) {
        float gz[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) gz[i] = g[i];
        if (zrows) {
          const float4* zr = reinterpret_cast<const float4*>(p.z + (m0 + m) * p.z_ld) + 2 * q;
          const float4 za = zr[0], zb = zr[1];
          gz[0] += za.x; gz[1] += za.y; gz[2] += za.z; gz[3] += za.w;
          gz[4] += zb.x; gz[5] += zb.y; gz[6] += zb.z; gz[7] += zb.w;
        }
        const uint32_t w4[4] = {xr[m].x, xr[m].y, xr[m].z, xr[m].w};
        float v[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a0 = bf16lo_to_f32(w4[j]), a1 = bf16hi_to_f32(w4[j]);
          ss[m] = fmaf(a0, a0, fmaf(a1, a1, ss[m]));
          v[2 * j] = a0 * gz[2 * j];
          v[2 * j + 1] = a1 * gz[2 * j + 1];
          mx[m] = fmaxf(mx[m], fmaxf(fabsf(v[2 * j]), fabsf(v[2 * j + 1])));
        }
        float4* ud = reinterpret_cast<float4*>(u + m * p.d_i + q * 8);
        ud[0] = make_float4(v[0], v[1], v[2], v[3]);
        ud[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kProMaxR; ++m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss[m] += __shfl_xor_sync(0xFFFFFFFFu, ss[m], o);
      mx[m] = fmaxf(mx[m], __shfl_xor_sync(0xFFFFFFFFu, mx[m], o));
    }
    if (lane == 0) {
      red[warp][m][0] = ss[m];
      red[warp][m][1] = mx[m];
    }
  }
  __syncthreads();
  if (tid < rows) {
    float s = 0.f, x = 0.f;
#pragma unroll
    for (int w = 0; w < kProWarps; ++w) {
      s += red[w][tid][0];
      x = fmaxf(x, red[w][tid][1]);
    }
    const float inv = norm ? 1.0f / sqrtf(s / static_cast<float>(p.d_i) + p.eps) : 1.0f;
    const float hmax = inv * x;  // max |h|: rounding is monotone, so this is max |fl(u inv)|
    s_inv[tid] = inv;
    if (kFp8) {
      const float sx = hmax > 0.f ? __fdiv_rn(hmax, 448.0f) : 1.0f;
      s_f[tid] = sx;
      if (hg == 0) p.rowscale[m0 + tid] = sx;
    } else {
      int e = hmax > 0.f ? ilogbf(hmax) - 13 : 0;  // max |h| / c_m in [2^13, 2^14)
      e = e < -100 ? -100 : (e > 100 ? 100 : e);
      s_f[tid] = inv * ldexpf(1.0f, -e);
      if (hg == 0) p.rowscale[m0 + tid] = ldexpf(1.0f, e);
    }
  }
  __syncthreads();
  if (tid == 0) PL_TLP(4);

  // 2. the activations (adapter group 0)
  if (hg == 0) {
    for (int64_t q = tid; q < n8; q += kProThreads) {
#pragma unroll
      for (int m = 0; m < kProMaxR; ++m) {
        if (m < rows) {
          const int64_t row = m0 + m;
          const float4* us = reinterpret_cast<const float4*>(u + m * p.d_i + q * 8);
          const float4 a = us[0], b = us[1];
          const float f = s_f[m];
          if (kFp8) {
            const float inv = s_inv[m];
            const float hv[8] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv, b.x * inv, b.y * inv, b.z * inv, b.w * inv};
            uint32_t w[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t c4 = 0;
#pragma unroll
              for (int i = 0; i < 4; i += 2) {
                // two codes per conversion; a value that rounds to zero keeps no sign
                uint32_t c2 = cvt_e4m3x2(__fdiv_rn(hv[4 * hh + i + 1], f), __fdiv_rn(hv[4 * hh + i], f));
                if ((c2 & 0x7Fu) == 0) c2 &= 0xFF00u;
                if ((c2 & 0x7F00u) == 0) c2 &= 0x00FFu;
                c4 |= c2 << (8 * i);
              }
              w[hh] = c4;
            }
            reinterpret_cast<uint2*>(p.qx + row * p.d_i)[q] = make_uint2(w[0], w[1]);
          } else {
            reinterpret_cast<uint4*>(p.hq + row * p.d_i)[q] =
                make_uint4(f32x2_to_f16x2(a.x * f, a.y * f), f32x2_to_f16x2(a.z * f, a.w * f),
                           f32x2_to_f16x2(b.x * f, b.y * f), f32x2_to_f16x2(b.z * f, b.w * f));
          }
        }
      }
    }
  }

  // 3. t = rs A_p u for adapter rows [j0, j1): warp w takes rows j0 + 4 (w mod nj) .. + 3 and
  //    K slice w / nj of ns
  const int nj = JG / 4, ns = kProWarps / nj;
  const int jb = j0 + 4 * (warp % nj), ks = warp / nj;
  const int64_t k0 = ks * n8 / ns, k1 = (ks + 1) * n8 / ns;
  const __nv_bfloat16* arow[4];
#pragma unroll
  for (int jr = 0; jr < 4; ++jr) arow[jr] = arow_of(jb + jr);
  float acc[4][kProMaxR];
#pragma unroll
  for (int jr = 0; jr < 4; ++jr)
#pragma unroll
    for (int m = 0; m < kProMaxR; ++m) acc[jr][m] = 0.f;
  const int qk0 = static_cast<int>(k0), qk1 = static_cast<int>(k1), di = static_cast<int>(p.d_i);  // d_i <= 8192 here
#pragma unroll 2
  for (int q = qk0 + lane; q < qk1; q += 32) {  // two iterations unrolled: their loads are in flight together
    float af[4][8];  // the adapter values of this piece, converted once for all token rows
#pragma unroll
    for (int jr = 0; jr < 4; ++jr) {
      const uint4 a = arow[jr] != nullptr ? __ldg(reinterpret_cast<const uint4*>(arow[jr]) + q) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w4[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        af[jr][2 * j] = bf16lo_to_f32(w4[j]);
        af[jr][2 * j + 1] = bf16hi_to_f32(w4[j]);
      }
    }
#pragma unroll
    for (int m = 0; m < kProMaxR; ++m) {
      if (m < rows) {
        const float4* us = reinterpret_cast<const float4*>(u + m * di + q * 8);
        const float4 ua = us[0], ub = us[1];
        const float uv[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
        for (int jr = 0; jr < 4; ++jr)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[jr][m] = fmaf(af[jr][e], uv[e], acc[jr][m]);
      }
    }
  }
#pragma unroll
  for (int jr = 0; jr < 4; ++jr)
#pragma unroll
    for (int m = 0; m < kProMaxR; ++m) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[jr][m] += __shfl_xor_sync(0xFFFFFFFFu, acc[jr][m], o);
      if (lane == 0) part[warp][jr][m] = acc[jr][m];
    }
  __syncthreads();
  // thread (jr, m, group) of each row group: the slices in order
  if (tid < JG * kProMaxR) {
    const int jl = tid / kProMaxR, m = tid % kProMaxR;  // adapter row j0 + jl, token row m
    const int jj = j0 + jl;
    if (jj < j1 && m < rows) {
      const int wg = jl / 4, jr = jl % 4;  // its warps: wg + nj s, s = 0 .. ns - 1
      float s = 0.f;
      for (int sl = 0; sl < ns; ++sl) s += part[wg + nj * sl][jr][m];
      p.t[(m0 + m) * p.t_ld + jj] = s_inv[m] * s;
    }
  }
  if (tid == 0) PL_TLP(3);
}

// ------------------------------------------------------------------ main kernel
__global__ void __launch_bounds__(kThreads, 1) k_tc_decode(const __grid_constant__ TcMaps maps,
                                                           const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sBa = smem + p.stage_region;  // [128][64] bf16: the B rows of the tile
  uint8_t* sTq = sBa + kBaBytes;          // [N][64] bf16: lambda t of the tokens
  Smem& S = *reinterpret_cast<Smem*>(sTq + p.tq_region);
  volatile int* abort_flag = &S.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gtile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  // the projection of this tile: the last one whose first tile is <= gtile
  int pj = 0;
#pragma unroll
  for (int q = 1; q < kMaxProj; ++q)
    if (q < p.n_proj && gtile >= p.proj[q].tile0) pj = q;
  const TcProjDev& P = p.proj[pj];
  const TcSetDev& Q = p.set[P.set];  // its input
  const int N = Q.N;
  // the stage region: weight stages of 18 KB from its start, then hst activation stages
  const uint32_t h_bytes = static_cast<uint32_t>(N) * 512u;
  const int hst = h_stages_for(N);
  const int wfit = static_cast<int>((p.stage_region - static_cast<uint32_t>(hst) * h_bytes) / kWStage);
  const int stages = wfit < kMaxStages ? wfit : kMaxStages;
  uint8_t* hreg = smem + static_cast<size_t>(stages) * kWStage;
  const CUtensorMap* map_codes = &maps.codes[pj];
  const CUtensorMap* map_scales = &maps.scales[pj];
  const CUtensorMap* map_hq = &maps.hq[P.set];
  const int tile = gtile - P.tile0;
  const int c0 = static_cast<int>((static_cast<int64_t>(split) * p.kc) / p.splits);
  const int c1 = static_cast<int>((static_cast<int64_t>(split + 1) * p.kc) / p.splits);
  const int nch = c1 - c0;
  const bool lora = P.r > 0;
  const bool lora_here = lora && split == 0;  // the split that adds the adapter's term
  // the up-projection accumulates into the weight buffer the next chunk would use, free
  // once the last chunk that used it has completed
  const int b_lora = nch % kAbuf;
  bool go = false;  // epilogue threads: this CTA's accumulators are valid

  const uint64_t pol_w = policy_evict_first();  // weights are streamed once
  const int pre = nch < stages ? nch : stages;
  const int32_t row0 = tile * kTileO;
  if (threadIdx.x == 0) {
    PL_TL(0);
    pdl_launch_dependents();
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&S.wfull[s]), 1);
      mbar_init(smem_u32(&S.empty[s]), kDeqWarps);  // released once dequantised
    }
    for (int s = 0; s < hst; ++s) {
      mbar_init(smem_u32(&S.hfull[s]), 1);
      mbar_init(smem_u32(&S.hempty[s]), kIssuers);  // released once its MMAs completed
    }
    for (int b = 0; b < kAbuf; ++b) {
      mbar_init(smem_u32(&S.a_full[b]), kDeqWarps);
      mbar_init(smem_u32(&S.a_empty[b]), kIssuers);
    }
    mbar_init(smem_u32(&S.d_full), kIssuers);
    mbar_init(smem_u32(&S.tq_full), kDeqWarps);
    S.abort_flag = 0;
    fence_mbar_init();
    // the first stages of weights do not depend on the prologue: issue them at once
    for (int c = 0; c < pre; ++c) {
      uint8_t* st = smem + static_cast<size_t>(c) * kWStage;
      const uint32_t wb = smem_u32(&S.wfull[c]);
      mbar_arrive_expect_tx(wb, kWStage);
      const int kc = c0 + c;
      PL_TLC(0, c);
      tma_load_2d_hint(smem_u32(st), map_codes, kc * (kChunkK / 2), row0, wb, pol_w);
      tma_load_2d_hint(smem_u32(st + kCodesBytes), map_scales, kc * (kChunkK / 16), row0, wb, pol_w);
    }
    tma_prefetch_desc(map_hq);
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
    // ---------------------------------------------------------------- weight producer
    // The weights never depend on the prologue: this thread streams them without waiting
    // for it, each stage as soon as the dequant warps have released it.
    if (lane == 0) {
      int c = pre;
      bool ok = true;
      while (ok && c < nch) {
        const int s = c % stages;
        ok = wait_or_abort(smem_u32(&S.empty[s]), ((c / stages) - 1) & 1, abort_flag);
        if (!ok) break;
        uint8_t* st = smem + static_cast<size_t>(s) * kWStage;
        const uint32_t wb = smem_u32(&S.wfull[s]);
        const int kc = c0 + c;
        PL_TLC(0, c);
        mbar_arrive_expect_tx(wb, kWStage);
        tma_load_2d_hint(smem_u32(st), map_codes, kc * (kChunkK / 2), row0, wb, pol_w);
        tma_load_2d_hint(smem_u32(st + kCodesBytes), map_scales, kc * (kChunkK / 16), row0, wb, pol_w);
        ++c;
      }
      if (*abort_flag)  // every issued copy must land before this CTA exits
        for (int d = (c - stages > 0 ? c - stages : 0); d < c; ++d) drain(smem_u32(&S.wfull[d % stages]), (d / stages) & 1);
    }
  } else if (warp == kHWarp) {
    // ---------------------------------------------------------------- activation producer
    if (lane == 0) {
      PL_TL(2);
      pdl_wait();  // the activations come from the prologue
      PL_TL(3);
      int c = 0;
      bool ok = true;
      while (ok && c < nch) {
        const int s = c % hst;
        if (c >= hst) ok = wait_or_abort(smem_u32(&S.hempty[s]), ((c / hst) - 1) & 1, abort_flag);
        if (!ok) break;
        uint8_t* st = hreg + static_cast<size_t>(s) * h_bytes;
        const uint32_t hb = smem_u32(&S.hfull[s]);
        mbar_arrive_expect_tx(hb, h_bytes);
        for (int q = 0; q < 4; ++q)
          tma_load_2d(smem_u32(st + q * N * 128), map_hq, (c0 + c) * kChunkK + 64 * q, 0, hb);
        ++c;
      }
      if (*abort_flag)
        for (int d = (c - hst > 0 ? c - hst : 0); d < c; ++d) drain(smem_u32(&S.hfull[d % hst]), (d / hst) & 1);
    }
  } else if (warp == 1 || warp == kIssuer1Warp) {
    // ---------------------------------------------------------------- MMA issuers
    // One thread can issue a tcgen05.mma only every few tens of ns, so two warps share the
    // work: issuer q takes K steps [8 q, 8 q + 8) of every chunk, weights (tensor memory) x
    // activations^T into its own partial accumulator; the epilogue adds the two.
    const int q = warp == 1 ? 0 : 1;
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kTileO, N, 0);
      const uint32_t dcol = tmem + kColAcc + 64u * static_cast<uint32_t>(q);
      const int k0 = 8 * q;
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        const int hs = c % hst, b = c % kAbuf;
        ok = wait_or_abort(smem_u32(&S.a_full[b]), (c / kAbuf) & 1, abort_flag);
        if (q == 0) PL_TLC(5, c);
        ok = ok && wait_or_abort(smem_u32(&S.hfull[hs]), (c / hst) & 1, abort_flag);
        if (!ok) break;
        if (q == 0) PL_TLC(1, c);
        tc_fence_after();
        const uint32_t hbase = smem_u32(hreg + static_cast<size_t>(hs) * h_bytes);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int kk = k0 + i;
          const uint64_t bdesc = smem_desc_sw128(hbase + (kk >> 2) * N * 128 + (kk & 3) * 32, 1024);
          mma_ts(dcol, tmem + kColA0 + 128u * b + kk * 8, bdesc, idesc, (c > 0 || i > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&S.a_empty[b]));
        tc_commit(smem_u32(&S.hempty[hs]));
      }
      if (ok && q == 0 && lora_here) {
        // lambda B t: K steps over the rank, B rows (as stored) x bf16(lambda t)^T, into a
        // weight buffer whose last chunk has completed (by both issuers)
        ok = wait_or_abort(smem_u32(&S.tq_full), 0, abort_flag) &&
             (nch < kAbuf || wait_or_abort(smem_u32(&S.a_empty[b_lora]), ((nch - kAbuf) / kAbuf) & 1, abort_flag));
        if (ok) {
          tc_fence_after();
          const uint32_t idesc_l = idesc_f16(kTileO, N, 1);
          const int ksteps = (P.r + 15) / 16;
          for (int kk = 0; kk < ksteps; ++kk)
            mma_ss(tmem + kColA0 + 128u * b_lora, smem_desc_sw128(smem_u32(sBa) + kk * 32, 1024),
                   smem_desc_sw128(smem_u32(sTq) + kk * 32, 1024), idesc_l, kk > 0 ? 1u : 0u);
        }
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
    if (threadIdx.x == 64) S.s_g = *P.s_g;  // weight inputs: never written by the preceding kernel
    if (lora_here) {
      // B rows of this tile into sBa (bf16, 128-byte swizzle, zero past r and past d_o):
      // thread et fills 16-byte pieces (row o, columns 8 j8 .. 8 j8 + 7)
      const int et0 = threadIdx.x - 64;
      const int64_t o0 = static_cast<int64_t>(tile) * kTileO;
      const int rows = static_cast<int>(P.d_o - o0 < kTileO ? P.d_o - o0 : kTileO);
      for (int i = et0; i < kTileO * 8; i += kEpiThreads) {
        const int o = i >> 3, j8 = i & 7;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (o < rows && 8 * j8 < P.r) {
          const __nv_bfloat16* src = P.B + (o0 + o) * P.r + 8 * j8;
          if ((P.r & 7) == 0) {
            v = *reinterpret_cast<const uint4*>(src);
          } else {
            uint16_t e[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) e[q] = 8 * j8 + q < P.r ? __bfloat16_as_ushort(src[q]) : 0;
            v = make_uint4(e[0] | (uint32_t(e[1]) << 16), e[2] | (uint32_t(e[3]) << 16),
                           e[4] | (uint32_t(e[5]) << 16), e[6] | (uint32_t(e[7]) << 16));
          }
        }
        *reinterpret_cast<uint4*>(sBa + o * 128 + ((j8 ^ (o & 7)) << 4)) = v;
      }
    }
    for (int c = 0; c < nch; ++c) {
      const int s = c % stages, b = c % kAbuf;
      ok = wait_or_abort(smem_u32(&S.wfull[s]), (c / stages) & 1, abort_flag);
      if (threadIdx.x == 64) PL_TLC(4, c);
      ok = ok && (c < kAbuf || wait_or_abort(smem_u32(&S.a_empty[b]), ((c / kAbuf) - 1) & 1, abort_flag));
      if (!ok) break;
      if (c == 0 && threadIdx.x == 64) PL_TL(4);
      if (threadIdx.x == 64) PL_TLC(3, c);
      const uint8_t* st = smem + static_cast<size_t>(s) * kWStage;
      const uint8_t* crow = st + row * 128;
      const uint2 sc8 = *reinterpret_cast<const uint2*>(st + kCodesBytes + row * 16 + g * 8);
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
      if (threadIdx.x == 64) PL_TLC(2, c);
      if (lane == 0) {
        mbar_arrive(smem_u32(&S.a_full[b]));
        mbar_arrive(smem_u32(&S.empty[s]));
      }
    }
    if (threadIdx.x == 64) PL_TL(5);
    // ---------------------------------------------------------------- lambda t operand
    pdl_wait();  // the row scales and t belong to this call's prologue
    const int et = threadIdx.x - 64;  // 0 .. 255
    if (lora_here) {
      // sTq[n][j] = bf16(lambda t[n][toff + j]), zero past r and past M, 16 bytes a thread
      const int mt = static_cast<int>(Q.M < N ? Q.M : N);
      for (int i = et; i < N * 8; i += kEpiThreads) {
        const int n = i >> 3, j8 = i & 7;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (n < mt && 8 * j8 < P.r) {
          const float* tr = Q.t + static_cast<int64_t>(n) * Q.t_ld + P.toff + 8 * j8;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = 8 * j8 + 2 * q < P.r ? P.lambda * tr[2 * q] : 0.f;
            const float hi = 8 * j8 + 2 * q + 1 < P.r ? P.lambda * tr[2 * q + 1] : 0.f;
            w[q] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
          }
        }
        *reinterpret_cast<uint4*>(sTq + n * 128 + ((j8 ^ (n & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();  // sBa and sTq are read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.tq_full));
    }
    // ---------------------------------------------------------------- epilogue, part 1
    ok = wait_or_abort(smem_u32(&S.d_full), 0, abort_flag) && ok;
    tc_fence_after();
    if (threadIdx.x == 64) PL_TL(7);
    if (et < N) S.rowscale[et] = et < Q.M ? Q.rowscale[et] : 0.f;
    go = named_bar_and(1, kEpiThreads, ok && !*abort_flag);  // one decision, publishes the row scales
    if (threadIdx.x == 64) PL_TL(8);
    if (go) {
      // y[n][o] = s_g c_n (D1 even + D1 odd)[o][n] + (lambda B t)[o][n]: stored at once
      // without a K split, else as this split's partial into red [N][128] (the stages)
      float* red = reinterpret_cast<float*>(smem);
      const float s_g = S.s_g;
      const int half = N / 2;  // 8, 16, 24 or 32 tokens per thread
      const int n0 = g * half;
      const uint32_t acc = tmem + lane_addr + kColAcc + static_cast<uint32_t>(n0);
      const uint32_t accl = tmem + lane_addr + kColA0 + 128u * b_lora + static_cast<uint32_t>(n0);
      const int64_t oo = static_cast<int64_t>(tile) * kTileO + row;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        if (cb * 8 < half) {  // 8 tokens at a time
          uint32_t da[8], db[8], dl[8];
          tmem_ld8(acc + cb * 8, da);
          tmem_ld8(acc + 64 + cb * 8, db);
          if (lora_here) tmem_ld8(accl + cb * 8, dl);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int n = n0 + cb * 8 + i;
            float v = s_g * S.rowscale[n] * (__uint_as_float(da[i]) + __uint_as_float(db[i]));
            if (lora_here) v += __uint_as_float(dl[i]);
            if (p.splits > 1) {
              red[n * kTileO + row] = v;
            } else if (n < Q.M && oo < P.d_o) {
              if (p.y_f32) static_cast<float*>(P.y)[n * P.d_o + oo] = v;
              else static_cast<__nv_bfloat16*>(P.y)[n * P.d_o + oo] = __float2bfloat16_rn(v);
            }
          }
        }
      }
    }
  }
  if (threadIdx.x == 64) PL_TL(9);
  tc_fence_before();
  __syncthreads();
  // ------------------------------------------------------------------ epilogue, part 2
  // With a K split: after a cluster barrier every CTA sums the partials of its row groups
  // (4 rows each, groups [32 split / S, 32 (split+1) / S)) over the S CTAs in split order
  // and writes y.
  if (p.splits > 1) cluster_sync();
  if (threadIdx.x == 0) PL_TL(10);
  if (p.splits > 1 && threadIdx.x >= 64 && threadIdx.x < 64 + kEpiThreads && go) {
    const int et = threadIdx.x - 64;
    const uint32_t red_addr = smem_u32(smem);
    const int mt = static_cast<int>(Q.M < N ? Q.M : N);
    const int g0 = (split * (kTileO / 4)) / p.splits, g1 = ((split + 1) * (kTileO / 4)) / p.splits;
    const int r0 = 4 * g0, nrows = 4 * (g1 - g0);
    const int ngrp = kEpiThreads / nrows;  // >= 2: a share has at most 128 rows
    const int rl = et % nrows, tg = et / nrows;
    if (tg < ngrp) {
      const int rr = r0 + rl;
      const int64_t oo = static_cast<int64_t>(tile) * kTileO + rr;
      for (int n = tg; n < mt; n += ngrp) {
        const uint32_t addr = red_addr + static_cast<uint32_t>((n * kTileO + rr) * 4);
        float part[kMaxSplit];
#pragma unroll
        for (int sp = 0; sp < kMaxSplit; ++sp)
          if (sp < p.splits) part[sp] = ld_dsmem_f32(mapa_shared(addr, sp));
        float v = 0.f;
#pragma unroll
        for (int sp = 0; sp < kMaxSplit; ++sp)
          if (sp < p.splits) v += part[sp];
        if (oo < P.d_o) {
          if (p.y_f32) static_cast<float*>(P.y)[n * P.d_o + oo] = v;
          else static_cast<__nv_bfloat16*>(P.y)[n * P.d_o + oo] = __float2bfloat16_rn(v);
        }
      }
    }
  }
  if (threadIdx.x == 64) PL_TL(11);
  if (p.splits > 1) cluster_sync();  // peers keep their shared memory until every reader is done
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

// Shared memory of the main kernel: the stage region (as many weight stages as fit, at
// most kMaxStages, then h_stages_for(N) activation stages), the B rows of the tile and
// lambda t (the up-projection's operands), the control block and 1 KB of alignment slack.
// With a K split the epilogue reuses the stage region for its partials ([N][128] FP32,
// 0.5 KB x N), which two weight stages always cover.  A member of a launch with fewer
// tokens than the largest lays its own stages out in the same region.  At most 165 KB, so
// that a prologue CTA (up to 57 KB) of the next call fits on the same SM: the next prologue
// then runs while this kernel's CTAs finish, and the next main kernel's CTAs do not wait for
// SMs that prologue CTAs hold (measured: 26.3 µs per decode-sweep batch against 27.1 µs with
// 227 KB and more weight stages; the 7B layer and the 32B stack 2-4 % faster too).
void stage_plan(int N, uint32_t& region, size_t& total) {
  const size_t limit = 165 * 1024;
  const size_t fixed = 1024 + kBaBytes + static_cast<size_t>(N) * 128 + sizeof(Smem);
  const size_t hpart = static_cast<size_t>(h_stages_for(N)) * static_cast<size_t>(N) * 512;
  int ws = static_cast<int>((limit - fixed - hpart) / kWStage);
  ws = ws > kMaxStages ? kMaxStages : (ws < 2 ? 2 : ws);
  region = static_cast<uint32_t>(static_cast<size_t>(ws) * kWStage + hpart);
  total = fixed + region;
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
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_pro_rows<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_pro_dec<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_pro_dec<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_pro_rows<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
  });
  return err;
}

// Clusters of `cs` main-kernel CTAs that can be resident at once (cached per N).
int max_active_clusters(int N, int cs) {
  static int cache[kMaxN / 16 + 1][kMaxSplit + 1];
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  int& c = cache[N / 16][cs];
  if (c == 0) {
    uint32_t region;
    size_t total;
    stage_plan(N, region, total);
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
int choose_splits(int N, int tiles, int kc) {
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= kMaxSplit && s <= kc; ++s) {
    const int clusters = max_active_clusters(N, s);
    const int waves = (tiles + clusters - 1) / clusters;
    const double cost = waves * (static_cast<double>((kc + s - 1) / s) + 1.5);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// Workspace of one launch: per input, the f16 rows [M][d_i], the row scales [M] and t [M][t_ld].
struct TcSetWs {
  __half* hq;
  float* rowscale;
  float* t;
  int t_ld;
};

size_t carve_sets(void* ws, int64_t d_i, const int64_t* Ms, const int* rtot, int n_sets, TcSetWs* out) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(ws);
  size_t off = 0;
  for (int s = 0; s < n_sets; ++s) {
    TcSetWs w{};
    w.hq = reinterpret_cast<__half*>(b + off);
    off += align_up(static_cast<size_t>(Ms[s]) * d_i * 2, 256);
    w.rowscale = reinterpret_cast<float*>(b + off);
    off += align_up(static_cast<size_t>(Ms[s]) * 4, 256);
    w.t_ld = rtot[s] > 0 ? (rtot[s] + 3) / 4 * 4 : 4;
    w.t = reinterpret_cast<float*>(b + off);
    off += align_up(static_cast<size_t>(Ms[s]) * w.t_ld * 4, 256);
    if (out != nullptr) out[s] = w;
  }
  return off;
}

// The row prologue's decomposition of one input: R token rows per CTA (their FP32 u, R d_i x 4
// bytes of shared memory, at most 160 KB), adapter groups of JG rows (fewer rows for long
// rows: with 8 (4 past d_i = 4096) each warp sums a quarter (an eighth) of K, a few pieces of
// 8 per lane).
void pro_plan(ProSet& q) {
  const int64_t fit = (160 * 1024) / (q.d_i * 4);
  int64_t r = q.M < kProMaxR ? q.M : kProMaxR;
  r = r < fit ? r : fit;
  q.R = r < 1 ? 1 : static_cast<int>(r);
  q.JG = q.d_i <= 4096 ? 8 : 4;
  q.H = q.rtot > 0 ? (q.rtot + q.JG - 1) / q.JG : 1;
}

// The cluster prologue (rows longer than kRowsMaxDi): input s takes clusters [cl0_s,
// cl0_s + ceil(M_s / R_s)) of kProMaxC CTAs, R_s = 1, 2 or 4 token rows each.
cudaError_t launch_pro_clusters(ProParams pr, bool fp8, cudaStream_t stream) {
  int clusters = 0;
  size_t pro_smem = 0;
  for (int s = 0; s < pr.n_sets; ++s) {
    ProSet& q = pr.set[s];
    q.R = q.M <= 16 ? 1 : (q.M <= 32 ? 2 : kProMaxR);
    q.C = kProMaxC;
    q.cl0 = clusters;
    clusters += static_cast<int>((q.M + q.R - 1) / q.R);
    const int64_t n8 = q.d_i / 8;
    const size_t need = static_cast<size_t>(q.R) * static_cast<size_t>((n8 + q.C - 1) / q.C) * 8 * 4;
    pro_smem = need > pro_smem ? need : pro_smem;
  }
  cudaLaunchAttribute pa[2];
  pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pa[0].val.programmaticStreamSerializationAllowed = 1;
  pa[1].id = cudaLaunchAttributeClusterDimension;
  pa[1].val.clusterDim.x = static_cast<unsigned>(kProMaxC);
  pa[1].val.clusterDim.y = 1;
  pa[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t c1{};
  c1.gridDim = dim3(static_cast<unsigned>(clusters * kProMaxC));
  c1.blockDim = dim3(kProThreads);
  c1.dynamicSmemBytes = pro_smem;
  c1.stream = stream;
  c1.attrs = pa;
  c1.numAttrs = 2;
  return fp8 ? cudaLaunchKernelEx(&c1, k_pro_dec<true>, pr) : cudaLaunchKernelEx(&c1, k_pro_dec<false>, pr);
}

// The row prologue: input s takes CTAs [cta0_s, cta0_s + ceil(M_s / R_s) H_s).  Rows longer than
// kRowsMaxDi take the cluster prologue (a CTA would hold too few rows of u), and so does the
// FP8 mode (measured: the W8A8 decode layer ran 17 % longer on the row prologue, whose CTAs each
// divide four whole rows).
cudaError_t launch_pro(ProParams pr, bool fp8, cudaStream_t stream) {
  if (fp8 || pr.set[0].d_i > kRowsMaxDi) return launch_pro_clusters(pr, fp8, stream);
  int ctas = 0;
  size_t pro_smem = 0;
  for (int s = 0; s < pr.n_sets; ++s) {
    ProSet& q = pr.set[s];
    pro_plan(q);
    q.cta0 = ctas;
    ctas += static_cast<int>((q.M + q.R - 1) / q.R) * q.H;
    const size_t need = static_cast<size_t>(q.R) * static_cast<size_t>(q.d_i) * 4;
    pro_smem = need > pro_smem ? need : pro_smem;
  }
  cudaLaunchAttribute pa[1];
  pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pa[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c1{};
  c1.gridDim = dim3(static_cast<unsigned>(ctas));
  c1.blockDim = dim3(kProThreads);
  c1.dynamicSmemBytes = pro_smem;
  c1.stream = stream;
  c1.attrs = pa;
  c1.numAttrs = 1;
  return fp8 ? cudaLaunchKernelEx(&c1, k_pro_rows<true>, pr) : cudaLaunchKernelEx(&c1, k_pro_rows<false>, pr);
}

}  // namespace

bool tc_supported(int64_t M, int64_t d_i, int64_t, int r) {
  return M >= 1 && M <= kMaxN && d_i >= kChunkK && d_i % kChunkK == 0 && d_i <= 32768 && r >= 0 && r <= kMaxR;
}

bool tc_batch_supported(int64_t d_i, const TcSet* sets, int n_sets, const TcProj* projs, int n_proj) {
  if (n_sets < 1 || n_sets > kMaxSets || n_proj < 1 || n_proj > kMaxProj) return false;
  int rtot[kMaxSets] = {0}, count[kMaxSets] = {0};
  for (int s = 0; s < n_sets; ++s)
    if (!tc_supported(sets[s].M, d_i, 1, 0)) return false;
  for (int i = 0; i < n_proj; ++i) {
    const int s = projs[i].set;
    if (s < 0 || s >= n_sets || projs[i].r < 0 || projs[i].r > kMaxR) return false;
    rtot[s] += projs[i].r;
    if (++count[s] > kMaxAdapt || rtot[s] > kMaxRTot) return false;
  }
  return true;
}

size_t tc_workspace_bytes(int64_t M, int64_t d_i, int64_t, int r) { return carve_sets(nullptr, d_i, &M, &r, 1, nullptr); }

size_t tc_batch_workspace_bytes(int64_t d_i, const TcSet* sets, int n_sets, const TcProj* projs, int n_proj) {
  int64_t Ms[kMaxSets];
  int rtot[kMaxSets] = {0};
  if (n_sets < 1 || n_sets > kMaxSets) return 0;
  for (int s = 0; s < n_sets; ++s) Ms[s] = sets[s].M;
  for (int i = 0; i < n_proj; ++i)
    if (projs[i].set >= 0 && projs[i].set < n_sets) rtot[projs[i].set] += projs[i].r;
  return carve_sets(nullptr, d_i, Ms, rtot, n_sets, nullptr);
}

cudaError_t launch_linear_tc_batch(int64_t d_i, float eps, const TcSet* sets, int n_sets, const TcProj* projs,
                                   int n_proj, bool y_f32, void* ws, cudaStream_t stream) {
  cudaError_t e = set_kernel_attributes();
  if (e != cudaSuccess) return e;
  int64_t Ms[kMaxSets];
  int rtot[kMaxSets] = {0}, toff[kMaxProj], tiles = 0, Nmax = 16;
  for (int s = 0; s < n_sets; ++s) {
    Ms[s] = sets[s].M;
    const int N = static_cast<int>((sets[s].M + 15) / 16 * 16);
    Nmax = N > Nmax ? N : Nmax;
  }
  for (int i = 0; i < n_proj; ++i) {
    toff[i] = rtot[projs[i].set];
    rtot[projs[i].set] += projs[i].r;
    tiles += static_cast<int>((projs[i].d_o + kTileO - 1) / kTileO);
  }
  TcSetWs w[kMaxSets];
  carve_sets(ws, d_i, Ms, rtot, n_sets, w);
  const int kc = static_cast<int>(d_i / kChunkK);
  const int splits = choose_splits(Nmax, tiles, kc);
  uint32_t stage_region;
  size_t smem;
  stage_plan(Nmax, stage_region, smem);  // the largest N sets the allocation
  const uint32_t tq_region = static_cast<uint32_t>(Nmax) * 128u;
  for (int s = 0; s < n_sets; ++s) {  // every member's own layout holds two weight stages
    const uint32_t N = static_cast<uint32_t>((sets[s].M + 15) / 16 * 16);
    const uint32_t hpart = static_cast<uint32_t>(h_stages_for(static_cast<int>(N))) * N * 512u;
    if (hpart + 2 * kWStage > stage_region) return cudaErrorInvalidValue;
  }

  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  bool ok = true;
  for (int s = 0; s < n_sets && ok; ++s)
    ok = encode_2d(&maps.hq[s], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w[s].hq, d_i, sets[s].M, 64,
                   static_cast<uint32_t>((sets[s].M + 15) / 16 * 16), CU_TENSOR_MAP_SWIZZLE_128B);
  // the main kernel's members in order of decreasing token count: the block scheduler starts
  // low tile indices first, so the members with the longest main loops get their SMs first
  int order[kMaxProj];
  for (int i = 0; i < n_proj; ++i) {
    int k = i;
    while (k > 0 && sets[projs[order[k - 1]].set].M < sets[projs[i].set].M) {
      order[k] = order[k - 1];
      --k;
    }
    order[k] = i;
  }
  for (int k = 0; k < n_proj && ok; ++k) {
    const int i = order[k];
    ok = encode_2d(&maps.codes[k], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, projs[i].codes, d_i / 2, projs[i].d_o, 128,
                   kTileO, CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_2d(&maps.scales[k], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, projs[i].scales, d_i / 16, projs[i].d_o, 16,
                   kTileO, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!ok) return cudaErrorInvalidValue;

  // prologue: per input, clusters of C CTAs over R token rows each, with the adapters of the
  // members that read it
  ProParams pr{};
  pr.n_sets = n_sets;
  for (int s = 0; s < n_sets; ++s) {
    ProSet& q = pr.set[s];
    q.x = static_cast<const __nv_bfloat16*>(sets[s].x);
    q.M = sets[s].M;
    q.d_i = d_i;
    q.w_norm = sets[s].w_norm;
    q.z = sets[s].w_norm != nullptr ? sets[s].z : nullptr;
    q.z_ld = sets[s].z_ld;
    q.eps = eps;
    q.hq = w[s].hq;
    q.rowscale = w[s].rowscale;
    q.t = w[s].t;
    q.t_ld = w[s].t_ld;
    q.rtot = rtot[s];
    for (int i = 0; i < n_proj; ++i)
      if (projs[i].set == s) {
        q.A[q.n_proj] = static_cast<const __nv_bfloat16*>(projs[i].A);
        q.r[q.n_proj] = projs[i].A != nullptr ? projs[i].r : 0;
        q.toff[q.n_proj] = toff[i];
        ++q.n_proj;
      }
  }
  e = launch_pro(pr, false, stream);
  if (e != cudaSuccess) return e;

  TcParams p{};
  p.d_i = d_i;
  p.splits = splits;
  p.kc = kc;
  p.stage_region = stage_region;
  p.tq_region = tq_region;
  p.n_proj = n_proj;
  p.y_f32 = y_f32 ? 1 : 0;
  for (int s = 0; s < n_sets; ++s)
    p.set[s] = TcSetDev{sets[s].M, static_cast<int>((sets[s].M + 15) / 16 * 16), w[s].rowscale, w[s].t, w[s].t_ld};
  for (int k = 0, t0 = 0; k < n_proj; ++k) {
    const int i = order[k];
    const bool lora = projs[i].r > 0 && projs[i].A != nullptr && projs[i].B != nullptr;
    p.proj[k].d_o = projs[i].d_o;
    p.proj[k].s_g = projs[i].s_g;
    p.proj[k].B = lora ? static_cast<const __nv_bfloat16*>(projs[i].B) : nullptr;
    p.proj[k].y = projs[i].y;
    p.proj[k].r = lora ? projs[i].r : 0;
    p.proj[k].toff = toff[i];
    p.proj[k].tile0 = t0;
    p.proj[k].lambda = projs[i].lambda;
    p.proj[k].set = projs[i].set;
    t0 += static_cast<int>((projs[i].d_o + kTileO - 1) / kTileO);
  }
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = static_cast<unsigned>(splits);
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t c2{};
  c2.gridDim = dim3(static_cast<unsigned>(tiles * splits));
  c2.blockDim = dim3(kThreads);
  c2.dynamicSmemBytes = smem;
  c2.stream = stream;
  c2.attrs = attrs;
  c2.numAttrs = 2;
  return cudaLaunchKernelEx(&c2, k_tc_decode, maps, p);
}

cudaError_t launch_pro_fp8(const void* x, int64_t M, int64_t d_i, const float* w_norm, const float* z, int64_t z_ld,
                           float eps, const void* A, int r, uint8_t* qx, float* s_x, float* t, int t_ld,
                           cudaStream_t stream) {
  cudaError_t e = set_kernel_attributes();
  if (e != cudaSuccess) return e;
  ProParams pr{};
  pr.n_sets = 1;
  ProSet& q = pr.set[0];
  q.x = static_cast<const __nv_bfloat16*>(x);
  q.M = M;
  q.d_i = d_i;
  q.w_norm = w_norm;
  q.z = w_norm != nullptr ? z : nullptr;
  q.z_ld = z_ld;
  q.eps = eps;
  q.qx = qx;
  q.rowscale = s_x;
  q.t = t;
  q.t_ld = t_ld;
  q.n_proj = 1;
  q.rtot = A != nullptr ? r : 0;
  q.A[0] = static_cast<const __nv_bfloat16*>(A);
  q.r[0] = q.rtot;
  q.toff[0] = 0;
  return launch_pro(pr, true, stream);
}

cudaError_t launch_linear_tc(const LinearArgs& a, cudaStream_t stream) {
  const TcSet set{a.x, a.M, a.w_norm, a.z, a.z_ld};
  TcProj pj{a.d_o, a.codes, a.scales, a.s_g, a.A, a.B, a.r, a.lambda, a.y, 0};
  return launch_linear_tc_batch(a.d_i, a.eps, &set, 1, &pj, 1, a.y_f32, a.ws, stream);
}

cudaError_t launch_act_prologue(const LinearArgs& a, __half* hq, float* rowscale, const ActConv& conv,
                                cudaStream_t stream, uint8_t* qx, float* s_x) {
  cudaError_t e = set_kernel_attributes();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int64_t a_slots = 0;
  for (int sg = 0; sg < conv.n; ++sg) a_slots += static_cast<int64_t>(conv.r[sg]) * a.d_i / 8;
  for (int zr = 0; zr < conv.n_zero_ranges; ++zr) a_slots += conv.n_zero[zr] / 4;
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
                            a.eps, hq, rowscale, qx, s_x, conv, n_row_ctas, wpr);
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
