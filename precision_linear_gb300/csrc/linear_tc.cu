// tcgen05 tensor-core NVFP4 + LoRA linear (decode, M <= 64), sm_103a.
//
// Computes the forward map of "QeRL: When Quantized Weights Help Reinforcement
// Learning, and Where the Evidence Stops", section 2.1 (y = W_hat h + lambda B (A h))
// on the section 3.1 NVFP4 backbone (w_hat = s_g s_b q) with the section 5.1
// RMSNorm-AQN input h = u (.) (w_norm + z).
//
// Orientation ("swap AB"): the 128 weight rows of a tile are the MMA's M dimension,
// the (padded) tokens its N dimension, d_i its K dimension.  Per CTA and K chunk of
// 256:
//   * warp 0 (one lane) TMA-loads the chunk's packed codes (128 rows x 128 B,
//     128-byte swizzle), its E4M3 scales (128 x 16 B) and the activations
//     (N rows x 256 halves, 128-byte swizzle, canonical K-major layout);
//   * warps 2..9 dequantise: each thread owns one weight row and half the chunk,
//     turns 8 codes per 32-bit word into 4 f16x2 words with the hardware E2M1
//     conversion, multiplies by the block scale (q * s_b is exact in f16), and
//     stores them into tensor memory, where they are the MMA's A operand;
//   * warp 1 (one lane) issues 16 tcgen05.mma kind::f16 (K = 16 each) with A from
//     tensor memory and B from the swizzled shared tile, FP32 accumulator D1 in
//     tensor memory; the CTA holding the tile's first K split also issues the LoRA
//     up-projection D2 = B_lora (bf16, in tensor memory) x (lambda t)^T (bf16 tile).
// Epilogue (warps 2..9): tcgen05.ld the accumulators, y = s_g c_m D1 + D2.  When a
// tile's K range is split across CTAs, each writes its FP32 partial to the
// workspace and the last CTA to arrive (atomic counter, no waiting) sums the
// partials in split order -- deterministic.
//
// The activations are prepared by k_tc_prologue: per token row it forms the
// RMSNorm-AQN h in FP32, picks a power-of-two c_m that brings max|h| to [2^13, 2^14),
// stores h / c_m as f16 (11-bit significand; no overflow), and computes the LoRA
// down-projection t = A h in FP32, stored as bf16(lambda t).  Both kernels use
// programmatic dependent launch: the main kernel starts streaming weights while
// the prologue runs and waits (griddepcontrol.wait) only before it reads the
// prologue's outputs; the prologue waits before it overwrites the workspace.
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
#define PL_TL(slot) do { if (blockIdx.x < 1024) g_tl_main[blockIdx.x][slot] = globaltimer_ns(); } while (0)
#define PL_TLP(slot) do { const unsigned b_ = blockIdx.x + gridDim.x * blockIdx.y; \
                          if (b_ < 256) g_tl_pro[b_][slot] = globaltimer_ns(); } while (0)
#else
#define PL_TL(slot) do { } while (0)
#define PL_TLP(slot) do { } while (0)
#endif

namespace {

constexpr int kTileO = 128;
constexpr int kChunkK = 256;
constexpr int kCodesBytes = kTileO * kChunkK / 2;     // 16 KB
constexpr int kScaleBytes = kTileO * kChunkK / 16;    // 2 KB
constexpr int kThreads = 320;
constexpr int kDeqWarps = 8;
constexpr int kMaxStages = 12;
constexpr int kMaxSplit = 8;
constexpr int kMaxN = 64;
constexpr int kRpad = 64;  // tq row: 64 bf16 (128 B), zero beyond r
constexpr uint32_t kTmemCols = 512;
// tensor-memory column map
constexpr uint32_t kColA0 = 0;  // A buffer b at kColA0 + 128 b
constexpr uint32_t kColD1 = 256;
constexpr uint32_t kColD2 = 320;
constexpr uint32_t kColA2 = 384;

struct TcParams {
  int64_t M, d_i, d_o;
  int N, r, tiles, splits, kc, stages;
  uint32_t stage_bytes;
  float lambda;
  const float* s_g;
  const float* rowscale;
  const __nv_bfloat16* Blora;
  void* y;
  int y_f32;
};

struct TcMaps {
  CUtensorMap codes, scales, hq, tq;
};

// ------------------------------------------------------------------ small helpers
PL_DEVINL uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
PL_DEVINL uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// 8 E2M1 codes (one 32-bit word, code k in nibble k) -> 4 f16x2 (codes 2p, 2p+1 in word p).
PL_DEVINL void e2m1x8_to_f16x8(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2, uint32_t& o3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3) : "r"(w));
}
PL_DEVINL void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
         "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
         "r"(v[15]) : "memory");
}
PL_DEVINL void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                 "=r"(v[7]) : "r"(taddr) : "memory");
}
PL_DEVINL void named_bar(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
PL_DEVINL void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
PL_DEVINL uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
PL_DEVINL float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// Named barrier that also ANDs a predicate over the participating threads.
PL_DEVINL bool named_bar_and(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %3, 0;\n\t"
               "bar.red.and.pred p, %1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(r) : "r"(id), "r"(n), "r"(pred ? 1u : 0u) : "memory");
  return r != 0;
}

struct Smem {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t a_full[2], a_empty[2];
  uint64_t d_full, tq_full, a2_full, drain;
  uint32_t tmem_base;
  int abort_flag;
  float rowscale[kMaxN];
};

// Wait that also gives up when another role of the CTA has already given up.
PL_DEVINL bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(&g_tc_status, kStatusTimeout);
        return false;
      }
    }
  }
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

// ------------------------------------------------------------------ prologue
constexpr int kProThreads = 256;

// One CTA per (group of TM token rows, group of 8 adapter rows).  Pass 1 reads x,
// w_norm and z with 16-byte loads, keeps hz = x (.) (w + z) in shared memory and
// reduces sum(x^2) and max|hz| per row; then h = hz / rms, the power-of-two row
// scale c_m, the f16 activations h / c_m (written by the CTAs of adapter group 0)
// and the LoRA down-projection of this CTA's 8 adapter rows, A is read once per
// TM tokens.
template <int TM>
__global__ void __launch_bounds__(kProThreads) k_tc_prologue(
    const __nv_bfloat16* __restrict__ x, int64_t M, int64_t d_i, const float* __restrict__ w_norm,
    const float* __restrict__ z, float eps, const __nv_bfloat16* __restrict__ A, int r, float lambda,
    __half* __restrict__ hq, float* __restrict__ rowscale, __nv_bfloat16* __restrict__ tq) {
  extern __shared__ float4 hz4[];  // [TM][d_i / 4]
  __shared__ float red[kProThreads / 32][8 * TM];
  __shared__ float s_inv[TM], s_c[TM];
  if (threadIdx.x == 0) {
    PL_TLP(0);
    pdl_launch_dependents();
  }
  pdl_wait();  // the previous call may still read this workspace
  if (threadIdx.x == 0) PL_TLP(1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * TM;
  const int tm = static_cast<int>(M - m0 < TM ? M - m0 : TM);
  const int jb = blockIdx.y;
  const int64_t nslot = d_i / 8;  // 8 elements per slot
  const bool norm = w_norm != nullptr;
  float ss[TM], mx[TM];
#pragma unroll
  for (int t = 0; t < TM; ++t) ss[t] = mx[t] = 0.f;
  for (int64_t sl = threadIdx.x; sl < nslot; sl += kProThreads) {
    float sc[8];
    if (norm) {
      const float4 w0 = reinterpret_cast<const float4*>(w_norm)[2 * sl];
      const float4 w1 = reinterpret_cast<const float4*>(w_norm)[2 * sl + 1];
      sc[0] = w0.x; sc[1] = w0.y; sc[2] = w0.z; sc[3] = w0.w;
      sc[4] = w1.x; sc[5] = w1.y; sc[6] = w1.z; sc[7] = w1.w;
      if (z != nullptr) {
        const float4 z0 = reinterpret_cast<const float4*>(z)[2 * sl];
        const float4 z1 = reinterpret_cast<const float4*>(z)[2 * sl + 1];
        sc[0] += z0.x; sc[1] += z0.y; sc[2] += z0.z; sc[3] += z0.w;
        sc[4] += z1.x; sc[5] += z1.y; sc[6] += z1.z; sc[7] += z1.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i] = 1.0f;
    }
#pragma unroll
    for (int t = 0; t < TM; ++t) {
      if (t < tm) {
        const uint4 v = reinterpret_cast<const uint4*>(x + (m0 + t) * d_i)[sl];
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        float h[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a0 = bf16lo_to_f32(u[j]), a1 = bf16hi_to_f32(u[j]);
          ss[t] = fmaf(a0, a0, ss[t]);
          ss[t] = fmaf(a1, a1, ss[t]);
          h[2 * j] = a0 * sc[2 * j];
          h[2 * j + 1] = a1 * sc[2 * j + 1];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[t] = fmaxf(mx[t], fabsf(h[i]));
        hz4[t * (d_i / 4) + 2 * sl] = make_float4(h[0], h[1], h[2], h[3]);
        hz4[t * (d_i / 4) + 2 * sl + 1] = make_float4(h[4], h[5], h[6], h[7]);
      }
    }
  }
  if (threadIdx.x == 0) PL_TLP(2);
#pragma unroll
  for (int t = 0; t < TM; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss[t] += __shfl_xor_sync(0xFFFFFFFFu, ss[t], o);
      mx[t] = fmaxf(mx[t], __shfl_xor_sync(0xFFFFFFFFu, mx[t], o));
    }
    if (lane == 0) {
      red[warp][t] = ss[t];
      red[warp][TM + t] = mx[t];
    }
  }
  __syncthreads();
  if (threadIdx.x < TM) {
    const int t = threadIdx.x;
    float tot = 0.f, hm = 0.f;
#pragma unroll
    for (int w = 0; w < kProThreads / 32; ++w) {
      tot += red[w][t];
      hm = fmaxf(hm, red[w][TM + t]);
    }
    const float inv = norm ? 1.0f / sqrtf(tot / static_cast<float>(d_i) + eps) : 1.0f;
    const float hmax = inv * hm;
    int e = hmax > 0.f ? ilogbf(hmax) - 13 : 0;  // max |h| / c_m in [2^13, 2^14)
    e = e < -100 ? -100 : (e > 100 ? 100 : e);
    s_inv[t] = inv;
    s_c[t] = ldexpf(1.0f, e);
    if (jb == 0 && t < tm) rowscale[m0 + t] = ldexpf(1.0f, e);
  }
  __syncthreads();
  if (jb == 0) {
    for (int64_t sl = threadIdx.x; sl < nslot; sl += kProThreads) {
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        if (t < tm) {
          const float f = s_inv[t] / s_c[t];
          const float4 h0 = hz4[t * (d_i / 4) + 2 * sl], h1 = hz4[t * (d_i / 4) + 2 * sl + 1];
          const __half2 p0 = __floats2half2_rn(h0.x * f, h0.y * f), p1 = __floats2half2_rn(h0.z * f, h0.w * f);
          const __half2 p2 = __floats2half2_rn(h1.x * f, h1.y * f), p3 = __floats2half2_rn(h1.z * f, h1.w * f);
          uint4 o;
          o.x = *reinterpret_cast<const uint32_t*>(&p0);
          o.y = *reinterpret_cast<const uint32_t*>(&p1);
          o.z = *reinterpret_cast<const uint32_t*>(&p2);
          o.w = *reinterpret_cast<const uint32_t*>(&p3);
          reinterpret_cast<uint4*>(hq + (m0 + t) * d_i)[sl] = o;
        }
      }
    }
    for (int i = threadIdx.x; i < TM * kRpad; i += kProThreads) {
      const int t = i / kRpad, j = i % kRpad;
      if (t < tm && j >= r) tq[(m0 + t) * kRpad + j] = __float2bfloat16_rn(0.f);
    }
  }
  if (threadIdx.x == 0) PL_TLP(3);
  if (A == nullptr || r == 0) return;
  // LoRA down-projection t = A h for adapter rows j0 .. j0 + 7, FP32
  const int j0 = 8 * jb;
  float acc[8][TM];
#pragma unroll
  for (int q = 0; q < 8; ++q)
#pragma unroll
    for (int t = 0; t < TM; ++t) acc[q][t] = 0.f;
#pragma unroll 2
  for (int64_t sl = threadIdx.x; sl < nslot; sl += kProThreads) {
    uint4 av[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      av[q] = (j0 + q < r) ? reinterpret_cast<const uint4*>(A + static_cast<int64_t>(j0 + q) * d_i)[sl]
                           : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int t = 0; t < TM; ++t) {
      const float4 h0 = hz4[t * (d_i / 4) + 2 * sl], h1 = hz4[t * (d_i / 4) + 2 * sl + 1];
      const float hh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t u[4] = {av[q].x, av[q].y, av[q].z, av[q].w};
        float a = acc[q][t];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          a = fmaf(bf16lo_to_f32(u[j]), hh[2 * j], a);
          a = fmaf(bf16hi_to_f32(u[j]), hh[2 * j + 1], a);
        }
        acc[q][t] = a;
      }
    }
  }
  if (threadIdx.x == 0) PL_TLP(4);
  __syncthreads();  // red[] is reused below
#pragma unroll
  for (int q = 0; q < 8; ++q)
#pragma unroll
    for (int t = 0; t < TM; ++t) {
      float v = acc[q][t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      if (lane == 0) red[warp][q * TM + t] = v;
    }
  __syncthreads();
  if (threadIdx.x < 8 * TM) {
    const int q = threadIdx.x / TM, t = threadIdx.x % TM;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kProThreads / 32; ++w) v += red[w][q * TM + t];
    if (t < tm && j0 + q < r) tq[(m0 + t) * kRpad + j0 + q] = __float2bfloat16_rn(lambda * s_inv[t] * v);
  }
  if (threadIdx.x == 0) PL_TLP(5);
}

// ------------------------------------------------------------------ main kernel
__global__ void __launch_bounds__(kThreads, 1) k_tc_decode(const __grid_constant__ TcMaps maps,
                                                           const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int N = p.N, stages = p.stages;
  uint8_t* tq_smem = smem + static_cast<size_t>(stages) * p.stage_bytes;
  Smem& S = *reinterpret_cast<Smem*>(tq_smem + N * 128);
  volatile int* abort_flag = &S.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  const int c0 = static_cast<int>((static_cast<int64_t>(split) * p.kc) / p.splits);
  const int c1 = static_cast<int>((static_cast<int64_t>(split + 1) * p.kc) / p.splits);
  const int nch = c1 - c0;
  const bool has_lora = (split == 0) && p.r > 0;
  const uint32_t h_bytes = static_cast<uint32_t>(N) * 512u;
  bool go = false;  // epilogue threads: this CTA's accumulators are valid

  if (threadIdx.x == 0) {
    PL_TL(0);
    pdl_launch_dependents();
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&S.full[s]), 1);
      mbar_init(smem_u32(&S.empty[s]), kDeqWarps + 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&S.a_full[b]), kDeqWarps);
      mbar_init(smem_u32(&S.a_empty[b]), 1);
    }
    mbar_init(smem_u32(&S.d_full), 1);
    mbar_init(smem_u32(&S.tq_full), 1);
    mbar_init(smem_u32(&S.a2_full), 4);
    mbar_init(smem_u32(&S.drain), 1);
    S.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&maps.codes);
    tma_prefetch_desc(&maps.scales);
    tma_prefetch_desc(&maps.hq);
    tma_prefetch_desc(&maps.tq);
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
      const uint64_t pol_w = policy_evict_first();  // weights are streamed once
      const int pre = nch < stages ? nch : stages;
      const int32_t row0 = tile * kTileO;
      // weights of the first stages do not depend on the prologue: issue them now
      for (int c = 0; c < pre; ++c) {
        uint8_t* st = smem + static_cast<size_t>(c) * p.stage_bytes;
        const uint32_t fb = smem_u32(&S.full[c]);
        mbar_arrive_expect_tx(fb, kCodesBytes + kScaleBytes + h_bytes);
        const int kc = c0 + c;
        tma_load_2d_hint(smem_u32(st), &maps.codes, kc * (kChunkK / 2), row0, fb, pol_w);
        tma_load_2d_hint(smem_u32(st + kCodesBytes + h_bytes), &maps.scales, kc * (kChunkK / 16), row0, fb, pol_w);
      }
      PL_TL(2);
      pdl_wait();  // activations come from the prologue
      PL_TL(3);
      for (int c = 0; c < pre; ++c) {
        uint8_t* st = smem + static_cast<size_t>(c) * p.stage_bytes;
        const uint32_t fb = smem_u32(&S.full[c]);
        const int kc = c0 + c;
        for (int q = 0; q < 4; ++q)
          tma_load_2d(smem_u32(st + kCodesBytes + q * N * 128), &maps.hq, kc * kChunkK + 64 * q, 0, fb);
      }
      if (has_lora) {
        const uint32_t tb = smem_u32(&S.tq_full);
        mbar_arrive_expect_tx(tb, static_cast<uint32_t>(N) * 128u);
        tma_load_2d(smem_u32(tq_smem), &maps.tq, 0, 0, tb);
      }
      int c = pre;
      for (; c < nch; ++c) {
        const int s = c % stages;
        if (!wait_or_abort(smem_u32(&S.empty[s]), ((c / stages) - 1) & 1, abort_flag)) break;
        uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
        const uint32_t fb = smem_u32(&S.full[s]);
        mbar_arrive_expect_tx(fb, kCodesBytes + kScaleBytes + h_bytes);
        const int kc = c0 + c;
        tma_load_2d_hint(smem_u32(st), &maps.codes, kc * (kChunkK / 2), row0, fb, pol_w);
        tma_load_2d_hint(smem_u32(st + kCodesBytes + h_bytes), &maps.scales, kc * (kChunkK / 16), row0, fb, pol_w);
        for (int q = 0; q < 4; ++q)
          tma_load_2d(smem_u32(st + kCodesBytes + q * N * 128), &maps.hq, kc * kChunkK + 64 * q, 0, fb);
      }
      if (*abort_flag) {
        // drain: every issued stage's copies must land before this CTA exits
        const int first = c - stages > 0 ? c - stages : 0;
        for (int d = first; d < c; ++d) {
          const uint32_t fb = smem_u32(&S.full[d % stages]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(fb, (d / stages) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kTileO, N, 0);
      const uint32_t idesc_l = idesc_f16(kTileO, N, 1);
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        const int s = c % stages, b = c & 1;
        ok = wait_or_abort(smem_u32(&S.a_full[b]), (c >> 1) & 1, abort_flag) &&
             wait_or_abort(smem_u32(&S.full[s]), (c / stages) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t hbase = smem_u32(smem + static_cast<size_t>(s) * p.stage_bytes + kCodesBytes);
#pragma unroll
        for (int kk = 0; kk < kChunkK / 16; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(hbase + (kk >> 2) * N * 128 + (kk & 3) * 32, 1024);
          mma_ts(tmem + kColD1, tmem + (kColA0 + 128u * b) + kk * 8, bdesc, idesc, (c > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&S.empty[s]));
        tc_commit(smem_u32(&S.a_empty[b]));
      }
      if (ok && has_lora) {
        ok = wait_or_abort(smem_u32(&S.a2_full), 0, abort_flag) &&
             wait_or_abort(smem_u32(&S.tq_full), 0, abort_flag);
        if (ok) {
          tc_fence_after();
          const uint32_t tbase = smem_u32(tq_smem);
          const int ksteps = (p.r + 15) / 16;
          for (int kk = 0; kk < ksteps; ++kk)
            mma_ts(tmem + kColD2, tmem + kColA2 + kk * 8, smem_desc_sw128(tbase + kk * 32, 1024), idesc_l,
                   kk > 0 ? 1u : 0u);
        }
      }
      PL_TL(6);
      tc_commit(smem_u32(&S.d_full));  // also reached on abort: tracks every MMA issued
    }
  } else {
    // ---------------------------------------------------------------- dequant + epilogue
    const int dw = warp - 2;             // 0..7
    const int quarter = warp & 3;        // tensor-memory lane quarter of this warp
    const int g = dw >> 2;               // K half of each chunk
    const int row = quarter * 32 + lane; // weight row within the tile
    const int64_t o = static_cast<int64_t>(tile) * kTileO + row;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    if (has_lora && g == 0) {
      // A operand of the LoRA up-projection: this row of B_lora, bf16 pairs, zero past r
      const int rp2 = (p.r + 15) / 16 * 8;  // columns in use
      for (int cb = 0; cb < rp2; cb += 16) {
        uint32_t vv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = 2 * (cb + i);
          uint32_t lo = 0u, hi = 0u;
          if (o < p.d_o && j < p.r) lo = __bfloat16_as_ushort(p.Blora[o * p.r + j]);
          if (o < p.d_o && j + 1 < p.r) hi = __bfloat16_as_ushort(p.Blora[o * p.r + j + 1]);
          vv[i] = lo | (hi << 16);
        }
        tmem_st16(tmem + lane_addr + kColA2 + cb, vv);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.a2_full));
    }
    for (int c = 0; c < nch; ++c) {
      const int s = c % stages, b = c & 1;
      ok = wait_or_abort(smem_u32(&S.full[s]), (c / stages) & 1, abort_flag) &&
           (c < 2 || wait_or_abort(smem_u32(&S.a_empty[b]), ((c >> 1) - 1) & 1, abort_flag));
      if (!ok) break;
      if (c == 0 && threadIdx.x == 64) PL_TL(4);
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
        tmem_st16(tmem + lane_addr + (kColA0 + 128u * b) + j * 16, v);
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
    // ---------------------------------------------------------------- epilogue
    ok = wait_or_abort(smem_u32(&S.d_full), 0, abort_flag) && ok;
    if (threadIdx.x == 64) PL_TL(7);
    tc_fence_after();
    pdl_wait();  // the row scales belong to this call's prologue
    const int et = threadIdx.x - 64;  // 0 .. 255
    if (et < N) S.rowscale[et] = et < p.M ? p.rowscale[et] : 0.f;
    // one decision for all epilogue threads (also publishes the row scales)
    go = named_bar_and(1, kDeqWarps * 32, ok && !*abort_flag);
    if (threadIdx.x == 64) PL_TL(8);
    if (go) {
      const float s_g = *p.s_g;
      const int half = N / 2;
      const int n0 = g * half;
      float* red = reinterpret_cast<float*>(smem);  // [N][128] partial, reuses stage 0
      for (int cb = 0; cb < half; cb += 8) {
        uint32_t d1[8], d2[8];
        tmem_ld8(tmem + lane_addr + kColD1 + n0 + cb, d1);
        if (has_lora) tmem_ld8(tmem + lane_addr + kColD2 + n0 + cb, d2);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = n0 + cb + i;
          float v = s_g * S.rowscale[n] * __uint_as_float(d1[i]);
          if (has_lora) v += __uint_as_float(d2[i]);
          if (p.splits == 1) {
            if (n < p.M && o < p.d_o) {
              if (p.y_f32) static_cast<float*>(p.y)[n * p.d_o + o] = v;
              else static_cast<__nv_bfloat16*>(p.y)[n * p.d_o + o] = __float2bfloat16_rn(v);
            }
          } else {
            red[n * kTileO + row] = v;
          }
        }
      }
    }
  }
  if (threadIdx.x == 64) PL_TL(9);
  tc_fence_before();
  __syncthreads();
  if (p.splits > 1) {
    // K splits of one tile form a cluster: after every CTA has its FP32 partial in
    // shared memory, CTA `split` sums rows [r0, r1) of all partials over DSMEM in
    // split order (deterministic) and writes them.
    cluster_sync();
    if (threadIdx.x == 0) PL_TL(10);
    if (threadIdx.x >= 64 && go) {
      const int et = threadIdx.x - 64;
      const int r0 = (split * kTileO) / p.splits, r1 = ((split + 1) * kTileO) / p.splits;
      const int nr = r1 - r0;
      const int mt = static_cast<int>(p.M < N ? p.M : N);
      const uint32_t red_addr = smem_u32(smem);
      for (int e = et; e < nr * mt; e += kDeqWarps * 32) {
        const int n = e / nr, rr = r0 + e % nr;
        const int64_t oo = static_cast<int64_t>(tile) * kTileO + rr;
        const uint32_t off = static_cast<uint32_t>((n * kTileO + rr) * 4);
        float acc = 0.f;
        for (int sp = 0; sp < p.splits; ++sp) acc += ld_dsmem_f32(mapa_shared(red_addr + off, sp));
        if (oo < p.d_o) {
          if (p.y_f32) static_cast<float*>(p.y)[n * p.d_o + oo] = acc;
          else static_cast<__nv_bfloat16*>(p.y)[n * p.d_o + oo] = __float2bfloat16_rn(acc);
        }
      }
    }
    if (threadIdx.x == 64) PL_TL(11);
    cluster_sync();  // peers keep their shared memory until every reader is done
    if (threadIdx.x == 0) PL_TL(12);
  }
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
  int N, tiles, kc, splits, stages, tm;
  uint32_t stage_bytes;
  size_t smem, pro_smem;
};

uint32_t stage_bytes_for(int N) { return kCodesBytes + kScaleBytes + static_cast<uint32_t>(N) * 512u; }

int stages_for(uint32_t stage_bytes) {
  int st = static_cast<int>((200u * 1024u) / stage_bytes);
  return st > kMaxStages ? kMaxStages : (st < 2 ? 2 : st);
}

size_t smem_for(int N) {
  const uint32_t sb = stage_bytes_for(N);
  return 1024 + static_cast<size_t>(stages_for(sb)) * sb + static_cast<size_t>(N) * 128 + sizeof(Smem);
}

cudaError_t set_kernel_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(k_tc_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_tc_prologue<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_tc_prologue<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_tc_prologue<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  });
  return err;
}

// Clusters of `cs` decode CTAs that can be resident at once (cached per N class).
int max_active_clusters(int N, int cs) {
  static int cache[kMaxN / 16 + 1][kMaxSplit + 1];
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  int& c = cache[N / 16][cs];
  if (c == 0) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(cs * 64));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_for(N);
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
int choose_splits(int N, int tiles, int kc, bool query) {
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= kMaxSplit && s <= kc; ++s) {
    const int clusters = query ? max_active_clusters(N, s) : 1024;
    const int waves = (tiles + clusters - 1) / clusters;
    const double cost = waves * (static_cast<double>((kc + s - 1) / s) + 1.5);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

Plan make_plan(int64_t M, int64_t d_i, int64_t d_o, bool query) {
  Plan pl{};
  pl.N = static_cast<int>((M + 15) / 16 * 16);
  pl.tiles = static_cast<int>((d_o + kTileO - 1) / kTileO);
  pl.kc = static_cast<int>(d_i / kChunkK);
  pl.splits = choose_splits(pl.N, pl.tiles, pl.kc, query);
  pl.stage_bytes = stage_bytes_for(pl.N);
  pl.stages = stages_for(pl.stage_bytes);
  pl.smem = smem_for(pl.N);
  const int64_t tm = (160 * 1024) / (d_i * 4);
  pl.tm = tm >= 4 ? 4 : (tm >= 2 ? 2 : 1);
  pl.pro_smem = static_cast<size_t>(pl.tm) * d_i * 4;
  return pl;
}

struct TcWs {
  __half* hq;
  float* rowscale;
  __nv_bfloat16* tq;
  size_t bytes;
};

TcWs carve(void* ws, int64_t M, int64_t d_i) {
  TcWs w{};
  const uintptr_t b = reinterpret_cast<uintptr_t>(ws);
  size_t off = 0;
  w.hq = reinterpret_cast<__half*>(b + off);
  off += align_up(static_cast<size_t>(M) * d_i * 2, 256);
  w.rowscale = reinterpret_cast<float*>(b + off);
  off += align_up(static_cast<size_t>(M) * 4, 256);
  w.tq = reinterpret_cast<__nv_bfloat16*>(b + off);
  off += align_up(static_cast<size_t>(M) * kRpad * 2, 256);
  w.bytes = off;
  return w;
}

template <int TM>
cudaError_t launch_prologue(const LinearArgs& a, const Plan& pl, const TcWs& w, cudaStream_t stream,
                            cudaLaunchAttribute* pdl) {
  const int ny = a.r > 0 ? (a.r + 7) / 8 : 1;
  cudaLaunchConfig_t c{};
  c.gridDim = dim3(static_cast<unsigned>((a.M + TM - 1) / TM), static_cast<unsigned>(ny));
  c.blockDim = dim3(kProThreads);
  c.dynamicSmemBytes = pl.pro_smem;
  c.stream = stream;
  c.attrs = pdl;
  c.numAttrs = 1;
  return cudaLaunchKernelEx(&c, k_tc_prologue<TM>, static_cast<const __nv_bfloat16*>(a.x), a.M, a.d_i, a.w_norm,
                            a.z, a.eps, static_cast<const __nv_bfloat16*>(a.A), a.r, a.lambda, w.hq, w.rowscale,
                            w.tq);
}

}  // namespace

bool tc_supported(int64_t M, int64_t d_i, int64_t, int r) {
  return M >= 1 && M <= kMaxN && d_i >= kChunkK && d_i % kChunkK == 0 && r >= 0 && r <= kRpad;
}

size_t tc_workspace_bytes(int64_t M, int64_t d_i, int64_t, int) { return carve(nullptr, M, d_i).bytes; }

cudaError_t launch_linear_tc(const LinearArgs& a, cudaStream_t stream) {
  cudaError_t e = set_kernel_attributes();
  if (e != cudaSuccess) return e;
  const Plan pl = make_plan(a.M, a.d_i, a.d_o, true);
  const TcWs w = carve(a.ws, a.M, a.d_i);
  TcMaps maps;
  bool ok = encode_2d(&maps.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, a.d_i / 2, a.d_o, 128, kTileO,
                      CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&maps.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.scales, a.d_i / 16, a.d_o, 16, kTileO,
                      CU_TENSOR_MAP_SWIZZLE_NONE) &&
            encode_2d(&maps.hq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.hq, a.d_i, a.M, 64, pl.N,
                      CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&maps.tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w.tq, kRpad, a.M, 64, pl.N,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;

  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = static_cast<unsigned>(pl.splits);
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;

  e = pl.tm == 4 ? launch_prologue<4>(a, pl, w, stream, attrs)
                 : (pl.tm == 2 ? launch_prologue<2>(a, pl, w, stream, attrs) : launch_prologue<1>(a, pl, w, stream, attrs));
  if (e != cudaSuccess) return e;

  TcParams p{};
  p.M = a.M;
  p.d_i = a.d_i;
  p.d_o = a.d_o;
  p.N = pl.N;
  p.r = a.r;
  p.tiles = pl.tiles;
  p.splits = pl.splits;
  p.kc = pl.kc;
  p.stages = pl.stages;
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
  c2.numAttrs = pl.splits > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&c2, k_tc_decode, maps, p);
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
#endif

uint32_t tc_read_and_clear_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(zero));
  return v;
}

}  // namespace pl
