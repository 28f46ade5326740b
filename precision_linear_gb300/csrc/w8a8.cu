// W8A8 rollout linear on FP8 E4M3 tensor cores (tcgen05 kind::f8f6f4), sm_103a.
//
// "QuRL: Low-Precision Reinforcement Learning for Efficient Reasoning" (reading notes,
// "method / overall framework"): before rollout the actor's weights are quantised with one
// scale per output channel and the activations with one scale per token, in INT8 or FP8,
// and rollout runs on 8-bit matrix products.  This is the FP8 form (on this part the FP8
// tensor rate far exceeds the INT8 one), with the frozen-backbone adapter of the QeRL
// forward map kept at full precision:
//   y[m, o] = s_x[m] s_w[o] sum_k q_x[m, k] q_w[o, k] + lambda sum_j B[o, j] t[m, j],
//   t = A h,  h = RMSNorm_AQN(x),  s_x = max_k |h[m, k]| / 448,  s_w = max_k |W[o, k]| / 448.
//
// k_w8_quant: one CTA per weight row: s_w = fp32(amax / 448) (1 for a zero row), codes
//   E4M3(fp32(w / s_w)), round to nearest even, saturating, +0 for values rounding to zero.
// The activations come from the cluster prologue of the tensor-core decode path in its FP8
// mode (linear_tc.cu): q_x, s_x and t = A h, FP32.
// k_w8_gemm (decode, M <= 64; a cluster of S CTAs per 128 weight rows x N tokens; CTA s takes the s-th slice
//   of K in chunks of 128):
//   * warp 0 TMA-loads per chunk the weight codes (128 rows x 128 B) and the activation codes
//     (N rows x 128 B), both with the 128-byte swizzle: they are the MMA operands as stored;
//   * warp 1 allocates tensor memory and one thread issues 4 MMAs per chunk (K = 32 each,
//     E4M3 x E4M3, FP32 accumulator, 128 x N); split 0 then adds the adapter as one more
//     K step of kind::f16 into the same accumulator: A' = B[o, :] / s_w[o] and
//     B' = lambda t[m, :] / s_x[m], both BF16, so that s_x s_w D carries lambda B t;
//   * warps 2..5 build A' and B' in shared memory while the main loop runs, then read the
//     accumulator, scale it by s_x s_w and write y (after summing the S partials of their
//     share of the rows over DSMEM, in split order, when K is split).
// k_w8_gemm_p (M > 64): the same arithmetic, persistent over tiles of 128 weight rows x 256
//   tokens with two accumulators (see its comment below).
// Every wait is bounded (200 ms); a wait that gives up sets the status word, the CTA drains
// its copies and MMAs, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace pl {

__device__ uint32_t g_w8_status = 0;

namespace {

constexpr int kTileO = 128;
constexpr int kChunk = 128;                 // K elements (bytes) of one stage
constexpr int kWBytes = kTileO * kChunk;    // 16 KB of weight codes per stage
constexpr int kMaxStages = 8;
constexpr int kThreads = 192;               // producer, MMA + TMEM, 4 epilogue warps
constexpr int kEpiThreads = 128;
constexpr int kMaxSplit = 8;
constexpr int kMaxR = 64;
constexpr int kLoraK = 64;                  // adapter K columns (zeros past r)

struct W8Params {
  int64_t M, d_i, d_o;
  int N, otiles, splits, kc, stages, n_tiles, mtiles;
  uint32_t stage_bytes, off_la, off_lb, off_ctrl;
  const float* s_w;   // [d_o]
  const float* s_x;   // [M]
  const float* t;     // [M][t_ld]: A h
  int t_ld;
  const __nv_bfloat16* B;  // [d_o][r] or null
  int r;
  float lambda;
  void* y;
  int y_f32;
};

struct W8Maps {
  CUtensorMap w, x;
};

struct W8Ctrl {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t lora_ready, d_full;
  uint32_t tmem_base;
  int abort_flag;
};

PL_DEVINL bool wait8(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return wait_or_abort_status(bar, parity, abort_flag, &g_w8_status);
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3, FP32 accumulator
PL_DEVINL void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accum) : "memory");
}

PL_DEVINL void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

PL_DEVINL uint32_t cluster_rank8() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// ------------------------------------------------------------------ weight quantiser
constexpr int kQThreads = 256;
__global__ void __launch_bounds__(kQThreads) k_w8_quant(const __nv_bfloat16* __restrict__ W, int64_t d_i,
                                                        uint8_t* __restrict__ codes, float* __restrict__ s_w) {
  __shared__ float red[kQThreads / 32];
  __shared__ float s_sh;
  const int64_t o = blockIdx.x;
  const uint4* wr = reinterpret_cast<const uint4*>(W + o * d_i);
  const int64_t n8 = d_i / 8;
  float mx = 0.f;
  for (int64_t i = threadIdx.x; i < n8; i += kQThreads) {
    const uint4 v = wr[i];
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fmaxf(fabsf(bf16lo_to_f32(w4[j])), fabsf(bf16hi_to_f32(w4[j]))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int w = 0; w < kQThreads / 32; ++w) a = fmaxf(a, red[w]);
    const float s = a > 0.f ? __fdiv_rn(a, 448.0f) : 1.0f;
    s_sh = s;
    s_w[o] = s;
  }
  __syncthreads();
  const float s = s_sh;
  uint2* cr = reinterpret_cast<uint2*>(codes + o * d_i);
  for (int64_t i = threadIdx.x; i < n8; i += kQThreads) {
    const uint4 v = wr[i];
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t c2 = cvt_e4m3x2(__fdiv_rn(bf16hi_to_f32(w4[j]), s), __fdiv_rn(bf16lo_to_f32(w4[j]), s));
      if ((c2 & 0x7Fu) == 0) c2 &= 0xFF00u;    // -0 -> +0
      if ((c2 & 0x7F00u) == 0) c2 &= 0x00FFu;
      c[j] = c2;
    }
    cr[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  }
}

// ------------------------------------------------------------------ GEMM
__global__ void __launch_bounds__(kThreads, 1) k_w8_gemm(const __grid_constant__ W8Maps maps,
                                                         const __grid_constant__ W8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  W8Ctrl& C = *reinterpret_cast<W8Ctrl*>(smem + p.off_ctrl);
  volatile int* abort_flag = &C.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, stages = p.stages, S = p.splits;
  const int split = static_cast<int>(cluster_rank8());
  const int tile = blockIdx.x / S;
  const int ot = tile % p.otiles, mt = tile / p.otiles;
  const int32_t row0 = ot * kTileO, tok0 = mt * N;
  const int c0 = static_cast<int>((static_cast<int64_t>(split) * p.kc) / S);
  const int c1 = static_cast<int>((static_cast<int64_t>(split + 1) * p.kc) / S);
  const int nch = c1 - c0;
  const bool lora = p.r > 0 && split == 0;  // the adapter term is added once
  const uint32_t x_bytes = static_cast<uint32_t>(N) * kChunk;
  const uint32_t tcols = N <= 32 ? 32u : (N <= 64 ? 64u : 128u);

  if (threadIdx.x == 0) {
    pdl_launch_dependents();
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&C.full[s]), 1);
      mbar_init(smem_u32(&C.empty[s]), 1);
    }
    mbar_init(smem_u32(&C.lora_ready), kEpiThreads / 32);
    mbar_init(smem_u32(&C.d_full), 1);
    C.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&C.tmem_base), tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;
  bool go = false;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const int pre = nch < stages ? nch : stages;
      // weights do not depend on the preceding kernel: the first stages go out at once
      for (int c = 0; c < pre; ++c) {
        const uint32_t fb = smem_u32(&C.full[c]);
        mbar_arrive_expect_tx(fb, kWBytes + x_bytes);
        tma_load_2d_hint(smem_u32(smem + c * p.stage_bytes), &maps.w, (c0 + c) * kChunk, row0, fb, pol_w);
      }
      pdl_wait();  // the activation codes come from the prologue
      for (int c = 0; c < pre; ++c)
        tma_load_2d(smem_u32(smem + c * p.stage_bytes + kWBytes), &maps.x, (c0 + c) * kChunk, tok0,
                    smem_u32(&C.full[c]));
      bool ok = true;
      int c = pre;
      for (; c < nch && ok; ++c) {
        const int s = c % stages;
        ok = wait8(smem_u32(&C.empty[s]), ((c / stages) - 1) & 1, abort_flag);
        if (!ok) break;
        const uint32_t fb = smem_u32(&C.full[s]);
        mbar_arrive_expect_tx(fb, kWBytes + x_bytes);
        tma_load_2d_hint(smem_u32(smem + s * p.stage_bytes), &maps.w, (c0 + c) * kChunk, row0, fb, pol_w);
        tma_load_2d(smem_u32(smem + s * p.stage_bytes + kWBytes), &maps.x, (c0 + c) * kChunk, tok0, fb);
      }
      if (*abort_flag)
        for (int d = (c - stages > 0 ? c - stages : 0); d < c; ++d) drain(smem_u32(&C.full[d % stages]), (d / stages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kTileO, N, 0);  // E4M3 x E4M3 shares the f16 field codes (0)
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        const int s = c % stages;
        ok = wait8(smem_u32(&C.full[s]), (c / stages) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t wa = smem_u32(smem + s * p.stage_bytes), xa = wa + kWBytes;
#pragma unroll
        for (int k = 0; k < kChunk / 32; ++k)
          mma_f8(tmem, smem_desc_sw128(wa + 32 * k, 1024), smem_desc_sw128(xa + 32 * k, 1024), idesc,
                 (c > 0 || k > 0) ? 1u : 0u);
        tc_commit(smem_u32(&C.empty[s]));
      }
      if (ok && lora) {
        ok = wait8(smem_u32(&C.lora_ready), 0, abort_flag);
        if (ok) {
          tc_fence_after();
          const uint32_t la = smem_u32(smem + p.off_la), lb = smem_u32(smem + p.off_lb);
          const uint32_t idesc_b = idesc_f16(kTileO, N, 1);
          const int ksteps = (p.r + 15) / 16;
#pragma unroll 1
          for (int k = 0; k < ksteps; ++k)
            mma_ss(tmem, smem_desc_sw128(la + 32 * k, 1024), smem_desc_sw128(lb + 32 * k, 1024), idesc_b,
                   (nch > 0 || k > 0) ? 1u : 0u);
        }
      }
      tc_commit(smem_u32(&C.d_full));  // also reached on abort: tracks every MMA issued
    }
  } else {
    // ---------------------------------------------------------------- adapter operands, epilogue
    const int et = threadIdx.x - 64;       // 0 .. 127
    const int quarter = warp & 3;          // tensor-memory lane quarter of this warp
    const int row = quarter * 32 + lane;   // weight row within the tile
    const int64_t o = static_cast<int64_t>(row0) + row;
    const float sw = o < p.d_o ? p.s_w[o] : 0.f;  // a weight input
    bool ok = true;
    if (lora) {
      // A' [128][64] = B[o, :] / s_w[o] (bf16, zeros past r and past d_o), one row per thread,
      // K-major 128-byte swizzled rows
      uint8_t* la = smem + p.off_la + row * 128;
#pragma unroll
      for (int j8 = 0; j8 < kLoraK / 8; ++j8) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int j = 8 * j8 + i;
          v[i] = (o < p.d_o && j < p.r) ? __bfloat162float(p.B[o * p.r + j]) / sw : 0.f;
        }
        *reinterpret_cast<uint4*>(la + ((j8 ^ (row & 7)) << 4)) =
            make_uint4(f32x2_to_bf16x2(v[0], v[1]), f32x2_to_bf16x2(v[2], v[3]), f32x2_to_bf16x2(v[4], v[5]),
                       f32x2_to_bf16x2(v[6], v[7]));
      }
      pdl_wait();  // t and s_x come from the prologue
      // B' [N][64] = lambda t[m, :] / s_x[m] (bf16, zeros past r and past M)
      for (int n = et; n < N; n += kEpiThreads) {
        const int64_t m = tok0 + n;
        const float f = m < p.M ? __fdiv_rn(p.lambda, p.s_x[m]) : 0.f;
        uint8_t* lb = smem + p.off_lb + n * 128;
#pragma unroll
        for (int j8 = 0; j8 < kLoraK / 8; ++j8) {
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int j = 8 * j8 + i;
            v[i] = (m < p.M && j < p.r) ? p.t[m * p.t_ld + j] * f : 0.f;
          }
          *reinterpret_cast<uint4*>(lb + ((j8 ^ (n & 7)) << 4)) =
              make_uint4(f32x2_to_bf16x2(v[0], v[1]), f32x2_to_bf16x2(v[2], v[3]), f32x2_to_bf16x2(v[4], v[5]),
                         f32x2_to_bf16x2(v[6], v[7]));
        }
      }
      fence_proxy_async_smem();  // read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.lora_ready));
    }
    ok = wait8(smem_u32(&C.d_full), 0, abort_flag) && ok;
    tc_fence_after();
    pdl_wait();  // s_x belongs to this call's prologue
    go = named_bar_and(1, kEpiThreads, ok && !*abort_flag);
    if (go) {
      // this thread's accumulator row, 16 tokens at a time: s_w s_x D (the adapter is in D)
      const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
      float* red = reinterpret_cast<float*>(smem);  // [N][128] partials of a split K (reuses the stages)
      for (int n0 = 0; n0 < N; n0 += 16) {
        uint32_t d[16];
        tmem_ld16(tmem + lane_addr + static_cast<uint32_t>(n0), d);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t m = tok0 + n0 + i;
          const float v = (m < p.M ? p.s_x[m] : 0.f) * sw * __uint_as_float(d[i]);
          if (S > 1) {
            red[(n0 + i) * kTileO + row] = v;
          } else if (m < p.M && o < p.d_o) {
            if (p.y_f32) static_cast<float*>(p.y)[m * p.d_o + o] = v;
            else static_cast<__nv_bfloat16*>(p.y)[m * p.d_o + o] = __float2bfloat16_rn(v);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (S > 1) {
    // the S partials of this CTA's share of the rows, in split order
    cluster_sync();
    if (threadIdx.x >= 64 && go) {
      const int et = threadIdx.x - 64;
      const int g0 = (split * (kTileO / 4)) / S, g1 = ((split + 1) * (kTileO / 4)) / S;
      const int r0 = 4 * g0, nrows = 4 * (g1 - g0);
      const uint32_t red_addr = smem_u32(smem);
      const int mt_rows = static_cast<int>(p.M - tok0 < N ? p.M - tok0 : N);
      for (int e = et; e < nrows * mt_rows; e += kEpiThreads) {
        const int rr = r0 + e % nrows, n = e / nrows;
        const int64_t oo = static_cast<int64_t>(row0) + rr;
        const uint32_t addr = red_addr + static_cast<uint32_t>((n * kTileO + rr) * 4);
        float part[kMaxSplit];
#pragma unroll
        for (int sp = 0; sp < kMaxSplit; ++sp)
          if (sp < S) part[sp] = ld_dsmem_f32(mapa_shared(addr, sp));
        float v = 0.f;
#pragma unroll
        for (int sp = 0; sp < kMaxSplit; ++sp)
          if (sp < S) v += part[sp];
        const int64_t m = tok0 + n;
        if (oo < p.d_o) {
          if (p.y_f32) static_cast<float*>(p.y)[m * p.d_o + oo] = v;
          else static_cast<__nv_bfloat16*>(p.y)[m * p.d_o + oo] = __float2bfloat16_rn(v);
        }
      }
    }
    cluster_sync();  // peers keep their shared memory until every reader is done
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

// ------------------------------------------------------------------ GEMM, large M
// k_w8_gemm_p: persistent, one CTA per SM over tiles of 128 weight rows x kPN tokens (the
// token tiles fastest, so that concurrent CTAs share their weight tile in L2 and the weights
// are read from DRAM about once; the activations, 1 byte per element, stay in L2); two
// accumulators of kPN columns, so that a tile's epilogue runs under the next tile's MMAs.
//   * warp 0 TMA-loads per chunk of 128 K the weight codes (16 KB) and the activation codes
//     (kPN rows, 32 KB) into a ring of kPStages stages;
//   * warp 1: one thread issues 4 MMAs per chunk (E4M3 x E4M3, K = 32, M = 128, N = kPN),
//     then the adapter's K steps (bf16 A' = B / s_w and B' = lambda t / s_x, as in
//     k_w8_gemm), and commits the accumulator;
//   * warps 2..5 write y = s_x s_w D of a finished tile, free its accumulator, then build the
//     next tile's adapter operands (the previous tile's adapter step has completed by then).
constexpr int kPN = 256;
constexpr int kPStages = 3;
constexpr uint32_t kPStageBytes = kWBytes + kPN * kChunk;  // 48 KB

struct W8PCtrl {
  uint64_t full[kPStages], empty[kPStages];
  uint64_t lora_ready, d_full[2], d_empty[2], mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(kThreads, 1) k_w8_gemm_p(const __grid_constant__ W8Maps maps,
                                                           const __grid_constant__ W8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  W8PCtrl& C = *reinterpret_cast<W8PCtrl*>(smem + p.off_ctrl);
  volatile int* abort_flag = &C.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool lora = p.r > 0;
  const int kc = p.kc;

  if (threadIdx.x == 0) {
    pdl_launch_dependents();
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(smem_u32(&C.full[s]), 1);
      mbar_init(smem_u32(&C.empty[s]), 1);
    }
    mbar_init(smem_u32(&C.lora_ready), kEpiThreads / 32);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&C.d_full[b]), 1);
      mbar_init(smem_u32(&C.d_empty[b]), kEpiThreads / 32);
    }
    mbar_init(smem_u32(&C.mma_done), 1);
    C.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&C.tmem_base), 2 * kPN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      pdl_wait();  // the activation codes come from the prologue
      bool ok = true;
      int64_t gs = 0;
      for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x) {
        const int32_t row0 = (tile / p.mtiles) * kTileO, tok0 = (tile % p.mtiles) * kPN;
        for (int c = 0; c < kc && ok; ++c, ++gs) {
          const int s = static_cast<int>(gs % kPStages);
          if (gs >= kPStages) ok = wait8(smem_u32(&C.empty[s]), static_cast<uint32_t>((gs / kPStages) - 1) & 1, abort_flag);
          if (!ok) break;
          const uint32_t fb = smem_u32(&C.full[s]);
          mbar_arrive_expect_tx(fb, kPStageBytes);
          tma_load_2d_hint(smem_u32(smem + s * kPStageBytes), &maps.w, c * kChunk, row0, fb, pol_w);
          tma_load_2d(smem_u32(smem + s * kPStageBytes + kWBytes), &maps.x, c * kChunk, tok0, fb);
        }
      }
      if (*abort_flag)
        for (int64_t d = gs - kPStages > 0 ? gs - kPStages : 0; d < gs; ++d)
          drain(smem_u32(&C.full[d % kPStages]), static_cast<uint32_t>(d / kPStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kTileO, kPN, 0);    // E4M3 x E4M3 shares the f16 field codes (0)
      const uint32_t idesc_b = idesc_f16(kTileO, kPN, 1);  // the adapter step: bf16
      const int ksteps = (p.r + 15) / 16;
      const uint32_t la = smem_u32(smem + p.off_la), lb = smem_u32(smem + p.off_lb);
      bool ok = true;
      int64_t gs = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x, ++it) {
        const int b = it & 1;
        if (it >= 2) ok = wait8(smem_u32(&C.d_empty[b]), ((it >> 1) - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(kPN * b);
        for (int c = 0; c < kc && ok; ++c, ++gs) {
          const int s = static_cast<int>(gs % kPStages);
          ok = wait8(smem_u32(&C.full[s]), static_cast<uint32_t>(gs / kPStages) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t wa = smem_u32(smem + s * kPStageBytes), xa = wa + kWBytes;
#pragma unroll
          for (int k = 0; k < kChunk / 32; ++k)
            mma_f8(d, smem_desc_sw128(wa + 32 * k, 1024), smem_desc_sw128(xa + 32 * k, 1024), idesc,
                   (c > 0 || k > 0) ? 1u : 0u);
          tc_commit(smem_u32(&C.empty[s]));
        }
        if (ok && lora) {
          ok = wait8(smem_u32(&C.lora_ready), it & 1, abort_flag);
          if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int k = 0; k < ksteps; ++k)
              mma_ss(d, smem_desc_sw128(la + 32 * k, 1024), smem_desc_sw128(lb + 32 * k, 1024), idesc_b, 1u);
          }
        }
        tc_commit(smem_u32(&C.d_full[b]));  // also reached on abort: tracks every MMA issued
      }
      tc_commit(smem_u32(&C.mma_done));
      drain(smem_u32(&C.mma_done), 0);  // tensor memory is freed only after the last MMA
    }
  } else {
    // ---------------------------------------------------------------- epilogue, adapter operands
    const int et = threadIdx.x - 64;       // 0 .. 127
    const int quarter = warp & 3;          // tensor-memory lane quarter of this warp
    const int row = quarter * 32 + lane;   // weight row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    pdl_wait();  // t and s_x come from the prologue
    // A' [128][64] = B[o, :] / s_w[o] and B' [kPN][64] = lambda t[m, :] / s_x[m] of a tile
    // (bf16, zeros past r, d_o and M; K-major 128-byte swizzled rows), then the arrival
    auto build_lora = [&](int tile) {
      const int64_t o = static_cast<int64_t>(tile / p.mtiles) * kTileO + row;
      const int64_t tok0 = static_cast<int64_t>(tile % p.mtiles) * kPN;
      const float sw = o < p.d_o ? p.s_w[o] : 1.f;
      uint8_t* la = smem + p.off_la + row * 128;
#pragma unroll
      for (int j8 = 0; j8 < kLoraK / 8; ++j8) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int j = 8 * j8 + i;
          v[i] = (o < p.d_o && j < p.r) ? __bfloat162float(p.B[o * p.r + j]) / sw : 0.f;
        }
        *reinterpret_cast<uint4*>(la + ((j8 ^ (row & 7)) << 4)) =
            make_uint4(f32x2_to_bf16x2(v[0], v[1]), f32x2_to_bf16x2(v[2], v[3]), f32x2_to_bf16x2(v[4], v[5]),
                       f32x2_to_bf16x2(v[6], v[7]));
      }
      for (int n = et; n < kPN; n += kEpiThreads) {
        const int64_t m = tok0 + n;
        const float f = m < p.M ? __fdiv_rn(p.lambda, p.s_x[m]) : 0.f;
        uint8_t* lb = smem + p.off_lb + n * 128;
#pragma unroll
        for (int j8 = 0; j8 < kLoraK / 8; ++j8) {
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int j = 8 * j8 + i;
            v[i] = (m < p.M && j < p.r) ? p.t[m * p.t_ld + j] * f : 0.f;
          }
          *reinterpret_cast<uint4*>(lb + ((j8 ^ (n & 7)) << 4)) =
              make_uint4(f32x2_to_bf16x2(v[0], v[1]), f32x2_to_bf16x2(v[2], v[3]), f32x2_to_bf16x2(v[4], v[5]),
                         f32x2_to_bf16x2(v[6], v[7]));
        }
      }
      fence_proxy_async_smem();  // read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.lora_ready));
    };
    bool ok = true;
    int it = 0;
    if (lora && static_cast<int>(blockIdx.x) < p.n_tiles) build_lora(blockIdx.x);
    for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x, ++it) {
      const int b = it & 1;
      ok = wait8(smem_u32(&C.d_full[b]), (it >> 1) & 1, abort_flag);
      ok = __all_sync(0xFFFFFFFFu, ok && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      const int64_t o = static_cast<int64_t>(tile / p.mtiles) * kTileO + row;
      const int64_t tok0 = static_cast<int64_t>(tile % p.mtiles) * kPN;
      const float sw = o < p.d_o ? p.s_w[o] : 0.f;
      for (int n0 = 0; n0 < kPN; n0 += 16) {
        uint32_t dv[16];
        tmem_ld16(tmem + lane_addr + static_cast<uint32_t>(kPN * b + n0), dv);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t m = tok0 + n0 + i;
          if (m < p.M && o < p.d_o) {
            const float v = p.s_x[m] * sw * __uint_as_float(dv[i]);
            if (p.y_f32) static_cast<float*>(p.y)[m * p.d_o + o] = v;
            else static_cast<__nv_bfloat16*>(p.y)[m * p.d_o + o] = __float2bfloat16_rn(v);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.d_empty[b]));
      if (lora && tile + static_cast<int>(gridDim.x) < p.n_tiles) build_lora(tile + gridDim.x);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kPN);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// Row-major [outer][inner] bytes, box of box_inner bytes x box_outer rows, 128-byte swizzle.
bool encode_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Workspace: the E4M3 activations, s_x and t = A h; at large M also the row prologue's f16
// rows and row scales, the f16 adapter (rows rounded up to 16, padding zero), the adapter
// down-projection's split partials and counters.
struct W8Ws {
  uint8_t* qx;
  float* s_x;
  float* t;
  int t_ld;
  __half* hq;
  float* rowscale;
  __half* A16;
  float* t_part;
  int* counters;
  size_t bytes;
};

W8Ws carve_w8(void* ws, int64_t M, int64_t d_i, int r) {
  W8Ws w{};
  const uintptr_t b = reinterpret_cast<uintptr_t>(ws);
  size_t off = 0;
  w.qx = reinterpret_cast<uint8_t*>(b + off);
  off += align_up(static_cast<size_t>(M) * d_i, 256);
  w.s_x = reinterpret_cast<float*>(b + off);
  off += align_up(static_cast<size_t>(M) * 4, 256);
  w.t_ld = r > 0 ? (r + 3) / 4 * 4 : 4;
  w.t = reinterpret_cast<float*>(b + off);
  off += align_up(static_cast<size_t>(M) * w.t_ld * 4, 256);
  if (M > 64 && r <= 32) {
    w.hq = reinterpret_cast<__half*>(b + off);
    off += align_up(static_cast<size_t>(M) * d_i * 2, 256);
    w.rowscale = reinterpret_cast<float*>(b + off);
    off += align_up(static_cast<size_t>(M) * 4, 256);
    if (r > 0) {
      const int r16 = (r + 15) / 16 * 16;
      w.A16 = reinterpret_cast<__half*>(b + off);
      off += align_up(static_cast<size_t>(r16) * d_i * 2, 256);
      w.t_part = reinterpret_cast<float*>(b + off);
      off += lora_down_t_scratch_bytes(M, r);
      w.counters = reinterpret_cast<int*>(b + off);
      off += align_up(static_cast<size_t>((M + 127) / 128 + 8) * 4, 256);
    }
  }
  w.bytes = off;
  return w;
}

}  // namespace

bool w8a8_supported(int64_t M, int64_t d_i, int64_t d_o, int r) {
  return M >= 1 && d_o >= 1 && d_i >= kChunk && d_i % kChunk == 0 && d_i <= 32768 && r >= 0 && r <= kMaxR;
}

size_t w8a8_workspace_bytes(int64_t M, int64_t d_i, int64_t, int r) { return carve_w8(nullptr, M, d_i, r).bytes; }

cudaError_t launch_w8a8_quantize(const void* W, int64_t d_o, int64_t d_i, uint8_t* codes, float* s_w,
                                 cudaStream_t stream) {
  k_w8_quant<<<static_cast<unsigned>(d_o), kQThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(W), d_i, codes,
                                                                    s_w);
  return cudaGetLastError();
}

cudaError_t launch_w8a8_linear(const W8Args& a, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(k_w8_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(k_w8_gemm_p, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const W8Ws w = carve_w8(a.ws, a.M, a.d_i, a.r);
  cudaError_t e = cudaSuccess;
  if (a.M > 64 && a.r <= 32) {
    // large M: the row prologue (E4M3 codes, s_x, f16 rows) and the adapter's down-projection
    // on the tensor cores (ranks up to 32), in place of the cluster prologue
    LinearArgs in{};
    in.x = a.x;
    in.M = a.M;
    in.d_i = a.d_i;
    in.w_norm = a.w_norm;
    in.z = a.w_norm ? a.z : nullptr;
    in.z_ld = (a.w_norm && a.z) ? a.z_ld : 0;
    in.eps = a.eps;
    ActConv conv{};
    if (a.r > 0) {
      const int r16 = (a.r + 15) / 16 * 16;
      conv.A[0] = a.A;
      conv.A16[0] = w.A16;
      conv.r[0] = a.r;
      conv.n = 1;
      conv.zero[conv.n_zero_ranges] = reinterpret_cast<float*>(w.counters);
      conv.n_zero[conv.n_zero_ranges++] = ((a.M + 127) / 128 + 3) / 4 * 4;
      if (r16 > a.r) {
        conv.zero[conv.n_zero_ranges] = reinterpret_cast<float*>(w.A16 + static_cast<int64_t>(a.r) * a.d_i);
        conv.n_zero[conv.n_zero_ranges++] = static_cast<int64_t>(r16 - a.r) * a.d_i / 2;
      }
    }
    e = launch_act_prologue(in, w.hq, w.rowscale, conv, stream, w.qx, w.s_x);
    if (e != cudaSuccess) return e;
    if (a.r > 0) {
      e = launch_lora_down_t(w.hq, a.M, a.d_i, w.A16, a.r, w.rowscale, w.t, w.t_ld, w.t_part, w.counters, stream);
      if (e != cudaSuccess) return e;
    }
  } else {
    e = launch_pro_fp8(a.x, a.M, a.d_i, a.w_norm, a.z, a.z_ld, a.eps, a.A, a.r, w.qx, w.s_x, w.t, w.t_ld, stream);
    if (e != cudaSuccess) return e;
  }

  W8Params p{};
  p.M = a.M;
  p.d_i = a.d_i;
  p.d_o = a.d_o;
  p.s_w = a.s_w;
  p.s_x = w.s_x;
  p.t = w.t;
  p.t_ld = w.t_ld;
  p.B = a.r > 0 ? static_cast<const __nv_bfloat16*>(a.B) : nullptr;
  p.r = a.r;
  p.lambda = a.lambda;
  p.y = a.y;
  p.y_f32 = a.y_f32 ? 1 : 0;
  p.kc = static_cast<int>(a.d_i / kChunk);
  p.otiles = static_cast<int>((a.d_o + kTileO - 1) / kTileO);
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  if (a.M > 64) {  // large M: the persistent kernel
    p.N = kPN;
    p.mtiles = static_cast<int>((a.M + kPN - 1) / kPN);
    p.n_tiles = p.otiles * p.mtiles;
    p.off_la = kPStages * kPStageBytes;
    p.off_lb = p.off_la + kTileO * 128;
    p.off_ctrl = static_cast<uint32_t>(align_up(p.off_lb + static_cast<size_t>(kPN) * 128, 128));
    W8Maps maps;
    if (!encode_u8(&maps.w, a.codes, a.d_i, a.d_o, kChunk, kTileO) || !encode_u8(&maps.x, w.qx, a.d_i, a.M, kChunk, kPN))
      return cudaErrorInvalidValue;
    cudaLaunchConfig_t c{};
    c.gridDim = dim3(static_cast<unsigned>(p.n_tiles < sm_count() ? p.n_tiles : sm_count()));
    c.blockDim = dim3(kThreads);
    c.dynamicSmemBytes = 1024 + p.off_ctrl + sizeof(W8PCtrl);
    c.stream = stream;
    c.attrs = pdl;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, k_w8_gemm_p, maps, p);
  }
  p.N = static_cast<int>((a.M + 15) / 16 * 16);
  const int mtiles = static_cast<int>((a.M + p.N - 1) / p.N);
  // split K when the tiles alone leave most SMs idle (decode)
  const int tiles = p.otiles * mtiles;
  int S = 1;
  while (S < kMaxSplit && S < p.kc && tiles * (S + 1) <= sm_count()) ++S;
  p.splits = S;
  p.stage_bytes = static_cast<uint32_t>(kWBytes + p.N * kChunk);
  const size_t fixed = 1024 + static_cast<size_t>(kTileO) * 128 + static_cast<size_t>(p.N) * 128 + sizeof(W8Ctrl);
  int st = static_cast<int>((227 * 1024 - fixed) / p.stage_bytes);
  st = st > kMaxStages ? kMaxStages : st;
  p.stages = st;
  p.off_la = static_cast<uint32_t>(st) * p.stage_bytes;
  p.off_lb = p.off_la + kTileO * 128;
  p.off_ctrl = static_cast<uint32_t>(align_up(p.off_lb + static_cast<size_t>(p.N) * 128, 128));
  const size_t smem = 1024 + p.off_ctrl + sizeof(W8Ctrl);
  if (st < 2 || (S > 1 && static_cast<size_t>(p.N) * kTileO * 4 > static_cast<size_t>(st) * p.stage_bytes))
    return cudaErrorInvalidValue;

  W8Maps maps;
  if (!encode_u8(&maps.w, a.codes, a.d_i, a.d_o, kChunk, kTileO) ||
      !encode_u8(&maps.x, w.qx, a.d_i, a.M, kChunk, p.N))
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attrs[2];
  attrs[0] = pdl[0];
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = static_cast<unsigned>(S);
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t c{};
  c.gridDim = dim3(static_cast<unsigned>(tiles * S));
  c.blockDim = dim3(kThreads);
  c.dynamicSmemBytes = smem;
  c.stream = stream;
  c.attrs = attrs;
  c.numAttrs = 2;
  return cudaLaunchKernelEx(&c, k_w8_gemm, maps, p);
}

uint32_t w8_read_and_clear_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_w8_status, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_w8_status, &zero, sizeof(zero));
  return v;
}

}  // namespace pl
