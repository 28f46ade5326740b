// Backward of the frozen-backbone NVFP4 + LoRA linear and its RMSNorm-AQN prologue, sm_103a.
//
// "QeRL: When Quantized Weights Help Reinforcement Learning, and Where the Evidence Stops",
// section 2.1 "Weight storage and trainable state are different budgets": the backbone
// W_hat is frozen, the gradients train A and B and still pass through the frozen quantised
// projection to reach the layers before it.  For the upstream gradient g = dL/dy [M, d_o]:
//   u  = lambda g B                      [M, r]
//   dh = g W_hat + u A                   [M, d_i]
//   dA = u^T h                           [r, d_i]
//   dB = lambda g^T (h A^T)              [d_o, r]
//   dx = rho s (.) dh - rho^3 x (sum_j x_j s_j dh_j) / d_i,  s = w_norm + z,
//   rho = (mean x^2 + eps)^(-1/2)        (section 5.1's norm; w_norm and z are not trained)
//
// Every contraction runs on the tensor cores (tcgen05.mma kind::f16, BF16 operands, FP32
// accumulation).  The contractions over tokens (dA, dB) and over the weight's output axis
// (dh) read operands whose contiguous axis is the MMA's M or N axis: those are fed
// MN-major (128-byte swizzled atoms of 8 K-lines x 64 elements), so nothing is transposed
// in memory:
//   k_bgemm<a_mn, b_mn>: D[128 rows][64 cols] = sum_k A[row, k] B[col, k], both operands by
//     TMA (K-major or MN-major), K split over a cluster with the partials added over DSMEM
//     in split order; it gives lambda t = lambda h A^T, u = lambda g B (B padded to 64
//     columns by k_pad_b), dA and dB;
//   k_bwd_dh: D1[128 rows of d_i][N tokens] = sum_o (s_b q)[o, i] g[t, o] and
//     D2 = sum_j A[j, i] u[t, j], dh = s_g D1 + D2: eight warps dequantise each 64-row slab of
//     codes (E2M1 x E4M3, exact in BF16) straight into the MN-major layout, g and u are
//     K-major TMA tiles, A an MN-major one;
//   k_bwd_norm: the RMSNorm-AQN backward, one CTA per token row.
// BF16 rounding enters through h, u and lambda t (relative 2^-9 per element); W_hat and g
// are exact.  Every wait is bounded (200 ms).
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace pl {

__device__ uint32_t g_bw_status = 0;

namespace {

constexpr int kBK = 64;               // K elements per stage: one 128-byte line of 16-bit values
constexpr uint32_t kAtomMN = 8192;    // bytes between the two 64-wide MN atoms of a 128-wide operand
constexpr int kMaxStages = 6;
constexpr int kMaxSplit = 8;

PL_DEVINL bool waitb(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return wait_or_abort_status(bar, parity, abort_flag, &g_bw_status);
}
PL_DEVINL void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
PL_DEVINL uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// ------------------------------------------------------------------ generic BF16 GEMM
struct BgParams {
  int rows, cols;     // problem rows (tiles of 128) and columns written (<= 64)
  int kc, splits, stages;
  uint32_t stage_bytes, off_ctrl;
  float scale;
  void* out;
  int out_bf16;       // 1: BF16 [rows][64] (all 64 columns), 0: FP32
  int transpose;      // FP32 only: 1 -> out[col * ld + row], 0 -> out[row * ld + col]
  int64_t ld;
};
struct BgMaps {
  CUtensorMap a, b;
};
struct BgCtrl {
  uint64_t full[kMaxStages], empty[kMaxStages], d_full;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int kBgThreads = 192;  // producer, MMA + TMEM, 4 epilogue warps
constexpr uint32_t kBgA = 16384, kBgB = 8192;

template <bool kAMN, bool kBMN>
__global__ void __launch_bounds__(kBgThreads, 1) k_bgemm(const __grid_constant__ BgMaps maps,
                                                         const __grid_constant__ BgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BgCtrl& C = *reinterpret_cast<BgCtrl*>(smem + p.off_ctrl);
  volatile int* abort_flag = &C.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits, split = static_cast<int>(cl_rank());
  const int tile = blockIdx.x / S;
  const int32_t row0 = tile * 128;
  const int c0 = static_cast<int>((static_cast<int64_t>(split) * p.kc) / S);
  const int c1 = static_cast<int>((static_cast<int64_t>(split + 1) * p.kc) / S);
  const int nch = c1 - c0, stages = p.stages;
  if (threadIdx.x == 0) {
    pdl_launch_dependents();
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&C.full[s]), 1);
      mbar_init(smem_u32(&C.empty[s]), 1);
    }
    mbar_init(smem_u32(&C.d_full), 1);
    C.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&C.tmem_base), 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;
  bool go = false;
  if (warp == 0) {
    if (lane == 0) {
      pdl_wait();  // both operands may come from the preceding kernels
      bool ok = true;
      int c = 0;
      for (; c < nch && ok; ++c) {
        const int s = c % stages;
        if (c >= stages) ok = waitb(smem_u32(&C.empty[s]), ((c / stages) - 1) & 1, abort_flag);
        if (!ok) break;
        const uint32_t fb = smem_u32(&C.full[s]);
        const uint32_t sa = smem_u32(smem + s * p.stage_bytes), sb = sa + kBgA;
        const int32_t k0 = (c0 + c) * kBK;
        mbar_arrive_expect_tx(fb, kBgA + kBgB);
        if (kAMN) {
          tma_load_2d(sa, &maps.a, row0, k0, fb);
          tma_load_2d(sa + kAtomMN, &maps.a, row0 + 64, k0, fb);
        } else {
          tma_load_2d(sa, &maps.a, k0, row0, fb);
        }
        if (kBMN) tma_load_2d(sb, &maps.b, 0, k0, fb);
        else tma_load_2d(sb, &maps.b, k0, 0, fb);
      }
      if (*abort_flag)
        for (int d = (c - stages > 0 ? c - stages : 0); d < c; ++d) drain(smem_u32(&C.full[d % stages]), (d / stages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_major(128, 64, 1, kAMN ? 1 : 0, kBMN ? 1 : 0);
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        const int s = c % stages;
        ok = waitb(smem_u32(&C.full[s]), (c / stages) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * p.stage_bytes), sb = sa + kBgA;
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const uint64_t ad = kAMN ? smem_desc_mn_sw128(sa + ks * 2048, kAtomMN, 1024) : smem_desc_sw128(sa + ks * 32, 1024);
          const uint64_t bd = kBMN ? smem_desc_mn_sw128(sb + ks * 2048, kAtomMN, 1024) : smem_desc_sw128(sb + ks * 32, 1024);
          mma_ss(tmem, ad, bd, idesc, (c > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&C.empty[s]));
      }
      tc_commit(smem_u32(&C.d_full));
    }
  } else {
    const int quarter = warp & 3, row = quarter * 32 + lane;
    bool ok = waitb(smem_u32(&C.d_full), 0, abort_flag);
    tc_fence_after();
    go = named_bar_and(1, 128, ok && !*abort_flag && nch > 0);
    float* red = reinterpret_cast<float*>(smem);  // [128][65] partials (reuses the stages)
    const int64_t r = static_cast<int64_t>(row0) + row;
    const uint32_t la = static_cast<uint32_t>(quarter * 32) << 16;
    for (int c16 = 0; c16 < 64 && go; c16 += 16) {
      uint32_t d[16];
      tmem_ld16(tmem + la + static_cast<uint32_t>(c16), d);
      tmem_ld_wait();
      if (S > 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) red[row * 65 + c16 + i] = __uint_as_float(d[i]);
      } else if (r < p.rows) {
        if (p.out_bf16) {
          uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + r * 64 + c16);
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            w[i] = f32x2_to_bf16x2(p.scale * __uint_as_float(d[2 * i]), p.scale * __uint_as_float(d[2 * i + 1]));
          o[0] = make_uint4(w[0], w[1], w[2], w[3]);
          o[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c16 + i < p.cols) {
              float* o = static_cast<float*>(p.out) + (p.transpose ? (c16 + i) * p.ld + r : r * p.ld + c16 + i);
              *o = p.scale * __uint_as_float(d[i]);
            }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (S > 1) {
    cluster_sync();
    // rows [128 split / S, 128 (split+1) / S) of the tile: the S partials in split order
    if (threadIdx.x >= 64 && go) {
      const int et = threadIdx.x - 64;
      const int ra = (128 * split) / S, rb = (128 * (split + 1)) / S;
      const uint32_t red_addr = smem_u32(smem);
      for (int e = et; e < (rb - ra) * 64; e += 128) {
        const int rr = ra + e / 64, col = e % 64;
        const uint32_t addr = red_addr + static_cast<uint32_t>((rr * 65 + col) * 4);
        float part[kMaxSplit];
#pragma unroll
        for (int sp = 0; sp < kMaxSplit; ++sp)
          if (sp < S) part[sp] = ld_dsmem_f32(mapa_shared(addr, sp));
        float v = 0.f;
#pragma unroll
        for (int sp = 0; sp < kMaxSplit; ++sp)
          if (sp < S) v += part[sp];
        v *= p.scale;
        const int64_t r = static_cast<int64_t>(row0) + rr;
        if (r >= p.rows) continue;
        if (p.out_bf16) static_cast<__nv_bfloat16*>(p.out)[r * 64 + col] = __float2bfloat16_rn(v);
        else if (col < p.cols) static_cast<float*>(p.out)[p.transpose ? col * p.ld + r : r * p.ld + col] = v;
      }
    }
    cluster_sync();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// ------------------------------------------------------------------ dh = g W_hat + u A
struct DhParams {
  int64_t M, d_i, d_o;
  int N, itiles, kc, stages, r16;
  uint32_t stage_bytes, off_deq, off_la, off_lb, off_ctrl;
  const float* s_g;
  float* dh;
};
struct DhMaps {
  CUtensorMap codes, scales, g, a, u;
};
struct DhCtrl {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t deq_full[2], deq_empty[2], lora_full, d_full;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int kDhThreads = 320;  // producer, MMA + TMEM, 8 dequant / epilogue warps
constexpr uint32_t kDhCodes = 64 * 64, kDhScales = 64 * 16, kDhDeq = 16384;

__global__ void __launch_bounds__(kDhThreads, 1) k_bwd_dh(const __grid_constant__ DhMaps maps,
                                                          const __grid_constant__ DhParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DhCtrl& C = *reinterpret_cast<DhCtrl*>(smem + p.off_ctrl);
  volatile int* abort_flag = &C.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, stages = p.stages, kc = p.kc;
  const int itile = blockIdx.x % p.itiles, mtile = blockIdx.x / p.itiles;
  const int32_t i0 = itile * 128, t0 = mtile * N;
  const uint32_t g_bytes = static_cast<uint32_t>(N) * 128u;
  // two accumulators of N columns: D1 (backbone) at column 0, D2 (adapter) at column acc2
  const uint32_t acc2 = N <= 32 ? 32u : (N <= 64 ? 64u : 128u), tcols = 2 * acc2;
  if (threadIdx.x == 0) {
    pdl_launch_dependents();
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&C.full[s]), 1);
      mbar_init(smem_u32(&C.empty[s]), 8 + 1);  // the dequant warps (codes, scales) and the MMAs (g)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&C.deq_full[b]), 8);
      mbar_init(smem_u32(&C.deq_empty[b]), 1);
    }
    mbar_init(smem_u32(&C.lora_full), 1);
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
      pdl_wait();  // g and u may come from the preceding kernels
      if (p.r16 > 0) {
        const uint32_t lb = smem_u32(&C.lora_full);
        mbar_arrive_expect_tx(lb, 2 * kAtomMN + g_bytes);
        tma_load_2d(smem_u32(smem + p.off_la), &maps.a, i0, 0, lb);
        tma_load_2d(smem_u32(smem + p.off_la) + kAtomMN, &maps.a, i0 + 64, 0, lb);
        tma_load_2d(smem_u32(smem + p.off_lb), &maps.u, 0, t0, lb);
      }
      bool ok = true;
      int c = 0;
      for (; c < kc && ok; ++c) {
        const int s = c % stages;
        if (c >= stages) ok = waitb(smem_u32(&C.empty[s]), ((c / stages) - 1) & 1, abort_flag);
        if (!ok) break;
        // stage: g (1024-byte aligned for the swizzle), codes, scales
        const uint32_t fb = smem_u32(&C.full[s]), st = smem_u32(smem + s * p.stage_bytes);
        mbar_arrive_expect_tx(fb, kDhCodes + kDhScales + g_bytes);
        tma_load_2d(st, &maps.g, c * kBK, t0, fb);
        tma_load_2d(st + g_bytes, &maps.codes, i0 / 2, c * kBK, fb);
        tma_load_2d(st + g_bytes + kDhCodes, &maps.scales, (i0 / 256) * 16, c * kBK, fb);
      }
      if (*abort_flag) {
        for (int d = (c - stages > 0 ? c - stages : 0); d < c; ++d) drain(smem_u32(&C.full[d % stages]), (d / stages) & 1);
        if (p.r16 > 0) drain(smem_u32(&C.lora_full), 0);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_major(128, N, 1, 1, 0);  // A (W_hat^T slab) MN-major, B (g) K-major
      bool ok = true;
      for (int c = 0; c < kc && ok; ++c) {
        const int s = c % stages, b = c & 1;
        ok = waitb(smem_u32(&C.deq_full[b]), (c >> 1) & 1, abort_flag) &&
             waitb(smem_u32(&C.full[s]), (c / stages) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + p.off_deq + b * kDhDeq);
        const uint32_t sg = smem_u32(smem + s * p.stage_bytes);
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks)
          mma_ss(tmem, smem_desc_mn_sw128(sa + ks * 2048, kAtomMN, 1024), smem_desc_sw128(sg + ks * 32, 1024), idesc,
                 (c > 0 || ks > 0) ? 1u : 0u);
        tc_commit(smem_u32(&C.deq_empty[b]));
        tc_commit(smem_u32(&C.empty[s]));
      }
      if (ok && p.r16 > 0) {
        ok = waitb(smem_u32(&C.lora_full), 0, abort_flag);
        if (ok) {
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + p.off_la), sb = smem_u32(smem + p.off_lb);
          for (int ks = 0; ks < p.r16; ++ks)
            mma_ss(tmem + acc2, smem_desc_mn_sw128(sa + ks * 2048, kAtomMN, 1024),
                   smem_desc_sw128(sb + ks * 32, 1024), idesc, ks > 0 ? 1u : 0u);
        }
      }
      tc_commit(smem_u32(&C.d_full));
    }
  } else {
    // ---------------------------------------------------------------- dequant, then epilogue
    const int et = threadIdx.x - 64;  // 0 .. 255
    const float s_g = *p.s_g;         // a weight input
    const int sc_off = (i0 % 256) / 16;
    bool ok = true;
    for (int c = 0; c < kc && ok; ++c) {
      const int s = c % stages, b = c & 1;
      ok = waitb(smem_u32(&C.full[s]), (c / stages) & 1, abort_flag) &&
           (c < 2 || waitb(smem_u32(&C.deq_empty[b]), ((c >> 1) - 1) & 1, abort_flag));
      if (!ok) break;
      const uint8_t* codes = smem + s * p.stage_bytes + N * 128;
      const uint8_t* scales = codes + kDhCodes;
      uint8_t* dq = smem + p.off_deq + b * kDhDeq;
      // 64 weight rows (K) x 16 pieces of 8 d_i values (MN); piece cc of row o goes to MN atom
      // cc / 8, K group o / 8, line o % 8, 16-byte slot (cc % 8) ^ (o % 8)
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int task = et + 256 * t, o = task >> 4, cc = task & 15;
        const uint32_t cw = *reinterpret_cast<const uint32_t*>(codes + o * 64 + cc * 4);
        const uint32_t sbyte = scales[o * 16 + sc_off + (cc >> 1)];
        const uint32_t s2 = cvt_e4m3x2_to_f16x2(sbyte | (sbyte << 8));
        uint32_t v[4];
        e2m1x8_to_f16x8(cw, v[0], v[1], v[2], v[3]);
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t h2 = hmul2_u32(v[i], s2);  // q s_b, exact in f16
          const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
          const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
          w[i] = f32x2_to_bf16x2(lo, hi);  // exact: at most 7 significant bits
        }
        const int kr = o & 7;
        *reinterpret_cast<uint4*>(dq + (cc >> 3) * kAtomMN + (o >> 3) * 1024 + kr * 128 + (((cc & 7) ^ kr) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_async_smem();  // read by the tensor cores
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&C.deq_full[b]));
        mbar_arrive(smem_u32(&C.empty[s]));
      }
    }
    ok = waitb(smem_u32(&C.d_full), 0, abort_flag) && ok;
    tc_fence_after();
    go = named_bar_and(1, 256, ok && !*abort_flag);
    if (go) {
      // lane quarter (warp % 4) x token half ((warp - 2) / 4): dh[t][i] = s_g D1[i][t] + D2[i][t]
      const int quarter = warp & 3, half = (warp - 2) >> 2;
      const int row = quarter * 32 + lane;
      const uint32_t la = static_cast<uint32_t>(quarter * 32) << 16;
      const int nh = N / 2;
      for (int n0 = half * nh; n0 < (half + 1) * nh; n0 += 8) {
        uint32_t d[8], e[8];
        tmem_ld8(tmem + la + static_cast<uint32_t>(n0), d);
        if (p.r16 > 0) tmem_ld8(tmem + la + acc2 + static_cast<uint32_t>(n0), e);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int64_t t = static_cast<int64_t>(t0) + n0 + i;
          const float v = s_g * __uint_as_float(d[i]) + (p.r16 > 0 ? __uint_as_float(e[i]) : 0.f);
          if (t < p.M) p.dh[t * p.d_i + i0 + row] = v;
        }
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

// B [d_o][r] -> Bp [d_o][64] (zeros past r), BF16: the MN-major operand of u = lambda g B.
__global__ void k_pad_b(const __nv_bfloat16* __restrict__ B, int64_t d_o, int r, __nv_bfloat16* __restrict__ Bp) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= d_o * 64) return;
  const int64_t o = i / 64;
  const int j = static_cast<int>(i % 64);
  Bp[i] = j < r ? B[o * r + j] : __float2bfloat16_rn(0.f);
}

// dx = rho s (.) dh - rho^3 x (sum_j x_j s_j dh_j) / d, one CTA per token row.
constexpr int kNbThreads = 256;
__global__ void __launch_bounds__(kNbThreads) k_bwd_norm(const __nv_bfloat16* __restrict__ x, int64_t d,
                                                         const float* __restrict__ w, const float* __restrict__ z,
                                                         int64_t z_ld, float eps, const float* __restrict__ dh,
                                                         float* __restrict__ dx) {
  __shared__ float red[2][kNbThreads / 32];
  const int64_t m = blockIdx.x;
  const __nv_bfloat16* xr = x + m * d;
  const float* zr = z != nullptr ? z + m * z_ld : nullptr;
  pdl_wait();  // dh comes from the preceding kernel
  float ss = 0.f, pr = 0.f;
  for (int64_t k = threadIdx.x; k < d; k += kNbThreads) {
    const float xv = __bfloat162float(xr[k]);
    const float s = w[k] + (zr != nullptr ? zr[k] : 0.f);
    ss = fmaf(xv, xv, ss);
    pr = fmaf(xv * s, dh[m * d + k], pr);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    pr += __shfl_xor_sync(0xFFFFFFFFu, pr, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = ss;
    red[1][threadIdx.x >> 5] = pr;
  }
  __syncthreads();
  float tss = 0.f, tpr = 0.f;
#pragma unroll
  for (int i = 0; i < kNbThreads / 32; ++i) {
    tss += red[0][i];
    tpr += red[1][i];
  }
  const float rho = 1.0f / sqrtf(tss / static_cast<float>(d) + eps);
  const float coef = rho * rho * rho * tpr / static_cast<float>(d);
  for (int64_t k = threadIdx.x; k < d; k += kNbThreads) {
    const float xv = __bfloat162float(xr[k]);
    const float s = w[k] + (zr != nullptr ? zr[k] : 0.f);
    dx[m * d + k] = rho * s * dh[m * d + k] - coef * xv;
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_bw() {
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

// Row-major [outer][inner] tensor of `esize`-byte elements; box box_inner x box_outer.
bool map2d(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* base, uint64_t inner, uint64_t outer,
           uint32_t box_inner, uint32_t box_outer, bool swizzle) {
  auto fn = encode_bw();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t bi, uint32_t bo) {
  return map2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, bi, bo, true);
}

cudaError_t set_attrs_bw() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    const int big = 227 * 1024;
    err = cudaFuncSetAttribute(k_bgemm<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(k_bgemm<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(k_bgemm<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(k_bwd_dh, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
  });
  return err;
}

cudaLaunchAttribute g_pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// D[rows][64] = sum over K of A[row, k] B[col, k]; maps prepared by the caller (A: box 64 x 128
// K-major or 64 x 64 MN-major; B: box 64 x 64).
template <bool kAMN, bool kBMN>
cudaError_t launch_bgemm(const BgMaps& maps, int64_t rows, int cols, int64_t K, float scale, void* out, bool bf16,
                         bool transpose, int64_t ld, cudaStream_t stream) {
  BgParams p{};
  p.rows = static_cast<int>(rows);
  p.cols = cols;
  p.kc = static_cast<int>((K + kBK - 1) / kBK);
  const int tiles = static_cast<int>((rows + 127) / 128);
  int S = 1;
  while (S < kMaxSplit && S < p.kc && tiles * (S + 1) <= sm_count()) ++S;
  p.splits = S;
  p.stage_bytes = kBgA + kBgB;
  p.stages = kMaxStages;
  p.off_ctrl = static_cast<uint32_t>(p.stages) * p.stage_bytes;
  p.scale = scale;
  p.out = out;
  p.out_bf16 = bf16 ? 1 : 0;
  p.transpose = transpose ? 1 : 0;
  p.ld = ld;
  cudaLaunchAttribute at[2] = {g_pdl_attr(), {}};
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = static_cast<unsigned>(S);
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t c{};
  c.gridDim = dim3(static_cast<unsigned>(tiles * S));
  c.blockDim = dim3(kBgThreads);
  c.dynamicSmemBytes = 1024 + p.off_ctrl + sizeof(BgCtrl);
  c.stream = stream;
  c.attrs = at;
  c.numAttrs = 2;
  return cudaLaunchKernelEx(&c, k_bgemm<kAMN, kBMN>, maps, p);
}

struct BwWs {
  __nv_bfloat16 *hb, *bp, *lu, *lt;
  float* dh;
  size_t bytes;
};

BwWs carve_bw(void* ws, int64_t M, int64_t d_i, int64_t d_o, bool norm, bool lora) {
  BwWs w{};
  const uintptr_t b = reinterpret_cast<uintptr_t>(ws);
  size_t off = 0;
  auto take = [&](size_t n) {
    const uintptr_t p = b + off;
    off += align_up(n, 256);
    return p;
  };
  w.hb = norm ? reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(M) * d_i * 2)) : nullptr;
  w.dh = norm ? reinterpret_cast<float*>(take(static_cast<size_t>(M) * d_i * 4)) : nullptr;
  w.bp = lora ? reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(d_o) * 64 * 2)) : nullptr;
  w.lu = lora ? reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(M) * 64 * 2)) : nullptr;
  w.lt = lora ? reinterpret_cast<__nv_bfloat16*>(take(static_cast<size_t>(M) * 64 * 2)) : nullptr;
  w.bytes = off;
  return w;
}

}  // namespace

bool backward_supported(int64_t M, int64_t d_i, int64_t d_o, int r) {
  // d_i % 256: the rows of block scales (d_i / 16 bytes) must be 16-byte multiples for TMA
  return M >= 1 && d_o >= 8 && d_o % 8 == 0 && d_i >= 256 && d_i % 256 == 0 && r >= 0 && r <= 64;
}

size_t backward_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r, bool norm) {
  return carve_bw(nullptr, M, d_i, d_o, norm, r > 0).bytes;
}

cudaError_t launch_backward(const BwArgs& a, cudaStream_t stream) {
  cudaError_t e = set_attrs_bw();
  if (e != cudaSuccess) return e;
  const bool norm = a.w_norm != nullptr, lora = a.r > 0;
  const BwWs w = carve_bw(a.ws, a.M, a.d_i, a.d_o, norm, lora);
  const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(a.g);
  // h in BF16: the norm's output, or x itself
  const __nv_bfloat16* hb = static_cast<const __nv_bfloat16*>(a.x);
  if (norm) {
    e = launch_rmsnorm_aqn(a.x, a.M, a.d_i, a.w_norm, a.z, a.z_ld, a.eps, w.hb, false, stream);
    if (e != cudaSuccess) return e;
    hb = w.hb;
  }
  if (lora) {
    const int64_t n = a.d_o * 64;
    k_pad_b<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(a.B), a.d_o,
                                                                     a.r, w.bp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    BgMaps m;
    // lambda t = lambda h A^T: rows = tokens, K = d_i, A and h both K-major
    if (!map_bf16(&m.a, hb, a.d_i, a.M, 64, 128) || !map_bf16(&m.b, a.A, a.d_i, a.r, 64, 64))
      return cudaErrorInvalidValue;
    if ((e = launch_bgemm<false, false>(m, a.M, 64, a.d_i, a.lambda, w.lt, true, false, 64, stream)) != cudaSuccess)
      return e;
    // u = lambda g B: rows = tokens, K = d_o, g K-major, B (padded) MN-major
    if (!map_bf16(&m.a, g, a.d_o, a.M, 64, 128) || !map_bf16(&m.b, w.bp, 64, a.d_o, 64, 64))
      return cudaErrorInvalidValue;
    if ((e = launch_bgemm<false, true>(m, a.M, 64, a.d_o, a.lambda, w.lu, true, false, 64, stream)) != cudaSuccess)
      return e;
  }
  // dh = s_g g (s_b q) + u A
  DhParams p{};
  p.M = a.M;
  p.d_i = a.d_i;
  p.d_o = a.d_o;
  p.N = a.M <= 128 ? static_cast<int>((a.M + 15) / 16 * 16) : 128;
  p.itiles = static_cast<int>(a.d_i / 128);
  p.kc = static_cast<int>((a.d_o + kBK - 1) / kBK);
  p.r16 = lora ? (a.r + 15) / 16 : 0;
  p.stage_bytes = static_cast<uint32_t>(align_up(static_cast<size_t>(p.N) * 128 + kDhCodes + kDhScales, 1024));
  const size_t fixed = 2 * kDhDeq + 2 * kAtomMN + static_cast<size_t>(p.N) * 128 + sizeof(DhCtrl) + 1024 + 256;
  int st = static_cast<int>((227 * 1024 - fixed) / p.stage_bytes);
  p.stages = st > kMaxStages ? kMaxStages : st;
  if (p.stages < 2) return cudaErrorInvalidValue;
  p.off_deq = static_cast<uint32_t>(p.stages) * p.stage_bytes;
  p.off_la = p.off_deq + 2 * kDhDeq;
  p.off_lb = p.off_la + 2 * kAtomMN;
  p.off_ctrl = static_cast<uint32_t>(align_up(p.off_lb + static_cast<size_t>(p.N) * 128, 128));
  p.s_g = a.s_g;
  p.dh = norm ? w.dh : a.dx;
  DhMaps dm;
  memset(&dm, 0, sizeof(dm));
  bool ok = map2d(&dm.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, a.d_i / 2, a.d_o, 64, 64, false) &&
            map2d(&dm.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.scales, a.d_i / 16, a.d_o, 16, 64, false) &&
            map_bf16(&dm.g, g, a.d_o, a.M, 64, p.N);
  if (ok && lora) ok = map_bf16(&dm.a, a.A, a.d_i, a.r, 64, 64) && map_bf16(&dm.u, w.lu, 64, a.M, 64, p.N);
  if (!ok) return cudaErrorInvalidValue;
  {
    cudaLaunchAttribute at[1] = {g_pdl_attr()};
    cudaLaunchConfig_t c{};
    c.gridDim = dim3(static_cast<unsigned>(p.itiles * ((a.M + p.N - 1) / p.N)));
    c.blockDim = dim3(kDhThreads);
    c.dynamicSmemBytes = 1024 + p.off_ctrl + sizeof(DhCtrl);
    c.stream = stream;
    c.attrs = at;
    c.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&c, k_bwd_dh, dm, p)) != cudaSuccess) return e;
  }
  if (norm) {
    cudaLaunchAttribute at[1] = {g_pdl_attr()};
    cudaLaunchConfig_t c{};
    c.gridDim = dim3(static_cast<unsigned>(a.M));
    c.blockDim = dim3(kNbThreads);
    c.stream = stream;
    c.attrs = at;
    c.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&c, k_bwd_norm, static_cast<const __nv_bfloat16*>(a.x), a.d_i, a.w_norm, a.z,
                                a.z != nullptr ? a.z_ld : int64_t{0}, a.eps, static_cast<const float*>(w.dh),
                                a.dx)) != cudaSuccess)
      return e;
  }
  if (lora && a.dA != nullptr) {
    // dA[j][i] = sum_t u[t][j] h[t][i]: rows = d_i, K = tokens, both MN-major
    BgMaps m;
    if (!map_bf16(&m.a, hb, a.d_i, a.M, 64, 64) || !map_bf16(&m.b, w.lu, 64, a.M, 64, 64)) return cudaErrorInvalidValue;
    if ((e = launch_bgemm<true, true>(m, a.d_i, a.r, a.M, 1.0f, a.dA, false, true, a.d_i, stream)) != cudaSuccess)
      return e;
  }
  if (lora && a.dB != nullptr) {
    // dB[o][j] = sum_t g[t][o] (lambda t)[t][j]: rows = d_o, K = tokens, both MN-major
    BgMaps m;
    if (!map_bf16(&m.a, g, a.d_o, a.M, 64, 64) || !map_bf16(&m.b, w.lt, 64, a.M, 64, 64)) return cudaErrorInvalidValue;
    if ((e = launch_bgemm<true, true>(m, a.d_o, a.r, a.M, 1.0f, a.dB, false, false, a.r, stream)) != cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

uint32_t bw_read_and_clear_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_bw_status, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_bw_status, &zero, sizeof(zero));
  return v;
}

}  // namespace pl
