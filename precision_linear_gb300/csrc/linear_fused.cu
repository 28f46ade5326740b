// Single-kernel tcgen05 NVFP4 + LoRA + RMSNorm-AQN linear for decode (M <= 64), sm_103a.
//
// Computes the forward map of "QeRL: When Quantized Weights Help Reinforcement
// Learning, and Where the Evidence Stops", section 2.1 (y = W_hat h + lambda B (A h)),
// on the section 3.1 NVFP4 backbone (w_hat = s_g s_b q), with the section 5.1 input
// h = x / rms(x) (.) (w_norm + z).
//
// Used when every CTA's slice of the K = d_i axis is at most 3 chunks of 256, so that
// the CTA holds all of its weights (dequantised, in tensor memory) and all of its
// activations (shared memory) at once.  A cluster of S CTAs covers 128 weight rows;
// CTA s takes chunks [s kc / S, (s+1) kc / S).  The norm is folded in by linearity:
//   y[m, o] = rs_m * ( sum_k W_hat[o, k] u[m, k] + lambda sum_j B[o, j] sum_k A[j, k] u[m, k] ),
//   u = x (.) (w_norm + z),   rs_m = 1 / sqrt(sum_k x[m, k]^2 / d_i + eps),
// so no CTA needs the whole row before its MMAs: each converts its own slice of u to
// f16 with a power-of-two scale c of its own (max |u c| in [2^13, 2^14)), and the
// per-split sums of x^2 are added up in the epilogue.
//
// Roles (14 warps):
//   warp 0       TMA: the CTA's codes and E4M3 scales and the LoRA A slice at once
//                (weights; they do not depend on the preceding kernel), then, after
//                the programmatic-dependent-launch wait, the x slice and the w_norm
//                and z slices;
//   warps 10-13  w_norm + z; A bf16 -> f16 in place; token rows of x from a shared
//                queue (sum of squares and max |u| of the row, then u c -> f16 in
//                place; the row sums go to every CTA of the cluster); then lane 0 of
//                each issues tcgen05.mma kind::f16 into its own accumulator (a single
//                issuing thread is latency-bound on these small MMAs): D1 += W_hat/s_g (tensor
//                memory) x u^T over even / odd K steps as the chunks are dequantised,
//                and Dt^T += u x A^T (shared memory) over even / odd K steps at once;
//                warps 12-13 then round t = Dt lambda / s_g to bf16 into shared memory
//                and the D1 issuer adds the up-projection as one more K step,
//                D1 += B t^T (bf16 operands, B as stored);
//   warps 2-9    B rows of the tile into shared memory (bf16); dequantise chunks
//                into two or three tensor-memory buffers (E2M1 -> f16 conversion,
//                times the block scale: exact in f16), take token rows from the
//                queue when the buffers are full, then the epilogue;
//   warp 1       tensor-memory allocation.
// Epilogue: each CTA's partial P = rs s_g D1 / c already holds its share of the LoRA
// path (by linearity the splits' B t_s add up to B t; rs is formed by warps 12-13 from
// every split's row sums, which arrive during the row conversion); it sends P, eight
// tokens at a time, with st.async into the shared memory of the peer that owns the
// row (peer p owns rows [128 p / S, 128 (p+1) / S)).  Each CTA sums what it owns in
// split order (deterministic) and writes y.
// The receive buffers have a region of their own when shared memory allows (then no
// cluster barrier comes between the MMAs and the exchange), else they lie over the
// stage region, after a cluster barrier.
//
// Every mbarrier wait is bounded (200 ms).  A wait that gives up sets the status word;
// the CTA still takes part in every cluster barrier and still sends its (then
// meaningless) share, so that no peer waits on it for ever, drains its own copies,
// frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace pl {

__device__ uint32_t g_fused_status = 0;

// Phase timestamps for development builds (-DPL_TIMELINE); compiled out otherwise.
#ifdef PL_TIMELINE
__device__ unsigned long long g_tl_fused[1024][64];
#define PL_TLF(slot) do { if (blockIdx.x < 1024) g_tl_fused[blockIdx.x][slot] = globaltimer_ns(); } while (0)
#else
#define PL_TLF(slot) do { } while (0)
#endif

namespace {

constexpr int kTileO = 128;
constexpr int kChunkK = 256;
constexpr int kCodesBytes = kTileO * kChunkK / 2;   // 16 KB
constexpr int kScaleBytes = kTileO * kChunkK / 16;  // 2 KB
constexpr int kMaxChunks = 3;
constexpr int kMaxSplit = 8;
constexpr int kMaxN = 64;
constexpr int kMaxRFused = 32;  // LoRA rank this kernel takes (B rows are held in registers)
constexpr int kDeqWarps = 8;
constexpr int kAcc = 2;  // D1 accumulators, each with its own issuing thread (even / odd K steps)
constexpr int kConvWarps = 4;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kEpiThreads = kDeqWarps * 32;
constexpr int kThreads = (2 + kDeqWarps + kConvWarps) * 32;  // 448
constexpr int kConvWarp0 = 2 + kDeqWarps;                    // first conversion warp
constexpr uint32_t kTmemCols = 512;
constexpr size_t kMinSmem = 120 * 1024;  // > half an SM: one CTA per SM, so its 512 TMEM columns are free

struct FParams {
  int64_t M, d_i, d_o;
  int N, Np, Mp, rb, r, S, kc, rows_max, nbuf;
  float lambda, eps, inv_d;
  const float* s_g;
  const float* w_norm;
  const float* z;
  const __nv_bfloat16* B;
  void* y;
  int y_f32;
  // shared-memory layout (byte offsets from the 1 KB-aligned base)
  uint32_t off_scales, off_x, off_a, off_gw, off_gz, off_q, off_ctrl;
  uint32_t off_rp;          // partial-output receive buffers
  uint32_t off_bq, off_tq;  // LoRA up-projection operands: B of the tile [128][64], t [N][64] (bf16, SW128)
  int alias_recv;           // 1: the receive buffers lie over the stage region (cluster barrier first)
  int lora_in_a;            // 1: the up-projection operands lie over the A slabs (written once Dt is done)
};

struct FMaps {
  CUtensorMap codes, scales, x, a;
};

struct Ctrl {
  uint64_t wfull[kMaxChunks];  // codes + scales of chunk c landed
  uint64_t a_full[kMaxChunks]; // chunk c dequantised into its tensor-memory buffer
  uint64_t a_empty[kMaxChunks]; // the MMAs reading buffer b are done
  uint64_t a_in, x_in, g_in;   // LoRA A slice, x slice, w_norm / z slices landed
  uint64_t g_ready;            // w_norm + z formed
  uint64_t rows_ready;         // every token row converted (one arrival per row)
  uint64_t a16_ready;          // the LoRA A slice converted to f16
  uint64_t dt_full;            // the LoRA down-projection MMAs done
  uint64_t lora_ready;         // B and t of the up-projection in shared memory
  uint64_t d_full;             // every MMA done
  uint64_t recv;               // the peers' partial outputs arrived
  uint64_t q_full;             // the peers' row sums of x^2 arrived
  uint64_t rs_ready;           // rs of every token row formed
  uint32_t tmem_base;
  int abort_flag;
  int next_row;                // token-row queue of the conversion
  alignas(16) float cinv[kMaxN];  // 1 / c of this split, per token row
  float rs[kMaxN];
};

__device__ __noinline__ bool wait_f_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return wait_or_abort_status(bar, parity, abort_flag, &g_fused_status);
}
// Bounded wait: the common case (already complete) inline, the polling loop out of line.
PL_DEVINL bool wait_f(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_try_wait(bar, parity) || wait_f_slow(bar, parity, abort_flag);
}
PL_DEVINL uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
PL_DEVINL void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
PL_DEVINL void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
PL_DEVINL void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
PL_DEVINL void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// 16 bytes into a peer's shared memory, completing 16 bytes of its mbarrier's transaction.
PL_DEVINL void st_async_f32x4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
               :: "r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar) : "memory");
}
PL_DEVINL void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
               :: "r"(addr), "r"(__float_as_uint(v)), "r"(bar) : "memory");
}
// One contiguous global -> shared copy (16-byte aligned, size a multiple of 16).
PL_DEVINL void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// First weight row of the share that CTA `s` of the cluster owns.
PL_DEVINL int owner_row0(int s, int S) { return (s * kTileO) / S; }

// Token rows of x (one warp): sum of squares and max |u| over this CTA's slice, then
// u c -> f16 in place.  Rows come two at a time from a queue shared by the conversion
// and dequant warps.  Lane l takes the 16-byte pieces l, l + 32, ... of a row (piece q:
// slab q / 8, column q % 8; one piece per lane per chunk), so its eight values of
// w_norm + z per piece stay in registers for every row, and the row's pieces stay in
// registers between the two passes.  Out of line: it is called from two roles.
__device__ __noinline__ void convert_rows_warp(uint8_t* smem, uint32_t off_x, const float* gsh, float* qrecv, Ctrl* C,
                                               int N, int nslab, int M, int S, int me, bool norm,
                                               volatile int* abort_flag) {
  constexpr int kRows = 1;
  const int lane = threadIdx.x & 31;
  const int nk = nslab / 4;  // pieces per lane: one per chunk
  const int ch = lane & 7;
  float g[kMaxChunks][8];
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    float4 ga = make_float4(1.f, 1.f, 1.f, 1.f), gb = ga;
    if (norm && k < nk) {
      const float4* g4 = reinterpret_cast<const float4*>(gsh) + (lane + 32 * k) * 2;
      ga = g4[0];
      gb = g4[1];
    }
    g[k][0] = ga.x; g[k][1] = ga.y; g[k][2] = ga.z; g[k][3] = ga.w;
    g[k][4] = gb.x; g[k][5] = gb.y; g[k][6] = gb.z; g[k][7] = gb.w;
  }
  // byte offset of this lane's piece k within a row n: slab (lane + 32 k) / 8, column ch
  auto piece = [&](int n, int k) {
    return off_x + static_cast<uint32_t>(n * 128 + ((lane >> 3) + 4 * k) * N * 128 + ((ch ^ (n & 7)) << 4));
  };
  const uint32_t q_bar = smem_u32(&C->q_full);
  for (;;) {
    int base = 0;
    if (lane == 0) base = atomicAdd(&C->next_row, kRows);
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (base >= M || *abort_flag) break;
    uint4 v[kRows][kMaxChunks];
    float ss[kRows], mx[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int n = base + r;
      ss[r] = 0.f;
      mx[r] = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxChunks; ++k) {
        v[r][k] = make_uint4(0u, 0u, 0u, 0u);
        if (k < nk && n < M) v[r][k] = *reinterpret_cast<const uint4*>(smem + piece(n, k));
        const uint32_t w[4] = {v[r][k].x, v[r][k].y, v[r][k].z, v[r][k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = bf16lo_to_f32(w[i]), x1 = bf16hi_to_f32(w[i]);
          ss[r] = fmaf(x0, x0, fmaf(x1, x1, ss[r]));
          mx[r] = fmaxf(mx[r], fmaxf(fabsf(x0 * g[k][2 * i]), fabsf(x1 * g[k][2 * i + 1])));
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        ss[r] += __shfl_xor_sync(0xFFFFFFFFu, ss[r], o);
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], o));
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int n = base + r;
      if (n >= M) continue;
      // c = 2^e with max |u| c in [2^13, 2^14): e from the exponent field of max |u|
      const int ex = static_cast<int>((__float_as_uint(mx[r]) >> 23) & 0xFFu) - 127;
      int e = mx[r] > 0.f ? 13 - ex : 0;
      e = e < -100 ? -100 : (e > 100 ? 100 : e);
      const float cs = __int_as_float((127 + e) << 23);
#pragma unroll
      for (int k = 0; k < kMaxChunks; ++k) {
        if (k < nk) {
          const uint32_t w[4] = {v[r][k].x, v[r][k].y, v[r][k].z, v[r][k].w};
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            o[i] = f32x2_to_f16x2(bf16lo_to_f32(w[i]) * (g[k][2 * i] * cs), bf16hi_to_f32(w[i]) * (g[k][2 * i + 1] * cs));
          *reinterpret_cast<uint4*>(smem + piece(n, k)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      if (lane == 0) {
        C->cinv[n] = __int_as_float((127 - e) << 23);
        if (norm) qrecv[me * N + n] = ss[r];
      } else if (norm && lane < S) {  // the row's sum of squares to every peer
        const uint32_t dst = static_cast<uint32_t>((me + lane) % S);
        st_async_f32(mapa_shared(smem_u32(&qrecv[me * N + n]), dst), ss[r], mapa_shared(q_bar, dst));
      }
    }
    fence_proxy_async_smem();  // the f16 operands are read by the tensor cores
    __syncwarp();
    if (lane == 0) {
      const int live = M - base < kRows ? M - base : kRows;
      for (int r = 0; r < live; ++r) mbar_arrive(smem_u32(&C->rows_ready));
    }
  }
  if (lane == 0) PL_TLF(32 + (threadIdx.x >> 5));
}

// The K steps q, q + Q, ... of one chunk (16 steps of 16): D (+)= W_hat/s_g (tensor
// memory, 8 columns per step) x u^T (shared memory; 2 units of 16 B per step, one slab
// per 4 steps).
template <int Q>
PL_DEVINL void mma_d1_chunk(uint32_t dtm, uint32_t abuf, uint64_t xc, uint32_t xslab, uint32_t idesc, int q,
                            bool first) {
#pragma unroll
  for (int i = 0; i < (kChunkK / 16 + Q - 1) / Q; ++i) {
    const int kk = q + Q * i;
    if (kk < kChunkK / 16)
      mma_ts(dtm, abuf + 8u * kk, xc + static_cast<uint64_t>((kk >> 2) * xslab + 2u * (kk & 3)), idesc,
             (!first || i > 0) ? 1u : 0u);
  }
}

// D1 issuer q of kAcc (one thread): K steps q, q + kAcc, ... of every chunk as it is
// dequantised, into accumulator q (a single issuing thread is latency-bound on these
// small MMAs); issuer 0 then adds the LoRA up-projection (rank rb, 0 for none) as one
// more K step.  Out of line: it is called from two warps.
__device__ __noinline__ void issue_d1_thread(Ctrl& C, int q, int nch, int nbuf, int N, int rb,
                                             uint32_t tmem, uint32_t col_d1, uint32_t x_addr, uint32_t bq_addr,
                                             uint32_t tq_addr, volatile int* abort_flag) {
  const uint32_t dtm = tmem + col_d1 + static_cast<uint32_t>(q * N);
  const uint64_t xd0 = smem_desc_sw128(x_addr, 1024);
  const uint32_t xslab = static_cast<uint32_t>(N) * 8u;  // one 64-element slab of u, in 16-byte units
  const uint32_t idesc = idesc_f16(kTileO, N, 0);
  bool go = wait_f(smem_u32(&C.rows_ready), 0, abort_flag);
  if (q == 0) PL_TLF(15);
  for (int c = 0; c < nch && go; ++c) {
    go = wait_f(smem_u32(&C.a_full[c]), 0, abort_flag);
    if (!go) break;
    if (q == 0) PL_TLF(23 + c);
    tc_fence_after();
    const uint64_t xc = xd0 + static_cast<uint64_t>(4u * c * xslab);
    const uint32_t ab = tmem + 128u * (c % nbuf);
    mma_d1_chunk<kAcc>(dtm, ab, xc, xslab, idesc, q, c == 0);
    if (q == 0) PL_TLF(26 + c);
    if (c + nbuf < nch) tc_commit(smem_u32(&C.a_empty[c % nbuf]));  // buffer reused by chunk c + nbuf
  }
  if (rb > 0 && q == 0 && go) {
    // the LoRA up-projection as one more K step: B (bf16, as stored) times
    // t = Dt lambda / s_g (bf16), which is lambda B A u in the units of D1
    go = wait_f(smem_u32(&C.lora_ready), 0, abort_flag);
    if (go) {
      tc_fence_after();
      const uint32_t idesc_l = idesc_f16(kTileO, N, 1);
      const uint64_t bd = smem_desc_sw128(bq_addr, 1024);
      const uint64_t td = smem_desc_sw128(tq_addr, 1024);
      for (int k = 0; k < rb / 16; ++k) mma_ss(dtm, bd + 2u * k, td + 2u * k, idesc_l, 1u);
    }
  }
  tc_commit(smem_u32(&C.d_full));  // also reached on abort: tracks every MMA issued
  if (q == 0) PL_TLF(8);
}

// The staged LoRA A slice, bf16 -> f16 in place (16 bytes per step; `who` of `nthreads`).
__device__ __noinline__ bool convert_a(uint8_t* a, uint32_t bytes, int who, int nthreads, uint32_t a_in,
                                       volatile int* abort_flag) {
  if (!wait_f(a_in, 0, abort_flag)) return false;
  uint4* a4 = reinterpret_cast<uint4*>(a);
  for (int i = who; i < static_cast<int>(bytes / 16); i += nthreads) {
    const uint4 v = a4[i];
    a4[i] = make_uint4(f32x2_to_f16x2(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x)),
                       f32x2_to_f16x2(bf16lo_to_f32(v.y), bf16hi_to_f32(v.y)),
                       f32x2_to_f16x2(bf16lo_to_f32(v.z), bf16hi_to_f32(v.z)),
                       f32x2_to_f16x2(bf16lo_to_f32(v.w), bf16hi_to_f32(v.w)));
  }
  return true;
}

__global__ void __launch_bounds__(kThreads, 1) k_fused_decode(const __grid_constant__ FMaps maps, const FParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl& C = *reinterpret_cast<Ctrl*>(smem + p.off_ctrl);
  volatile int* abort_flag = &C.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S, N = p.N;
  const int M = static_cast<int>(p.M);
  const int me = static_cast<int>(cluster_rank());
  const int tile = blockIdx.x / S;
  const int c0 = (me * p.kc) / S, c1 = ((me + 1) * p.kc) / S;
  const int nch = c1 - c0;
  const int nslab = nch * 4;  // 64-element k slabs of this CTA
  const bool lora = p.r > 0, norm = p.w_norm != nullptr, noise = norm && p.z != nullptr;
  const int R0 = owner_row0(me, S), rows_own = owner_row0(me + 1, S) - R0;
  const int32_t row0 = tile * kTileO;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t x_bytes = static_cast<uint32_t>(nslab) * N * 128u;
  const uint32_t a_bytes = static_cast<uint32_t>(nslab) * p.rb * 128u;
  const uint32_t g_bytes = static_cast<uint32_t>(nch) * kChunkK * 4u;
  const int nbuf = p.nbuf;  // tensor-memory weight buffers (2 or 3) of 128 columns
  const uint32_t colD1 = 128u * nbuf, colDta = colD1 + kAcc * N, colDtb = colDta + p.rb;

  if (threadIdx.x == 0) {
    PL_TLF(0);
    pdl_launch_dependents();
    for (int c = 0; c < kMaxChunks; ++c) {
      mbar_init(smem_u32(&C.wfull[c]), 1);
      mbar_init(smem_u32(&C.a_full[c]), kDeqWarps);
    }
    for (int b = 0; b < kMaxChunks; ++b) mbar_init(smem_u32(&C.a_empty[b]), kAcc);  // the D1 issuers
    mbar_init(smem_u32(&C.a_in), 1);
    mbar_init(smem_u32(&C.x_in), 1);
    mbar_init(smem_u32(&C.g_in), 1);
    mbar_init(smem_u32(&C.g_ready), kConvWarps);
    mbar_init(smem_u32(&C.rows_ready), M);
    mbar_init(smem_u32(&C.a16_ready), kConvWarps + 1);  // + warp 1 (its share of A)
    mbar_init(smem_u32(&C.dt_full), 2);
    mbar_init(smem_u32(&C.lora_ready), 4 + 2);  // 4 dequant warps (B), 2 conversion warps (t)
    mbar_init(smem_u32(&C.d_full), kAcc);
    mbar_init(smem_u32(&C.recv), 1);
    mbar_init(smem_u32(&C.q_full), 1);
    mbar_init(smem_u32(&C.rs_ready), 2);  // warps kConvWarp0 + 2, + 3
    fence_mbar_init();
    mbar_arrive_expect_tx(smem_u32(&C.q_full), norm ? static_cast<uint32_t>((S - 1) * M * 4) : 0u);
    PL_TLF(16);
    const uint64_t pol = policy_evict_first();  // weights are streamed once
    for (int c = 0; c < nch; ++c) {
      const uint32_t wb = smem_u32(&C.wfull[c]);
      mbar_arrive_expect_tx(wb, kCodesBytes + kScaleBytes);
      tma_load_2d_hint(sbase + c * kCodesBytes, &maps.codes, (c0 + c) * (kChunkK / 2), row0, wb, pol);
      tma_load_2d_hint(sbase + p.off_scales + c * kScaleBytes, &maps.scales, (c0 + c) * (kChunkK / 16), row0, wb,
                       pol);
    }
    PL_TLF(17);
    if (lora) {
      const uint32_t ab = smem_u32(&C.a_in);
      mbar_arrive_expect_tx(ab, a_bytes);
      for (int j = 0; j < nslab; ++j)
        tma_load_2d(sbase + p.off_a + j * p.rb * 128, &maps.a, c0 * kChunkK + 64 * j, 0, ab);
    }
    tma_prefetch_desc(&maps.x);
    C.abort_flag = 0;
    C.next_row = 0;
    PL_TLF(18);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&C.tmem_base), kTmemCols);
    tmem_relinquish();
    if (lane == 0) PL_TLF(19);
  }
  if (threadIdx.x >= 64 && threadIdx.x < 64 + kMaxN) C.cinv[threadIdx.x - 64] = 1.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) PL_TLF(20);
  // every CTA's barriers are initialised before any peer touches them (the init fence
  // above orders the initialisation; the arrive itself need not)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  cluster_wait();
  const uint32_t tmem = C.tmem_base;
  if (threadIdx.x == 0) PL_TLF(1);

  float* qrecv = reinterpret_cast<float*>(smem + p.off_q);  // [S][N]: sums of x^2 of every split
  const float* gsh = reinterpret_cast<const float*>(smem + p.off_gw);

  auto convert_rows = [&]() {
    convert_rows_warp(smem, p.off_x, gsh, qrecv, &C, N, nslab, M, S, me, norm, abort_flag);
  };

  auto issue_d1 = [&](int q) {
    issue_d1_thread(C, q, nch, nbuf, N, lora ? p.rb : 0, tmem, colD1, sbase + p.off_x, sbase + p.off_bq,
                    sbase + p.off_tq, abort_flag);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      pdl_wait();  // x, w_norm and z may come from the preceding kernel
      PL_TLF(2);
      const uint32_t xb = smem_u32(&C.x_in);
      mbar_arrive_expect_tx(xb, x_bytes);
      for (int j = 0; j < nslab; ++j) tma_load_2d(sbase + p.off_x + j * N * 128, &maps.x, c0 * kChunkK + 64 * j, 0, xb);
      const int64_t k0 = static_cast<int64_t>(c0) * kChunkK;
      if (norm) {
        const uint32_t gb = smem_u32(&C.g_in);
        mbar_arrive_expect_tx(gb, noise ? 2 * g_bytes : g_bytes);
        bulk_g2s(sbase + p.off_gw, p.w_norm + k0, g_bytes, gb);
        if (noise) bulk_g2s(sbase + p.off_gz, p.z + k0, g_bytes, gb);
      }
      // every copy lands before the stage region is handed to the peers
      for (int c = 0; c < nch; ++c) drain(smem_u32(&C.wfull[c]), 0);
      if (lora) drain(smem_u32(&C.a_in), 0);
      if (norm) drain(smem_u32(&C.g_in), 0);
      drain(xb, 0);
    }
    __syncwarp();
    if (p.alias_recv) {
      cluster_arrive();
      cluster_wait();
    }
    cluster_arrive_relaxed();
  } else if (warp == 1) {
    if (lora) convert_a(smem + p.off_a, a_bytes, kConvThreads + lane, kConvThreads + 32, smem_u32(&C.a_in), abort_flag);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&C.a16_ready));
    if (p.alias_recv) {
      cluster_arrive();
      cluster_wait();
    }
    cluster_arrive_relaxed();
  } else if (warp >= kConvWarp0) {
    // ---------------------------------------------------------------- activations, then MMA issue
    const int cw = warp - kConvWarp0;              // 0..3
    const int ct = threadIdx.x - kConvWarp0 * 32;  // 0..127
    static_assert((kConvWarp0 + 2) % 4 == 0, "warps kConvWarp0 + 2, + 3 hold tensor-memory lanes 0-63");
    bool ok = true;
    if (lora)  // A lands early (a weight): convert it while x is still on its way
      ok = convert_a(smem + p.off_a, a_bytes, ct, kConvThreads + 32, smem_u32(&C.a_in), abort_flag);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&C.a16_ready));
    if (ct == 0) PL_TLF(21);
    if (norm) {
      ok = wait_f(smem_u32(&C.g_in), 0, abort_flag) && ok;
      if (noise) {
        float4* gw = reinterpret_cast<float4*>(smem + p.off_gw);
        const float4* gz = reinterpret_cast<const float4*>(smem + p.off_gz);
        for (int k4 = ct; k4 < nch * kChunkK / 4; k4 += kConvThreads) {
          float4 a = gw[k4];
          const float4 b = gz[k4];
          a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
          gw[k4] = a;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&C.g_ready));
    if (ct == 0) PL_TLF(3);
    ok = wait_f(smem_u32(&C.g_ready), 0, abort_flag) && wait_f(smem_u32(&C.x_in), 0, abort_flag) && ok;
    if (ct == 0) PL_TLF(4);
    convert_rows();  // also fences and arrives on rows_ready
    if (ct == 0) PL_TLF(5);
    const bool tpart = cw >= 2;
    if (lane == 0) {
      if (!tpart) {
        issue_d1(cw);  // D1 issuers 0 and 1
      } else if (lora) {
        // the LoRA down-projection needs no weight buffer: all of it at once, even / odd
        // K steps into Dta / Dtb (cw 2 / 3)
        const int par = cw & 1;
        const uint32_t dtm = tmem + (cw == 2 ? colDta : colDtb);
        const uint64_t xd0 = smem_desc_sw128(sbase + p.off_x, 1024) + 2u * par;
        const uint32_t xslab = static_cast<uint32_t>(N) * 8u, aslab = static_cast<uint32_t>(p.rb) * 8u;
        bool go = wait_f(smem_u32(&C.rows_ready), 0, abort_flag) && wait_f(smem_u32(&C.a16_ready), 0, abort_flag);
        const uint32_t idesc = idesc_f16(kTileO, p.rb, 0);
        const uint64_t ad0 = smem_desc_sw128(sbase + p.off_a, 1024) + 2u * par;
        for (int c = 0; c < nch && go; ++c) {
          // A operand: 128 rows of u (rows >= N read bytes of the following slabs and
          // regions, inside this CTA's allocation; they only feed unread lanes)
          const uint64_t xc = xd0 + static_cast<uint64_t>(4u * c * xslab);
          const uint64_t acd = ad0 + static_cast<uint64_t>(4u * c * aslab);
#pragma unroll
          for (int h = 0; h < kChunkK / 32; ++h)
            mma_ss(dtm, xc + (h >> 1) * xslab + 4u * (h & 1), acd + (h >> 1) * aslab + 4u * (h & 1), idesc,
                   (c > 0 || h > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&C.dt_full));
      }
    }
    __syncwarp();
    if (tpart && lora) {
      // t = (Dta + Dtb) lambda / s_g -> bf16, one token row per lane (warps 12 / 13 hold
      // tensor-memory lanes 0-31 / 32-63), K-major 128-byte swizzled rows of 64 elements
      bool tok = wait_f(smem_u32(&C.dt_full), 0, abort_flag);
      tc_fence_after();
      const int n = (cw - 2) * 32 + lane;
      const float lam_sg = __fdividef(p.lambda, *p.s_g);
      uint8_t* tq = smem + p.off_tq + n * 128;
      const uint32_t la = static_cast<uint32_t>((cw - 2) * 32) << 16;
#pragma unroll
      for (int j8 = 0; j8 < kMaxRFused / 8; ++j8) {
        if (j8 * 8 < p.rb) {
          uint32_t a8[8], b8[8];
          tmem_ld8(tmem + la + colDta + j8 * 8, a8);
          tmem_ld8(tmem + la + colDtb + j8 * 8, b8);
          tmem_ld_wait();
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            w[q] = f32x2_to_bf16x2((__uint_as_float(a8[2 * q]) + __uint_as_float(b8[2 * q])) * lam_sg,
                                   (__uint_as_float(a8[2 * q + 1]) + __uint_as_float(b8[2 * q + 1])) * lam_sg);
          if (n < N && tok) *reinterpret_cast<uint4*>(tq + ((j8 ^ (n & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.lora_ready));
    }
    if (tpart) {
      // rs_n = 1 / sqrt(sum over the splits of sum_k x[n, k]^2 / d_i + eps), one token row
      // per lane, once every split's row sums are in (the local ones: rows_ready)
      const bool qok = wait_f(smem_u32(&C.rows_ready), 0, abort_flag) && wait_f(smem_u32(&C.q_full), 0, abort_flag);
      const int n = (cw - 2) * 32 + lane;
      if (n < M) {
        float rs = 1.f;
        if (norm && qok) {
          float tot = 0.f;
          for (int s = 0; s < S; ++s) tot += qrecv[s * N + n];
          asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(rs) : "f"(tot * p.inv_d + p.eps));
        }
        C.rs[n] = rs;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.rs_ready));
    }
    __syncwarp();
    if (p.alias_recv) {
      cluster_arrive();
      cluster_wait();
    }
    cluster_arrive_relaxed();
  } else {
    // ---------------------------------------------------------------- dequant + epilogue
    const int dw = warp - 2;              // 0..7
    const int quarter = warp & 3;         // tensor-memory lane quarter of this warp
    const int g = dw >> 2;                // K half of each chunk
    const int row = quarter * 32 + lane;  // weight row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int et = threadIdx.x - 64;      // 0 .. 255
    const float s_g = *p.s_g;             // a weight input: not written by the preceding kernel
    // B rows of the up-projection operand (K-major, 128-byte swizzled; columns >= r are
    // 0), one row per g == 0 thread, from global memory (a weight)
    auto write_bq = [&](bool wait_dt) {
      if (g == 0) {
        uint32_t bq[kMaxRFused / 2];
#pragma unroll
        for (int j = 0; j < kMaxRFused / 2; ++j) bq[j] = 0u;
        const int64_t o = static_cast<int64_t>(row0) + row;
        if (o < p.d_o) {
          if ((p.r & 7) == 0) {
            const uint4* src = reinterpret_cast<const uint4*>(p.B + o * p.r);
#pragma unroll
            for (int q = 0; q < kMaxRFused / 8; ++q)
              if (8 * q < p.r) {
                const uint4 v = src[q];
                bq[4 * q] = v.x; bq[4 * q + 1] = v.y; bq[4 * q + 2] = v.z; bq[4 * q + 3] = v.w;
              }
          } else {
            const uint16_t* src = reinterpret_cast<const uint16_t*>(p.B + o * p.r);
#pragma unroll
            for (int j = 0; j < kMaxRFused; ++j)
              if (j < p.r) bq[j >> 1] |= static_cast<uint32_t>(src[j]) << (16 * (j & 1));
          }
        }
        // over the A slabs: only once the down-projection is done with them
        const bool w_ok = !wait_dt || wait_f(smem_u32(&C.dt_full), 0, abort_flag);
        uint8_t* bqs = smem + p.off_bq + row * 128;
#pragma unroll
        for (int j8 = 0; j8 < kMaxRFused / 8; ++j8)
          if (j8 * 8 < p.rb && w_ok)
            *reinterpret_cast<uint4*>(bqs + ((j8 ^ (row & 7)) << 4)) =
                make_uint4(bq[4 * j8], bq[4 * j8 + 1], bq[4 * j8 + 2], bq[4 * j8 + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&C.lora_ready));
      }
    };
    if (lora && !p.lora_in_a) write_bq(false);
    bool ok = true, converted = false;
    for (int c = 0; c < nch; ++c) {
      if (c == nbuf) {  // buffer 0 is needed again: help with the activations first
        if (et == 0) PL_TLF(7);
        ok = wait_f(smem_u32(&C.g_ready), 0, abort_flag) && wait_f(smem_u32(&C.x_in), 0, abort_flag) && ok;
        convert_rows();
        converted = true;
      }
      const int b = c % nbuf;
      ok = ok && wait_f(smem_u32(&C.wfull[c]), 0, abort_flag) &&
           (c < nbuf || wait_f(smem_u32(&C.a_empty[b]), 0, abort_flag));
      if (!ok) break;
      if (c == 0 && et == 0) PL_TLF(6);
      const uint8_t* crow = smem + c * kCodesBytes + row * 128;
      const uint2 sc8 = *reinterpret_cast<const uint2*>(smem + p.off_scales + c * kScaleBytes + row * 16 + g * 8);
      const uint32_t sc_words[2] = {sc8.x, sc8.y};
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = 4 * g + jj;  // 16-byte piece of the row (32 codes, 2 scale blocks)
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
        tmem_st16(tmem + lane_addr + 128u * b + j * 16, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.a_full[c]));
    }
    if (!converted) {
      if (et == 0) PL_TLF(7);
      ok = wait_f(smem_u32(&C.g_ready), 0, abort_flag) && wait_f(smem_u32(&C.x_in), 0, abort_flag) && ok;
      convert_rows();
    }
    if (lora && p.lora_in_a) write_bq(true);
    // ---------------------------------------------------------------- epilogue: gather
    ok = wait_f(smem_u32(&C.d_full), 0, abort_flag) && ok;
    if (et == 0) PL_TLF(9);
    tc_fence_after();
    const int half = N / 2, n0 = g * half;  // tokens [n0, n0 + half) of D1 for this thread
    const int Mp = p.Mp;
    // rs_ready also orders the reads of 1 / c: its arrivals follow a wait on rows_ready
    ok = wait_f(smem_u32(&C.rs_ready), 0, abort_flag) && ok;
    const bool good = ok && !*abort_flag;
    if (p.alias_recv) {  // the receive buffers lie over the stage region: every CTA is done with it
      cluster_arrive();
      cluster_wait();
    }
    if (et == 0) PL_TLF(10);
    // ---------------------------------------------------------------- epilogue: exchange
    // P[row, n] = rs_n s_g D1[row, n] / c_n (this split's share of y), 8 tokens at a time,
    // straight into the shared memory of the CTA that owns the row
    const uint32_t recv_bar = smem_u32(&C.recv);
    {
      const int o = ((row + 1) * S - 1) >> 7;  // the owner: owner_row0(o, S) <= row < owner_row0(o + 1, S)
      const int rl = row - owner_row0(o, S);
      const uint32_t dst = sbase + p.off_rp + static_cast<uint32_t>(((me * p.rows_max + rl) * p.Np + n0) * 4);
      const uint32_t rdst = mapa_shared(dst, static_cast<uint32_t>(o)), rbar = mapa_shared(recv_bar, o);
#pragma unroll 1
      for (int i = 0; i < half && n0 + i < Mp; i += 8) {
        uint32_t a8[8], b8[8];
        tmem_ld8(tmem + lane_addr + colD1 + n0 + i, a8);
        tmem_ld8(tmem + lane_addr + colD1 + N + n0 + i, b8);
        tmem_ld_wait();
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int n = n0 + i + j;
          v[j] = good ? C.rs[n] * C.cinv[n] * s_g * (__uint_as_float(a8[j]) + __uint_as_float(b8[j])) : 0.f;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (n0 + i + 4 * h < Mp) {
            const float4 f = make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
            const uint32_t off = static_cast<uint32_t>(4 * (i + 4 * h));
            if (o == me) *reinterpret_cast<float4*>(smem + (dst - sbase) + off) = f;
            else st_async_f32x4(rdst + off, f, rbar);
          }
        }
      }
    }
    if (et == 0) {
      const uint32_t per_peer = static_cast<uint32_t>(rows_own * Mp * 4);
      mbar_arrive_expect_tx(recv_bar, per_peer * static_cast<uint32_t>(S - 1));
      PL_TLF(11);
    }
    named_bar(1, kEpiThreads);  // this CTA's own shares are in place
    ok = wait_f(recv_bar, 0, abort_flag) && good;
    cluster_arrive_relaxed();  // nothing more lands here (released at the exit barrier)
    if (et == 0) PL_TLF(12);
    // ---------------------------------------------------------------- epilogue: combine
    if (ok) {
      const float* rp = reinterpret_cast<const float*>(smem + p.off_rp);
      const int items = rows_own * (Mp / 4);
      for (int e = et; e < items; e += kEpiThreads) {
        const int rl = e % rows_own, n4 = 4 * (e / rows_own);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int s = 0; s < S; ++s) {
          const float4 v = *reinterpret_cast<const float4*>(rp + (s * p.rows_max + rl) * p.Np + n4);
          acc[0] += v.x; acc[1] += v.y; acc[2] += v.z; acc[3] += v.w;
        }
        const int64_t oo = static_cast<int64_t>(row0) + R0 + rl;
        if (oo < p.d_o) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int n = n4 + q;
            if (n < M) {
              const float v = acc[q];
              if (p.y_f32) static_cast<float*>(p.y)[static_cast<int64_t>(n) * p.d_o + oo] = v;
              else static_cast<__nv_bfloat16*>(p.y)[static_cast<int64_t>(n) * p.d_o + oo] = __float2bfloat16_rn(v);
            }
          }
        }
      }
    }
  }
  if (threadIdx.x == 64) PL_TLF(13);
  // no CTA leaves while a peer may still write into its shared memory (also when a
  // bounded wait gave up: every CTA reaches this barrier)
  __syncwarp();
  cluster_wait();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) PL_TLF(14);
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

struct FPlan {
  int N, Np, rb, S, kc, tiles, rows_max, nchmax, alias_recv, lora_in_a;
  uint32_t off_scales, off_x, off_a, off_gw, off_gz, off_q, off_ctrl, off_rp, off_bq, off_tq;
  size_t smem;
};

uint32_t al1k(size_t v) { return static_cast<uint32_t>(align_up(v, 1024)); }

// Shared-memory layout for S splits; false if it does not fit.
bool layout(FPlan& f, int r) {
  const int nslab = f.nchmax * 4;
  f.off_scales = static_cast<uint32_t>(f.nchmax * kCodesBytes);
  f.off_x = al1k(f.off_scales + static_cast<size_t>(f.nchmax) * kScaleBytes);
  f.off_a = al1k(f.off_x + static_cast<size_t>(nslab) * f.N * 128);
  f.off_gw = al1k(f.off_a + static_cast<size_t>(nslab) * f.rb * 128);
  f.off_gz = f.off_gw + f.nchmax * kChunkK * 4;
  f.off_q = f.off_gz + f.nchmax * kChunkK * 4;
  f.off_ctrl = f.off_q + static_cast<uint32_t>(align_up(static_cast<size_t>(f.S) * f.N * 4, 16));
  f.off_ctrl = static_cast<uint32_t>(align_up(f.off_ctrl, 128));
  size_t end = f.off_ctrl + sizeof(Ctrl);
  // the LoRA-down MMA reads 128 rows of every u slab (rows >= N are don't-care)
  const size_t read_end = f.off_x + static_cast<size_t>(nslab - 1) * f.N * 128 + 128 * 128;
  if (end < read_end) end = read_end;
  // Two buffers may have a region of their own or share one:
  //  - the LoRA up-projection operands (B [128][64] and t [N][64], bf16): own region, or
  //    over the A slabs, which are free once the down-projection is done;
  //  - the partial-output receive buffers P [S][rows_max][Np]: own region (peers may send
  //    as soon as they are done), or over the stage region, which every CTA of the
  //    cluster must have finished with first.
  const size_t base = align_up(end, 1024);
  const size_t lora_bytes = r > 0 ? static_cast<size_t>(kTileO) * 128 + align_up(static_cast<size_t>(f.N) * 128, 1024) : 0;
  const size_t a_region = f.off_gw - f.off_a;
  const size_t rp_bytes = static_cast<size_t>(f.S) * f.rows_max * f.Np * 4;
  bool placed = false;
  for (int opt = 0; opt < 4 && !placed; ++opt) {
    const bool l_in_a = opt == 1 || opt == 2, rp_alias = opt >= 2;
    if (l_in_a && (r == 0 || lora_bytes > a_region)) continue;
    if (rp_alias && rp_bytes > f.off_gw) continue;
    size_t e = base;
    f.off_bq = f.off_tq = 0;
    if (r > 0) {
      const size_t lb = l_in_a ? f.off_a : e;
      f.off_bq = static_cast<uint32_t>(lb);
      f.off_tq = static_cast<uint32_t>(lb + static_cast<size_t>(kTileO) * 128);
      if (!l_in_a) e += lora_bytes;
    }
    f.off_rp = rp_alias ? 0u : static_cast<uint32_t>(e);
    if (!rp_alias) e += rp_bytes;
    if (e + 1024 > 227 * 1024) continue;  // + alignment slack
    f.lora_in_a = l_in_a ? 1 : 0;
    f.alias_recv = rp_alias ? 1 : 0;
    f.smem = e + 1024;
    if (f.smem < kMinSmem) f.smem = kMinSmem;
    placed = true;
  }
  // tensor memory: 2 weight buffers of 128 columns, D1 twice (N), Dt twice (rb)
  const bool tmem_ok = 256 + 2 * f.N + 2 * f.rb <= static_cast<int>(kTmemCols);
  return placed && tmem_ok;
}

int max_active_clusters(size_t smem, int cs) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(cs * 64));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(cs);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_fused_decode, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  return n;
}

cudaError_t set_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(k_fused_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  return err;
}

// Split count S: the largest (at most 8) for which the grid is one wave on the SMs,
// every CTA's slice is at most 3 chunks, shared memory fits and all clusters can be
// resident at once; none -> this path does not apply.
bool make_plan(int64_t M, int64_t d_i, int64_t d_o, int r, FPlan& out) {
  if (M < 1 || M > kMaxN || d_i < kChunkK || d_i % kChunkK != 0 || r < 0 || r > kMaxRFused || d_o < 1) return false;
  FPlan f{};
  f.N = static_cast<int>((M + 15) / 16 * 16);
  f.Np = f.N + 4;
  f.rb = r > 0 ? (r + 15) / 16 * 16 : 16;
  f.kc = static_cast<int>(d_i / kChunkK);
  const int64_t tiles = (d_o + kTileO - 1) / kTileO;
  if (tiles > 4096) return false;
  f.tiles = static_cast<int>(tiles);
  if (set_attributes() != cudaSuccess) return false;
  const int smin = (f.kc + kMaxChunks - 1) / kMaxChunks;
  const int smax = f.kc < kMaxSplit ? f.kc : kMaxSplit;
  for (int S = smax; S >= smin; --S) {
    if (static_cast<int64_t>(f.tiles) * S > sm_count()) continue;
    FPlan g = f;
    g.S = S;
    g.nchmax = (f.kc + S - 1) / S;
    g.rows_max = (kTileO + S - 1) / S;
    if (!layout(g, r)) continue;
    if (max_active_clusters(g.smem, S) < f.tiles) continue;
    out = g;
    return true;
  }
  return false;
}

struct PlanKey {
  int64_t M, d_i, d_o;
  int r;
  int dev;
};
struct PlanEntry {
  PlanKey k;
  bool ok;
  FPlan f;
};

bool cached_plan(int64_t M, int64_t d_i, int64_t d_o, int r, FPlan& out) {
  static std::mutex mu;
  static PlanEntry cache[64];
  static int used = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < used; ++i) {
    const PlanKey& k = cache[i].k;
    if (k.M == M && k.d_i == d_i && k.d_o == d_o && k.r == r && k.dev == dev) {
      out = cache[i].f;
      return cache[i].ok;
    }
  }
  FPlan f{};
  const bool ok = make_plan(M, d_i, d_o, r, f);
  PlanEntry& e = cache[used < 64 ? used++ : (used = 1, 0)];
  e.k = PlanKey{M, d_i, d_o, r, dev};
  e.ok = ok;
  e.f = f;
  out = f;
  return ok;
}

}  // namespace

bool fused_supported(int64_t M, int64_t d_i, int64_t d_o, int r) {
  FPlan f;
  return cached_plan(M, d_i, d_o, r, f);
}

cudaError_t launch_linear_fused(const LinearArgs& a, cudaStream_t stream) {
  FPlan f;
  if (!cached_plan(a.M, a.d_i, a.d_o, a.r, f)) return cudaErrorInvalidValue;
  FMaps maps;
  bool ok = encode_2d(&maps.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, a.d_i / 2, a.d_o, 128, kTileO,
                      CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&maps.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.scales, a.d_i / 16, a.d_o, 16, kTileO,
                      CU_TENSOR_MAP_SWIZZLE_NONE) &&
            encode_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.x, a.d_i, a.M, 64, f.N,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok && a.r > 0)
    ok = encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.A, a.d_i, a.r, 64, f.rb,
                   CU_TENSOR_MAP_SWIZZLE_128B);
  else
    maps.a = maps.x;  // unused
  if (!ok) return cudaErrorInvalidValue;

  FParams p{};
  p.M = a.M;
  p.d_i = a.d_i;
  p.d_o = a.d_o;
  p.N = f.N;
  p.Np = f.Np;
  p.Mp = static_cast<int>((a.M + 3) / 4 * 4);
  p.rb = f.rb;
  p.r = a.r;
  p.S = f.S;
  p.kc = f.kc;
  p.rows_max = f.rows_max;
  // tensor memory: nbuf weight buffers of 128 columns, D1 twice (N), Dt twice (rb)
  p.nbuf = 384 + 2 * f.N + 2 * f.rb <= static_cast<int>(kTmemCols) ? 3 : 2;
  p.lambda = a.lambda;
  p.eps = a.eps;
  p.inv_d = 1.0f / static_cast<float>(a.d_i);
  p.s_g = a.s_g;
  p.w_norm = a.w_norm;
  p.z = a.z;
  p.B = static_cast<const __nv_bfloat16*>(a.B);
  p.y = a.y;
  p.y_f32 = a.y_f32 ? 1 : 0;
  p.off_scales = f.off_scales;
  p.off_x = f.off_x;
  p.off_a = f.off_a;
  p.off_gw = f.off_gw;
  p.off_gz = f.off_gz;
  p.off_q = f.off_q;
  p.off_ctrl = f.off_ctrl;
  p.off_rp = f.off_rp;
  p.off_bq = f.off_bq;
  p.off_tq = f.off_tq;
  p.alias_recv = f.alias_recv;
  p.lora_in_a = f.lora_in_a;

  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = static_cast<unsigned>(f.S);
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t c{};
  c.gridDim = dim3(static_cast<unsigned>(f.tiles * f.S));
  c.blockDim = dim3(kThreads);
  c.dynamicSmemBytes = f.smem;
  c.stream = stream;
  c.attrs = attrs;
  c.numAttrs = 2;
  return cudaLaunchKernelEx(&c, k_fused_decode, maps, p);
}

#ifdef PL_TIMELINE
extern "C" int pl_debug_read_timeline_fused(unsigned long long* out) {
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  return cudaMemcpyFromSymbol(out, g_tl_fused, sizeof(g_tl_fused)) != cudaSuccess ? 2 : 0;
}
#endif

uint32_t fused_read_and_clear_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_fused_status, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_fused_status, &zero, sizeof(zero));
  return v;
}

}  // namespace pl
