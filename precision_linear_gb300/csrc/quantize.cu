// NVFP4 quantiser: tensor amax -> per-16-block E4M3 scale -> E2M1 codes, packed.
//
// Source: "QeRL: When Quantized Weights Help Reinforcement Learning, and Where the
// Evidence Stops", section 3.1 (E2M1 grid, one E4M3 scale per 16 weights, FP32
// tensor scale, reconstruction w_hat = s_g s_b q and argmin q = argmin|w - s_g s_b q|)
// and step 4-5 of its backbone-preparation algorithm (quantise, pack).
//
// Arithmetic contract (FP32, round to nearest even), bit-exact with the oracle:
//   s_g  = amax_t / 2688           (1 if amax_t == 0)
//   s_b  = E4M3_satfinite( amax_b / (6 * s_g) )
//   S    = s_g * s_b
//   code = E2M1_satfinite( |w| / S ) with the sign of w, +0 for magnitude 0, 0 if S == 0.
//
// Three launches after a 4-byte memset of s_g:
//   k_amax     grid-stride max|w| over the BF16 words; atomicMax of the FP32 bit
//              pattern into s_g (non-negative floats order like their bits).
//   k_quant    one thread per 16-weight block: 32-byte load, block amax, scale,
//              codes, 8-byte + 1-byte stores (a warp moves 1 KB in, 288 B out).
//   k_finalize turns the accumulated amax into s_g in place.
//
// The UAQ fold (invariant scaling, "QuRL" reading notes, section 3: W X = (W / s)(s X))
// quantises W' = fp32(W / s) instead: the same three kernels with kFold, which divide
// every loaded weight by s (IEEE division) and derive the tensor and block scales from
// fp32(amax / s) -- equal to the maximum of the divided values, since rounding a quotient
// by a positive s is monotone.
//
// The quotient |w|/S decides a code only through which E2M1 rounding interval it
// falls in.  k_quant therefore evaluates |w| * (1/S) scaled by (1 -+ 2^-21), a band
// that provably brackets the correctly rounded quotient (reciprocal and products
// each add at most 2^-24 relative error); when both ends give the same code that
// code is the contract's.  Only when a threshold falls inside the band (rare) does
// the block redo its codes with the IEEE division __fdiv_rn.
#include "common.cuh"

namespace pl {
namespace {

constexpr int kThreads = 256;

PL_DEVINL uint32_t absmax_bf16x2(uint32_t w) {
  return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu);
}

__global__ void __launch_bounds__(kThreads) k_amax(const uint4* __restrict__ W, size_t n_vec,
                                                   uint32_t* __restrict__ amax_bits) {
  uint32_t m = 0;
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
  for (; i + 3 * stride < n_vec; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcs(W + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      m = max(m, max(max(absmax_bf16x2(v[u].x), absmax_bf16x2(v[u].y)),
                     max(absmax_bf16x2(v[u].z), absmax_bf16x2(v[u].w))));
  }
  for (; i < n_vec; i += stride) {
    uint4 v = __ldcs(W + i);
    m = max(m, max(max(absmax_bf16x2(v.x), absmax_bf16x2(v.y)),
                   max(absmax_bf16x2(v.z), absmax_bf16x2(v.w))));
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < kThreads / 32 ? red[threadIdx.x] : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (threadIdx.x == 0 && m != 0) atomicMax(amax_bits, m << 16);  // bf16 -> f32 bits
  }
}

PL_DEVINL float tensor_scale_from_amax(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
}

// Clear the sign of every nibble whose magnitude is 0 (no -0 codes).
PL_DEVINL uint32_t drop_negative_zero(uint32_t w) {
  const uint32_t mag = w & 0x77777777u;
  const uint32_t nz = (mag | (mag >> 1) | (mag >> 2)) & 0x11111111u;
  return mag | (w & (nz << 3));
}

// Codes of 16 values f[] scaled by `y` (f * y rounded in FP32, then E2M1).
PL_DEVINL void codes16(const float (&f)[16], float y, uint32_t& w0, uint32_t& w1) {
  uint32_t b[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) b[p] = cvt_e2m1x2(__fmul_rn(f[2 * p + 1], y), __fmul_rn(f[2 * p], y));
  w0 = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  w1 = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
}

template <bool kFold>
__global__ void __launch_bounds__(kThreads) k_quant(const uint4* __restrict__ W, size_t n_blocks,
                                                    const uint32_t* __restrict__ amax_bits,
                                                    uint2* __restrict__ codes,
                                                    uint8_t* __restrict__ scales, float fold_s) {
  float amax_t = __uint_as_float(*amax_bits);
  if constexpr (kFold) amax_t = __fdiv_rn(amax_t, fold_s);
  const float s_g = tensor_scale_from_amax(amax_t);
  const float six_sg = __fmul_rn(6.0f, s_g);
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  for (size_t b = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; b < n_blocks; b += stride) {
    const uint4 v0 = __ldcs(W + 2 * b), v1 = __ldcs(W + 2 * b + 1);
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
    uint32_t am = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[2 * i] = bf16lo_to_f32(u[i]);
      f[2 * i + 1] = bf16hi_to_f32(u[i]);
      am = max(am, absmax_bf16x2(u[i]));
    }
    float amax_b = __uint_as_float(am << 16);
    if constexpr (kFold) {
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = __fdiv_rn(f[i], fold_s);
      amax_b = __fdiv_rn(amax_b, fold_s);
    }
    const float t = __fdiv_rn(amax_b, six_sg);
    const uint32_t sb = cvt_e4m3x2(0.0f, t) & 0xFFu;
    const float S = __fmul_rn(s_g, e4m3_to_f32(sb));
    uint32_t w0 = 0, w1 = 0;
    if (S != 0.0f) {
      bool exact = !(S >= 0x1p-125f && S <= 0x1p125f);
      if (!exact) {
        const float y = __frcp_rn(S);
        uint32_t l0, l1, h0, h1;
        codes16(f, __fmul_rn(y, 1.0f - 0x1p-21f), l0, l1);
        codes16(f, __fmul_rn(y, 1.0f + 0x1p-21f), h0, h1);
        w0 = l0;
        w1 = l1;
        exact = (l0 != h0) || (l1 != h1);
      }
      if (exact) {
        uint32_t bb[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const float q1 = copysignf(__fdiv_rn(fabsf(f[2 * p + 1]), S), f[2 * p + 1]);
          const float q0 = copysignf(__fdiv_rn(fabsf(f[2 * p]), S), f[2 * p]);
          bb[p] = cvt_e2m1x2(q1, q0);
        }
        w0 = bb[0] | (bb[1] << 8) | (bb[2] << 16) | (bb[3] << 24);
        w1 = bb[4] | (bb[5] << 8) | (bb[6] << 16) | (bb[7] << 24);
      }
      w0 = drop_negative_zero(w0);
      w1 = drop_negative_zero(w1);
    }
    __stcs(codes + b, make_uint2(w0, w1));
    scales[b] = static_cast<uint8_t>(sb);
  }
}

template <bool kFold>
__global__ void k_finalize(float* s_g, float fold_s) {
  if (threadIdx.x == 0) {
    float amax = __uint_as_float(*reinterpret_cast<const uint32_t*>(s_g));
    if constexpr (kFold) amax = __fdiv_rn(amax, fold_s);
    *s_g = tensor_scale_from_amax(amax);
  }
}

// The norm-scale half of the fold: w' = fp32(w * s), elementwise.
__global__ void __launch_bounds__(kThreads) k_fold_norm(const float* __restrict__ w, int64_t d, float s,
                                                        float* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < d; i += stride)
    out[i] = __fmul_rn(w[i], s);
}

}  // namespace

cudaError_t launch_quantize(const void* W, int64_t d_o, int64_t d_i, uint8_t* codes,
                            uint8_t* scales, float* s_g, cudaStream_t stream, float fold_s) {
  const bool fold = fold_s != 1.0f;  // W / 1 == W exactly: the plain kernels
  const size_t n = static_cast<size_t>(d_o) * static_cast<size_t>(d_i);
  const size_t n_vec = n / 8;        // 16-byte words of 8 bf16
  const size_t n_blocks = n / 16;    // 16-weight blocks
  cudaError_t e = cudaMemsetAsync(s_g, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  size_t g1 = (n_vec + kThreads * 4 - 1) / (kThreads * 4);
  g1 = g1 < 1 ? 1 : (g1 > static_cast<size_t>(sms) * 8 ? static_cast<size_t>(sms) * 8 : g1);
  k_amax<<<static_cast<unsigned>(g1), kThreads, 0, stream>>>(static_cast<const uint4*>(W), n_vec,
                                                             reinterpret_cast<uint32_t*>(s_g));
  size_t g2 = (n_blocks + kThreads - 1) / kThreads;
  g2 = g2 < 1 ? 1 : (g2 > static_cast<size_t>(sms) * 16 ? static_cast<size_t>(sms) * 16 : g2);
  if (fold) {
    k_quant<true><<<static_cast<unsigned>(g2), kThreads, 0, stream>>>(
        static_cast<const uint4*>(W), n_blocks, reinterpret_cast<const uint32_t*>(s_g),
        reinterpret_cast<uint2*>(codes), scales, fold_s);
    k_finalize<true><<<1, 32, 0, stream>>>(s_g, fold_s);
  } else {
    k_quant<false><<<static_cast<unsigned>(g2), kThreads, 0, stream>>>(
        static_cast<const uint4*>(W), n_blocks, reinterpret_cast<const uint32_t*>(s_g),
        reinterpret_cast<uint2*>(codes), scales, 1.0f);
    k_finalize<false><<<1, 32, 0, stream>>>(s_g, 1.0f);
  }
  return cudaGetLastError();
}

cudaError_t launch_fold_norm(const float* w, int64_t d, float s, float* out, cudaStream_t stream) {
  int64_t g = (d + kThreads - 1) / kThreads;
  g = g > 1024 ? 1024 : g;
  k_fold_norm<<<static_cast<unsigned>(g), kThreads, 0, stream>>>(w, d, s, out);
  return cudaGetLastError();
}

}  // namespace pl
