// Generic CUDA-core NVFP4 + LoRA linear for shapes the tensor-core path does not
// take (d_i % 256 != 0).  Correct for every M >= 1, d_i % 16 == 0, r <= 64.
//
// Forward map ("QeRL: When Quantized Weights Help Reinforcement Learning, and Where
// the Evidence Stops", section 2.1): y = W_hat h + lambda B (A h), with h the
// section 5.1 RMSNorm-AQN of x when a norm scale is given, x itself otherwise, and
// W_hat = s_g s_b q (section 3.1).
//
// Two kernels:
//   k_prologue  one CTA per token row: h (FP32) into the workspace, then
//               t = A h (FP32, r values) by one warp per adapter row.
//   k_main      one warp per (output row o, group of 16 tokens): lanes stride over
//               the 16-weight blocks of row o, decode 16 weights to FP32 once and
//               FMA them against the 16 tokens' h; warp-shuffle reduction, then
//               y = s_g acc + lambda B[o,:] t[m,:] rounded to BF16.
#include "common.cuh"

namespace pl {
namespace {

constexpr int kProThreads = 256;
constexpr int kMainWarps = 8;
constexpr int kTok = 16;
constexpr int kRmax = 64;

struct GenericWs {
  float* h;   // [M][d_i]
  float* t;   // [M][kRmax]
};

GenericWs carve(void* ws, int64_t M, int64_t d_i) {
  char* p = static_cast<char*>(ws);
  GenericWs w;
  w.h = reinterpret_cast<float*>(p);
  p += align_up(static_cast<size_t>(M) * d_i * sizeof(float), 256);
  w.t = reinterpret_cast<float*>(p);
  return w;
}

__global__ void __launch_bounds__(kProThreads) k_prologue(const __nv_bfloat16* __restrict__ x, int64_t d_i,
                                                          const float* __restrict__ w_norm,
                                                          const float* __restrict__ z, int64_t z_ld,
                                                          float eps, const __nv_bfloat16* __restrict__ A,
                                                          int r, float* __restrict__ h, float* __restrict__ t) {
  __shared__ float red[kProThreads / 32];
  const int64_t m = blockIdx.x;
  if (z != nullptr) z += m * z_ld;  // this row's noise state (z_ld = 0: shared)
  const __nv_bfloat16* xr = x + m * d_i;
  float* hr = h + m * d_i;
  float inv = 1.0f;
  if (w_norm != nullptr) {
    float ss = 0.f;
    for (int64_t k = threadIdx.x; k < d_i; k += kProThreads) {
      const float a = __bfloat162float(xr[k]);
      ss = fmaf(a, a, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kProThreads / 32; ++w) tot += red[w];
    inv = 1.0f / sqrtf(tot / static_cast<float>(d_i) + eps);
  }
  for (int64_t k = threadIdx.x; k < d_i; k += kProThreads) {
    float v = __bfloat162float(xr[k]);
    if (w_norm != nullptr) v = (v * inv) * (w_norm[k] + (z != nullptr ? z[k] : 0.f));
    hr[k] = v;
  }
  __syncthreads();
  if (A == nullptr || r == 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < r; j += kProThreads / 32) {
    const __nv_bfloat16* Aj = A + static_cast<int64_t>(j) * d_i;
    float acc = 0.f;
    for (int64_t k = lane; k < d_i; k += 32) acc = fmaf(__bfloat162float(Aj[k]), hr[k], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) t[m * kRmax + j] = acc;
  }
}

// E2M1 code -> value, from the bit fields (sign | 2-bit exponent | 1-bit mantissa).
PL_DEVINL float e2m1_value(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float mag = e == 0 ? 0.5f * static_cast<float>(m)
                           : __uint_as_float((126u + e) << 23 | (m << 22));
  return (c & 8u) ? -mag : mag;
}

__global__ void __launch_bounds__(kMainWarps * 32) k_main(const uint8_t* __restrict__ codes,
                                                          const uint8_t* __restrict__ scales,
                                                          const float* __restrict__ s_g_ptr,
                                                          const float* __restrict__ h,
                                                          const float* __restrict__ t,
                                                          const __nv_bfloat16* __restrict__ B, int r,
                                                          float lambda, int64_t M, int64_t d_i,
                                                          int64_t d_o, void* __restrict__ y, bool y_f32) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t o = static_cast<int64_t>(blockIdx.x) * kMainWarps + warp;
  if (o >= d_o) return;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTok;
  const int ntok = static_cast<int>(M - m0 < kTok ? M - m0 : kTok);
  const int64_t nb = d_i / 16;
  float acc[kTok];
#pragma unroll
  for (int i = 0; i < kTok; ++i) acc[i] = 0.f;
  const uint8_t* crow = codes + o * (d_i / 2);
  const uint8_t* srow = scales + o * nb;
  for (int64_t b = lane; b < nb; b += 32) {
    const uint2 cw = *reinterpret_cast<const uint2*>(crow + 8 * b);
    const float sb = e4m3_to_f32(srow[b]);
    float w[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = ((i < 4 ? cw.x : cw.y) >> (8 * (i & 3))) & 0xFFu;
      w[2 * i] = e2m1_value(byte & 0xFu) * sb;
      w[2 * i + 1] = e2m1_value(byte >> 4) * sb;
    }
#pragma unroll
    for (int i = 0; i < kTok; ++i) {
      if (i < ntok) {
        const float4* hp = reinterpret_cast<const float4*>(h + (m0 + i) * d_i + 16 * b);
        float a = acc[i];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 hv = hp[q];
          a = fmaf(w[4 * q], hv.x, a);
          a = fmaf(w[4 * q + 1], hv.y, a);
          a = fmaf(w[4 * q + 2], hv.z, a);
          a = fmaf(w[4 * q + 3], hv.w, a);
        }
        acc[i] = a;
      }
    }
  }
  const float s_g = *s_g_ptr;
  const float bj = (B != nullptr && lane < r) ? __bfloat162float(B[o * r + lane]) : 0.f;
  const float bj2 = (B != nullptr && lane + 32 < r) ? __bfloat162float(B[o * r + lane + 32]) : 0.f;
  for (int i = 0; i < ntok; ++i) {
    float a = acc[i];
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, s);
    float l = 0.f;
    if (B != nullptr && r > 0) {
      const float* tr = t + (m0 + i) * kRmax;
      l = bj * (lane < r ? tr[lane] : 0.f) + bj2 * (lane + 32 < r ? tr[lane + 32] : 0.f);
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, s);
    }
    if (lane == 0) {
      const float v = fmaf(lambda, l, s_g * a);
      if (y_f32)
        static_cast<float*>(y)[(m0 + i) * d_o + o] = v;
      else
        static_cast<__nv_bfloat16*>(y)[(m0 + i) * d_o + o] = __float2bfloat16_rn(v);
    }
  }
}

}  // namespace

size_t generic_workspace_bytes(int64_t M, int64_t d_i, int64_t, int) {
  return align_up(static_cast<size_t>(M) * d_i * sizeof(float), 256) +
         align_up(static_cast<size_t>(M) * kRmax * sizeof(float), 256);
}

cudaError_t launch_linear_generic(const LinearArgs& a, cudaStream_t stream) {
  GenericWs w = carve(a.ws, a.M, a.d_i);
  const bool lora = a.A != nullptr && a.B != nullptr && a.r > 0;
  k_prologue<<<static_cast<unsigned>(a.M), kProThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.x), a.d_i, a.w_norm, a.z, a.z_ld, a.eps,
      lora ? static_cast<const __nv_bfloat16*>(a.A) : nullptr, lora ? a.r : 0, w.h, w.t);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((a.d_o + kMainWarps - 1) / kMainWarps),
            static_cast<unsigned>((a.M + kTok - 1) / kTok));
  k_main<<<grid, kMainWarps * 32, 0, stream>>>(
      a.codes, a.scales, a.s_g, w.h, w.t, lora ? static_cast<const __nv_bfloat16*>(a.B) : nullptr,
      lora ? a.r : 0, a.lambda, a.M, a.d_i, a.d_o, a.y, a.y_f32);
  return cudaGetLastError();
}

}  // namespace pl
