// RMSNorm with the AQN noise folded into the scale.
//
// Source: "QeRL: When Quantized Weights Help Reinforcement Learning, and Where the
// Evidence Stops", section 5.1: u = x / sqrt(d^-1 sum_j x_j^2 + delta),
// h_z = u (.) (w + z).  The noised scale w + z is formed in FP32 (BF16 spacing near
// 1 is 2^-7, coarser than the noise sigma of 1e-2 .. 5e-3), then the product is
// rounded once to BF16.
//
// One CTA per row; 16-byte loads of 8 BF16; the row's sum of squares is reduced in
// FP32 (warp shuffles, then one shared-memory pass), and the row is read a second
// time (from L1/L2) to write h.
#include "common.cuh"

namespace pl {
namespace {

constexpr int kThreads = 256;

PL_DEVINL float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) s += red[w];
  return s;
}

template <bool kF32>
__global__ void __launch_bounds__(kThreads) k_rmsnorm_aqn(const uint4* __restrict__ x, int64_t d,
                                                          const float* __restrict__ w_norm,
                                                          const float* __restrict__ z, int64_t z_ld,
                                                          float eps, void* __restrict__ h) {
  __shared__ float red[kThreads / 32];
  const int64_t nv = d / 8;
  const uint4* xr = x + blockIdx.x * nv;
  if (z != nullptr) z += static_cast<int64_t>(blockIdx.x) * z_ld;  // this row's noise state
  float ss = 0.f;
  for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
    const uint4 v = xr[i];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16lo_to_f32(u[j]), b = bf16hi_to_f32(u[j]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  const float total = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(total / static_cast<float>(d) + eps);
  for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
    const uint4 v = xr[i];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    float hv[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t k = 8 * i + 2 * j;
      float s0 = w_norm[k], s1 = w_norm[k + 1];
      if (z != nullptr) {
        s0 += z[k];
        s1 += z[k + 1];
      }
      hv[2 * j] = (bf16lo_to_f32(u[j]) * inv) * s0;
      hv[2 * j + 1] = (bf16hi_to_f32(u[j]) * inv) * s1;
    }
    if (kF32) {
      float4* hr = static_cast<float4*>(h) + (blockIdx.x * nv + i) * 2;
      hr[0] = make_float4(hv[0], hv[1], hv[2], hv[3]);
      hr[1] = make_float4(hv[4], hv[5], hv[6], hv[7]);
    } else {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(hv[2 * j], hv[2 * j + 1]);
        o[j] = *reinterpret_cast<const uint32_t*>(&p);
      }
      static_cast<uint4*>(h)[blockIdx.x * nv + i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm_aqn(const void* x, int64_t M, int64_t d, const float* w_norm,
                               const float* z, int64_t z_ld, float eps, void* h, bool h_f32,
                               cudaStream_t stream) {
  if (h_f32)
    k_rmsnorm_aqn<true><<<static_cast<unsigned>(M), kThreads, 0, stream>>>(
        static_cast<const uint4*>(x), d, w_norm, z, z_ld, eps, h);
  else
    k_rmsnorm_aqn<false><<<static_cast<unsigned>(M), kThreads, 0, stream>>>(
        static_cast<const uint4*>(x), d, w_norm, z, z_ld, eps, h);
  return cudaGetLastError();
}

}  // namespace pl
