// AQN noise state on the device, sm_103a.
//
// "QeRL: When Quantized Weights Help Reinforcement Learning, and Where the Evidence
// Stops": the noise z enters the RMSNorm scale (section 5.1, h = u (.) (w + z)), its
// standard deviation follows the staged schedule of section 5.2, and it is drawn from a
// recorded seed under a declared persistence scope (section 6).  This kernel writes
// z [n_scopes][d] = sigma * N(0, 1) draws for scope indices scope0 .. scope0 + n_scopes - 1
// of one norm; the state is a pure function of (seed, norm index, scope index, channel),
// so a rollout, response or token can replay its noise exactly.
//
// Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC 2011) restated from its definition: ten rounds of two 32x32 -> 64-bit
// products (multipliers 0xD2511F53, 0xCD9E8D57), the high halves mixed with the other two
// words and the key, the key bumped by 0x9E3779B9 / 0xBB67AE85 after every round.
// Key = seed (low word first); counter = (block b, norm index, scope low word, scope high
// word); block b gives channels 4b .. 4b+3.  Each word x becomes u = (2 (x >> 9) + 1) 2^-24
// (exact in FP32, inside (0, 1)); Box-Muller turns (u0, u1) into rho cos(2 pi u1),
// rho sin(2 pi u1) with rho = sqrt(-2 ln u0), and (u2, u3) likewise.  FP32 arithmetic with
// the IEEE square root, logf and sincospif (no fast-math), then the multiply by sigma.
//
// One thread per block of four channels, a grid-stride loop, plain stores: z is a few
// KB to a few MB, written once per noise state.
#include "internal.h"

namespace pl {
namespace {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t hi0 = __umulhi(kPhiloxM0, c.x), lo0 = kPhiloxM0 * c.x;
    const uint32_t hi1 = __umulhi(kPhiloxM1, c.z), lo1 = kPhiloxM1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return c;
}

// 23 random bits as an odd multiple of 2^-24: exact in FP32, never 0 or 1.
__device__ __forceinline__ float uniform24(uint32_t x) {
  return __uint2float_rn(2u * (x >> 9) + 1u) * 0x1p-24f;
}

__global__ void __launch_bounds__(256) k_aqn_noise(uint32_t k0, uint32_t k1, uint32_t norm_id, uint64_t scope0,
                                                   int64_t n_scopes, int64_t d, float sigma,
                                                   float* __restrict__ z) {
  const int64_t nb = (d + 3) / 4;
  const int64_t total = nb * n_scopes;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total; g += stride) {
    const int64_t s = g / nb, b = g - s * nb;
    const uint64_t sc = scope0 + static_cast<uint64_t>(s);
    const uint4 x = philox4x32_10(
        make_uint4(static_cast<uint32_t>(b), norm_id, static_cast<uint32_t>(sc), static_cast<uint32_t>(sc >> 32)),
        k0, k1);
    const float rho_a = sqrtf(-2.0f * logf(uniform24(x.x)));
    const float rho_b = sqrtf(-2.0f * logf(uniform24(x.z)));
    float sa, ca, sb, cb;
    sincospif(2.0f * uniform24(x.y), &sa, &ca);
    sincospif(2.0f * uniform24(x.w), &sb, &cb);
    const float v[4] = {sigma * (rho_a * ca), sigma * (rho_a * sa), sigma * (rho_b * cb), sigma * (rho_b * sb)};
    float* out = z + s * d + 4 * b;
    const int64_t left = d - 4 * b;  // 1 .. 4 channels of this block exist
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q < left) out[q] = v[q];
  }
}

}  // namespace

cudaError_t launch_aqn_noise(uint64_t seed, uint32_t norm_id, uint64_t scope0, int64_t n_scopes, int64_t d,
                             float sigma, float* z, cudaStream_t stream) {
  const int threads = 256;
  const int64_t total = (d + 3) / 4 * n_scopes;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = 8ll * sm_count();  // a few waves at most; the loop covers the rest
  if (blocks > cap) blocks = cap;
  k_aqn_noise<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32), norm_id, scope0, n_scopes, d, sigma, z);
  return cudaGetLastError();
}

}  // namespace pl
