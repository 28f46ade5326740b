// Internal host-side interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pl {

// Device-side status bits set by bounded waits that gave up.
enum : uint32_t { kStatusTimeout = 1u, kStatusRange = 2u };

// ---- quantize.cu
// fold_s != 1 quantises fp32(W / fold_s) (the UAQ fold); 1 is the plain quantiser.
cudaError_t launch_quantize(const void* W, int64_t d_o, int64_t d_i, uint8_t* codes,
                            uint8_t* scales, float* s_g, cudaStream_t stream, float fold_s = 1.0f);
// out[i] = fp32(w[i] * s), i < d: the norm-scale half of the UAQ fold.
cudaError_t launch_fold_norm(const float* w, int64_t d, float s, float* out, cudaStream_t stream);

// ---- norm.cu
// z_ld: 0 = one noise vector for every row, else row m's vector starts at z + m * z_ld.
cudaError_t launch_rmsnorm_aqn(const void* x, int64_t M, int64_t d, const float* w_norm,
                               const float* z, int64_t z_ld, float eps, void* h, bool h_f32,
                               cudaStream_t stream);

// Arguments of one linear call, shared by every path.
struct LinearArgs {
  const void* x;        // bf16 [M][d_i]
  int64_t M, d_i, d_o;
  const uint8_t* codes;   // [d_o][d_i/2]
  const uint8_t* scales;  // [d_o][d_i/16]
  const float* s_g;       // [1]
  const void* A;          // bf16 [r][d_i] or null
  const void* B;          // bf16 [d_o][r] or null
  int r;
  float lambda;
  const float* w_norm;    // [d_i] or null
  const float* z;         // [d_i] (z_ld == 0) or [M] rows of z_ld floats, or null
  int64_t z_ld;           // 0: one noise vector for every row; else elements between rows
  float eps;
  void* y;                // [M][d_o], bf16 or fp32
  bool y_f32;
  void* ws;               // workspace
  size_t ws_bytes;
};

// ---- linear_generic.cu (CUDA cores, any d_i % 16 == 0)
size_t generic_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r);
cudaError_t launch_linear_generic(const LinearArgs& a, cudaStream_t stream);

// ---- linear_tc.cu (tcgen05; d_i % 256 == 0)
// One input of a launch of the two-kernel decode path: x and its norm and noise.
struct TcSet {
  const void* x;  // bf16 [M][d_i]
  int64_t M;
  const float* w_norm;  // or null
  const float* z;
  int64_t z_ld;
};
// One projection (member) of such a launch; `set` is the index of the input it reads.
struct TcProj {
  int64_t d_o;
  const uint8_t* codes;
  const uint8_t* scales;
  const float* s_g;
  const void* A;  // bf16 [r][d_i] or null
  const void* B;  // bf16 [d_o][r] or null
  int r;          // 0 when A or B is null
  float lambda;
  void* y;        // [M][d_o]
  int set;
};
bool tc_supported(int64_t M, int64_t d_i, int64_t d_o, int r);
// at most 8 inputs and 8 members, at most 4 members and 128 adapter rows per input, M <= 64
bool tc_batch_supported(int64_t d_i, const TcSet* sets, int n_sets, const TcProj* projs, int n_proj);
size_t tc_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r);
size_t tc_batch_workspace_bytes(int64_t d_i, const TcSet* sets, int n_sets, const TcProj* projs, int n_proj);
cudaError_t launch_linear_tc(const LinearArgs& a, cudaStream_t stream);
// one prologue over every input, one main kernel over every member's weight tiles
cudaError_t launch_linear_tc_batch(int64_t d_i, float eps, const TcSet* sets, int n_sets, const TcProj* projs,
                                   int n_proj, bool y_f32, void* ws, cudaStream_t stream);
uint32_t tc_read_and_clear_status();
cudaError_t launch_wait_timeout_probe(cudaStream_t stream);
// The row prologue on its own: hq = f16(RMSNorm_AQN(x) / rowscale) [M][d_i], rowscale
// [M] (powers of two), A16 = f16(A) [r][d_i], and n_zero zeros (a multiple of 4) at zero.
// The adapters a row prologue converts to f16, one segment per projection of a large-M
// group, and the float ranges it zeroes (counters, padding rows of the f16 adapters).
constexpr int kMaxActConv = 4;
struct ActConv {
  const void* A[kMaxActConv];   // bf16 [r][d_i]
  __half* A16[kMaxActConv];     // f16 [r][d_i]
  int r[kMaxActConv];
  int n;
  float* zero[kMaxActConv + 1];     // floats to zero
  int64_t n_zero[kMaxActConv + 1];  // a multiple of 4
  int n_zero_ranges;
};
// The row prologue of the large-M paths: hq = f16(h / c_m) and c_m per row, the adapters of
// `conv`; with qx / s_x also the W8A8 form's E4M3 codes and per-row scale of h.
cudaError_t launch_act_prologue(const LinearArgs& a, __half* hq, float* rowscale, const ActConv& conv,
                                cudaStream_t stream, uint8_t* qx = nullptr, float* s_x = nullptr);

// ---- linear_fused.cu (tcgen05, one kernel; M <= 64 and at most 3 K chunks of 256 per CTA)
bool fused_supported(int64_t M, int64_t d_i, int64_t d_o, int r);
cudaError_t launch_linear_fused(const LinearArgs& a, cudaStream_t stream);
uint32_t fused_read_and_clear_status();

// ---- linear_prefill.cu (tcgen05 persistent GEMM; M > 64, d_i % 256 == 0, r <= 32)
bool prefill_supported(int64_t M, int64_t d_i, int64_t d_o, int r);
size_t prefill_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r);
cudaError_t launch_linear_prefill(const LinearArgs& a, cudaStream_t stream);
// A group of projections on one input at large M (q/k/v, gate/up): one row prologue, one
// LoRA down-projection per adapter, one contraction over every member's weight tiles.
// `in` carries the input, norm, noise, eps, y_f32 and the workspace; the members' fields
// are those of the group entry (TcProj::set unused).
constexpr int kMaxPrefillGroup = 4;
bool prefill_group_supported(int64_t M, int64_t d_i, const TcProj* projs, int n);
// The adapter's down-projection of the W8A8 form at large M: t[m][j] = c_m (A16 hq)[m][j] in
// FP32 from the row prologue's f16 rows, with A16 [r16(r)][d_i] (padding rows zero) and the
// counters [ceil(M / 128)] zeroed beforehand; t_part takes lora_down_t_scratch_bytes.
size_t lora_down_t_scratch_bytes(int64_t M, int r);
cudaError_t launch_lora_down_t(const __half* hq, int64_t M, int64_t d_i, const __half* A16, int r,
                               const float* rowscale, float* t, int t_ld, float* t_part, int* counters,
                               cudaStream_t stream);
size_t prefill_group_workspace_bytes(int64_t M, int64_t d_i, const TcProj* projs, int n);
cudaError_t launch_linear_prefill_group(const LinearArgs& in, const TcProj* projs, int n, cudaStream_t stream);
uint32_t prefill_read_and_clear_status();

// ---- w8a8.cu (FP8 E4M3 W8A8 linear; d_i % 128 == 0)
struct W8Args {
  const void* x;         // bf16 [M][d_i]
  int64_t M, d_i, d_o;
  const uint8_t* codes;  // E4M3 [d_o][d_i]
  const float* s_w;      // [d_o]
  const void* A;         // bf16 [r][d_i] or null
  const void* B;         // bf16 [d_o][r] or null
  int r;
  float lambda;
  const float* w_norm;
  const float* z;
  int64_t z_ld;
  float eps;
  void* y;
  bool y_f32;
  void* ws;
};
bool w8a8_supported(int64_t M, int64_t d_i, int64_t d_o, int r);
size_t w8a8_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r);
cudaError_t launch_w8a8_quantize(const void* W, int64_t d_o, int64_t d_i, uint8_t* codes, float* s_w,
                                 cudaStream_t stream);
cudaError_t launch_w8a8_linear(const W8Args& a, cudaStream_t stream);
uint32_t w8_read_and_clear_status();
// linear_tc.cu: the cluster prologue in its FP8 mode (per-token E4M3 codes, s_x, t = A h)
cudaError_t launch_pro_fp8(const void* x, int64_t M, int64_t d_i, const float* w_norm, const float* z, int64_t z_ld,
                           float eps, const void* A, int r, uint8_t* qx, float* s_x, float* t, int t_ld,
                           cudaStream_t stream);

// ---- backward.cu (frozen-backbone backward; d_i % 256 == 0, d_o % 8 == 0)
struct BwArgs {
  const void* g;          // bf16 [M][d_o]
  int64_t M, d_i, d_o;
  const uint8_t* codes;
  const uint8_t* scales;
  const float* s_g;
  const void* A;          // bf16 [r][d_i] or null
  const void* B;          // bf16 [d_o][r] or null
  int r;                  // 0 when A or B is null
  float lambda;
  const void* x;          // bf16 [M][d_i]
  const float* w_norm;    // or null
  const float* z;
  int64_t z_ld;
  float eps;
  float* dx;              // [M][d_i]
  float* dA;              // [r][d_i] or null
  float* dB;              // [d_o][r] or null
  void* ws;
};
bool backward_supported(int64_t M, int64_t d_i, int64_t d_o, int r);
size_t backward_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r, bool norm);
cudaError_t launch_backward(const BwArgs& a, cudaStream_t stream);
uint32_t bw_read_and_clear_status();

// ---- aqn.cu: z [n_scopes][d] = sigma * Philox4x32-10 / Box-Muller normals
cudaError_t launch_aqn_noise(uint64_t seed, uint32_t norm_id, uint64_t scope0, int64_t n_scopes, int64_t d,
                             float sigma, float* z, cudaStream_t stream);

// ---- api.cu
int sm_count();            // SMs of the current device (cached)
bool device_supported();   // the current device is one this library runs on (compute capability 10.3)

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace pl
