// C ABI of libprecision_linear: argument checks, device check, dispatch.
// Declarations and the contract of every entry point are in include/precision_linear.h.
#include <atomic>
#include <cmath>
#include <mutex>

#include "../../include/precision_linear.h"
#include "internal.h"

namespace {

std::atomic<int> g_fail_next_launch{0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The noise state's row stride: 0 (one vector for every row) or a multiple of 4 that is
// at least the row length, with every row's offset representable.
bool z_ld_ok(int64_t z_ld, int64_t M, int64_t d) {
  if (z_ld == 0) return true;
  return z_ld >= d && z_ld % 4 == 0 && z_ld <= (int64_t{1} << 40) / (M > 0 ? M : 1);
}

pl_status check_launch(cudaError_t e) {
  if (g_fail_next_launch.exchange(0) != 0) return PL_ERR_CUDA;
  return e == cudaSuccess ? PL_OK : PL_ERR_CUDA;
}

struct DevInfo {
  int ok = -1;  // -1 unknown, 0 unsupported, 1 supported
  int sms = 0;
};
constexpr int kMaxDev = 64;
DevInfo g_dev[kMaxDev];
std::mutex g_dev_mu;

pl_status device_check() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return PL_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.ok < 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return PL_ERR_DEVICE;
    }
    d.ok = (major == 10 && minor == 3) ? 1 : 0;
    d.sms = sms;
  }
  return d.ok == 1 ? PL_OK : PL_ERR_DEVICE;
}

}  // namespace

namespace pl {
bool device_supported() { return device_check() == PL_OK; }

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDev) return 148;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  return g_dev[dev].sms > 0 ? g_dev[dev].sms : 148;
}
}  // namespace pl

extern "C" {

const char* pl_status_string(pl_status s) {
  switch (s) {
    case PL_OK: return "PL_OK";
    case PL_ERR_NULL: return "PL_ERR_NULL: a required pointer is NULL";
    case PL_ERR_SHAPE: return "PL_ERR_SHAPE: size out of range or not a multiple of the block";
    case PL_ERR_ALIGN: return "PL_ERR_ALIGN: pointer not 16-byte aligned";
    case PL_ERR_RANK: return "PL_ERR_RANK: LoRA rank out of range";
    case PL_ERR_DEVICE: return "PL_ERR_DEVICE: no current CUDA device of compute capability 10.3";
    case PL_ERR_CUDA: return "PL_ERR_CUDA: CUDA launch or runtime call failed";
    case PL_ERR_WORKSPACE: return "PL_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case PL_ERR_TIMEOUT: return "PL_ERR_TIMEOUT: a bounded device-side wait gave up";
    case PL_ERR_RANGE: return "PL_ERR_RANGE: an intermediate left its number format's range";
    case PL_ERR_OVERLAP: return "PL_ERR_OVERLAP: a batch's output overlaps another output or an input";
  }
  return "unknown pl_status";
}

int pl_version(void) { return 200; }

size_t pl_nvfp4_bytes(int64_t d_o, int64_t d_i) {
  if (d_o < 1 || d_i < 16 || d_i % 16 != 0) return 0;
  const size_t P = static_cast<size_t>(d_o) * static_cast<size_t>(d_i);
  return P / 2 + P / 16;
}

size_t pl_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r) {
  if (M < 1 || d_o < 1 || d_i < 16 || d_i % 16 != 0 || r < 0 || r > 64) return 0;
  size_t g = pl::generic_workspace_bytes(M, d_i, d_o, r);
  size_t t = pl::tc_supported(M, d_i, d_o, r) ? pl::tc_workspace_bytes(M, d_i, d_o, r) : 0;
  const size_t f = pl::prefill_supported(M, d_i, d_o, r) ? pl::prefill_workspace_bytes(M, d_i, d_o, r) : 0;
  t = t > f ? t : f;
  return g > t ? g : t;
}

pl_status pl_nvfp4_quantize(const void* W, int64_t d_o, int64_t d_i, uint8_t* codes,
                            uint8_t* scales, float* s_g, pl_stream_t stream) {
  if (!W || !codes || !scales || !s_g) return PL_ERR_NULL;
  if (d_o < 1 || d_i < 16 || d_i % 16 != 0) return PL_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(s_g) & 3u)) return PL_ERR_ALIGN;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  return check_launch(pl::launch_quantize(W, d_o, d_i, codes, scales, s_g,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

pl_status pl_nvfp4_quantize_uaq(const void* W, int64_t d_o, int64_t d_i, float s, uint8_t* codes,
                                uint8_t* scales, float* s_g, pl_stream_t stream) {
  if (!W || !codes || !scales || !s_g) return PL_ERR_NULL;
  if (d_o < 1 || d_i < 16 || d_i % 16 != 0 || !(s > 0.f) || !std::isfinite(s)) return PL_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(s_g) & 3u)) return PL_ERR_ALIGN;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  return check_launch(pl::launch_quantize(W, d_o, d_i, codes, scales, s_g,
                                          reinterpret_cast<cudaStream_t>(stream), s));
}

pl_status pl_uaq_fold_norm(const float* w_norm, int64_t d, float s, float* out, pl_stream_t stream) {
  if (!w_norm || !out) return PL_ERR_NULL;
  if (d < 1 || d > (1ll << 40) || !(s > 0.f) || !std::isfinite(s)) return PL_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(w_norm) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u)) return PL_ERR_ALIGN;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  return check_launch(pl::launch_fold_norm(w_norm, d, s, out, reinterpret_cast<cudaStream_t>(stream)));
}

pl_status pl_rmsnorm_aqn(const void* x, int64_t M, int64_t d, const float* w_norm,
                         const float* z, int64_t z_ld, float eps, void* h, int h_dtype, pl_stream_t stream) {
  if (!x || !w_norm || !h) return PL_ERR_NULL;
  if (M < 1 || d < 8 || d % 8 != 0 || M > 0x7FFFFFFF) return PL_ERR_SHAPE;
  if (h_dtype != PL_DTYPE_BF16 && h_dtype != PL_DTYPE_F32) return PL_ERR_SHAPE;
  if (z && !z_ld_ok(z_ld, M, d)) return PL_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(h) || (z && !aligned16(z))) return PL_ERR_ALIGN;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  return check_launch(pl::launch_rmsnorm_aqn(x, M, d, w_norm, z, z ? z_ld : 0, eps, h, h_dtype == PL_DTYPE_F32,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

pl_status pl_nvfp4_lora_linear(const void* x, int64_t M, int64_t d_i, int64_t d_o,
                               const uint8_t* codes, const uint8_t* scales, const float* s_g,
                               const void* A, const void* B, int r, float lambda,
                               const float* w_norm, const float* z, int64_t z_ld, float eps, void* y,
                               int y_dtype, void* workspace, size_t ws_bytes, pl_stream_t stream) {
  if (!x || !codes || !scales || !s_g || !y) return PL_ERR_NULL;
  if (M < 1 || d_o < 1 || d_i < 16 || d_i % 16 != 0 || M > (1ll << 24) || d_o > (1ll << 31) ||
      d_i > (1ll << 31))
    return PL_ERR_SHAPE;
  if (y_dtype != PL_DTYPE_BF16 && y_dtype != PL_DTYPE_F32) return PL_ERR_SHAPE;
  if (r < 0 || r > 64) return PL_ERR_RANK;
  if (w_norm && z && !z_ld_ok(z_ld, M, d_i)) return PL_ERR_SHAPE;
  const bool lora = r > 0 && A != nullptr && B != nullptr;
  if (r > 0 && (A == nullptr) != (B == nullptr)) return PL_ERR_NULL;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(y) ||
      (lora && (!aligned16(A) || !aligned16(B))) || (w_norm && !aligned16(w_norm)) || (z && !aligned16(z)))
    return PL_ERR_ALIGN;
  const size_t need = pl_workspace_bytes(M, d_i, d_o, r);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PL_ERR_WORKSPACE;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  pl::LinearArgs a{x, M, d_i, d_o, codes, scales, s_g, lora ? A : nullptr, lora ? B : nullptr,
                   lora ? r : 0, lambda, w_norm, w_norm ? z : nullptr, (w_norm && z) ? z_ld : 0, eps, y,
                   y_dtype == PL_DTYPE_F32,
                   workspace, ws_bytes};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the one-kernel path takes one noise vector per call; per-row states go to the two-kernel
  // path, whose prologue reads them row by row
  if (a.z_ld == 0 && pl::fused_supported(M, d_i, d_o, a.r)) return check_launch(pl::launch_linear_fused(a, s));
  if (pl::tc_supported(M, d_i, d_o, a.r)) return check_launch(pl::launch_linear_tc(a, s));
  if (pl::prefill_supported(M, d_i, d_o, a.r)) return check_launch(pl::launch_linear_prefill(a, s));
  return check_launch(pl::launch_linear_generic(a, s));
}

// Host checks shared by the group and batch entries for one projection.
pl_status check_proj(int64_t d_o, const uint8_t* codes, const uint8_t* scales, const float* s_g, const void* A,
                     const void* B, int r, const void* y) {
  if (!codes || !scales || !s_g || !y) return PL_ERR_NULL;
  if (d_o < 1 || d_o > (1ll << 31)) return PL_ERR_SHAPE;
  if (r < 0 || r > 64) return PL_ERR_RANK;
  if (r > 0 && (A == nullptr) != (B == nullptr)) return PL_ERR_NULL;
  const bool lora = r > 0 && A != nullptr && B != nullptr;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(y) || (lora && (!aligned16(A) || !aligned16(B))))
    return PL_ERR_ALIGN;
  return PL_OK;
}

pl::TcProj tc_proj(int64_t d_o, const uint8_t* codes, const uint8_t* scales, const float* s_g, const void* A,
                   const void* B, int r, float lambda, void* y, int set) {
  const bool lora = r > 0 && A != nullptr && B != nullptr;
  return pl::TcProj{d_o, codes, scales, s_g, lora ? A : nullptr, lora ? B : nullptr, lora ? r : 0, lambda, y, set};
}

size_t pl_workspace_bytes_group(int64_t M, int64_t d_i, const pl_nvfp4_proj* projs, int n_proj) {
  if (!projs || n_proj < 1 || n_proj > PL_MAX_GROUP) return 0;
  size_t need = 0;
  pl::TcProj tp[PL_MAX_GROUP];
  for (int i = 0; i < n_proj; ++i) {
    const size_t w = pl_workspace_bytes(M, d_i, projs[i].d_o, projs[i].r);
    if (w == 0) return 0;
    need = need > w ? need : w;
    tp[i] = tc_proj(projs[i].d_o, projs[i].codes, projs[i].scales, projs[i].s_g, projs[i].A_bf16, projs[i].B_bf16,
                    projs[i].r, projs[i].lambda, projs[i].y, 0);
    tp[i].r = projs[i].r;  // the workspace is sized for the declared ranks
  }
  if (pl::tc_supported(M, d_i, 1, 0)) {
    const pl::TcSet set{nullptr, M, nullptr, nullptr, 0};
    const size_t g = pl::tc_batch_workspace_bytes(d_i, &set, 1, tp, n_proj);
    need = need > g ? need : g;
  }
  if (pl::prefill_group_supported(M, d_i, tp, n_proj)) {
    const size_t g = pl::prefill_group_workspace_bytes(M, d_i, tp, n_proj);
    need = need > g ? need : g;
  }
  return need;
}

pl_status pl_nvfp4_lora_linear_group(const void* x, int64_t M, int64_t d_i, const float* w_norm, const float* z,
                                     int64_t z_ld, float eps, const pl_nvfp4_proj* projs, int n_proj, int y_dtype,
                                     void* workspace, size_t ws_bytes, pl_stream_t stream) {
  if (!x || !projs) return PL_ERR_NULL;
  if (n_proj < 1 || n_proj > PL_MAX_GROUP) return PL_ERR_SHAPE;
  if (M < 1 || d_i < 16 || d_i % 16 != 0 || M > (1ll << 24) || d_i > (1ll << 31)) return PL_ERR_SHAPE;
  if (y_dtype != PL_DTYPE_BF16 && y_dtype != PL_DTYPE_F32) return PL_ERR_SHAPE;
  if (w_norm && z && !z_ld_ok(z_ld, M, d_i)) return PL_ERR_SHAPE;
  if (!aligned16(x) || (w_norm && !aligned16(w_norm)) || (z && !aligned16(z))) return PL_ERR_ALIGN;
  pl::TcProj tp[PL_MAX_GROUP];
  for (int i = 0; i < n_proj; ++i) {
    const pl_nvfp4_proj& q = projs[i];
    const pl_status st = check_proj(q.d_o, q.codes, q.scales, q.s_g, q.A_bf16, q.B_bf16, q.r, q.y);
    if (st != PL_OK) return st;
    tp[i] = tc_proj(q.d_o, q.codes, q.scales, q.s_g, q.A_bf16, q.B_bf16, q.r, q.lambda, q.y, 0);
  }
  const size_t need = pl_workspace_bytes_group(M, d_i, projs, n_proj);
  if (!workspace || need == 0 || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PL_ERR_WORKSPACE;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // one launch pair for the whole group on the two-kernel decode path, one row pass and one
  // contraction at large M; otherwise one call per projection, in order
  const pl::TcSet set{x, M, w_norm, w_norm ? z : nullptr, (w_norm && z) ? z_ld : 0};
  if (n_proj > 1 && pl::tc_batch_supported(d_i, &set, 1, tp, n_proj))
    return check_launch(pl::launch_linear_tc_batch(d_i, eps, &set, 1, tp, n_proj, y_dtype == PL_DTYPE_F32,
                                                   workspace, s));
  if (n_proj > 1 && pl::prefill_group_supported(M, d_i, tp, n_proj)) {
    pl::LinearArgs in{};
    in.x = x;
    in.M = M;
    in.d_i = d_i;
    in.w_norm = w_norm;
    in.z = w_norm ? z : nullptr;
    in.z_ld = (w_norm && z) ? z_ld : 0;
    in.eps = eps;
    in.y_f32 = y_dtype == PL_DTYPE_F32;
    in.ws = workspace;
    in.ws_bytes = ws_bytes;
    return check_launch(pl::launch_linear_prefill_group(in, tp, n_proj, s));
  }
  for (int i = 0; i < n_proj; ++i) {
    st = pl_nvfp4_lora_linear(x, M, d_i, tp[i].d_o, tp[i].codes, tp[i].scales, tp[i].s_g, tp[i].A, tp[i].B, tp[i].r,
                              tp[i].lambda, w_norm, z, z_ld, eps, tp[i].y, y_dtype, workspace, ws_bytes, stream);
    if (st != PL_OK) return st;
  }
  return PL_OK;
}

namespace {
// The distinct inputs of a batch (calls with the same x, M, w_norm, z and z_ld share one) and
// each call's index among them.
int batch_sets(const pl_nvfp4_call* calls, int n, pl::TcSet* sets, int* which) {
  int n_sets = 0;
  for (int i = 0; i < n; ++i) {
    const pl_nvfp4_call& c = calls[i];
    const float* z = c.w_norm ? c.z : nullptr;
    const int64_t z_ld = (c.w_norm && c.z) ? c.z_ld : 0;
    int s = 0;
    while (s < n_sets && !(sets[s].x == c.x_bf16 && sets[s].M == c.M && sets[s].w_norm == c.w_norm &&
                           sets[s].z == z && sets[s].z_ld == z_ld))
      ++s;
    if (s == n_sets) sets[n_sets++] = pl::TcSet{c.x_bf16, c.M, c.w_norm, z, z_ld};
    which[i] = s;
  }
  return n_sets;
}

bool ranges_overlap(uintptr_t a0, size_t an, uintptr_t b0, size_t bn) { return a0 < b0 + bn && b0 < a0 + an; }
}  // namespace

size_t pl_workspace_bytes_batch(int64_t d_i, const pl_nvfp4_call* calls, int n_calls) {
  if (!calls || n_calls < 1 || n_calls > PL_MAX_BATCH) return 0;
  size_t need = 0;
  for (int i = 0; i < n_calls; ++i) {
    const size_t w = pl_workspace_bytes(calls[i].M, d_i, calls[i].d_o, calls[i].r);
    if (w == 0) return 0;
    need = need > w ? need : w;
  }
  pl::TcSet sets[PL_MAX_BATCH];
  int which[PL_MAX_BATCH];
  const int n_sets = batch_sets(calls, n_calls, sets, which);
  pl::TcProj tp[PL_MAX_BATCH];
  for (int i = 0; i < n_calls; ++i)
    tp[i] = pl::TcProj{calls[i].d_o, calls[i].codes, calls[i].scales, calls[i].s_g, calls[i].A_bf16, calls[i].B_bf16,
                       calls[i].r, calls[i].lambda, calls[i].y, which[i]};
  if (pl::tc_batch_supported(d_i, sets, n_sets, tp, n_calls)) {
    const size_t g = pl::tc_batch_workspace_bytes(d_i, sets, n_sets, tp, n_calls);
    need = need > g ? need : g;
  }
  return need;
}

pl_status pl_nvfp4_lora_linear_batch(int64_t d_i, float eps, const pl_nvfp4_call* calls, int n_calls, int y_dtype,
                                     void* workspace, size_t ws_bytes, pl_stream_t stream) {
  if (!calls) return PL_ERR_NULL;
  if (n_calls < 1 || n_calls > PL_MAX_BATCH || d_i < 16 || d_i % 16 != 0 || d_i > (1ll << 31)) return PL_ERR_SHAPE;
  if (y_dtype != PL_DTYPE_BF16 && y_dtype != PL_DTYPE_F32) return PL_ERR_SHAPE;
  const size_t ysz = y_dtype == PL_DTYPE_F32 ? 4 : 2;
  for (int i = 0; i < n_calls; ++i) {
    const pl_nvfp4_call& c = calls[i];
    if (!c.x_bf16) return PL_ERR_NULL;
    if (c.M < 1 || c.M > (1ll << 24)) return PL_ERR_SHAPE;
    if (c.w_norm && c.z && !z_ld_ok(c.z_ld, c.M, d_i)) return PL_ERR_SHAPE;
    if (!aligned16(c.x_bf16) || (c.w_norm && !aligned16(c.w_norm)) || (c.z && !aligned16(c.z))) return PL_ERR_ALIGN;
    const pl_status st = check_proj(c.d_o, c.codes, c.scales, c.s_g, c.A_bf16, c.B_bf16, c.r, c.y);
    if (st != PL_OK) return st;
  }
  // independent calls: no output may overlap another call's output or any call's activations
  for (int i = 0; i < n_calls; ++i) {
    const uintptr_t yi = reinterpret_cast<uintptr_t>(calls[i].y);
    const size_t ni = static_cast<size_t>(calls[i].M) * calls[i].d_o * ysz;
    for (int j = 0; j < n_calls; ++j) {
      const uintptr_t xj = reinterpret_cast<uintptr_t>(calls[j].x_bf16);
      if (ranges_overlap(yi, ni, xj, static_cast<size_t>(calls[j].M) * d_i * 2)) return PL_ERR_OVERLAP;
      if (j != i && ranges_overlap(yi, ni, reinterpret_cast<uintptr_t>(calls[j].y),
                                   static_cast<size_t>(calls[j].M) * calls[j].d_o * ysz))
        return PL_ERR_OVERLAP;
    }
  }
  const size_t need = pl_workspace_bytes_batch(d_i, calls, n_calls);
  if (!workspace || need == 0 || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PL_ERR_WORKSPACE;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  pl::TcSet sets[PL_MAX_BATCH];
  int which[PL_MAX_BATCH];
  const int n_sets = batch_sets(calls, n_calls, sets, which);
  pl::TcProj tp[PL_MAX_BATCH];
  for (int i = 0; i < n_calls; ++i)
    tp[i] = tc_proj(calls[i].d_o, calls[i].codes, calls[i].scales, calls[i].s_g, calls[i].A_bf16, calls[i].B_bf16,
                    calls[i].r, calls[i].lambda, calls[i].y, which[i]);
  if (n_calls > 1 && pl::tc_batch_supported(d_i, sets, n_sets, tp, n_calls))
    return check_launch(pl::launch_linear_tc_batch(d_i, eps, sets, n_sets, tp, n_calls, y_dtype == PL_DTYPE_F32,
                                                   workspace, reinterpret_cast<cudaStream_t>(stream)));
  for (int i = 0; i < n_calls; ++i) {
    const pl_nvfp4_call& c = calls[i];
    st = pl_nvfp4_lora_linear(c.x_bf16, c.M, d_i, c.d_o, c.codes, c.scales, c.s_g, c.A_bf16, c.B_bf16, c.r, c.lambda,
                              c.w_norm, c.z, c.z_ld, eps, c.y, y_dtype, workspace, ws_bytes, stream);
    if (st != PL_OK) return st;
  }
  return PL_OK;
}

size_t pl_w8a8_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r) {
  if (!pl::w8a8_supported(M, d_i, d_o, r) || M > (1ll << 24)) return 0;
  return pl::w8a8_workspace_bytes(M, d_i, d_o, r);
}

pl_status pl_w8a8_quantize_weight(const void* W, int64_t d_o, int64_t d_i, uint8_t* codes, float* s_w,
                                  pl_stream_t stream) {
  if (!W || !codes || !s_w) return PL_ERR_NULL;
  if (d_o < 1 || d_o > 0x7FFFFFFF || d_i < 16 || d_i % 16 != 0) return PL_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(s_w) & 3u)) return PL_ERR_ALIGN;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  return check_launch(pl::launch_w8a8_quantize(W, d_o, d_i, codes, s_w, reinterpret_cast<cudaStream_t>(stream)));
}

pl_status pl_w8a8_lora_linear(const void* x, int64_t M, int64_t d_i, int64_t d_o, const uint8_t* codes,
                              const float* s_w, const void* A, const void* B, int r, float lambda,
                              const float* w_norm, const float* z, int64_t z_ld, float eps, void* y, int y_dtype,
                              void* workspace, size_t ws_bytes, pl_stream_t stream) {
  if (!x || !codes || !s_w || !y) return PL_ERR_NULL;
  if (M < 1 || M > (1ll << 24) || d_o < 1 || d_o > (1ll << 31) || d_i < 128 || d_i % 128 != 0 || d_i > 32768)
    return PL_ERR_SHAPE;
  if (y_dtype != PL_DTYPE_BF16 && y_dtype != PL_DTYPE_F32) return PL_ERR_SHAPE;
  if (r < 0 || r > 64) return PL_ERR_RANK;
  if (r > 0 && (A == nullptr) != (B == nullptr)) return PL_ERR_NULL;
  if (w_norm && z && !z_ld_ok(z_ld, M, d_i)) return PL_ERR_SHAPE;
  const bool lora = r > 0 && A != nullptr && B != nullptr;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(y) || (reinterpret_cast<uintptr_t>(s_w) & 3u) ||
      (lora && (!aligned16(A) || !aligned16(B))) || (w_norm && !aligned16(w_norm)) || (z && !aligned16(z)))
    return PL_ERR_ALIGN;
  const size_t need = pl_w8a8_workspace_bytes(M, d_i, d_o, r);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PL_ERR_WORKSPACE;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  pl::W8Args a{x, M, d_i, d_o, codes, s_w, lora ? A : nullptr, lora ? B : nullptr, lora ? r : 0, lambda, w_norm,
               w_norm ? z : nullptr, (w_norm && z) ? z_ld : 0, eps, y, y_dtype == PL_DTYPE_F32, workspace};
  return check_launch(pl::launch_w8a8_linear(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t pl_backward_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r, int with_norm) {
  if (!pl::backward_supported(M, d_i, d_o, r) || M > (1ll << 24)) return 0;
  return pl::backward_workspace_bytes(M, d_i, d_o, r, with_norm != 0);
}

pl_status pl_nvfp4_lora_linear_backward(const void* g, int64_t M, int64_t d_i, int64_t d_o, const uint8_t* codes,
                                        const uint8_t* scales, const float* s_g, const void* A, const void* B, int r,
                                        float lambda, const void* x, const float* w_norm, const float* z,
                                        int64_t z_ld, float eps, float* dx, float* dA, float* dB, void* workspace,
                                        size_t ws_bytes, pl_stream_t stream) {
  if (!g || !codes || !scales || !s_g || !dx || !x) return PL_ERR_NULL;
  if (M < 1 || M > (1ll << 24) || d_o < 8 || d_o % 8 != 0 || d_o > (1ll << 31) || d_i < 256 || d_i % 256 != 0 ||
      d_i > (1ll << 31))
    return PL_ERR_SHAPE;
  if (r < 0 || r > 64) return PL_ERR_RANK;
  if (r > 0 && (A == nullptr) != (B == nullptr)) return PL_ERR_NULL;
  if (w_norm && z && !z_ld_ok(z_ld, M, d_i)) return PL_ERR_SHAPE;
  const bool lora = r > 0 && A != nullptr && B != nullptr;
  if (!aligned16(g) || !aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(dx) ||
      (lora && (!aligned16(A) || !aligned16(B))) || (w_norm && !aligned16(w_norm)) || (z && !aligned16(z)) ||
      (dA && !aligned16(dA)) || (dB && (reinterpret_cast<uintptr_t>(dB) & 3u)))
    return PL_ERR_ALIGN;
  const size_t need = pl_backward_workspace_bytes(M, d_i, d_o, lora ? r : 0, w_norm != nullptr);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PL_ERR_WORKSPACE;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  pl::BwArgs a{g, M, d_i, d_o, codes, scales, s_g, lora ? A : nullptr, lora ? B : nullptr, lora ? r : 0, lambda, x,
               w_norm, w_norm ? z : nullptr, (w_norm && z) ? z_ld : 0, eps, dx, lora ? dA : nullptr,
               lora ? dB : nullptr, workspace};
  return check_launch(pl::launch_backward(a, reinterpret_cast<cudaStream_t>(stream)));
}

int pl_aqn_stage(int64_t done, int64_t total) {
  if (total < 1 || done < 0) return -1;
  // ten equal parts of the planned horizon, the product taken in 128 bits
  if (done >= total) return 9;
  const int64_t k = static_cast<int64_t>((static_cast<__int128>(10) * done) / total);
  return k > 9 ? 9 : static_cast<int>(k);
}

float pl_aqn_sigma(int stage, float sigma_start, float sigma_end) {
  if (stage < 0 || stage > 9 || !(sigma_start > 0.f) || !(sigma_end > 0.f) || !std::isfinite(sigma_start) ||
      !std::isfinite(sigma_end))
    return -1.f;
  if (stage == 0) return 0.f;
  const double s0 = sigma_start, s1 = sigma_end;
  return static_cast<float>(s0 * std::pow(s1 / s0, (stage - 1) / 8.0));
}

pl_status pl_aqn_noise(uint64_t seed, uint32_t norm_id, uint64_t scope0, int64_t n_scopes, int64_t d,
                       float sigma, float* z, pl_stream_t stream) {
  if (!z) return PL_ERR_NULL;
  if (d < 1 || n_scopes < 1 || d > (1ll << 31) || n_scopes > (1ll << 31) || d * n_scopes > (1ll << 40) ||
      !(sigma >= 0.f) || !std::isfinite(sigma))
    return PL_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(z) & 3u) return PL_ERR_ALIGN;
  pl_status st = device_check();
  if (st != PL_OK) return st;
  return check_launch(pl::launch_aqn_noise(seed, norm_id, scope0, n_scopes, d, sigma, z,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

pl_status pl_last_device_status(pl_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return PL_ERR_CUDA;
  uint32_t bits = pl::tc_read_and_clear_status() | pl::fused_read_and_clear_status() |
                  pl::prefill_read_and_clear_status() | pl::w8_read_and_clear_status() |
                  pl::bw_read_and_clear_status();
  if (bits & pl::kStatusTimeout) return PL_ERR_TIMEOUT;
  return (bits & pl::kStatusRange) ? PL_ERR_RANGE : PL_OK;
}

int pl_debug_linear_path(int64_t M, int64_t d_i, int64_t d_o, int r) {
  if (M < 1 || d_o < 1 || d_i < 16 || d_i % 16 != 0 || r < 0 || r > 64 || device_check() != PL_OK) return -1;
  if (pl::fused_supported(M, d_i, d_o, r)) return 2;
  if (pl::tc_supported(M, d_i, d_o, r)) return 1;
  if (pl::prefill_supported(M, d_i, d_o, r)) return 3;
  return 0;
}

void pl_debug_fail_next_launch(int armed) { g_fail_next_launch.store(armed ? 1 : 0); }

pl_status pl_debug_wait_timeout_probe(pl_stream_t stream) {
  pl_status st = device_check();
  if (st != PL_OK) return st;
  return check_launch(pl::launch_wait_timeout_probe(reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
