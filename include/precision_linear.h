/*
 * precision_linear.h -- C ABI of the NVFP4 + LoRA + AQN-RMSNorm linear for GB300.
 *
 * The frozen-backbone linear layer of quantised RL rollout:
 *
 *     y = W_hat . h + lambda . B (A . h),    h = RMSNorm_AQN(x) = u (.) (w_norm + z),
 *     u = x / sqrt(mean(x^2) + eps),        W_hat = s_g . s_b . q  (NVFP4)
 *
 * Sources: "QeRL: When Quantized Weights Help Reinforcement Learning, and Where
 * the Evidence Stops" (zhongzhuzhou.org) -- section 2.1 (forward map of LoRA on
 * a quantised backbone), section 3.1 (NVFP4: E2M1 codes, one E4M3 scale per 16
 * weights, one FP32 tensor scale, reconstruction and argmin equations, 9P/16
 * storage), section 5.1 (noise folded into the RMSNorm scale).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensors are dense and row-major.  "BF16" buffers hold IEEE bfloat16,
 *    "FP32" buffers IEEE float.
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise, on the
 *    current CUDA device.  The caller owns all memory; the library never
 *    allocates device memory on these paths.  Scratch lives in the caller's
 *    workspace (see pl_workspace_bytes).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and never synchronise the host.
 *  - Errors are return codes.  Argument checks (NULL, sizes, alignment, rank,
 *    workspace size) are done on the host before anything is launched; a call
 *    that fails them launches nothing.  Launch failures map to PL_ERR_CUDA.
 *    Device-side waits are bounded: one that gives up records a device status
 *    word, read (with a stream synchronise) by pl_last_device_status.
 *  - Device requirement: compute capability 10.3 (GB300, sm_103a), else
 *    PL_ERR_DEVICE.
 *
 * NVFP4 layout (canonical, what pl_nvfp4_quantize writes and the linear reads)
 * ---------------------------------------------------------------------------
 *  codes  uint8 [d_o][d_i/2]  : byte (o, k/2) = code(o,k) | code(o,k+1) << 4, k even.
 *                               A code is 4-bit E2M1: sign | 2 exponent bits | 1
 *                               mantissa bit, magnitudes {0,.5,1,1.5,2,3,4,6}.
 *  scales uint8 [d_o][d_i/16] : OCP FP8 E4M3 ("FN") block scale of weights
 *                               (o, 16j .. 16j+15).
 *  s_g    float [1]           : FP32 tensor scale (device memory).
 *  Blocks of 16 run along d_i, so d_i % 16 == 0.  Total 9*d_o*d_i/16 bytes + 4.
 */
#ifndef PRECISION_LINEAR_H
#define PRECISION_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pl_stream_t;

/* Element type of an output buffer.  Arithmetic is FP32 either way; a BF16
 * output is the round-to-nearest-even BF16 of exactly the FP32 value the FP32
 * output would hold. */
typedef enum pl_dtype {
  PL_DTYPE_BF16 = 0,
  PL_DTYPE_F32 = 1
} pl_dtype;

typedef enum pl_status {
  PL_OK = 0,
  PL_ERR_NULL = 1,      /* a required pointer is NULL                         */
  PL_ERR_SHAPE = 2,     /* a size is out of range or breaks a divisibility rule */
  PL_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned                   */
  PL_ERR_RANK = 4,      /* LoRA rank out of range (0..64)                     */
  PL_ERR_DEVICE = 5,    /* no current CUDA device of compute capability 10.3  */
  PL_ERR_CUDA = 6,      /* a CUDA runtime call or kernel launch failed        */
  PL_ERR_WORKSPACE = 7, /* workspace NULL, misaligned or smaller than needed  */
  PL_ERR_TIMEOUT = 8,   /* a bounded device-side wait gave up                 */
  PL_ERR_RANGE = 9,     /* reserved: an intermediate left its number format's
                           range (no current path raises it)                  */
  PL_ERR_OVERLAP = 10   /* a batch's output overlaps another output or an input */
} pl_status;

/* Static, human-readable name of a status code.  Never NULL. */
const char* pl_status_string(pl_status status);

/* ABI version of this header (major * 100 + minor): 200 (z_ld added to
 * pl_rmsnorm_aqn and pl_nvfp4_lora_linear). */
int pl_version(void);

/* Bytes of the packed NVFP4 payload plus block scales for a [d_o, d_i] weight:
 * d_o*d_i/2 + d_o*d_i/16 (= 9P/16, QeRL review section 3.1 memory equation),
 * not counting the 4-byte tensor scale.  0 if the shape is invalid. */
size_t pl_nvfp4_bytes(int64_t d_o, int64_t d_i);

/* Workspace bytes pl_nvfp4_lora_linear needs for this shape (any path the
 * library may choose for it).  The workspace is caller-owned device memory,
 * 256-byte aligned, reusable across calls on one stream; its contents on entry
 * do not matter.  Calls that run concurrently need separate workspaces. */
size_t pl_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r);

/* NVFP4 quantiser (section 3.1, "Quantize values to E2M1 codes; retain block
 * E4M3 scales and tensor-global scales" in the backbone-preparation algorithm).
 *
 *  W_bf16  in : BF16 [d_o][d_i], finite values.
 *  codes   out: uint8 [d_o][d_i/2]  (layout above)
 *  scales  out: uint8 [d_o][d_i/16]
 *  s_g     out: float[1], device
 * Arithmetic (bit-exact contract, FP32 IEEE round-to-nearest):
 *  s_g = max|W| / 2688 (2688 = 6*448; 1 if W is all zero);
 *  s_b = E4M3_rne_satfinite( amax_block / (6*s_g) );
 *  code = nearest E2M1 value to |w| / (s_g*s_b), ties to the even code,
 *         saturating at 6, sign from w, +0 for zero; 0 when s_g*s_b == 0.
 * Requirements: d_o >= 1, 1 <= d_i, d_i % 16 == 0; W, codes 16-byte aligned.
 * Launches three kernels (tensor amax, block quantise, scale finalise) after a
 * 4-byte memset of s_g, which serves as the amax accumulator until the end. */
pl_status pl_nvfp4_quantize(const void* W_bf16, int64_t d_o, int64_t d_i,
                            uint8_t* codes, uint8_t* scales, float* s_g,
                            pl_stream_t stream);

/* Update-aware quantisation fold ("QuRL: Low-Precision Reinforcement Learning for
 * Efficient Reasoning", reading notes section 3: a linear layer is invariant under
 * W X = (W / s)(s X), the factor on X absorbed by the normalisation before it; the
 * method folds s > 1, once, before training; s = 1.5 in its runs).
 *
 * pl_nvfp4_quantize_uaq: pl_nvfp4_quantize of W' = fp32(W / s) (IEEE division of every
 *   weight): s_g = fp32(max|W'| / 2688), block scales and codes of W' under the same
 *   contract.  s == 1 is exactly pl_nvfp4_quantize.  Requirements as pl_nvfp4_quantize,
 *   plus s finite and > 0 (PL_ERR_SHAPE).  For s >= 1 (the method's own setting) every
 *   W / s is finite; for s < 1 the caller must keep max|W| / s below the FP32 maximum
 *   (3.4e38), else s_g, scales and codes are not meaningful (not checked).
 * pl_uaq_fold_norm: out[i] = fp32(w_norm[i] * s), i < d (FP32 [d] in and out, device,
 *   4-byte aligned; out may equal w_norm).  Requirements: 1 <= d <= 2^40, s finite and > 0
 *   (PL_ERR_SHAPE), pointers non-NULL (PL_ERR_NULL) and 4-byte aligned (PL_ERR_ALIGN); one
 *   kernel launch, asynchronous.  The folded pair (W', w') gives the same layer up to the
 *   quantisation of W'. */
pl_status pl_nvfp4_quantize_uaq(const void* W_bf16, int64_t d_o, int64_t d_i, float s,
                                uint8_t* codes, uint8_t* scales, float* s_g, pl_stream_t stream);
pl_status pl_uaq_fold_norm(const float* w_norm, int64_t d, float s, float* out, pl_stream_t stream);

/* The AQN noise state z of a call (section 5.1 folds it into the norm scale; section 6,
 * "A training algorithm that exposes the stochastic state", lets the caller declare its
 * persistence scope: one state per rollout, per response or per token).
 *  z NULL     : no noise.
 *  z_ld == 0  : z is one FP32 vector [d], the state of every token row (per-rollout
 *               scope, or any call whose rows share a state).
 *  z_ld >= d  : z holds one FP32 vector per token row: row m's state starts at
 *               z + m * z_ld (per-response or per-token scope in a batched call; e.g.
 *               the [n_scopes][d] output of pl_aqn_noise with z_ld = d).
 * z_ld must be 0 or a multiple of 4 that is >= d (else PL_ERR_SHAPE). */

/* RMSNorm with AQN noise folded into the scale (section 5.1):
 *   h[m, :] = x[m, :] / sqrt(mean_j x[m, j]^2 + eps) (.) (w_norm + z_m)
 *  x_bf16 in : BF16 [M][d];  w_norm in: FP32 [d];  z, z_ld: the noise state (above),
 *  z_m its vector for row m;  h out: [M][d] of h_dtype (BF16 rounds to nearest even).
 *  w_norm + z_m is formed in FP32.  Requirements: M >= 1, d >= 8, d % 8 == 0, x and h
 *  16-byte aligned, z 16-byte aligned, h_dtype a pl_dtype. */
pl_status pl_rmsnorm_aqn(const void* x_bf16, int64_t M, int64_t d,
                         const float* w_norm, const float* z, int64_t z_ld, float eps,
                         void* h, int h_dtype, pl_stream_t stream);

/* The quantised-backbone LoRA linear (section 2.1 forward map, with the
 * section 5.1 prologue when w_norm is given):
 *   h = RMSNorm_AQN(x; w_norm, z, eps)   if w_norm != NULL,  else h = x;
 *   y[m, o] = sum_k W_hat[o, k] h[m, k] + lambda * sum_j B[o, j] (sum_k A[j, k] h[m, k])
 *  x_bf16  in : BF16 [M][d_i]
 *  codes, scales, s_g in: NVFP4 weight [d_o][d_i] (layout above)
 *  A_bf16  in : BF16 [r][d_i], B_bf16 in: BF16 [d_o][r]; both NULL or r == 0
 *               means no adapter.
 *  w_norm  in : FP32 [d_i] or NULL (no norm: z is then ignored)
 *  z, z_ld in : the noise state (above) over d = d_i
 *  y       out: [M][d_o] of y_dtype (a pl_dtype)
 *  workspace  : device scratch of at least pl_workspace_bytes(M, d_i, d_o, r).
 * Accumulation is FP32.  M <= 64 runs the decode path, larger M the prefill
 * path; both use tcgen05 tensor cores when d_i % 256 == 0 and a generic CUDA-core
 * kernel otherwise.  Requirements: M >= 1, d_o >= 1, d_i >= 16, d_i % 16 == 0,
 * 0 <= r <= 64; x, codes, scales, A, B, w_norm, z, y 16-byte aligned. */
pl_status pl_nvfp4_lora_linear(const void* x_bf16, int64_t M, int64_t d_i, int64_t d_o,
                               const uint8_t* codes, const uint8_t* scales, const float* s_g,
                               const void* A_bf16, const void* B_bf16, int r, float lambda,
                               const float* w_norm, const float* z, int64_t z_ld, float eps,
                               void* y, int y_dtype, void* workspace, size_t workspace_bytes,
                               pl_stream_t stream);

/* A group of projections that read the same input: in a decoder layer the projections
 * behind one RMSNorm (q, k and v behind the attention norm; gate and up behind the FFN
 * norm) share x, w_norm and the noise state z (QeRL section 5.1, "Deriving the RMSNorm
 * identity": one noise vector is folded into each norm, so Q, K and V share one and
 * Gate and Up the other).  One projection of a group: */
typedef struct pl_nvfp4_proj {
  int64_t d_o;             /* output features of this projection                        */
  const uint8_t* codes;    /* NVFP4 weight [d_o][d_i] (layout above)                     */
  const uint8_t* scales;
  const float* s_g;        /* device scalar                                               */
  const void* A_bf16;      /* BF16 [r][d_i] or NULL (with B_bf16 NULL or r == 0: no adapter) */
  const void* B_bf16;      /* BF16 [d_o][r] or NULL                                       */
  int r;                   /* 0 .. 64                                                     */
  float lambda;
  void* y;                 /* [M][d_o] of the group's y_dtype                             */
} pl_nvfp4_proj;

/* Most projections in one group call. */
#define PL_MAX_GROUP 8

/* Workspace bytes pl_nvfp4_lora_linear_group needs (0 for an invalid group). */
size_t pl_workspace_bytes_group(int64_t M, int64_t d_i, const pl_nvfp4_proj* projs, int n_proj);

/* pl_nvfp4_lora_linear of every projection of `projs` on the same x, w_norm, z, z_ld and
 * eps: y_p = W_hat_p h + lambda_p B_p (A_p h), h = RMSNorm_AQN(x) (x when w_norm is NULL).
 * Results equal those of separate calls within the linear's tolerance.  For decode batch
 * sizes (M <= 64, d_i % 256 == 0, at most 4 projections, sum of ranks <= 128) the group
 * runs as one prologue (h once, t_p = A_p h once per projection) and one main kernel over
 * the weight tiles of all projections.  For large M (M > 64, d_i % 256 == 0, at most 4
 * projections, ranks <= 32) it runs as one row pass (h / c_m once), one adapter
 * down-projection per projection and one contraction over the weight tiles of all
 * projections.  Otherwise the projections run one after another.
 * Requirements: those of pl_nvfp4_lora_linear for every projection, 1 <= n_proj <=
 * PL_MAX_GROUP; the y buffers must not overlap one another or any input.  `projs` is a
 * HOST array, read during the call only. */
pl_status pl_nvfp4_lora_linear_group(const void* x_bf16, int64_t M, int64_t d_i,
                                     const float* w_norm, const float* z, int64_t z_ld, float eps,
                                     const pl_nvfp4_proj* projs, int n_proj, int y_dtype,
                                     void* workspace, size_t workspace_bytes, pl_stream_t stream);

/* W8A8 rollout linear ("QuRL: Low-Precision Reinforcement Learning for Efficient
 * Reasoning", reading notes, "method / overall framework": the actor is quantised before
 * rollout with one scale per output channel for the weights and one per token for the
 * activations, INT8 or FP8; rollout runs on 8-bit matrix products).  This library takes the
 * FP8 E4M3 form (the 8-bit tensor-core rate of this part).  Symmetric absmax scales, no
 * zero point:
 *   s_w[o] = max_k |W[o, k]| / 448,  q_w = E4M3(W / s_w)       (pl_w8a8_quantize_weight)
 *   s_x[m] = max_k |h[m, k]| / 448,  q_x = E4M3(h / s_x),  h = RMSNorm_AQN(x)
 *   y[m, o] = s_x[m] s_w[o] sum_k q_x[m, k] q_w[o, k] + lambda sum_j B[o, j] (A h)[m, j]
 * with the adapter on the unquantised h, as on the NVFP4 path.  FP32 IEEE arithmetic for the
 * scales and quotients, round to nearest even onto E4M3, saturating at 448, +0 for values
 * that round to zero, s = 1 for an all-zero row.
 *
 * pl_w8a8_quantize_weight: W_bf16 BF16 [d_o][d_i] in; codes uint8 [d_o][d_i] and s_w FP32
 *   [d_o] out (device).  Bit-exact contract.  Requirements: d_o >= 1, d_i >= 16, d_i % 16 == 0,
 *   W and codes 16-byte aligned, s_w 4-byte aligned.  One kernel launch.
 * pl_w8a8_lora_linear: arguments as pl_nvfp4_lora_linear, with the weight given as codes and
 *   s_w.  Requirements: 1 <= M <= 2^24, 128 <= d_i <= 32768, d_i % 128 == 0, 0 <= r <= 64,
 *   alignment as pl_nvfp4_lora_linear, a workspace of pl_w8a8_workspace_bytes.  Two kernel
 *   launches (activation prologue, FP8 tensor-core GEMM), asynchronous. */
size_t pl_w8a8_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r);
pl_status pl_w8a8_quantize_weight(const void* W_bf16, int64_t d_o, int64_t d_i, uint8_t* codes, float* s_w,
                                  pl_stream_t stream);
pl_status pl_w8a8_lora_linear(const void* x_bf16, int64_t M, int64_t d_i, int64_t d_o,
                              const uint8_t* codes, const float* s_w,
                              const void* A_bf16, const void* B_bf16, int r, float lambda,
                              const float* w_norm, const float* z, int64_t z_ld, float eps,
                              void* y, int y_dtype, void* workspace, size_t workspace_bytes,
                              pl_stream_t stream);

/* Backward of the frozen-backbone linear (QeRL section 2.1, "Weight storage and trainable
 * state are different budgets": the quantised backbone is frozen, the gradients train A and
 * B and still pass through the frozen projection to the layers before it), with the
 * RMSNorm-AQN prologue's backward when w_norm is given (w_norm and z are not trained):
 *   u  = lambda g B;   dh = g W_hat + u A;   dA = u^T h;   dB = lambda g^T (h A^T)
 *   dx = rho s (.) dh - rho^3 x (sum_j x_j s_j dh_j) / d_i,  s = w_norm + z_m,
 *   rho = (mean_j x_j^2 + eps)^(-1/2),  h = RMSNorm_AQN(x)   (h = x and dx = dh without norm)
 *  g_bf16 in : BF16 [M][d_o], the upstream gradient dL/dy
 *  codes, scales, s_g, A_bf16, B_bf16, r, lambda: the forward call's weight and adapter
 *  x_bf16 in : BF16 [M][d_i], the forward input; w_norm, z, z_ld, eps as in the forward
 *  dx     out: FP32 [M][d_i];  dA out: FP32 [r][d_i] or NULL;  dB out: FP32 [d_o][r] or NULL
 *  workspace : pl_backward_workspace_bytes(M, d_i, d_o, r, w_norm != NULL), 256-byte aligned.
 * All contractions on tensor cores with BF16 operands (W_hat and g exact; h, u and h A^T
 * rounded to BF16) and FP32 accumulation; every sum in a fixed order (repeatable bit for
 * bit).  Requirements: M >= 1, d_i >= 256, d_i % 256 == 0, d_o % 8 == 0, 0 <= r <= 64; g,
 * codes, scales, x, dx, A, B, w_norm, z, dA 16-byte aligned, dB 4-byte aligned.  Up to
 * eight kernel launches, asynchronous. */
size_t pl_backward_workspace_bytes(int64_t M, int64_t d_i, int64_t d_o, int r, int with_norm);
pl_status pl_nvfp4_lora_linear_backward(const void* g_bf16, int64_t M, int64_t d_i, int64_t d_o,
                                        const uint8_t* codes, const uint8_t* scales, const float* s_g,
                                        const void* A_bf16, const void* B_bf16, int r, float lambda,
                                        const void* x_bf16, const float* w_norm, const float* z,
                                        int64_t z_ld, float eps, float* dx, float* dA, float* dB,
                                        void* workspace, size_t workspace_bytes, pl_stream_t stream);

/* A batch of independent calls of the linear, each with its own input: e.g. the
 * projections of several decode streams, or of one layer whose projections read different
 * inputs.  One call of a batch (every field as the argument of the same name of
 * pl_nvfp4_lora_linear): */
typedef struct pl_nvfp4_call {
  const void* x_bf16;      /* BF16 [M][d_i]                                               */
  int64_t M;
  int64_t d_o;
  const uint8_t* codes;
  const uint8_t* scales;
  const float* s_g;
  const void* A_bf16;
  const void* B_bf16;
  int r;
  float lambda;
  const float* w_norm;
  const float* z;
  int64_t z_ld;
  void* y;                 /* [M][d_o] of the batch's y_dtype                             */
} pl_nvfp4_call;

/* Most calls in one batch. */
#define PL_MAX_BATCH 8

/* Workspace bytes pl_nvfp4_lora_linear_batch needs (0 for an invalid batch). */
size_t pl_workspace_bytes_batch(int64_t d_i, const pl_nvfp4_call* calls, int n_calls);

/* Every call of `calls` (a HOST array, read during the call only), with the same d_i and
 * eps: results equal those of separate pl_nvfp4_lora_linear calls within the linear's
 * tolerance.  The calls must be independent: no call's y may overlap another call's y or
 * any call's x (else PL_ERR_OVERLAP, nothing launched).  Calls with the same x, M, w_norm,
 * z and z_ld share one prologue row pass (a group).  For decode batch sizes (every M <= 64,
 * d_i % 256 == 0, at most 8 calls, at most 4 calls per distinct input) the batch runs as one
 * prologue and one main kernel over the weight tiles of every call, so that the weight
 * streams of the calls overlap; otherwise the calls run one after another.  Requirements:
 * those of pl_nvfp4_lora_linear for every call, 1 <= n_calls <= PL_MAX_BATCH. */
pl_status pl_nvfp4_lora_linear_batch(int64_t d_i, float eps, const pl_nvfp4_call* calls, int n_calls,
                                     int y_dtype, void* workspace, size_t workspace_bytes,
                                     pl_stream_t stream);

/* Bytes of the scratch array behind pl_nvfp4_lora_linear_static_ws. */
#define PL_STATIC_WORKSPACE_BYTES ((size_t)8 << 20)

/* pl_nvfp4_lora_linear without a caller-provided workspace.  (No counterpart in
 * the pages: it is an interface convenience, not part of the method.)
 *
 * For callers that cannot allocate device memory themselves -- for example a
 * plug-in that receives only raw input and output pointers from a host program
 * owning every allocation, or a serving loop that must not call cudaMalloc because
 * it synchronises the device and the caching allocator is out of reach.  The
 * caller still passes all inputs and the output; the scratch the call needs lives
 * in one library-owned device array of PL_STATIC_WORKSPACE_BYTES (8 MiB) that
 * every device loading this library keeps until the process exits.
 *
 * Arguments, layouts, arithmetic and status codes are those of
 * pl_nvfp4_lora_linear with z_ld = 0 (one noise vector for every row); additionally
 * PL_ERR_WORKSPACE is returned, with nothing
 * launched, when pl_workspace_bytes(M, d_i, d_o, r) exceeds
 * PL_STATIC_WORKSPACE_BYTES (e.g. M = 64 decode fits for d_i up to 28672).
 * The call allocates nothing.  Every call looks up the array's device address on the
 * current device (cudaGetSymbolAddress; the first lookup on a device loads the module, so
 * make the first call on a device before any stream capture).  All calls share the one
 * array and it keeps the
 * last call's contents (nothing in it needs to start at zero): calls that may
 * overlap on the GPU -- on different streams, or concurrently from several host
 * threads -- race on it and must be serialised by the caller. */
pl_status pl_nvfp4_lora_linear_static_ws(const void* x_bf16, int64_t M, int64_t d_i, int64_t d_o,
                                         const uint8_t* codes, const uint8_t* scales, const float* s_g,
                                         const void* A_bf16, const void* B_bf16, int r, float lambda,
                                         const float* w_norm, const float* z, float eps,
                                         void* y, int y_dtype, pl_stream_t stream);

/* AQN noise state: the staged schedule (section 5.2), its stage (section 6) and the
 * device draw of z that pl_rmsnorm_aqn and pl_nvfp4_lora_linear take (section 5.1).
 *
 * pl_aqn_stage: the schedule stage after `done` of `total` planned updates, ten
 *   equal parts of the horizon: min(9, floor(10 done / total)); stage 0 is the
 *   warm-up without noise.  Host only.  Returns -1 when total < 1 or done < 0. */
int pl_aqn_stage(int64_t done, int64_t total);

/* pl_aqn_sigma: sigma_0 = 0 and, for k = 1 .. 9,
 *   sigma_k = sigma_start * (sigma_end / sigma_start) ^ ((k - 1) / 8),
 * so stage 1 is sigma_start and stage 9 sigma_end.  Computed in double, returned
 * rounded to float.  Host only.  Returns -1 for a stage outside 0 .. 9 or a start or
 * end that is not positive and finite. */
float pl_aqn_sigma(int stage, float sigma_start, float sigma_end);

/* pl_aqn_noise: z[s][j] = sigma * n_j(seed, norm_id, scope0 + s), s < n_scopes, j < d.
 * The state is a pure function of its arguments, so a rollout, a response or a token
 * (the persistence scope the caller declares through the scope index) replays it
 * exactly; norm_id names the RMSNorm (one vector per norm, shared by the projections
 * that read it).  Draws: Philox4x32-10 (Salmon et al., SC 2011) with key = seed (low
 * word first) and counter = (j / 4, norm_id, scope low word, scope high word); each
 * output word x gives u = (2 (x >> 9) + 1) * 2^-24; channels 4b, 4b+1 are rho cos(2 pi
 * u1), rho sin(2 pi u1) with rho = sqrt(-2 ln u0) from words 0..1 of block b, channels
 * 4b+2, 4b+3 the same from words 2..3; FP32 with the IEEE square root, logf and
 * sincospif, then times sigma.
 *  z out: FP32 [n_scopes][d], device, 4-byte aligned (caller-owned).
 * Requirements: 1 <= d <= 2^31, 1 <= n_scopes <= 2^31, d * n_scopes <= 2^40, sigma
 * finite and >= 0 (PL_ERR_SHAPE otherwise, nothing launched).  One kernel launch,
 * asynchronous on `stream`. */
pl_status pl_aqn_noise(uint64_t seed, uint32_t norm_id, uint64_t scope0, int64_t n_scopes, int64_t d,
                       float sigma, float* z, pl_stream_t stream);

/* Synchronises `stream`, then returns and clears the device status word: set by
 * bounded device-side waits that gave up (PL_ERR_TIMEOUT; that call's y is then not
 * valid), else PL_OK. */
pl_status pl_last_device_status(pl_stream_t stream);

/* Test hook: which kernel path pl_nvfp4_lora_linear takes for this shape on the
 * current device with one noise vector per call (z_ld = 0; with one per row, path 2 becomes
 * path 1): 2 = one fused tcgen05 kernel (every CTA's K slice on chip),
 * 1 = tcgen05 prologue + main kernel (M <= 64), 3 = large-M tcgen05 path (row
 * prologue, LoRA down-projection, persistent NVFP4 GEMM), 0 = generic CUDA-core
 * kernels, -1 = invalid shape or unsupported device.  Launches nothing. */
int pl_debug_linear_path(int64_t M, int64_t d_i, int64_t d_o, int r);

/* Test hook: when `armed` is non-zero the next launch-checking step of any call
 * reports a launch failure (PL_ERR_CUDA) as if the CUDA runtime had returned
 * one, without faulting anything.  One-shot; 0 disarms. */
void pl_debug_fail_next_launch(int armed);

/* Test hook: launches one tiny kernel whose bounded wait on a barrier that nothing
 * completes gives up after 2 ms, exactly as a stalled pipeline wait would; the
 * device status word then reads PL_ERR_TIMEOUT through pl_last_device_status.
 * Faults nothing and leaves the context usable. */
pl_status pl_debug_wait_timeout_probe(pl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PRECISION_LINEAR_H */
