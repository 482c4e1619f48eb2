/*
 * coda.h -- C ABI of the GB300 (sm_103a) fused GEMM-epilogue library.
 *
 * The library implements the hot path of "CODA: Rewriting Transformer Blocks
 * as GEMM-Epilogue Programs", forward and backward, as the CODA news write-up
 * describes it
 * (KuCoin news, "CODA new research optimizes transformer training with
 * GEMM-epilogue programming"; the same article on itsolotime.com and on
 * KuCoin's Arabic site):
 *
 *   section "CODA: the treasure hidden in the epilogue":
 *     GEMM -> residual add -> RMSNorm -> GEMM.  RMSNorm's per-row scale r is a
 *     scalar shared by the whole row, so it commutes with the next matmul and
 *     can be applied in the second GEMM's epilogue; the first GEMM's epilogue
 *     then only computes local partial RMS statistics, which a very light
 *     auxiliary reduction kernel folds into r.  SwiGLU admits the same
 *     reparameterisation.
 *   section "five blocks and a Lego language":
 *     the epilogue primitives used here -- element-wise transforms (residual
 *     add, activation), vector load (the broadcast RMSNorm weight, folded into
 *     the next weight here) and block reduction (local RMS).
 *
 * The block computed by a chain of calls (row i of M tokens, hidden width N):
 *     h    = R + X . W1                                coda_gemm_residual_partial_rms
 *     r_i  = 1 / sqrt(mean_j h_ij^2 + eps)             coda_rms_reduce
 *     W2'  = diag(gamma) . W2                          coda_fold_gamma (once per weight)
 *     Z    = diag(r) . h . W2'      == RMSNorm(h).W2   coda_gemm_rowscale
 *     act  = silu(r h Wg') * (r h Wu')                 coda_gemm_swiglu
 * with RMSNorm(h)_ij = h_ij * r_i * gamma_j and silu(x) = x / (1 + e^-x).
 * Further calls fold r into the consumer GEMM (coda_gemm_*_fused_rms), run a
 * residual GEMM and its consumer as one launch (coda_block_*), rotate Q and K
 * in the QKV GEMM's epilogue (coda_gemm_rowscale_rope), give the backward of
 * the block (coda_gemm_grad_norm, coda_rmsnorm_backward, coda_gemm with
 * either operand layout, coda_gemm_swiglu_save / coda_gemm_swiglu_backward),
 * quantise to FP8 (coda_amax, coda_quantize_e4m3), and run an FP8 block in
 * one launch that quantises its own operands (coda_block_*_fp8).
 *
 * Conventions shared by every call
 *   - Matrices are row-major.  Activations are [rows, K]; a weight W [K, N]
 *     is passed as its transpose W^T [N, K] (the nn.Linear weight layout), so
 *     both GEMM operands are K-major.
 *   - Pointers are DEVICE pointers unless stated otherwise, 16-byte aligned.
 *     Every row of every matrix must start on a 16-byte boundary: K and the
 *     output width must be multiples of 4 (CODA_F32), 8 (CODA_BF16) or 16
 *     (CODA_E4M3 operands).
 *   - Sizes are int64_t; M may be 0 (nothing is launched), N and K must be
 *     positive; every dimension must be below 2^31, every matrix below 2^60
 *     elements, and a GEMM below 2^30 output tiles of 128 x 128.
 *   - Ownership: the caller owns all memory.  The library never allocates,
 *     frees or synchronises; every call only enqueues work on `stream`
 *     (cudaStream_t; NULL = the legacy default stream) and returns.
 *   - Outputs must not overlap any input or each other (checked on the
 *     address ranges; CODA_ERR_INVALID_ARG otherwise).
 *   - Errors: argument checks run before anything is enqueued and return
 *     CODA_ERR_INVALID_ARG (nothing written); CUDA errors from encoding or
 *     launching return CODA_ERR_CUDA.  coda_last_error() describes the last
 *     failure of the calling thread.  Device-side wait timeouts (a kernel
 *     that gave up instead of hanging) are reported by coda_get_device_status().
 *   - dtype: CODA_F32 = fp32 operands and outputs (tensor cores in tf32 with
 *     fp32 accumulation); CODA_BF16 = bf16 operands and outputs (fp32
 *     accumulation); CODA_E4M3 = OCP FP8 e4m3 GEMM operands, each with a
 *     per-tensor fp32 dequantisation scale (device pointer), fp32
 *     accumulation, bf16 residual and outputs.
 */
#ifndef CODA_H_
#define CODA_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define CODA_API __attribute__((visibility("default")))
#else
#define CODA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CODA_OK = 0,
  CODA_ERR_INVALID_ARG = 1,
  CODA_ERR_UNSUPPORTED = 2,
  CODA_ERR_CUDA = 3,
  CODA_ERR_TIMEOUT = 4
} coda_status;

typedef enum { CODA_F32 = 0, CODA_BF16 = 1, CODA_E4M3 = 2 } coda_dtype;

/* Storage of a GEMM operand: CODA_K_MAJOR = rows of the output dimension
 * with K contiguous ([M, K] / [N, K]); CODA_MN_MAJOR = rows of K with the
 * output dimension contiguous ([K, M] / [K, N], i.e. the transpose). */
typedef enum { CODA_K_MAJOR = 0, CODA_MN_MAJOR = 1 } coda_layout;

/* Library version, major * 10000 + minor * 100 + patch. */
CODA_API int coda_version(void);

/* Human-readable name of a status code (static string). */
CODA_API const char* coda_status_string(coda_status s);

/* Message describing the last failed call on this host thread (static,
 * thread-local storage; "" if none). */
CODA_API const char* coda_last_error(void);

/* Number of partial-sum columns T = ceil(N / 128) that
 * coda_gemm_residual_partial_rms writes per row for hidden width N: the
 * caller allocates P as fp32 [M, T].  Returns -1 for N <= 0. */
CODA_API int64_t coda_partial_cols(int64_t N);

/* One-time weight transform W' = diag(gamma) . W (not on the pages as a
 * separate step: it is where the broadcast RMSNorm weight of the "five
 * blocks" section goes once r has been moved past the GEMM).
 *   Wt      [N_out, K] input weight W^T (dtype CODA_F32 or CODA_BF16)
 *   gamma   [K] fp32 RMSNorm weight of the hidden dimension K
 *   Wt_out  [N_out, K] output W'^T, same dtype: Wt_out[n, k] = Wt[n, k] * gamma[k]
 *           (computed in fp32, rounded to nearest-even once).  May not alias Wt.
 * For FP8, fold in bf16 or fp32 first, then coda_amax + coda_quantize_e4m3. */
CODA_API coda_status coda_fold_gamma(const void* Wt, const float* gamma, void* Wt_out, int64_t N_out, int64_t K,
                            coda_dtype dtype, cudaStream_t stream);

/* GEMM1 with the residual add and the partial RMS statistics in its epilogue
 * (section "CODA: the treasure hidden in the epilogue"):
 *   h[i, j]  = R[i, j] + sum_k X[i, k] * W1t[j, k]        (fp32 accumulate, stored
 *                                                           rounded to the output type)
 *   P[i, g]  = sum over j in [128 g, 128 g + 128) of h[i, j]^2   (of the stored h)
 *   X   [M, K]   dtype operands (CODA_E4M3: e4m3 bytes)
 *   W1t [N, K]   dtype operands
 *   R   [M, N]   residual: fp32 for CODA_F32, else bf16
 *   H   [M, N]   output h, same type as R.  Must not alias R.
 *   P   [M, coda_partial_cols(N)] fp32 output
 *   scale_x, scale_w: CODA_E4M3 only (device fp32 scalars; the product
 *           X.W1t is multiplied by *scale_x * *scale_w); must be NULL otherwise.
 *   amax_h: nullable device fp32 scalar; when given it receives max |h|
 *           (overwritten, not accumulated), for quantising h to FP8 next. */
CODA_API coda_status coda_gemm_residual_partial_rms(const void* X, const void* W1t, const void* R, void* H, float* P,
                                           int64_t M, int64_t N, int64_t K, coda_dtype dtype,
                                           const float* scale_x, const float* scale_w, float* amax_h,
                                           cudaStream_t stream);

/* The auxiliary reduction ("a very light auxiliary reduction kernel"):
 *   r[i] = 1 / sqrt( (sum_g P[i, g]) / N + eps )
 *   P [M, coda_partial_cols(N)] fp32 partials of a hidden width N; r [M] fp32.
 *   eps >= 0 and finite. */
CODA_API coda_status coda_rms_reduce(const float* P, int64_t M, int64_t N, float eps, float* r, cudaStream_t stream);

/* GEMM2 with RMSNorm's row scale applied in its epilogue:
 *   Z[i, n] = r[i] * sum_k H[i, k] * W2t[n, k]
 * which equals RMSNorm(h) . W2 when W2t = (diag(gamma) W2)^T from coda_fold_gamma.
 *   H [M, K], W2t [N2, K] dtype operands; r [M] fp32 (required);
 *   Z [M, N2]: fp32 for CODA_F32, else bf16.
 *   scale_h, scale_w: as for coda_gemm_residual_partial_rms. */
CODA_API coda_status coda_gemm_rowscale(const void* H, const void* W2t, const float* r, void* Z, int64_t M, int64_t N2,
                               int64_t K, coda_dtype dtype, const float* scale_h, const float* scale_w,
                               cudaStream_t stream);

/* RoPE in the QKV GEMM's epilogue (the CODA write-up, section "CODA: the
 * treasure hidden in the epilogue", lists rotary position embedding among the
 * operations the same reparameterisation moves into an epilogue).  Reading:
 * RoFormer's rotation with interleaved pairs.  For output row i at position
 * p_i, every head of head_dim columns among the first rope_cols columns (the
 * Q and K heads of a fused QKV weight; V follows unrotated), and pair j:
 *   phi = p_i * base^(-2j / head_dim)
 *   (z_2j, z_2j+1) <- (z_2j cos phi - z_2j+1 sin phi, z_2j sin phi + z_2j+1 cos phi)
 * applied in fp32 to Z = r * (H . W2t^T) before the single rounding to the
 * output type.  The angle is formed in fp32 and reduced by whole turns, so its
 * error is about 1.2e-7 * phi radians (2.4e-4 at phi = 2047).
 *
 * As coda_gemm_rowscale (r given) or coda_gemm_rowscale_fused_rms (P and eps
 * given, r_out nullable): exactly one of r and P.
 *   head_dim: a multiple of 8 (bf16, e4m3 operands) or 4 (fp32);
 *   rope_cols: a multiple of head_dim, at most N2 (0 = no rotation);
 *   base: finite, > 1 (500000 for LLaMA-3);
 *   positions: [M] int32, or NULL for p_i = i mod seq_len (rows batch-major). */
CODA_API coda_status coda_gemm_rowscale_rope(const void* H, const void* W2t, const float* r, const float* P,
                                             float eps, float* r_out, void* Z, int64_t M, int64_t N2, int64_t K,
                                             coda_dtype dtype, const float* scale_h, const float* scale_w,
                                             int64_t head_dim, int64_t rope_cols, double base, int64_t seq_len,
                                             const int32_t* positions, cudaStream_t stream);

/* Gate/up GEMM with SwiGLU (and the row scale) in its epilogue:
 *   G = r . (H . Wgt^T),  U = r . (H . Wut^T)   (row scale applied to both
 *   before the non-linearity),  Act[i, n] = silu(G[i, n]) * U[i, n]
 *   H [M, K], Wgt [I, K], Wut [I, K] dtype operands; r [M] fp32 or NULL (= 1);
 *   Act [M, I]: fp32 for CODA_F32, else bf16.
 *   scale_h, scale_wg, scale_wu: CODA_E4M3 only, NULL otherwise.
 *   amax_act: nullable; receives max |Act| (overwritten). */
CODA_API coda_status coda_gemm_swiglu(const void* H, const void* Wgt, const void* Wut, const float* r, void* Act, int64_t M,
                             int64_t I, int64_t K, coda_dtype dtype, const float* scale_h, const float* scale_wg,
                             const float* scale_wu, float* amax_act, cudaStream_t stream);

/* The auxiliary reduction folded into the second GEMM (the natural next step
 * after section "CODA: the treasure hidden in the epilogue" calls the
 * reduction "very light"): as coda_gemm_rowscale, except that each epilogue
 * thread reduces its own row's partial sums of squares to r exactly as
 * coda_rms_reduce does (same summation order, so the same bits), saving one
 * launch and the round trip of r.
 *   P [M, coda_partial_cols(K)] fp32: the partials written by the
 *     coda_gemm_residual_partial_rms that produced h (RMSNorm width = K here);
 *     for CODA_E4M3, H is the quantised h and P still comes from the bf16 h.
 *   eps: finite, >= 0.
 *   r_out: nullable; receives r [M] (written once per row).
 * Other arguments as for coda_gemm_rowscale. */
CODA_API coda_status coda_gemm_rowscale_fused_rms(const void* H, const void* W2t, const float* P, float eps,
                                                  float* r_out, void* Z, int64_t M, int64_t N2, int64_t K,
                                                  coda_dtype dtype, const float* scale_h, const float* scale_w,
                                                  cudaStream_t stream);

/* coda_gemm_swiglu with the reduction folded in, as for
 * coda_gemm_rowscale_fused_rms: r is computed per row from P (K columns of h)
 * and applied to gate and up before silu; r_out nullable. */
CODA_API coda_status coda_gemm_swiglu_fused_rms(const void* H, const void* Wgt, const void* Wut, const float* P,
                                                float eps, float* r_out, void* Act, int64_t M, int64_t I, int64_t K,
                                                coda_dtype dtype, const float* scale_h, const float* scale_wg,
                                                const float* scale_wu, float* amax_act, cudaStream_t stream);

/* The whole block in ONE persistent launch: GEMM1 with the residual add and
 * partial RMS, then the consuming GEMM with the reduction folded into its
 * epilogue (the single-launch chain that the "very light" reduction of
 * section "CODA: the treasure hidden in the epilogue" makes possible).  The
 * consuming GEMM's tiles of a row band start as soon as every GEMM1 tile of
 * that band has stored h and P, filling the SMs that GEMM1's last wave leaves
 * idle.  Results equal the separate calls bit for bit.
 *   coda_block_rowscale:  h = R + X.W1t^T, P, r (r_out, nullable), Z = diag(r) h W2t^T
 *   coda_block_swiglu:    h, P, r, Act = silu(r h Wgt^T) * (r h Wut^T)
 *   X [M, K]; W1t [N, K]; R, H [M, N]; P [M, coda_partial_cols(N)] fp32;
 *   W2t [N2, N] / Wgt, Wut [I, N] (gamma folded in); Z [M, N2] / Act [M, I].
 *   dtype: CODA_F32 or CODA_BF16 (CODA_E4M3 -> CODA_ERR_UNSUPPORTED: FP8
 *     quantises h with its per-tensor amax, which needs all of h first).
 *   workspace: device memory of coda_block_workspace_bytes(M) bytes, zeroed
 *     by the caller before its first use; every call leaves it zeroed again
 *     (the last CTA to finish resets it), so it can be reused without a
 *     memset.  Calls that share a workspace must not overlap on the GPU.
 *   Co-residency: the band waits need every CTA of the grid resident at
 *   once.  The grid never exceeds the CTAs that fit on an idle GPU, and the
 *   kernel is launched cooperatively, which makes the runtime either start
 *   the whole grid together or fail the launch (CODA_ERR_CUDA).  If a device
 *   or runtime refuses a cooperative launch of a clustered grid, the library
 *   notes that once per device and launches plainly from then on (as it
 *   does when the environment sets CODA_NO_COOPERATIVE, for profilers that
 *   cannot replay a cooperative clustered launch); the co-residency then
 *   rests on the caller: while such a launch runs, no
 *   kernel on another stream may hold SMs that its CTAs need.  If that
 *   contract is broken, a band wait runs out after 2 s and the call reports
 *   CODA_ERR_TIMEOUT through coda_get_device_status(), with partial outputs;
 *   it does not hang.  Every wait is bounded the same way. */
CODA_API int64_t coda_block_workspace_bytes(int64_t M);
CODA_API coda_status coda_block_rowscale(const void* X, const void* W1t, const void* R, const void* W2t, float eps,
                                         void* H, float* P, float* r_out, void* Z, int64_t M, int64_t N, int64_t K,
                                         int64_t N2, coda_dtype dtype, void* workspace, cudaStream_t stream);
CODA_API coda_status coda_block_swiglu(const void* X, const void* W1t, const void* R, const void* Wgt,
                                       const void* Wut, float eps, void* H, float* P, float* r_out, void* Act,
                                       int64_t M, int64_t N, int64_t K, int64_t I, coda_dtype dtype, void* workspace,
                                       cudaStream_t stream);

/* FP8 (e4m3) forms of the one-launch blocks (the CODA write-up, section "lazy
 * tax of large-model training": FP8 GEMMs make the memory-bound neighbours a
 * larger share of the step, which is what fusing them removes).  Per-tensor
 * scales s = amax / 448 (1 for an all-zero tensor), codes e4m3(x / s)
 * rounded to nearest even and saturated, exactly as coda_quantize_e4m3.
 * One launch computes, for the consumer Z / Act:
 *   [Aq = e4m3(A / scale_a), scale_a = amax_a / 448]   when A is given
 *   h = R + scale_a scale_w1 (Aq . W1t^T)              bf16, with P and
 *   amax_h = max |h|, then scale_h = amax_h / 448, Hq = e4m3(h / scale_h)
 *   r = 1 / sqrt(sum_g P[i, g] / N + eps)               (r_out, nullable)
 *   coda_block_rowscale_fp8: Z = r scale_h scale_w2 (Hq . W2t^T)       bf16
 *   coda_block_swiglu_fp8:   Act = silu(r s_h s_wg (Hq . Wgt^T)) *
 *                                  (r s_h s_wu (Hq . Wut^T))          bf16,
 *                            amax_act = max |Act| (nullable)
 * Results equal the separate calls (coda_quantize_e4m3, the e4m3 residual
 * GEMM, coda_quantize_e4m3 of h, the e4m3 consumer with the reduction
 * folded in) bit for bit.  Warps of every CTA quantise h band by band once
 * every CTA is past the residual GEMM; the consumer starts on a band as soon
 * as its e4m3 copy is complete.
 *   A [M, K] bf16, nullable: with A, amax_a (its max |x|, final before the
 *     call) is read and Aq [M, K] and scale_a are written by the launch;
 *     without A, Aq and scale_a are the given e4m3 operand and its scale.
 *   W1t [N, K], W2t [N2, N], Wgt, Wut [I, N]: e4m3 bytes (gamma folded in
 *     before quantising) with device scalar scales.  R [M, N] bf16.
 *   Outputs: H [M, N] bf16, P [M, coda_partial_cols(N)] fp32, amax_h, Hq
 *     [M, N] e4m3, scale_h, Z [M, N2] / Act [M, I] bf16, amax_act; the
 *     library zeroes amax_h and amax_act itself (asynchronously on stream).
 *   K, N multiples of 16; N2 / I multiples of 8.  M = 0 zeroes amax_h and
 *   amax_act and writes nothing else.
 *   workspace: coda_block_fp8_workspace_bytes(M) bytes, zeroed before its
 *     first use and left zeroed by every call; calls sharing it must not
 *     overlap on the GPU.  Co-residency and bounded waits as for
 *     coda_block_swiglu (CODA_ERR_TIMEOUT through coda_get_device_status()). */
CODA_API int64_t coda_block_fp8_workspace_bytes(int64_t M);
CODA_API coda_status coda_block_swiglu_fp8(const void* A, const float* amax_a, uint8_t* Aq, float* scale_a,
                                           const uint8_t* W1t, const float* scale_w1, const void* R,
                                           const uint8_t* Wgt, const float* scale_wg, const uint8_t* Wut,
                                           const float* scale_wu, float eps, void* H, float* P, float* r_out,
                                           float* amax_h, uint8_t* Hq, float* scale_h, void* Act, float* amax_act,
                                           int64_t M, int64_t N, int64_t K, int64_t I, void* workspace,
                                           cudaStream_t stream);
CODA_API coda_status coda_block_rowscale_fp8(const void* A, const float* amax_a, uint8_t* Aq, float* scale_a,
                                             const uint8_t* W1t, const float* scale_w1, const void* R,
                                             const uint8_t* W2t, const float* scale_w2, float eps, void* H, float* P,
                                             float* r_out, float* amax_h, uint8_t* Hq, float* scale_h, void* Z,
                                             int64_t M, int64_t N, int64_t K, int64_t N2, void* workspace,
                                             cudaStream_t stream);

/* coda_block_rowscale with RoPE on the consuming GEMM's leading columns (the
 * Q and K heads of a fused QKV weight), as coda_gemm_rowscale_rope does it:
 * the LLaMA block tail's next-layer QKV projection, normalised, projected and
 * rotated in the same launch as the down projection and its residual add.
 * head_dim, rope_cols, base, seq_len and positions as for
 * coda_gemm_rowscale_rope; the other arguments as for coda_block_rowscale. */
CODA_API coda_status coda_block_rowscale_rope(const void* X, const void* W1t, const void* R, const void* W2t,
                                              float eps, void* H, float* P, float* r_out, void* Z, int64_t M,
                                              int64_t N, int64_t K, int64_t N2, coda_dtype dtype, int64_t head_dim,
                                              int64_t rope_cols, double base, int64_t seq_len,
                                              const int32_t* positions, void* workspace, cudaStream_t stream);

/* coda_block_swiglu for callers that cannot allocate device memory (no
 * counterpart in the CODA write-ups: it exists for the way some programs
 * manage memory).  Runtimes that own all device memory and give a kernel
 * library no workspace, and hot paths that must not call cudaMalloc (which
 * may synchronise the device), can use this form: it takes no workspace and
 * allocates nothing.  Its band counters live in a fixed array inside the
 * library (4100 bytes on every GPU that loads it, held until the process
 * exits).
 *   Limit: M <= 131072 rows; larger M returns CODA_ERR_INVALID_ARG.
 *   The first call on a device looks up the array's device address for that
 *   device (with it current); make that first call before any stream capture.
 *   The address is kept for the life of the process: after cudaDeviceReset
 *   on a device, do not call this entry point on that device again.
 *   Arguments are checked before anything is enqueued: a rejected call
 *   leaves the shared array as it was.
 *   Every call shares the one array: each call zeroes the counters it uses
 *   (an asynchronous memset on `stream`) before its kernel, so calls that
 *   overlap on the GPU, on any streams, race and must not be issued.
 *   Other arguments and results as for coda_block_swiglu. */
CODA_API coda_status coda_block_swiglu_noalloc(const void* X, const void* W1t, const void* R, const void* Wgt,
                                               const void* Wut, float eps, void* H, float* P, float* r_out,
                                               void* Act, int64_t M, int64_t N, int64_t K, int64_t I,
                                               coda_dtype dtype, cudaStream_t stream);

/* General GEMM on the same tcgen05 kernels, for the transposed products of
 * the block's backward pass (dX = dh . W1, dW = X^T . dh, ...):
 *   D[m, n] = row_scale[m] * col_scale[n] * sum_k A(m, k) B(n, k)
 *   A(m, k) = A[m*K + k] (CODA_K_MAJOR) or A[k*M + m] (CODA_MN_MAJOR)
 *   B(n, k) = B[n*K + k] (CODA_K_MAJOR) or B[k*N + n] (CODA_MN_MAJOR)
 * row_scale [M], col_scale [N]: nullable fp32 (= 1).  D [M, N] in the output
 * type of dtype (fp32 for CODA_F32, else bf16).  dtype CODA_F32 or
 * CODA_BF16; MN-major operands are bf16 only, and an MN-major A needs an
 * MN-major B.  Every stored row must be a multiple of 16 bytes. */
CODA_API coda_status coda_gemm(const void* A, coda_layout a_layout, const void* B, coda_layout b_layout, void* D,
                               int64_t M, int64_t N, int64_t K, coda_dtype dtype, const float* row_scale,
                               const float* col_scale, cudaStream_t stream);

/* ---- Backward of the block (the CODA write-up, section "CODA: the treasure
 * hidden in the epilogue": when the forward epilogue is block-local the
 * backward inherits the same GEMM + epilogue structure).  bf16 only.
 * Forward being differentiated: h = R + X W1, r_i = 1/sqrt(mean_j h_ij^2 + eps),
 * y = h r gamma, then Z = y W2 or act = silu(y Wg) (y Wu).  Gradients:
 *   dy     = dZ . W2                    coda_gemm_grad_norm (also S)
 *   dh     = r gamma dy - h r^3/N sum_j gamma_j dy_j h_j (+ dH_in)
 *   dgamma = sum_i dy h r,  Yt = r h    coda_rmsnorm_backward
 *   dX = dh . W1^T, dW1 = X^T dh, dW2 = (Yt^T dZ) diag(gamma)   coda_gemm
 *   SwiGLU: dAct = dOut . Wd, dG = dAct U silu'(G), dU = dAct silu(G)
 *                                       coda_gemm_swiglu_backward
 */

/* dY = dOut . Wt with the row reduction of RMSNorm's backward in the epilogue:
 *   dY[i, j] = sum_k dOut[i, k] Wt[k, j]        (Wt [K, N]: the forward weight
 *                                                as stored, W^T of its GEMM)
 *   S[i, g]  = sum over j in [128 g, 128 g + 128) of gamma_j dY_ij H_ij
 *              (of the stored, rounded dY; H [M, N] is the forward's h)
 *   dOut [M, K], dY [M, N] bf16; gamma [N] fp32; S [M, coda_partial_cols(N)] fp32.
 * For the SwiGLU block, dOut = dG || dU [M, 2I] and Wt = Wg^T || Wu^T stacked
 * as [2I, N] (the forward's Wgt above Wut, unfolded). */
CODA_API coda_status coda_gemm_grad_norm(const void* dOut, const void* Wt, const void* H, const float* gamma,
                                         void* dY, float* S, int64_t M, int64_t N, int64_t K, coda_dtype dtype,
                                         cudaStream_t stream);

/* Elementwise RMSNorm backward from coda_gemm_grad_norm's dY and S:
 *   c_i = r_i^3 / N * sum_g S[i, g];  dH = r gamma dY - c H (+ dH_in);
 *   Yt = r H (the operand of the weight gradient);  dgamma_j = sum_i dY H r.
 * dY, H, dH_in (nullable), dH, Yt: [M, N] bf16; r [M], gamma [N], dgamma [N]
 * fp32.  workspace: coda_rmsnorm_backward_workspace_bytes(M, N) bytes of
 * device memory (dgamma partials, summed in a fixed order: deterministic).
 * N a multiple of 8. */
CODA_API int64_t coda_rmsnorm_backward_workspace_bytes(int64_t M, int64_t N);
CODA_API coda_status coda_rmsnorm_backward(const void* dY, const void* H, const float* r, const float* gamma,
                                           const float* S, const void* dH_in, void* dH, void* Yt, float* dgamma,
                                           float* workspace, int64_t M, int64_t N, cudaStream_t stream);

/* The forward SwiGLU GEMM that also saves its pre-activations for the
 * backward (the "matrix block store" primitive of the write-up's section
 * "five blocks and a Lego language"): as coda_gemm_swiglu (r given) or
 * coda_gemm_swiglu_fused_rms (P, eps, r_out), exactly one of r and P, plus
 *   GU [M, 2I] bf16: G = r (H Wgt^T) in columns [0, I), U = r (H Wut^T) in [I, 2I).
 * bf16 only; I a multiple of 64 (the G half is stored in 64-column boxes that
 * must not reach into the U half). */
CODA_API coda_status coda_gemm_swiglu_save(const void* H, const void* Wgt, const void* Wut, const float* r,
                                           const float* P, float eps, float* r_out, void* Act, void* GU, int64_t M,
                                           int64_t I, int64_t K, coda_dtype dtype, cudaStream_t stream);

/* SwiGLU backward in the epilogue of the GEMM that produces its upstream
 * gradient (the down projection's dAct = dOut . Wd):
 *   dAct[i, n] = sum_k dOut[i, k] Wt[k, n]    (Wt [K, I]: the down weight as stored)
 *   dG = dAct U silu'(G),  dU = dAct silu(G),  silu'(x) = s(x) (1 + x (1 - s(x)))
 * GU [M, 2I]: the forward's pre-activations G || U (saved by
 * coda_gemm_swiglu_save); dGU [M, 2I] receives dG || dU.  dAct itself never
 * reaches memory.  I a multiple of 64. */
CODA_API coda_status coda_gemm_swiglu_backward(const void* dOut, const void* Wt, const void* GU, void* dGU,
                                               int64_t M, int64_t I, int64_t K, coda_dtype dtype,
                                               cudaStream_t stream);

/* Per-tensor absolute maximum: *amax = max_i |x_i| over n elements of
 * dtype CODA_F32 or CODA_BF16 (overwritten).  n may be 0 (amax = 0).
 * The FP8 operands of the block's LLaMA-8B workload use per-tensor scales. */
CODA_API coda_status coda_amax(const void* x, int64_t n, coda_dtype dtype, float* amax, cudaStream_t stream);

/* Per-tensor FP8 quantisation with the scale s = amax / 448 (s = 1 when
 * amax == 0): q_i = e4m3(x_i / s), where x_i / s is the correctly rounded fp32
 * quotient, then rounded to nearest-even and saturated to +-448 (OCP e4m3, no
 * infinities).  x [n] CODA_F32 or CODA_BF16; amax: device fp32 scalar from
 * coda_amax or from a GEMM's amax output; q [n] bytes; x and q 16-byte
 * aligned, any n >= 0 (a tail of n mod 16 elements takes a scalar path);
 * scale: device fp32 scalar receiving s, the dequantisation scale to pass to
 * the GEMMs.  q and scale may not overlap x or amax. */
CODA_API coda_status coda_quantize_e4m3(const void* x, int64_t n, coda_dtype dtype, const float* amax, uint8_t* q,
                               float* scale, cudaStream_t stream);

/* Self-test of the failure path, with no GPU fault: enqueues one block whose
 * thread waits on a shared-memory mbarrier that nothing signals.  The wait is
 * bounded by timeout_ns of the GPU's global timer, like every wait inside the
 * GEMM kernels (which use 2 s).  When the limit runs out the thread raises
 * the timeout bit of the device status word and the kernel returns, so the
 * next coda_get_device_status() reports CODA_ERR_TIMEOUT and the context
 * stays usable.  Not on the pages: a diagnostic of this library.
 *   timeout_ns in [1e3, 1e10] (else CODA_ERR_INVALID_ARG, nothing enqueued). */
CODA_API coda_status coda_selftest_wait_timeout(int64_t timeout_ns, cudaStream_t stream);

/* Synchronises the current device, then reads and clears the device status
 * word: CODA_ERR_TIMEOUT if any kernel since the last call gave up on a
 * bounded wait, CODA_ERR_CUDA if the device reports an error, else CODA_OK. */
CODA_API coda_status coda_get_device_status(void);

#ifdef __cplusplus
}
#endif
#endif /* CODA_H_ */
