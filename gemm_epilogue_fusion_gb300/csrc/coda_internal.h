// Internal interface between the C ABI (coda_abi.cu) and the kernel
// translation units.  Host and device code both see these definitions.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace coda {

// r = 1 / sqrt(sum_t p[t] / n + eps) for one row's T partial sums of squares,
// summed in one fixed order (16-byte groups when T % 4 == 0) so that the
// reduction kernel and the fused epilogue give identical bits.
__device__ __forceinline__ float row_rstd(const float* __restrict__ p, int T, float n, float eps) {
  float s = 0.0f;
  if ((T & 3) == 0) {
    const float4* p4 = reinterpret_cast<const float4*>(p);
    for (int t = 0; t < T / 4; ++t) {
      const float4 v = __ldg(p4 + t);
      s += (v.x + v.y) + (v.z + v.w);
    }
  } else {
    for (int t = 0; t < T; ++t) s += __ldg(p + t);
  }
  return 1.0f / sqrtf(s / n + eps);
}

// Epilogue programs of the persistent GEMM (see gemm_epilogue.cuh).
// Backward programs:
//   kEpiGradNorm   dY = acc stored; P[row, g] = sum over the 128-column group g of
//                  col_scale_j * dY_j * H_j, with H TMA-loaded (RMSNorm backward's
//                  row reduction, on the stored dY)
//   kEpiSwiGLUBwd  acc = dAct; with the saved pre-activations G, U loaded:
//                  dG = dAct U silu'(G), dU = dAct silu(G), stored side by side
//   kEpiSwiGLUSave SwiGLU that also stores the pre-activations G = r g and
//                  U = r u (bf16) side by side, for the backward
enum Epilogue {
  kEpiResidualPartialRms = 0,
  kEpiRowScale = 1,
  kEpiSwiGLU = 2,
  kEpiGradNorm = 3,
  kEpiSwiGLUBwd = 4,
  kEpiSwiGLUSave = 5
};

// Width, in output columns, of one partial sum-of-squares group written by the
// residual epilogue: P has ceil(N / kPartialCols) columns.
constexpr int kPartialCols = 128;

// Arguments of the fused epilogue programs (all device pointers).
struct EpiParams {
  const float* r;         // row scale [M]: used by the row-scale and SwiGLU programs when P_in is null
                          // (nullable for SwiGLU: 1)
  const float* P_in;      // row-scale / SwiGLU: partial sums of squares [M, T_in] of the previous
                          // residual GEMM; when set, the epilogue reduces them to r itself
  int T_in;               // columns of P_in
  float n_norm;           // RMSNorm width N the partials cover (the GEMM's K)
  float eps;
  float* r_out;           // nullable: with P_in, the tiles of the first column band store r [M]
  float* P;               // residual program: partial sums of squares [M, T]
  int T;                  // columns of P
  const float* scale_a;   // E4M3 operands: dequantisation scale of A, else null
  const float* scale_b;   // ... of B (SwiGLU: of the gate weight)
  const float* scale_b2;  // SwiGLU: of the up weight
  float* amax_out;        // nullable: max |stored output|, combined with atomicMax (caller zeroes it)
  // row-scale program only: RoPE on the first rope_cols output columns (0 = none)
  const int* rope_pos;    // [M] positions; null = row % rope_seq
  int rope_seq, rope_half, rope_cols;
  float rope_log2b;       // log2(base) / rope_half
  const float* col_scale; // row-scale program: nullable [N_out], multiplies output column n;
                          // grad-norm program: gamma [N_out]
  int gu_off;             // SwiGLU backward: column offset of U (and dU) in the [M, 2 I] tensors
};

// Second phase of a two-phase launch (the consuming GEMM of the block).
struct PhaseB {
  int epi = -1;            // kEpiRowScale or kEpiSwiGLU; -1 = one-phase launch
  const void* A = nullptr;  // h [M, K] (phase A's output)
  const void* B = nullptr;  // weight [N_out, K]; SwiGLU: gate weight
  const void* B2 = nullptr; // SwiGLU: up weight
  void* D = nullptr;        // output [M, N_out]
  int N_out = 0, K = 0;
  EpiParams ep = {};
};

// FP8 one-launch block: the e4m3 copies that the launch itself makes.  h
// (phase A's bf16 output) is quantised once every phase-A tile has stored it
// and folded its |h| into amax_h; with `a` set, phase A's A operand is
// quantised from its bf16 source first (amax_a final before the launch).
// Both run in the quantiser warps, band by band, so the consuming GEMM
// starts on a band as soon as its e4m3 copy is complete.
struct QuantArgs {
  const void* h = nullptr;        // h [M, N] bf16: phase A's output
  uint8_t* hq = nullptr;          // its e4m3 copy: phase B's A operand
  float* amax_h = nullptr;        // max |h| (zeroed before the launch)
  float* scale_h = nullptr;       // written: amax_h / 448 (1 if zero)
  const void* a = nullptr;        // nullable: bf16 source of phase A's A operand [M, K]
  uint8_t* aq = nullptr;          // its e4m3 copy: phase A's A operand
  const float* amax_a = nullptr;  // max |a|
  float* scale_a = nullptr;       // written: amax_a / 448
};

// Counters of a two-phase launch's workspace, in units of unsigned, for m
// row bands: [0, m) band ready (h and P stored), [m] CTAs done (the last one
// resets every counter); FP8 blocks add [m + 1] CTAs past phase A, [m + 2,
// 2m + 2) bands of h quantised, [2m + 2, 3m + 2) bands of A quantised.
__host__ __device__ constexpr int64_t block_counters(int64_t m_bands, bool fp8) {
  return fp8 ? 3 * m_bands + 2 : m_bands + 1;
}

struct GemmProblem {
  int epi;                 // Epilogue
  const void* A;           // [M, K] K-major activations
  const void* B;           // [N_out, K] K-major weight (W^T); SwiGLU: gate weight [I, K]
  const void* B2;          // SwiGLU: up weight [I, K]; else null
  const void* R;           // residual program: [M, N_out] residual; else null
  void* D;                 // [M, N_out] output
  int M, N_out, K;
  EpiParams ep;
  cudaStream_t stream;
  bool pdl;                // launch with programmatic stream serialisation
  void* GU = nullptr;      // kEpiSwiGLUSave: G || U output [M, 2 N_out]
  bool a_mn = false;       // A stored [K, M] (MN-major) instead of [M, K]
  bool b_mn = false;       // B stored [K, N_out] instead of [N_out, K]
  PhaseB b;                // consuming GEMM of a two-phase launch
  unsigned* band_ready;    // two-phase: block_counters(ceil(M / tile rows), fp8) zeroed counters
  bool fp8_block = false;  // two-phase e4m3: h quantised in the launch (QuantArgs)
  QuantArgs q;
};

// One launcher per operand kind; each lives in its own translation unit so
// the three compile in parallel.  They return cudaSuccess or the CUDA error
// of the tensor-map encode / launch, with a message in *msg.
cudaError_t launch_gemm_bf16(const GemmProblem& p, const char** msg);
cudaError_t launch_gemm_tf32(const GemmProblem& p, const char** msg);
cudaError_t launch_gemm_e4m3(const GemmProblem& p, const char** msg);
unsigned read_clear_status_bf16();
unsigned read_clear_status_tf32();
unsigned read_clear_status_e4m3();

// Element-wise and reduction kernels (coda_aux.cu).
cudaError_t launch_rms_reduce(const float* P, int64_t M, int T, int64_t N, float eps, float* r,
                              cudaStream_t s, bool pdl);
cudaError_t launch_fold_gamma(const void* Wt, const float* gamma, void* Wt_out, int64_t N_out, int64_t K,
                              bool f32, cudaStream_t s);
int64_t rmsnorm_bwd_chunks(int64_t M);
cudaError_t launch_rmsnorm_backward(const void* dY, const void* H, const float* r, const float* gamma,
                                    const float* S, int T, const void* dH_in, void* dH, void* Yt, float* dgamma,
                                    float* part, int64_t M, int64_t N, cudaStream_t s);
cudaError_t launch_amax(const void* x, int64_t n, bool f32, float* amax, cudaStream_t s);
cudaError_t launch_quantize_e4m3(const void* x, int64_t n, bool f32, const float* amax, uint8_t* q,
                                 float* scale, cudaStream_t s);
unsigned read_clear_status_aux();

// Host helpers (coda_abi.cu).
int device_sm_count();
// 2-D row-major tensor map with 128-byte swizzle: `inner` contiguous
// elements per row, `outer` rows, rows `row_bytes` apart; box of
// box_inner x box_outer elements.
CUresult encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// Launch `kernel` with the given shape, optionally with programmatic stream
// serialisation (PDL), so its prologue overlaps the previous kernel's tail,
// in clusters of `cluster` CTAs along x, and as a cooperative launch (every
// CTA of the grid resident at once, or the launch fails).
cudaError_t launch_ex(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      void** args, int cluster = 1, bool cooperative = false);

// A two-phase launch (band waits between CTAs) first asks for a cooperative
// launch, which makes the co-residency of its grid a guarantee.  What to do
// with that attempt's result:
//   kCoopDone      launched
//   kCoopFallback  the runtime or device does not take a cooperative launch
//                  of this form (with clusters): launch it plainly, on a
//                  grid no larger than the co-resident CTAs of an idle GPU
//   kCoopError     any other error, cudaErrorCooperativeLaunchTooLarge
//                  included: report it, never launch a grid that might not
//                  fit
enum CoopAction { kCoopDone = 0, kCoopFallback = 1, kCoopError = 2 };
inline CoopAction cooperative_action(cudaError_t e) {
  if (e == cudaSuccess) return kCoopDone;
  if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue || e == cudaErrorInvalidConfiguration)
    return kCoopFallback;
  return kCoopError;
}

// One launch of a grid whose CTAs wait on each other: `launch(cooperative)`
// issues one attempt.  With try_coop, the cooperative form goes first and
// the plain form follows only on kCoopFallback (*refused is then set, so the
// caller can skip the attempt on that device from then on).
template <class F>
cudaError_t launch_coresident(F&& launch, bool try_coop, bool* refused) {
  *refused = false;
  if (try_coop) {
    const cudaError_t e = launch(true);
    if (cooperative_action(e) != kCoopFallback) return e;
    (void)cudaGetLastError();  // a refused launch configuration is not sticky: clear it
    *refused = true;
  }
  return launch(false);
}

}  // namespace coda
