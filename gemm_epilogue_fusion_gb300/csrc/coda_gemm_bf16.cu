// Instantiations of the fused GEMM-epilogue kernels for bf16 operands
// (residual + partial RMS, row scale, SwiGLU programs).
#include "gemm_epilogue.cuh"

namespace coda {

cudaError_t launch_gemm_bf16(const GemmProblem& p, const char** msg) { return launch_gemm<kKindBF16>(p, msg); }

unsigned read_clear_status_bf16() { return read_clear_status_impl(); }

}  // namespace coda
