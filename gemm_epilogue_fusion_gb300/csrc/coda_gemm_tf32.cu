// Instantiations of the fused GEMM-epilogue kernels for tf32 operands
// (residual + partial RMS, row scale, SwiGLU programs).
#include "gemm_epilogue.cuh"

namespace coda {

cudaError_t launch_gemm_tf32(const GemmProblem& p, const char** msg) { return launch_gemm<kKindTF32>(p, msg); }

unsigned read_clear_status_tf32() { return read_clear_status_impl(); }

}  // namespace coda
