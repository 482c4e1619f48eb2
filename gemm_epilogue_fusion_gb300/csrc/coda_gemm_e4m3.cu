// Instantiations of the fused GEMM-epilogue kernels for e4m3 operands
// (residual + partial RMS, row scale, SwiGLU programs).
#include "gemm_epilogue.cuh"

namespace coda {

cudaError_t launch_gemm_e4m3(const GemmProblem& p, const char** msg) { return launch_gemm<kKindE4M3>(p, msg); }

unsigned read_clear_status_e4m3() { return read_clear_status_impl(); }

}  // namespace coda
