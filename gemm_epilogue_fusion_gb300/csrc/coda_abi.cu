// C ABI of the fused GEMM-epilogue library: argument validation, dispatch to
// the kernel translation units, error reporting.  Nothing here allocates or
// synchronises (except coda_get_device_status, which says so).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cinttypes>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <utility>

#include "coda.h"
#include "coda_internal.h"

namespace coda {
// The failure-path self-test kernel's launcher (coda_aux.cu).
cudaError_t launch_wait_probe(int64_t timeout_ns, cudaStream_t s);
}  // namespace coda

namespace {

thread_local char g_msg[512] = "";
// Largest M that coda_block_swiglu_noalloc accepts (its counters are built in).
constexpr int kNoAllocMaxRows = 131072;

coda_status fail(coda_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
coda_status fail(coda_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

coda_status cuda_fail(cudaError_t e, const char* what) {
  return fail(CODA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int elem_bytes(coda_dtype d) { return d == CODA_F32 ? 4 : d == CODA_BF16 ? 2 : 1; }
// residual / output element size for GEMMs with this operand type
int out_bytes(coda_dtype d) { return d == CODA_F32 ? 4 : 2; }
bool valid_dtype(int d) { return d == CODA_F32 || d == CODA_BF16 || d == CODA_E4M3; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  const char* name;
  uintptr_t lo, hi;  // [lo, hi)
};
Range rng(const char* name, const void* p, int64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {name, a, a + static_cast<uintptr_t>(bytes)};
}
bool overlap(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// Every output range against every input range and every other output.
coda_status check_overlaps(const Range* outs, int n_out, const Range* ins, int n_in) {
  for (int i = 0; i < n_out; ++i) {
    for (int j = 0; j < n_in; ++j)
      if (overlap(outs[i], ins[j]))
        return fail(CODA_ERR_INVALID_ARG, "output %s overlaps input %s", outs[i].name, ins[j].name);
    for (int j = i + 1; j < n_out; ++j)
      if (overlap(outs[i], outs[j]))
        return fail(CODA_ERR_INVALID_ARG, "outputs %s and %s overlap", outs[i].name, outs[j].name);
  }
  return CODA_OK;
}

#define REQUIRE(cond, ...)                                 \
  do {                                                     \
    if (!(cond)) return fail(CODA_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

coda_status check_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(CODA_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(CODA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return CODA_OK;
}

coda_status check_scalar_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(CODA_ERR_INVALID_ARG, "%s is NULL", name);
  if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0) return fail(CODA_ERR_INVALID_ARG, "%s is not 4-byte aligned", name);
  return CODA_OK;
}

#define TRY(expr)                        \
  do {                                   \
    coda_status s_ = (expr);             \
    if (s_ != CODA_OK) return s_;        \
  } while (0)

// Byte extents of every operand of an M x N x K product must fit int64, and
// the kernels' tile indices are 32-bit: bound both at the smallest tile,
// 128 x 128 outputs.  M, N, K are already within [0, 2^31).
coda_status check_extents(int64_t M, int64_t N, int64_t K, const char* nname) {
  REQUIRE(M * N < (int64_t(1) << 60) && M * K < (int64_t(1) << 60) && N * K < (int64_t(1) << 60),
          "M = %" PRId64 ", %s = %" PRId64 ", K = %" PRId64 ": a matrix of 2^60 elements or more", M, nname, N, K);
  REQUIRE(((M + 127) / 128) * ((N + 127) / 128) < INT32_MAX / 2,
          "M = %" PRId64 ", %s = %" PRId64 ": too many output tiles for the kernels' 32-bit tile indices", M, nname, N);
  return CODA_OK;
}

// Shape rules common to the GEMM calls.
coda_status check_gemm_dims(int64_t M, int64_t N, int64_t K, coda_dtype dt, const char* nname) {
  REQUIRE(valid_dtype(dt), "unknown dtype %d", static_cast<int>(dt));
  REQUIRE(M >= 0 && M < INT32_MAX, "M = %" PRId64 " out of range [0, 2^31)", M);
  REQUIRE(N > 0 && N < INT32_MAX, "%s = %" PRId64 " out of range [1, 2^31)", nname, N);
  REQUIRE(K > 0 && K < INT32_MAX, "K = %" PRId64 " out of range [1, 2^31)", K);
  REQUIRE((K * elem_bytes(dt)) % 16 == 0, "K = %" PRId64 " must be a multiple of %d for this dtype (16-byte rows)", K,
          16 / elem_bytes(dt));
  REQUIRE((N * out_bytes(dt)) % 16 == 0, "%s = %" PRId64 " must be a multiple of %d for this dtype (16-byte rows)",
          nname, N, 16 / out_bytes(dt));
  return check_extents(M, N, K, nname);
}

coda_status check_scales(coda_dtype dt, const float* a, const char* an, const float* b, const char* bn,
                         const float* c = nullptr, const char* cn = nullptr) {
  if (dt == CODA_E4M3) {
    TRY(check_scalar_ptr(a, an));
    TRY(check_scalar_ptr(b, bn));
    if (cn) TRY(check_scalar_ptr(c, cn));
  } else {
    REQUIRE(a == nullptr && b == nullptr && c == nullptr, "FP8 scales must be NULL unless dtype is CODA_E4M3");
  }
  return CODA_OK;
}

coda_status run_gemm(coda_dtype dt, const coda::GemmProblem& p) {
  const char* msg = "";
  cudaError_t e;
  switch (dt) {
    case CODA_BF16: e = coda::launch_gemm_bf16(p, &msg); break;
    case CODA_F32: e = coda::launch_gemm_tf32(p, &msg); break;
    default: e = coda::launch_gemm_e4m3(p, &msg); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, msg);
  return CODA_OK;
}

// Programmatic dependent launch (kernel prologues overlap the previous
// kernel's tail) is on unless CODA_NO_PDL is set in the environment.
bool use_pdl() {
  static const bool on = getenv("CODA_NO_PDL") == nullptr;
  return on;
}

coda_status zero_scalar(float* p, cudaStream_t s) {
  if (p == nullptr) return CODA_OK;
  cudaError_t e = cudaMemsetAsync(p, 0, sizeof(float), s);
  return e == cudaSuccess ? CODA_OK : cuda_fail(e, "cudaMemsetAsync(amax)");
}

}  // namespace

// ------------------------------------------------------------ host helpers ----
namespace coda {

int device_sm_count() {
  // host threads may ask at once: each slot is written with the same value
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

CUresult encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

cudaError_t launch_ex(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      void** args, int cluster, bool cooperative) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  int n = 0;
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelExC(&cfg, kernel, args);
}

}  // namespace coda

// ------------------------------------------------------------------- ABI ----
extern "C" {

int coda_version(void) { return 100; }

const char* coda_status_string(coda_status s) {
  switch (s) {
    case CODA_OK: return "CODA_OK";
    case CODA_ERR_INVALID_ARG: return "CODA_ERR_INVALID_ARG";
    case CODA_ERR_UNSUPPORTED: return "CODA_ERR_UNSUPPORTED";
    case CODA_ERR_CUDA: return "CODA_ERR_CUDA";
    case CODA_ERR_TIMEOUT: return "CODA_ERR_TIMEOUT";
  }
  return "unknown coda_status";
}

const char* coda_last_error(void) { return g_msg; }

int64_t coda_partial_cols(int64_t N) {
  if (N <= 0) return -1;
  return (N + coda::kPartialCols - 1) / coda::kPartialCols;
}

coda_status coda_fold_gamma(const void* Wt, const float* gamma, void* Wt_out, int64_t N_out, int64_t K,
                            coda_dtype dtype, cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(dtype == CODA_F32 || dtype == CODA_BF16, "coda_fold_gamma: dtype must be CODA_F32 or CODA_BF16");
  REQUIRE(N_out >= 0 && K > 0 && N_out < INT32_MAX && K < INT32_MAX && N_out * K < (int64_t(1) << 60),
          "coda_fold_gamma: bad shape");
  REQUIRE((K * elem_bytes(dtype)) % 16 == 0, "coda_fold_gamma: K must give 16-byte rows");
  if (N_out == 0) return CODA_OK;
  TRY(check_ptr(Wt, "Wt"));
  TRY(check_ptr(gamma, "gamma"));
  TRY(check_ptr(Wt_out, "Wt_out"));
  const int64_t wb = N_out * K * elem_bytes(dtype);
  const Range outs[] = {rng("Wt_out", Wt_out, wb)};
  const Range ins[] = {rng("Wt", Wt, wb), rng("gamma", gamma, K * 4)};
  TRY(check_overlaps(outs, 1, ins, 2));
  cudaError_t e = coda::launch_fold_gamma(Wt, gamma, Wt_out, N_out, K, dtype == CODA_F32, stream);
  return e == cudaSuccess ? CODA_OK : cuda_fail(e, "coda_fold_gamma launch");
}

coda_status coda_gemm_residual_partial_rms(const void* X, const void* W1t, const void* R, void* H, float* P,
                                           int64_t M, int64_t N, int64_t K, coda_dtype dtype,
                                           const float* scale_x, const float* scale_w, float* amax_h,
                                           cudaStream_t stream) {
  g_msg[0] = 0;
  TRY(check_gemm_dims(M, N, K, dtype, "N"));
  TRY(check_scales(dtype, scale_x, "scale_x", scale_w, "scale_w"));
  if (amax_h) TRY(check_scalar_ptr(amax_h, "amax_h"));
  if (M == 0) return zero_scalar(amax_h, stream);
  TRY(check_ptr(X, "X"));
  TRY(check_ptr(W1t, "W1t"));
  TRY(check_ptr(R, "R"));
  TRY(check_ptr(H, "H"));
  TRY(check_ptr(P, "P"));
  const int64_t T = coda_partial_cols(N);
  const int ob = out_bytes(dtype), ib = elem_bytes(dtype);
  const Range outs[] = {rng("H", H, M * N * ob), rng("P", P, M * T * 4), rng("amax_h", amax_h, amax_h ? 4 : 0)};
  const Range ins[] = {rng("X", X, M * K * ib), rng("W1t", W1t, N * K * ib), rng("R", R, M * N * ob),
                       rng("scale_x", scale_x, scale_x ? 4 : 0), rng("scale_w", scale_w, scale_w ? 4 : 0)};
  TRY(check_overlaps(outs, 3, ins, 5));
  TRY(zero_scalar(amax_h, stream));
  coda::GemmProblem p = {};
  p.epi = coda::kEpiResidualPartialRms;
  p.A = X;
  p.B = W1t;
  p.R = R;
  p.D = H;
  p.M = static_cast<int>(M);
  p.N_out = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.ep.P = P;
  p.ep.T = static_cast<int>(T);
  p.ep.scale_a = scale_x;
  p.ep.scale_b = scale_w;
  p.ep.amax_out = amax_h;
  p.stream = stream;
  p.pdl = use_pdl();
  return run_gemm(dtype, p);
}

coda_status coda_rms_reduce(const float* P, int64_t M, int64_t N, float eps, float* r, cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(M >= 0 && M < INT32_MAX, "coda_rms_reduce: M out of range");
  REQUIRE(N > 0 && N < INT32_MAX, "coda_rms_reduce: N out of range");
  REQUIRE(std::isfinite(eps) && eps >= 0.0f, "coda_rms_reduce: eps must be finite and >= 0");
  if (M == 0) return CODA_OK;
  TRY(check_ptr(P, "P"));
  TRY(check_ptr(r, "r"));
  const int64_t T = coda_partial_cols(N);
  const Range outs[] = {rng("r", r, M * 4)};
  const Range ins[] = {rng("P", P, M * T * 4)};
  TRY(check_overlaps(outs, 1, ins, 1));
  cudaError_t e = coda::launch_rms_reduce(P, M, static_cast<int>(T), N, eps, r, stream, use_pdl());
  return e == cudaSuccess ? CODA_OK : cuda_fail(e, "coda_rms_reduce launch");
}

}  // extern "C"

namespace {

// RoPE arguments of the row-scale program.
struct RopeArgs {
  int64_t head_dim, rope_cols;
  double base;
  int64_t seq_len;
  const int32_t* positions;
};

// Checks of the RoPE arguments of a row-scale program with N2 output columns.
coda_status check_rope(const RopeArgs* rope, int64_t M, int64_t N2, coda_dtype dtype) {
  const int64_t chunk = 16 / out_bytes(dtype);  // columns per 16-byte store chunk
  REQUIRE(rope->head_dim > 0 && rope->head_dim % chunk == 0,
          "head_dim must be a positive multiple of %" PRId64 " for this dtype", chunk);
  REQUIRE(rope->rope_cols >= 0 && rope->rope_cols <= N2 && rope->rope_cols % rope->head_dim == 0,
          "rope_cols must be a multiple of head_dim within [0, N2]");
  REQUIRE(std::isfinite(rope->base) && rope->base > 1.0, "base must be finite and > 1");
  REQUIRE(rope->positions != nullptr || (rope->seq_len > 0 && rope->seq_len < INT32_MAX),
          "seq_len must be in [1, 2^31) when positions is NULL");
  if (M > 0 && rope->positions) TRY(check_scalar_ptr(rope->positions, "positions"));
  return CODA_OK;
}

// The RoPE fields of a row-scale program's epilogue.
void set_rope(coda::EpiParams& ep, const RopeArgs* rope) {
  if (rope == nullptr || rope->rope_cols <= 0) return;
  ep.rope_pos = rope->positions;
  ep.rope_seq = static_cast<int>(rope->positions ? 1 : rope->seq_len);
  ep.rope_half = static_cast<int>(rope->head_dim / 2);
  ep.rope_cols = static_cast<int>(rope->rope_cols);
  ep.rope_log2b = static_cast<float>(std::log2(rope->base) / static_cast<double>(rope->head_dim / 2));
}

// Shared by the row-scale calls: r given, or reduced in the epilogue from P;
// optionally RoPE on the leading columns.
coda_status gemm_rowscale_impl(const void* H, const void* W2t, const float* r, const float* P, float eps,
                               float* r_out, void* Z, int64_t M, int64_t N2, int64_t K, coda_dtype dtype,
                               const float* scale_h, const float* scale_w, cudaStream_t stream,
                               const RopeArgs* rope = nullptr) {
  g_msg[0] = 0;
  if (rope) TRY(check_rope(rope, M, N2, dtype));
  TRY(check_gemm_dims(M, N2, K, dtype, "N2"));
  TRY(check_scales(dtype, scale_h, "scale_h", scale_w, "scale_w"));
  if (P) REQUIRE(std::isfinite(eps) && eps >= 0.0f, "eps must be finite and >= 0");
  if (M == 0) return CODA_OK;
  TRY(check_ptr(H, "H"));
  TRY(check_ptr(W2t, "W2t"));
  TRY(check_ptr(Z, "Z"));
  if (P) {
    TRY(check_ptr(P, "P"));
    if (r_out) TRY(check_scalar_ptr(r_out, "r_out"));
  } else {
    TRY(check_ptr(r, "r"));
  }
  const int ob = out_bytes(dtype), ib = elem_bytes(dtype);
  const int64_t T = coda_partial_cols(K);
  const Range outs[] = {rng("Z", Z, M * N2 * ob), rng("r_out", r_out, r_out ? M * 4 : 0)};
  const Range ins[] = {rng("H", H, M * K * ib), rng("W2t", W2t, N2 * K * ib), rng("r", r, r ? M * 4 : 0),
                       rng("P", P, P ? M * T * 4 : 0), rng("scale_h", scale_h, scale_h ? 4 : 0),
                       rng("scale_w", scale_w, scale_w ? 4 : 0),
                       rng("positions", rope ? rope->positions : nullptr, rope && rope->positions ? M * 4 : 0)};
  TRY(check_overlaps(outs, 2, ins, 7));
  coda::GemmProblem p = {};
  p.epi = coda::kEpiRowScale;
  p.A = H;
  p.B = W2t;
  p.D = Z;
  p.M = static_cast<int>(M);
  p.N_out = static_cast<int>(N2);
  p.K = static_cast<int>(K);
  p.ep.r = P ? nullptr : r;
  p.ep.P_in = P;
  p.ep.T_in = static_cast<int>(T);
  p.ep.n_norm = static_cast<float>(K);
  p.ep.eps = eps;
  p.ep.r_out = P ? r_out : nullptr;
  p.ep.scale_a = scale_h;
  p.ep.scale_b = scale_w;
  set_rope(p.ep, rope);
  p.stream = stream;
  p.pdl = use_pdl();
  return run_gemm(dtype, p);
}

// Shared by the SwiGLU calls.
coda_status gemm_swiglu_impl(const void* H, const void* Wgt, const void* Wut, const float* r, const float* P,
                             float eps, float* r_out, void* Act, int64_t M, int64_t I, int64_t K, coda_dtype dtype,
                             const float* scale_h, const float* scale_wg, const float* scale_wu, float* amax_act,
                             cudaStream_t stream) {
  g_msg[0] = 0;
  TRY(check_gemm_dims(M, I, K, dtype, "I"));
  TRY(check_scales(dtype, scale_h, "scale_h", scale_wg, "scale_wg", scale_wu, "scale_wu"));
  if (P) REQUIRE(std::isfinite(eps) && eps >= 0.0f, "eps must be finite and >= 0");
  if (amax_act) TRY(check_scalar_ptr(amax_act, "amax_act"));
  if (M == 0) return zero_scalar(amax_act, stream);
  TRY(check_ptr(H, "H"));
  TRY(check_ptr(Wgt, "Wgt"));
  TRY(check_ptr(Wut, "Wut"));
  if (P) {
    TRY(check_ptr(P, "P"));
    if (r_out) TRY(check_scalar_ptr(r_out, "r_out"));
  } else if (r) {
    TRY(check_scalar_ptr(r, "r"));
  }
  TRY(check_ptr(Act, "Act"));
  const int ob = out_bytes(dtype), ib = elem_bytes(dtype);
  const int64_t T = coda_partial_cols(K);
  const Range outs[] = {rng("Act", Act, M * I * ob), rng("amax_act", amax_act, amax_act ? 4 : 0),
                        rng("r_out", r_out, r_out ? M * 4 : 0)};
  const Range ins[] = {rng("H", H, M * K * ib),
                       rng("Wgt", Wgt, I * K * ib),
                       rng("Wut", Wut, I * K * ib),
                       rng("r", r, r ? M * 4 : 0),
                       rng("P", P, P ? M * T * 4 : 0),
                       rng("scale_h", scale_h, scale_h ? 4 : 0),
                       rng("scale_wg", scale_wg, scale_wg ? 4 : 0),
                       rng("scale_wu", scale_wu, scale_wu ? 4 : 0)};
  TRY(check_overlaps(outs, 3, ins, 8));
  TRY(zero_scalar(amax_act, stream));
  coda::GemmProblem p = {};
  p.epi = coda::kEpiSwiGLU;
  p.A = H;
  p.B = Wgt;
  p.B2 = Wut;
  p.D = Act;
  p.M = static_cast<int>(M);
  p.N_out = static_cast<int>(I);
  p.K = static_cast<int>(K);
  p.ep.r = P ? nullptr : r;
  p.ep.P_in = P;
  p.ep.T_in = static_cast<int>(T);
  p.ep.n_norm = static_cast<float>(K);
  p.ep.eps = eps;
  p.ep.r_out = P ? r_out : nullptr;
  p.ep.scale_a = scale_h;
  p.ep.scale_b = scale_wg;
  p.ep.scale_b2 = scale_wu;
  p.ep.amax_out = amax_act;
  p.stream = stream;
  p.pdl = use_pdl();
  return run_gemm(dtype, p);
}

}  // namespace

extern "C" {

coda_status coda_gemm_rowscale(const void* H, const void* W2t, const float* r, void* Z, int64_t M, int64_t N2,
                               int64_t K, coda_dtype dtype, const float* scale_h, const float* scale_w,
                               cudaStream_t stream) {
  if (r == nullptr && M > 0) {
    g_msg[0] = 0;
    return fail(CODA_ERR_INVALID_ARG, "r is NULL");
  }
  return gemm_rowscale_impl(H, W2t, r, nullptr, 0.0f, nullptr, Z, M, N2, K, dtype, scale_h, scale_w, stream);
}

coda_status coda_gemm_rowscale_fused_rms(const void* H, const void* W2t, const float* P, float eps, float* r_out,
                                         void* Z, int64_t M, int64_t N2, int64_t K, coda_dtype dtype,
                                         const float* scale_h, const float* scale_w, cudaStream_t stream) {
  if (P == nullptr && M > 0) {
    g_msg[0] = 0;
    return fail(CODA_ERR_INVALID_ARG, "P is NULL");
  }
  return gemm_rowscale_impl(H, W2t, nullptr, P, eps, r_out, Z, M, N2, K, dtype, scale_h, scale_w, stream);
}

coda_status coda_gemm_rowscale_rope(const void* H, const void* W2t, const float* r, const float* P, float eps,
                                    float* r_out, void* Z, int64_t M, int64_t N2, int64_t K, coda_dtype dtype,
                                    const float* scale_h, const float* scale_w, int64_t head_dim, int64_t rope_cols,
                                    double base, int64_t seq_len, const int32_t* positions, cudaStream_t stream) {
  if (M > 0 && (r == nullptr) == (P == nullptr)) {
    g_msg[0] = 0;
    return fail(CODA_ERR_INVALID_ARG, "exactly one of r and P must be given");
  }
  const RopeArgs rope = {head_dim, rope_cols, base, seq_len, positions};
  return gemm_rowscale_impl(H, W2t, P ? nullptr : r, P, eps, P ? r_out : nullptr, Z, M, N2, K, dtype, scale_h,
                            scale_w, stream, &rope);
}

coda_status coda_gemm_swiglu(const void* H, const void* Wgt, const void* Wut, const float* r, void* Act, int64_t M,
                             int64_t I, int64_t K, coda_dtype dtype, const float* scale_h, const float* scale_wg,
                             const float* scale_wu, float* amax_act, cudaStream_t stream) {
  return gemm_swiglu_impl(H, Wgt, Wut, r, nullptr, 0.0f, nullptr, Act, M, I, K, dtype, scale_h, scale_wg, scale_wu,
                          amax_act, stream);
}

coda_status coda_gemm_swiglu_fused_rms(const void* H, const void* Wgt, const void* Wut, const float* P, float eps,
                                       float* r_out, void* Act, int64_t M, int64_t I, int64_t K, coda_dtype dtype,
                                       const float* scale_h, const float* scale_wg, const float* scale_wu,
                                       float* amax_act, cudaStream_t stream) {
  if (P == nullptr && M > 0) {
    g_msg[0] = 0;
    return fail(CODA_ERR_INVALID_ARG, "P is NULL");
  }
  return gemm_swiglu_impl(H, Wgt, Wut, nullptr, P, eps, r_out, Act, M, I, K, dtype, scale_h, scale_wg, scale_wu,
                          amax_act, stream);
}

coda_status coda_gemm(const void* A, coda_layout a_layout, const void* B, coda_layout b_layout, void* D, int64_t M,
                      int64_t N, int64_t K, coda_dtype dtype, const float* row_scale, const float* col_scale,
                      cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(dtype == CODA_F32 || dtype == CODA_BF16, "coda_gemm: dtype must be CODA_F32 or CODA_BF16");
  REQUIRE((a_layout == CODA_K_MAJOR || a_layout == CODA_MN_MAJOR) && (b_layout == CODA_K_MAJOR || b_layout == CODA_MN_MAJOR),
          "unknown layout");
  const bool a_mn = a_layout == CODA_MN_MAJOR, b_mn = b_layout == CODA_MN_MAJOR;
  REQUIRE(!(a_mn || b_mn) || dtype == CODA_BF16, "MN-major operands are bf16 only");
  REQUIRE(!(a_mn && !b_mn), "an MN-major A needs an MN-major B");
  REQUIRE(M >= 0 && M < INT32_MAX && N > 0 && N < INT32_MAX && K > 0 && K < INT32_MAX, "bad shape");
  TRY(check_extents(M, N, K, "N"));
  const int eb = elem_bytes(dtype), ob = out_bytes(dtype);
  REQUIRE(((a_mn ? M : K) * eb) % 16 == 0, "A's rows must be a multiple of 16 bytes");
  REQUIRE(((b_mn ? N : K) * eb) % 16 == 0, "B's rows must be a multiple of 16 bytes");
  REQUIRE((N * ob) % 16 == 0, "D's rows must be a multiple of 16 bytes");
  if (M == 0) return CODA_OK;
  TRY(check_ptr(A, "A"));
  TRY(check_ptr(B, "B"));
  TRY(check_ptr(D, "D"));
  if (row_scale) TRY(check_scalar_ptr(row_scale, "row_scale"));
  if (col_scale) TRY(check_scalar_ptr(col_scale, "col_scale"));
  const Range outs[] = {rng("D", D, M * N * ob)};
  const Range ins[] = {rng("A", A, M * K * eb), rng("B", B, N * K * eb),
                       rng("row_scale", row_scale, row_scale ? M * 4 : 0),
                       rng("col_scale", col_scale, col_scale ? N * 4 : 0)};
  TRY(check_overlaps(outs, 1, ins, 4));
  coda::GemmProblem p = {};
  p.epi = coda::kEpiRowScale;
  p.A = A;
  p.B = B;
  p.D = D;
  p.M = static_cast<int>(M);
  p.N_out = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.ep.r = row_scale;
  p.ep.col_scale = col_scale;
  p.a_mn = a_mn;
  p.b_mn = b_mn;
  p.stream = stream;
  p.pdl = use_pdl();
  return run_gemm(dtype, p);
}

coda_status coda_gemm_grad_norm(const void* dOut, const void* Wt, const void* H, const float* gamma, void* dY,
                                float* S, int64_t M, int64_t N, int64_t K, coda_dtype dtype, cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(dtype == CODA_BF16, "coda_gemm_grad_norm: dtype must be CODA_BF16");
  TRY(check_gemm_dims(M, N, K, dtype, "N"));
  if (M == 0) return CODA_OK;
  TRY(check_ptr(dOut, "dOut"));
  TRY(check_ptr(Wt, "Wt"));
  TRY(check_ptr(H, "H"));
  TRY(check_ptr(gamma, "gamma"));
  TRY(check_ptr(dY, "dY"));
  TRY(check_ptr(S, "S"));
  const int64_t T = coda_partial_cols(N);
  const Range outs[] = {rng("dY", dY, M * N * 2), rng("S", S, M * T * 4)};
  const Range ins[] = {rng("dOut", dOut, M * K * 2), rng("Wt", Wt, K * N * 2), rng("H", H, M * N * 2),
                       rng("gamma", gamma, N * 4)};
  TRY(check_overlaps(outs, 2, ins, 4));
  coda::GemmProblem p = {};
  p.epi = coda::kEpiGradNorm;
  p.A = dOut;
  p.B = Wt;
  p.R = H;
  p.D = dY;
  p.M = static_cast<int>(M);
  p.N_out = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.ep.P = S;
  p.ep.T = static_cast<int>(T);
  p.ep.col_scale = gamma;
  p.b_mn = true;
  p.stream = stream;
  p.pdl = use_pdl();
  return run_gemm(dtype, p);
}

int64_t coda_rmsnorm_backward_workspace_bytes(int64_t M, int64_t N) {
  if (M < 0 || N <= 0) return -1;
  return coda::rmsnorm_bwd_chunks(M) * N * static_cast<int64_t>(sizeof(float));
}

coda_status coda_rmsnorm_backward(const void* dY, const void* H, const float* r, const float* gamma, const float* S,
                                  const void* dH_in, void* dH, void* Yt, float* dgamma, float* workspace, int64_t M,
                                  int64_t N, cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(M >= 0 && M < INT32_MAX && N > 0 && N < INT32_MAX && N % 8 == 0 && M * N < (int64_t(1) << 60),
          "coda_rmsnorm_backward: M in [0, 2^31), N a positive multiple of 8, M N below 2^60");
  if (M == 0) {
    TRY(check_scalar_ptr(dgamma, "dgamma"));
    cudaError_t e = cudaMemsetAsync(dgamma, 0, static_cast<size_t>(N) * sizeof(float), stream);
    return e == cudaSuccess ? CODA_OK : cuda_fail(e, "cudaMemsetAsync(dgamma)");
  }
  for (const auto& pr : {std::make_pair(dY, "dY"), std::make_pair(H, "H"), std::make_pair(static_cast<const void*>(dH), "dH"),
                         std::make_pair(static_cast<const void*>(Yt), "Yt"), std::make_pair(static_cast<const void*>(gamma), "gamma"),
                         std::make_pair(static_cast<const void*>(dgamma), "dgamma"),
                         std::make_pair(static_cast<const void*>(workspace), "workspace")})
    TRY(check_ptr(pr.first, pr.second));
  TRY(check_scalar_ptr(r, "r"));
  TRY(check_scalar_ptr(S, "S"));
  if (dH_in) TRY(check_ptr(dH_in, "dH_in"));
  const int64_t T = coda_partial_cols(N);
  const int64_t mn = M * N * 2;
  const Range outs[] = {rng("dH", dH, mn), rng("Yt", Yt, mn), rng("dgamma", dgamma, N * 4),
                        rng("workspace", workspace, coda_rmsnorm_backward_workspace_bytes(M, N))};
  const Range ins[] = {rng("dY", dY, mn), rng("H", H, mn), rng("r", r, M * 4), rng("gamma", gamma, N * 4),
                       rng("S", S, M * T * 4), rng("dH_in", dH_in, dH_in ? mn : 0)};
  TRY(check_overlaps(outs, 4, ins, 6));
  cudaError_t e = coda::launch_rmsnorm_backward(dY, H, r, gamma, S, static_cast<int>(T), dH_in, dH, Yt, dgamma,
                                                workspace, M, N, stream);
  return e == cudaSuccess ? CODA_OK : cuda_fail(e, "coda_rmsnorm_backward launch");
}

coda_status coda_gemm_swiglu_save(const void* H, const void* Wgt, const void* Wut, const float* r, const float* P,
                                  float eps, float* r_out, void* Act, void* GU, int64_t M, int64_t I, int64_t K,
                                  coda_dtype dtype, cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(dtype == CODA_BF16, "coda_gemm_swiglu_save: dtype must be CODA_BF16");
  // a 64-column box of the G half must not reach into the U half
  REQUIRE(I % 64 == 0, "coda_gemm_swiglu_save: I must be a multiple of 64");
  REQUIRE(M <= 0 || (r == nullptr) != (P == nullptr), "exactly one of r and P must be given");
  TRY(check_gemm_dims(M, I, K, dtype, "I"));
  if (P) REQUIRE(std::isfinite(eps) && eps >= 0.0f, "eps must be finite and >= 0");
  if (M == 0) return CODA_OK;
  TRY(check_ptr(H, "H"));
  TRY(check_ptr(Wgt, "Wgt"));
  TRY(check_ptr(Wut, "Wut"));
  TRY(check_ptr(Act, "Act"));
  TRY(check_ptr(GU, "GU"));
  if (P) TRY(check_ptr(P, "P"));
  else TRY(check_scalar_ptr(r, "r"));
  if (r_out) TRY(check_scalar_ptr(r_out, "r_out"));
  const int64_t T = coda_partial_cols(K);
  const Range outs[] = {rng("Act", Act, M * I * 2), rng("GU", GU, M * 2 * I * 2),
                        rng("r_out", r_out, (P && r_out) ? M * 4 : 0)};
  const Range ins[] = {rng("H", H, M * K * 2), rng("Wgt", Wgt, I * K * 2), rng("Wut", Wut, I * K * 2),
                       rng("r", r, r ? M * 4 : 0), rng("P", P, P ? M * T * 4 : 0)};
  TRY(check_overlaps(outs, 3, ins, 5));
  coda::GemmProblem p = {};
  p.epi = coda::kEpiSwiGLUSave;
  p.A = H;
  p.B = Wgt;
  p.B2 = Wut;
  p.D = Act;
  p.GU = GU;
  p.M = static_cast<int>(M);
  p.N_out = static_cast<int>(I);
  p.K = static_cast<int>(K);
  p.ep.r = P ? nullptr : r;
  p.ep.P_in = P;
  p.ep.T_in = static_cast<int>(T);
  p.ep.n_norm = static_cast<float>(K);
  p.ep.eps = eps;
  p.ep.r_out = P ? r_out : nullptr;
  p.ep.gu_off = static_cast<int>(I);
  p.stream = stream;
  p.pdl = use_pdl();
  return run_gemm(dtype, p);
}

coda_status coda_gemm_swiglu_backward(const void* dOut, const void* Wt, const void* GU, void* dGU, int64_t M,
                                      int64_t I, int64_t K, coda_dtype dtype, cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(dtype == CODA_BF16, "coda_gemm_swiglu_backward: dtype must be CODA_BF16");
  REQUIRE(I % 64 == 0, "coda_gemm_swiglu_backward: I must be a multiple of 64");
  TRY(check_gemm_dims(M, I, K, dtype, "I"));
  if (M == 0) return CODA_OK;
  TRY(check_ptr(dOut, "dOut"));
  TRY(check_ptr(Wt, "Wt"));
  TRY(check_ptr(GU, "GU"));
  TRY(check_ptr(dGU, "dGU"));
  const Range outs[] = {rng("dGU", dGU, M * 2 * I * 2)};
  const Range ins[] = {rng("dOut", dOut, M * K * 2), rng("Wt", Wt, K * I * 2), rng("GU", GU, M * 2 * I * 2)};
  TRY(check_overlaps(outs, 1, ins, 3));
  coda::GemmProblem p = {};
  p.epi = coda::kEpiSwiGLUBwd;
  p.A = dOut;
  p.B = Wt;
  p.R = GU;
  p.D = dGU;
  p.M = static_cast<int>(M);
  p.N_out = static_cast<int>(I);
  p.K = static_cast<int>(K);
  p.ep.gu_off = static_cast<int>(I);
  p.b_mn = true;
  p.stream = stream;
  p.pdl = use_pdl();
  return run_gemm(dtype, p);
}

int64_t coda_block_workspace_bytes(int64_t M) {
  if (M < 0) return -1;
  return ((M + 127) / 128 + 1) * static_cast<int64_t>(sizeof(unsigned));
}

}  // extern "C"

namespace {

// Shared by the one-launch blocks: residual GEMM (phase A) and its consumer
// (phase B) with the reduction folded into the consumer's epilogue.  Checks
// every argument and fills *p; enqueues nothing.  M == 0 leaves p->M at 0
// (nothing to launch).
coda_status block_prepare(int epi_b, const void* X, const void* W1t, const void* R, const void* Wb, const void* Wb2,
                          float eps, void* H, float* P, float* r_out, void* Out, int64_t M, int64_t N, int64_t K,
                          int64_t N_out, coda_dtype dtype, void* workspace, cudaStream_t stream,
                          coda::GemmProblem* pp) {
  g_msg[0] = 0;
  *pp = coda::GemmProblem{};
  if (dtype == CODA_E4M3)
    return fail(CODA_ERR_UNSUPPORTED,
                "one-launch blocks take CODA_F32 or CODA_BF16: FP8 needs the per-tensor amax of h before its consumer");
  TRY(check_gemm_dims(M, N, K, dtype, "N"));
  TRY(check_gemm_dims(M, N_out, N, dtype, epi_b == coda::kEpiSwiGLU ? "I" : "N2"));
  REQUIRE(std::isfinite(eps) && eps >= 0.0f, "eps must be finite and >= 0");
  if (M == 0) return CODA_OK;
  TRY(check_ptr(X, "X"));
  TRY(check_ptr(W1t, "W1t"));
  TRY(check_ptr(R, "R"));
  TRY(check_ptr(Wb, epi_b == coda::kEpiSwiGLU ? "Wgt" : "W2t"));
  if (epi_b == coda::kEpiSwiGLU) TRY(check_ptr(Wb2, "Wut"));
  TRY(check_ptr(H, "H"));
  TRY(check_ptr(P, "P"));
  if (r_out) TRY(check_scalar_ptr(r_out, "r_out"));
  TRY(check_ptr(Out, epi_b == coda::kEpiSwiGLU ? "Act" : "Z"));
  TRY(check_ptr(workspace, "workspace"));
  const int ob = out_bytes(dtype), ib = elem_bytes(dtype);
  const int64_t T = coda_partial_cols(N);
  const Range outs[] = {rng("H", H, M * N * ob), rng("P", P, M * T * 4), rng("r_out", r_out, r_out ? M * 4 : 0),
                        rng(epi_b == coda::kEpiSwiGLU ? "Act" : "Z", Out, M * N_out * ob),
                        rng("workspace", workspace, coda_block_workspace_bytes(M))};
  const Range ins[] = {rng("X", X, M * K * ib), rng("W1t", W1t, N * K * ib), rng("R", R, M * N * ob),
                       rng("W", Wb, N_out * N * ib), rng("Wut", Wb2, Wb2 ? N_out * N * ib : 0)};
  TRY(check_overlaps(outs, 5, ins, 5));
  coda::GemmProblem& p = *pp;
  p.epi = coda::kEpiResidualPartialRms;
  p.A = X;
  p.B = W1t;
  p.R = R;
  p.D = H;
  p.M = static_cast<int>(M);
  p.N_out = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.ep.P = P;
  p.ep.T = static_cast<int>(T);
  p.b.epi = epi_b;
  p.b.A = H;
  p.b.B = Wb;
  p.b.B2 = Wb2;
  p.b.D = Out;
  p.b.N_out = static_cast<int>(N_out);
  p.b.K = static_cast<int>(N);
  p.b.ep.P_in = P;
  p.b.ep.T_in = static_cast<int>(T);
  p.b.ep.n_norm = static_cast<float>(N);
  p.b.ep.eps = eps;
  p.b.ep.r_out = r_out;
  p.band_ready = static_cast<unsigned*>(workspace);
  p.stream = stream;
  p.pdl = use_pdl();
  return CODA_OK;
}

coda_status block_impl(int epi_b, const void* X, const void* W1t, const void* R, const void* Wb, const void* Wb2,
                       float eps, void* H, float* P, float* r_out, void* Out, int64_t M, int64_t N, int64_t K,
                       int64_t N_out, coda_dtype dtype, void* workspace, cudaStream_t stream) {
  coda::GemmProblem p;
  TRY(block_prepare(epi_b, X, W1t, R, Wb, Wb2, eps, H, P, r_out, Out, M, N, K, N_out, dtype, workspace, stream, &p));
  if (p.M == 0) return CODA_OK;
  return run_gemm(dtype, p);
}

}  // namespace

extern "C" {

coda_status coda_block_rowscale(const void* X, const void* W1t, const void* R, const void* W2t, float eps, void* H,
                                float* P, float* r_out, void* Z, int64_t M, int64_t N, int64_t K, int64_t N2,
                                coda_dtype dtype, void* workspace, cudaStream_t stream) {
  return block_impl(coda::kEpiRowScale, X, W1t, R, W2t, nullptr, eps, H, P, r_out, Z, M, N, K, N2, dtype, workspace,
                    stream);
}

coda_status coda_block_rowscale_rope(const void* X, const void* W1t, const void* R, const void* W2t, float eps,
                                     void* H, float* P, float* r_out, void* Z, int64_t M, int64_t N, int64_t K,
                                     int64_t N2, coda_dtype dtype, int64_t head_dim, int64_t rope_cols, double base,
                                     int64_t seq_len, const int32_t* positions, void* workspace,
                                     cudaStream_t stream) {
  coda::GemmProblem p;
  TRY(block_prepare(coda::kEpiRowScale, X, W1t, R, W2t, nullptr, eps, H, P, r_out, Z, M, N, K, N2, dtype, workspace,
                    stream, &p));
  const RopeArgs rope = {head_dim, rope_cols, base, seq_len, positions};
  TRY(check_rope(&rope, M, N2, dtype));
  if (p.M == 0) return CODA_OK;
  const int ob = out_bytes(dtype);
  const int64_t T = coda_partial_cols(N);
  const Range outs[] = {rng("H", H, M * N * ob), rng("P", P, M * T * 4), rng("r_out", r_out, r_out ? M * 4 : 0),
                        rng("Z", Z, M * N2 * ob), rng("workspace", workspace, coda_block_workspace_bytes(M))};
  const Range ins[] = {rng("positions", positions, positions ? M * 4 : 0)};
  TRY(check_overlaps(outs, 5, ins, 1));
  set_rope(p.b.ep, &rope);
  return run_gemm(dtype, p);
}

coda_status coda_block_swiglu(const void* X, const void* W1t, const void* R, const void* Wgt, const void* Wut,
                              float eps, void* H, float* P, float* r_out, void* Act, int64_t M, int64_t N, int64_t K,
                              int64_t I, coda_dtype dtype, void* workspace, cudaStream_t stream) {
  return block_impl(coda::kEpiSwiGLU, X, W1t, R, Wgt, Wut, eps, H, P, r_out, Act, M, N, K, I, dtype, workspace,
                    stream);
}

int64_t coda_block_fp8_workspace_bytes(int64_t M) {
  if (M < 0) return -1;
  return coda::block_counters((M + 127) / 128, true) * static_cast<int64_t>(sizeof(unsigned));
}

}  // extern "C"

namespace {

// Shared by the FP8 one-launch blocks.  Phase A: h = R + dequant(Aq . W1t^T)
// with P and amax_h; the quantiser warps then write Hq = e4m3(h / scale_h);
// phase B: the consumer on Hq with the reduction folded in.  With A_bf16
// given, the quantiser warps first write Aq = e4m3(A / (amax_a / 448)).
coda_status block_fp8_impl(int epi_b, const void* A_bf16, const float* amax_a, uint8_t* Aq, float* scale_a,
                           const uint8_t* W1t, const float* scale_w1, const void* R, const uint8_t* Wb,
                           const float* scale_wb, const uint8_t* Wb2, const float* scale_wb2, float eps, void* H,
                           float* P, float* r_out, float* amax_h, uint8_t* Hq, float* scale_h, void* Out,
                           float* amax_out, int64_t M, int64_t N, int64_t K, int64_t N_out, void* workspace,
                           cudaStream_t stream) {
  g_msg[0] = 0;
  const bool swiglu = epi_b == coda::kEpiSwiGLU;
  TRY(check_gemm_dims(M, N, K, CODA_E4M3, "N"));
  TRY(check_gemm_dims(M, N_out, N, CODA_E4M3, swiglu ? "I" : "N2"));
  REQUIRE(std::isfinite(eps) && eps >= 0.0f, "eps must be finite and >= 0");
  TRY(check_scalar_ptr(amax_h, "amax_h"));
  if (amax_out) TRY(check_scalar_ptr(amax_out, "amax_act"));
  if (M == 0) {
    TRY(zero_scalar(amax_h, stream));
    return zero_scalar(amax_out, stream);
  }
  const bool quant_a = A_bf16 != nullptr;
  if (quant_a) {
    TRY(check_ptr(A_bf16, "A"));
    TRY(check_scalar_ptr(amax_a, "amax_a"));
  }
  TRY(check_ptr(Aq, "Aq"));
  TRY(check_scalar_ptr(scale_a, "scale_a"));
  TRY(check_ptr(W1t, "W1t"));
  TRY(check_scalar_ptr(scale_w1, "scale_w1"));
  TRY(check_ptr(R, "R"));
  TRY(check_ptr(Wb, swiglu ? "Wgt" : "W2t"));
  TRY(check_scalar_ptr(scale_wb, swiglu ? "scale_wg" : "scale_w2"));
  if (swiglu) {
    TRY(check_ptr(Wb2, "Wut"));
    TRY(check_scalar_ptr(scale_wb2, "scale_wu"));
  }
  TRY(check_ptr(H, "H"));
  TRY(check_ptr(P, "P"));
  if (r_out) TRY(check_scalar_ptr(r_out, "r_out"));
  TRY(check_ptr(Hq, "Hq"));
  TRY(check_scalar_ptr(scale_h, "scale_h"));
  TRY(check_ptr(Out, swiglu ? "Act" : "Z"));
  TRY(check_ptr(workspace, "workspace"));
  const int64_t T = coda_partial_cols(N);
  const char* out_name = swiglu ? "Act" : "Z";
  // the launch writes Aq and scale_a when it quantises A; else it reads them
  const Range outs[] = {rng("H", H, M * N * 2), rng("P", P, M * T * 4), rng("r_out", r_out, r_out ? M * 4 : 0),
                        rng("amax_h", amax_h, 4), rng("Hq", Hq, M * N), rng("scale_h", scale_h, 4),
                        rng(out_name, Out, M * N_out * 2), rng("amax_act", amax_out, amax_out ? 4 : 0),
                        rng("workspace", workspace, coda_block_fp8_workspace_bytes(M)),
                        rng("Aq", quant_a ? Aq : nullptr, quant_a ? M * K : 0),
                        rng("scale_a", quant_a ? scale_a : nullptr, quant_a ? 4 : 0)};
  const Range ins[] = {rng("A", A_bf16, quant_a ? M * K * 2 : 0), rng("amax_a", amax_a, quant_a ? 4 : 0),
                       rng("Aq", quant_a ? nullptr : Aq, quant_a ? 0 : M * K),
                       rng("scale_a", quant_a ? nullptr : scale_a, quant_a ? 0 : 4), rng("W1t", W1t, N * K),
                       rng("scale_w1", scale_w1, 4), rng("R", R, M * N * 2), rng("W", Wb, N_out * N),
                       rng("scale_w", scale_wb, 4), rng("Wut", Wb2, Wb2 ? N_out * N : 0),
                       rng("scale_wu", scale_wb2, Wb2 ? 4 : 0)};
  TRY(check_overlaps(outs, 11, ins, 11));
  TRY(zero_scalar(amax_h, stream));
  TRY(zero_scalar(amax_out, stream));
  coda::GemmProblem p = {};
  p.epi = coda::kEpiResidualPartialRms;
  p.A = Aq;
  p.B = W1t;
  p.R = R;
  p.D = H;
  p.M = static_cast<int>(M);
  p.N_out = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.ep.P = P;
  p.ep.T = static_cast<int>(T);
  p.ep.scale_a = scale_a;
  p.ep.scale_b = scale_w1;
  p.ep.amax_out = amax_h;
  p.b.epi = epi_b;
  p.b.A = Hq;
  p.b.B = Wb;
  p.b.B2 = Wb2;
  p.b.D = Out;
  p.b.N_out = static_cast<int>(N_out);
  p.b.K = static_cast<int>(N);
  p.b.ep.P_in = P;
  p.b.ep.T_in = static_cast<int>(T);
  p.b.ep.n_norm = static_cast<float>(N);
  p.b.ep.eps = eps;
  p.b.ep.r_out = r_out;
  p.b.ep.scale_a = scale_h;
  p.b.ep.scale_b = scale_wb;
  p.b.ep.scale_b2 = scale_wb2;
  p.b.ep.amax_out = amax_out;
  p.band_ready = static_cast<unsigned*>(workspace);
  p.fp8_block = true;
  p.q.h = H;
  p.q.hq = Hq;
  p.q.amax_h = amax_h;
  p.q.scale_h = scale_h;
  p.q.a = A_bf16;
  p.q.aq = Aq;
  p.q.amax_a = amax_a;
  p.q.scale_a = scale_a;
  p.stream = stream;
  p.pdl = use_pdl();
  return run_gemm(CODA_E4M3, p);
}

}  // namespace

extern "C" {

coda_status coda_block_swiglu_fp8(const void* X, const float* amax_x, uint8_t* Xq, float* scale_x, const uint8_t* W1t,
                                  const float* scale_w1, const void* R, const uint8_t* Wgt, const float* scale_wg,
                                  const uint8_t* Wut, const float* scale_wu, float eps, void* H, float* P,
                                  float* r_out, float* amax_h, uint8_t* Hq, float* scale_h, void* Act,
                                  float* amax_act, int64_t M, int64_t N, int64_t K, int64_t I, void* workspace,
                                  cudaStream_t stream) {
  return block_fp8_impl(coda::kEpiSwiGLU, X, amax_x, Xq, scale_x, W1t, scale_w1, R, Wgt, scale_wg, Wut, scale_wu, eps,
                        H, P, r_out, amax_h, Hq, scale_h, Act, amax_act, M, N, K, I, workspace, stream);
}

coda_status coda_block_rowscale_fp8(const void* X, const float* amax_x, uint8_t* Xq, float* scale_x,
                                    const uint8_t* W1t, const float* scale_w1, const void* R, const uint8_t* W2t,
                                    const float* scale_w2, float eps, void* H, float* P, float* r_out,
                                    float* amax_h, uint8_t* Hq, float* scale_h, void* Z, int64_t M, int64_t N,
                                    int64_t K, int64_t N2, void* workspace, cudaStream_t stream) {
  return block_fp8_impl(coda::kEpiRowScale, X, amax_x, Xq, scale_x, W1t, scale_w1, R, W2t, scale_w2, nullptr, nullptr,
                        eps, H, P, r_out, amax_h, Hq, scale_h, Z, nullptr, M, N, K, N2, workspace, stream);
}

coda_status coda_amax(const void* x, int64_t n, coda_dtype dtype, float* amax, cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(dtype == CODA_F32 || dtype == CODA_BF16, "coda_amax: dtype must be CODA_F32 or CODA_BF16");
  REQUIRE(n >= 0 && n < (int64_t(1) << 60), "coda_amax: n out of range [0, 2^60)");
  TRY(check_scalar_ptr(amax, "amax"));
  TRY(zero_scalar(amax, stream));
  if (n == 0) return CODA_OK;
  TRY(check_ptr(x, "x"));
  const Range outs[] = {rng("amax", amax, 4)};
  const Range ins[] = {rng("x", x, n * elem_bytes(dtype))};
  TRY(check_overlaps(outs, 1, ins, 1));
  cudaError_t e = coda::launch_amax(x, n, dtype == CODA_F32, amax, stream);
  return e == cudaSuccess ? CODA_OK : cuda_fail(e, "coda_amax launch");
}

coda_status coda_quantize_e4m3(const void* x, int64_t n, coda_dtype dtype, const float* amax, uint8_t* q,
                               float* scale, cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(dtype == CODA_F32 || dtype == CODA_BF16, "coda_quantize_e4m3: dtype must be CODA_F32 or CODA_BF16");
  REQUIRE(n >= 0 && n < (int64_t(1) << 60), "coda_quantize_e4m3: n out of range [0, 2^60)");
  TRY(check_scalar_ptr(amax, "amax"));
  TRY(check_scalar_ptr(scale, "scale"));
  if (n > 0) {
    TRY(check_ptr(x, "x"));
    TRY(check_ptr(q, "q"));
  }
  const Range outs[] = {rng("q", q, n), rng("scale", scale, 4)};
  const Range ins[] = {rng("x", x, n * elem_bytes(dtype)), rng("amax", amax, 4)};
  TRY(check_overlaps(outs, 2, ins, 2));
  cudaError_t e = coda::launch_quantize_e4m3(x, n, dtype == CODA_F32, amax, q, scale, stream);
  return e == cudaSuccess ? CODA_OK : cuda_fail(e, "coda_quantize_e4m3 launch");
}

coda_status coda_selftest_wait_timeout(int64_t timeout_ns, cudaStream_t stream) {
  g_msg[0] = 0;
  REQUIRE(timeout_ns >= 1000 && timeout_ns <= 10000000000LL,
          "coda_selftest_wait_timeout: timeout_ns must lie in [1e3, 1e10]");
  cudaError_t e = coda::launch_wait_probe(timeout_ns, stream);
  return e == cudaSuccess ? CODA_OK : cuda_fail(e, "coda_selftest_wait_timeout launch");
}

coda_status coda_get_device_status(void) {
  g_msg[0] = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  const unsigned s = coda::read_clear_status_bf16() | coda::read_clear_status_tf32() |
                     coda::read_clear_status_e4m3() | coda::read_clear_status_aux();
  if (s == ~0u) return fail(CODA_ERR_CUDA, "could not read the device status word");
  if (s & 1u) return fail(CODA_ERR_TIMEOUT, "a kernel gave up on a bounded wait (timeout)");
  return CODA_OK;
}

}  // extern "C"

// --------------------------------------------------- allocation-free block ----
// Some callers cannot call cudaMalloc at all: runtimes that own every byte of
// device memory and hand a kernel library no workspace, and hot paths where
// an allocation (which may synchronise the device) is not acceptable.  For
// them coda_block_swiglu_noalloc keeps the one-launch block's band counters
// in this file-scope device array instead of a caller workspace.  Every GPU
// that loads the library holds it (4100 bytes) until the process exits.
static __device__ __align__(256) unsigned g_noalloc_band_counters[(kNoAllocMaxRows + 127) / 128 + 1];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// The array's name is only a host-side stand-in: the kernel needs its device
// address, looked up once per device with that device current.
coda_status noalloc_counters(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(CODA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_band_counters);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(band counters)");
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return CODA_OK;
}

}  // namespace

extern "C" coda_status coda_block_swiglu_noalloc(const void* X, const void* W1t, const void* R, const void* Wgt,
                                                 const void* Wut, float eps, void* H, float* P, float* r_out,
                                                 void* Act, int64_t M, int64_t N, int64_t K, int64_t I,
                                                 coda_dtype dtype, cudaStream_t stream) {
  g_msg[0] = 0;
  if (M > kNoAllocMaxRows)
    return fail(CODA_ERR_INVALID_ARG,
                "M = %" PRId64 " exceeds the %d rows of the library's built-in band counters; use coda_block_swiglu "
                "with a workspace",
                M, kNoAllocMaxRows);
  if (M <= 0) return coda_block_swiglu(X, W1t, R, Wgt, Wut, eps, H, P, r_out, Act, M, N, K, I, dtype, nullptr, stream);
  void* counters = nullptr;
  TRY(noalloc_counters(&counters));
  // every argument is checked before anything is enqueued, so a rejected
  // call leaves the shared array untouched
  coda::GemmProblem p;
  TRY(block_prepare(coda::kEpiSwiGLU, X, W1t, R, Wgt, Wut, eps, H, P, r_out, Act, M, N, K, I, dtype, counters, stream,
                    &p));
  // every call shares the array: start from zero whatever the last call left
  const int64_t bytes = coda_block_workspace_bytes(M);
  cudaError_t e = cudaMemsetAsync(counters, 0, static_cast<size_t>(bytes), stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(band counters)");
  return run_gemm(dtype, p);
}
