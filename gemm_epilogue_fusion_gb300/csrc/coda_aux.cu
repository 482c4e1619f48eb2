// Memory-bound helper kernels of the fused block:
//   rms_reduce      the "very light auxiliary reduction kernel" of the CODA
//                   write-up's section "CODA: the treasure hidden in the
//                   epilogue": r_i = 1/sqrt(sum_g P[i, g] / N + eps)
//   fold_gamma      W'^T[n, k] = W^T[n, k] * gamma[k] (RMSNorm weight folded
//                   into the next GEMM's weight, once per weight)
//   amax, quantize  per-tensor FP8 e4m3 scaling of GEMM operands
// None of them waits on anything, so none can time out.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "coda_internal.h"
#include "fp8_e4m3.cuh"
#include "sm103_ptx.cuh"

namespace coda {
namespace {

// One thread per row; a row's T partials are contiguous (16-byte loads when
// T is a multiple of 4, which keeps every row 16-byte aligned).  The same
// row_rstd() runs inside the row-scale and SwiGLU epilogues when they are
// given the partials instead of r.
__global__ void __launch_bounds__(256) rms_reduce_kernel(const float* __restrict__ P, int M, int T, float n,
                                                         float eps, float* __restrict__ r) {
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= M) return;
  r[i] = row_rstd(P + static_cast<int64_t>(i) * T, T, n, eps);
}

// One 16-byte vector of W^T per thread and row: 8 bf16 or 4 fp32 elements.
// Thread x of the grid owns the vector column x (K gives 16-byte rows, so a
// vector never straddles two rows), loads its gamma once, and walks the rows
// blockIdx.y, blockIdx.y + gridDim.y, ...
template <bool F32>
__global__ void __launch_bounds__(256) fold_gamma_kernel(const uint4* __restrict__ W, const float* __restrict__ gamma,
                                                         uint4* __restrict__ out, int64_t n_rows, int64_t row_vecs) {
  constexpr int VEC = F32 ? 4 : 8;
  const int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (c >= row_vecs) return;
  float g[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) g[e] = __ldg(gamma + c * VEC + e);
#pragma unroll 4
  for (int64_t r = blockIdx.y; r < n_rows; r += gridDim.y) {
    const int64_t v = r * row_vecs + c;
    uint4 w = __ldg(W + v);
    if constexpr (F32) {
      float4 f = *reinterpret_cast<float4*>(&w);
      f.x *= g[0];
      f.y *= g[1];
      f.z *= g[2];
      f.w *= g[3];
      out[v] = *reinterpret_cast<uint4*>(&f);
    } else {
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        h[e] = __floats2bfloat162_rn(f.x * g[2 * e], f.y * g[2 * e + 1]);
      }
      out[v] = w;
    }
  }
}

__device__ __forceinline__ float block_max(float v) {
  __shared__ float red[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  }
  return v;
}

// max |x| over n elements; 16-byte vectors plus a scalar tail.  The result
// is combined with atomicMax on the bit pattern (order-preserving for
// non-negative floats) into *amax, which the caller zeroed.
template <bool F32>
__global__ void __launch_bounds__(256) amax_kernel(const void* __restrict__ x, int64_t n, float* amax) {
  pdl_wait();
  constexpr int VEC = F32 ? 4 : 8;
  const int64_t n_vec = n / VEC;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  float m = 0.0f;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < n_vec;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    uint4 w = __ldg(xv + v);
    if constexpr (F32) {
      const float4 f = *reinterpret_cast<float4*>(&w);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
    } else {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
  }
  if (blockIdx.x == 0) {
    for (int64_t i = n_vec * VEC + threadIdx.x; i < n; i += blockDim.x) {
      const float f = F32 ? reinterpret_cast<const float*>(x)[i]
                          : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[i]);
      m = fmaxf(m, fabsf(f));
    }
  }
  m = block_max(m);
  if (threadIdx.x == 0) atomicMax(reinterpret_cast<int*>(amax), __float_as_int(m));
}

// 16 elements per thread: 16 bytes of q.
template <bool F32, bool FAST>
__device__ __forceinline__ void quantize_range(const void* __restrict__ x, int64_t n, float s, float inv,
                                               uint8_t* __restrict__ q) {
  const int64_t n16 = n / 16;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < n16;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float f[16];
    if constexpr (F32) {
      const float4* xv = reinterpret_cast<const float4*>(x) + v * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 a = __ldg(xv + j);
        f[4 * j] = a.x;
        f[4 * j + 1] = a.y;
        f[4 * j + 2] = a.z;
        f[4 * j + 3] = a.w;
      }
    } else {
      const uint4* xv = reinterpret_cast<const uint4*>(x) + v * 2;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint4 w = __ldg(xv + j);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 t = __bfloat1622float2(h[e]);
          f[8 * j + 2 * e] = t.x;
          f[8 * j + 2 * e + 1] = t.y;
        }
      }
    }
    reinterpret_cast<uint4*>(q)[v] = e4m3x16<FAST>(f, s, inv);
  }
  if (blockIdx.x == 0) {
    for (int64_t i = n16 * 16 + threadIdx.x; i < n; i += blockDim.x) {
      const float f = F32 ? reinterpret_cast<const float*>(x)[i]
                          : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[i]);
      q[i] = static_cast<uint8_t>(to_e4m3x2<FAST>(f, 0.0f, s, inv) & 0xFF);
    }
  }
}

template <bool F32>
__global__ void __launch_bounds__(256) quantize_kernel(const void* __restrict__ x, int64_t n,
                                                       const float* __restrict__ amax, uint8_t* __restrict__ q,
                                                       float* __restrict__ scale) {
  pdl_wait();
  const float s = e4m3_scale(*amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale = s;
  if (e4m3_fast_scale(s)) {  // uniform over the launch
    quantize_range<F32, true>(x, n, s, __frcp_rn(s), q);
  } else {
    quantize_range<F32, false>(x, n, s, 0.0f, q);
  }
}

// RMSNorm backward on [M, N] (y = h r gamma), given dY and the grad-norm
// GEMM's partials S[i, g] = sum over group g of gamma_j dY_ij h_ij:
//   c_i   = r_i^3 / N * sum_g S[i, g]
//   dh_ij = r_i gamma_j dY_ij - c_i h_ij (+ dH_in_ij)
//   Yt_ij = r_i h_ij                       (the weight gradient's operand)
//   part[chunk, j] = sum over the chunk's rows of dY_ij h_ij r_i  (dgamma partials)
// Block: kBwdThreads threads x 8 columns each, one chunk of kBwdRows rows.
constexpr int kBwdRows = 64;
constexpr int kBwdThreads = 128;

__global__ void __launch_bounds__(kBwdThreads) rmsnorm_bwd_kernel(
    const uint4* __restrict__ dY, const uint4* __restrict__ H, const float* __restrict__ r,
    const float* __restrict__ gamma, const float* __restrict__ S, int T, const uint4* __restrict__ dH_in,
    uint4* __restrict__ dH, uint4* __restrict__ Yt, float* __restrict__ part, int M, int N) {
  __shared__ float s_r[kBwdRows], s_c[kBwdRows];
  const int row0 = blockIdx.y * kBwdRows;
  if (threadIdx.x < kBwdRows) {
    const int i = row0 + threadIdx.x;
    float ri = 0.0f, ci = 0.0f;
    if (i < M) {
      ri = r[i];
      float sum = 0.0f;
      for (int t = 0; t < T; ++t) sum += S[static_cast<int64_t>(i) * T + t];
      ci = ri * ri * ri / static_cast<float>(N) * sum;
    }
    s_r[threadIdx.x] = ri;
    s_c[threadIdx.x] = ci;
  }
  __syncthreads();
  const int col = (blockIdx.x * kBwdThreads + threadIdx.x) * 8;
  if (col >= N) return;
  float g[8], dg[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    g[e] = __ldg(gamma + col + e);
    dg[e] = 0.0f;
  }
  const int nv = N / 8;
  const int rows = min(kBwdRows, M - row0);
  const uint4 zero = make_uint4(0, 0, 0, 0);
  // one row of this thread's 8 columns: stores dh and r h, accumulates dgamma
  auto row_out = [&](int ii, int64_t v, const uint4& a, const uint4& b, const uint4& d) {
    const float ri = s_r[ii], ci = s_c[ii];
    const __nv_bfloat162* ya = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&b);
    const __nv_bfloat162* dd = reinterpret_cast<const __nv_bfloat162*>(&d);
    uint4 o1, o2;
    __nv_bfloat162* w1 = reinterpret_cast<__nv_bfloat162*>(&o1);
    __nv_bfloat162* w2 = reinterpret_cast<__nv_bfloat162*>(&o2);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 y = __bfloat1622float2(ya[e]), h = __bfloat1622float2(hb[e]), x = __bfloat1622float2(dd[e]);
      w1[e] = __floats2bfloat162_rn(ri * g[2 * e] * y.x - ci * h.x + x.x, ri * g[2 * e + 1] * y.y - ci * h.y + x.y);
      w2[e] = __floats2bfloat162_rn(ri * h.x, ri * h.y);
      dg[2 * e] += y.x * h.x * ri;
      dg[2 * e + 1] += y.y * h.y * ri;
    }
    dH[v] = o1;
    Yt[v] = o2;
  };
  // rows in groups of 4: all loads of a group are issued before any use, so
  // a thread keeps 8-12 16-byte loads in flight; rows are still consumed in
  // order, so dgamma's partial sums are unchanged
  int ii = 0;
  for (; ii + 4 <= rows; ii += 4) {
    uint4 a[4], b[4], d[4];
    int64_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      v[u] = static_cast<int64_t>(row0 + ii + u) * nv + col / 8;
      a[u] = __ldg(dY + v[u]);
      b[u] = __ldg(H + v[u]);
      d[u] = dH_in ? __ldg(dH_in + v[u]) : zero;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) row_out(ii + u, v[u], a[u], b[u], d[u]);
  }
  for (; ii < rows; ++ii) {
    const int64_t v = static_cast<int64_t>(row0 + ii) * nv + col / 8;
    row_out(ii, v, __ldg(dY + v), __ldg(H + v), dH_in ? __ldg(dH_in + v) : zero);
  }
  float4* pp = reinterpret_cast<float4*>(part + static_cast<int64_t>(blockIdx.y) * N + col);
  pp[0] = make_float4(dg[0], dg[1], dg[2], dg[3]);
  pp[1] = make_float4(dg[4], dg[5], dg[6], dg[7]);
}

// dgamma[j] = sum over chunks of part[chunk, j]: the 8 warps of a block each
// sum every 8th chunk in chunk order for 32 columns, then warp 0 adds the 8
// partial sums in warp order.  The order is fixed, so the result is the same
// on every run.
constexpr int kColSumWarps = 8;
__global__ void __launch_bounds__(32 * kColSumWarps) column_sum_kernel(const float* __restrict__ part, int chunks,
                                                                       int N, float* __restrict__ out) {
  __shared__ float s[kColSumWarps][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + lane;
  float acc = 0.0f;
  if (j < N)
    for (int c = w; c < chunks; c += kColSumWarps) acc += part[static_cast<int64_t>(c) * N + j];
  s[w][lane] = acc;
  __syncthreads();
  if (w == 0 && j < N) {
    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < kColSumWarps; ++k) sum += s[k][lane];
    out[j] = sum;
  }
}

// Status word of this translation unit, read back (and cleared) by
// read_clear_status_aux(): the wait probe's timeout bit.
__device__ unsigned g_aux_status;

// Self-test of the failure path: one thread waits on an mbarrier that nothing
// signals, bounded by timeout_ns of %globaltimer like every wait of the GEMM
// kernels, then raises the timeout bit and returns, leaving the context usable.
__global__ void __launch_bounds__(32) wait_probe_kernel(uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  const uint32_t a = smem_u32(&bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, 0u)) {  // phase 0 of a fresh barrier never completes
    if (globaltimer_ns() - t0 > timeout_ns) {
      atomicOr(&g_aux_status, kDevTimeout);
      return;
    }
  }
}

int grid_for(int64_t work_items, int threads) {
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  int64_t g = (work_items + threads - 1) / threads;
  if (g > cap) g = cap;
  return g < 1 ? 1 : static_cast<int>(g);
}

}  // namespace

cudaError_t launch_rms_reduce(const float* P, int64_t M, int T, int64_t N, float eps, float* r, cudaStream_t s,
                              bool pdl) {
  int m = static_cast<int>(M);
  float n = static_cast<float>(N);
  void* args[] = {&P, &m, &T, &n, &eps, &r};
  return launch_ex(reinterpret_cast<const void*>(rms_reduce_kernel), dim3((m + 255) / 256), dim3(256), 0, s, pdl,
                   args);
}

cudaError_t launch_fold_gamma(const void* Wt, const float* gamma, void* Wt_out, int64_t N_out, int64_t K, bool f32,
                              cudaStream_t s) {
  const int64_t row_vecs = K / (f32 ? 4 : 8);
  const unsigned gx = static_cast<unsigned>((row_vecs + 255) / 256);
  // about 8 blocks per SM in all, each walking every gridDim.y-th row
  int64_t gy = (static_cast<int64_t>(device_sm_count()) * 8 + gx - 1) / gx;
  gy = gy < N_out ? gy : N_out;
  gy = gy < 65535 ? gy : 65535;
  const dim3 grid(gx, static_cast<unsigned>(gy > 0 ? gy : 1));
  if (f32)
    fold_gamma_kernel<true><<<grid, 256, 0, s>>>(static_cast<const uint4*>(Wt), gamma, static_cast<uint4*>(Wt_out),
                                                 N_out, row_vecs);
  else
    fold_gamma_kernel<false><<<grid, 256, 0, s>>>(static_cast<const uint4*>(Wt), gamma, static_cast<uint4*>(Wt_out),
                                                  N_out, row_vecs);
  return cudaGetLastError();
}

int64_t rmsnorm_bwd_chunks(int64_t M) { return (M + kBwdRows - 1) / kBwdRows; }

cudaError_t launch_rmsnorm_backward(const void* dY, const void* H, const float* r, const float* gamma,
                                    const float* S, int T, const void* dH_in, void* dH, void* Yt, float* dgamma,
                                    float* part, int64_t M, int64_t N, cudaStream_t s) {
  const int chunks = static_cast<int>(rmsnorm_bwd_chunks(M));
  const dim3 grid(static_cast<unsigned>((N / 8 + kBwdThreads - 1) / kBwdThreads), static_cast<unsigned>(chunks));
  rmsnorm_bwd_kernel<<<grid, kBwdThreads, 0, s>>>(
      static_cast<const uint4*>(dY), static_cast<const uint4*>(H), r, gamma, S, T, static_cast<const uint4*>(dH_in),
      static_cast<uint4*>(dH), static_cast<uint4*>(Yt), part, static_cast<int>(M), static_cast<int>(N));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  column_sum_kernel<<<static_cast<unsigned>((N + 31) / 32), 32 * kColSumWarps, 0, s>>>(part, chunks, static_cast<int>(N),
                                                                                dgamma);
  return cudaGetLastError();
}

cudaError_t launch_amax(const void* x, int64_t n, bool f32, float* amax, cudaStream_t s) {
  const int g = grid_for(n / (f32 ? 4 : 8) + 1, 256);
  if (f32)
    amax_kernel<true><<<g, 256, 0, s>>>(x, n, amax);
  else
    amax_kernel<false><<<g, 256, 0, s>>>(x, n, amax);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const void* x, int64_t n, bool f32, const float* amax, uint8_t* q, float* scale,
                                 cudaStream_t s) {
  const int g = grid_for(n / 16 + 1, 256);
  if (f32)
    quantize_kernel<true><<<g, 256, 0, s>>>(x, n, amax, q, scale);
  else
    quantize_kernel<false><<<g, 256, 0, s>>>(x, n, amax, q, scale);
  return cudaGetLastError();
}

cudaError_t launch_wait_probe(int64_t timeout_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(static_cast<uint64_t>(timeout_ns));
  return cudaGetLastError();
}

unsigned read_clear_status_aux() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_aux_status, sizeof(v)) != cudaSuccess) return ~0u;
  if (cudaMemcpyToSymbol(g_aux_status, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
  return v;
}

}  // namespace coda
