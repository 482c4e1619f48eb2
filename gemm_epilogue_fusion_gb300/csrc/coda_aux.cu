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

// 16 bytes of W^T per thread: 8 bf16 or 4 fp32 elements of one row (K gives
// 16-byte rows, so a vector never straddles two rows).
template <bool F32>
__global__ void __launch_bounds__(256) fold_gamma_kernel(const uint4* __restrict__ W, const float* __restrict__ gamma,
                                                         uint4* __restrict__ out, int64_t n_vec, int64_t K) {
  constexpr int VEC = F32 ? 4 : 8;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < n_vec;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t k0 = (v * VEC) % K;
    uint4 w = W[v];
    if constexpr (F32) {
      float4 f = *reinterpret_cast<float4*>(&w);
      f.x *= gamma[k0];
      f.y *= gamma[k0 + 1];
      f.z *= gamma[k0 + 2];
      f.w *= gamma[k0 + 3];
      out[v] = *reinterpret_cast<uint4*>(&f);
    } else {
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        h[e] = __floats2bfloat162_rn(f.x * gamma[k0 + 2 * e], f.y * gamma[k0 + 2 * e + 1]);
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

__device__ __forceinline__ float e4m3_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

// q = e4m3(x / s), round-to-nearest-even, saturating (cvt ... .satfinite).
__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi, float s) {
  return __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(lo, s), __fdiv_rn(hi, s)), __NV_SATFINITE, __NV_E4M3);
}

// 16 elements per thread: 16 bytes of q.
template <bool F32>
__global__ void __launch_bounds__(256) quantize_kernel(const void* __restrict__ x, int64_t n,
                                                       const float* __restrict__ amax, uint8_t* __restrict__ q,
                                                       float* __restrict__ scale) {
  pdl_wait();
  const float s = e4m3_scale(*amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale = s;
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
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = static_cast<uint32_t>(to_e4m3x2(f[4 * j], f[4 * j + 1], s)) |
             (static_cast<uint32_t>(to_e4m3x2(f[4 * j + 2], f[4 * j + 3], s)) << 16);
    reinterpret_cast<uint4*>(q)[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (blockIdx.x == 0) {
    for (int64_t i = n16 * 16 + threadIdx.x; i < n; i += blockDim.x) {
      const float f = F32 ? reinterpret_cast<const float*>(x)[i]
                          : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[i]);
      q[i] = static_cast<uint8_t>(to_e4m3x2(f, 0.0f, s) & 0xFF);
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
  const int64_t n_vec = N_out * K / (f32 ? 4 : 8);
  const int g = grid_for(n_vec, 256);
  if (f32)
    fold_gamma_kernel<true><<<g, 256, 0, s>>>(static_cast<const uint4*>(Wt), gamma, static_cast<uint4*>(Wt_out),
                                              n_vec, K);
  else
    fold_gamma_kernel<false><<<g, 256, 0, s>>>(static_cast<const uint4*>(Wt), gamma, static_cast<uint4*>(Wt_out),
                                               n_vec, K);
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

unsigned read_clear_status_aux() { return 0u; }

}  // namespace coda
