// Per-tensor FP8 (OCP E4M3) quantisation of GEMM operands, shared by the
// standalone quantise kernel (coda_aux.cu) and the quantiser warps of the
// FP8 one-launch blocks (gemm_epilogue.cuh), so both decide every code the
// same way: s = amax / 448 (1 for an all-zero tensor), q = E4M3(x / s) with
// round-to-nearest-even and saturation to +-448.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace coda {

__device__ __forceinline__ float e4m3_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

// The quotient's fast form is valid for s in this range (nothing underflows).
__device__ __forceinline__ bool e4m3_fast_scale(float s) { return s >= 0x1p-100f && s <= 0x1p100f; }

// x / s rounded to nearest, without a divide per element.  With inv the
// correctly rounded reciprocal of s: q0 = x * inv is within an ulp of x / s,
// the residual x - s * q0 is exact in one FMA, and q0 + residual * inv rounds
// to the correctly rounded quotient (Markstein's theorem on FMA division,
// IBM J. Res. Dev. 34(1), 1990).  It holds while nothing underflows, which the
// caller ensures by taking this path only when e4m3_fast_scale(s).
__device__ __forceinline__ float div_rn_by(float x, float s, float inv) {
  const float q0 = __fmul_rn(x, inv);
  return fmaf(fmaf(-s, q0, x), inv, q0);
}

// The same quotient for two values on the packed fp32 pipe: the .f32x2
// multiply and FMA round each lane to nearest exactly as their scalar forms
// (no flush of subnormals), so the results are the scalar ones bit for bit,
// in half the instructions.
__device__ __forceinline__ float2 div_rn_by2(float2 x, float s, float inv) {
  const float2 q0 = fmul2(x, make_float2(inv, inv));
  return ffma2(ffma2(make_float2(-s, -s), q0, x), make_float2(inv, inv), q0);
}

// q = e4m3(x / s), round-to-nearest-even, saturating (cvt ... .satfinite).
template <bool FAST>
__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi, float s, float inv) {
  const float2 q = FAST ? div_rn_by2(make_float2(lo, hi), s, inv) : make_float2(__fdiv_rn(lo, s), __fdiv_rn(hi, s));
  return __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
}

// 16 floats -> 16 e4m3 codes (16 bytes, element order kept).
template <bool FAST>
__device__ __forceinline__ uint4 e4m3x16(const float (&f)[16], float s, float inv) {
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    o[j] = static_cast<uint32_t>(to_e4m3x2<FAST>(f[4 * j], f[4 * j + 1], s, inv)) |
           (static_cast<uint32_t>(to_e4m3x2<FAST>(f[4 * j + 2], f[4 * j + 3], s, inv)) << 16);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 16 bf16 values (two 16-byte words) -> 16 floats.
__device__ __forceinline__ void bf16x16_to_float(const uint4& w0, const uint4& w1, float (&f)[16]) {
  const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&w0);
  const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&w1);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 a = __bfloat1622float2(h0[e]);
    const float2 b = __bfloat1622float2(h1[e]);
    f[2 * e] = a.x;
    f[2 * e + 1] = a.y;
    f[8 + 2 * e] = b.x;
    f[8 + 2 * e + 1] = b.y;
  }
}

}  // namespace coda
