// Device-side elementwise math: bf16 packing and the activations of the
// column-parallel epilogue with their derivatives.  The activations act
// coordinate by coordinate, which is why they commute with the column split
// ("02 — Tensor Parallelism", section "The MLP pairing").
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "tp.h"

namespace tp {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Two floats -> one 32-bit word of two bf16 (lo = a, hi = b), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t w, float& a, float& b) {
  a = __uint_as_float(w << 16);
  b = __uint_as_float(w & 0xFFFF0000u);
}

// IEEE fp16 pairs (the attention kernels keep Q, K, V, P, dO and dS in fp16).
__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void unpack_f16x2(uint32_t w, float& a, float& b) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  const float2 f = __half22float2(h);
  a = f.x;
  b = f.y;
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kSqrt2OverPi = 0.7978845608028654f;
constexpr float kGeluC = 0.044715f;
constexpr float kInvSqrt2 = 0.7071067811865476f;
constexpr float kInvSqrt2Pi = 0.3989422804014327f;

__device__ __forceinline__ float act_apply(int act, float z) {
  switch (act) {
    case TP_ACT_RELU:
      return fmaxf(z, 0.0f);
    case TP_ACT_GELU_TANH: {
      const float u = kSqrt2OverPi * fmaf(kGeluC * z, z * z, z);
      return 0.5f * z * (1.0f + tanh_fast(u));
    }
    case TP_ACT_GELU_ERF:
      return 0.5f * z * (1.0f + erff(z * kInvSqrt2));
    default:
      return z;
  }
}

__device__ __forceinline__ float act_grad(int act, float z) {
  switch (act) {
    case TP_ACT_RELU:
      return z > 0.0f ? 1.0f : 0.0f;
    case TP_ACT_GELU_TANH: {
      const float u = kSqrt2OverPi * fmaf(kGeluC * z, z * z, z);
      const float th = tanh_fast(u);
      const float du = kSqrt2OverPi * fmaf(3.0f * kGeluC * z, z, 1.0f);
      return 0.5f * (1.0f + th) + 0.5f * z * (1.0f - th * th) * du;
    }
    case TP_ACT_GELU_ERF:
      return 0.5f * (1.0f + erff(z * kInvSqrt2)) + z * kInvSqrt2Pi * expf(-0.5f * z * z);
    default:
      return 1.0f;
  }
}

// Compile-time forms: one activation per kernel instantiation keeps the
// unrolled epilogue small.
template <int ACT>
__device__ __forceinline__ float act_apply_t(float z) {
  if constexpr (ACT == TP_ACT_RELU) {
    return fmaxf(z, 0.0f);
  } else if constexpr (ACT == TP_ACT_GELU_TANH) {
    const float u = kSqrt2OverPi * fmaf(kGeluC * z, z * z, z);
    return 0.5f * z * (1.0f + tanh_fast(u));
  } else if constexpr (ACT == TP_ACT_GELU_ERF) {
    return 0.5f * z * (1.0f + erff(z * kInvSqrt2));
  } else {
    return z;
  }
}

template <int ACT>
__device__ __forceinline__ float act_grad_t(float z) {
  if constexpr (ACT == TP_ACT_RELU) {
    return z > 0.0f ? 1.0f : 0.0f;
  } else if constexpr (ACT == TP_ACT_GELU_TANH) {
    const float u = kSqrt2OverPi * fmaf(kGeluC * z, z * z, z);
    const float th = tanh_fast(u);
    const float du = kSqrt2OverPi * fmaf(3.0f * kGeluC * z, z, 1.0f);
    return 0.5f * (1.0f + th) + 0.5f * z * (1.0f - th * th) * du;
  } else if constexpr (ACT == TP_ACT_GELU_ERF) {
    return 0.5f * (1.0f + erff(z * kInvSqrt2)) + z * kInvSqrt2Pi * expf(-0.5f * z * z);
  } else {
    return 1.0f;
  }
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Gradient of a = silu(g) u given da:  d up = da silu(g),  d gate = da u silu'(g) with
// silu'(g) = s (1 + g (1 - s)), s = sigmoid(g).
__device__ __forceinline__ void swiglu_grad(float g, float u, float da, float& dg, float& du) {
  const float s = 1.0f / (1.0f + expf(-g));
  dg = da * u * (s * (1.0f + g * (1.0f - s)));
  du = da * (g * s);
}

}  // namespace tp
