// common.cuh -- device helpers shared by the selective-scan kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Steps between the state checkpoints of the backward pass's recomputation.
constexpr int kCkSteps = 16;

// ---- element conversions --------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// ---- MUFU wrappers ---------------------------------------------------------------
// 2^x on the special-function unit; results below 2^-126 flush to zero, which only
// drops contributions that are already far below fp32 resolution of the state.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Decay factor exp(dt * A) for one state. The bf16 path takes 2^(dt * A * log2 e) on
// the SFU (A2 = A * log2 e prepared once per channel). The fp32 path must be close to
// correctly rounded: a long-memory state (A-bar near 1) amplifies any bias in A-bar
// by about 1 / (1 - A-bar), so it evaluates exp in double from the exact product.
template <bool kAccurate>
__device__ __forceinline__ float decay(float dt, float A, float A2) {
  if (kAccurate) return (float)exp((double)dt * (double)A);
  return ex2(dt * A2);
}

// B-bar factor of the exact zero-order hold for one diagonal entry A of the state
// matrix: (exp(dt A) - 1) / A, with its limit dt at A = 0, so that B-bar = factor * B.
// expm1 keeps the factor accurate when dt A is small (no cancellation in exp - 1); the
// fp32 I/O path evaluates it in double like its decay.
template <bool kAccurate>
__device__ __forceinline__ float zoh_factor(float dt, float A) {
  if (A == 0.f) return dt;
  if (kAccurate) return (float)(expm1((double)dt * (double)A) / (double)A);
  return expm1f(dt * A) / A;
}

// ---- step-size map and gate -----------------------------------------------------
// Accurate softplus log(1 + e^r): identity above 20 (the remainder e^-20 is below
// fp32 resolution of r), log1p otherwise.
__device__ __forceinline__ float softplus_precise(float r) {
  return r > 20.f ? r : log1pf(expf(r));
}

// Accurate SiLU z * sigmoid(z).
__device__ __forceinline__ float silu_precise(float z) {
  return z / (1.f + expf(-z));
}

// ---- device-side error word (bounded waits set it instead of trapping) -----------
// Defined here: the library is one translation unit (ssm_abi.cu includes every kernel).
__device__ int g_ssm_error = 0;

}  // namespace ssm
