// common.cuh -- small device helpers shared by the mLSTM kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mlstm {

// ---------------------------------------------------------------- storage conversions
template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------- gate math
// log sigmoid(x) = min(x, 0) - log(1 + exp(-|x|)): the exponent is never positive.
__device__ __forceinline__ float log_sigmoid(float x) { return fminf(x, 0.f) - log1pf(expf(-fabsf(x))); }
// log f of the forget-gate variant: f = sigmoid(f~) (log sigmoid(f~)) or f = exp(f~) (f~ itself)
__device__ __forceinline__ float log_forget(float x, int exp_fg) { return exp_fg ? x : log_sigmoid(x); }

// ---------------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace mlstm
