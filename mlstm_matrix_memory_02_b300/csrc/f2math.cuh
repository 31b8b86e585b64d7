// f2math.cuh -- packed fp32-pair arithmetic and 16-bit conversions shared by the tensor-core
// kernels (sm_103a: one f32x2 instruction works on two lanes of data).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace mlstm {

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2unpack(uint64_t x, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// bf16 pair -> fp32 pair
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) { return f2pack(bf16_lo(w), bf16_hi(w)); }
// fp32 pair -> fp16 pair (round to nearest)
__device__ __forceinline__ uint32_t f2_to_h2(uint64_t x) {
  float lo, hi;
  f2unpack(x, lo, hi);
  return pack_half2(lo, hi);
}
// bf16 pair -> fp16 pair (exact for values inside the fp16 range)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) { return pack_half2(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ float f2sum(uint64_t x) {
  float lo, hi;
  f2unpack(x, lo, hi);
  return lo + hi;
}

}  // namespace mlstm
