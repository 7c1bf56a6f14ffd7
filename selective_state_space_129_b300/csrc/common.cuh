// Device helpers shared by the scan kernels of libm3scan.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace m3 {

// Activation loads/stores: fp32 or bf16 storage, fp32 arithmetic.
template <typename T>
__device__ __forceinline__ float ld_act(const T* p);
template <>
__device__ __forceinline__ float ld_act<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_act<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st_act(T* p, float v);
template <>
__device__ __forceinline__ void st_act<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_act<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

// Reduce an angle to [-pi, pi] by subtracting the nearest multiple of 2*pi.
// 2*pi is split in two parts (Cody & Waite's additive range reduction): the
// head has few significant bits so that k*head is exact for the small k seen
// here, the tail carries the remaining bits of 2*pi.
__device__ __forceinline__ float wrap_angle(float a) {
  const float kInvTwoPi = 0.159154943091895335768883763372514362f;
  const float kTwoPiHead = 6.28125f;
  const float kTwoPiTail = 1.93530717958647692528676655900576839e-3f;
  const float k = rintf(a * kInvTwoPi);
  return fmaf(-k, kTwoPiTail, fmaf(-k, kTwoPiHead, a));
}

}  // namespace m3
