// MXFP8 block rule shared by the quantising kernels (OCP Microscaling: scale
// 2^(floor(log2 amax) - 8) as a biased UE8M0 byte, elements rounded to nearest-even E4M3
// with saturation, all-zero block -> byte 127) and the scale-atom byte position.
#pragma once
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mok {

__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  if (amax == 0.f) return 127u;  // all-zero block
  const int biased = (int)((__float_as_uint(amax) >> 23) & 0xFF);
  const int b = biased - 8;      // floor(log2 amax) - 8, biased by 127
  return (uint32_t)(b < 0 ? 0 : b);
}
// 2^(127 - byte): the factor that maps the block onto E4M3's range
__device__ __forceinline__ float mx_inv_scale(uint32_t byte) {
  return __uint_as_float((254u - byte) << 23);
}
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
// byte of (row m, K index k) inside its 512-byte atom (128 rows x 4 blocks of 32 along K)
__device__ __forceinline__ size_t atom_byte(int m, int k) {
  return (size_t)(16 * (m & 31) + 4 * ((m & 127) >> 5) + ((k & 127) >> 5));
}

}  // namespace mok
