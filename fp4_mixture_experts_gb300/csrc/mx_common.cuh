// MXFP8 block quantisation (OCP Microscaling v1.0 conversion, E4M3 element,
// one E8M0 scale per 32 elements), shared by the activation quantiser, the
// quantising gather and the block-scaled W13 epilogue.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace moe_fp4 {

// floor(log2(v)) of a nonzero bf16 magnitude given by its 15 low bits.
__device__ __forceinline__ int bf16_floor_log2(uint32_t mag) {
  const int e = (int)(mag >> 7);
  if (e > 0) return e - 127;
  return -133 + (31 - __clz(mag));  // subnormal: mag * 2^-133, mag in [1, 127]
}

// E8M0 scale byte of a block from its largest bf16 magnitude (15 low bits):
// 2^(floor(log2 amax) - 8), exponent clamped at -127; 0 for an all-zero
// block; 0xFF (NaN) for a block holding an infinity or a NaN.
__device__ __forceinline__ uint32_t mx_scale_byte(uint32_t amax) {
  if (amax >= 0x7F80u) return 0xFFu;
  const int s = amax == 0 ? -127 : max(bf16_floor_log2(amax) - 8, -127);
  return (uint32_t)(s + 127);
}

// E4M3 code of a bf16 value divided by the block scale (scale byte < 0xFF):
// v * 2^(127 - byte) is exact (a normal fp32 power of two for bytes 0..254),
// then rounded to nearest even and saturated at +-448.
__device__ __forceinline__ uint32_t mx_e4m3_code(uint32_t bf16_bits, uint32_t scale_byte) {
  const float inv = __uint_as_float((254u - scale_byte) << 23);  // 2^(127 - byte)
  const float v = __uint_as_float(bf16_bits << 16) * inv;
  return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

}  // namespace moe_fp4
