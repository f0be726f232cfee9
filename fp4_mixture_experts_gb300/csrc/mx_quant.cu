// MXFP8 quantisation of bf16 rows, the activation operand of a block-scaled
// tensor-core product (E4M3 elements, one E8M0 scale per 32 elements along
// the row, OCP Microscaling v1.0 conversion).
//
// One thread per 32-element block: four 16-byte loads, the block's largest
// magnitude from the bf16 bit patterns (with the sign bit cleared, bit order
// is magnitude order), its exponent minus 8 (the largest E4M3 exponent) as
// the scale, then every element times the exact power of two 2^-scale goes
// through the CUDA fp8 conversion (round to nearest even, saturating at the
// largest finite E4M3); two 16-byte stores of codes and one scale byte.  A
// block holding an infinity or a NaN gets the NaN scale byte 0xFF and NaN
// codes (0x7F): its value is undefined, as the MX format has no other way to
// carry it.  The kernel is bound by HBM: 2 bytes read and 1 + 1/32 written
// per element.
#include <cuda_fp8.h>

#include "moe_fp4_internal.cuh"
#include "mx_common.cuh"

namespace moe_fp4 {
namespace {

__global__ void __launch_bounds__(256)
mxfp8_quantize_kernel(const uint4* __restrict__ x, long long n_blocks, uint4* __restrict__ codes,
                      uint8_t* __restrict__ scales) {
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < n_blocks;
       b += (long long)gridDim.x * blockDim.x) {
    uint32_t w[16];  // 32 bf16, two per word, the even element in the low half
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 q = x[4 * b + i];
      w[4 * i] = q.x;
      w[4 * i + 1] = q.y;
      w[4 * i + 2] = q.z;
      w[4 * i + 3] = q.w;
    }
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = max(amax, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    const uint32_t sb = mx_scale_byte(amax);
    if (sb == 0xFFu) {  // an infinity or a NaN in the block (bf16 exponent field all ones)
      const uint4 nan4 = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      codes[2 * b] = nan4;
      codes[2 * b + 1] = nan4;
      scales[b] = 0xFF;
      continue;
    }
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t a = w[2 * i], c = w[2 * i + 1];
      out[i] = mx_e4m3_code(a & 0xFFFFu, sb) | (mx_e4m3_code(a >> 16, sb) << 8) |
               (mx_e4m3_code(c & 0xFFFFu, sb) << 16) | (mx_e4m3_code(c >> 16, sb) << 24);
    }
    codes[2 * b] = make_uint4(out[0], out[1], out[2], out[3]);
    codes[2 * b + 1] = make_uint4(out[4], out[5], out[6], out[7]);
    scales[b] = (uint8_t)sb;
  }
}

}  // namespace

cudaError_t launch_mxfp8_quantize(const uint16_t* x, long long rows, int K, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t st) {
  const long long n_blocks = rows * (K / 32);
  if (n_blocks <= 0) return cudaSuccess;
  long long grid = (n_blocks + 255) / 256;
  const long long cap = (long long)num_sms() * 16;
  if (grid > cap) grid = cap;
  mxfp8_quantize_kernel<<<(unsigned)grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(x), n_blocks,
                                                        reinterpret_cast<uint4*>(codes), scales);
  return cudaGetLastError();
}

}  // namespace moe_fp4

extern "C" int moe_fp4_mxfp8_quantize(const void* x_bf16, int64_t rows, int32_t K, uint8_t* codes, uint8_t* scales,
                                      void* cuda_stream) {
  using namespace moe_fp4;
  if (rows < 0 || K <= 0 || K % 32 != 0) return MOE_FP4_ERR_INVALID_ARG;
  if (rows == 0) return MOE_FP4_OK;  // nothing to do; the pointers are not looked at
  if (!x_bf16 || !codes || !scales) return MOE_FP4_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x_bf16) & 15) || (reinterpret_cast<uintptr_t>(codes) & 15))
    return MOE_FP4_ERR_INVALID_ARG;
  return launch_mxfp8_quantize(static_cast<const uint16_t*>(x_bf16), (long long)rows, K, codes, scales,
                               static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
             ? MOE_FP4_OK
             : MOE_FP4_ERR_CUDA;
}
