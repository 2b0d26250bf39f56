// MXFP8 encoding helpers shared by the quantizers and the fused quantization in
// the FP8 gate/up GEMM's epilogue: E4M3 elements, one power-of-two scale per 32
// consecutive elements along K stored as an 8-bit biased exponent, and the
// 512-byte scale atoms the tensor cores' block-scaled MMA reads (xtuner PR
// "Decouple expert parallelism from FSDP sharding (dp2ep layout)", "Changes":
// tile-wise scaled Float8; the format is the OCP microscaling MXFP8).
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

// X = floor(log2(amax)) - 8 (E4M3's largest exponent), clamped to [-127, 127];
// -127 for an all-zero block.
__device__ __forceinline__ int mx_exponent(float amax) {
  if (!(amax > 0.f)) return -127;
  int ex;
  frexpf(amax, &ex);                        // amax = m * 2^ex, m in [0.5, 1)
  int X = (ex - 1) - 8;                     // floor(log2 amax) - E4M3's largest exponent
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// 2^-X as a float (X in [-127, 126]: the result is a normal float).
__device__ __forceinline__ float inv_pow2(int X) { return __int_as_float((127 - X) << 23); }

// Four values to E4M3 (round to nearest even, saturating at 448), packed.
__device__ __forceinline__ uint32_t to_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// Byte of row r's j-th K32 scale in a 512-byte atom of 128 rows x 4 scales.
__device__ __forceinline__ size_t atom_byte(long long atom, int r, int j) {
  return static_cast<size_t>(atom) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

}  // namespace moe
