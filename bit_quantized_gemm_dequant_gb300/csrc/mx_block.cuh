// MXFP4 block arithmetic shared by the standalone quantizer and the GEMM that
// quantizes its A operand itself.
//
// "量化推理引擎中的微缩放格式前瞻：MXFP4 矩阵乘法 Kernel 原理", §三
// (pack_tensor_to_mxfp4_layout): per 32-element block, amax clamped at 1e-8,
// e = ceil(log2(amax / 6)), v = x / 2^e, nearest E2M1 grid point with the
// first (smaller) one on a tie; the scale byte is the biased exponent e + 127.
#pragma once

#include <cstdint>

namespace wq {

// Block exponent e = ceil(log2(q)) with q = amax / 6 rounded to FP32, read off
// amax's own bits (amax already clamped to >= 1e-8).  With amax = m 2^E
// (1 <= m < 2): amax / 6 = (m / 1.5) 2^(E-2), and m / 1.5 lies in (1, 4/3)
// when m > 1.5 (e = E - 1) and in [2/3, 1] otherwise (e = E - 2).  Rounding
// m / 1.5 to FP32 never lands on 1 from either side except at m = 1.5 itself,
// so e = E - 2 + [m > 1.5].  amax and q are normal because amax >= 1e-8.
// (Equal to the rounded quotient's ceil(log2) for every mantissa, checked
// exhaustively.)
__device__ __forceinline__ int mx_block_exponent(float amax) {
  const uint32_t ab = __float_as_uint(amax);
  return static_cast<int>(ab >> 23) - 129 + ((ab & 0x7FFFFFu) > 0x400000u);
}

// 2^-e as a float (exact: |e| stays well inside the normal range here).
__device__ __forceinline__ float mx_inv_scale(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

__device__ __forceinline__ uint32_t e2m1_code(float x, float inv_scale) {
  // v = x * 2^-e is exact (a power-of-two scaling) and |v| <= 6.  The index
  // of the nearest grid point, the smaller one on a tie (the first index of
  // the argmin), is the number of grid midpoints strictly below |v|:
  //   |v| >= 1: the grid is every float with one mantissa bit from 1 to 6.
  //             Adding just under half a unit of that bit (2^21 - 1) and
  //             truncating rounds to nearest with ties to the smaller
  //             magnitude; the index is 2 * (unbiased exponent + 1) plus the
  //             kept mantissa bit, i.e. (bits >> 22) - 252.
  //   |v| < 1:  the grid is 0, 0.5, 1, with midpoints 0.25 and 0.75.
  // Non-negative float bits compare like the floats.  This equals counting
  // the seven midpoints (0.25 .. 5) one by one for every float32 in [0, 6].
  const uint32_t a = __float_as_uint(x * inv_scale) & 0x7FFFFFFFu;
  const uint32_t big = ((a + 0x1FFFFFu) >> 22) - 252u;
  const uint32_t small = (a > 0x3E800000u) + (a > 0x3F400000u);  // 0.25f, 0.75f
  const uint32_t j = a >= 0x3F800000u ? big : small;              // 1.0f
  return (x < 0.0f ? 8u : 0u) | j;
}

// Eight elements (one thread's quarter of a block) -> eight packed codes.
__device__ __forceinline__ uint32_t e2m1_word(const float (&xs)[8], float inv_scale) {
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) word |= e2m1_code(xs[i], inv_scale) << (4 * i);
  return word;
}

}  // namespace wq
