// NVFP4 quantizer: FP32 rows -> 16-element E2M1 blocks, E4M3 block scales and
// one FP32 tensor scale.
//
// The format is the one "Triton 工业级融合微算子编写：W4A16 极速切片矩阵乘与
// Blackwell NVFP4 硬件指令实装" §三 names: E2M1 elements under a two-level
// block scaling with an FP8 local scale, executed natively by the tensor
// cores.  The page gives no block size or encoding; the reading implemented
// here is 16-element blocks, scale s = e4m3(amax_block / (6 g)) (round to
// nearest even, saturating at 448) and tensor scale g = amax_tensor / 2688,
// with each element the nearest E2M1 grid point to x / (s g), the smaller one
// on a tie ("量化推理引擎中的微缩放格式前瞻：MXFP4 矩阵乘法 Kernel 原理" §三
// chooses its elements that way).  Every division and product is a single
// IEEE float32 operation rounded to nearest, so the bytes match a float32
// restatement of those steps exactly.
//
// Three launches on the stream: the tensor amax (an atomic max over the
// float bits, kept in the tensor-scale word), the quantization (which reads
// it), and a one-thread step that turns the amax into g.  HBM-bound: the
// source is read twice (4 + 4 B per element) and 0.5 + 1/16 B written.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kThreads = 256;  // one float4 per thread, four threads per 16-element block
constexpr float kScaleRange = 2688.0f;  // 6 (largest E2M1) x 448 (largest E4M3)

__device__ __forceinline__ float4 load4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ float amax4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// Tensor amax: the largest |x| over the rows [row0, row0 + gridDim.y); the
// non-negative float bits order like the floats, so an integer atomic max
// over them is a float max.
__global__ void __launch_bounds__(kThreads)
nv_amax_kernel(NvQuantArgs p, int row0) {
  const int r = row0 + blockIdx.y;
  const int c4 = blockIdx.x * kThreads + threadIdx.x;
  float m = 0.0f;
  if (c4 < p.cols / 4) m = amax4(load4(p.src + static_cast<int64_t>(r) * p.ld_src + 4 * c4));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0 && m > 0.0f)
    atomicMax(reinterpret_cast<unsigned int*>(p.tensor_scale), __float_as_uint(m));
}

// g from the amax the first kernel left in the tensor-scale word.
__device__ __forceinline__ float tensor_scale_of(float amax) {
  return amax > 0.0f ? __fdiv_rn(amax, kScaleRange) : 1.0f;
}

// Index of the nearest E2M1 grid point to |v|, the smaller one on a tie: the
// number of grid midpoints (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) strictly
// below |v|.  |v| can exceed 6 when the block scale was rounded down; it
// still maps to 6.
__device__ __forceinline__ uint32_t e2m1_index(float v) {
  const float a = fabsf(v);
  return (a > 0.25f) + (a > 0.75f) + (a > 1.25f) + (a > 1.75f) + (a > 2.5f) + (a > 3.5f) + (a > 5.0f);
}

__global__ void __launch_bounds__(kThreads)
nv_quantize_kernel(NvQuantArgs p, int row0) {
  const int r = row0 + blockIdx.y;
  const int c4 = blockIdx.x * kThreads + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool live = c4 < p.cols / 4;  // cols is a multiple of 16: a block is live or dead as a whole
  const float4 x = live ? load4(p.src + static_cast<int64_t>(r) * p.ld_src + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
  float m = amax4(x);
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));  // the block's amax in all four lanes
  const float g = tensor_scale_of(__uint_as_float(*reinterpret_cast<const unsigned int*>(p.tensor_scale)));
  const float sb_f = __fdiv_rn(m, __fmul_rn(6.0f, g));
  const __nv_fp8_storage_t sb = __nv_cvt_float_to_fp8(sb_f, __NV_SATFINITE, __NV_E4M3);
  const float d = __fmul_rn(__half2float(__half(__nv_cvt_fp8_to_halfraw(sb, __NV_E4M3))), g);
  uint32_t codes = 0;
  if (d > 0.0f) {
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      codes |= ((xs[i] < 0.0f ? 8u : 0u) | e2m1_index(__fdiv_rn(xs[i], d))) << (4 * i);
  }
  // Lane 4k gathers the block's four 16-bit code groups into 8 bytes.
  const uint32_t pair = codes | (__shfl_down_sync(0xffffffffu, codes, 1) << 16);
  const uint32_t pair_hi = __shfl_down_sync(0xffffffffu, pair, 2);
  if (live && (lane & 3) == 0) {
    *reinterpret_cast<uint2*>(p.data + static_cast<int64_t>(r) * p.ld_data + 2 * c4) = make_uint2(pair, pair_hi);
    p.scales[static_cast<int64_t>(r) * p.ld_scales + c4 / 4] = sb;
  }
}

__global__ void nv_tensor_scale_kernel(float* tensor_scale) {
  *tensor_scale = tensor_scale_of(__uint_as_float(*reinterpret_cast<const unsigned int*>(tensor_scale)));
}

}  // namespace

cudaError_t launch_nv_quantize(const NvQuantArgs& a, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(a.tensor_scale, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  const int cx = (a.cols / 4 + kThreads - 1) / kThreads;
  if (a.rows > 0 && a.cols > 0) {
    for (int r0 = 0; r0 < a.rows; r0 += 65535) {  // grid y is at most 65535 rows per launch
      const int n = a.rows - r0 < 65535 ? a.rows - r0 : 65535;
      nv_amax_kernel<<<dim3(cx, n), kThreads, 0, s>>>(a, r0);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    for (int r0 = 0; r0 < a.rows; r0 += 65535) {
      const int n = a.rows - r0 < 65535 ? a.rows - r0 : 65535;
      nv_quantize_kernel<<<dim3(cx, n), kThreads, 0, s>>>(a, r0);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  nv_tensor_scale_kernel<<<1, 1, 0, s>>>(a.tensor_scale);
  return cudaGetLastError();
}

}  // namespace wq
