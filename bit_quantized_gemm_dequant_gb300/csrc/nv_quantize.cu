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
// Three launches on the stream after zeroing the tensor-scale word: the
// tensor amax (kept in that word), the quantization (which reads it), and a
// one-thread step that turns the amax into g.  HBM-bound: the
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

// Tensor amax.  Each block takes one 1024-column slice of every gridDim.y-th
// row (four rows in flight per thread), reduces in shared memory and makes
// one atomic max on the tensor-scale word: non-negative float bits order like
// the floats, so an integer max over them is a float max.  Plain cached loads,
// so that an operand that fits in L2 is still there for the second pass.
constexpr int kAmaxRowsInFlight = 4;

__global__ void __launch_bounds__(kThreads)
nv_amax_kernel(NvQuantArgs p) {
  const int c4 = blockIdx.x * kThreads + threadIdx.x;
  float m = 0.0f;
  if (c4 < p.cols / 4) {
    const float* col = p.src + 4 * static_cast<int64_t>(c4);
    const int step = gridDim.y;
    int r = blockIdx.y;
    for (; r + (kAmaxRowsInFlight - 1) * step < p.rows; r += kAmaxRowsInFlight * step) {
      float4 v[kAmaxRowsInFlight];
#pragma unroll
      for (int i = 0; i < kAmaxRowsInFlight; ++i)
        v[i] = __ldg(reinterpret_cast<const float4*>(col + static_cast<int64_t>(r + i * step) * p.ld_src));
#pragma unroll
      for (int i = 0; i < kAmaxRowsInFlight; ++i) m = fmaxf(m, amax4(v[i]));
    }
    for (; r < p.rows; r += step)
      m = fmaxf(m, amax4(__ldg(reinterpret_cast<const float4*>(col + static_cast<int64_t>(r) * p.ld_src))));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float warp_max[kThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, warp_max[w]);
    if (m > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(p.tensor_scale), __float_as_uint(m));
  }
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

// The same index for v = RN(a / d) (a >= 0, d > 0), without the division.
// Each midpoint t has at most three significant bits and an even last
// mantissa bit, so RN(a/d) > t exactly when a/d exceeds t + ulp(t)/2 (a tie
// rounds to the even t), i.e. when a - t*d > h*d with h = ulp(t)/2, a power
// of two.  The FMA forms a - t*d exactly where it matters: when
// |a - t*d| <= 4h*d the difference is a multiple of 2^-25 * 2^(e_t + e_d)
// below 2^-21 * 2^(e_t + e_d), at most four significant bits; beyond that,
// rounding cannot carry it across h*d.  h*d is exact while d >= 2^-100 (the
// caller divides otherwise).  Three comparisons, a binary search over the
// seven midpoints.  hd[i] = h_i * d.
__device__ __forceinline__ uint32_t e2m1_index_quotient(float a, float d, const float (&hd)[7]) {
  const bool b2 = __fmaf_rn(-1.75f, d, a) > hd[3];
  const float t1 = b2 ? 3.5f : 0.75f, h1 = b2 ? hd[5] : hd[1];
  const bool b1 = __fmaf_rn(-t1, d, a) > h1;
  const float t0 = b2 ? (b1 ? 5.0f : 2.5f) : (b1 ? 1.25f : 0.25f);
  const float h0 = b2 ? (b1 ? hd[6] : hd[4]) : (b1 ? hd[2] : hd[0]);
  const bool b0 = __fmaf_rn(-t0, d, a) > h0;
  return (b2 ? 4u : 0u) + (b1 ? 2u : 0u) + (b0 ? 1u : 0u);
}

// One 16-element block per four lanes: the block amax by two shuffles, the
// E4M3 scale, then each lane's four codes.  Lane 4k gathers the block's four
// 16-bit code groups into 8 bytes.
__device__ __forceinline__ void quantize_row4(const NvQuantArgs& p, int r, int c4, bool live, float4 x, float g,
                                              int lane) {
  float m = amax4(x);
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));  // the block's amax in all four lanes
  const float sb_f = __fdiv_rn(m, __fmul_rn(6.0f, g));
  const __nv_fp8_storage_t sb = __nv_cvt_float_to_fp8(sb_f, __NV_SATFINITE, __NV_E4M3);
  const float d = __fmul_rn(__half2float(__half(__nv_cvt_fp8_to_halfraw(sb, __NV_E4M3))), g);
  uint32_t codes = 0;
  const float xs[4] = {x.x, x.y, x.z, x.w};
  if (d >= 0x1p-100f) {
    // ulp(t)/2 of the midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, times d.
    const float hd[7] = {d * 0x1p-26f, d * 0x1p-25f, d * 0x1p-24f, d * 0x1p-24f, d * 0x1p-23f, d * 0x1p-23f,
                         d * 0x1p-22f};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      codes |= ((xs[i] < 0.0f ? 8u : 0u) | e2m1_index_quotient(fabsf(xs[i]), d, hd)) << (4 * i);
  } else if (d > 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      codes |= ((xs[i] < 0.0f ? 8u : 0u) | e2m1_index(__fdiv_rn(xs[i], d))) << (4 * i);
  }
  const uint32_t pair = codes | (__shfl_down_sync(0xffffffffu, codes, 1) << 16);
  const uint32_t pair_hi = __shfl_down_sync(0xffffffffu, pair, 2);
  if (live && (lane & 3) == 0) {
    *reinterpret_cast<uint2*>(p.data + static_cast<int64_t>(r) * p.ld_data + 2 * c4) = make_uint2(pair, pair_hi);
    p.scales[static_cast<int64_t>(r) * p.ld_scales + c4 / 4] = sb;
  }
}

// Each block takes one 1024-column slice of every gridDim.y-th row, loading
// four rows before quantizing them.  The columns past the matrix are whole
// dead blocks (cols is a multiple of 16): they quantize zeros and store
// nothing, but still take part in the shuffles.
constexpr int kQuantRowsInFlight = 4;

__global__ void __launch_bounds__(kThreads)
nv_quantize_kernel(NvQuantArgs p) {
  const int c4 = blockIdx.x * kThreads + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool live = c4 < p.cols / 4;
  const float g = tensor_scale_of(__uint_as_float(*reinterpret_cast<const unsigned int*>(p.tensor_scale)));
  const float* col = p.src + 4 * static_cast<int64_t>(c4);
  const int step = gridDim.y;
  int r = blockIdx.y;
  for (; r + (kQuantRowsInFlight - 1) * step < p.rows; r += kQuantRowsInFlight * step) {
    float4 x[kQuantRowsInFlight];
#pragma unroll
    for (int i = 0; i < kQuantRowsInFlight; ++i)
      x[i] = live ? load4(col + static_cast<int64_t>(r + i * step) * p.ld_src) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kQuantRowsInFlight; ++i) quantize_row4(p, r + i * step, c4, live, x[i], g, lane);
  }
  for (; r < p.rows; r += step) {
    const float4 x = live ? load4(col + static_cast<int64_t>(r) * p.ld_src) : make_float4(0.f, 0.f, 0.f, 0.f);
    quantize_row4(p, r, c4, live, x, g, lane);
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
    // About 16 blocks per SM in each pass; each strides over the rows.
    int ry = (sm_count() * 16 + cx - 1) / cx;
    ry = ry < a.rows ? ry : a.rows;
    nv_amax_kernel<<<dim3(cx, ry), kThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    nv_quantize_kernel<<<dim3(cx, ry), kThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  nv_tensor_scale_kernel<<<1, 1, 0, s>>>(a.tensor_scale);
  return cudaGetLastError();
}

}  // namespace wq
