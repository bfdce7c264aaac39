// MXFP4 quantizer: FP32 rows -> 32-element E2M1 blocks + E8M0 scales.
//
// Defined by "量化推理引擎中的微缩放格式前瞻：MXFP4 矩阵乘法 Kernel 原理", §三
// (pack_tensor_to_mxfp4_layout): per 32-element block, amax clamped at 1e-8,
// e = ceil(log2(amax / 6)), v = x / 2^e, nearest E2M1 grid point with the
// first (smaller) one on a tie.  §一: data and scale segments are separate.
//
// HBM-bound: 4 B read + 0.5 B + 1/32 B written per element.  Four threads
// own one block: each loads 32 contiguous bytes (two 128-bit loads), the
// block amax is a 4-lane shuffle max, and each thread stores one 32-bit word
// of packed codes, so a warp reads 1 KB and writes 128 B contiguously.
#include "mx_block.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // blocks in flight per thread quad

// Element offsets of 32-element block `item` in the source, data and scale
// arrays.  kDense: rows are packed back to back (every leading dimension is
// the row length), so the block index alone gives them; otherwise the row is
// found with a 32-bit division (the launcher keeps block counts below 2^31).
template <bool kDense>
__device__ __forceinline__ void block_offsets(const MxQuantArgs& p, uint32_t blocks_per_row, uint32_t item,
                                              int64_t& src, int64_t& data, int64_t& sc) {
  if (kDense) {
    src = static_cast<int64_t>(item) * 32;
    data = static_cast<int64_t>(item) * 16;
    sc = item;
  } else {
    const uint32_t r = item / blocks_per_row, b = item - r * blocks_per_row;
    src = static_cast<int64_t>(r) * p.ld_src + b * 32;
    data = static_cast<int64_t>(r) * p.ld_data + b * 16;
    sc = static_cast<int64_t>(r) * p.ld_scales + b;
  }
}

template <bool kDense>
__global__ void __launch_bounds__(kThreads, 3)
mx_quantize_kernel(MxQuantArgs p, uint32_t n_items) {
  // A warp owns 8 consecutive blocks (1 KB of source) per step; the loop
  // bound is warp-uniform so that every lane reaches the quad shuffles.
  const int lane = threadIdx.x & 31;
  const int quad_lane = lane & 3;
  const uint32_t blocks_per_row = static_cast<uint32_t>(p.cols / 32);
  const uint32_t warp0 = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t step = ((gridDim.x * kThreads) >> 5) * 8;

  for (uint32_t base = warp0 * 8; base < n_items; base += step * kUnroll) {
    float4 v[kUnroll][2];
    int64_t src[kUnroll], data[kUnroll], sc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t item = base + u * step + (lane >> 2);
      if (item < n_items) {
        block_offsets<kDense>(p, blocks_per_row, item, src[u], data[u], sc[u]);
        const float4* ps = reinterpret_cast<const float4*>(p.src + src[u] + quad_lane * 8);
        v[u][0] = __ldcs(ps);
        v[u][1] = __ldcs(ps + 1);
      } else {
        src[u] = -1;
        v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float xs[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                           v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(xs[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      amax = fmaxf(amax, 1e-8f);
      const int e = mx_block_exponent(amax);
      const uint32_t word = e2m1_word(xs, mx_inv_scale(e));
      if (src[u] >= 0) {
        __stcs(reinterpret_cast<unsigned int*>(p.data + data[u] + quad_lane * 4), word);
        if (quad_lane == 0) p.scales[sc[u]] = static_cast<uint8_t>(e + 127);
      }
    }
  }
}

}  // namespace

cudaError_t launch_mx_quantize(const MxQuantArgs& a, cudaStream_t s) {
  const int64_t n_items = static_cast<int64_t>(a.rows) * (a.cols / 32);
  if (n_items == 0) return cudaSuccess;
  // 32-bit block indices: under 2^31 blocks (a 256 GB source) the loop
  // counter cannot wrap.
  if (n_items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int64_t blocks_per_cta = kThreads / 4;  // one 32-element block per thread quad
  int64_t ctas = (n_items + blocks_per_cta * kUnroll - 1) / (blocks_per_cta * kUnroll);
  const bool dense = a.ld_src == a.cols && a.ld_data == a.cols / 2 && a.ld_scales == a.cols / 32;
  auto kern = dense ? mx_quantize_kernel<true> : mx_quantize_kernel<false>;
  // One wave of as many CTAs as the SMs hold at once (registers decide: at
  // least 3 by the launch bounds).
  static PerDevice<int> per_sm[2];
  int n = 3;  // the launch bounds' minimum, if the query fails
  per_sm[dense].get(n, [&](int& v) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kThreads, 0) == cudaSuccess && v >= 1;
  });
  const int64_t cap = static_cast<int64_t>(sm_count()) * n;
  if (ctas > cap) ctas = cap;
  kern<<<static_cast<unsigned>(ctas), kThreads, 0, s>>>(a, static_cast<uint32_t>(n_items));
  return cudaGetLastError();
}

}  // namespace wq
