// FP4 block scales: row-major bytes -> the tensor cores' chunk layout.
//
// The block-scaled MMAs ("量化推理引擎中的微缩放格式前瞻：MXFP4 矩阵乘法 Kernel
// 原理" §二.1-§二.2: one scale per 32-element E2M1 block, the exponents added
// inside the dot product; NVFP4 as read from "W4A16 量化" §三: one E4M3 scale
// per 16 elements) take their scales from tensor memory, which
// tcgen05.cp 32x128b.warpx4 fills from 512-byte shared-memory chunks of 128
// rows x 4 scale bytes.  With the scales already in that order in global
// memory, the GEMMs move them with plain bulk copies and start the MMAs as
// soon as a stage lands.  The layout is defined beside tc_sf_chunks.
//
// One CTA of 128 threads per (row group of 128 rows, four chunks): thread r
// reads 16 scale bytes of row r (one 128-bit load when aligned and in range,
// else byte loads with the padding value outside the matrix), and after a
// shared-memory exchange writes line r % 32 of chunk r / 32, four rows' words
// gathered into one 16-byte store; a warp stores one whole chunk.
#include "tc_common.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

__global__ void __launch_bounds__(128)
fp4_scales_tc_kernel(const uint8_t* __restrict__ S, int64_t lds, int rows, int nb, uint8_t* __restrict__ out,
                     int chunks, uint32_t fill) {
  __shared__ uint32_t tile[128][5];  // 4 words per row; stride 5 keeps the gathers conflict-free
  tc::griddep_launch_dependents();
  tc::griddep_wait();  // S may come from the kernel before this one
  const int r = threadIdx.x, g = blockIdx.y, c0 = 4 * blockIdx.x;
  const int row = g * 128 + r, b0 = 4 * c0;  // 16 blocks from b0
  uint32_t w[4] = {fill, fill, fill, fill};
  if (row < rows && b0 < nb) {
    const uint8_t* p = S + static_cast<int64_t>(row) * lds + b0;
    if (b0 + 16 <= nb && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
      w[0] = v.x;
      w[1] = v.y;
      w[2] = v.z;
      w[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (b0 + i < nb) {
          const int sh = 8 * (i & 3);
          w[i >> 2] = (w[i >> 2] & ~(0xFFu << sh)) | (static_cast<uint32_t>(__ldg(p + i)) << sh);
        }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) tile[r][j] = w[j];
  __syncthreads();
  const int j = r >> 5, l = r & 31;
  if (c0 + j < chunks) {
    const uint4 o = make_uint4(tile[l][j], tile[l + 32][j], tile[l + 64][j], tile[l + 96][j]);
    *reinterpret_cast<uint4*>(out + (static_cast<int64_t>(g) * chunks + c0 + j) * kTcSfChunk + 16 * l) = o;
  }
}

}  // namespace

cudaError_t launch_fp4_scales_tc(bool nv, int rows, int K, const uint8_t* S, int64_t lds, uint8_t* out,
                                 cudaStream_t s) {
  const int chunks = tc_sf_chunks(nv, K);
  const int groups = (rows + 255) / 256 * 2;
  if (chunks == 0 || groups == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((chunks + 3) / 4, groups);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fp4_scales_tc_kernel, S, lds, rows, K / (nv ? 16 : 32), out, chunks,
                                           nv ? 0u : 0x7F7F7F7Fu);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace wq
