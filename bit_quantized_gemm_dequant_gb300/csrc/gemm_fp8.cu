// FP8 e4m3 GEMM with per-tensor scales on the 5th-generation tensor cores.
//
// Defined by "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核" (kernel listing
// and the 精度管理 bullet): e4m3fn A [M, K] and B [K, N], FP32 accumulation,
// the per-tensor scales applied once to the accumulator, BF16 output.
//
// Design: one 128 x 256 output tile per CTA, K in 128-byte steps.
//   warp 0      TMA producer: A box 128(k) x 128(m) and two B boxes
//               128(n) x 128(k), 128-byte swizzle, into a 4-stage ring.
//   warp 1      TMEM allocator and MMA issuer: per stage, 4 K-steps x two
//               tcgen05.mma.kind::f8f6f4 of 128 x 128 x 32 (A K-major, B
//               MN-major straight from the [K, N] layout, no transpose pass),
//               accumulating into 256 TMEM columns; tcgen05.commit frees the
//               stage, and a last commit hands the accumulator over.
//   warps 2-5   epilogue: tcgen05.ld of their 32-lane quarter, scale, round to
//               BF16 and store.
// The page's Ada/Hopper tiles (128 x 64 x 32, multicast TMA) are not used:
// each CTA loads its own tiles.
#include <cuda_bf16.h>

#include "tc_common.cuh"
#include "tma_host.h"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK;             // 16 KB
constexpr int kBHalfBytes = 128 * BK;        // 16 KB: 128 n x 128 k
constexpr int kStageBytes = kABytes + 2 * kBHalfBytes;
constexpr int kTmemCols = 256;
constexpr int kThreads = 192;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /* barriers */ + 1024 /* alignment slack */;

__global__ void __launch_bounds__(kThreads, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, Fp8GemmArgs p,
                int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* accum = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int KT = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(accum, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tmA);
    tc::tma_prefetch_desc(&tmB);
    int issued = 0;
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % kStages;
      if (!tc::mbar_wait(&empty[s], ((kt / kStages) & 1) ^ 1, abort, err, kSiteGemmProducer)) break;
      uint8_t* st = smem + s * kStageBytes;
      tc::mbar_arrive_expect_tx(&full[s], kStageBytes);
      tc::tma_load_2d(st, &tmA, kt * BK, m0, &full[s]);
      tc::tma_load_2d(st + kABytes, &tmB, n0, kt * BK, &full[s]);
      tc::tma_load_2d(st + kABytes + kBHalfBytes, &tmB, n0 + 128, kt * BK, &full[s]);
      issued = kt + 1;
    }
    if (*abort) {  // let the copies already issued land before the CTA exits
      for (int kt = issued > kStages ? issued - kStages : 0; kt < issued; ++kt)
        tc::mbar_wait_drain(&full[kt % kStages], (kt / kStages) & 1);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = tc::idesc_dense(/*E4M3*/ 0, /*E4M3*/ 0, /*A K-major*/ 0, /*B MN-major*/ 1, 128, 128);
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % kStages;
      if (!tc::mbar_wait(&full[s], (kt / kStages) & 1, abort, err, kSiteGemmMma)) break;
      tc::tc_fence_after();
      const uint32_t a = tc::smem_u32(smem + s * kStageBytes);
      const uint32_t b = a + kABytes;
#pragma unroll
      for (int j = 0; j < BK / 32; ++j) {
        const uint64_t adesc = tc::smem_desc(a + 32 * j, 1024, 1024, tc::kSwizzle128B);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t bdesc = tc::smem_desc(b + h * kBHalfBytes + 32 * 128 * j, 1024, 1024, tc::kSwizzle128B);
          tc::mma_f8f6f4(tmem + 128 * h, adesc, bdesc, idesc, (kt | j) != 0);
        }
      }
      tc::tc_commit(&empty[s]);
    }
    tc::tc_commit(accum);  // arrives once every MMA above has completed
  } else if (warp >= 2) {
    const bool ok = tc::mbar_wait(accum, 0, abort, err, kSiteGemmEpilogue);
    tc::tc_fence_after();
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = m0 + 32 * q + lane;
    const float scale = p.scale_a * p.scale_b;
    __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C);
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tc::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + 32 * c, r);
      tc::tmem_ld_wait();
      if (!ok || row >= p.M) continue;
      const int col0 = n0 + 32 * c;
      __nv_bfloat16* dst = C + static_cast<int64_t>(row) * p.ldc + col0;
      if (col0 + 32 <= p.N) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t pk[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[8 * v + 2 * t]) * scale,
                                                            __uint_as_float(r[8 * v + 2 * t + 1]) * scale);
            pk[t] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(dst + 8 * v) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      } else {
        for (int t = 0; t < 32 && col0 + t < p.N; ++t) dst[t] = __float2bfloat16_rn(__uint_as_float(r[t]) * scale);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_fp8_gemm(const Fp8GemmArgs& a, cudaStream_t s) {
  if (a.K == 0)
    return cudaMemset2DAsync(a.C, a.ldc * 2, 0, static_cast<size_t>(a.N) * 2, a.M, s);
  CUtensorMap tA, tB;
  cudaError_t e = make_tmap_2d(&tA, a.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.K, a.M, a.lda, BK, BM,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&tB, a.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, a.K, a.ldb, 128, BK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  static bool configured = false;
  if (!configured) {
    e = cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM);
  fp8_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(tA, tB, a, device_error_word());
  return cudaGetLastError();
}

}  // namespace wq
