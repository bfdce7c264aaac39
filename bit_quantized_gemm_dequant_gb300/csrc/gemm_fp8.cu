// FP8 e4m3 GEMM with per-tensor scales on the 5th-generation tensor cores.
//
// Defined by "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核" (kernel listing
// and the 精度管理 bullet): e4m3fn A [M, K] and B [K, N], FP32 accumulation,
// the per-tensor scales applied once to the accumulator, BF16 output.
//
// Design: a persistent kernel, one CTA per SM, output tiles of 128 x BN
// (BN = 256, or 128 when M is small so that more SMs share the weight
// stream) handed out round-robin; K in 128-byte steps.
//   warp 0      TMA producer: A box 128(k) x 128(m) and BN/128 B boxes
//               128(n) x 128(k), 128-byte swizzle, into a 4-stage ring that
//               runs continuously across the CTA's tiles.
//   warp 1      TMEM allocator and MMA issuer: per stage, 4 K-steps of one
//               tcgen05.mma.kind::f8f6f4 of 128 x BN x 32 (A K-major, B
//               MN-major straight from the [K, N] layout, no transpose pass)
//               into one of two TMEM accumulators; tcgen05.commit frees the
//               stage and, after the last K step, hands the accumulator over.
//   warps 2-5   epilogue: tcgen05.ld of their 32-lane quarter, scale, round to
//               BF16 and store, then release the accumulator — while the MMA
//               warp already fills the other one.
// The page's Ada/Hopper tiles (128 x 64 x 32, multicast TMA) are not used:
// each CTA loads its own tiles.
#include <cuda_bf16.h>

#include "tc_common.cuh"
#include "tma_host.h"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int BM = 128, BK = 128;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK;       // 16 KB
constexpr int kBHalfBytes = 128 * BK;  // 16 KB: 128 n x 128 k
constexpr int kThreads = 192;

template <int HALVES>
struct Fp8Cfg {
  static constexpr int BN = 128 * HALVES;
  static constexpr int kStageBytes = kABytes + HALVES * kBHalfBytes;
  static constexpr int kAccCols = BN;
  static constexpr int kTmemCols = 2 * BN;  // two accumulators
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 1024;
};

template <int HALVES>
__global__ void __launch_bounds__(kThreads, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, Fp8GemmArgs p,
                int* err) {
  using Cfg = Fp8Cfg<HALVES>;
  constexpr int BN = Cfg::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * Cfg::kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;   // [2] MMA -> epilogue
  uint64_t* acc_empty = acc_full + 2;     // [2] epilogue -> MMA
  uint64_t* drain = acc_empty + 2;        // MMAs in flight after a give-up
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (p.M + BM - 1) / BM;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int tiles = m_tiles * n_tiles;
  const int KT = (p.K + BK - 1) / BK;
  // Tile order: bands of kBand row tiles, M fastest within a band.  A round
  // of tiles then reads kBand row panels of A and a few column panels of B
  // (about 40 MB at 8192^3) instead of every row panel of A (64 MB), which
  // L2 could not keep while C streams out.
  constexpr int kBand = 32;
  auto band_rows = [&](int t) {
    const int m_base = t / (kBand * n_tiles) * kBand;
    return m_tiles - m_base < kBand ? m_tiles - m_base : kBand;
  };
  auto tile_m = [&](int t) {
    const int b = t / (kBand * n_tiles);
    return b * kBand + (t - b * kBand * n_tiles) % band_rows(t);
  };
  auto tile_n = [&](int t) { return (t - t / (kBand * n_tiles) * kBand * n_tiles) / band_rows(t); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    tc::mbar_init(drain, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  tc::cta_barrier();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Tile t -> (tile_m(t), tile_n(t)): consecutive tiles walk down M within a
  // band, so the CTAs running at the same time share B columns.
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tmA);
    tc::tma_prefetch_desc(&tmB);
    int it = 0, issued = 0;
    for (int t = blockIdx.x; t < tiles && !*abort; t += gridDim.x) {
      const int m0 = tile_m(t) * BM, n0 = tile_n(t) * BN;
      for (int kt = 0; kt < KT; ++kt, ++it) {
        const int s = it % kStages;
        if (!tc::mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, abort, err, kSiteGemmProducer)) break;
        uint8_t* st = smem + s * Cfg::kStageBytes;
        tc::mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
        tc::tma_load_2d(st, &tmA, kt * BK, m0, &full[s]);
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
          tc::tma_load_2d(st + kABytes + h * kBHalfBytes, &tmB, n0 + 128 * h, kt * BK, &full[s]);
        issued = it + 1;
      }
    }
    if (*abort)  // let the copies already issued land before the CTA exits
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        tc::mbar_wait_drain(&full[i % kStages], (i / kStages) & 1);
  } else if (warp == 1 && lane == 0) {
    // One 128 x BN x 32 MMA per K slice: A is read once per slice.  B is
    // MN-major: its BN / 128 swizzle atoms along N are the B boxes, kBHalfBytes
    // apart (the descriptor's leading byte offset); 8-row K groups are 1 KB
    // apart (stride byte offset).
    constexpr uint32_t idesc = tc::idesc_dense(/*E4M3*/ 0, /*E4M3*/ 0, /*A K-major*/ 0, /*B MN-major*/ 1, 128, BN);
    int it = 0, local = 0;
    for (int t = blockIdx.x; t < tiles && !*abort; t += gridDim.x, ++local) {
      const int buf = local & 1;
      if (!tc::mbar_wait(&acc_empty[buf], ((local >> 1) & 1) ^ 1, abort, err, kSiteGemmTmemFree)) break;
      tc::tc_fence_after();
      const uint32_t acc = tmem + buf * Cfg::kAccCols;
      bool ok = true;
      for (int kt = 0; kt < KT; ++kt, ++it) {
        const int s = it % kStages;
        if (!tc::mbar_wait(&full[s], (it / kStages) & 1, abort, err, kSiteGemmMma)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t a = tc::smem_u32(smem + s * Cfg::kStageBytes);
        const uint32_t b = a + kABytes;
#pragma unroll
        for (int j = 0; j < BK / 32; ++j) {
          const uint64_t adesc = tc::smem_desc(a + 32 * j, 1024, 1024, tc::kSwizzle128B);
          const uint64_t bdesc = tc::smem_desc(b + 32 * 128 * j, kBHalfBytes, 1024, tc::kSwizzle128B);
          tc::mma_f8f6f4(acc, adesc, bdesc, idesc, (kt | j) != 0);
        }
        tc::tc_commit(&empty[s]);
      }
      if (!ok) break;
      tc::tc_commit(&acc_full[buf]);  // arrives once every MMA of the tile has completed
    }
    // After a give-up: wait (bounded) until every MMA issued so far has
    // completed, so that none still writes TMEM when it is freed.
    if (*abort) {
      tc::tc_commit(drain);
      tc::mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 2) {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const float scale = p.scale_a * p.scale_b;
    __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C);
    int local = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++local) {
      const int buf = local & 1;
      const bool ok = tc::mbar_wait(&acc_full[buf], (local >> 1) & 1, abort, err, kSiteGemmEpilogue);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::tc_fence_after();
      const int m0 = tile_m(t) * BM, n0 = tile_n(t) * BN;
      const int row = m0 + 32 * q + lane;
      const uint32_t acc = tmem + buf * Cfg::kAccCols + (static_cast<uint32_t>(32 * q) << 16);
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(acc + 32 * c, r);
        tc::tmem_ld_wait();
        if (c == BN / 32 - 1) {  // accumulator fully read: hand it back to the MMA warp
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
        }
        if (row >= p.M) continue;
        const int col0 = n0 + 32 * c;
        __nv_bfloat16* dst = C + static_cast<int64_t>(row) * p.ldc + col0;
        if (col0 + 32 <= p.N) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t pk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[8 * v + 2 * u]) * scale,
                                                              __uint_as_float(r[8 * v + 2 * u + 1]) * scale);
              pk[u] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(dst + 8 * v) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u)
            if (col0 + u < p.N) dst[u] = __float2bfloat16_rn(__uint_as_float(r[u]) * scale);
        }
      }
    }
  }
  tc::tc_fence_before();
  tc::cta_barrier();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <int HALVES>
cudaError_t launch_variant(const Fp8GemmArgs& a, cudaStream_t s) {
  using Cfg = Fp8Cfg<HALVES>;
  CUtensorMap tA, tB;
  cudaError_t e = make_tmap_2d(&tA, a.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.K, a.M, a.lda, BK, BM,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&tB, a.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, a.K, a.ldb, 128, BK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  auto kern = fp8_gemm_kernel<HALVES>;
  static PerDevice<bool> configured;
  bool done = false;
  if (!configured.get(done, [&](bool& v) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
        v = true;
        return e == cudaSuccess;
      }))
    return e;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + Cfg::BN - 1) / Cfg::BN);
  const int grid = tiles < sm_count() ? tiles : sm_count();
  kern<<<grid, kThreads, Cfg::kSmemBytes, s>>>(tA, tB, a, device_error_word());
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_gemm(const Fp8GemmArgs& a, cudaStream_t s) {
  if (a.K == 0) return cudaMemset2DAsync(a.C, a.ldc * 2, 0, static_cast<size_t>(a.N) * 2, a.M, s);
  // Small M: 128-column tiles put twice as many SMs on the weight stream.
  return a.M <= 64 ? launch_variant<1>(a, s) : launch_variant<2>(a, s);
}

}  // namespace wq
