// Weight-only GEMM for large M (prefill): W4A16 / W8A16 on the 5th-generation
// tensor cores, dequantizing in registers straight into tensor memory.
//
// Defined by "Triton 工业级融合微算子编写：W4A16 极速切片矩阵乘与 Blackwell NVFP4
// 硬件指令实装" §二 (INT4 codes, even k in the low nibble, (q - 8) * s[n],
// FP32 accumulation) and "Triton 量化算子：W8A16 权重量化融合矩阵乘法" Step 1 /
// Step 3 (INT8, Y = X (W_int8 S)).
//
// The product is computed transposed, Y^T[n, m] = sum_k W[k, n] X[m, k], so
// that the dequantized weights are the MMA's A operand and can live in TMEM:
//   warp 0      TMA producer: X tile 256(m) x 64(k) fp16 (128-byte swizzle)
//               and the packed weight tile (INT4 32 x 128 bytes, INT8 64 x 128
//               bytes, no swizzle) into a shared-memory ring.
//   warps 2-5   dequant: lane L of warp w owns weight column n = 32*(w%4) + L
//               (its TMEM lane).  It reads its column of the packed tile
//               byte by byte, turns every byte into exact fp16 values (INT4:
//               0x6400 | nibble = 1024 + q, minus 1032; INT8: byte ^ 0x80 |
//               0x6400, minus 1152) and writes 32 fp16 pairs (one 64-k slice)
//               with tcgen05.st into a ring of A buffers in TMEM.  The
//               dequantized weight never touches shared or global memory.
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma.kind::f16 with A
//               from TMEM (128 n x 16 k) and B = the X tile from shared memory
//               (K-major), 128 x 256 x 16, four per 64-k slice.
//   warps 2-5   then the epilogue: tcgen05.ld of the 128 x 256 accumulator,
//               multiply by the per-column scale (exact to move out of the K
//               sum: it is per column), round to fp16 and store; a warp writes
//               32 consecutive columns of one row of Y per store.
// Column-grouped scales and zero points ("Triton 量化算子：W8A16 权重量化融合矩
// 阵乘法", 扩展说明): the scale of column n is scales[n / group_n], and a
// zero point z replaces the fixed 8 (INT4) or 0 (INT8) in the constant each
// thread subtracts for its own column.
#include <cuda_fp16.h>

#include "tc_common.cuh"
#include "tma_host.h"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int BN = 128;            // weight columns per CTA (MMA M)
constexpr int BK = 64;             // k per stage
constexpr int kStages = 4;         // shared-memory ring
constexpr int kAStages = 4;        // TMEM A ring
constexpr int kThreads = 192;
constexpr int kAColsPerStage = BK / 2;  // fp16 pairs per TMEM lane

template <int BITS, int BM>
struct WoGemmCfg {
  static constexpr int kXBytes = BM * BK * 2;
  static constexpr int kWRows = BITS == 4 ? BK / 2 : BK;
  static constexpr int kWBytes = kWRows * BN;
  static constexpr int kStageBytes = ((kXBytes + kWBytes + 1023) / 1024) * 1024;
  static constexpr int kAccCols = BM;
  static constexpr int kTmemCols = 512;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 1024;
  static_assert(kAccCols + kAStages * kAColsPerStage <= kTmemCols, "TMEM budget");
};

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

template <int BITS, int BM>
__global__ void __launch_bounds__(kThreads, 1)
wo_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, WoArgs p,
               int* err) {
  using Cfg = WoGemmCfg<BITS, BM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * Cfg::kStageBytes);
  uint64_t* empty = full + kStages;       // MMA done with X (commit) + 4 dequant warps done with W
  uint64_t* a_full = empty + kStages;     // 4 dequant warps wrote the TMEM A slice
  uint64_t* a_empty = a_full + kAStages;  // MMA done with the TMEM A slice (commit)
  uint64_t* accum = a_empty + kAStages;
  uint64_t* drain = accum + 1;            // MMAs in flight after a give-up
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int KT = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 5);
    }
    for (int t = 0; t < kAStages; ++t) {
      tc::mbar_init(&a_full[t], 4);
      tc::mbar_init(&a_empty[t], 1);
    }
    tc::mbar_init(accum, 1);
    tc::mbar_init(drain, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_ring = tmem + Cfg::kAccCols;

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmX);
      tc::tma_prefetch_desc(&tmW);
      int issued = 0;
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % kStages;
        if (!tc::mbar_wait(&empty[s], ((kt / kStages) & 1) ^ 1, abort, err, kSiteGemmProducer)) break;
        uint8_t* st = smem + s * Cfg::kStageBytes;
        tc::mbar_arrive_expect_tx(&full[s], Cfg::kXBytes + Cfg::kWBytes);
        tc::tma_load_2d(st, &tmX, kt * BK, m0, &full[s]);
        tc::tma_load_2d(st + Cfg::kXBytes, &tmW, n0, kt * Cfg::kWRows, &full[s]);
        issued = kt + 1;
      }
      if (*abort)
        for (int kt = issued > kStages ? issued - kStages : 0; kt < issued; ++kt)
          tc::mbar_wait_drain(&full[kt % kStages], (kt / kStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_dense(/*F16*/ 0, /*F16*/ 0, 0, 0, 128, BM);
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % kStages, t = kt % kAStages;
        if (!tc::mbar_wait(&full[s], (kt / kStages) & 1, abort, err, kSiteGemmMma)) break;
        if (!tc::mbar_wait(&a_full[t], (kt / kAStages) & 1, abort, err, kSiteGemmMma)) break;
        tc::tc_fence_after();
        const uint32_t xs = tc::smem_u32(smem + s * Cfg::kStageBytes);
#pragma unroll
        for (int j = 0; j < BK / 16; ++j) {
          const uint64_t bdesc = tc::smem_desc(xs + 32 * j, 1024, 1024, tc::kSwizzle128B);
          mma_f16_tmem_a(tmem, a_ring + t * kAColsPerStage + 8 * j, bdesc, idesc, (kt | j) != 0);
        }
        tc::tc_commit(&empty[s]);
        tc::tc_commit(&a_empty[t]);
      }
      tc::tc_commit(accum);
      // After a give-up: wait (bounded) until every MMA issued so far has
      // completed, so that none still reads or writes TMEM when it is freed.
      if (*abort) {
        tc::tc_commit(drain);
        tc::mbar_wait_drain(drain, 0);
      }
    }
  } else {
    // Dequant warps, then the epilogue.
    const int q = warp & 3;
    const int nl = 32 * q + lane;  // this thread's weight column inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    const int gn = n0 + nl;
    // The fp16 constant the dequantization subtracts from 1024 + q (INT4) or
    // 1152 + q (INT8): the fixed zero point, or this column's group zero point
    // (1024 + z and 1152 + z are integers below 2048, exact in fp16).
    uint32_t sub = BITS == 4 ? 0x64086408u : 0x64806480u;
    if (p.zeros != nullptr && gn < p.N) {
      const int g = gn / p.group_n;
      const uint32_t z = BITS == 4 ? static_cast<uint32_t>(static_cast<const uint8_t*>(p.zeros)[g])
                                   : static_cast<uint32_t>(static_cast<int>(static_cast<const int8_t*>(p.zeros)[g]) + 128);
      sub = (0x6400u | z) * 0x10001u;
    }
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % kStages, t = kt % kAStages;
      bool ok = tc::mbar_wait(&full[s], (kt / kStages) & 1, abort, err, kSiteGemmProducer);
      ok = ok && tc::mbar_wait(&a_empty[t], ((kt / kAStages) & 1) ^ 1, abort, err, kSiteGemmTmemFree);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint8_t* wt = smem + s * Cfg::kStageBytes + Cfg::kXBytes + nl;
      uint32_t r[32];
      if constexpr (BITS == 4) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const uint32_t b = wt[c * BN];  // codes of k = 2c (low nibble), 2c + 1
          const uint32_t v = ((b * 0x1001u) & 0x000F000Fu) | 0x64006400u;
          r[c] = h2_sub(v, sub);  // minus 1024 + zero point
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const uint32_t b = static_cast<uint32_t>(wt[(2 * c) * BN]) | (static_cast<uint32_t>(wt[(2 * c + 1) * BN]) << 16);
          r[c] = h2_sub((b ^ 0x00800080u) | 0x64006400u, sub);  // minus 1152 + zero point
        }
      }
      tc::fence_proxy_async_smem();  // generic reads of the tile before its TMA refill
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[s]);  // this warp is done with the packed tile
      tc::tc_fence_after();
      tmem_st_32x32b_x32(a_ring + t * kAColsPerStage + lane_off, r);
      tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&a_full[t]);
    }
    const bool done = tc::mbar_wait(accum, 0, abort, err, kSiteGemmEpilogue);
    tc::tc_fence_after();
    const float sc = (gn < p.N) ? __half2float(static_cast<const __half*>(p.scales)[gn / p.group_n]) : 0.0f;
    __half* Y = static_cast<__half*>(p.Y);
    for (int c = 0; c < BM / 32; ++c) {
      uint32_t v[32];
      tc::tmem_ld_32x32b_x32(tmem + lane_off + 32 * c, v);
      tc::tmem_ld_wait();
      if (!done || gn >= p.N) continue;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int gm = m0 + 32 * c + i;
        if (gm < p.M) Y[static_cast<int64_t>(gm) * p.ldy + gn] = __float2half_rn(sc * __uint_as_float(v[i]));
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <int BITS, int BM>
cudaError_t launch_tc(const WoArgs& a, cudaStream_t s) {
  using Cfg = WoGemmCfg<BITS, BM>;
  CUtensorMap tX, tW;
  cudaError_t e = make_tmap_2d(&tX, a.X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.K, a.M, a.ldx * 2, BK, BM,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const uint64_t w_rows = BITS == 4 ? a.K / 2 : a.K;
  e = make_tmap_2d(&tW, a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, w_rows, a.ldw, BN, Cfg::kWRows,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  auto kern = wo_gemm_kernel<BITS, BM>;
  static PerDevice<bool> configured;
  bool done = false;
  if (!configured.get(done, [&](bool& v) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
        v = true;
        return e == cudaSuccess;
      }))
    return e;
  dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM);
  kern<<<grid, kThreads, Cfg::kSmemBytes, s>>>(tX, tW, a, device_error_word());
  return cudaGetLastError();
}

}  // namespace

// Rows of X per CTA.  A CTA's time is set mostly by its K loop (weight
// dequantization and the ring), not by its rows: a 128-row CTA takes about
// 0.85x a 256-row one.  So take 128-row tiles, which use twice the SMs, when
// they need no more waves (M = 512 at N = 4096: 128 CTAs instead of 64).
int wo_gemm_rows(int M, int N) {
  const int64_t sms = sm_count(), nt = (N + BN - 1) / BN;
  auto waves = [&](int bm) { return (nt * ((M + bm - 1) / bm) + sms - 1) / sms; };
  return waves(128) <= waves(256) ? 128 : 256;
}

cudaError_t launch_wo_gemm(const WoArgs& a, int bits, cudaStream_t s) {
  if (a.K == 0) return cudaMemset2DAsync(a.Y, a.ldy * 2, 0, static_cast<size_t>(a.N) * 2, a.M, s);
  if (wo_gemm_rows(a.M, a.N) == 128) return bits == 4 ? launch_tc<4, 128>(a, s) : launch_tc<8, 128>(a, s);
  return bits == 4 ? launch_tc<4, 256>(a, s) : launch_tc<8, 256>(a, s);
}

}  // namespace wq
