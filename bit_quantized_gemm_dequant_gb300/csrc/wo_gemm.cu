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
//   warps 2-9   dequant, two warps per TMEM lane quarter taking alternate
//               64-k steps (two steps in flight per CTA): lane L of warp w
//               owns weight column n = 32*(w%4) + L (its TMEM lane).  It reads its column of the packed tile
//               byte by byte, turns every byte into exact fp16 values (INT4:
//               0x6400 | nibble = 1024 + q, minus 1032; INT8: byte ^ 0x80 |
//               0x6400, minus 1152) and writes 32 fp16 pairs (one 64-k slice)
//               with tcgen05.st into a ring of A buffers in TMEM.  The
//               dequantized weight never touches shared or global memory.
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma.kind::f16 with A
//               from TMEM (128 n x 16 k) and B = the X tile from shared memory
//               (K-major), 128 x 256 x 16, four per 64-k slice.
//   warps 2-9   then the epilogue: tcgen05.ld of the 128 x 256 accumulator
//               (the two warps of a lane quarter take alternate 32 columns),
//               multiply by the per-column scale (exact to move out of the K
//               sum: it is per column), round to fp16 and store; a warp writes
//               32 consecutive columns of one row of Y per store.
// Column-grouped scales and zero points ("Triton 量化算子：W8A16 权重量化融合矩
// 阵乘法", 扩展说明): the scale of column n is scales[n / group_n], and a
// zero point z replaces the fixed 8 (INT4) or 0 (INT8) in the constant each
// thread subtracts for its own column.
//
// Mid M (16 < M <= 64, the "tile per (M, N, K)" choice of the W4A16 page §二
// at a shape between decode and prefill): one 64-row activation tile, so each
// weight is dequantized exactly once, and the K loop of every 128-column tile
// split among the S CTAs of a thread-block cluster so that tiles x S fills
// the GPU (two CTAs per SM).  Each CTA parks its 128 x 64 FP32 partial in its
// own shared memory; after a cluster barrier CTA r reads rows r*64/S ..
// (r+1)*64/S - 1 of every peer's partial through distributed shared memory,
// adds them in rank order (deterministic), scales, rounds and stores; a
// second cluster barrier keeps each CTA's shared memory alive until its peers
// are done reading it.  These launches use programmatic dependent launch, so
// a call's prologue overlaps the previous kernel's tail.
#include <cuda_fp16.h>

#include "tc_common.cuh"
#include "tma_host.h"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int BN = 128;            // weight columns per CTA (MMA M)
constexpr int kXBoxK = 64;         // k per X box (128 bytes of fp16: one swizzle span)
constexpr int kDequantWarps = 8;   // two per TMEM lane quarter
constexpr int kThreads = (2 + kDequantWarps) * 32;
constexpr int kMidRows = 64;       // activation rows of the mid-M (cluster K-split) instance
constexpr int kMaxClusterK = 8;    // portable cluster size

constexpr int kSmPerSmem = 228 * 1024;  // shared memory of one SM
constexpr int kSmemPerCtaReserved = 1024;

template <int BITS, int BM>
struct WoGemmCfg {
  // k per stage.  A stage has a fixed cost (the barrier round trips of its
  // TMA -> dequant -> MMA chain), so fewer, larger stages pay off where the
  // ring still holds several: INT4 at every tile height (W4A16 4096^3 went
  // from 138 to 118 us, M = 64 at N = 11008 from 18.1 to 16.3 us) and INT8 at
  // 128 rows (M = 512: 34.5 to 28.4 us).  INT8 keeps 64 at 64 rows (three
  // stages instead of six: 5% slower) and at 256 rows (two stages: 19% slower).
  static constexpr int kBK = (BITS == 4 || BM == 128) ? 128 : 64;
  static constexpr int kXBoxes = kBK / kXBoxK;     // X boxes per stage
  static constexpr int kACols = kBK / 2;           // TMEM columns (fp16 pairs) per A slice
  static constexpr int kXBytes = BM * kBK * 2;
  static constexpr int kWRows = BITS == 4 ? kBK / 2 : kBK;
  static constexpr int kWBytes = kWRows * BN;
  static constexpr int kStageBytes = ((kXBytes + kWBytes + 1023) / 1024) * 1024;
  static constexpr int kAccCols = BM;
  static constexpr int kTmemCols = BM == kMidRows ? 256 : 512;  // mid M: two CTAs per SM
  static constexpr int kCtasPerSm = 512 / kTmemCols;
  // TMEM A ring: the columns the accumulator leaves, at most 8 slices.
  static constexpr int kAStagesFit = (kTmemCols - kAccCols) / kACols;
  static constexpr int kAStages = kAStagesFit > 8 ? 8 : kAStagesFit;
  // Shared-memory ring: as deep as the SM's share for kCtasPerSm CTAs allows
  // (at most 8 stages).  The ring also keeps a (kCtasPerSm + 1)-th CTA off
  // the SM: it could not get tensor memory and would stall in its allocation
  // until a neighbour left.
  static constexpr int kStagesFit = (kSmPerSmem / kCtasPerSm - kSmemPerCtaReserved - 2048) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 1024;
  static_assert(kStages >= 2, "ring depth");
  static_assert((kSmemBytes + kSmemPerCtaReserved) * (kCtasPerSm + 1) > kSmPerSmem, "one CTA too many per SM");
  static_assert(kAccCols + kAStages * kACols <= kTmemCols, "TMEM budget");
  static_assert(kAStages >= 2, "TMEM A ring depth");
  // Mid M: the FP32 partial tile [BM rows][BN columns] reuses the idle ring.
  static_assert(BM != kMidRows || BM * BN * 4 <= kStages * kStageBytes, "partial tile fits in the ring");
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

__device__ __forceinline__ uint32_t h2_bits2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

template <int BITS, int BM, bool kCluster>
__global__ void __launch_bounds__(kThreads, kCluster ? 2 : 1)  // mid M: two CTAs per SM
wo_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, WoArgs p,
               int* err) {
  using Cfg = WoGemmCfg<BITS, BM>;
  constexpr int kStages = Cfg::kStages;
  constexpr int kAStages = Cfg::kAStages;
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
  const int KT = (p.K + Cfg::kBK - 1) / Cfg::kBK;
  // This CTA's 128-column tile and its k-tiles [kt0, kt0 + nk): all of K, or
  // (cluster K-split) the rank's share.
  int n_tile = blockIdx.x, rank = 0, S = 1;
  if constexpr (kCluster) {
    rank = static_cast<int>(tc::cluster_ctarank());
    S = static_cast<int>(tc::cluster_nctarank());
    n_tile = blockIdx.x / S;
    tc::griddep_launch_dependents();
  }
  const int n0 = n_tile * BN, m0 = blockIdx.y * BM;
  const int kt0 = static_cast<int>(static_cast<int64_t>(rank) * KT / S);
  const int nk = static_cast<int>(static_cast<int64_t>(rank + 1) * KT / S) - kt0;

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
  tc::cta_barrier();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_ring = tmem + Cfg::kAccCols;
  // Programmatic dependent launch: everything above overlapped the previous
  // kernel; no thread reads global memory before that kernel has finished.
  if constexpr (kCluster) tc::griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmX);
      tc::tma_prefetch_desc(&tmW);
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % kStages, kt = kt0 + i;
        if (!tc::mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1, abort, err, kSiteGemmProducer)) break;
        uint8_t* st = smem + s * Cfg::kStageBytes;
        tc::mbar_arrive_expect_tx(&full[s], Cfg::kXBytes + Cfg::kWBytes);
#pragma unroll
        for (int h = 0; h < Cfg::kXBoxes; ++h)
          tc::tma_load_2d(st + h * BM * kXBoxK * 2, &tmX, kt * Cfg::kBK + h * kXBoxK, m0, &full[s]);
        tc::tma_load_2d(st + Cfg::kXBytes, &tmW, n0, kt * Cfg::kWRows, &full[s]);
        issued = i + 1;
      }
      if (*abort)
        for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
          tc::mbar_wait_drain(&full[i % kStages], (i / kStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_dense(/*F16*/ 0, /*F16*/ 0, 0, 0, 128, BM);
      for (int i = 0; i < nk; ++i) {
        const int s = i % kStages, t = i % kAStages;
        if (!tc::mbar_wait(&full[s], (i / kStages) & 1, abort, err, kSiteGemmMma)) break;
        if (!tc::mbar_wait(&a_full[t], (i / kAStages) & 1, abort, err, kSiteGemmMma)) break;
        tc::tc_fence_after();
        const uint32_t xs = tc::smem_u32(smem + s * Cfg::kStageBytes);
#pragma unroll
        for (int j = 0; j < Cfg::kBK / 16; ++j) {  // 16 k per MMA, four per 64-k X box
          const uint64_t bdesc =
              tc::smem_desc(xs + (j / 4) * BM * kXBoxK * 2 + 32 * (j % 4), 1024, 1024, tc::kSwizzle128B);
          mma_f16_tmem_a(tmem, a_ring + t * Cfg::kACols + 8 * j, bdesc, idesc, (i | j) != 0);
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
    // Dequant warps, then the epilogue.  Group dg (0 or 1) of the lane
    // quarter q takes local steps dg, dg + 2, ... and accumulator chunks dg,
    // dg + 2, ...
    const int q = warp & 3, dg = (warp - 2) >> 2;
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
    for (int i = dg; i < nk; i += 2) {
      const int s = i % kStages, t = i % kAStages;
      bool ok = tc::mbar_wait(&full[s], (i / kStages) & 1, abort, err, kSiteGemmProducer);
      ok = ok && tc::mbar_wait(&a_empty[t], ((i / kAStages) & 1) ^ 1, abort, err, kSiteGemmTmemFree);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint8_t* wt = smem + s * Cfg::kStageBytes + Cfg::kXBytes + nl;
      tc::tc_fence_after();
      // The stage's k in 64-k halves (32 fp16 pairs each), so that one half's
      // registers are live at a time.
#pragma unroll 1
      for (int h = 0; h < Cfg::kXBoxes; ++h) {
        uint32_t r[32];
        if constexpr (BITS == 4) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint32_t b = wt[(32 * h + c) * BN];  // codes of k = 2c (low nibble), 2c + 1 of the half
            const uint32_t v = ((b * 0x1001u) & 0x000F000Fu) | 0x64006400u;
            r[c] = h2_sub(v, sub);  // minus 1024 + zero point
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int row = 64 * h + 2 * c;
            const uint32_t b = static_cast<uint32_t>(wt[row * BN]) | (static_cast<uint32_t>(wt[(row + 1) * BN]) << 16);
            r[c] = h2_sub((b ^ 0x00800080u) | 0x64006400u, sub);  // minus 1152 + zero point
          }
        }
        tmem_st_32x32b_x32(a_ring + t * Cfg::kACols + 32 * h + lane_off, r);
      }
      tc::fence_proxy_async_smem();  // generic reads of the tile before its TMA refill
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[s]);  // this warp is done with the packed tile
      tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&a_full[t]);
    }
    const bool done = tc::mbar_wait(accum, 0, abort, err, kSiteGemmEpilogue);
    tc::tc_fence_after();
    if constexpr (kCluster) {
      // Park the partial tile, row-major [BM][BN], in the idle ring: every
      // load has landed and every MMA has completed (accum).
      float* part = reinterpret_cast<float*>(smem);
#pragma unroll 1
      for (int c = dg; c < BM / 32; c += 2) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + lane_off + 32 * c, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) part[(32 * c + i) * BN + nl] = __uint_as_float(v[i]);
      }
    }
    const float sc = (gn < p.N) ? __half2float(static_cast<const __half*>(p.scales)[gn / p.group_n]) : 0.0f;
    __half* Y = static_cast<__half*>(p.Y);
    for (int c = dg; c < (kCluster ? 0 : BM / 32); c += 2) {
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
  tc::cta_barrier();
  if constexpr (kCluster) {
    // Every CTA of the cluster gets here (all its waits are bounded), so the
    // two cluster barriers end.  First: all partial tiles are in place.
    tc::cluster_sync_all();
    if (warp >= 2) {
      // Rows r0 .. r1 - 1 of the tile, four columns per item; the S peers'
      // float4s of an item (plain loads through generic addresses, which the
      // compiler batches) are added in rank order.
      const int r0 = rank * BM / S;
      const int r1 = min((rank + 1) * BM / S, p.M - m0);
      const float4* part = reinterpret_cast<const float4*>(smem);
      const float4* peer[kMaxClusterK];
#pragma unroll
      for (int q = 0; q < kMaxClusterK; ++q) peer[q] = tc::peer_ptr(part, q < S ? q : 0);
      const __half* scales = static_cast<const __half*>(p.scales);
      __half* Y = static_cast<__half*>(p.Y);
      const bool live = !*abort;
      for (int it = threadIdx.x - 64; it < (r1 - r0) * (BN / 4); it += kThreads - 64) {
        const int r = r0 + it / (BN / 4), c4 = it % (BN / 4);
        const int off = r * (BN / 4) + c4;
        float4 v[kMaxClusterK];
#pragma unroll
        for (int q = 0; q < kMaxClusterK; ++q)
          if (q < S) v[q] = peer[q][off];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kMaxClusterK; ++q)
          if (q < S) {
            acc.x += v[q].x;
            acc.y += v[q].y;
            acc.z += v[q].z;
            acc.w += v[q].w;
          }
        const int gn = n0 + 4 * c4;
        if (!live || gn >= p.N) continue;
        const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
        __half h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          h[j] = __float2half_rn(gn + j < p.N ? __half2float(scales[(gn + j) / p.group_n]) * a4[j] : 0.0f);
        __half* dst = Y + static_cast<int64_t>(m0 + r) * p.ldy + gn;
        if (gn + 4 <= p.N) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(h2_bits2(h[0], h[1]), h2_bits2(h[2], h[3]));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (gn + j < p.N) dst[j] = h[j];
        }
      }
    }
    // Second: no CTA leaves (releasing its shared memory) while a peer may
    // still read its partial tile.
    tc::cluster_sync_all();
  }
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <int BITS, int BM, bool kCluster>
cudaError_t configure_tc() {
  static PerDevice<bool> configured;
  bool done = false;
  cudaError_t e = cudaSuccess;
  if (!configured.get(done, [&](bool& v) {
        e = cudaFuncSetAttribute(wo_gemm_kernel<BITS, BM, kCluster>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 WoGemmCfg<BITS, BM>::kSmemBytes);
        if (e == cudaSuccess)
          e = cudaFuncSetAttribute(wo_gemm_kernel<BITS, BM, kCluster>,
                                   cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        v = true;
        return e == cudaSuccess;
      }))
    return e == cudaSuccess ? cudaErrorUnknown : e;
  return cudaSuccess;
}

template <int BITS, int BM>
cudaError_t launch_tc(const WoArgs& a, cudaStream_t s) {
  using Cfg = WoGemmCfg<BITS, BM>;
  CUtensorMap tX, tW;
  cudaError_t e = make_tmap_2d(&tX, a.X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.K, a.M, a.ldx * 2, kXBoxK, BM,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const uint64_t w_rows = BITS == 4 ? a.K / 2 : a.K;
  e = make_tmap_2d(&tW, a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, w_rows, a.ldw, BN, Cfg::kWRows,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  if ((e = configure_tc<BITS, BM, false>()) != cudaSuccess) return e;
  dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM);
  wo_gemm_kernel<BITS, BM, false><<<grid, kThreads, Cfg::kSmemBytes, s>>>(tX, tW, a, device_error_word());
  return cudaGetLastError();
}

// Mid M: the K-split size S of each 128-column tile's cluster.  As many CTAs
// as the GPU holds at once (tiles x S, with the kCtasPerSm CTAs per SM that
// the ring and tensor-memory sizes admit), S at most the portable cluster
// size and at most the number of 64-k steps.
template <int BITS>
int mid_split(int N, int K) {
  using Cfg = WoGemmCfg<BITS, kMidRows>;
  const int64_t tiles = (N + BN - 1) / BN, kt = (K + Cfg::kBK - 1) / Cfg::kBK;
  int64_t S = static_cast<int64_t>(sm_count()) * Cfg::kCtasPerSm / tiles;
  if (S > kMaxClusterK) S = kMaxClusterK;
  if (S > kt) S = kt;
  return S < 1 ? 1 : static_cast<int>(S);
}

template <int BITS>
cudaError_t launch_mid(const WoArgs& a, cudaStream_t s) {
  using Cfg = WoGemmCfg<BITS, kMidRows>;
  CUtensorMap tX, tW;
  cudaError_t e = make_tmap_2d(&tX, a.X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.K, a.M, a.ldx * 2, kXBoxK, kMidRows,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const uint64_t w_rows = BITS == 4 ? a.K / 2 : a.K;
  e = make_tmap_2d(&tW, a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, w_rows, a.ldw, BN, Cfg::kWRows,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  if ((e = configure_tc<BITS, kMidRows, true>()) != cudaSuccess) return e;
  const int S = mid_split<BITS>(a.N, a.K);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((a.N + BN - 1) / BN * S), 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, wo_gemm_kernel<BITS, kMidRows, true>, tX, tW, a, device_error_word());
  if (e != cudaSuccess) return e;
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
  if (a.M <= kMidRows) return bits == 4 ? launch_mid<4>(a, s) : launch_mid<8>(a, s);
  if (wo_gemm_rows(a.M, a.N) == 128) return bits == 4 ? launch_tc<4, 128>(a, s) : launch_tc<8, 128>(a, s);
  return bits == 4 ? launch_tc<4, 256>(a, s) : launch_tc<8, 256>(a, s);
}

}  // namespace wq
