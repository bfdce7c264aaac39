// Skinny GEMMs for small M (decode): W4A16, W8A16 and the M <= 16 FP8 GEMM.
//
// Defined by "Triton 工业级融合微算子编写：W4A16 极速切片矩阵乘与 Blackwell NVFP4
// 硬件指令实装" §二 (INT4: byte row k/2, even k in the low nibble, weight
// (q - 8) * s[n], FP32 accumulation, FP16 output) and "Triton 量化算子：W8A16
// 权重量化融合矩阵乘法" Step 1 / Step 3 (INT8: Y = X (W_int8 S), W [K, N]); and
// "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核" (e4m3 A [M, K] x B [K, N],
// FP32 accumulation, acc * scale_a * scale_b, BF16 output) — at M <= 16 that
// GEMM is a weight stream exactly like W8A16 (B has the same [K, N] byte
// layout), so it shares this path.
//
// Design (HBM-bound; the packed weights are read from HBM exactly once):
//   * One CTA of twelve warps per SM.  A work unit is one chunk of one
//     128-column tile: 32 rows x 128 bytes of the packed weight matrix (64 k
//     for INT4, 32 k for INT8 and e4m3).  The CTA's local units are dealt to
//     its warps round-robin, and every warp streams its own units: lane 0
//     issues the TMA loads of the unit's weight box (128-byte swizzle) and of
//     the matching activation box into one of the warp's own ring slots
//     (three per warp where they fit, else two), and refills a slot as soon as
//     the warp has consumed it.  About 144 KB of weights per SM are in flight,
//     no warp waits for another to free a slot, and none waits on a global
//     load.  A slot is only ever filled and read by one warp, in order (an
//     mbarrier wait names only the parity of a phase, so a reader that could
//     reach a slot two fills ahead would take a stale phase for a fresh one).
//   * A consumer thread reads 16-byte vectors of packed weights from shared
//     memory (rows 2c, 2c + 1, ... so that, with the swizzle, the eight lanes
//     of a quarter-warp hit eight different bank groups) and dequantizes them
//     in registers straight into the A operand of mma.sync (Y^T = W^T X^T:
//     weight columns are the MMA rows, the M <= 16 activation rows the MMA
//     columns).  INT4 codes become exact fp16 (q - 8) with one LOP3 (0x6400 |
//     nibble = 1024 + nibble) and one HSUB2/HFMA2 per two weights; INT8 with
//     one LOP3 (byte ^ 0x80 | 0x6400) and one HSUB2.  The per-column scale
//     factors out of the K sum and is applied once in the epilogue (exact
//     reordering: it is per column).
//   * e4m3 needs no dequantization: four K rows of 16 bytes are turned into
//     K-contiguous 4-byte words by a 4 x 4 byte transpose (PRMT) and fed to
//     mma.sync.m16n8k32.e4m3.
//   * MMA k-order: any bijection between the MMA's k slots and the real k
//     indices gives the same sum as long as the weight and activation
//     fragments use the same one.  Each fragment slot pair is mapped to the
//     weight rows a thread loads (see the per-mode comments), and the
//     activation fragment is gathered from shared memory in that order.
//   * Work split, one of three plans per shape (make_plan):
//       - one CTA per tile when the tiles fill at least half the SMs: no
//         split of K, no hand-shake;
//       - otherwise a cluster of S CTAs per tile, each streaming a slice of
//         K; the partial tiles meet in distributed shared memory, each CTA
//         pushing the other CTAs' slices into their receive areas with
//         st.async (no CTA reads another's shared memory);
//       - otherwise stream-K: the grid is the SM count and the (M tile,
//         128-column tile, chunk) units are dealt out as equal contiguous
//         runs; a tile split between CTAs meets in the caller's workspace,
//         where the last CTA to arrive (per-tile counter) adds the parts in
//         CTA order and resets the counter.
//     In every plan the warps' partial sums of a tile meet in shared memory
//     (lane-native float4 layout, conflict free) and every sum runs in a
//     fixed order, so results are deterministic.
//   * Column-grouped scales and zero points ("Triton 量化算子：W8A16 权重量化
//     融合矩阵乘法", 扩展说明) are a separate compile-time instance: the zero
//     point enters through the activation row sums, once per tile.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "skinny_common.cuh"
#include "tc_common.cuh"
#include "tma_host.h"
#include "wq_internal.h"

namespace wq {
namespace {

// Stream-K plan: U = tiles * chunks units over G CTAs; CTA b owns units
// [b*U/G, (b+1)*U/G).
// cluster > 1: the grid is tiles * cluster CTAs in clusters of that size;
// CTA b's run is then chunks [r ch / S, (r + 1) ch / S) of tile b / S (r its
// rank), and the cluster adds its partial tiles through distributed shared
// memory instead of the workspace.
using Plan = SkinnyPlan;

// Number of CTAs whose runs touch tile T.
__device__ __forceinline__ int tile_contributors(int T, int64_t U, int G, int ch) {
  return unit_owner(static_cast<int64_t>(T + 1) * ch - 1, U, G) - unit_owner(static_cast<int64_t>(T) * ch, U, G) + 1;
}


// kZp: the weight-only modes with zero points (a separate instance, so that
// the symmetric kernels carry none of their code).
template <int BITS, int MT, bool kZp>
__global__ void __launch_bounds__(kThreads, 1)
wo_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, SkinnyArgs p,
                 Plan pl, int* err) {
  using C = Cfg<BITS, MT>;
  constexpr int D = C::kDepth;
  constexpr int kFinElems = (C::kOutF4 + kThreads - 1) / kThreads;  // partial elements a thread finishes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* ring = smem;
  float4* red = reinterpret_cast<float4*>(smem + C::kRingBytes);  // [kRedBufs][kOutF4]
  float4* rx = red + kRedBufs * C::kOutF4;  // [S][kOutF4 / S]: peer q's part of this CTA's slice at q
  float* col_fac = reinterpret_cast<float*>(rx + C::kOutF4);  // [kTileN] output factors
  float* col_zf = col_fac + kTileN;  // [kTileN] zero-point correction factors
  uint64_t* full =
      reinterpret_cast<uint64_t*>(smem + C::kRingBytes + C::kRedBytes + C::kRxBytes + C::kFacBytes);
  volatile int* abort = reinterpret_cast<volatile int*>(full + C::kStages);
  volatile int* last_flag = abort + 1;  // [2]
  uint64_t* rx_bar = reinterpret_cast<uint64_t*>(const_cast<int*>(abort) + 4);  // 8-byte aligned

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.x, G = gridDim.x;
  const int64_t U = pl.units;
  const int ch = pl.chunks;
  const int64_t lo = unit_lo(b, U, G);
  const int n_local = static_cast<int>(unit_lo(b + 1, U, G) - lo);
  // This warp's units are local indices warp, warp + kWarps, ...; its k-th
  // unit goes to its own slot warp * D + k % D.
  const int n_mine = n_local > warp ? (n_local - warp + kWarps - 1) / kWarps : 0;

  // The next call in the stream may start claiming SMs as this grid's CTAs
  // leave; it waits (griddep_wait) before touching memory this grid writes.
  tc::griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) tc::mbar_init(&full[s], 1);
    if (pl.cluster > 1) tc::mbar_init(rx_bar, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  tc::cta_barrier();
  if (pl.cluster > 1) {
    // The receive barrier expects the other CTAs' slices of this CTA's part of
    // the tile; every CTA's barrier is armed before any CTA sends.
    if (threadIdx.x == 0)
      tc::mbar_arrive_expect_tx(rx_bar, static_cast<uint32_t>((pl.cluster - 1) * (C::kOutF4 / pl.cluster) * 16));
    tc::cluster_sync_all();
  }

  // Lane 0 of a warp starts the TMA loads of the warp's units in order; the
  // cursor (tile, chunk) of the next one advances by kWarps units at a time
  // (no division in the loop).
  int cur_n = 0, cur_m = 0, cur_c = 0;  // n tile, m tile, chunk
  if (n_mine > 0) {
    const int64_t u = lo + warp;
    const int t0 = static_cast<int>(u / ch);
    cur_c = static_cast<int>(u - static_cast<int64_t>(t0) * ch);
    cur_n = t0 % pl.n_tiles;
    cur_m = t0 / pl.n_tiles;
  }
  auto issue = [&](int k) {
    const int s = warp * D + k % D;
    uint8_t* slot = ring + s * C::kSlotBytes;
    tc::mbar_arrive_expect_tx(&full[s], kWBytes + C::kXBytes);
    tc::tma_load_2d(slot, &tmW, cur_n * kTileN, cur_c * kBoxRows, &full[s]);
    tc::tma_load_2d(slot + kWBytes, &tmX, cur_c * C::kChunkK, cur_m * C::kRows, &full[s]);
    cur_c += kWarps;
    while (cur_c >= ch) {
      cur_c -= ch;
      if (++cur_n == pl.n_tiles) {
        cur_n = 0;
        ++cur_m;
      }
    }
  };
  // With static weights (the caller's promise that no kernel still running
  // writes W), the first round's weight boxes go straight into the ring
  // while the previous kernel of the stream may still be running; their
  // activation boxes, which that kernel may be writing, follow the wait.
  int early = 0;
  int early_m[D], early_c[D];
  if (lane == 0) {
    tc::tma_prefetch_desc(&tmW);
    tc::tma_prefetch_desc(&tmX);
    if (p.early_w) {
#pragma unroll
      for (int k = 0; k < D; ++k) {
        if (k >= n_mine) break;
        uint8_t* slot = ring + (warp * D + k) * C::kSlotBytes;
        tc::mbar_arrive_expect_tx(&full[warp * D + k], kWBytes + C::kXBytes);
        tc::tma_load_2d(slot, &tmW, cur_n * kTileN, cur_c * kBoxRows, &full[warp * D + k]);
        early_m[k] = cur_m;
        early_c[k] = cur_c;
        early = k + 1;
        cur_c += kWarps;
        while (cur_c >= ch) {
          cur_c -= ch;
          if (++cur_n == pl.n_tiles) {
            cur_n = 0;
            ++cur_m;
          }
        }
      }
    } else {
      // Pull the warp's first weight boxes into L2 while the previous kernel
      // of the stream may still be running (a prefetch cannot read stale data).
      int pn = cur_n, pc = cur_c;
      for (int k = 0; k < D && k < n_mine; ++k) {
        tc::tma_prefetch_l2_2d(&tmW, pn * kTileN, pc * kBoxRows);
        pc += kWarps;
        while (pc >= ch) {
          pc -= ch;
          if (++pn == pl.n_tiles) pn = 0;
        }
      }
    }
  }
  // Everything below reads inputs or writes outputs and workspace that
  // earlier work in the stream may still own.
  tc::griddep_wait();
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < D; ++k)
      if (k < early)
        tc::tma_load_2d(ring + (warp * D + k) * C::kSlotBytes + kWBytes, &tmX, early_c[k] * C::kChunkK,
                        early_m[k] * C::kRows, &full[warp * D + k]);
    for (int k = early; k < D && k < n_mine; ++k) issue(k);
  }

  int* ws_count = static_cast<int*>(p.ws);
  float4* ws_part = reinterpret_cast<float4*>(static_cast<uint8_t*>(p.ws) + kCounterBytes);
  const int t = threadIdx.x;
  int k = 0;  // the warp's next unit to consume
  bool ok = true;
  int pend0 = -1, pend1 = -1;  // shared tiles of this run (its first and last segment at most)
  const bool stage_fac = BITS != kE4m3 && (pl.cluster > 1 || pl.grid == pl.tiles);
  int fac_n_base = 0;  // n_base of the staged factors
  // Factors of element e's two columns in the current tile.
  auto fin_factors = [&](int e) {
    if (!stage_fac) return elem_factors<BITS>(p, e, fac_n_base);
    const int col = elem_col(e);
    return make_float2(col_fac[col], col_fac[col + 1]);
  };
  // One segment per tile the CTA's run touches.
  for (int i = 0; i < n_local;) {
    const int64_t u0 = lo + i;
    const int T = static_cast<int>(u0 / ch);
    const int64_t seg_end = static_cast<int64_t>(T + 1) * ch < lo + n_local ? static_cast<int64_t>(T + 1) * ch
                                                                             : lo + n_local;
    const int seg = static_cast<int>(seg_end - u0);
    const int m_base = (T / pl.n_tiles) * C::kRows, n_base = (T % pl.n_tiles) * kTileN;
    fac_n_base = n_base;
    // The first element this thread finishes if the tile ends here (the CTA's
    // own tile, or its slice of a cluster's tile).
    const int e_first = pl.cluster > 1 ? static_cast<int>(tc::cluster_ctarank()) * C::kOutF4 / pl.cluster + t : t;
    // Plans with one segment per CTA stage the tile's per-column scales in
    // shared memory now, while the first weight boxes are in flight, so that
    // the epilogue does not wait on global loads after the stream.
    if (stage_fac && t < kTileN) {
      const int gn = n_base + t;
      col_fac[t] = gn < p.N ? __half2float(static_cast<const __half*>(p.scales)[gn / p.group_n]) : 0.0f;
    }
    // With zero points, each column's factor for the activation-sum term:
    // INT8 sums x (1152 + q) and corr holds -1152 sum x, so corr (1152 + z) /
    // 1152 completes sum x (q - z); INT4 sums x (q - 8) and corr holds sum x,
    // so corr (8 - z) does.
    if (kZp && t < kTileN) {
      const int gn = n_base + t;
      float f = 0.0f;
      if (gn < p.N) {
        const int g = gn / p.group_n;
        if constexpr (BITS == kInt8)
          f = static_cast<float>(1152 + static_cast<const int8_t*>(p.zeros)[g]) * (1.0f / 1152.0f);
        else
          f = static_cast<float>(8 - static_cast<int>(static_cast<const uint8_t*>(p.zeros)[g]));
      }
      col_zf[t] = f;
    }

    float acc[MT][8][4], corr[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[mt][q][r] = 0.0f;
#pragma unroll
      for (int r = 0; r < 4; ++r) corr[mt][r] = 0.0f;
    }

    for (; ok && k < n_mine && warp + k * kWarps < i + seg; ++k) {
      const int s = warp * D + k % D;
      ok = __all_sync(0xffffffffu, tc::mbar_wait_sleep(&full[s], (k / D) & 1, abort, err, kSiteGemmMma, p.wait_ns));
      if (!ok) break;
      const uint8_t* slot = ring + s * C::kSlotBytes;
      UnitRegs<BITS, MT> ur;
      load_unit<BITS, MT>(ur, slot, slot + kWBytes, g, c);
      // The slot's next contents arrive through TMA (async proxy): order the
      // warp's generic-proxy reads of the slot before lane 0 refills it, and
      // refill it before the math, so that the copy overlaps the math.
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && k + D < n_mine) issue(k + D);
      compute_unit<BITS, MT, kZp && BITS == kInt4>(acc, corr, ur);
    }
    if constexpr (kZp) {
      // Per-column zero points: corr times the column's factor (staged at the
      // start of the segment; the barrier makes it visible).  acc[mt][q][r]
      // is column 16g + 2q + r / 2 of the tile.
      cta_sync();
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[mt][q][r] += corr[mt][r] * col_zf[16 * g + 2 * q + (r >> 1)];
    } else if constexpr (BITS == kInt8) {
      // The correction is the same for every MMA row (weight column).
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[mt][q][r] += corr[mt][r];
    }

    // Warp w adds into buffer w % kRedBufs in round w / kRedBufs; the buffers
    // are then summed in index order (a fixed order: deterministic).
    float4* buf = red + (warp % kRedBufs) * C::kOutF4;
    for (int r = 0; r < kRedRounds; ++r) {
      if (warp / kRedBufs == r) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 v = make_float4(acc[mt][q][0], acc[mt][q][1], acc[mt][q][2], acc[mt][q][3]);
            float4* d = buf + (mt * 8 + q) * 32 + lane;
            if (r > 0) v = f4add(*d, v);
            *d = v;
          }
      }
      cta_sync();
    }

    // A tile inside the run is this CTA's alone: finish it now.  Only the
    // first and the last segment of a contiguous run can share their tile
    // with other CTAs; their partial tiles go to the workspace now, and the
    // hand-shake with the other contributors waits for the end of the run,
    // so that it never stalls the stream.
    if (pl.cluster > 1) {
      // The cluster's CTAs each hold one part of this tile, and CTA q
      // finishes slice q of it.  Each CTA adds its four buffers and sends
      // every other slice straight into the owner's receive area (one-way
      // stores that count toward the owner's receive barrier); the owner
      // then adds the S parts of its slice in rank order, so the result does
      // not depend on arrival order.  No CTA reads another's shared memory,
      // so none has to wait for its peers before leaving.
      const int S = pl.cluster, r = static_cast<int>(tc::cluster_ctarank());
      const int slice = C::kOutF4 / S;
      for (int e = t; e < C::kOutF4; e += kThreads) {
        const int q = e / slice;
        if (q == r) continue;
        float4 v = red[e];
#pragma unroll
        for (int b2 = 1; b2 < kRedBufs; ++b2) v = f4add(v, red[b2 * C::kOutF4 + e]);
        tc::st_async_f4(tc::dsmem_addr(rx + r * slice + (e - q * slice), q), v, tc::dsmem_addr(rx_bar, q));
      }
      if (t < slice) {
        const int e = e_first;  // r * slice + t
        float4 own = red[e];
#pragma unroll
        for (int b2 = 1; b2 < kRedBufs; ++b2) own = f4add(own, red[b2 * C::kOutF4 + e]);
        const bool got = tc::mbar_wait_cluster(rx_bar, 0, err, kSiteClusterRecv);
        const int rows_valid = p.M - m_base < C::kRows ? p.M - m_base : C::kRows;
        if (got && elem_live(e, rows_valid)) {
          float4 sum = r == 0 ? own : rx[t];
          for (int q = 1; q < S; ++q) sum = f4add(sum, q == r ? own : rx[q * slice + t]);
          store_elem<BITS>(p, e, m_base, n_base, sum, fin_factors(e));
        }
      }
    } else if (seg == ch || tile_contributors(T, U, G, ch) == 1) {  // the whole tile is in this run
      const int rows_valid = p.M - m_base < C::kRows ? p.M - m_base : C::kRows;
#pragma unroll
      for (int j = 0; j < kFinElems; ++j) {
        const int e = t + j * kThreads;
        if (e >= C::kOutF4 || !elem_live(e, rows_valid)) continue;
        float4 v = red[e];
#pragma unroll
        for (int q = 1; q < kRedBufs; ++q) v = f4add(v, red[q * C::kOutF4 + e]);
        store_elem<BITS>(p, e, m_base, n_base, v, fin_factors(e));
      }
    } else {
      const int f0 = unit_owner(static_cast<int64_t>(T) * ch, U, G);
      float4* mine = ws_part + (static_cast<size_t>(T) * pl.slots + (b - f0)) * C::kOutF4;
      const int rows_valid = p.M - m_base < C::kRows ? p.M - m_base : C::kRows;
      for (int e = t; e < C::kOutF4; e += kThreads) {
        if (!elem_live(e, rows_valid)) continue;
        float4 v = red[e];
#pragma unroll
        for (int q = 1; q < kRedBufs; ++q) v = f4add(v, red[q * C::kOutF4 + e]);
        __stcg(mine + e, v);
      }
      if (pend0 < 0) pend0 = T; else pend1 = T;
    }
    cta_sync();  // `red` is reused by the next segment
    i += seg;
  }

  // Hand-shake for the shared tiles: publish this CTA's partials, count it in
  // on each tile, and finish the tiles it was the last to reach (summing the
  // partials in CTA order, so the result does not depend on who came last).
  if (pend0 >= 0) {
    __threadfence();
    cta_sync();
    if (t < 2) {
      const int T = t == 0 ? pend0 : pend1;
      last_flag[t] = T >= 0 && atomicAdd(&ws_count[T], 1) == tile_contributors(T, U, G, ch) - 1;
    }
    cta_sync();
    for (int j = 0; j < 2; ++j) {
      if (last_flag[j] == 0) continue;
      __threadfence();
      const int T = j == 0 ? pend0 : pend1;
      const int contributors = tile_contributors(T, U, G, ch);
      const int m_base = (T / pl.n_tiles) * C::kRows, n_base = (T % pl.n_tiles) * kTileN;
      const int rows_valid = p.M - m_base < C::kRows ? p.M - m_base : C::kRows;
      const float4* src = ws_part + static_cast<size_t>(T) * pl.slots * C::kOutF4;
      for (int e = t; e < C::kOutF4; e += kThreads) {
        if (!elem_live(e, rows_valid)) continue;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        // Eight partial tiles in flight at a time; summed in contributor order.
        for (int q0 = 0; q0 < contributors; q0 += 8) {
          float4 v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            v[q] = q0 + q < contributors ? __ldcg(src + static_cast<size_t>(q0 + q) * C::kOutF4 + e)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int q = 0; q < 8; ++q) sum = f4add(sum, v[q]);
        }
        store_elem<BITS>(p, e, m_base, n_base, sum, elem_factors<BITS>(p, e, n_base));
      }
      if (t == 0) ws_count[T] = 0;  // ready for the next call
    }
  }

  // After a give-up, let this warp's copies still in flight land before the
  // CTA exits (no TMA write may target the shared memory of a finished CTA).
  if (!ok && lane == 0)
    for (int kk = k; kk < n_mine && kk < k + D; ++kk) tc::mbar_wait_drain(&full[warp * D + kk % D], (kk / D) & 1);
}

// Opt the kernel into its dynamic shared memory (above the 48 KB default);
// must precede both the occupancy query and the first launch.
template <int BITS, int MT, bool kZp = false>
cudaError_t configure_kernel() {
  static PerDevice<cudaError_t> status;
  cudaError_t e = cudaSuccess;
  status.get(e, [&e](cudaError_t& v) {
    v = e = cudaFuncSetAttribute(wo_skinny_kernel<BITS, MT, kZp>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Cfg<BITS, MT>::kSmemBytes));
    return v == cudaSuccess;
  });
  return e;
}

template <int BITS, int MT>
int ctas_per_sm() {
  static PerDevice<int> cached;
  int n = 1;
  if (!cached.get(n, [](int& v) {
        return configure_kernel<BITS, MT>() == cudaSuccess &&
               cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, wo_skinny_kernel<BITS, MT, false>, kThreads,
                                                             Cfg<BITS, MT>::kSmemBytes) == cudaSuccess &&
               v >= 1;
      }))
    return 1;  // not cached: a later call may succeed
  return n;
}

// Clusters of S of these CTAs that the GPU holds at once (0 when it holds
// none or the query fails; not cached then).
template <int BITS, int MT>
int max_clusters(int S) {
  static PerDevice<int> cached[9];
  if (S < 2 || S > 8) return 0;
  int n = 0;
  cached[S].get(n, [S](int& v) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<BITS, MT>::kSmemBytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return configure_kernel<BITS, MT>() == cudaSuccess &&
           cudaOccupancyMaxActiveClusters(&v, wo_skinny_kernel<BITS, MT, false>, &cfg) == cudaSuccess && v >= 1;
  });
  return n;  // 0 when the query failed (not cached: a later call may succeed)
}

template <int BITS, int MT>
Plan make_plan(int M, int N, int K) {
  using C = Cfg<BITS, MT>;
  Plan pl;
  pl.mt = MT;
  pl.ws_bytes = 0;
  pl.n_tiles = (N + kTileN - 1) / kTileN;
  pl.tiles = pl.n_tiles * ((M + C::kRows - 1) / C::kRows);
  pl.chunks = (K + C::kChunkK - 1) / C::kChunkK;
  pl.units = static_cast<int64_t>(pl.tiles) * pl.chunks;
  const int64_t cap = static_cast<int64_t>(sm_count()) * ctas_per_sm<BITS, MT>();
  pl.grid = static_cast<int>(pl.units < cap ? pl.units : cap);
  // Enough tiles to occupy at least half of the GPU: one CTA per tile, no
  // split of K, so no hand-shake between CTAs (its round trips cost more than
  // the SMs left idle).
  if (2 * static_cast<int64_t>(pl.tiles) >= cap && pl.tiles <= cap) pl.grid = pl.tiles;
  pl.slots = 1;
  pl.cluster = 1;
  // Fewer tiles: split each tile's K among a cluster of S CTAs that reduce
  // through distributed shared memory (no workspace, no round trip through
  // L2), if the clusters fit in one wave and cover at least half the GPU.
  if (2 * static_cast<int64_t>(pl.tiles) < cap) {
    for (int S = 8; S >= 2; S /= 2) {
      const int64_t g = static_cast<int64_t>(pl.tiles) * S;
      if (g <= cap && 2 * g >= cap && S <= pl.chunks && pl.tiles <= max_clusters<BITS, MT>(S)) {
        pl.cluster = S;
        pl.grid = static_cast<int>(g);
        return pl;
      }
    }
  }
  if (pl.tiles > kMaxSplitTiles) {  // too many tiles for the counter area: one CTA per tile, no split
    pl.grid = pl.tiles;
    return pl;
  }
  for (int T = 0; T < pl.tiles; ++T) {
    const int n = unit_owner(static_cast<int64_t>(T + 1) * pl.chunks - 1, pl.units, pl.grid) -
                  unit_owner(static_cast<int64_t>(T) * pl.chunks, pl.units, pl.grid) + 1;
    if (n > pl.slots) pl.slots = n;
  }
  if (pl.slots > 1) pl.ws_bytes = kCounterBytes + static_cast<size_t>(pl.tiles) * pl.slots * C::kOutF4 * 16;
  return pl;
}

template <int BITS, int MT, bool kZp>
cudaError_t launch_variant(const SkinnyArgs& a, const Plan& pl, cudaStream_t s) {
  using C = Cfg<BITS, MT>;
  cudaError_t e = configure_kernel<BITS, MT, kZp>();
  if (e != cudaSuccess) return e;
  CUtensorMap tW, tX;
  const uint64_t rows = BITS == kInt4 ? a.K / 2 : a.K;
  // 128-byte L2 fetches: the weight boxes' rows are 128 bytes, and the
  // neighbouring tile's bytes belong to another CTA (0.5% faster than 256).
  e = make_tmap_2d(&tW, a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, rows, a.ldw, kTileN, kBoxRows,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e != cudaSuccess) return e;
  const CUtensorMapSwizzle xs = C::kXRowBytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : C::kXRowBytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_32B;
  if constexpr (BITS == kE4m3)
    e = make_tmap_2d(&tX, a.X, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.K, a.M, a.ldx, C::kChunkK, C::kRows, xs);
  else
    e = make_tmap_2d(&tX, a.X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.K, a.M, a.ldx * 2, C::kChunkK, C::kRows, xs);
  if (e != cudaSuccess) return e;
  // Launched as a programmatic dependent of the previous kernel in the stream:
  // its prologue and weight prefetch overlap that kernel's tail.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pl.cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = pl.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, wo_skinny_kernel<BITS, MT, kZp>, tW, tX, a, pl, device_error_word());
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The plan's M-tile height (mt) picks the kernel instance.
template <int BITS>
cudaError_t launch_mode(const SkinnyArgs& a, const Plan& pl, cudaStream_t s) {
  if constexpr (BITS != kE4m3) {
    if (a.zeros != nullptr)
      return pl.mt == 2 ? launch_variant<BITS, 2, true>(a, pl, s) : launch_variant<BITS, 1, true>(a, pl, s);
  }
  return pl.mt == 2 ? launch_variant<BITS, 2, false>(a, pl, s) : launch_variant<BITS, 1, false>(a, pl, s);
}

template <int BITS>
Plan mode_plan(int M, int N, int K) {
  return M > 8 ? make_plan<BITS, 2>(M, N, K) : make_plan<BITS, 1>(M, N, K);
}

}  // namespace

SkinnyPlan plan_skinny(int M, int N, int K, int mode) {
  if (M <= 0 || N <= 0 || K <= 0) return SkinnyPlan{};
  return mode == 4 ? mode_plan<kInt4>(M, N, K) : mode == 8 ? mode_plan<kInt8>(M, N, K) : mode_plan<kE4m3>(M, N, K);
}

cudaError_t launch_wo_skinny(const WoArgs& a, int bits, const SkinnyPlan& pl, cudaStream_t s) {
  if (a.K == 0) return cudaMemset2DAsync(a.Y, a.ldy * 2, 0, static_cast<size_t>(a.N) * 2, a.M, s);
  const SkinnyArgs sa{a.M, a.N, a.K, a.X, a.ldx, a.W, a.ldw, a.scales, 1.0f, a.Y, a.ldy, a.ws, a.zeros, a.group_n,
                      skinny_wait_ns(), static_weights() ? 1 : 0};
  return bits == 4 ? launch_mode<kInt4>(sa, pl, s) : launch_mode<kInt8>(sa, pl, s);
}

cudaError_t launch_fp8_skinny(const Fp8GemmArgs& a, const SkinnyPlan& pl, cudaStream_t s) {
  if (a.K == 0) return cudaMemset2DAsync(a.C, a.ldc * 2, 0, static_cast<size_t>(a.N) * 2, a.M, s);
  const SkinnyArgs sa{a.M, a.N, a.K, a.A, a.lda, a.B, a.ldb, nullptr, a.scale_a * a.scale_b, a.C, a.ldc, a.ws,
                      nullptr, 1, skinny_wait_ns()};
  return launch_mode<kE4m3>(sa, pl, s);
}

}  // namespace wq

// --------------------------------------------------------------------------
// Built-in scratch for callers that cannot allocate device memory.
//
// Some callers may not allocate at call time: an engine plugin whose enqueue
// step must not allocate, a real-time loop that forbids cudaMalloc/cudaFree
// once it runs, or a runtime that plans every device byte ahead.  For them the
// INT8 skinny path can keep its split-K scratch (tile counters and partial
// sums) in this fixed array instead of a caller workspace.  Every GPU that
// loads the library holds the array until the process exits.
namespace wq {

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

cudaError_t noalloc_scratch(void** ptr) {
  // The array's host-side name is not a device address: look the address up
  // once per device, with that device current.
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

size_t skinny_counter_bytes() { return kCounterBytes; }

}  // namespace wq
