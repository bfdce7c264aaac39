// Batched weight-only GEMMs for small M (decode): up to kMaxBatch independent
// W4A16 or W8A16 problems in one launch.
//
// Each problem is defined as for the per-call kernels: "Triton 工业级融合微算子
// 编写：W4A16 极速切片矩阵乘与 Blackwell NVFP4 硬件指令实装" §二 (INT4: byte row k/2,
// even k in the low nibble, weight (q - 8) * s[n], FP32 accumulation, FP16
// output) and "Triton 量化算子：W8A16 权重量化融合矩阵乘法" Step 1 / Step 3 (INT8:
// Y = X (W_int8 S), W [K, N]); column-grouped scales as in that page's 扩展说明.
//
// Why a batch: at M <= 16 one GEMM moves 8 to 60 MB, a few microseconds of
// HBM time, and every launch pays a fixed ramp (dependency release, first
// data latency, the last warps' tail, the reduction) of the same order.  A
// decoder step runs several independent projections on the same activations
// (or on activations that are ready at the same time); one launch streams all
// of their weights through the same per-warp TMA rings, so the ramp is paid
// once and HBM stays busy across problem boundaries.
//
// Work split ("ordered stream-K"): the units (one chunk of 32 packed weight
// rows of one 128-column tile) of all problems are laid end to end, problem by
// problem, tile by tile, and the grid (one CTA per SM) takes equal contiguous
// runs of them.  A run covers whole tiles, which the CTA finishes alone, and
// at most two tiles it shares with its neighbours.  A shared tile is finished
// by one CTA, its finalizer (the middle CTA when three runs touch it, else the
// one holding its last units); the other CTAs publish their partial tiles to
// the workspace.  Every CTA computes the pieces it publishes FIRST and the
// piece it finalizes LAST, so a finalizer normally finds the other parts
// already published when it needs them: the hand-shake sits off the critical
// path, and no CTA waits for anything before publishing (no cycle of waits).
// The finalizer adds the parts in CTA order, so the result is deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "skinny_common.cuh"
#include "tc_common.cuh"
#include "tma_host.h"
#include "wq_internal.h"

namespace wq {
namespace {

struct BatchProb {
  SkinnyArgs a;
  int n_tiles;   // 128-column tiles
  int tiles;     // n_tiles * M tiles
  int chunks;    // units per tile
  int unit_off;  // first unit of this problem in the batch
  int tile_off;  // first tile of this problem in the batch (workspace counters)
};

struct BatchTable {
  CUtensorMap tmW[kMaxBatch];
  CUtensorMap tmX[kMaxBatch];
  BatchProb prob[kMaxBatch];
  int count;
  int units;
  uint64_t wait_ns;  // limit of a bounded wait before the kernel gives up
};

struct TileRef {
  int p;       // problem
  int t;       // tile within the problem
  int ts, te;  // the tile's units [ts, te) in the batch
};

// The problem and tile that hold unit u (problems with no units are not in
// the table, so the unit offsets strictly increase).
__device__ __forceinline__ TileRef tile_of(const BatchTable& tb, int u) {
  int p = 0;
  while (p + 1 < tb.count && tb.prob[p + 1].unit_off <= u) ++p;
  const int ch = tb.prob[p].chunks;
  const int t = (u - tb.prob[p].unit_off) / ch;
  const int ts = tb.prob[p].unit_off + t * ch;
  return TileRef{p, t, ts, ts + ch};
}

// The CTA that finishes a tile touched by several runs: the middle one when
// exactly three runs touch it, else the one holding the tile's last units.
__device__ __forceinline__ int finalizer(int bf, int bl) { return bl - bf == 2 ? bf + 1 : bl; }

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// A contiguous range of units, processed as a whole, in the CTA's order.
struct Piece {
  int s, e;
};

template <int BITS, int MT>
__global__ void __launch_bounds__(kThreads, 1)
wo_batched_kernel(const __grid_constant__ BatchTable tb, int* ws_count, float4* ws_part, int* err) {
  using C = Cfg<BITS, MT>;
  constexpr int D = C::kDepth;
  constexpr int kFinElems = (C::kOutF4 + kThreads - 1) / kThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* ring = smem;
  float4* red = reinterpret_cast<float4*>(smem + C::kRingBytes);  // [kRedBufs][kOutF4]
  float* col_fac = reinterpret_cast<float*>(smem + C::kRingBytes + C::kRedBytes + C::kRxBytes);  // [kTileN]
  uint64_t* full =
      reinterpret_cast<uint64_t*>(smem + C::kRingBytes + C::kRedBytes + C::kRxBytes + C::kFacBytes);
  volatile int* abort = reinterpret_cast<volatile int*>(full + C::kStages);
  volatile int* fin_ok = abort + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int t = threadIdx.x;
  const int b = blockIdx.x, G = gridDim.x;
  const int U = tb.units;
  const int lo = static_cast<int>(unit_lo(b, U, G)), hi = static_cast<int>(unit_lo(b + 1, U, G));
  const int n_local = hi - lo;
  const int n_mine = n_local > warp ? (n_local - warp + kWarps - 1) / kWarps : 0;

  // This CTA's pieces in processing order: the shared pieces it publishes,
  // then its whole tiles, then the shared piece it finalizes.
  Piece P[3];
  int np = 0;
  if (n_local > 0) {
    const TileRef A = tile_of(tb, lo), Z = tile_of(tb, hi - 1);
    if (A.ts == Z.ts) {
      P[np++] = Piece{lo, hi};
    } else {
      const bool f_split = lo != A.ts, l_split = hi != Z.te;
      const bool f_fin = f_split && finalizer(unit_owner(A.ts, U, G), unit_owner(A.te - 1, U, G)) == b;
      if (f_split && !f_fin) P[np++] = Piece{lo, A.te};
      if (l_split) P[np++] = Piece{Z.ts, hi};
      const int mid_s = f_split ? A.te : lo, mid_e = l_split ? Z.ts : hi;
      if (mid_s < mid_e) P[np++] = Piece{mid_s, mid_e};
      if (f_fin) P[np++] = Piece{lo, A.te};
    }
  }

  tc::griddep_launch_dependents();
  if (t == 0) {
    for (int s = 0; s < C::kStages; ++s) tc::mbar_init(&full[s], 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  tc::cta_barrier();

  // Issue cursor of this warp: piece cp, batch unit cu, and its problem,
  // tile and chunk (cb, ct, cc), advanced by kWarps units at a time.
  int cp = 0, cu = 0, cb = 0, ct = 0, cc = 0;
  auto decompose = [&]() {
    const TileRef r = tile_of(tb, cu);
    cb = r.p;
    ct = r.t;
    cc = cu - r.ts;
  };
  auto advance = [&]() {
    cu += kWarps;
    if (cu >= P[cp].e) {
      int over = cu - P[cp].e;
      ++cp;
      while (cp < np && over >= P[cp].e - P[cp].s) {
        over -= P[cp].e - P[cp].s;
        ++cp;
      }
      if (cp < np) {
        cu = P[cp].s + over;
        decompose();
      }
      return;
    }
    cc += kWarps;
    int ch = tb.prob[cb].chunks;
    while (cc >= ch) {  // the next tile, possibly of the next problem (cu stays inside the piece)
      cc -= ch;
      if (++ct == tb.prob[cb].tiles) {
        ct = 0;
        ++cb;
        ch = tb.prob[cb].chunks;
      }
    }
  };
  if (n_mine > 0) {
    int v = warp, base = 0;
    while (v >= base + (P[cp].e - P[cp].s)) {
      base += P[cp].e - P[cp].s;
      ++cp;
    }
    cu = P[cp].s + (v - base);
    decompose();
  }
  auto issue = [&](int k) {
    const int s = warp * D + k % D;
    uint8_t* slot = ring + s * C::kSlotBytes;
    const int nt = tb.prob[cb].n_tiles;
    const int mt = ct / nt, nt_i = ct - mt * nt;
    tc::mbar_arrive_expect_tx(&full[s], kWBytes + C::kXBytes);
    tc::tma_load_2d(slot, &tb.tmW[cb], nt_i * kTileN, cc * kBoxRows, &full[s]);
    tc::tma_load_2d(slot + kWBytes, &tb.tmX[cb], cc * C::kChunkK, mt * C::kRows, &full[s]);
    advance();
  };
  if (lane == 0) {
    for (int p = 0; p < tb.count; ++p) {
      tc::tma_prefetch_desc(&tb.tmW[p]);
      tc::tma_prefetch_desc(&tb.tmX[p]);
    }
  }
  // Inputs and outputs (and the workspace) may still belong to earlier work
  // in the stream until this returns.
  tc::griddep_wait();
  if (lane == 0)
    for (int k = 0; k < D && k < n_mine; ++k) issue(k);

  int k = 0;  // the warp's next unit to consume
  bool ok = true;
  int i = 0;  // local index of the current segment's first unit
  for (int pc = 0; pc < np; ++pc) {
    for (int u0 = P[pc].s; u0 < P[pc].e;) {
      const TileRef T = tile_of(tb, u0);
      const int u1 = T.te < P[pc].e ? T.te : P[pc].e;
      const int seg = u1 - u0;
      const BatchProb& bp = tb.prob[T.p];
      const SkinnyArgs& pa = bp.a;
      const int m_base = (T.t / bp.n_tiles) * C::kRows, n_base = (T.t % bp.n_tiles) * kTileN;
      const bool whole = u0 == T.ts && u1 == T.te;
      const int bf = whole ? b : unit_owner(T.ts, U, G), bl = whole ? b : unit_owner(T.te - 1, U, G);
      const bool fin = !whole && finalizer(bf, bl) == b;
      if (!whole && !fin) {
        // nothing to stage: the published part carries no scale
      } else if (t < kTileN) {
        const int gn = n_base + t;
        col_fac[t] = gn < pa.N ? __half2float(static_cast<const __half*>(pa.scales)[gn / pa.group_n]) : 0.0f;
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
        ok = __all_sync(0xffffffffu, tc::mbar_wait_sleep(&full[s], (k / D) & 1, abort, err, kSiteGemmMma, tb.wait_ns));
        if (!ok) break;
        const uint8_t* slot = ring + s * C::kSlotBytes;
        UnitRegs<BITS, MT> ur;
        load_unit<BITS, MT>(ur, slot, slot + kWBytes, g, c);
        // Generic-proxy reads of the slot before its TMA refill.
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && k + D < n_mine) issue(k + D);
        compute_unit<BITS, MT, false>(acc, corr, ur);
      }
      if constexpr (BITS == kInt8) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int q = 0; q < 8; ++q)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[mt][q][r] += corr[mt][r];
      }
      // The warps' partial tiles meet in shared memory (fixed order).
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
      const int rows_valid = pa.M - m_base < C::kRows ? pa.M - m_base : C::kRows;
      if (whole) {
#pragma unroll
        for (int j = 0; j < kFinElems; ++j) {
          const int e = t + j * kThreads;
          if (e >= C::kOutF4 || !elem_live(e, rows_valid)) continue;
          float4 v = red[e];
#pragma unroll
          for (int q = 1; q < kRedBufs; ++q) v = f4add(v, red[q * C::kOutF4 + e]);
          const int col = elem_col(e);
          store_elem<BITS>(pa, e, m_base, n_base, v, make_float2(col_fac[col], col_fac[col + 1]));
        }
      } else if (!fin) {
        // Publish this CTA's part: slot 0 holds the part of the tile its run
        // starts in, slot 1 the part of the tile its run ends in.
        float4* mine = ws_part + (static_cast<size_t>(b) * 2 + (T.ts < lo ? 0 : 1)) * C::kOutF4;
        for (int e = t; e < C::kOutF4; e += kThreads) {
          if (!elem_live(e, rows_valid)) continue;
          float4 v = red[e];
#pragma unroll
          for (int q = 1; q < kRedBufs; ++q) v = f4add(v, red[q * C::kOutF4 + e]);
          __stcg(mine + e, v);
        }
        __threadfence();
        cta_sync();
        if (t == 0) atomicAdd(&ws_count[bp.tile_off + T.t], 1);
      } else {
        float4 own[kFinElems];
#pragma unroll
        for (int j = 0; j < kFinElems; ++j) {
          const int e = t + j * kThreads;
          own[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (e >= C::kOutF4) continue;
          own[j] = red[e];
#pragma unroll
          for (int q = 1; q < kRedBufs; ++q) own[j] = f4add(own[j], red[q * C::kOutF4 + e]);
        }
        // Wait (bounded) until the other CTAs touching the tile have
        // published their parts.
        if (t == 0) {
          int* cnt = &ws_count[bp.tile_off + T.t];
          bool got = ld_acquire(cnt) >= bl - bf;
          if (!got) {
            const uint64_t t0 = tc::globaltimer_ns();
            while (!(got = ld_acquire(cnt) >= bl - bf)) {
              if (tc::globaltimer_ns() - t0 > tb.wait_ns) {
                if (err) atomicCAS(err, 0, kSiteBatchRecv);
                *abort = 1;
                break;
              }
              __nanosleep(64);
            }
          }
          __threadfence();
          *fin_ok = got;
          if (got) *cnt = 0;  // ready for the next call
        }
        cta_sync();
        if (*fin_ok) {
#pragma unroll
          for (int j = 0; j < kFinElems; ++j) {
            const int e = t + j * kThreads;
            if (e >= C::kOutF4 || !elem_live(e, rows_valid)) continue;
            float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int q = bf; q <= bl; ++q) {
              if (q == b) {
                sum = f4add(sum, own[j]);
              } else {
                const int lo_q = static_cast<int>(unit_lo(q, U, G));
                const float4* part = ws_part + (static_cast<size_t>(q) * 2 + (T.ts < lo_q ? 0 : 1)) * C::kOutF4;
                sum = f4add(sum, __ldcg(part + e));
              }
            }
            const int col = elem_col(e);
            store_elem<BITS>(pa, e, m_base, n_base, sum, make_float2(col_fac[col], col_fac[col + 1]));
          }
        }
      }
      cta_sync();  // `red` and the factors are reused by the next segment
      i += seg;
      u0 = u1;
    }
  }

  // After a give-up, let this warp's copies still in flight land before the
  // CTA exits (no TMA write may target the shared memory of a finished CTA).
  if (!ok && lane == 0)
    for (int kk = k; kk < n_mine && kk < k + D; ++kk) tc::mbar_wait_drain(&full[warp * D + kk % D], (kk / D) & 1);
}

template <int BITS, int MT>
cudaError_t configure_batched() {
  static PerDevice<cudaError_t> status;
  cudaError_t e = cudaSuccess;
  status.get(e, [&e](cudaError_t& v) {
    v = e = cudaFuncSetAttribute(wo_batched_kernel<BITS, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Cfg<BITS, MT>::kSmemBytes));
    return v == cudaSuccess;
  });
  return e;
}

template <int BITS, int MT>
size_t batched_ws_bytes(int grid) {
  return kCounterBytes + static_cast<size_t>(grid) * 2 * Cfg<BITS, MT>::kOutF4 * 16;
}

template <int BITS, int MT>
cudaError_t launch_batched_variant(const WoArgs* probs, int count, const BatchPlan& pl, void* ws, cudaStream_t s) {
  using C = Cfg<BITS, MT>;
  cudaError_t e = configure_batched<BITS, MT>();
  if (e != cudaSuccess) return e;
  BatchTable tb = {};
  tb.wait_ns = skinny_wait_ns();
  int units = 0, tiles = 0, n = 0;
  for (int i = 0; i < count; ++i) {
    const WoArgs& a = probs[i];
    if (a.M == 0 || a.N == 0 || a.K == 0) continue;
    BatchProb& bp = tb.prob[n];
    bp.a = SkinnyArgs{a.M, a.N, a.K, a.X, a.ldx, a.W, a.ldw, a.scales, 1.0f, a.Y, a.ldy, nullptr, nullptr, a.group_n,
                      tb.wait_ns};
    bp.n_tiles = (a.N + kTileN - 1) / kTileN;
    bp.tiles = bp.n_tiles * ((a.M + C::kRows - 1) / C::kRows);
    bp.chunks = (a.K + C::kChunkK - 1) / C::kChunkK;
    bp.unit_off = units;
    bp.tile_off = tiles;
    units += bp.tiles * bp.chunks;
    tiles += bp.tiles;
    const uint64_t rows = BITS == kInt4 ? a.K / 2 : a.K;
    // 128-byte L2 fetches: a CTA's run walks one tile's K range, so the 128
    // bytes next to a box row (the neighbouring tile) are read by another CTA
    // much later; with 256-byte fetches they were fetched twice (ncu: 288 MB
    // of DRAM reads for 227 MB of weights, 229 MB with 128-byte fetches).
    e = make_tmap_2d(&tb.tmW[n], a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, rows, a.ldw, kTileN, kBoxRows,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
    if (e != cudaSuccess) return e;
    const CUtensorMapSwizzle xs = C::kXRowBytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : C::kXRowBytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_32B;
    e = make_tmap_2d(&tb.tmX[n], a.X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.K, a.M, a.ldx * 2, C::kChunkK, C::kRows, xs);
    if (e != cudaSuccess) return e;
    ++n;
  }
  tb.count = n;
  tb.units = units;
  if (n == 0 || units != pl.units || pl.grid < 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int* ws_count = static_cast<int*>(ws);
  float4* ws_part = reinterpret_cast<float4*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  e = cudaLaunchKernelEx(&cfg, wo_batched_kernel<BITS, MT>, tb, ws_count, ws_part, device_error_word());
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

BatchPlan plan_batched(const WoArgs* probs, int count, int bits) {
  BatchPlan pl = {};
  int mt = 1;
  int64_t units = 0, tiles = 0;
  for (int i = 0; i < count; ++i) {
    const WoArgs& a = probs[i];
    if (a.M == 0 || a.N == 0 || a.K == 0) continue;
    if (a.M > 8) mt = 2;
  }
  const int rows = 8 * mt, chunk_k = bits == 4 ? 64 : 32;
  for (int i = 0; i < count; ++i) {
    const WoArgs& a = probs[i];
    if (a.M == 0 || a.N == 0 || a.K == 0) continue;
    const int64_t t = static_cast<int64_t>((a.N + kTileN - 1) / kTileN) * ((a.M + rows - 1) / rows);
    tiles += t;
    units += t * ((a.K + chunk_k - 1) / chunk_k);
  }
  pl.mt = mt;
  if (units == 0) return pl;
  if (tiles > kMaxSplitTiles || units >= (int64_t(1) << 31) / 2) {
    pl.unsupported = true;
    return pl;
  }
  pl.units = static_cast<int>(units);
  const int sms = sm_count();
  pl.grid = static_cast<int>(units < sms ? units : sms);
  pl.ws_bytes = bits == 4 ? (mt == 2 ? batched_ws_bytes<kInt4, 2>(pl.grid) : batched_ws_bytes<kInt4, 1>(pl.grid))
                          : (mt == 2 ? batched_ws_bytes<kInt8, 2>(pl.grid) : batched_ws_bytes<kInt8, 1>(pl.grid));
  return pl;
}

cudaError_t launch_wo_batched(const WoArgs* probs, int count, int bits, const BatchPlan& pl, void* ws,
                              cudaStream_t s) {
  for (int i = 0; i < count; ++i) {  // K = 0 problems: Y = 0
    const WoArgs& a = probs[i];
    if (a.M > 0 && a.N > 0 && a.K == 0) {
      const cudaError_t e = cudaMemset2DAsync(a.Y, a.ldy * 2, 0, static_cast<size_t>(a.N) * 2, a.M, s);
      if (e != cudaSuccess) return e;
    }
  }
  if (pl.units == 0) return cudaSuccess;
  if (bits == 4)
    return pl.mt == 2 ? launch_batched_variant<kInt4, 2>(probs, count, pl, ws, s)
                      : launch_batched_variant<kInt4, 1>(probs, count, pl, ws, s);
  return pl.mt == 2 ? launch_batched_variant<kInt8, 2>(probs, count, pl, ws, s)
                    : launch_batched_variant<kInt8, 1>(probs, count, pl, ws, s);
}

}  // namespace wq
