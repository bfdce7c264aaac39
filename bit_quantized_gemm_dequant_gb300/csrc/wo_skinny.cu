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
//   * A CTA owns 128 output columns and a slice of K.  One producer thread
//     streams the packed weight tile of every 64-k chunk (INT8: 64 rows x 128
//     bytes, INT4: 32 rows x 128 bytes) with TMA into a 64 KB shared-memory
//     ring, so up to 64 KB per CTA (three CTAs per SM) is in flight no matter
//     what the consumers are doing.
//   * Consumer warps take the chunks round-robin.  Each thread reads 16-byte
//     vectors of packed weights from shared memory and dequantizes them in
//     registers straight into the A operand of mma.sync.m16n8k16
//     (Y^T = W^T X^T: weight columns are the MMA rows, the M <= 16 activation
//     rows the MMA columns).  INT4 codes become exact fp16 (q - 8) with one
//     LOP3 (0x6400 | nibble = 1024 + nibble) and one HSUB2/HFMA2 per two
//     weights; INT8 with one LOP3 (byte ^ 0x80 | 0x6400) and one HSUB2.  The
//     per-column scale factors out of the K sum and is applied once in the
//     epilogue (exact reordering: it is per column).
//   * e4m3 needs no dequantization: four K rows of 16 bytes are turned into
//     K-contiguous 4-byte words by a 4 x 4 byte transpose (8 PRMT per 16
//     bytes) and fed to mma.sync.m16n8k32.e4m3; the activation fragment is
//     4 consecutive bytes of a row of A.
//   * INT4 MMA k-order: a register of the A fragment holds the low (or high)
//     nibbles of the same byte column from K-pair rows c and c + 4, so one
//     PRMT serves four weights; the activation fragment is permuted to the
//     same k order (k0+2c, k0+2c+8 | k0+2c+1, k0+2c+9).
//   * Stream-K split: the grid is exactly the number of CTAs the GPU holds at
//     once (three per SM), and the (M tile, 128-column tile, 64-k chunk) work
//     units are dealt out as equal contiguous runs, so every SM streams the
//     same number of bytes and the launch is a single wave.  Consumer warps
//     reduce a tile's partial sums through shared memory; when a tile is
//     split between CTAs, each writes its partial tile to the caller's
//     workspace and the last one to arrive (per-tile counter) adds them in a
//     fixed order, so the result is deterministic, and resets the counter.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "tc_common.cuh"
#include "tma_host.h"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kTileN = 256;       // output columns per tile: 256-byte rows per TMA box row
constexpr int kHalfN = 128;       // columns per consumer warp (a warp pair splits a tile)
constexpr int kChunkK = 32;       // k per pipeline stage
constexpr int kRingBytes = 48 * 1024;
constexpr int kConsumers = 4;     // consumer warps (plus one producer warp)
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kCtasPerSm = 3;
// Workspace layout: a fixed counter area first (one int per tile, at most
// kMaxSplitTiles tiles), so that the counters of any shape sit in bytes that
// every call leaves zero; the partial tiles follow.
constexpr int kMaxSplitTiles = 16384;
constexpr size_t kCounterBytes = kMaxSplitTiles * sizeof(int);

// Operand modes: packed INT4 weights, INT8 weights, e4m3 B operand.
constexpr int kInt4 = 4, kInt8 = 8, kE4m3 = 9;

// What the three modes share at the kernel boundary.  Weight-only: X fp16
// (ldx in elements), per-column fp16 scales, Y fp16.  e4m3: X = A bytes
// (ldx in bytes), the scalar scale_a * scale_b, Y = C bf16.
struct SkinnyArgs {
  int M, N, K;
  const void* X; int64_t ldx;
  const void* W; int64_t ldw;
  const void* scales; float scale;
  void* Y; int64_t ldy;
  void* ws;
};

template <int BITS>
struct Ring {
  static constexpr int kRows = BITS == kInt4 ? kChunkK / 2 : kChunkK;  // rows of the packed tile
  static constexpr int kStageBytes = kRows * kTileN;
  static constexpr int kStages = kRingBytes / kStageBytes;
  // Slot i % kStages holds local chunk i and chunk i is consumed by warp pair
  // i % 2: with an even slot count every slot belongs to one pair, which
  // waits on it in order, so a wait can never see the slot's phase from two
  // fills back (the parity of an mbarrier phase repeats every two phases).
  static_assert(kStages % 2 == 0, "each ring slot must belong to one warp pair");
};

template <int MT>
constexpr size_t skinny_smem_bytes() {
  return kRingBytes + sizeof(float) * 8 * MT * kTileN + 512 + 128;
}

// Stream-K plan: U = tiles * chunks units over G CTAs; CTA b owns units
// [b*U/G, (b+1)*U/G).
struct Plan {
  int n_tiles, tiles, chunks, grid, slots;
  int64_t units;
};

__host__ __device__ __forceinline__ int64_t unit_lo(int b, int64_t U, int G) { return (int64_t)b * U / G; }
// The CTA whose run contains unit u.
__host__ __device__ __forceinline__ int unit_owner(int64_t u, int64_t U, int G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

__device__ __forceinline__ uint32_t ldg_x2(const __half* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16832_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 4 x 4 byte transpose: words r0..r3 (rows, bytes = columns) -> c0..c3
// (columns, bytes = rows 0..3).
__device__ __forceinline__ void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3, uint32_t (&c)[4]) {
  const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r2, r3, 0x5140);
  const uint32_t t2 = __byte_perm(r0, r1, 0x7362), t3 = __byte_perm(r2, r3, 0x7362);
  c[0] = __byte_perm(t0, t1, 0x5410);
  c[1] = __byte_perm(t0, t1, 0x7632);
  c[2] = __byte_perm(t2, t3, 0x5410);
  c[3] = __byte_perm(t2, t3, 0x7632);
}

// One 32-k step of e4m3: v[0..3] = rows 4c .. 4c+3 and v[4..7] = rows
// 16 + 4c .. 16 + 4c + 3 of the step, 16 columns each.  MMA i takes columns
// 2i (MMA row g) and 2i + 1 (row g + 8).
template <int MT>
__device__ __forceinline__ void fp8_step(float (&acc)[MT][8][4], const uint4* v, const uint32_t (&xb)[MT][2]) {
  const uint32_t lo[4][4] = {{v[0].x, v[1].x, v[2].x, v[3].x}, {v[0].y, v[1].y, v[2].y, v[3].y},
                             {v[0].z, v[1].z, v[2].z, v[3].z}, {v[0].w, v[1].w, v[2].w, v[3].w}};
  const uint32_t hi[4][4] = {{v[4].x, v[5].x, v[6].x, v[7].x}, {v[4].y, v[5].y, v[6].y, v[7].y},
                             {v[4].z, v[5].z, v[6].z, v[7].z}, {v[4].w, v[5].w, v[6].w, v[7].w}};
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // columns 4j .. 4j + 3
    uint32_t cl[4], ch[4];
    transpose4x4(lo[j][0], lo[j][1], lo[j][2], lo[j][3], cl);
    transpose4x4(hi[j][0], hi[j][1], hi[j][2], hi[j][3], ch);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        mma16832_e4m3(acc[mt][2 * j + h], cl[2 * h], cl[2 * h + 1], ch[2 * h], ch[2 * h + 1], xb[mt][0], xb[mt][1]);
  }
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// fp16 pair {1024 + lo nibble of byte 0, 1024 + lo nibble of byte 2} -> minus 1032.
__device__ __forceinline__ uint32_t int4_lo_pair(uint32_t u) {
  const uint32_t t = (u & 0x000F000Fu) | 0x64006400u;
  return h2_bits(__hsub2(bits_h2(t), bits_h2(0x64086408u)));  // 1032 = 1024 + 8
}
// fp16 pair {1024 + 16 * hi nibble, ...} -> /16 - 72 = hi - 8.
__device__ __forceinline__ uint32_t int4_hi_pair(uint32_t u) {
  const uint32_t t = (u & 0x00F000F0u) | 0x64006400u;
  return h2_bits(__hfma2(bits_h2(t), bits_h2(0x2C002C00u), bits_h2(0xD480D480u)));  // 1/16, -72
}
// fp16 pair {1024 + (byte0 ^ 0x80), 1024 + (byte2 ^ 0x80)} -> minus 1152 = signed bytes.
__device__ __forceinline__ uint32_t int8_pair(uint32_t u) {
  const uint32_t t = (u & 0x00FF00FFu) ^ 0x64806480u;
  return h2_bits(__hsub2(bits_h2(t), bits_h2(0x64806480u)));  // 1152 = 1024 + 128
}

// One 16-k step: dequantize the thread's weight vectors and issue the MMAs.
// INT4: wv[0] = K-pair row c, wv[1] = row c + 4 of the step's 8 K-pair rows.
// INT8: wv[0..3] = rows 2c, 2c + 1, 2c + 8, 2c + 9 of the step's 16 rows.
template <int BITS, int MT>
__device__ __forceinline__ void wo_step(float (&acc)[MT][8][4], const uint4* wv, const uint32_t (&xb)[MT][2]) {
  if constexpr (BITS == kInt4) {
    const uint32_t wa[4] = {wv[0].x, wv[0].y, wv[0].z, wv[0].w};
    const uint32_t wb[4] = {wv[1].x, wv[1].y, wv[1].z, wv[1].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t u = __byte_perm(wa[j], wb[j], h ? 0x7632 : 0x5410);
        const uint32_t a0 = int4_lo_pair(u), a2 = int4_hi_pair(u);
        const uint32_t a1 = int4_lo_pair(u >> 8), a3 = int4_hi_pair(u >> 8);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma16816(acc[mt][2 * j + h], a0, a1, a2, a3, xb[mt][0], xb[mt][1]);
      }
    }
  } else {
    const uint32_t w0[4] = {wv[0].x, wv[0].y, wv[0].z, wv[0].w};
    const uint32_t w1[4] = {wv[1].x, wv[1].y, wv[1].z, wv[1].w};
    const uint32_t w2[4] = {wv[2].x, wv[2].y, wv[2].z, wv[2].w};
    const uint32_t w3[4] = {wv[3].x, wv[3].y, wv[3].z, wv[3].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t sel = h ? 0x7632 : 0x5410;
        const uint32_t ulo = __byte_perm(w0[j], w1[j], sel);
        const uint32_t uhi = __byte_perm(w2[j], w3[j], sel);
        const uint32_t a0 = int8_pair(ulo), a1 = int8_pair(ulo >> 8);
        const uint32_t a2 = int8_pair(uhi), a3 = int8_pair(uhi >> 8);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma16816(acc[mt][2 * j + h], a0, a1, a2, a3, xb[mt][0], xb[mt][1]);
      }
    }
  }
}

// 4 consecutive e4m3 bytes of A at k .. k+3, zero beyond K (0x7F would be NaN).
__device__ __forceinline__ uint32_t ldg_e4m3x4(const uint8_t* row, int k, int K) {
  if (k + 4 <= K) return __ldg(reinterpret_cast<const unsigned int*>(row + k));
  uint32_t w = 0;
  for (int i = 0; i < 4; ++i)
    if (k + i < K) w |= static_cast<uint32_t>(__ldg(row + k + i)) << (8 * i);
  return w;
}

// Activation fragments of one chunk (rows 8mt + g of this M tile): four
// 16-k steps of fp16 X, or two 32-k steps of e4m3 A.
template <int BITS, int MT>
__device__ __forceinline__ void load_x_chunk(uint32_t (&xb)[4][MT][2], const SkinnyArgs& p, int m_base,
                                             int k_chunk, int g, int c) {
  if constexpr (BITS == kE4m3) {
    const uint8_t* X = static_cast<const uint8_t*>(p.X);
#pragma unroll
    for (int j = 0; j < kChunkK / 32; ++j) {
      const int ka = k_chunk + 32 * j + 4 * c, kb = ka + 16;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int m = m_base + 8 * mt + g;
        const uint8_t* xr = X + static_cast<int64_t>(m) * p.ldx;
        xb[j][mt][0] = (m < p.M && ka < p.K) ? ldg_e4m3x4(xr, ka, p.K) : 0u;
        xb[j][mt][1] = (m < p.M && kb < p.K) ? ldg_e4m3x4(xr, kb, p.K) : 0u;
      }
    }
  } else {
    const __half* X = static_cast<const __half*>(p.X);
#pragma unroll
    for (int j = 0; j < kChunkK / 16; ++j) {
      const int ka = k_chunk + 16 * j + 2 * c, kb = ka + 8;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int m = m_base + 8 * mt + g;
        const bool mok = m < p.M;
        const __half* xr = X + static_cast<int64_t>(m) * p.ldx;
        const uint32_t pa = (mok && ka < p.K) ? ldg_x2(xr + ka) : 0u;
        const uint32_t pb = (mok && kb < p.K) ? ldg_x2(xr + kb) : 0u;
        if constexpr (BITS == kInt4) {
          xb[j][mt][0] = __byte_perm(pa, pb, 0x5410);  // {x[k0+2c], x[k0+2c+8]}
          xb[j][mt][1] = __byte_perm(pa, pb, 0x7632);  // {x[k0+2c+1], x[k0+2c+9]}
        } else {
          xb[j][mt][0] = pa;
          xb[j][mt][1] = pb;
        }
      }
    }
  }
}

// Barrier over the consumer warps only (the producer keeps streaming).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
}

template <int BITS, int MT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
wo_skinny_kernel(const __grid_constant__ CUtensorMap tmW, SkinnyArgs p, Plan pl, int* err) {
  using R = Ring<BITS>;
  constexpr int kRows = 8 * MT;
  constexpr int kOut = kRows * kTileN;  // outputs per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128 - (tc::smem_u32(smem_raw) & 127)) & 127);
  uint8_t* ring = smem;
  float* part = reinterpret_cast<float*>(smem + kRingBytes);  // [kRows][kTileN]
  uint64_t* full = reinterpret_cast<uint64_t*>(part + kOut);
  uint64_t* empty = full + R::kStages;
  volatile int* abort = reinterpret_cast<volatile int*>(empty + R::kStages);
  volatile int* last_flag = abort + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.x, G = gridDim.x;
  const int64_t U = pl.units;
  const int ch = pl.chunks;
  const int64_t lo = unit_lo(b, U, G);
  const int n_local = static_cast<int>(unit_lo(b + 1, U, G) - lo);

  if (threadIdx.x == 0) {
    for (int s = 0; s < R::kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 2);  // both warps of the consuming pair
    }
    *abort = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // Producer: one elected thread keeps the ring full across the CTA's run.
    if (lane == 0 && n_local > 0) {
      tc::tma_prefetch_desc(&tmW);
      int issued = 0;
      for (int i = 0; i < n_local; ++i) {
        const int64_t u = lo + i;
        const int T = static_cast<int>(u / ch), chunk = static_cast<int>(u % ch);
        const int s = i % R::kStages;
        if (!tc::mbar_wait(&empty[s], ((i / R::kStages) & 1) ^ 1, abort, err, kSiteGemmProducer)) break;
        tc::mbar_arrive_expect_tx(&full[s], R::kStageBytes);
        tc::tma_load_2d(ring + s * R::kStageBytes, &tmW, (T % pl.n_tiles) * kTileN, chunk * R::kRows, &full[s]);
        issued = i + 1;
      }
      // Let the last copies land before this thread leaves: the CTA must not
      // exit with TMA writes into its shared memory still in flight.
      for (int i = issued > R::kStages ? issued - R::kStages : 0; i < issued; ++i)
        tc::mbar_wait_drain(&full[i % R::kStages], (i / R::kStages) & 1);
    }
    return;
  }

  // Consumers: one segment per tile the run touches.
  int* ws_count = static_cast<int*>(p.ws);
  float* ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(p.ws) + kCounterBytes);
  const __half* S = static_cast<const __half*>(p.scales);
  uint32_t xb[4][MT][2];
  for (int i = 0; i < n_local;) {
    const int64_t u0 = lo + i;
    const int T = static_cast<int>(u0 / ch);
    const int64_t seg_end = static_cast<int64_t>(T + 1) * ch < lo + n_local ? static_cast<int64_t>(T + 1) * ch
                                                                             : lo + n_local;
    const int seg = static_cast<int>(seg_end - u0);
    const int m_base = (T / pl.n_tiles) * kRows, n_base = (T % pl.n_tiles) * kTileN;
    const int chunk0 = static_cast<int>(u0 - static_cast<int64_t>(T) * ch);

    float acc[MT][8][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[mt][q][r] = 0.0f;

    // Warp pair (warp >> 1) takes the chunks whose local index has its
    // parity (so it always uses the same ring slots); the two warps of a pair
    // take the two 128-column halves of the tile.
    const int half = warp & 1, pair = warp >> 1;
    for (int j = ((i & 1) == pair) ? 0 : 1; j < seg; j += kConsumers / 2) {
      const int li = i + j;
      const int s = li % R::kStages;
      load_x_chunk<BITS, MT>(xb, p, m_base, (chunk0 + j) * kChunkK, g, c);
      const bool ok = tc::mbar_wait(&full[s], (li / R::kStages) & 1, abort, err, kSiteGemmMma);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint8_t* st = ring + s * R::kStageBytes + kHalfN * half + 16 * g;
      if constexpr (BITS == kE4m3) {
#pragma unroll
        for (int q = 0; q < kChunkK / 32; ++q) {  // 32-k steps
          uint4 v[8];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            v[r] = *reinterpret_cast<const uint4*>(st + (32 * q + 4 * c + r) * kTileN);
            v[4 + r] = *reinterpret_cast<const uint4*>(st + (32 * q + 16 + 4 * c + r) * kTileN);
          }
          fp8_step<MT>(acc, v, xb[q]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < kChunkK / 16; ++q) {  // 16-k steps
          uint4 wv[BITS == kInt4 ? 2 : 4];
          if constexpr (BITS == kInt4) {
            wv[0] = *reinterpret_cast<const uint4*>(st + (8 * q + c) * kTileN);
            wv[1] = *reinterpret_cast<const uint4*>(st + (8 * q + c + 4) * kTileN);
          } else {
            wv[0] = *reinterpret_cast<const uint4*>(st + (16 * q + 2 * c) * kTileN);
            wv[1] = *reinterpret_cast<const uint4*>(st + (16 * q + 2 * c + 1) * kTileN);
            wv[2] = *reinterpret_cast<const uint4*>(st + (16 * q + 2 * c + 8) * kTileN);
            wv[3] = *reinterpret_cast<const uint4*>(st + (16 * q + 2 * c + 9) * kTileN);
          }
          wo_step<BITS, MT>(acc, wv, xb[q]);
        }
      }
      // The slot's next contents arrive through TMA (async proxy): order this
      // thread's generic-proxy reads of the slot before releasing it.
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[s]);
    }

    // Sum the two warp pairs' partial tiles in a fixed order.  acc[mt][q]
    // covers MMA rows (weight columns) 128 * half + 16g + 2q and + 1, MMA
    // columns (rows of X) 8mt + 2c and 8mt + 2c + 1.
    for (int r = 0; r < kConsumers / 2; ++r) {
      if (pair == r) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int n = kHalfN * half + 16 * g + 2 * q, m = 8 * mt + 2 * c;
            float2* p0 = reinterpret_cast<float2*>(part + m * kTileN + n);
            float2* p1 = reinterpret_cast<float2*>(part + (m + 1) * kTileN + n);
            float2 v0 = make_float2(acc[mt][q][0], acc[mt][q][2]);
            float2 v1 = make_float2(acc[mt][q][1], acc[mt][q][3]);
            if (r > 0) {
              const float2 o0 = *p0, o1 = *p1;
              v0.x += o0.x; v0.y += o0.y; v1.x += o1.x; v1.y += o1.y;
            }
            *p0 = v0;
            *p1 = v1;
          }
      }
      consumer_sync();
    }

    // Finish the tile, or hand this CTA's share to the last contributor.
    // Only the tile's valid rows travel through the workspace.
    const int f0 = unit_owner(static_cast<int64_t>(T) * ch, U, G);
    const int f1 = unit_owner(static_cast<int64_t>(T + 1) * ch - 1, U, G);
    const int contributors = f1 - f0 + 1;
    const int t = threadIdx.x;  // 0 .. 127 across the consumer warps
    const int rows_valid = p.M - m_base < kRows ? p.M - m_base : kRows;
    const int n_out = rows_valid * kTileN;
    bool finish = true;
    const float* src = part;
    if (contributors > 1) {
      float* mine = ws_part + (static_cast<size_t>(T) * pl.slots + (b - f0)) * kOut;
      for (int o = 4 * t; o < n_out; o += 4 * kConsumers * 32)
        __stcg(reinterpret_cast<float4*>(mine + o), *reinterpret_cast<const float4*>(part + o));
      __threadfence();
      consumer_sync();
      if (t == 0) *last_flag = (atomicAdd(&ws_count[T], 1) == contributors - 1);
      consumer_sync();
      finish = *last_flag != 0;
      if (finish) __threadfence();
      src = ws_part + static_cast<size_t>(T) * pl.slots * kOut;
    }
    if (finish) {
      for (int o = 4 * t; o < n_out; o += 4 * kConsumers * 32) {
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        if (contributors > 1) {
          // Eight partial tiles in flight at a time; summed in contributor order.
          for (int q0 = 0; q0 < contributors; q0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              v[u] = q0 + u < contributors
                         ? __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(q0 + u) * kOut + o))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              sum.x += v[u].x; sum.y += v[u].y; sum.z += v[u].z; sum.w += v[u].w;
            }
          }
        } else {
          sum = *reinterpret_cast<const float4*>(src + o);
        }
        const int m = o / kTileN, n = o % kTileN;
        const int gm = m_base + m;
        const float v[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int gn = n_base + n + e;
          if (gn >= p.N) continue;
          if constexpr (BITS == kE4m3)
            static_cast<__nv_bfloat16*>(p.Y)[static_cast<int64_t>(gm) * p.ldy + gn] = __float2bfloat16_rn(v[e] * p.scale);
          else
            static_cast<__half*>(p.Y)[static_cast<int64_t>(gm) * p.ldy + gn] = __float2half_rn(__half2float(S[gn]) * v[e]);
        }
      }
      if (contributors > 1 && t == 0) ws_count[T] = 0;  // ready for the next call
    }
    consumer_sync();  // `part` is rewritten by the next segment
    i += seg;
  }
}

// Opt the kernel into its dynamic shared memory (above the 48 KB default);
// must precede both the occupancy query and the first launch.
template <int BITS, int MT>
cudaError_t configure_kernel() {
  static cudaError_t status = cudaFuncSetAttribute(wo_skinny_kernel<BITS, MT>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(skinny_smem_bytes<MT>()));
  return status;
}

template <int BITS, int MT>
int ctas_per_sm() {
  static int cached = 0;
  if (cached == 0) {
    int n = 0;
    if (configure_kernel<BITS, MT>() != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, wo_skinny_kernel<BITS, MT>, kThreads,
                                                      skinny_smem_bytes<MT>()) != cudaSuccess || n < 1)
      return 1;  // not cached: a later call may succeed
    cached = n;
  }
  return cached;
}

template <int BITS, int MT>
Plan make_plan(int M, int N, int K) {
  Plan pl;
  pl.n_tiles = (N + kTileN - 1) / kTileN;
  pl.tiles = pl.n_tiles * ((M + 8 * MT - 1) / (8 * MT));
  pl.chunks = (K + kChunkK - 1) / kChunkK;
  pl.units = static_cast<int64_t>(pl.tiles) * pl.chunks;
  const int64_t cap = static_cast<int64_t>(sm_count()) * ctas_per_sm<BITS, MT>();
  pl.grid = static_cast<int>(pl.units < cap ? pl.units : cap);
  pl.slots = 1;
  if (pl.tiles > kMaxSplitTiles) {  // too many tiles for the counter area: one CTA per tile, no split
    pl.grid = pl.tiles;
    return pl;
  }
  for (int T = 0; T < pl.tiles; ++T) {
    const int n = unit_owner(static_cast<int64_t>(T + 1) * pl.chunks - 1, pl.units, pl.grid) -
                  unit_owner(static_cast<int64_t>(T) * pl.chunks, pl.units, pl.grid) + 1;
    if (n > pl.slots) pl.slots = n;
  }
  return pl;
}

template <int BITS, int MT>
size_t plan_workspace(int M, int N, int K) {
  const Plan pl = make_plan<BITS, MT>(M, N, K);
  if (pl.slots == 1) return 0;
  return kCounterBytes + static_cast<size_t>(pl.tiles) * pl.slots * (8 * MT) * kTileN * sizeof(float);
}

template <int BITS, int MT>
cudaError_t launch_variant(const SkinnyArgs& a, cudaStream_t s) {
  using R = Ring<BITS>;
  const size_t smem = skinny_smem_bytes<MT>();
  auto kern = wo_skinny_kernel<BITS, MT>;
  cudaError_t e = configure_kernel<BITS, MT>();
  if (e != cudaSuccess) return e;
  const Plan pl = make_plan<BITS, MT>(a.M, a.N, a.K);
  CUtensorMap tW;
  const uint64_t rows = BITS == kInt4 ? a.K / 2 : a.K;
  e = make_tmap_2d(&tW, a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, rows, a.ldw, kTileN, R::kRows,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  kern<<<pl.grid, kThreads, smem, s>>>(tW, a, pl, device_error_word());
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_mode(const SkinnyArgs& a, cudaStream_t s) {
  return a.M > 8 ? launch_variant<BITS, 2>(a, s) : launch_variant<BITS, 1>(a, s);
}

template <int BITS>
size_t mode_workspace(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return M > 8 ? plan_workspace<BITS, 2>(M, N, K) : plan_workspace<BITS, 1>(M, N, K);
}

}  // namespace

size_t wo_skinny_workspace(int M, int N, int K, int bits) {
  return bits == 4 ? mode_workspace<kInt4>(M, N, K) : mode_workspace<kInt8>(M, N, K);
}

size_t fp8_skinny_workspace(int M, int N, int K) { return mode_workspace<kE4m3>(M, N, K); }

cudaError_t launch_wo_skinny(const WoArgs& a, int bits, cudaStream_t s) {
  if (a.K == 0) return cudaMemset2DAsync(a.Y, a.ldy * 2, 0, static_cast<size_t>(a.N) * 2, a.M, s);
  const SkinnyArgs sa{a.M, a.N, a.K, a.X, a.ldx, a.W, a.ldw, a.scales, 1.0f, a.Y, a.ldy, a.ws};
  return bits == 4 ? launch_mode<kInt4>(sa, s) : launch_mode<kInt8>(sa, s);
}

cudaError_t launch_fp8_skinny(const Fp8GemmArgs& a, void* ws, cudaStream_t s) {
  if (a.K == 0) return cudaMemset2DAsync(a.C, a.ldc * 2, 0, static_cast<size_t>(a.N) * 2, a.M, s);
  const SkinnyArgs sa{a.M, a.N, a.K, a.A, a.lda, a.B, a.ldb, nullptr, a.scale_a * a.scale_b, a.C, a.ldc, ws};
  return launch_mode<kE4m3>(sa, s);
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
