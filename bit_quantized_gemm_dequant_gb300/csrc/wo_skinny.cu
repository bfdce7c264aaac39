// Weight-only GEMM for small M (decode): W4A16 and W8A16.
//
// Defined by "Triton 工业级融合微算子编写：W4A16 极速切片矩阵乘与 Blackwell NVFP4
// 硬件指令实装" §二 (INT4: byte row k/2, even k in the low nibble, weight
// (q - 8) * s[n], FP32 accumulation, FP16 output) and "Triton 量化算子：W8A16
// 权重量化融合矩阵乘法" Step 1 / Step 3 (INT8: Y = X (W_int8 S), W [K, N]).
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
#include <cuda_fp16.h>

#include <mutex>

#include "tc_common.cuh"
#include "tma_host.h"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kTileN = 128;       // output columns per CTA
constexpr int kChunkK = 64;       // k per pipeline stage
constexpr int kRingBytes = 64 * 1024;
constexpr int kConsumers = 4;     // consumer warps (plus one producer warp)
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kCtasPerSm = 3;
// Workspace layout: a fixed counter area first (one int per tile, at most
// kMaxSplitTiles tiles), so that the counters of any shape sit in bytes that
// every call leaves zero; the partial tiles follow.
constexpr int kMaxSplitTiles = 16384;
constexpr size_t kCounterBytes = kMaxSplitTiles * sizeof(int);

template <int BITS>
struct Ring {
  static constexpr int kRows = BITS == 4 ? kChunkK / 2 : kChunkK;  // rows of the packed tile
  static constexpr int kStageBytes = kRows * kTileN;
  static constexpr int kStages = kRingBytes / kStageBytes;
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
  if constexpr (BITS == 4) {
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

// Activation fragments of the 4 steps of one chunk (rows 8mt + g of this M tile).
template <int BITS, int MT>
__device__ __forceinline__ void load_x_chunk(uint32_t (&xb)[4][MT][2], const WoArgs& p, int m_base, int k_chunk,
                                             int g, int c) {
  const __half* X = static_cast<const __half*>(p.X);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int ka = k_chunk + 16 * j + 2 * c, kb = ka + 8;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int m = m_base + 8 * mt + g;
      const bool mok = m < p.M;
      const __half* xr = X + static_cast<int64_t>(m) * p.ldx;
      const uint32_t pa = (mok && ka < p.K) ? ldg_x2(xr + ka) : 0u;
      const uint32_t pb = (mok && kb < p.K) ? ldg_x2(xr + kb) : 0u;
      if constexpr (BITS == 4) {
        xb[j][mt][0] = __byte_perm(pa, pb, 0x5410);  // {x[k0+2c], x[k0+2c+8]}
        xb[j][mt][1] = __byte_perm(pa, pb, 0x7632);  // {x[k0+2c+1], x[k0+2c+9]}
      } else {
        xb[j][mt][0] = pa;
        xb[j][mt][1] = pb;
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
wo_skinny_kernel(const __grid_constant__ CUtensorMap tmW, WoArgs p, Plan pl, int* err) {
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
      tc::mbar_init(&empty[s], 1);
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
      if (*abort)
        for (int i = issued > R::kStages ? issued - R::kStages : 0; i < issued; ++i)
          tc::mbar_wait_drain(&full[i % R::kStages], (i / R::kStages) & 1);
    }
    return;
  }

  // Consumers: one segment per tile the run touches.
  int* ws_count = static_cast<int*>(p.ws);
  float* ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(p.ws) + kCounterBytes);
  const __half* S = static_cast<const __half*>(p.scales);
  __half* Y = static_cast<__half*>(p.Y);
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

    for (int j = warp; j < seg; j += kConsumers) {
      const int li = i + j;
      const int s = li % R::kStages;
      load_x_chunk<BITS, MT>(xb, p, m_base, (chunk0 + j) * kChunkK, g, c);
      const bool ok = tc::mbar_wait(&full[s], (li / R::kStages) & 1, abort, err, kSiteGemmMma);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint8_t* st = ring + s * R::kStageBytes + 16 * g;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 wv[BITS == 4 ? 2 : 4];
        if constexpr (BITS == 4) {
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
      // The slot's next contents arrive through TMA (async proxy): order this
      // thread's generic-proxy reads of the slot before releasing it.
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[s]);
    }

    // Sum the consumer warps' partial tiles in a fixed order.  acc[mt][q]
    // covers MMA rows (weight columns) 16g + 2q and 16g + 2q + 1, MMA columns
    // (rows of X) 8mt + 2c and 8mt + 2c + 1.
    for (int r = 0; r < kConsumers; ++r) {
      if (warp == r) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int n = 16 * g + 2 * q, m = 8 * mt + 2 * c;
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
    const int f0 = unit_owner(static_cast<int64_t>(T) * ch, U, G);
    const int f1 = unit_owner(static_cast<int64_t>(T + 1) * ch - 1, U, G);
    const int contributors = f1 - f0 + 1;
    const int t = threadIdx.x;  // 0 .. 127 across the consumer warps
    bool finish = true;
    const float* src = part;
    if (contributors > 1) {
      float* mine = ws_part + (static_cast<size_t>(T) * pl.slots + (b - f0)) * kOut;
      for (int o = 4 * t; o < kOut; o += 4 * kConsumers * 32)
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
      for (int o = 4 * t; o < kOut; o += 4 * kConsumers * 32) {
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        if (contributors > 1) {
          for (int q = 0; q < contributors; ++q) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(q) * kOut + o));
            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
          }
        } else {
          sum = *reinterpret_cast<const float4*>(src + o);
        }
        const int m = o / kTileN, n = o % kTileN;
        const int gm = m_base + m;
        const float v[4] = {sum.x, sum.y, sum.z, sum.w};
        if (gm < p.M)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int gn = n_base + n + e;
            if (gn < p.N) Y[static_cast<int64_t>(gm) * p.ldy + gn] = __float2half_rn(__half2float(S[gn]) * v[e]);
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
cudaError_t launch_variant(const WoArgs& a, cudaStream_t s) {
  using R = Ring<BITS>;
  const size_t smem = skinny_smem_bytes<MT>();
  auto kern = wo_skinny_kernel<BITS, MT>;
  cudaError_t e = configure_kernel<BITS, MT>();
  if (e != cudaSuccess) return e;
  const Plan pl = make_plan<BITS, MT>(a.M, a.N, a.K);
  CUtensorMap tW;
  const uint64_t rows = BITS == 4 ? a.K / 2 : a.K;
  e = make_tmap_2d(&tW, a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, rows, a.ldw, kTileN, R::kRows,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  kern<<<pl.grid, kThreads, smem, s>>>(tW, a, pl, device_error_word());
  return cudaGetLastError();
}

}  // namespace

size_t wo_skinny_workspace(int M, int N, int K, int bits) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const bool two = M > 8;
  if (bits == 4) return two ? plan_workspace<4, 2>(M, N, K) : plan_workspace<4, 1>(M, N, K);
  return two ? plan_workspace<8, 2>(M, N, K) : plan_workspace<8, 1>(M, N, K);
}

cudaError_t launch_wo_skinny(const WoArgs& a, int bits, cudaStream_t s) {
  if (a.K == 0) return cudaMemset2DAsync(a.Y, a.ldy * 2, 0, static_cast<size_t>(a.N) * 2, a.M, s);
  const bool two = a.M > 8;
  if (bits == 4) return two ? launch_variant<4, 2>(a, s) : launch_variant<4, 1>(a, s);
  return two ? launch_variant<8, 2>(a, s) : launch_variant<8, 1>(a, s);
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
