// Weight-only GEMM for small M (decode): W4A16 and W8A16.
//
// Defined by "Triton 工业级融合微算子编写：W4A16 极速切片矩阵乘与 Blackwell NVFP4
// 硬件指令实装" §二 (INT4: byte row k/2, even k in the low nibble, weight
// (q - 8) * s[n], FP32 accumulation, FP16 output) and "Triton 量化算子：W8A16
// 权重量化融合矩阵乘法" Step 1 / Step 3 (INT8: Y = X (W_int8 S), W [K, N]).
//
// Design (HBM-bound; the packed weights are read exactly once):
//   * A warp owns 128 output columns and a slice of K.  Each thread streams
//     16-byte vectors of packed weights with non-allocating 128-bit loads
//     (a warp covers 128 contiguous bytes per weight row), a whole slice of
//     loads in flight before any math.
//   * The weights are dequantized in registers straight into the A operand
//     of mma.sync.m16n8k16 (Y^T = W^T X^T: weight columns are the MMA rows,
//     the M <= 16 activation rows the MMA columns).  The dequantized weight
//     never touches shared or global memory.  INT4 codes become exact fp16
//     (q - 8) with one LOP3 (0x6400 | nibble = 1024 + nibble) and one
//     HSUB2/HFMA2 per two weights; INT8 with one LOP3 (byte ^ 0x80 | 0x6400)
//     and one HSUB2.  The per-column scale factors out of the K sum and is
//     applied once in the epilogue (exact reordering: it is per column).
//   * Split-K: the warps of a CTA take different K slices and reduce through
//     shared memory; the CTAs of a thread-block cluster (up to 8) take
//     further slices and reduce through distributed shared memory, each CTA
//     finishing a 1/C share of the columns.  No workspace, one launch.
//   * INT4 MMA k-order: a register of the A fragment holds the low (or high)
//     nibbles of the same byte column from K-pair rows c and c + 4, so one
//     PRMT serves four weights; the activation fragment is permuted to the
//     same k order (k0+2c, k0+2c+8 | k0+2c+1, k0+2c+9).
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "wq_internal.h"

namespace cg = cooperative_groups;

namespace wq {
namespace {

constexpr int kTileN = 128;       // output columns per warp (and per CTA)
constexpr int kRedPad = 4;        // shared-memory row padding (floats)

__device__ __forceinline__ uint4 ldg_stream16(const uint8_t* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16 bytes at p, of which only the first `valid` (0..16) are read.
__device__ __forceinline__ uint4 ldg_vec16(const uint8_t* p, int valid) {
  if (valid >= 16) return ldg_stream16(p);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  for (int i = 0; i < valid; ++i) w[i >> 2] |= static_cast<uint32_t>(p[i]) << (8 * (i & 3));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t ldg_x2(const __half* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
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

template <int BITS>
struct WoTraits;
template <>
struct WoTraits<4> {
  static constexpr int kVecs = 2;    // 16-byte weight vectors per thread per 16-k step
  static constexpr int kDepth = 8;   // steps whose loads are in flight together
};
template <>
struct WoTraits<8> {
  static constexpr int kVecs = 4;
  static constexpr int kDepth = 4;
};

// One 16-k step: dequantize the thread's weight vectors and issue the MMAs.
template <int BITS, int MT>
__device__ __forceinline__ void wo_step(float (&acc)[MT][8][4], const uint4 (&wv)[WoTraits<BITS>::kVecs],
                                        const uint32_t (&xb)[MT][2]) {
  if constexpr (BITS == 4) {
    const uint32_t wa[4] = {wv[0].x, wv[0].y, wv[0].z, wv[0].w};  // K-pair row c
    const uint32_t wb[4] = {wv[1].x, wv[1].y, wv[1].z, wv[1].w};  // K-pair row c + 4
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
    const uint32_t w0[4] = {wv[0].x, wv[0].y, wv[0].z, wv[0].w};  // row k0 + 2c
    const uint32_t w1[4] = {wv[1].x, wv[1].y, wv[1].z, wv[1].w};  // row k0 + 2c + 1
    const uint32_t w2[4] = {wv[2].x, wv[2].y, wv[2].z, wv[2].w};  // row k0 + 2c + 8
    const uint32_t w3[4] = {wv[3].x, wv[3].y, wv[3].z, wv[3].w};  // row k0 + 2c + 9
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

// grid.x = n_tiles * C (cluster of C CTAs per 128-column tile), grid.y = M tiles
// of 8 * MT rows.  Dynamic shared memory: partial tiles of every warp plus
// the CTA's reduced tile.
template <int BITS, int MT, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
wo_skinny_kernel(WoArgs p) {
  using T = WoTraits<BITS>;
  constexpr int kRows = 8 * MT;
  constexpr int kLd = kTileN + kRedPad;
  extern __shared__ float smem[];
  float* red = smem;                              // [WARPS][kRows][kLd]
  float* part = smem + WARPS * kRows * kLd;       // [kRows][kTileN]

  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int tile = blockIdx.x / C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int n_base = tile * kTileN;
  const int m_base = blockIdx.y * kRows;

  const int steps = (p.K + 15) / 16;
  const int slices = C * WARPS;
  const int slice = rank * WARPS + warp;
  const int s_begin = static_cast<int>((static_cast<int64_t>(steps) * slice) / slices);
  const int s_end = static_cast<int>((static_cast<int64_t>(steps) * (slice + 1)) / slices);

  const uint8_t* W = static_cast<const uint8_t*>(p.W);
  const __half* X = static_cast<const __half*>(p.X);
  const int col = n_base + 16 * g;
  const int col_valid = min(16, max(0, p.N - col));
  const int w_rows = BITS == 4 ? p.K / 2 : p.K;

  float acc[MT][8][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[mt][i][r] = 0.0f;

  for (int s0 = s_begin; s0 < s_end; s0 += T::kDepth) {
    uint4 wv[T::kDepth][T::kVecs];
    uint32_t xb[T::kDepth][MT][2];
#pragma unroll
    for (int d = 0; d < T::kDepth; ++d) {
      const int st = s0 + d;
      const bool live = st < s_end;
      const int k0 = st * 16;
#pragma unroll
      for (int v = 0; v < T::kVecs; ++v) {
        int row;
        if constexpr (BITS == 4) row = k0 / 2 + c + 4 * v;
        else row = k0 + 2 * c + (v & 1) + 8 * (v >> 1);
        const bool ok = live && row < w_rows && col_valid > 0;
        wv[d][v] = ok ? ldg_vec16(W + static_cast<int64_t>(row) * p.ldw + col, col_valid) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int m = m_base + 8 * mt + g;
        const bool mok = live && m < p.M;
        const __half* xr = X + static_cast<int64_t>(m) * p.ldx;
        const int ka = k0 + 2 * c, kb = k0 + 2 * c + 8;
        const uint32_t pa = (mok && ka < p.K) ? ldg_x2(xr + ka) : 0u;
        const uint32_t pb = (mok && kb < p.K) ? ldg_x2(xr + kb) : 0u;
        if constexpr (BITS == 4) {
          xb[d][mt][0] = __byte_perm(pa, pb, 0x5410);  // {x[k0+2c], x[k0+2c+8]}
          xb[d][mt][1] = __byte_perm(pa, pb, 0x7632);  // {x[k0+2c+1], x[k0+2c+9]}
        } else {
          xb[d][mt][0] = pa;
          xb[d][mt][1] = pb;
        }
      }
    }
#pragma unroll
    for (int d = 0; d < T::kDepth; ++d) wo_step<BITS, MT>(acc, wv[d], xb[d]);
  }

  // Per-warp partial tiles -> shared memory.  acc[mt][i] covers MMA rows
  // (weight columns) 16g + 2i and 16g + 2i + 1, MMA columns (rows of X)
  // 8mt + 2c and 8mt + 2c + 1.
  float* rw = red + warp * kRows * kLd;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int n = 16 * g + 2 * i;
      const int m = 8 * mt + 2 * c;
      *reinterpret_cast<float2*>(rw + m * kLd + n) = make_float2(acc[mt][i][0], acc[mt][i][2]);
      *reinterpret_cast<float2*>(rw + (m + 1) * kLd + n) = make_float2(acc[mt][i][1], acc[mt][i][3]);
    }
  __syncthreads();
  for (int o = threadIdx.x; o < kRows * kTileN; o += WARPS * 32) {
    const int m = o / kTileN, n = o % kTileN;
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) sum += red[(w * kRows + m) * kLd + n];
    part[o] = sum;
  }
  // Cluster-wide reduction: CTA `rank` finishes columns [lo, hi) of the tile
  // from every CTA's reduced tile (distributed shared memory).
  cluster.sync();
  const int span = kTileN / C;
  const int lo = rank * span, hi = (rank == C - 1) ? kTileN : lo + span;
  const __half* S = static_cast<const __half*>(p.scales);
  __half* Y = static_cast<__half*>(p.Y);
  for (int o = threadIdx.x; o < kRows * (hi - lo); o += WARPS * 32) {
    const int m = o / (hi - lo), n = lo + o % (hi - lo);
    float sum = 0.0f;
    for (int q = 0; q < C; ++q) sum += cluster.map_shared_rank(part, q)[m * kTileN + n];
    const int gm = m_base + m, gn = n_base + n;
    if (gm < p.M && gn < p.N)
      Y[static_cast<int64_t>(gm) * p.ldy + gn] = __float2half_rn(__half2float(S[gn]) * sum);
  }
  cluster.sync();  // keep every CTA's shared memory alive until all reads are done
}

template <int BITS, int MT, int WARPS>
cudaError_t launch_variant(const WoArgs& a, int C, cudaStream_t s) {
  constexpr int kRows = 8 * MT;
  const size_t smem = sizeof(float) * (WARPS * kRows * (kTileN + kRedPad) + kRows * kTileN);
  auto kern = wo_skinny_kernel<BITS, MT, WARPS>;
  static bool configured = false;  // per instantiation; a benign race sets it twice
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int n_tiles = (a.N + kTileN - 1) / kTileN;
  const int m_tiles = (a.M + kRows - 1) / kRows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_tiles * C), static_cast<unsigned>(m_tiles), 1);
  cfg.blockDim = dim3(WARPS * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

int wo_skinny_max_m() { return 16; }

// Split-K heuristic: one warp per (128 columns, K slice); enough warps to keep
// about 16 per SM busy, at least two 16-k steps per warp, clusters of 1..8.
int wo_skinny_cluster(int N, int K, int warps) {
  const int n_tiles = (N + kTileN - 1) / kTileN;
  const int steps = (K + 15) / 16;
  const int target_warps = sm_count() * 16;
  int C = target_warps / (n_tiles * warps);
  C = C < 1 ? 1 : (C > 8 ? 8 : C);
  while (C > 1 && steps < 2 * C * warps) --C;
  return C;
}

cudaError_t launch_wo_skinny(const WoArgs& a, int bits, cudaStream_t s) {
  constexpr int kWarps = 8;
  const int C = wo_skinny_cluster(a.N, a.K, kWarps);
  const bool two = a.M > 8;
  if (bits == 4) return two ? launch_variant<4, 2, kWarps>(a, C, s) : launch_variant<4, 1, kWarps>(a, C, s);
  return two ? launch_variant<8, 2, kWarps>(a, C, s) : launch_variant<8, 1, kWarps>(a, C, s);
}

}  // namespace wq
