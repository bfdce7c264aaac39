// Device pieces shared by the skinny weight-stream kernels (the per-call
// kernel in wo_skinny.cu and the batched one in wo_batched.cu): tile and ring
// geometry, the fragment loads, the in-register dequantization and mma.sync
// steps, and the epilogue stores.  Everything sits in an unnamed namespace, so
// every translation unit that includes this gets its own copy.
//
// Defined by "Triton 工业级融合微算子编写：W4A16 极速切片矩阵乘与 Blackwell NVFP4
// 硬件指令实装" §二 (INT4 codes, even k in the low nibble, (q - 8) * s[n]),
// "Triton 量化算子：W8A16 权重量化融合矩阵乘法" Step 1 / Step 3 (INT8, W [K, N])
// and "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核" (e4m3 operands).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_common.cuh"

namespace wq {
namespace {

constexpr int kTileN = 128;                  // output columns per tile = bytes per weight box row
constexpr int kBoxRows = 32;                 // packed weight rows per unit
constexpr int kWBytes = kBoxRows * kTileN;   // 4 KB of packed weights per unit
constexpr int kWarps = 12;                   // warps per CTA; each loads and consumes its own units
constexpr int kThreads = kWarps * 32;
constexpr int kRedRounds = 3;                // rounds of the in-CTA reduction
constexpr int kRedBufs = kWarps / kRedRounds;  // shared-memory partial tiles
static_assert(kWarps % kRedRounds == 0, "reduction rounds must split the warps evenly");
constexpr int kSmemLimit = 227 * 1024;
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
  const void* zeros;  // weight-only: one zero point per column group, or nullptr
  int group_n;        // weight-only: columns per scale / zero-point group
  uint64_t wait_ns = 2000000000ull;  // limit of a bounded wait before the kernel gives up
  // The caller promised static weights (wq_set_static_weights): the first
  // weight boxes may be loaded before the grid dependency wait.
  int early_w = 0;
};

// The deepest per-warp ring (2..8 slots) whose slots, one 8-byte barrier
// each, and the fixed areas fit in the shared-memory budget.
constexpr int ring_depth(int slot_bytes, int fixed_bytes) {
  int d = 8;
  while (d > 2 && kWarps * d * (slot_bytes + 8) + fixed_bytes > kSmemLimit) --d;
  return d;
}

template <int BITS, int MT>
struct Cfg {
  static constexpr int kChunkK = BITS == kInt4 ? 64 : 32;   // k per unit
  static constexpr int kXRowBytes = kChunkK * (BITS == kE4m3 ? 1 : 2);  // 128, 64 or 32
  static constexpr int kRows = 8 * MT;                      // activation rows per M tile
  static constexpr int kXBytes = kRows * kXRowBytes;        // activation box
  static constexpr int kXAlloc = (kXBytes + 1023) / 1024 * 1024;
  static constexpr int kSlotBytes = kWBytes + kXAlloc;      // 1 KB multiple: swizzle atoms stay aligned
  static constexpr int kOutF4 = MT * 8 * 32;                // float4 per partial tile (lane-native)
  static constexpr int kRedBytes = kRedBufs * kOutF4 * 16;
  static constexpr int kRxBytes = kOutF4 * 16;              // cluster peers' slices of the partial tile
  static constexpr int kFacBytes = 2 * kTileN * 4;          // the tile's output and zero-point factors
  static constexpr int kFixedBytes = kRedBytes + kRxBytes + kFacBytes + 1024 + 64;  // + alignment slack, flags
  // Units in flight per warp: as many as fit in shared memory (two to eight).
  static constexpr int kDepth = ring_depth(kSlotBytes, kFixedBytes);
  static constexpr int kStages = kWarps * kDepth;
  static constexpr int kRingBytes = kStages * kSlotBytes;
  static constexpr size_t kSmemBytes = kRingBytes + kStages * 8 + kFixedBytes;
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
};

// Offset of byte `o` of a densely packed box after the TMA swizzle whose span
// is `cpr` 16-byte chunks (2, 4, 8 for 32, 64, 128 bytes): the chunk index
// (bits 4..) is XORed with bits 7.. of the offset.  Boxes sit 1 KB aligned.
__device__ __forceinline__ int swz(int o, int cpr) { return o ^ (((o >> 7) & (cpr - 1)) << 4); }


__host__ __device__ __forceinline__ int64_t unit_lo(int b, int64_t U, int G) { return (int64_t)b * U / G; }
// The CTA whose run contains unit u.
__host__ __device__ __forceinline__ int unit_owner(int64_t u, int64_t U, int G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
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

// One 32-k step of e4m3: v[0..3] feed k slots 4c .. 4c+3 and v[4..7] slots
// 16 + 4c .. 16 + 4c + 3, 16 columns each.  MMA i takes columns 2i (MMA row
// g) and 2i + 1 (row g + 8).
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
// fp16 pair {1024 + (byte0 ^ 0x80), 1024 + (byte2 ^ 0x80)} = 1152 + the signed
// bytes (exact).  The offset is not subtracted here: the MMA sums
// (1152 + w) x, and one extra MMA per k step with a constant -1152 operand
// (kInt8Offset) takes 1152 * sum(x) back out, in FP32.
__device__ __forceinline__ uint32_t int8_pair(uint32_t u) { return (u & 0x00FF00FFu) ^ 0x64806480u; }
constexpr uint32_t kInt8Offset = 0xE480E480u;  // fp16 pair {-1152, -1152}
constexpr uint32_t kOnes = 0x3C003C00u;        // fp16 pair {1, 1}

// One 16-k step: dequantize the thread's weight vectors and issue the MMAs.
// INT4: wv[0], wv[1] = K-pair rows 2c, 2c + 1 of the step's 8 (k = 4c ..
//   4c + 3); slots (2c, 2c+1) take k (4c, 4c+2) and slots (2c+8, 2c+9) take
//   k (4c+1, 4c+3).
// INT8: wv[0..3] = rows 2c, 2c + 1, 2c + 8, 2c + 9 of the step's 16 (natural
//   k order).
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

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint32_t lds16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

// One unit, held in registers: the thread's 8 weight vectors (16 bytes each)
// and its activation fragments.  Reading the whole unit out of its ring slot
// first lets the slot be refilled while the math runs.
template <int BITS, int MT>
struct UnitRegs {
  static constexpr int kXWords = BITS == kInt4 ? 4 * MT * 2 : (BITS == kInt8 ? 2 * MT * 2 : MT * 2);
  uint4 w[8];
  uint32_t x[kXWords];
};

// Load one unit from its ring slot: w = 32 swizzled weight rows of 128 bytes,
// x = the swizzled activation box (row m = 8 mt + g of this M tile).  The
// thread's 16-byte column group is g; rows r with r % 8 == 2c sit at swizzled
// column o0, rows with r % 8 == 2c + 1 at o1.
template <int BITS, int MT>
__device__ __forceinline__ void load_unit(UnitRegs<BITS, MT>& u, const uint8_t* w, const uint8_t* x, int g, int c) {
  using C = Cfg<BITS, MT>;
  constexpr int cpr = C::kXRowBytes / 16;
  const int o0 = (g ^ (2 * c)) << 4, o1 = (g ^ (2 * c + 1)) << 4;
  if constexpr (BITS == kE4m3) {
    // Slots 4c .. 4c+3 <- rows 2c, 2c+1, 2c+8, 2c+9; slots 16+4c .. <- rows
    // 2c+16, 2c+17, 2c+24, 2c+25: activation bytes at the same k.
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int r = (8 * mt + g) * C::kXRowBytes + 2 * c;
      u.x[2 * mt] = lds16(x + swz(r, cpr)) | (lds16(x + swz(r + 8, cpr)) << 16);
      u.x[2 * mt + 1] = lds16(x + swz(r + 16, cpr)) | (lds16(x + swz(r + 24, cpr)) << 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = 2 * c + 8 * i;  // rows row, row + 1
      u.w[(i & 1) * 2 + (i >> 1) * 4] = lds128(w + row * kTileN + o0);
      u.w[(i & 1) * 2 + (i >> 1) * 4 + 1] = lds128(w + (row + 1) * kTileN + o1);
    }
  } else if constexpr (BITS == kInt8) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int r = (8 * mt + g) * C::kXRowBytes + 32 * q + 4 * c;
        u.x[(q * MT + mt) * 2] = lds32(x + swz(r, cpr));           // k 16q + 2c, +1
        u.x[(q * MT + mt) * 2 + 1] = lds32(x + swz(r + 16, cpr));  // k 16q + 2c + 8, +9
      }
      const int row = 16 * q + 2 * c;
      u.w[4 * q] = lds128(w + row * kTileN + o0);
      u.w[4 * q + 1] = lds128(w + (row + 1) * kTileN + o1);
      u.w[4 * q + 2] = lds128(w + (row + 8) * kTileN + o0);
      u.w[4 * q + 3] = lds128(w + (row + 9) * kTileN + o1);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint2 pp = lds64(x + swz((8 * mt + g) * C::kXRowBytes + 32 * q + 8 * c, cpr));  // k 16q + 4c .. +3
        u.x[(q * MT + mt) * 2] = __byte_perm(pp.x, pp.y, 0x5410);      // {x[4c], x[4c+2]}
        u.x[(q * MT + mt) * 2 + 1] = __byte_perm(pp.x, pp.y, 0x7632);  // {x[4c+1], x[4c+3]}
      }
      const int row = 8 * q + 2 * c;
      u.w[2 * q] = lds128(w + row * kTileN + o0);
      u.w[2 * q + 1] = lds128(w + (row + 1) * kTileN + o1);
    }
  }
}

// The math of one unit from registers.  kSumX (INT4 with zero points): one
// extra MMA per k step against a constant 1.0 operand sums the activations
// into corr, for the zero-point correction.
template <int BITS, int MT, bool kSumX = false>
__device__ __forceinline__ void compute_unit(float (&acc)[MT][8][4], float (&corr)[MT][4], const UnitRegs<BITS, MT>& u) {
  if constexpr (BITS == kE4m3) {
    uint32_t xb[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      xb[mt][0] = u.x[2 * mt];
      xb[mt][1] = u.x[2 * mt + 1];
    }
    fp8_step<MT>(acc, u.w, xb);
  } else {
    constexpr int kSteps = BITS == kInt4 ? 4 : 2;
    constexpr int kVec = 8 / kSteps;  // weight vectors per 16-k step
#pragma unroll
    for (int q = 0; q < kSteps; ++q) {
      uint32_t xb[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        xb[mt][0] = u.x[(q * MT + mt) * 2];
        xb[mt][1] = u.x[(q * MT + mt) * 2 + 1];
      }
      wo_step<BITS, MT>(acc, u.w + kVec * q, xb);
      if constexpr (BITS == kInt8) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          mma16816(corr[mt], kInt8Offset, kInt8Offset, kInt8Offset, kInt8Offset, xb[mt][0], xb[mt][1]);
      } else if constexpr (kSumX) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma16816(corr[mt], kOnes, kOnes, kOnes, kOnes, xb[mt][0], xb[mt][1]);
      }
    }
  }
}

// Write two adjacent outputs (row gm, columns gn and gn + 1) of the final
// result, skipping columns at or beyond N; f = the factors of the two columns.
template <int BITS>
__device__ __forceinline__ void store_pair(const SkinnyArgs& p, int gm, int gn, float v0, float v1, float2 f) {
  if (gn >= p.N) return;
  const bool two = gn + 1 < p.N;
  if constexpr (BITS == kE4m3) {
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.Y) + static_cast<int64_t>(gm) * p.ldy + gn;
    if (two)
      *reinterpret_cast<__nv_bfloat162*>(y) = __floats2bfloat162_rn(v0 * f.x, v1 * f.y);
    else
      *y = __float2bfloat16_rn(v0 * f.x);
  } else {
    __half* y = static_cast<__half*>(p.Y) + static_cast<int64_t>(gm) * p.ldy + gn;
    if (two)
      *reinterpret_cast<__half2*>(y) = __floats2half2_rn(f.x * v0, f.y * v1);
    else
      *y = __float2half_rn(f.x * v0);
  }
}

// Lane-native partial element e = (mt * 8 + q) * 32 + lane holds acc[mt][q]
// of that lane: rows 8mt + 2c (.x, .z) and 8mt + 2c + 1 (.y, .w), columns
// 16g + 2q (.x, .y) and 16g + 2q + 1 (.z, .w), with g = lane / 4, c = lane % 4.
__device__ __forceinline__ int elem_col(int e) { return 16 * ((e & 31) >> 2) + 2 * ((e >> 5) & 7); }

// The output factors of element e's two columns: the per-column scales
// (weight-only) or scale_a * scale_b (e4m3); columns at or beyond N read 0.
template <int BITS>
__device__ __forceinline__ float2 elem_factors(const SkinnyArgs& p, int e, int n_base) {
  if constexpr (BITS == kE4m3) {
    return make_float2(p.scale, p.scale);
  } else {
    const int gn = n_base + elem_col(e);
    const __half* S = static_cast<const __half*>(p.scales);
    return make_float2(gn < p.N ? __half2float(S[gn / p.group_n]) : 0.0f,
                       gn + 1 < p.N ? __half2float(S[(gn + 1) / p.group_n]) : 0.0f);
  }
}

template <int BITS>
__device__ __forceinline__ void store_elem(const SkinnyArgs& p, int e, int m_base, int n_base, float4 v, float2 f) {
  const int gm = m_base + 8 * (e >> 8) + 2 * (e & 3), gn = n_base + elem_col(e);
  if (gm < p.M) store_pair<BITS>(p, gm, gn, v.x, v.z, f);
  if (gm + 1 < p.M) store_pair<BITS>(p, gm + 1, gn, v.y, v.w, f);
}


__device__ __forceinline__ bool elem_live(int e, int rows_valid) { return 8 * (e >> 8) + 2 * (e & 3) < rows_valid; }

__device__ __forceinline__ float4 f4add(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// Barrier over the CTA's warps (all of them load and consume).
// All kThreads threads of the CTA, on barrier 1 (barrier 0 is cta_barrier's).
// Non-aligned: it counts threads, so lanes of a warp may arrive apart.
__device__ __forceinline__ void cta_sync() {
  asm volatile("barrier.sync 1, %0;" ::"n"(kThreads) : "memory");
}

}  // namespace
}  // namespace wq
