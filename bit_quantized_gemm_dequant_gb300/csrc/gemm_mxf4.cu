// MXFP4 GEMM C = A * W^T on the block-scaled 5th-generation tensor cores.
//
// Defined by "量化推理引擎中的微缩放格式前瞻：MXFP4 矩阵乘法 Kernel 原理": §二.1
// (block dot product dC = S_A S_W sum_{i<32} a w over each 32-element K block)
// and §二.2 (S_A S_W = 2^(E_A + E_W - 254)); §三: C = A @ W^T, A [M, K],
// W [N, K], both split along K into 32-element E2M1 blocks with one E8M0
// exponent each.
//
// The page's CPU simulator adds exponents and shifts in software; here the
// exponent addition happens inside tcgen05.mma.kind::mxf4.block_scale: the
// E2M1 operands stay packed (two per byte) from HBM to the tensor core, and
// the UE8M0 block scales ride along in tensor memory.
//
// Design: one 128 x 256 output tile per CTA, K in 256-element (128-byte)
// steps through a 4-stage ring.
//   warp 0      producer.  Lane 0 issues the TMA loads of the A and W data
//               tiles (A 128 rows, W 256 rows, x 128 bytes, 128-byte swizzle)
//               and three bulk copies of the step's scale chunks (A's row
//               group, W's two), all counted on the stage's one barrier.  The
//               scales arrive already in the tensor cores' chunk layout
//               (fp4_scales.cu), so the stage is ready for the MMA warp the
//               moment it lands.
//   warp 1      TMEM allocator and MMA issuer: per stage, six (MXFP4) or
//               twelve (NVFP4) tcgen05.cp 32x128b.warpx4 (scale chunks ->
//               TMEM) and four tcgen05.mma 128 x 256 x 64 (one per 64-element
//               K slice; the A tile is read once per slice), the scale bytes
//               chosen by the descriptor's scale-factor ids.
//   warps 2-5   epilogue: tcgen05.ld and FP32 stores.
#include "mx_block.cuh"
#include "tc_common.cuh"
#include "tma_host.h"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int BM = 128, BN = 256;
constexpr int BKB = 128;                    // K bytes per stage (256 E2M1 elements)
constexpr int kStages = 4;
constexpr int kABytes = BM * BKB;           // 16 KB
constexpr int kBBytes = BN * BKB;           // 32 KB
constexpr int kSfChunk = kTcSfChunk;        // 128 rows x 4 scale bytes
constexpr int kSfBytes = 12 * kSfChunk;     // 6 KB: the step's scale chunks (NVFP4 12, MXFP4 6)
constexpr int kStageBytes = kABytes + kBBytes + kSfBytes;  // 54 KB (multiple of 1024)
constexpr int kAccCols = BN;                // FP32 accumulator columns
constexpr int kTmemCols = 512;              // accumulator + 4 stages of scale columns, rounded up
constexpr int kThreads = 192;
constexpr int kBarOffset = kStages * kStageBytes;  // barriers after the ring
constexpr int kSmemBytes = kBarOffset + 1024 + 1024;

// The two FP4 formats.  MXFP4: 32-element blocks with E8M0 scales, 8 scale
// bytes per row per K step (two chunks per row group), scales in pairs per
// TMEM word (scale_vec::2X).  NVFP4: 16-element blocks with E4M3 scales, 16
// scale bytes per row per K step (four chunks per row group), one TMEM word
// of four scales per MMA (scale_vec::4X), and two FP32 tensor scales applied
// in the epilogue.
template <bool kNv>
struct Fmt {
  static constexpr int kBlock = kNv ? 16 : 32;          // elements per scale
  static constexpr int kSfPerStep = BKB * 2 / kBlock;   // scale bytes per row per K step
  static constexpr int kWords = kSfPerStep / 4;         // 4-byte chunk lines per row per K step
  static constexpr int kChunks = 3 * kWords;            // 512-byte chunks per K step (A, W 0-127, W 128-255)
  static constexpr int kSfCols = 4 * kChunks;           // TMEM columns per stage
  static constexpr uint32_t kPiece = kWords * kSfChunk;  // bytes of one row group's chunks per K step
};
static_assert(3 * Fmt<true>::kPiece <= kSfBytes && 3 * Fmt<false>::kPiece <= kSfBytes, "scale area");
static_assert(kAccCols + kStages * Fmt<true>::kSfCols <= kTmemCols, "TMEM budget");
static_assert(kAccCols + kStages * Fmt<false>::kSfCols <= kTmemCols, "TMEM budget");

// K splits: when the output tiles cannot fill half the GPU (M = 128 at
// N = 8192: 32 tiles), split K so that tiles x splits fill it, keeping at
// least four K steps per split and at most the portable cluster size.  A
// tile's splits are one thread-block cluster and add their partial tiles in
// distributed shared memory, in rank order: the result is deterministic.
constexpr int kMaxSplits = 8;
// The receive area recv[S][ceil(BM / S)][BN / 4] float4 fits in the idle ring
// for every S (S ceil(BM / S) <= BM + S - 1).
static_assert((BM + kMaxSplits - 1) * BN * 4 <= kStages * kStageBytes, "receive area fits in the idle ring");
constexpr int kRxBarOffset = 256;  // the receive barrier's byte offset in the barrier area

// Returns 0 when the 128 x 256 tiles fill half the GPU (the persistent
// kernel); otherwise the number of K splits of the narrow kernel, whose tiles
// are 128 x kNarrowN: half-width tiles give twice the CTAs for the same split
// and a third of the partial bytes exchanged in the cluster (which that
// exchange is bound by).
constexpr int kNarrowN = 128;

int mx_splits(int M, int N, int K) {
  const int m_tiles = (M + BM - 1) / BM;
  const int sms = sm_count();
  if (2 * ((N + BN - 1) / BN) * m_tiles >= sms) return 0;
  const int tiles = ((N + kNarrowN - 1) / kNarrowN) * m_tiles;
  const int kt = (K / 2 + BKB - 1) / BKB;
  int S = sms / tiles;
  if (S > kt / 4) S = kt / 4;
  if (S > kMaxSplits) S = kMaxSplits;
  return S < 1 ? 1 : S;
}
static_assert(kStageBytes % 1024 == 0, "stage alignment");

// One K step's operands into ring stage `st`: [A tile][W tile][scale area].
// The scale area takes kWords chunks (from chunk kt * kWords) of A's row group
// m0 / 128, then of W's row groups n0 / 128 and n0 / 128 + 1 (W's rows are
// padded to a multiple of 256, so both exist), the order the scale copies
// into TMEM read them.  The W half and the A half are issued separately, so
// that a launch that quantizes A first can start W's stream before A exists.
// Each half issues its scale pieces (to `sbar`) before its tile (to `bar`):
// the pieces are small and land first, and a consumer that waits on a
// separate scale barrier can move them into TMEM while the tiles stream in.
// TN: the tile's width (W rows), 256 or 128; a 128-wide tile takes only the
// first W half of the stage and of the scale area.
template <bool kNv, int TN = BN>
__device__ __forceinline__ void load_stage_w(uint8_t* st, const CUtensorMap* tmW, const MxGemmArgs& p, int n0, int kt,
                                             uint64_t* bar, uint64_t* sbar) {
  constexpr uint32_t kPiece = Fmt<kNv>::kPiece;
  const int64_t chunks = tc_sf_chunks(kNv, p.K);
  const uint8_t* w = p.SW + ((n0 / 128) * chunks + static_cast<int64_t>(kt) * Fmt<kNv>::kWords) * kSfChunk;
  uint8_t* sf = st + kABytes + kBBytes;
  tc::bulk_load(sf + kPiece, w, kPiece, sbar);
  if (TN == 256) tc::bulk_load(sf + 2 * kPiece, w + chunks * kSfChunk, kPiece, sbar);
  tc::tma_load_2d(st + kABytes, tmW, kt * BKB, n0, bar);
}

template <bool kNv>
__device__ __forceinline__ void load_stage_a(uint8_t* st, const CUtensorMap* tmA, const MxGemmArgs& p, int m0, int kt,
                                             uint64_t* bar, uint64_t* sbar) {
  const int64_t chunks = tc_sf_chunks(kNv, p.K);
  tc::bulk_load(st + kABytes + kBBytes,
                p.SA + ((m0 / 128) * chunks + static_cast<int64_t>(kt) * Fmt<kNv>::kWords) * kSfChunk,
                Fmt<kNv>::kPiece, sbar);
  tc::tma_load_2d(st, tmA, kt * BKB, m0, bar);
}

// Bytes one stage's copies deliver: the scale pieces, the two tiles, both.
__host__ __device__ constexpr uint32_t stage_sf_tx(bool nv, int tn = BN) {
  return (1 + tn / 128) * (nv ? Fmt<true>::kPiece : Fmt<false>::kPiece);
}
__host__ __device__ constexpr uint32_t stage_tile_tx(int tn = BN) { return kABytes + tn * BKB; }
__host__ __device__ constexpr uint32_t stage_tx(bool nv, int tn = BN) { return stage_tile_tx(tn) + stage_sf_tx(nv, tn); }

// One K step on the tensor cores, in two parts: copy_scales moves the
// stage's scale chunks into its TMEM columns, mma_tiles issues four
// 128 x TN x 64 block-scaled MMAs that read them.  The MMAs may be issued
// right after the copies (a copy followed by an MMA is ordered in the tensor
// pipe); issuing the copies earlier takes their latency off the MMAs' path.
//   MXFP4: TMEM [A kb 0-3][A kb 4-7][W 0-127 kb 0-3][W 128-255 kb 0-3]
//          [W 0-127 kb 4-7][W 128-255 kb 4-7], 4 columns each; MMA j takes
//          the byte pair 2 (j % 2) of column 4 (j / 2) (A) and 8 + 8 (j / 2)
//          (W: the N = 256 MMA reads W rows 128-255 four columns after rows
//          0-127).
//   NVFP4: TMEM [A j=0..3][W 0-127 j=0][W 128-255 j=0] .. [W 0-127 j=3][W 128-255 j=3];
//          MMA j takes the whole word of column 4 j (A) and 16 + 8 j (W).
// A 128-wide tile (TN = 128) copies only A's and W rows 0-127's chunks (the
// first two thirds of the scale area) and issues 128 x 128 x 64 MMAs.
// Four consecutive 32-bit TMEM columns of this warp's 32 lanes (one row per
// thread), from registers; complete once tmem_st_wait returns.
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// First TMEM column (relative to the stage's scale columns) of the stage's
// scale chunk c, in the scale area's order (A, W rows 0-127, W rows 128-255).
template <bool kNv>
__device__ __forceinline__ constexpr int sf_column(int c) {
  if constexpr (!kNv) {
    return 4 * ((c == 3 || c == 4) ? 7 - c : c);  // chunk order 0, 1, 2, 4, 3, 5
  } else {
    const int grp = c / 4, j = c % 4;
    return grp == 0 ? 4 * j : 16 + 8 * j + (grp == 2 ? 4 : 0);
  }
}

// Each chunk is 32 lines of 16 bytes; line i goes to lane i of every lane
// quarter, as four columns.
template <bool kNv, int TN = BN>
__device__ __forceinline__ void copy_scales(uint32_t sf, uint32_t sf_col) {
#pragma unroll
  for (int c = 0; c < (TN == 256 ? 3 : 2) * Fmt<kNv>::kWords; ++c)
    tc::tmem_cp_32x128b_warpx4(sf_col + sf_column<kNv>(c),
                               tc::smem_desc(sf + c * kSfChunk, 16, 128, tc::kSwizzleNone));
}

template <bool kNv, int TN = BN>
__device__ __forceinline__ void mma_tiles(uint32_t tmem, uint32_t a, uint32_t b, uint32_t sf_col, bool first) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // 64 elements = 32 bytes per MMA
    const uint64_t adesc = tc::smem_desc(a + 32 * j, 1024, 1024, tc::kSwizzle128B);
    const uint64_t bdesc = tc::smem_desc(b + 32 * j, 1024, 1024, tc::kSwizzle128B);
    if constexpr (!kNv) {
      const uint32_t id = 2 * (j & 1);
      const uint32_t idesc = tc::idesc_block_scaled(/*E2M1*/ 1, /*E2M1*/ 1, BM, TN, id, id);
      tc::mma_mxf4(tmem, adesc, bdesc, idesc, sf_col + 4 * (j >> 1), sf_col + 8 + 8 * (j >> 1), !first || j != 0);
    } else {
      constexpr uint32_t idesc = tc::idesc_block_scaled(/*E2M1*/ 1, /*E2M1*/ 1, BM, TN, 0, 0, /*UE4M3*/ 0);
      tc::mma_mxf4nvf4_4x(tmem, adesc, bdesc, idesc, sf_col + 4 * j, sf_col + 16 + 8 * j, !first || j != 0);
    }
  }
}

template <bool kNv, int TN = BN>
__device__ __forceinline__ void mma_step(uint32_t tmem, uint32_t a, uint32_t b, uint32_t sf, uint32_t sf_col,
                                         bool first) {
  copy_scales<kNv, TN>(sf, sf_col);
  mma_tiles<kNv, TN>(tmem, a, b, sf_col, first);
}

// Product of the two tensor scales (NVFP4), 1 for MXFP4.
template <bool kNv>
__device__ __forceinline__ float tensor_scale(const MxGemmArgs& p) {
  if constexpr (kNv) return __fmul_rn(*p.ga, *p.gw);
  return 1.0f;
}


// ------------------------------------------------ A quantized in the launch
// mx_gemm_fp4_qa: the MXFP4 page's flow quantizes both operands before the
// GEMM (§三); here A's quantization is the first phase of the GEMM launch.
// Every CTA quantizes its share of A into the workspace (codes, and scales
// already in the tensor-core layout), the grid meets at one barrier, and the
// GEMM proper reads A from there through the same TMA and bulk copies as
// always.  Each element is quantized exactly once, with the arithmetic of
// mx_quantize_fp4 (mx_block.cuh), so the codes and the result are those of
// quantize-then-GEMM, bit for bit.
//
// Items are (row r < M rounded up to 256, chunk c < kc): blocks 4c .. 4c + 3
// of row r, 128 elements, for a group of 16 threads (four per block, eight
// elements each), numbered row by row.  The items of A's rows and those of
// the padding rows (scale 2^0, no codes: their data reads as zero through
// the tensor map) are split over the CTAs separately, so that every CTA gets
// the same share of real rows.  A group handles kQaUnroll items per round
// and loads the next round's elements before it quantizes the current ones,
// so the loads stay in flight while the arithmetic runs.
constexpr int kQaUnroll = 4;

// This CTA's items: local index v < n maps to real item r0 + v (v < nr) or
// padding item p0 + v - nr.
struct QaItems {
  uint32_t chunks, nb, r0, nr, p0, n;
  __device__ __forceinline__ uint32_t item(uint32_t v) const { return v < nr ? r0 + v : p0 + (v - nr); }
};

__device__ __forceinline__ QaItems qa_items(const MxGemmArgs& p) {
  QaItems q;
  q.chunks = static_cast<uint32_t>(tc_sf_chunks(false, p.K));
  q.nb = static_cast<uint32_t>(p.K / 32);
  const uint32_t real = static_cast<uint32_t>(p.M) * q.chunks;
  const uint32_t pad = static_cast<uint32_t>((p.M + 255) / 256 * 256 - p.M) * q.chunks;  // total < 2^31 (host check)
  const uint64_t G = gridDim.x * gridDim.y * gridDim.z;
  const uint64_t b = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  q.r0 = static_cast<uint32_t>(b * real / G);
  q.nr = static_cast<uint32_t>((b + 1) * real / G) - q.r0;
  q.p0 = real + static_cast<uint32_t>(b * pad / G);
  q.n = q.nr + (real + static_cast<uint32_t>((b + 1) * pad / G) - q.p0);
  return q;
}

// One round's loads: this thread's eight elements of local item base + grp + u ngrp,
// and each item's row and chunk column (kept for the quantization step).
__device__ __forceinline__ void qa_load(const MxGemmArgs& p, const QaItems& q, uint32_t base, uint32_t grp,
                                        uint32_t ngrp, uint32_t j, uint32_t qq, float4 (&v)[kQaUnroll][2],
                                        uint32_t (&rows)[kQaUnroll], uint32_t (&cols)[kQaUnroll]) {
#pragma unroll
  for (int u = 0; u < kQaUnroll; ++u) {
    const uint32_t lv = base + grp + u * ngrp;
    const uint32_t item = q.item(lv);
    const uint32_t row = item / q.chunks, col = item - row * q.chunks, blk = 4 * col + j;
    rows[u] = row;
    cols[u] = col;
    if (lv < q.n && row < static_cast<uint32_t>(p.M) && blk < q.nb) {
      const float4* src = reinterpret_cast<const float4*>(p.A32 + static_cast<int64_t>(row) * p.lda32 + 32 * blk + 8 * qq);
      v[u][0] = __ldcs(src);
      v[u][1] = __ldcs(src + 1);
    } else {
      v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

__device__ void quantize_a_share(const MxGemmArgs& p) {
  const QaItems q = qa_items(p);
  const int lane = threadIdx.x & 31, t16 = lane & 15;
  const uint32_t grp = threadIdx.x >> 4, ngrp = blockDim.x >> 4;
  const uint32_t j = t16 >> 2, qq = t16 & 3;  // block within the item, quarter within the block
  const uint32_t step = ngrp * kQaUnroll;
  float4 nxt[kQaUnroll][2];
  uint32_t nrow[kQaUnroll], ncol[kQaUnroll];
  if (q.n > 0) qa_load(p, q, 0, grp, ngrp, j, qq, nxt, nrow, ncol);
  // The loop bound is the same for every thread, so all lanes reach the shuffles.
  for (uint32_t base = 0; base < q.n; base += step) {
    float4 v[kQaUnroll][2];
    uint32_t crow[kQaUnroll], ccol[kQaUnroll];
#pragma unroll
    for (int u = 0; u < kQaUnroll; ++u) {
      v[u][0] = nxt[u][0];
      v[u][1] = nxt[u][1];
      crow[u] = nrow[u];
      ccol[u] = ncol[u];
    }
    if (base + step < q.n) qa_load(p, q, base + step, grp, ngrp, j, qq, nxt, nrow, ncol);
#pragma unroll
    for (int u = 0; u < kQaUnroll; ++u) {
      const bool item_ok = base + grp + u * ngrp < q.n;
      const uint32_t row = crow[u], col = ccol[u];
      const uint32_t blk = 4 * col + j;
      const bool real = item_ok && row < static_cast<uint32_t>(p.M) && blk < q.nb;
      const float xs[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                           v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(xs[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      amax = fmaxf(amax, 1e-8f);
      const int e = mx_block_exponent(amax);
      const uint32_t word = e2m1_word(xs, mx_inv_scale(e));
      if (real) *reinterpret_cast<uint32_t*>(p.Aq + static_cast<int64_t>(row) * p.ldq + 16 * blk + 4 * qq) = word;
      // The four blocks' scale bytes, gathered from the quad leaders of this
      // 16-thread group, form one word of the chunk line.
      const uint32_t sb = real ? static_cast<uint32_t>(e + 127) : 0x7Fu;
      const int g0 = lane & 16;
      const uint32_t sw = __shfl_sync(0xffffffffu, sb, g0) | (__shfl_sync(0xffffffffu, sb, g0 + 4) << 8) |
                          (__shfl_sync(0xffffffffu, sb, g0 + 8) << 16) | (__shfl_sync(0xffffffffu, sb, g0 + 12) << 24);
      if (t16 == 0 && item_ok)
        *reinterpret_cast<uint32_t*>(p.SAq + (static_cast<int64_t>(row / 128) * q.chunks + col) * kSfChunk +
                                     16 * (row % 32) + 4 * ((row / 32) % 4)) = sw;
    }
  }
}

// One barrier over the whole grid (the launch is cooperative, so every CTA is
// resident).  Word 0 of grid_bar counts arrivals, word 1 departures; the last
// CTA to leave zeroes both, so the next call finds them zero.  Returns false,
// with the error recorded and *abort raised, if the other CTAs do not all
// arrive within the wait limit.  Before it, each thread fences its global
// writes for the async proxy (the GEMM reads them with TMA and bulk copies).
__device__ bool grid_barrier(unsigned* bar, volatile int* abort, int* err) {
  tc::fence_proxy_async_all();
  tc::cta_barrier();
  if (threadIdx.x == 0) {
    const unsigned G = gridDim.x * gridDim.y * gridDim.z;
    __threadfence();
    atomicAdd(&bar[0], 1u);
    const uint64_t t0 = tc::globaltimer_ns();
    bool ok = true;
    // Spin for the first few microseconds (the CTAs normally arrive within
    // one or two), then poll with a short sleep; give up after the limit.
    for (uint32_t it = 0; tc::ld_acquire_gpu(&bar[0]) < G; ++it) {
      if ((it & 63u) != 63u) continue;
      const uint64_t dt = tc::globaltimer_ns() - t0;
      if (dt > 2000000000ull) {
        if (err) atomicCAS(err, 0, kSiteGridBarrier);
        *abort = 1;
        ok = false;
        break;
      }
      if (dt > 8000u) __nanosleep(64);
    }
    if (ok && atomicAdd(&bar[1], 1u) == G - 1) {
      atomicExch(&bar[0], 0u);
      atomicExch(&bar[1], 0u);
    }
    __threadfence();
  }
  tc::cta_barrier();
  tc::fence_proxy_async_all();
  return !*abort;
}

// Transpose a 32 x 32 block held one row per lane (lane i: v[j] = B[i][j])
// into one column per lane (lane j: v[i] = B[i][j]), with five butterfly
// stages of register exchanges between lanes.
__device__ __forceinline__ void warp_transpose32(uint32_t (&v)[32], int lane) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j & m) continue;
      const uint32_t send = upper ? v[j] : v[j + m];
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
      if (upper) v[j] = recv;
      else v[j + m] = recv;
    }
  }
}

template <bool kNv, bool kQA, int TN>
__global__ void __launch_bounds__(kThreads, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, MxGemmArgs p,
               int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* accum = empty + kStages;
  uint64_t* drain = accum + 1;  // MMAs in flight after a give-up
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // Split K: counts the peers' parts of this CTA's rows as they arrive.
  uint64_t* rx_bar = reinterpret_cast<uint64_t*>(smem + kBarOffset + kRxBarOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * TN;
  // K steps [kt0, kt1) of this CTA: all of K, or split z of gridDim.z.
  const int KT_all = (p.K / 2 + BKB - 1) / BKB;
  const int kt0 = static_cast<int>(static_cast<int64_t>(blockIdx.z) * KT_all / gridDim.z);
  const int kt1 = static_cast<int>(static_cast<int64_t>(blockIdx.z + 1) * KT_all / gridDim.z);
  const int KT = kt1 - kt0;  // steps here; step kt0 + i uses ring slot i % kStages

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(accum, 1);
    tc::mbar_init(drain, 1);
    if (gridDim.z > 1) {
      // Armed now, long before any peer sends (after the cluster barrier that
      // follows every CTA's MMAs): (S - 1) parts of this CTA's rows.
      const int S = gridDim.z, rank = static_cast<int>(blockIdx.z);
      const int rows = (rank + 1) * BM / S - rank * BM / S;
      tc::mbar_init(rx_bar, 1);
      tc::mbar_arrive_expect_tx(rx_bar, static_cast<uint32_t>((S - 1) * rows * TN * 4));
    }
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  tc::cta_barrier();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the scale re-layout: every read
  // of the inputs and every write of C comes after this.
  tc::griddep_wait();
  // Quantizing A first: the W halves of the first stages (fresh ring slots)
  // are issued before, so that W's stream overlaps A's quantization.
  const int pre = kQA ? (KT < kStages ? KT : kStages) : 0;
  if constexpr (kQA) {
    if (warp == 0 && lane == 0) {
      tc::tma_prefetch_desc(&tmW);
      for (int i = 0; i < pre; ++i) {
        tc::mbar_arrive_expect_tx(&full[i], stage_tx(kNv, TN));
        load_stage_w<kNv, TN>(smem + i * kStageBytes, &tmW, p, n0, kt0 + i, &full[i], &full[i]);
      }
    }
    quantize_a_share(p);
    grid_barrier(p.grid_bar, abort, err);
  }

  if (kQA && *abort) {
    // The grid barrier gave up: no role runs (the cluster steps below still
    // do).  The early W copies are in flight: complete their stages with the
    // A halves (in-bounds reads of the workspace) and wait for them.
    if (warp == 0 && lane == 0) {
      for (int i = 0; i < pre; ++i) load_stage_a<kNv>(smem + i * kStageBytes, &tmA, p, m0, kt0 + i, &full[i], &full[i]);
      for (int i = 0; i < pre; ++i) tc::mbar_wait_drain(&full[i], 0);
    }
  } else if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmA);
      tc::tma_prefetch_desc(&tmW);
    }
    int issued = 0;
    for (int i = 0; i < KT; ++i) {
      const int kt = kt0 + i, s = i % kStages;
      uint8_t* st = smem + s * kStageBytes;
      if (i < pre) {  // W half already issued
        if (lane == 0) load_stage_a<kNv>(st, &tmA, p, m0, kt, &full[s], &full[s]);
        issued = i + 1;
        continue;
      }
      const bool free_slot = tc::mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1, abort, err, kSiteGemmProducer);
      if (!__all_sync(0xffffffffu, free_slot)) break;  // warp-uniform exit
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(&full[s], stage_tx(kNv, TN));
        load_stage_a<kNv>(st, &tmA, p, m0, kt, &full[s], &full[s]);
        load_stage_w<kNv, TN>(st, &tmW, p, n0, kt, &full[s], &full[s]);
      }
      issued = i + 1;
    }
    if (*abort && lane == 0) {
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        tc::mbar_wait_drain(&full[i % kStages], (i / kStages) & 1);
    }
  } else if (warp == 1 && lane == 0) {
    for (int i = 0; i < KT; ++i) {
      const int s = i % kStages;
      if (!tc::mbar_wait(&full[s], (i / kStages) & 1, abort, err, kSiteGemmMma)) break;
      tc::tc_fence_after();
      const uint32_t a = tc::smem_u32(smem + s * kStageBytes);
      const uint32_t b = a + kABytes;
      const uint32_t sf = b + kBBytes;
      const uint32_t sf_col = tmem + kAccCols + s * Fmt<kNv>::kSfCols;
      mma_step<kNv, TN>(tmem, a, b, sf, sf_col, i == 0);
      tc::tc_commit(&empty[s]);
    }
    tc::tc_commit(accum);
    // After a give-up: wait (bounded) until every MMA and scale copy issued
    // so far has completed, so that none still uses TMEM when it is freed.
    if (*abort) {
      tc::tc_commit(drain);
      tc::mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 2) {
    const float gs = tensor_scale<kNv>(p);
    const bool ok = tc::mbar_wait(accum, 0, abort, err, kSiteGemmEpilogue);
    tc::tc_fence_after();
    // Split K: the accumulator stays in tensor memory until the cluster
    // exchange below.
    if (gridDim.z == 1) {
      const int q = warp & 3;
      const int row = m0 + 32 * q + lane;
      for (int c = 0; c < TN / 32; ++c) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + 32 * c, r);
        tc::tmem_ld_wait();
        if (!ok) continue;
        if constexpr (kNv) {
#pragma unroll
          for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * gs);
        }
        if (row >= p.M) continue;
        const int col0 = n0 + 32 * c;
        float* dst = p.C + static_cast<int64_t>(row) * p.ldc + col0;
        if (col0 + 32 <= p.N) {
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<uint4*>(dst + 4 * v) = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (col0 + t < p.N) dst[t] = __uint_as_float(r[t]);
        }
      }
    }
  }
  tc::tc_fence_before();
  tc::cta_barrier();
  if (gridDim.z > 1) {
    // Split K over the S CTAs of the cluster: rank k finishes rows
    // [k BM / S, (k + 1) BM / S) of the tile.  Every CTA gets here (all its
    // waits are bounded).  After the cluster barrier every CTA's MMAs are
    // done, so every ring is idle and becomes the receive area
    // recv[S][rmax][TN / 4]: part j of the owner's rows from rank j, the
    // float4s of each 32-column group rotated by the row (conflict-free
    // stores and loads).  Each epilogue warp sends its 32 accumulator rows
    // straight from tensor memory to their owners with one-way stores that
    // count toward the owner's receive barrier (its own rows with plain
    // stores); no CTA reads another's shared memory, so none waits for its
    // peers before leaving.  The owner adds the S parts in rank order, so the
    // result does not depend on arrival order.  (Pulling the parts with
    // loads, or sending row blocks with bulk copies, measured no faster: the
    // 96 KB each CTA exchanges at S = 4 is bound by the cluster network.)
    const int S = gridDim.z, rank = static_cast<int>(tc::cluster_ctarank());
    const int rmax = (BM + S - 1) / S;
    tc::cluster_sync_all();
    tc::tc_fence_after();
    float4* recv = reinterpret_cast<float4*>(smem);
    if (warp >= 2) {
      const int q = warp & 3;
      const int row = 32 * q + lane;                 // tile row = TMEM lane
      const int k = ((row + 1) * S - 1) / BM;         // its owner
      const int lr = row - k * BM / S;                // row within the owner's rows
      const int base = (rank * rmax + lr) * (TN / 4);  // this part's row in the owner's recv
      const uint32_t peer_recv = tc::dsmem_addr(recv, k);
      const uint32_t peer_bar = tc::dsmem_addr(rx_bar, k);
      for (int c = 0; c < TN / 32; ++c) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + 32 * c, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const int slot = base + 8 * c + ((v + lr) & 7);
          const float4 val = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                         __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          if (k == rank) recv[slot] = val;
          else tc::st_async_f4(peer_recv + 16u * static_cast<uint32_t>(slot), val, peer_bar);
        }
      }
    }
    tc::cta_barrier();  // this CTA's own part is in place
    // The peers' parts (bounded wait; the peers always send, so the wait
    // normally ends; a CTA that gives up leaves without storing).
    const bool got = tc::mbar_wait_cluster(rx_bar, 0, err, kSiteClusterRecv);
    const float gs = tensor_scale<kNv>(p);
    const bool live = got && !*abort;
    const int r0 = rank * BM / S, rows = (rank + 1) * BM / S - r0;
    const int n_items = rows * (TN / 4);
    for (int it = threadIdx.x; it < n_items; it += blockDim.x) {
      const int lr = it / (TN / 4), c4 = it % (TN / 4);
      const int slot = lr * (TN / 4) + (c4 & ~7) + (((c4 & 7) + lr) & 7);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < kMaxSplits; ++j)
        if (j < S) {
          const float4 v = recv[j * rmax * (TN / 4) + slot];
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
      if constexpr (kNv) {
        acc.x *= gs;
        acc.y *= gs;
        acc.z *= gs;
        acc.w *= gs;
      }
      const int row = m0 + r0 + lr, col = n0 + 4 * c4;
      if (!live || row >= p.M || col >= p.N) continue;
      float* dst = p.C + static_cast<int64_t>(row) * p.ldc + col;
      if (col + 4 <= p.N) {
        *reinterpret_cast<float4*>(dst) = acc;  // C 16-byte aligned, ldc a multiple of 4
      } else {
        const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (col + t < p.N) dst[t] = a4[t];
      }
    }
  }
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Persistent variant (one CTA per SM, output tiles handed out round-robin,
// walking down M so that the CTAs running at the same time share W tiles in
// L2).  The ring runs continuously across a CTA's tiles.  There is one
// accumulator (two 128 x 256 FP32 tiles and the staged scale columns do not
// fit in TMEM together), so the epilogue hands it back as soon as it has read
// it into registers and stores C while the next tile's MMAs run: eight
// epilogue warps, each holding 32 rows x 128 columns.  TMEM hands each lane
// one row; each 32 x 32 block is transposed across the warp first, so that
// every store instruction writes one whole 128-byte row of C.  (Writing rows
// per thread, 32 rows per instruction, either held the accumulator for a
// third of each tile or, done after the hand-back, flooded the SM's memory
// path and starved the next tile's TMA loads.)
//   warp 0      TMA producer (data tiles and scale chunks)
//   warp 1      TMEM allocator and MMA issuer
//   warps 2-9   epilogue: warp w reads TMEM lanes 32 (w % 4) .. (the lane
//               quarter it may access) and columns 128 ((w - 2) / 4) ..
constexpr int kPThreads = 320;
constexpr int kEpiWarps = 8;

// Wait for an accumulator hand-off that is normally microseconds away: poll
// with a short sleep between tries, so that the waiting warps leave the
// shared-memory barrier unit to the roles on the critical path.  Bounded like
// mbar_wait.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity, volatile int* abort, int* err,
                                                  int site, uint64_t limit_ns = 2000000000ull) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::globaltimer_ns();
  for (;;) {
    __nanosleep(256);
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (tc::globaltimer_ns() - t0 > limit_ns) {
      if (err) atomicCAS(err, 0, site);
      *abort = 1;
      return false;
    }
  }
}

template <bool kNv, bool kQA>
__global__ void __launch_bounds__(kPThreads, 1)
mx_gemm_persistent(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, MxGemmArgs p,
                   int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;     // MMA -> epilogue
  uint64_t* acc_empty = acc_full + 1;       // epilogue warps -> MMA
  uint64_t* drain = acc_empty + 1;          // MMAs in flight after a give-up
  uint64_t* sfull = drain + 1;              // producer -> scale stagers: a stage's scale pieces landed
  uint64_t* sf_ready = sfull + kStages;     // scale stagers -> MMA: a stage's scales are in TMEM
  // Who moves the scale chunks into TMEM.  NVFP4 (12 chunks a step): the
  // epilogue warps, between accumulator drains, with tcgen05.st.  MXFP4 (6
  // chunks): the MMA thread, with tcgen05.cp just before the step's MMAs,
  // and the pieces land with the tiles on `full`.  Measured on 8192^3:
  // staging took NVFP4 from 346 to 307 us but MXFP4 from 259 to 274 us.
  constexpr bool kStageSf = kNv;
  uint64_t* sbar = kStageSf ? sfull : full;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_ready + kStages);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = (p.K / 2 + BKB - 1) / BKB;
  const int m_tiles = (p.M + BM - 1) / BM, n_tiles = (p.N + BN - 1) / BN;
  const int tiles = m_tiles * n_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
      tc::mbar_init(&sfull[s], 1);
      tc::mbar_init(&sf_ready[s], kEpiWarps);
    }
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(acc_empty, kEpiWarps);
    tc::mbar_init(drain, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  tc::cta_barrier();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the scale re-layout: every read
  // of the inputs and every write of C comes after this.
  tc::griddep_wait();
  // Quantizing A first: the W halves of the first tile's first stages are
  // issued before, so that W's stream overlaps A's quantization (the grid is
  // at most one CTA per tile, so every CTA has a first tile).
  const int pre = kQA ? (KT < kStages ? KT : kStages) : 0;
  const int m00 = (static_cast<int>(blockIdx.x) % m_tiles) * BM, n00 = (static_cast<int>(blockIdx.x) / m_tiles) * BN;
  if constexpr (kQA) {
    if (warp == 0 && lane == 0) {
      tc::tma_prefetch_desc(&tmW);
      for (int i = 0; i < pre; ++i) {
        if (kStageSf) tc::mbar_arrive_expect_tx(&sfull[i], stage_sf_tx(kNv));
        tc::mbar_arrive_expect_tx(&full[i], kStageSf ? stage_tile_tx() : stage_tx(kNv));
        load_stage_w<kNv>(smem + i * kStageBytes, &tmW, p, n00, i, &full[i], &sbar[i]);
      }
    }
    quantize_a_share(p);
    grid_barrier(p.grid_bar, abort, err);
  }

  if (kQA && *abort) {
    // The grid barrier gave up: no role runs.  Complete the early stages
    // with their A halves and wait for them, so no copy is left in flight.
    if (warp == 0 && lane == 0) {
      for (int i = 0; i < pre; ++i) load_stage_a<kNv>(smem + i * kStageBytes, &tmA, p, m00, i, &full[i], &sbar[i]);
      for (int i = 0; i < pre; ++i) {
        tc::mbar_wait_drain(&full[i], 0);
        if (kStageSf) tc::mbar_wait_drain(&sfull[i], 0);
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmA);
      tc::tma_prefetch_desc(&tmW);
    }
    int it = 0, issued = 0;
    bool go = true;
    for (int t = blockIdx.x; t < tiles && go; t += gridDim.x) {
      const int m0 = (t % m_tiles) * BM, n0 = (t / m_tiles) * BN;
      for (int kt = 0; kt < KT; ++kt, ++it) {
        const int s = it % kStages;
        uint8_t* st = smem + s * kStageBytes;
        if (it < pre) {  // W half already issued (first tile, fresh slot)
          if (lane == 0) load_stage_a<kNv>(st, &tmA, p, m0, kt, &full[s], &sbar[s]);
          issued = it + 1;
          continue;
        }
        const bool free_slot = tc::mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, abort, err, kSiteGemmProducer);
        if (!__all_sync(0xffffffffu, free_slot)) {
          go = false;
          break;
        }
        if (lane == 0) {
          if (kStageSf) tc::mbar_arrive_expect_tx(&sfull[s], stage_sf_tx(kNv));
          tc::mbar_arrive_expect_tx(&full[s], kStageSf ? stage_tile_tx() : stage_tx(kNv));
          load_stage_a<kNv>(st, &tmA, p, m0, kt, &full[s], &sbar[s]);
          load_stage_w<kNv>(st, &tmW, p, n0, kt, &full[s], &sbar[s]);
        }
        issued = it + 1;
      }
    }
    if (*abort && lane == 0) {
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
        tc::mbar_wait_drain(&full[i % kStages], (i / kStages) & 1);
        if (kStageSf) tc::mbar_wait_drain(&sfull[i % kStages], (i / kStages) & 1);
      }
    }
  } else if (warp == 1 && lane == 0) {
    int it = 0, local = 0;
    for (int t = blockIdx.x; t < tiles && !*abort; t += gridDim.x, ++local) {
      if (!tc::mbar_wait(acc_empty, (local & 1) ^ 1, abort, err, kSiteGemmTmemFree)) break;
      tc::tc_fence_after();
      bool ok = true;
      for (int kt = 0; kt < KT; ++kt, ++it) {
        const int s = it % kStages;
        if ((kStageSf && !tc::mbar_wait(&sf_ready[s], (it / kStages) & 1, abort, err, kSiteGemmMma)) ||
            !tc::mbar_wait(&full[s], (it / kStages) & 1, abort, err, kSiteGemmMma)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t a = tc::smem_u32(smem + s * kStageBytes);
        const uint32_t sf_col = tmem + kAccCols + s * Fmt<kNv>::kSfCols;
        if constexpr (!kStageSf) copy_scales<kNv>(a + kABytes + kBBytes, sf_col);
        mma_tiles<kNv>(tmem, a, a + kABytes, sf_col, kt == 0);
        tc::tc_commit(&empty[s]);
      }
      if (!ok) break;
      tc::tc_commit(acc_full);  // arrives once every MMA of the tile has completed
    }
    // After a give-up: wait (bounded) until every MMA and scale copy issued
    // so far has completed, so that none still uses TMEM when it is freed.
    if (*abort) {
      tc::tc_commit(drain);
      tc::mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 2) {
    // With kStageSf the epilogue warps also move every stage's scale chunks
    // into TMEM (shared memory -> registers -> tcgen05.st), so that the
    // tensor pipe issues nothing but MMAs.  Warp (q, h) writes lane quarter
    // q of the stage's chunks h kHalf .. h kHalf + kHalf - 1.  Staging runs
    // up to kStages steps ahead of the MMAs; a tile's accumulator is drained
    // once the next tile's first steps are staged, so that their MMAs can
    // start as soon as the accumulator is handed back.
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;   // column half: 128 h .. 128 h + 127; chunk half
    const float gs = tensor_scale<kNv>(p);
    const uint32_t lanes = static_cast<uint32_t>(32 * q) << 16;
    // Drain tile t (this CTA's tile number `local`) from TMEM to C.
    auto drain_tile = [&](int t, int local) -> bool {
      const bool ok = mbar_wait_backoff(acc_full, local & 1, abort, err, kSiteGemmEpilogue);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc::tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld_32x32b_x32(tmem + lanes + 128 * h + 32 * c, r[c]);
      tc::tmem_ld_wait();
      // The accumulator is in registers: hand it back to the MMA warp.
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty);
      if constexpr (kNv) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int u = 0; u < 32; ++u) r[c][u] = __float_as_uint(__uint_as_float(r[c][u]) * gs);
      }
      // After the transpose lane l holds column n0 + 32 c + l of rows
      // row0 .. row0 + 31.
      const int row0 = (t % m_tiles) * BM + 32 * q, n0 = (t / m_tiles) * BN + 128 * h;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int col = n0 + 32 * c + lane;
        warp_transpose32(r[c], lane);
        if (col >= p.N) continue;
        float* dst = p.C + static_cast<int64_t>(row0) * p.ldc + col;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (row0 + i < p.M) dst[static_cast<int64_t>(i) * p.ldc] = __uint_as_float(r[c][i]);
      }
      return true;
    };
    if constexpr (!kStageSf) {
      int local = 0;
      for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++local)
        if (!drain_tile(t, local)) break;
    } else {
      constexpr int kHalf = Fmt<kNv>::kChunks / 2;
      const int ahead = KT < kStages ? KT : kStages;
      bool ok = true;
      int it = 0, local = 0;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++local) {
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int s = it % kStages;
          ok = tc::mbar_wait_sleep(&sfull[s], (it / kStages) & 1, abort, err, kSiteGemmEpilogue);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          const uint8_t* sf = smem + s * kStageBytes + kABytes + kBBytes;
          const uint32_t col = tmem + lanes + kAccCols + s * Fmt<kNv>::kSfCols;
#pragma unroll
          for (int i = 0; i < kHalf; ++i) {
            const int c = h * kHalf + i;
            tmem_st_32x32b_x4(col + sf_column<kNv>(c),
                                  *reinterpret_cast<const uint4*>(sf + c * kSfChunk + 16 * lane));
          }
          tmem_st_wait();
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sf_ready[s]);
          if (kt == ahead - 1 && local > 0 && !drain_tile(t - static_cast<int>(gridDim.x), local - 1)) {
            ok = false;
            break;
          }
        }
      }
      if (ok && local > 0) drain_tile(blockIdx.x + (local - 1) * static_cast<int>(gridDim.x), local - 1);
    }
  }
  tc::tc_fence_before();
  tc::cta_barrier();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace {

// kQA: A arrives as FP32 and is quantized in the same launch (MXFP4 only).
// That launch is cooperative (its CTAs meet at a grid barrier), so its grid
// must be resident at once: the persistent grid is one CTA per SM at most,
// and a K split is narrowed until the occupancy query says its clusters fit.
template <bool kNv, bool kQA = false>
cudaError_t launch_fp4_gemm(const MxGemmArgs& a, cudaStream_t s) {
  if (a.K == 0)
    return cudaMemset2DAsync(a.C, a.ldc * 4, 0, static_cast<size_t>(a.N) * 4, a.M, s);
  // splits == 0: the persistent kernel on 128 x 256 tiles; otherwise the
  // narrow kernel on 128 x 128 tiles, K split over `splits` CTAs.
  int splits = mx_splits(a.M, a.N, a.K);
  const int tn = splits == 0 ? BN : kNarrowN;
  CUtensorMap tA, tW;
  cudaError_t e = kQA ? make_tmap_2d(&tA, a.Aq, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.K / 2, a.M, a.ldq, BKB, BM,
                                     CU_TENSOR_MAP_SWIZZLE_128B)
                      : make_tmap_2d(&tA, a.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.K / 2, a.M, a.lda, BKB, BM,
                                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&tW, a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.K / 2, a.N, a.ldw, BKB, tn, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const int m_tiles = (a.M + BM - 1) / BM, n_tiles = (a.N + tn - 1) / tn, tiles = m_tiles * n_tiles;
  // Both kernels start as programmatic dependents of the launch before them
  // (normally the scale re-layout) and wait for it before touching memory.
  cudaLaunchConfig_t cfg = {};
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  attr[0].id = kQA ? cudaLaunchAttributeCooperative : cudaLaunchAttributeProgrammaticStreamSerialization;
  if (kQA) attr[0].val.cooperative = 1;
  else attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (splits == 0) {  // persistent: one CTA per SM
    auto pk = mx_gemm_persistent<kNv, kQA>;
    static PerDevice<bool> pconfigured;
    bool pdone = false;
    if (!pconfigured.get(pdone, [&](bool& v) {
          e = cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
          v = true;
          return e == cudaSuccess;
        }))
      return e;
    cfg.blockDim = dim3(kPThreads);
    cfg.gridDim = dim3(tiles < sm_count() ? tiles : sm_count());
    e = cudaLaunchKernelEx(&cfg, pk, tA, tW, a, device_error_word());
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  auto kern = mx_gemm_kernel<kNv, kQA, kNarrowN>;
  static PerDevice<bool> configured;
  bool done = false;
  if (!configured.get(done, [&](bool& v) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        v = true;
        return e == cudaSuccess;
      }))
    return e;
  if (kQA) {
    // The cooperative launch needs every cluster resident at once.  (With
    // at most 2 x 76 narrow tiles the grid of a split of 1 is one wave.)
    for (; splits > 1; --splits) {
      cudaLaunchConfig_t q = cfg;
      cudaLaunchAttribute ca[1];
      ca[0].id = cudaLaunchAttributeClusterDimension;
      ca[0].val.clusterDim.x = 1;
      ca[0].val.clusterDim.y = 1;
      ca[0].val.clusterDim.z = splits;
      q.attrs = ca;
      q.numAttrs = 1;
      q.blockDim = dim3(kThreads);
      q.gridDim = dim3(n_tiles, m_tiles, splits);
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &q) == cudaSuccess && clusters >= tiles) break;
    }
  }
  // Split K: each tile's splits form a thread-block cluster (along z) that
  // adds its partial tiles in distributed shared memory.
  cfg.blockDim = dim3(kThreads);
  cfg.gridDim = dim3(n_tiles, m_tiles, splits);
  if (splits > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = splits;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, kern, tA, tW, a, device_error_word());
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mx_gemm(const MxGemmArgs& a, cudaStream_t s) { return launch_fp4_gemm<false>(a, s); }

cudaError_t launch_mx_gemm_qa(const MxGemmArgs& a, cudaStream_t s) { return launch_fp4_gemm<false, true>(a, s); }

cudaError_t launch_nv_gemm(const MxGemmArgs& a, cudaStream_t s) { return launch_fp4_gemm<true>(a, s); }

}  // namespace wq
