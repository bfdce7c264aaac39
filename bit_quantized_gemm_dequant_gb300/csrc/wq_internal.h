// Internal declarations shared by the libwq translation units (host side).
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "../../include/wq.h"

namespace wq {

// Host-side one-time setup per device (a kernel's shared-memory attribute, an
// occupancy count), safe to call from several host threads: get(init) runs
// init(value) for the current device until it succeeds once, and returns the
// stored value afterwards (lock-free once set).  A failed init is not stored,
// so a later call tries again.
constexpr int kMaxDevices = 64;
int current_device();  // cudaGetDevice, clamped to [0, kMaxDevices)

template <typename T>
class PerDevice {
 public:
  template <typename F>
  bool get(T& out, F&& init) {
    const int d = current_device();
    if (ready_[d].load(std::memory_order_acquire)) {
      out = value_[d];
      return true;
    }
    std::lock_guard<std::mutex> lock(mu_);
    if (!ready_[d].load(std::memory_order_relaxed)) {
      T v{};
      if (!init(v)) return false;
      value_[d] = v;
      ready_[d].store(true, std::memory_order_release);
    }
    out = value_[d];
    return true;
  }

 private:
  std::mutex mu_;
  std::atomic<bool> ready_[kMaxDevices] = {};
  T value_[kMaxDevices] = {};
};

// Limit of the skinny kernels' bounded waits (2 s unless a test shortened it
// with wq_debug_set_wait_limit).
uint64_t skinny_wait_ns();
// wq_set_static_weights: whether callers promised that no kernel still
// running when a weight-only call launches writes its weights or scales.
bool static_weights();

// Device error word written by kernels whose bounded waits give up.  Lives in
// wq_api.cu; kernels receive its device address as a parameter.
int* device_error_word();

// Site codes recorded in the device error word.
enum ErrorSite : int {
  kSiteNone = 0,
  kSiteGemmProducer = 1,   // TMA producer waited too long for a free stage
  kSiteGemmMma = 2,        // MMA issuer waited too long for a full stage
  kSiteGemmEpilogue = 3,   // epilogue waited too long for the accumulator
  kSiteGemmTmemFree = 4,   // MMA issuer waited too long for the epilogue
  kSiteClusterRecv = 5,    // a CTA waited too long for its cluster peers' partial sums
  kSiteBatchRecv = 6,      // a batched-call CTA waited too long for its neighbours' published parts
  kSiteGridBarrier = 7,    // a CTA of the quantize-then-GEMM launch waited too long for the others
};

struct WoArgs {           // weight-only GEMM (W4A16 / W8A16)
  int M, N, K;
  const void* X; int64_t ldx;
  const void* W; int64_t ldw;
  const void* scales;
  void* Y; int64_t ldy;
  void* ws; size_t ws_bytes;  // caller scratch (split-K partial sums and tile counters)
  // Column groups: scales[n / group_n]; zeros (uint8 for INT4, int8 for
  // INT8, one per group) or nullptr for the fixed zero point (8 / 0).
  const void* zeros = nullptr;
  int group_n = 1;
};

struct MxQuantArgs {
  int rows, cols;
  const float* src; int64_t ld_src;
  uint8_t* data; int64_t ld_data;
  uint8_t* scales; int64_t ld_scales;
};

// Block scales of the FP4 GEMMs in the tensor cores' layout.  Rows are padded
// to a multiple of 256 and K to a multiple of 256 elements.  Row group g (rows
// 128 g .. 128 g + 127) holds tc_sf_chunks(nv, K) chunks of 512 bytes; chunk c
// holds the scales of blocks 4 c .. 4 c + 3 of the group's rows, the scale of
// row r and block b at byte 16 (r % 32) + 4 ((r / 32) % 4) + b % 4: the order
// in which tcgen05.cp 32x128b.warpx4 copies a chunk into four TMEM columns.
// Chunk (g, c) starts at byte 512 (g tc_sf_chunks + c).  Padding holds a
// finite scale (2^0 for E8M0, 0 for E4M3), so zero-filled data stays zero.
constexpr int kTcSfChunk = 512;
__host__ __device__ inline int tc_sf_chunks(bool nv, int K) { return ((K + 255) / 256) * (nv ? 4 : 2); }
inline size_t tc_sf_bytes(bool nv, int rows, int K) {
  return static_cast<size_t>((rows + 255) / 256) * 2 * tc_sf_chunks(nv, K) * kTcSfChunk;
}

struct MxGemmArgs {  // MXFP4 and NVFP4 GEMMs
  int M, N, K;
  const uint8_t* A; int64_t lda;
  const uint8_t* SA;  // A's block scales, tensor-core layout
  const uint8_t* W; int64_t ldw;
  const uint8_t* SW;  // W's block scales, tensor-core layout
  float* C; int64_t ldc;
  const float* ga = nullptr;  // NVFP4: the tensor scales of A and W (device memory)
  const float* gw = nullptr;
  // mx_gemm_fp4_qa: A arrives as FP32 (A32, row stride lda32 elements) and
  // the launch quantizes it first, into codes Aq [M, K/2] (row stride ldq) and
  // scales SA (the tensor-core layout) in the workspace, meeting at a grid
  // barrier whose two words are grid_bar.
  const float* A32 = nullptr; int64_t lda32 = 0;
  uint8_t* Aq = nullptr; int64_t ldq = 0;
  uint8_t* SAq = nullptr;
  unsigned* grid_bar = nullptr;
};

struct NvQuantArgs {
  int rows, cols;
  const float* src; int64_t ld_src;
  uint8_t* data; int64_t ld_data;
  uint8_t* scales; int64_t ld_scales;
  float* tensor_scale;  // device: receives the tensor scale
};

struct Fp8GemmArgs {
  int M, N, K;
  const uint8_t* A; int64_t lda;
  const uint8_t* B; int64_t ldb;
  float scale_a, scale_b;
  void* C; int64_t ldc;
  void* ws; size_t ws_bytes;  // caller scratch of the small-M path
};

// Work split of one call of the skinny weight-stream kernel, computed once
// per call (plan_skinny) so that the workspace check and the launch see the
// same plan.  U = tiles * chunks units over `grid` CTAs; CTA b owns units
// [b*U/G, (b+1)*U/G).  cluster > 1: the grid is tiles * cluster CTAs in
// clusters of that size; CTA b's run is then chunks [r ch / S, (r + 1) ch / S)
// of tile b / S (r its rank), and the cluster adds its partial tiles through
// distributed shared memory instead of the workspace.
struct SkinnyPlan {
  int n_tiles, tiles, chunks, grid, slots, cluster;
  int64_t units;
  int mt;           // 8-row activation groups per M tile (1 or 2): the kernel instance
  size_t ws_bytes;  // workspace this plan needs (0: every tile finished by one CTA or one cluster)
};
// mode: 4 (INT4), 8 (INT8) or 9 (e4m3 B operand of the small-M FP8 GEMM).
// An empty problem gives a zero plan.
SkinnyPlan plan_skinny(int M, int N, int K, int mode);

// Launchers (one per kernel family).  Each returns a cudaError_t from the
// launch; argument validation happened in wq_api.cu.
cudaError_t launch_wo_skinny(const WoArgs& a, int bits, const SkinnyPlan& pl, cudaStream_t s);
cudaError_t launch_wo_gemm(const WoArgs& a, int bits, cudaStream_t s);
cudaError_t launch_mx_quantize(const MxQuantArgs& a, cudaStream_t s);
cudaError_t launch_mx_gemm(const MxGemmArgs& a, cudaStream_t s);
cudaError_t launch_mx_gemm_qa(const MxGemmArgs& a, cudaStream_t s);  // A from FP32 in the same launch
// Row-major block scales S [rows, K / block] (row stride lds bytes) -> the
// tensor-core layout above, tc_sf_bytes(nv, rows, K) bytes at out.
cudaError_t launch_fp4_scales_tc(bool nv, int rows, int K, const uint8_t* S, int64_t lds, uint8_t* out,
                                 cudaStream_t s);
cudaError_t launch_nv_gemm(const MxGemmArgs& a, cudaStream_t s);
cudaError_t launch_nv_quantize(const NvQuantArgs& a, cudaStream_t s);
cudaError_t launch_fp8_gemm(const Fp8GemmArgs& a, cudaStream_t s);



// Batched skinny weight-only GEMMs (wo_batched.cu): up to kMaxBatch problems
// of one weight kind in one launch.  Problems with M, N or K = 0 take no
// units (K = 0 ones get Y = 0 from the launcher).
constexpr int kMaxBatch = 8;
struct BatchPlan {
  int units;         // units of all problems
  int grid;          // CTAs (one per SM, at most one per unit)
  int mt;            // 8-row activation groups per M tile: 2 if any problem has M > 8
  size_t ws_bytes;   // workspace: the tile counters and two published parts per CTA
  bool unsupported;  // too many tiles or units for one launch
};
BatchPlan plan_batched(const WoArgs* probs, int count, int bits);
cudaError_t launch_wo_batched(const WoArgs* probs, int count, int bits, const BatchPlan& pl, void* ws,
                              cudaStream_t s);

// Small-M FP8 (M <= kFp8SkinnyMaxM) runs on the skinny path as an e4m3
// weight stream.
constexpr int kFp8SkinnyMaxM = 16;
cudaError_t launch_fp8_skinny(const Fp8GemmArgs& a, const SkinnyPlan& pl, cudaStream_t s);

int sm_count();

// Built-in scratch of the allocation-free INT8 entry point (wo_skinny.cu).
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
cudaError_t noalloc_scratch(void** ptr);  // device address on the current device
size_t skinny_counter_bytes();            // leading counter area that must start at zero

}  // namespace wq
