// C ABI of libwq: host-side argument validation and shape dispatch.  Every
// entry point checks its arguments before any CUDA call and returns a WQ_*
// status; no exception crosses the boundary.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "wq_internal.h"

namespace wq {

namespace {
__device__ int g_device_error;  // first site code recorded by a bounded wait

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int launch_status(cudaError_t e) {
  if (e == cudaSuccess) return WQ_OK;
  cudaGetLastError();  // clear the sticky-free launch error so later calls are unaffected
  return WQ_ERR_LAUNCH;
}
}  // namespace

namespace {
std::atomic<uint64_t> g_skinny_wait_ns{2000000000ull};
}  // namespace

uint64_t skinny_wait_ns() { return g_skinny_wait_ns.load(std::memory_order_relaxed); }
std::atomic<int> g_static_weights{0};
bool static_weights() { return g_static_weights.load(std::memory_order_relaxed) != 0; }

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) d = 0;
  return d;
}

int* device_error_word() {
  static PerDevice<int*> words;
  int* ptr = nullptr;
  words.get(ptr, [](int*& p) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_device_error) != cudaSuccess) return false;
    p = static_cast<int*>(a);
    return true;
  });
  return ptr;  // nullptr if the lookup failed: kernels then record nothing
}

int sm_count() {
  static PerDevice<int> counts;
  int n = 0;
  if (!counts.get(n, [](int& v) {
        return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, current_device()) == cudaSuccess && v > 0;
      }))
    n = 148;  // the query failed (the launch that follows reports the error)
  return n;
}

// Shared validation of the weight-only GEMMs.
static int check_weight_only(int M, int N, int K, const void* X, int64_t ldx, const void* W, int64_t ldw,
                             const void* scales, const void* Y, int64_t ldy) {
  if (M < 0 || N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return WQ_OK;
  if (!Y || !scales || (K > 0 && (!X || !W))) return WQ_ERR_INVALID_ARG;
  if (K % 2) return WQ_ERR_INVALID_ARG;
  if (ldy < N || (K > 0 && ldx < K)) return WQ_ERR_INVALID_ARG;
  if (!aligned(Y, 16) || !aligned(scales, 2) || ldy % 8) return WQ_ERR_MISALIGNED;
  if (K > 0 && (!aligned(X, 16) || !aligned(W, 16) || ldx % 8 || ldw % 16)) return WQ_ERR_MISALIGNED;
  return WQ_OK;
}

// M up to this bound runs the split-K skinny path (HBM-bound); larger M the
// tensor-memory GEMM (up to 64 rows: one activation tile with K split over a
// cluster; beyond: 128- or 256-row tiles).
constexpr int kSkinnyMaxM = 16;
// The batched call runs every problem on the skinny kernel.
constexpr int kBatchedMaxM = 64;

// The tiled GEMMs put 128-row M tiles on the grid's y dimension (at most
// 65535 blocks); larger M is refused on the host instead of failing to launch.
constexpr int64_t kMaxTiledM = int64_t(65535) * 128;

static size_t weight_only_workspace(int bits, int M, int N, int K) {
  return (M > 0 && M <= kSkinnyMaxM) ? plan_skinny(M, N, K, bits).ws_bytes : 0;
}

// The skinny path's plan is made once here: the workspace is checked against
// this plan's need and the same plan is launched.
static int run_weight_only(int bits, int M, int N, int K, const void* X, int64_t ldx, const void* W, int64_t ldw,
                           const void* scales, void* Y, int64_t ldy, void* ws, size_t ws_bytes, cudaStream_t s,
                           const void* zeros = nullptr, int group_n = 1) {
  if (M == 0 || N == 0) return WQ_OK;
  if (M > kMaxTiledM) return WQ_ERR_UNSUPPORTED;
  WoArgs a{M, N, K, X, ldx, W, ldw, scales, Y, ldy, ws, ws_bytes, zeros, group_n};
  if (M > kSkinnyMaxM) return launch_status(launch_wo_gemm(a, bits, s));
  const SkinnyPlan pl = plan_skinny(M, N, K, bits);
  if (ws_bytes < pl.ws_bytes || (pl.ws_bytes > 0 && (!ws || !aligned(ws, 16)))) return WQ_ERR_WORKSPACE;
  return launch_status(launch_wo_skinny(a, bits, pl, s));
}

}  // namespace wq

using namespace wq;

extern "C" {

int wq_gemm_w4a16(int M, int N, int K, const void* X, int64_t ldx, const uint8_t* Wq, int64_t ldw,
                  const void* scales, void* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                  wq_stream_t stream) {
  int st = check_weight_only(M, N, K, X, ldx, Wq, ldw, scales, Y, ldy);
  if (st != WQ_OK || M == 0 || N == 0) return st;
  if (K > 0 && ldw < N) return WQ_ERR_INVALID_ARG;
  return run_weight_only(4, M, N, K, X, ldx, Wq, ldw, scales, Y, ldy, workspace, ws_bytes,
                         reinterpret_cast<cudaStream_t>(stream));
}

int wq_gemm_w8a16(int M, int N, int K, const void* X, int64_t ldx, const int8_t* W, int64_t ldw,
                  const void* scales, void* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                  wq_stream_t stream) {
  if (K % 2 && K > 0 && M >= 0 && N >= 0) return WQ_ERR_UNSUPPORTED;
  int st = check_weight_only(M, N, K, X, ldx, W, ldw, scales, Y, ldy);
  if (st != WQ_OK || M == 0 || N == 0) return st;
  if (K > 0 && ldw < N) return WQ_ERR_INVALID_ARG;
  return run_weight_only(8, M, N, K, X, ldx, W, ldw, scales, Y, ldy, workspace, ws_bytes,
                         reinterpret_cast<cudaStream_t>(stream));
}

int wq_gemm_w4a16_grouped(int M, int N, int K, const void* X, int64_t ldx, const uint8_t* Wq, int64_t ldw,
                          const void* scales, const uint8_t* zeros, int group_n, void* Y, int64_t ldy,
                          void* workspace, size_t ws_bytes, wq_stream_t stream) {
  if (group_n < 1) return WQ_ERR_INVALID_ARG;
  int st = check_weight_only(M, N, K, X, ldx, Wq, ldw, scales, Y, ldy);
  if (st != WQ_OK || M == 0 || N == 0) return st;
  if (K > 0 && ldw < N) return WQ_ERR_INVALID_ARG;
  return run_weight_only(4, M, N, K, X, ldx, Wq, ldw, scales, Y, ldy, workspace, ws_bytes,
                         reinterpret_cast<cudaStream_t>(stream), zeros, group_n);
}

int wq_gemm_w8a16_grouped(int M, int N, int K, const void* X, int64_t ldx, const int8_t* W, int64_t ldw,
                          const void* scales, const int8_t* zeros, int group_n, void* Y, int64_t ldy,
                          void* workspace, size_t ws_bytes, wq_stream_t stream) {
  if (group_n < 1) return WQ_ERR_INVALID_ARG;
  if (K % 2 && K > 0 && M >= 0 && N >= 0) return WQ_ERR_UNSUPPORTED;
  int st = check_weight_only(M, N, K, X, ldx, W, ldw, scales, Y, ldy);
  if (st != WQ_OK || M == 0 || N == 0) return st;
  if (K > 0 && ldw < N) return WQ_ERR_INVALID_ARG;
  return run_weight_only(8, M, N, K, X, ldx, W, ldw, scales, Y, ldy, workspace, ws_bytes,
                         reinterpret_cast<cudaStream_t>(stream), zeros, group_n);
}

int wq_gemm_w8a16_noalloc(int M, int N, int K, const void* X, int64_t ldx, const int8_t* W, int64_t ldw,
                          const void* scales, void* Y, int64_t ldy, wq_stream_t stream) {
  if (K % 2 && K > 0 && M >= 0 && N >= 0) return WQ_ERR_UNSUPPORTED;
  int st = check_weight_only(M, N, K, X, ldx, W, ldw, scales, Y, ldy);
  if (st != WQ_OK || M == 0 || N == 0) return st;
  if (K > 0 && ldw < N) return WQ_ERR_INVALID_ARG;
  if (M > kMaxTiledM) return WQ_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  WoArgs a{M, N, K, X, ldx, W, ldw, scales, Y, ldy, nullptr, 0, nullptr, 1};
  if (M > kSkinnyMaxM) return launch_status(launch_wo_gemm(a, 8, s));
  // One plan for the size check and the launch.
  const SkinnyPlan pl = plan_skinny(M, N, K, 8);
  if (pl.ws_bytes > kNoAllocScratchBytes) return WQ_ERR_WORKSPACE;  // beyond the built-in scratch
  if (pl.ws_bytes > 0) {
    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return launch_status(cudaErrorInvalidValue);
    // The array keeps the previous call's bytes: the tile counters must start at zero.
    if (cudaMemsetAsync(scratch, 0, skinny_counter_bytes(), s) != cudaSuccess) return launch_status(cudaErrorInvalidValue);
    a.ws = scratch;
    a.ws_bytes = kNoAllocScratchBytes;
  }
  return launch_status(launch_wo_skinny(a, 8, pl, s));
}

// Batched weight-only GEMMs: every problem is checked like a single call and
// the batch is planned once; the same plan serves the workspace check and the
// launch.
static int prepare_batched(int bits, int count, const wq_problem* problems, WoArgs (&a)[kMaxBatch], BatchPlan& pl) {
  if (count < 1 || count > kMaxBatch || !problems) return WQ_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    const wq_problem& q = problems[i];
    if (q.group_n < 1) return WQ_ERR_INVALID_ARG;
    if (bits == 8 && q.K % 2 && q.K > 0 && q.M >= 0 && q.N >= 0) return WQ_ERR_UNSUPPORTED;
    const int st = check_weight_only(q.M, q.N, q.K, q.X, q.ldx, q.W, q.ldw, q.scales, q.Y, q.ldy);
    if (st != WQ_OK) return st;
    if (q.M > 0 && q.N > 0 && q.K > 0 && q.ldw < q.N) return WQ_ERR_INVALID_ARG;
    if (q.M > kBatchedMaxM) return WQ_ERR_UNSUPPORTED;
    a[i] = WoArgs{q.M, q.N, q.K, q.X, q.ldx, q.W, q.ldw, q.scales, q.Y, q.ldy, nullptr, 0, nullptr, q.group_n};
  }
  pl = plan_batched(a, count, bits);
  return pl.unsupported ? WQ_ERR_UNSUPPORTED : WQ_OK;
}

static int run_batched(int bits, int count, const wq_problem* problems, void* ws, size_t ws_bytes, cudaStream_t s) {
  WoArgs a[kMaxBatch];
  BatchPlan pl = {};
  const int st = prepare_batched(bits, count, problems, a, pl);
  if (st != WQ_OK) return st;
  if (ws_bytes < pl.ws_bytes || (pl.ws_bytes > 0 && (!ws || !aligned(ws, 16)))) return WQ_ERR_WORKSPACE;
  return launch_status(launch_wo_batched(a, count, bits, pl, ws, s));
}

int mx_quantize_fp4(int rows, int cols, const float* src, int64_t ld_src, uint8_t* data, int64_t ld_data,
                    uint8_t* scales, int64_t ld_scales, wq_stream_t stream) {
  if (rows < 0 || cols < 0 || cols % 32) return WQ_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return WQ_OK;
  if (!src || !data || !scales) return WQ_ERR_INVALID_ARG;
  if (ld_src < cols || ld_data < cols / 2 || ld_scales < cols / 32) return WQ_ERR_INVALID_ARG;
  if (!aligned(src, 16) || ld_src % 4 || !aligned(data, 4) || ld_data % 4) return WQ_ERR_MISALIGNED;
  if (static_cast<int64_t>(rows) * (cols / 32) >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;  // 32-bit block ids
  MxQuantArgs a{rows, cols, src, ld_src, data, ld_data, scales, ld_scales};
  return launch_status(launch_mx_quantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

// FP4 GEMMs.  The kernels read block scales in the tensor-core layout
// (tc_sf_chunks); the row-major entry points first rearrange both operands'
// scales into the caller's workspace.
static size_t fp4_ws_a_bytes(bool nv, int M, int K) { return (tc_sf_bytes(nv, M, K) + 255) & ~size_t(255); }

static int check_fp4_gemm(bool nv, int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* W, int64_t ldw,
                          const float* C, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0 || K % (nv ? 16 : 32)) return WQ_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return WQ_OK;
  if (!C || (K > 0 && (!A || !W))) return WQ_ERR_INVALID_ARG;
  if (ldc < N || (K > 0 && (lda < K / 2 || ldw < K / 2))) return WQ_ERR_INVALID_ARG;
  if (!aligned(C, 16) || ldc % 4) return WQ_ERR_MISALIGNED;
  if (K > 0 && (!aligned(A, 16) || !aligned(W, 16) || lda % 16 || ldw % 16)) return WQ_ERR_MISALIGNED;
  if (M > kMaxTiledM || N > kMaxTiledM) return WQ_ERR_UNSUPPORTED;
  return WQ_OK;
}

// Row-major scales -> workspace in the tensor-core layout, then the GEMM.
static int fp4_gemm_rowmajor(bool nv, MxGemmArgs a, const uint8_t* SA, int64_t ldsa, const uint8_t* SW, int64_t ldsw,
                             void* workspace, size_t ws_bytes, cudaStream_t s) {
  const int st = check_fp4_gemm(nv, a.M, a.N, a.K, a.A, a.lda, a.W, a.ldw, a.C, a.ldc);
  if (st != WQ_OK || a.M == 0 || a.N == 0) return st;
  if (a.K > 0) {
    if (!SA || !SW) return WQ_ERR_INVALID_ARG;
    const int nb = a.K / (nv ? 16 : 32);
    if (ldsa < nb || ldsw < nb) return WQ_ERR_INVALID_ARG;
    if (ws_bytes < wq_workspace_size(nv ? WQ_OP_NV_GEMM : WQ_OP_MX_GEMM, a.M, a.N, a.K) || !workspace ||
        !aligned(workspace, 256))
      return WQ_ERR_WORKSPACE;
    uint8_t* sa_tc = static_cast<uint8_t*>(workspace);
    uint8_t* sw_tc = sa_tc + fp4_ws_a_bytes(nv, a.M, a.K);
    cudaError_t e = launch_fp4_scales_tc(nv, a.M, a.K, SA, ldsa, sa_tc, s);
    if (e == cudaSuccess) e = launch_fp4_scales_tc(nv, a.N, a.K, SW, ldsw, sw_tc, s);
    if (e != cudaSuccess) return launch_status(e);
    a.SA = sa_tc;
    a.SW = sw_tc;
  }
  return launch_status(nv ? launch_nv_gemm(a, s) : launch_mx_gemm(a, s));
}

// Scales already in the tensor-core layout.
static int fp4_gemm_tc(bool nv, const MxGemmArgs& a, size_t sa_bytes, size_t sw_bytes, cudaStream_t s) {
  const int st = check_fp4_gemm(nv, a.M, a.N, a.K, a.A, a.lda, a.W, a.ldw, a.C, a.ldc);
  if (st != WQ_OK || a.M == 0 || a.N == 0) return st;
  if (a.K > 0) {
    if (!a.SA || !a.SW) return WQ_ERR_INVALID_ARG;
    if (sa_bytes < tc_sf_bytes(nv, a.M, a.K) || sw_bytes < tc_sf_bytes(nv, a.N, a.K)) return WQ_ERR_INVALID_ARG;
    if (!aligned(a.SA, 16) || !aligned(a.SW, 16)) return WQ_ERR_MISALIGNED;
  }
  return launch_status(nv ? launch_nv_gemm(a, s) : launch_mx_gemm(a, s));
}

int mx_gemm_fp4(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* SA, int64_t ldsa,
                const uint8_t* W, int64_t ldw, const uint8_t* SW, int64_t ldsw, float* C, int64_t ldc,
                void* workspace, size_t ws_bytes, wq_stream_t stream) {
  MxGemmArgs a{M, N, K, A, lda, nullptr, W, ldw, nullptr, C, ldc};
  return fp4_gemm_rowmajor(false, a, SA, ldsa, SW, ldsw, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int mx_gemm_fp4_tc(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* SA, size_t sa_bytes,
                   const uint8_t* W, int64_t ldw, const uint8_t* SW, size_t sw_bytes, float* C, int64_t ldc,
                   wq_stream_t stream) {
  MxGemmArgs a{M, N, K, A, lda, SA, W, ldw, SW, C, ldc};
  return fp4_gemm_tc(false, a, sa_bytes, sw_bytes, reinterpret_cast<cudaStream_t>(stream));
}

// mx_gemm_fp4_qa workspace: the grid barrier's words, A's codes, A's scales
// (tensor-core layout), each part starting on a 256-byte boundary.
static int64_t qa_ldq(int K) { return (static_cast<int64_t>(K / 2) + 15) / 16 * 16; }
static size_t qa_codes_bytes(int M, int K) { return (static_cast<size_t>(M) * qa_ldq(K) + 255) & ~size_t(255); }
constexpr size_t kQaBarrierBytes = 256;

int mx_gemm_fp4_qa(int M, int N, int K, const float* A, int64_t lda, const uint8_t* W, int64_t ldw, const uint8_t* SW,
                   size_t sw_bytes, float* C, int64_t ldc, void* workspace, size_t ws_bytes, wq_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || K % 32) return WQ_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return WQ_OK;
  if (!C || ldc < N) return WQ_ERR_INVALID_ARG;
  if (!aligned(C, 16) || ldc % 4) return WQ_ERR_MISALIGNED;
  if (M > kMaxTiledM || N > kMaxTiledM) return WQ_ERR_UNSUPPORTED;
  if (K > 0) {
    if (!A || !W || !SW || lda < K || ldw < K / 2) return WQ_ERR_INVALID_ARG;
    if (sw_bytes < tc_sf_bytes(false, N, K)) return WQ_ERR_INVALID_ARG;
    if (!aligned(A, 16) || lda % 4 || !aligned(W, 16) || ldw % 16 || !aligned(SW, 16)) return WQ_ERR_MISALIGNED;
    // 32-bit item counters in the quantize phase
    if (static_cast<int64_t>((M + 255) / 256 * 256) * tc_sf_chunks(false, K) >= (int64_t(1) << 31))
      return WQ_ERR_UNSUPPORTED;
    if (ws_bytes < wq_workspace_size(WQ_OP_MX_GEMM_QA, M, N, K) || !workspace || !aligned(workspace, 256))
      return WQ_ERR_WORKSPACE;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  MxGemmArgs a{M, N, K, nullptr, 0, nullptr, W, ldw, SW, C, ldc};
  a.A32 = A;
  a.lda32 = lda;
  a.grid_bar = reinterpret_cast<unsigned*>(ws);
  a.Aq = ws + kQaBarrierBytes;
  a.ldq = qa_ldq(K);
  a.SAq = a.Aq + qa_codes_bytes(M, K);
  a.A = a.Aq;
  a.lda = a.ldq;
  a.SA = a.SAq;
  return launch_status(launch_mx_gemm_qa(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t fp4_scales_tc_size(int format, int rows, int K) {
  if ((format != WQ_FP4_MX && format != WQ_FP4_NV) || rows <= 0 || K <= 0) return 0;
  if (K % (format == WQ_FP4_NV ? 16 : 32)) return 0;
  return tc_sf_bytes(format == WQ_FP4_NV, rows, K);
}

int fp4_scales_tc(int format, int rows, int K, const uint8_t* S, int64_t lds, uint8_t* out, size_t out_bytes,
                  wq_stream_t stream) {
  if (format != WQ_FP4_MX && format != WQ_FP4_NV) return WQ_ERR_INVALID_ARG;
  const bool nv = format == WQ_FP4_NV;
  if (rows < 0 || K < 0 || K % (nv ? 16 : 32)) return WQ_ERR_INVALID_ARG;
  if (rows == 0 || K == 0) return WQ_OK;
  if (!S || !out || lds < K / (nv ? 16 : 32)) return WQ_ERR_INVALID_ARG;
  if (out_bytes < tc_sf_bytes(nv, rows, K)) return WQ_ERR_INVALID_ARG;
  if (!aligned(out, 16)) return WQ_ERR_MISALIGNED;
  if (rows > kMaxTiledM) return WQ_ERR_UNSUPPORTED;
  return launch_status(launch_fp4_scales_tc(nv, rows, K, S, lds, out, reinterpret_cast<cudaStream_t>(stream)));
}

int nv_quantize_fp4(int rows, int cols, const float* src, int64_t ld_src, uint8_t* data, int64_t ld_data,
                    uint8_t* scales, int64_t ld_scales, float* tensor_scale, wq_stream_t stream) {
  if (rows < 0 || cols < 0 || cols % 16 || !tensor_scale) return WQ_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0) {
    if (!src || !data || !scales) return WQ_ERR_INVALID_ARG;
    if (ld_src < cols || ld_data < cols / 2 || ld_scales < cols / 16) return WQ_ERR_INVALID_ARG;
    if (!aligned(src, 16) || ld_src % 4 || !aligned(data, 8) || ld_data % 8) return WQ_ERR_MISALIGNED;
    if (static_cast<int64_t>(rows) * (cols / 16) >= (int64_t(1) << 31)) return WQ_ERR_UNSUPPORTED;
  }
  if (!aligned(tensor_scale, 4)) return WQ_ERR_MISALIGNED;
  NvQuantArgs a{rows, cols, src, ld_src, data, ld_data, scales, ld_scales, tensor_scale};
  return launch_status(launch_nv_quantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

static int check_nv_scales(int M, int N, int K, const float* scale_a, const float* scale_w) {
  if (M <= 0 || N <= 0 || K <= 0) return WQ_OK;
  if (!scale_a || !scale_w) return WQ_ERR_INVALID_ARG;
  if (!aligned(scale_a, 4) || !aligned(scale_w, 4)) return WQ_ERR_MISALIGNED;
  return WQ_OK;
}

int nv_gemm_fp4(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* SA, int64_t ldsa,
                const float* scale_a, const uint8_t* W, int64_t ldw, const uint8_t* SW, int64_t ldsw,
                const float* scale_w, float* C, int64_t ldc, void* workspace, size_t ws_bytes, wq_stream_t stream) {
  const int st = check_fp4_gemm(true, M, N, K, A, lda, W, ldw, C, ldc);
  if (st != WQ_OK) return st;
  const int sg = check_nv_scales(M, N, K, scale_a, scale_w);
  if (sg != WQ_OK) return sg;
  MxGemmArgs a{M, N, K, A, lda, nullptr, W, ldw, nullptr, C, ldc, scale_a, scale_w};
  return fp4_gemm_rowmajor(true, a, SA, ldsa, SW, ldsw, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int nv_gemm_fp4_tc(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* SA, size_t sa_bytes,
                   const float* scale_a, const uint8_t* W, int64_t ldw, const uint8_t* SW, size_t sw_bytes,
                   const float* scale_w, float* C, int64_t ldc, wq_stream_t stream) {
  const int st = check_fp4_gemm(true, M, N, K, A, lda, W, ldw, C, ldc);
  if (st != WQ_OK) return st;
  const int sg = check_nv_scales(M, N, K, scale_a, scale_w);
  if (sg != WQ_OK) return sg;
  MxGemmArgs a{M, N, K, A, lda, SA, W, ldw, SW, C, ldc, scale_a, scale_w};
  return fp4_gemm_tc(true, a, sa_bytes, sw_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int fp8_gemm(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb, float scale_a,
             float scale_b, void* C, int64_t ldc, void* workspace, size_t ws_bytes, wq_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return WQ_OK;
  if (!C || (K > 0 && (!A || !B))) return WQ_ERR_INVALID_ARG;
  if (ldc < N || (K > 0 && (lda < K || ldb < N))) return WQ_ERR_INVALID_ARG;
  if (!aligned(C, 16) || ldc % 8) return WQ_ERR_MISALIGNED;
  if (K > 0 && (!aligned(A, 16) || !aligned(B, 16) || lda % 16 || ldb % 16)) return WQ_ERR_MISALIGNED;
  // The tiled path counts its 128 x 256 tiles in 32 bits.
  if (M > kFp8SkinnyMaxM && (M > kMaxTiledM || N > kMaxTiledM)) return WQ_ERR_UNSUPPORTED;
  Fp8GemmArgs a{M, N, K, A, lda, B, ldb, scale_a, scale_b, C, ldc, workspace, ws_bytes};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M > kFp8SkinnyMaxM) return launch_status(launch_fp8_gemm(a, s));
  // One plan for the workspace check and the launch.
  const SkinnyPlan pl = plan_skinny(M, N, K, 9);
  if (ws_bytes < pl.ws_bytes || (pl.ws_bytes > 0 && (!workspace || !aligned(workspace, 16)))) return WQ_ERR_WORKSPACE;
  return launch_status(launch_fp8_skinny(a, pl, s));
}

int wq_gemm_w4a16_batched(int count, const wq_problem* problems, void* workspace, size_t ws_bytes,
                          wq_stream_t stream) {
  return run_batched(4, count, problems, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int wq_gemm_w8a16_batched(int count, const wq_problem* problems, void* workspace, size_t ws_bytes,
                          wq_stream_t stream) {
  return run_batched(8, count, problems, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t wq_batched_workspace_size(int op, int count, const wq_problem* problems) {
  if (op != WQ_OP_W4A16 && op != WQ_OP_W8A16) return 0;
  WoArgs a[kMaxBatch];
  BatchPlan pl = {};
  return prepare_batched(op == WQ_OP_W4A16 ? 4 : 8, count, problems, a, pl) == WQ_OK ? pl.ws_bytes : 0;
}

size_t wq_workspace_size(int op, int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if (op == WQ_OP_W4A16 && K % 2 == 0) return weight_only_workspace(4, M, N, K);
  if (op == WQ_OP_W8A16 && K % 2 == 0) return weight_only_workspace(8, M, N, K);
  if (op == WQ_OP_FP8_GEMM && M <= kFp8SkinnyMaxM) return plan_skinny(M, N, K, 9).ws_bytes;
  if (op == WQ_OP_MX_GEMM_QA && K % 32 == 0)
    return kQaBarrierBytes + qa_codes_bytes(M, K) + tc_sf_bytes(false, M, K);
  if ((op == WQ_OP_MX_GEMM && K % 32 == 0) || (op == WQ_OP_NV_GEMM && K % 16 == 0)) {
    const bool nv = op == WQ_OP_NV_GEMM;
    return fp4_ws_a_bytes(nv, M, K) + tc_sf_bytes(nv, N, K);
  }
  return 0;
}

const char* wq_status_string(int status) {
  switch (status) {
    case WQ_OK: return "WQ_OK";
    case WQ_ERR_INVALID_ARG: return "WQ_ERR_INVALID_ARG: null pointer, negative size, bad multiple or leading dimension";
    case WQ_ERR_MISALIGNED: return "WQ_ERR_MISALIGNED: pointer or leading dimension breaks the alignment rule";
    case WQ_ERR_UNSUPPORTED: return "WQ_ERR_UNSUPPORTED: shape form not served";
    case WQ_ERR_WORKSPACE: return "WQ_ERR_WORKSPACE: workspace smaller than wq_workspace_size()";
    case WQ_ERR_LAUNCH: return "WQ_ERR_LAUNCH: CUDA launch error";
    case WQ_ERR_DEVICE: return "WQ_ERR_DEVICE: a kernel gave up a bounded wait";
    default: return "WQ_ERR_UNKNOWN";
  }
}

int wq_get_device_error(wq_stream_t stream, int* site) {
  int* word = device_error_word();
  if (!word) return WQ_ERR_LAUNCH;
  int host = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&host, word, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return WQ_ERR_LAUNCH;
  if (cudaMemsetAsync(word, 0, sizeof(int), s) != cudaSuccess) return WQ_ERR_LAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return WQ_ERR_LAUNCH;
  if (site) *site = host;
  return host ? WQ_ERR_DEVICE : WQ_OK;
}

int wq_set_static_weights(int enable) {
  return g_static_weights.exchange(enable ? 1 : 0, std::memory_order_relaxed);
}

int wq_debug_set_wait_limit(int64_t ns) {
  g_skinny_wait_ns.store(ns > 0 ? static_cast<uint64_t>(ns) : 2000000000ull, std::memory_order_relaxed);
  return WQ_OK;
}

int wq_version(void) { return 400; }  // 0.4.0: NVFP4 quantizer and GEMM

}  // extern "C"
