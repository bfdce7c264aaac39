/*
 * wq.h — C ABI of libwq, a fused on-the-fly-dequantization GEMM library for
 * one NVIDIA GB300 (sm_103a).
 *
 * Pages the operations are defined by (cited by title and section):
 *   [W4A16]  "Triton 工业级融合微算子编写：W4A16 极速切片矩阵乘与 Blackwell NVFP4
 *            硬件指令实装", §二 fused W4A16 kernel.
 *   [MXFP4]  "量化推理引擎中的微缩放格式前瞻：MXFP4 矩阵乘法 Kernel 原理", §一
 *            micro-block layout, §二 tiling equations, §三 simulator.
 *   [W8A16]  "Triton 量化算子：W8A16 权重量化融合矩阵乘法 (Quantization GEMM)",
 *            Step 1 formula, Step 3 signature and layout, reference solution.
 *   [FP8]    "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核", kernel
 *            listing and the 精度管理 (precision management) bullet.
 *   [W4A16] §三 also names NVFP4, the format of nv_quantize_fp4 / nv_gemm_fp4.
 *
 * Conventions for every entry point below
 *   - Matrices are row-major.  A leading dimension ("ld*") is the distance in
 *     ELEMENTS between consecutive rows (bytes for the uint8 arrays); the
 *     inner stride is always 1.  Non-unit inner strides are not expressible.
 *   - All array pointers are DEVICE pointers (cudaMalloc'd or otherwise
 *     device-accessible).  The caller owns every buffer, including the
 *     optional workspace; the library allocates nothing and keeps no pointer
 *     after the call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Inputs must stay valid and outputs untouched until the stream
 *     work completes.  Outputs must not alias inputs.
 *   - Every call validates its arguments on the host before launching.  On an
 *     invalid argument it returns a WQ_ERR_* code and launches nothing.  No
 *     C++ exception crosses this boundary.
 *   - M, N or K equal to 0 is a valid empty problem: nothing is launched and
 *     WQ_OK is returned (for K == 0 with M, N > 0 the GEMMs write zeros).
 *   - Inputs must be finite; NaN/Inf inputs give unspecified (but in-bounds)
 *     results.
 *   - Shapes beyond the kernels' grid limits return WQ_ERR_UNSUPPORTED without
 *     launching: M > 8,388,480 (65535 tiles of 128 rows) for the weight-only
 *     and MXFP4 GEMMs and for the FP8 GEMM at M > 16 (there also
 *     N > 8,388,480), and 2^31 or more 32-element blocks for mx_quantize_fp4.
 */
#ifndef WQ_H_
#define WQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t / CUstream, so either may be passed. */
typedef struct CUstream_st* wq_stream_t;

/* Status codes. */
#define WQ_OK 0
#define WQ_ERR_INVALID_ARG 1  /* null pointer, negative size, ld < row width, bad K multiple */
#define WQ_ERR_MISALIGNED 2   /* base pointer or leading dimension breaks the 16-byte rule */
#define WQ_ERR_UNSUPPORTED 3  /* shape form the kernels do not serve (documented per call) */
#define WQ_ERR_WORKSPACE 4    /* workspace smaller than wq_workspace_size() */
#define WQ_ERR_LAUNCH 5       /* CUDA reported an error when launching */
#define WQ_ERR_DEVICE 6       /* a kernel gave up a bounded wait (see wq_get_device_error) */

/* Operation ids for wq_workspace_size(). */
#define WQ_OP_W4A16 0
#define WQ_OP_W8A16 1
#define WQ_OP_MX_QUANTIZE 2
#define WQ_OP_MX_GEMM 3
#define WQ_OP_FP8_GEMM 4
#define WQ_OP_NV_GEMM 5
#define WQ_OP_MX_GEMM_QA 6

/*
 * wq_gemm_w4a16 — Y = X * ((q - 8) * s), INT4 weights dequantized on chip.
 *
 * [W4A16] §二: the packed INT4 weight byte row k/2 holds the codes of k and
 * k+1; the code of k is (byte >> ((k % 2) * 4)) & 0xF (even k in the low
 * nibble); the weight is (q - 8) * s[n]; products accumulate in FP32 and the
 * result is stored as FP16.  The dequantized weight never leaves the chip.
 *
 *   M, N, K  problem size; K must be even (two codes per byte).
 *   X        fp16 [M, K], row stride ldx (elements, ldx >= K).
 *   Wq       uint8 [K/2, N], row stride ldw (bytes, ldw >= N).
 *   scales   fp16 [N], one per output column.
 *   Y        fp16 [M, N] output, row stride ldy (elements, ldy >= N).
 *   workspace, ws_bytes  device scratch of at least
 *            wq_workspace_size(WQ_OP_W4A16, M, N, K) bytes, 16-byte aligned
 *            (may be NULL when that size is 0).  For M <= 16 the K dimension
 *            may be split across CTAs that meet here: the first 64 KiB hold
 *            one counter per tile, the partial sums of split tiles follow.
 *            (16 < M <= 64 splits K inside a thread-block cluster and needs
 *            no workspace; larger M needs none either.)  Zero-fill the
 *            workspace once before its first use; every call that returns
 *            WQ_OK leaves the counter area zero again (the rest is scratch),
 *            so one buffer serves any sequence of calls and shapes on one
 *            stream.  Two calls in flight at the same time must not share a
 *            workspace.  After WQ_ERR_DEVICE zero it again before reuse.  Too
 *            small: WQ_ERR_WORKSPACE.
 * Alignment: X, Wq, Y 16-byte aligned; ldx and ldy multiples of 8; ldw a
 * multiple of 16; scales 2-byte aligned.  Otherwise WQ_ERR_MISALIGNED.
 */
int wq_gemm_w4a16(int M, int N, int K, const void* X, int64_t ldx,
                  const uint8_t* Wq, int64_t ldw, const void* scales,
                  void* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                  wq_stream_t stream);

/*
 * wq_gemm_w8a16 — Y = X * (W_int8 * S), INT8 weights dequantized on chip.
 *
 * [W8A16] Step 1 (Y = X x (W_int8 x S)) and Step 3 (X fp16 [M, K], W int8
 * [K, N], S fp16 [N] one scale per column, Y fp16 [M, N]); symmetric, no zero
 * point; FP32 accumulation as in the reference solution.
 *
 *   M, N, K  problem size; K must be even (the kernels pair K rows).
 *   X        fp16 [M, K], row stride ldx (elements).
 *   W        int8 [K, N], row stride ldw (bytes).
 *   scales   fp16 [N].
 *   Y        fp16 [M, N], row stride ldy (elements).
 *   workspace, ws_bytes  as for wq_gemm_w4a16, sized by
 *            wq_workspace_size(WQ_OP_W8A16, M, N, K).
 * Alignment: as for wq_gemm_w4a16.  Odd K returns WQ_ERR_UNSUPPORTED.
 */
int wq_gemm_w8a16(int M, int N, int K, const void* X, int64_t ldx,
                  const int8_t* W, int64_t ldw, const void* scales,
                  void* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                  wq_stream_t stream);

/*
 * wq_gemm_w8a16_noalloc — wq_gemm_w8a16 without a caller workspace.
 *
 * The pages have no counterpart to this entry point: it exists for callers
 * that cannot allocate device memory when they call (an engine plugin whose
 * enqueue step may not allocate, a real-time loop that forbids cudaMalloc and
 * cudaFree after start-up, a runtime that plans every device byte ahead).
 * It computes exactly what wq_gemm_w8a16 computes, with the same arguments
 * minus the workspace, and allocates nothing: the split-K scratch of the
 * small-M path lives in a fixed 1 MiB array of device memory inside the
 * library, which every GPU that loads the library holds until the process
 * exits.
 *
 *   - Shapes whose scratch need (wq_workspace_size(WQ_OP_W8A16, M, N, K))
 *     exceeds 1 MiB return WQ_ERR_WORKSPACE without launching.  Only
 *     shapes whose K is split across CTAs through scratch need any (small N
 *     with long K); most decode shapes need none.
 *   - The first call on a device looks up the array's device address; make
 *     that first call before capturing the stream into a CUDA graph.
 *   - Each call clears the array's counter area on `stream` before its
 *     kernel.  All calls share the one array, so calls that overlap on the
 *     GPU (different streams, or the same stream from different threads
 *     without ordering) race and give wrong results.
 */
int wq_gemm_w8a16_noalloc(int M, int N, int K, const void* X, int64_t ldx,
                          const int8_t* W, int64_t ldw, const void* scales,
                          void* Y, int64_t ldy, wq_stream_t stream);

/*
 * wq_gemm_w4a16_grouped, wq_gemm_w8a16_grouped — weight-only GEMMs whose
 * scales, and optional zero points, are shared by groups of columns.
 *
 * [W8A16] 扩展说明 (extensions): when N is large several columns may share one
 * scale, and a zero_point turns the symmetric scheme asymmetric; [W4A16] §一:
 * the dequantization w = (w_int4 - zero_point) * scale.  Columns
 * g*group_n .. (g+1)*group_n - 1 share scale s[g] and zero point z[g] (the
 * last group may be shorter):
 *     Y[m, n] = sum_k X[m, k] * (q[k, n] - z[n / group_n]) * s[n / group_n],
 * q being the INT4 code (0..15, unpacked as for wq_gemm_w4a16) or the INT8
 * value.  Both factors are constant along K; the products accumulate in FP32
 * and Y is stored as FP16.
 *
 *   group_n  columns per group, >= 1 (otherwise WQ_ERR_INVALID_ARG).
 *   scales   fp16 [ceil(N / group_n)], 2-byte aligned.
 *   zeros    NULL for the symmetric scheme (zero point 8 for INT4, 0 for
 *            INT8), else [ceil(N / group_n)] zero points: uint8 for INT4 (any
 *            value 0..255), int8 for INT8.
 *   Every other argument, the workspace size (wq_workspace_size with
 *   WQ_OP_W4A16 or WQ_OP_W8A16) and the alignment rules are those of
 *   wq_gemm_w4a16 / wq_gemm_w8a16.
 * group_n = 1 with zeros = NULL computes exactly what wq_gemm_w4a16 and
 * wq_gemm_w8a16 compute.
 */
int wq_gemm_w4a16_grouped(int M, int N, int K, const void* X, int64_t ldx,
                          const uint8_t* Wq, int64_t ldw, const void* scales,
                          const uint8_t* zeros, int group_n,
                          void* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                          wq_stream_t stream);
int wq_gemm_w8a16_grouped(int M, int N, int K, const void* X, int64_t ldx,
                          const int8_t* W, int64_t ldw, const void* scales,
                          const int8_t* zeros, int group_n,
                          void* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                          wq_stream_t stream);

/*
 * Batched weight-only GEMMs for decode-sized M: up to WQ_MAX_BATCH
 * independent problems of one weight kind in one launch.
 *
 * Every problem computes what wq_gemm_w4a16 / wq_gemm_w8a16 compute ([W4A16]
 * §二; [W8A16] Step 1 and Step 3), with group_n columns sharing one scale as
 * for the _grouped calls (group_n = 1: per-column scales, the pages'
 * layout); the symmetric zero points (8 for INT4, 0 for INT8) apply.  The
 * pages have no batched call: each of their kernels computes one product.
 * The batch exists because at M <= 16 a product moves only a few
 * microseconds' worth of HBM traffic and every launch pays a fixed ramp and
 * tail of the same order; one launch streams all the problems' weights
 * back to back and pays it once.  The results equal the single calls' within
 * the usual rounding (the K sums are split differently), and are
 * deterministic.
 *
 *   count     number of problems, 1..WQ_MAX_BATCH.
 *   problems  host array of `count` descriptors (read during the call only):
 *               M, N, K   sizes; 0 <= M <= 64 (larger M: WQ_ERR_UNSUPPORTED);
 *                         K even; a problem with M or N = 0 is skipped, one
 *                         with K = 0 gets Y = 0;
 *               X, ldx    fp16 [M, K] activations;
 *               W, ldw    packed INT4 uint8 [K/2, N] (wq_gemm_w4a16_batched)
 *                         or int8 [K, N] (wq_gemm_w8a16_batched);
 *               scales    fp16 [ceil(N / group_n)];
 *               group_n   columns per scale, >= 1;
 *               Y, ldy    fp16 [M, N] output.
 *             Alignment and leading-dimension rules are those of the single
 *             calls.  No output may overlap another problem's output or any
 *             input.
 *   workspace, ws_bytes  device scratch of at least
 *             wq_batched_workspace_size(op, count, problems) bytes, 16-byte
 *             aligned: a counter area (zero-fill once before first use;
 *             every call that returns WQ_OK leaves it zero) and the partial
 *             tiles that neighbouring CTAs hand to each other.  Two calls in
 *             flight at the same time must not share a workspace; after
 *             WQ_ERR_DEVICE zero it again.  Too small: WQ_ERR_WORKSPACE.
 * Errors: count outside 1..WQ_MAX_BATCH or problems == NULL give
 * WQ_ERR_INVALID_ARG; each problem is checked as its single call would be.
 */
#define WQ_MAX_BATCH 8

typedef struct wq_problem {
  int M, N, K;
  const void* X;
  int64_t ldx;
  const void* W;
  int64_t ldw;
  const void* scales;
  int group_n;
  void* Y;
  int64_t ldy;
} wq_problem;

int wq_gemm_w4a16_batched(int count, const wq_problem* problems, void* workspace, size_t ws_bytes,
                          wq_stream_t stream);
int wq_gemm_w8a16_batched(int count, const wq_problem* problems, void* workspace, size_t ws_bytes,
                          wq_stream_t stream);

/* Workspace bytes a batched call needs (op = WQ_OP_W4A16 or WQ_OP_W8A16) on
 * the current device; 0 when the batch is invalid or needs none. */
size_t wq_batched_workspace_size(int op, int count, const wq_problem* problems);

/*
 * mx_quantize_fp4 — quantize FP32 rows to MXFP4 (E2M1 elements, E8M0 scales).
 *
 * [MXFP4] §三 simulator, per 32-element block of each row:
 *   amax = max(max|x|, 1e-8); e = ceil(log2(amax / 6)) (exact, amax/6 in
 *   FP32); E = e + 127; v = x / 2^e; magnitude index j = nearest point of
 *   {0, .5, 1, 1.5, 2, 3, 4, 6} to |v|, the smaller one on a tie; sign bit set
 *   when x < 0; code = sign << 3 | j.
 * [MXFP4] §一: data and scale segments are separate arrays.
 *
 *   rows, cols  source size; cols must be a multiple of 32.
 *   src         fp32 [rows, cols], row stride ld_src (elements).
 *   data        uint8 [rows, cols/2] output: element 2t in the low nibble and
 *               2t+1 in the high nibble of byte t; row stride ld_data (bytes).
 *   scales      uint8 [rows, cols/32] output E8M0 bytes; row stride ld_scales.
 * Alignment: src 16-byte aligned and ld_src a multiple of 4; data 4-byte
 * aligned and ld_data a multiple of 4.  The output is bit-exact with the
 * definition above.
 */
int mx_quantize_fp4(int rows, int cols, const float* src, int64_t ld_src,
                    uint8_t* data, int64_t ld_data, uint8_t* scales,
                    int64_t ld_scales, wq_stream_t stream);

/*
 * mx_gemm_fp4 — C = A * W^T for MXFP4 operands, FP32 output.
 *
 * [MXFP4] §二.1 and §二.2: for every output (m, n) and 32-element K block k,
 *   dC = 2^(E_A[m,k] + E_W[n,k] - 254) * sum_{i<32} a[m,k,i] * w[n,k,i],
 * summed over the blocks in FP32 (§三: C = A @ W^T with A [M, K], W [N, K]).
 *
 *   M, N, K  problem size; K must be a multiple of 32.
 *   A, SA    A's data uint8 [M, K/2] (row stride lda bytes) and E8M0 scales
 *            uint8 [M, K/32] (row stride ldsa bytes), as mx_quantize_fp4
 *            writes them.
 *   W, SW    the same for W [N, K] (row strides ldw, ldsw).
 *   C        fp32 [M, N] output, row stride ldc (elements).
 *   workspace, ws_bytes  at least wq_workspace_size(WQ_OP_MX_GEMM, M, N, K)
 *            bytes, 256-byte aligned: the call first rewrites both scale
 *            arrays there in the tensor-core layout (fp4_scales_tc), then
 *            runs mx_gemm_fp4_tc.  Too small or NULL (K > 0):
 *            WQ_ERR_WORKSPACE.  Two calls in flight must not share it.
 * Alignment: A, W 16-byte aligned with lda, ldw multiples of 16; C 16-byte
 * aligned with ldc a multiple of 4.  M and N at most 65535 * 128.
 * When the output tiles are too few to fill the GPU (small M), K is split
 * across the CTAs of a thread-block cluster, which add their FP32 partial
 * tiles in distributed shared memory in a fixed order.  Every shape writes C
 * once, and two calls on the same inputs give identical bits.
 */
int mx_gemm_fp4(int M, int N, int K, const uint8_t* A, int64_t lda,
                const uint8_t* SA, int64_t ldsa, const uint8_t* W,
                int64_t ldw, const uint8_t* SW, int64_t ldsw, float* C,
                int64_t ldc, void* workspace, size_t ws_bytes,
                wq_stream_t stream);

/*
 * fp4_scales_tc — rearrange FP4 block scales into the tensor-core layout
 * that mx_gemm_fp4_tc and nv_gemm_fp4_tc read.
 *
 * The block-scaled tensor cores ([MXFP4] §二.1-§二.2: the block exponents
 * enter the dot product in hardware) read scales from tensor memory, copied
 * there in 512-byte chunks of 128 rows x 4 blocks.  This call writes the
 * scales in that order once, so that a GEMM moves them with plain bulk
 * copies.  For weights, do it once when the weights are loaded.
 *
 *   format   WQ_FP4_MX (E8M0 scales of 32-element blocks, K % 32 == 0) or
 *            WQ_FP4_NV (E4M3 scales of 16-element blocks, K % 16 == 0).
 *   rows, K  the operand's rows and K in elements (the scale array is
 *            [rows, K / block]).
 *   S        uint8 [rows, K / block] scales, row stride lds bytes (any
 *            alignment), as mx_quantize_fp4 / nv_quantize_fp4 write them.
 *   out      device buffer of at least fp4_scales_tc_size(format, rows, K)
 *            bytes (out_bytes), 16-byte aligned.
 * Layout of out: rows padded to a multiple of 256 and K to a multiple of
 * 256 elements; row group g = rows 128 g .. 128 g + 127 holds
 * Kc = (K_padded / 256) * (2 for MX, 4 for NV) chunks of 512 bytes; chunk
 * c of group g starts at byte 512 (g Kc + c) and holds blocks 4 c .. 4 c + 3
 * of the group's rows, the scale of row r, block b at byte
 * 16 (r % 32) + 4 ((r / 32) % 4) + b % 4.  Padding holds 0x7F (2^0) for
 * MX and 0x00 for NV.
 */
#define WQ_FP4_MX 0
#define WQ_FP4_NV 1
size_t fp4_scales_tc_size(int format, int rows, int K);
int fp4_scales_tc(int format, int rows, int K, const uint8_t* S, int64_t lds,
                  uint8_t* out, size_t out_bytes, wq_stream_t stream);

/*
 * mx_gemm_fp4_tc — mx_gemm_fp4 with both scale arrays already in the
 * tensor-core layout (fp4_scales_tc): no workspace, one kernel launch.
 *
 *   SA, sa_bytes  A's scales from fp4_scales_tc(WQ_FP4_MX, M, K, ...) and
 *                 that buffer's size; SW, sw_bytes the same for W (N rows).
 *                 A buffer smaller than fp4_scales_tc_size: WQ_ERR_INVALID_ARG.
 *   Every other argument, the result and the alignment rules are those of
 *   mx_gemm_fp4; SA and SW must be 16-byte aligned.
 */
int mx_gemm_fp4_tc(int M, int N, int K, const uint8_t* A, int64_t lda,
                   const uint8_t* SA, size_t sa_bytes, const uint8_t* W,
                   int64_t ldw, const uint8_t* SW, size_t sw_bytes, float* C,
                   int64_t ldc, wq_stream_t stream);

/*
 * mx_gemm_fp4_qa — C = MXFP4(A) * W^T with A given in FP32, quantized inside
 * the GEMM's own launch.
 *
 * [MXFP4] §三: the simulator quantizes both A and W to MXFP4 (32-element
 * blocks, E8M0 exponents, nearest E2M1 codes) and then runs the block-scaled
 * GEMM.  Here W is quantized beforehand (weights) and A, the activations, is
 * quantized by the GEMM launch itself: every CTA first quantizes its share
 * of A with exactly mx_quantize_fp4's arithmetic, into the workspace, the
 * grid meets at one barrier, and the GEMM reads those codes and scales.
 * No separate quantize launch and no re-layout of A's scales; C equals
 * mx_quantize_fp4 of A followed by mx_gemm_fp4, bit for bit.
 *
 *   A        fp32 [M, K], row stride lda (elements); K % 32 == 0.
 *   W, SW    W's codes uint8 [N, K/2] (row stride ldw) and its scales in
 *            the tensor-core layout (fp4_scales_tc with WQ_FP4_MX, N rows),
 *            sw_bytes the size of that buffer.
 *   C        fp32 [M, N], row stride ldc.
 *   workspace, ws_bytes  at least wq_workspace_size(WQ_OP_MX_GEMM_QA, M, N,
 *            K) bytes, 256-byte aligned.  Its first 8 bytes (the grid
 *            barrier's counters) must be zero before the first call; every
 *            call that returns WQ_OK leaves them zero.  After WQ_ERR_DEVICE
 *            zero them again.  Two calls in flight must not share it.  After
 *            the call the workspace holds the quantized A, for reuse: its
 *            codes uint8 [M, ldq] at byte 256 (ldq = K/2 rounded up to a
 *            multiple of 16, the codes of mx_quantize_fp4 in the first K/2
 *            bytes of each row), then, at the next 256-byte boundary, its
 *            scales in the tensor-core layout (fp4_scales_tc of A's scales).
 * Alignment: A 16-byte aligned with lda a multiple of 4; W, SW 16-byte
 * aligned with ldw a multiple of 16; C as for mx_gemm_fp4.
 * The launch is cooperative (all of its CTAs are resident at once); when
 * its CTAs cannot all be resident the call returns WQ_ERR_LAUNCH.
 */
int mx_gemm_fp4_qa(int M, int N, int K, const float* A, int64_t lda,
                   const uint8_t* W, int64_t ldw, const uint8_t* SW,
                   size_t sw_bytes, float* C, int64_t ldc, void* workspace,
                   size_t ws_bytes, wq_stream_t stream);

/*
 * nv_quantize_fp4 — quantize FP32 rows to NVFP4: E2M1 elements in 16-element
 * blocks, one E4M3 scale per block, one FP32 scale per tensor.
 *
 * [W4A16] §三 names NVFP4 as E2M1 elements under a two-level block scaling
 * with an FP8 local block scale, executed natively by the 5th-generation
 * tensor cores, and gives no block size or encoding.  The reading: 16-element
 * blocks along the row; with g = amax(|src|) / 2688 (6 x 448; g = 1 for an
 * all-zero tensor), each block's scale is s = e4m3(amax_block / (6 g)), the
 * nearest E4M3 value with ties to the even code, saturating at 448; each
 * element's code is the nearest E2M1 grid point to x / (s g), the smaller one
 * on a tie, with the sign bit set when x < 0 ([MXFP4] §三 chooses elements the
 * same way); a block whose scale is 0 is all code 0.  Every step is one
 * float32 operation rounded to nearest, so the bytes are exact.
 *
 *   rows, cols    source size; cols must be a multiple of 16.
 *   src           fp32 [rows, cols], row stride ld_src (elements).
 *   data          uint8 [rows, cols/2] output (element 2t in the low nibble
 *                 of byte t), row stride ld_data (bytes).
 *   scales        uint8 [rows, cols/16] output E4M3 bytes, row stride ld_scales.
 *   tensor_scale  device pointer to one float that receives g (it also holds
 *                 the running amax while the call runs).
 * Alignment: src 16-byte aligned, ld_src a multiple of 4; data 8-byte aligned,
 * ld_data a multiple of 8; tensor_scale 4-byte aligned.
 * The source is read twice (amax, then the codes).
 */
int nv_quantize_fp4(int rows, int cols, const float* src, int64_t ld_src,
                    uint8_t* data, int64_t ld_data, uint8_t* scales,
                    int64_t ld_scales, float* tensor_scale, wq_stream_t stream);

/*
 * nv_gemm_fp4 — C = A * W^T for NVFP4 operands, FP32 output.
 *
 * [W4A16] §三 (NVFP4 on the 5th-generation tensor cores; reading as for
 * nv_quantize_fp4) and [MXFP4] §二.1 (the block dot product): for every output
 * (m, n) and 16-element K block b,
 *   dC = sA[m, b] * sW[n, b] * sum_{i<16} a[m, b, i] * w[n, b, i],
 * C = gA * gW * sum_b dC, accumulated in FP32 by the block-scaled tensor
 * cores (kind::mxf4nvf4, E4M3 scales).
 *
 *   M, N, K   problem size; K must be a multiple of 16.
 *   A, SA     A's data uint8 [M, K/2] (row stride lda) and E4M3 scales uint8
 *             [M, K/16] (row stride ldsa), as nv_quantize_fp4 writes them.
 *   scale_a   device pointer to A's tensor scale gA (from nv_quantize_fp4).
 *   W, SW, scale_w  the same for W [N, K].
 *   C         fp32 [M, N] output, row stride ldc (elements).
 *   workspace, ws_bytes  at least wq_workspace_size(WQ_OP_NV_GEMM, M, N, K)
 *             bytes, 256-byte aligned, used as in mx_gemm_fp4 (the scales
 *             are rewritten there, then nv_gemm_fp4_tc runs).
 * Alignment: as for mx_gemm_fp4, plus scale_a and scale_w 4-byte aligned.
 * Small M splits K across a cluster of CTAs as mx_gemm_fp4 does; the result
 * is deterministic.
 */
int nv_gemm_fp4(int M, int N, int K, const uint8_t* A, int64_t lda,
                const uint8_t* SA, int64_t ldsa, const float* scale_a,
                const uint8_t* W, int64_t ldw, const uint8_t* SW,
                int64_t ldsw, const float* scale_w, float* C, int64_t ldc,
                void* workspace, size_t ws_bytes, wq_stream_t stream);

/*
 * nv_gemm_fp4_tc — nv_gemm_fp4 with both E4M3 scale arrays already in the
 * tensor-core layout (fp4_scales_tc with WQ_FP4_NV): no workspace.
 * SA/sa_bytes and SW/sw_bytes as for mx_gemm_fp4_tc; everything else as for
 * nv_gemm_fp4.
 */
int nv_gemm_fp4_tc(int M, int N, int K, const uint8_t* A, int64_t lda,
                   const uint8_t* SA, size_t sa_bytes, const float* scale_a,
                   const uint8_t* W, int64_t ldw, const uint8_t* SW,
                   size_t sw_bytes, const float* scale_w, float* C,
                   int64_t ldc, wq_stream_t stream);

/*
 * fp8_gemm — C = bf16((A * B) * scale_a * scale_b) for e4m3 operands.
 *
 * [FP8] kernel listing and 精度管理 bullet: e4m3fn inputs, FP32 accumulation,
 * the per-tensor scales applied once to the accumulator, BF16 output
 * (round to nearest even).
 *
 *   M, N, K  problem size (any K).
 *   A        e4m3fn bytes [M, K], row stride lda (bytes).
 *   B        e4m3fn bytes [K, N], row stride ldb (bytes).
 *   scale_a, scale_b  per-tensor FP32 scales, passed by value.
 *   C        bf16 [M, N] output, row stride ldc (elements).
 *   workspace, ws_bytes  at least wq_workspace_size(WQ_OP_FP8_GEMM, M, N, K)
 *            bytes: for M <= 16 the K dimension is split across CTAs and the
 *            contract of wq_gemm_w4a16's workspace applies (zero-fill once;
 *            calls leave the counter area zero); 0 bytes otherwise.
 * Alignment: A, B, C 16-byte aligned; lda, ldb multiples of 16; ldc a
 * multiple of 8.
 */
int fp8_gemm(int M, int N, int K, const uint8_t* A, int64_t lda,
             const uint8_t* B, int64_t ldb, float scale_a, float scale_b,
             void* C, int64_t ldc, void* workspace, size_t ws_bytes,
             wq_stream_t stream);

/* Scratch bytes an operation needs for this shape on the current device (0
 * when none).  The size depends on the device's SM count. */
size_t wq_workspace_size(int op, int M, int N, int K);

/* Static, human-readable name of a status code (never NULL). */
const char* wq_status_string(int status);

/*
 * Read and clear the device error word that kernels set when a bounded
 * wait (an mbarrier or cluster handshake) gives up instead of hanging.
 * Synchronizes `stream`.  Returns WQ_OK when no kernel gave up, otherwise
 * WQ_ERR_DEVICE and stores the recorded site code in *site (if non-NULL).
 */
int wq_get_device_error(wq_stream_t stream, int* site);

/*
 * wq_set_static_weights — the caller's promise that weights are static.
 *
 * Off by default.  With enable != 0 the caller promises that, for every
 * later call of wq_gemm_w4a16, wq_gemm_w8a16 and their _grouped and
 * _noalloc forms, no kernel that may still be running when the call is
 * launched writes its weight array (Wq / W) or its scales and zero points:
 * the weights are loaded once and only read afterwards, as in inference.
 * The decode (M <= 16) kernels then start loading their first weight boxes
 * into shared memory while the kernel before them on the stream is still
 * finishing (they are launched as programmatic dependents), instead of only
 * prefetching them into L2; activations are still read, and outputs
 * written, only after that kernel has completed.  Results are identical
 * either way.  Breaking the promise (writing a weight array in a kernel
 * that overlaps a later call) can make that call compute with stale
 * weights.  Process-wide; applies to calls launched afterwards, from any
 * host thread.  Returns the previous setting (0 or 1).  The pages have no
 * counterpart: it is a launch-overlap switch, not a new operation.
 */
int wq_set_static_weights(int enable);

/*
 * wq_debug_set_wait_limit — testing hook: the limit (in nanoseconds) after
 * which the skinny weight-stream kernels (wq_gemm_w4a16, wq_gemm_w8a16, their
 * _grouped, _noalloc and _batched forms, and fp8_gemm at M <= 16) give up a
 * bounded wait, record the site in the device error word (see
 * wq_get_device_error) and return, instead of waiting on.  ns <= 0 restores
 * the default of 2 s.  Applies to calls launched afterwards, from any host
 * thread.  With a very short limit a call gives up almost at once and its
 * output is not computed; nothing is left in flight when it returns, and the
 * next call with the default limit computes normally.  The pages have no
 * counterpart: it exists so that tests can exercise the give-up path without
 * faulting or hanging a GPU.  Always returns WQ_OK.
 */
int wq_debug_set_wait_limit(int64_t ns);

/* Library version, as major * 10000 + minor * 100 + patch. */
int wq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WQ_H_ */
