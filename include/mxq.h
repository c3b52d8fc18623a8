/*
 * mxq.h -- C ABI of the GB300 (sm_103a) MX quantized-training library.
 *
 * The library implements the hot path of microscaling (MX) quantized
 * training: block-of-32 quantization of bf16 tensors to E4M3 (MXFP8) or
 * E2M1 (MXFP4) element codes with one E8M0 shared exponent per block, a
 * fixed 32-point Hadamard rotation fused into the quantizer, and the
 * block-scaled GEMM that consumes the codes for the forward, dgrad and Wgrad
 * products.
 *
 * Sources of the operations (cited per entry point below):
 *  [AMD-FP4]  "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題" (hzrcw.cc):
 *             §02 microscaling (each small block has its own dynamic
 *             exponent), the deterministic Hadamard rotation on the Wgrad
 *             path, the per-path FP4 study (forward, activation gradient,
 *             weight gradient); §03 native FP4 GEMMs on the GPU.
 *  [MINDSPEED] "MindSpeed LLM FSDP2量化特性：低比特大模型训练完全指南",
 *             第 1 步 (recipe dynamic_MX-1-1-32_E4M3_E4M3_E4M3): MX
 *             granularity, block size 32, E4M3 for inputs, weights and
 *             gradients.
 *  [LUMEN]    "Lumen：AMD原生大模型量化训练框架的技术突破与实践", §1: FP8
 *             E4M3 / MXFP8 / FP4 formats.
 *  Bit layouts and rounding (none are printed on those pages) follow the
 *  OCP Microscaling Formats (MX) v1.0 and OCP FP8 specifications.
 *
 * Conventions shared by every call
 *  - All pointers named x, codes, scales, A, B, C, out, workspace are DEVICE
 *    pointers owned by the caller; the library never frees or keeps them.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work on that stream and returns;
 *    argument errors are reported synchronously, device-side errors (a wait
 *    that timed out) by mxq_check().
 *  - Tensors are row-major.  A [rows, cols] bf16 tensor has row stride cols.
 *  - E4M3 and E5M2 codes take one byte per element.  E2M1 codes take half a
 *    byte: two per byte along the blocked axis, the even element in the low
 *    nibble.
 *  - E8M0 scale bytes: value 2^(s-127); 0xFF marks a block that held a NaN
 *    or an infinity (its codes are then all zero).  An all-zero block has
 *    scale 0x00.
 *  - Shared exponent e = floor(log2(amax)) - emax_elem (emax_elem = 8 for
 *    E4M3, 15 for E5M2, 2 for E2M1), clamped to [-127, 127]; elements
 *    x * 2^-e are rounded to nearest, ties to even, saturating at 448
 *    (E4M3), 57344 (E5M2) or 6 (E2M1); a negative value that rounds to zero
 *    keeps its sign.
 *  - Pointers to bf16 data and to codes must be 16-byte aligned; scales may
 *    have any alignment.
 *  - No call allocates device memory.
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXQ_OK = 0,
  MXQ_ERR_ARG = 1,          /* a size, enum or pointer argument is invalid   */
  MXQ_ERR_ALIGN = 2,        /* a pointer or a dimension breaks an alignment rule */
  MXQ_ERR_UNSUPPORTED = 3,  /* valid request the library does not implement   */
  MXQ_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed               */
  MXQ_ERR_TIMEOUT = 5,      /* a device-side wait gave up (see mxq_check)      */
  MXQ_ERR_WORKSPACE = 6,    /* workspace too small                             */
  MXQ_ERR_BOUNDS = 7        /* bounds-checked build only: a kernel computed an
                               index outside the extent its arguments imply
                               (the access was skipped; see mxq_check)       */
} mxq_status;

/* Element formats: E4M3 and E5M2 (MXFP8, one byte per element) and E2M1
   (MXFP4, packed two per byte).  E5M2: [LUMEN] §1 names FP8 E5M2 beside
   E4M3; OCP MX v1.0 lists it as the second MXFP8 element type. */
typedef enum { MXQ_E4M3 = 0, MXQ_E2M1 = 1, MXQ_E5M2 = 2 } mxq_fmt;

typedef enum {
  /* blocks of 32 run along cols; codes [rows][cols] (E2M1: [rows][cols/2]),
     scales [rows][cols/32] */
  MXQ_ROWWISE = 0,
  /* blocks of 32 run along rows; output stored transposed: codes
     [cols][rows] (E2M1: [cols][rows/2]), scales [cols][rows/32].  Row c of
     the output holds input column c in row order (the Wgrad operand). */
  MXQ_COLWISE_T = 1
} mxq_layout;

typedef enum { MXQ_OUT_F32 = 0, MXQ_OUT_BF16 = 1 } mxq_out;

/*
 * Layout of the E8M0 scale bytes of a quantized operand with `lines` rows
 * (output rows: rows for MXQ_ROWWISE, cols for MXQ_COLWISE_T) and a blocked
 * dimension of `blocked` elements (32 per block):
 *  MXQ_SCALES_ROWMAJOR: [lines][blocked / 32] bytes.
 *  MXQ_SCALES_TC: the layout the tensor cores read the block scales in
 *    (tcgen05.cp 32x128b.warpx4): 512-byte chunks, one per 128 lines x 4
 *    blocks; chunk (line / 128) * (blocked / 128) + block / 4 holds the
 *    byte of (line, block) at (line % 32) * 16 + ((line % 128) / 32) * 4 +
 *    block % 4.  Lines past the end of the last 128-line tile hold zeros.
 *    Size: mxq_scales_tc_bytes().  Needs blocked % 128 == 0 (E4M3, E5M2)
 *    or % 256 == 0 (E2M1, whole GEMM stages) and a 16-byte aligned buffer.
 *    A GEMM given scales in this layout (mxq_gemm_ex) skips its scale
 *    re-layout pass and needs no workspace.
 */
typedef enum { MXQ_SCALES_ROWMAJOR = 0, MXQ_SCALES_TC = 1 } mxq_scale_layout;

/* Library version, (major << 16) | minor. */
int mxq_version(void);

/* Human-readable name of a status code (static string). */
const char* mxq_status_str(int status);

/*
 * MX quantization of a bf16 tensor x [rows][cols].
 *   [AMD-FP4] §02 (per-block dynamic exponent), [MINDSPEED] 第 1 步
 *   (block 32, E4M3).
 * layout: MXQ_ROWWISE needs cols % 32 == 0; MXQ_COLWISE_T needs
 *   rows % 32 == 0 and cols % 8 == 0.
 * fmt: MXQ_E4M3, MXQ_E5M2 or MXQ_E2M1.  codes / scales: outputs in the
 * layout above.
 * rows == 0 or cols == 0 is a no-op.  Dimensions must be < 2^31.
 */
mxq_status mxq_quantize(const void* x, int64_t rows, int64_t cols, int layout, int fmt,
                        void* codes, uint8_t* scales, void* stream);

/*
 * Fixed 32-point Hadamard rotation of every block along the quantization
 * axis, then MX quantization of the rotated values.
 *   [AMD-FP4] §02: a deterministic (fixed, not random) orthogonal rotation
 *   applied before the MXFP4 quantization of the weight-gradient operands.
 * The rotation is the natural-order Sylvester transform H_32/sqrt(32):
 * radix-2 stages with half-width 1, 2, 4, 8, 16 in fp32, each add and
 * subtract rounded to nearest (no fused operations), then one multiply by
 * RN_fp32(2^-2.5).  The fp32 result is quantized without a bf16 rounding.
 * Arguments and preconditions as mxq_quantize.
 */
mxq_status mxq_hadamard_quantize(const void* x, int64_t rows, int64_t cols, int layout, int fmt,
                                 void* codes, uint8_t* scales, void* stream);

/*
 * One read of x [rows][cols] produces both the row-wise output (fmt_r,
 * Hadamard if had_r != 0) and the column-wise transposed output (fmt_c,
 * Hadamard if had_c != 0).  The forward/dgrad operand and the Wgrad operand
 * of the same tensor ([AMD-FP4] §02) come from a single pass.
 * Needs rows % 32 == 0, cols % 32 == 0; fmt_r and fmt_c are each MXQ_E4M3,
 * MXQ_E5M2 or MXQ_E2M1 ([LUMEN] §1 names FP8 E5M2 beside E4M3), in any
 * pairing.  Outputs as in mxq_quantize.
 */
mxq_status mxq_quantize_dual(const void* x, int64_t rows, int64_t cols,
                             int fmt_r, int had_r, void* codes_r, uint8_t* scales_r,
                             int fmt_c, int had_c, void* codes_c, uint8_t* scales_c,
                             void* stream);

/*
 * mxq_quantize / mxq_hadamard_quantize (hadamard != 0) with the scales in
 * the given mxq_scale_layout.  MXQ_SCALES_ROWMAJOR is exactly mxq_quantize.
 */
mxq_status mxq_quantize_ex(const void* x, int64_t rows, int64_t cols, int layout, int fmt,
                           int hadamard, void* codes, uint8_t* scales, int scale_layout,
                           void* stream);

/* mxq_quantize_dual with both outputs' scales in the given mxq_scale_layout. */
mxq_status mxq_quantize_dual_ex(const void* x, int64_t rows, int64_t cols,
                                int fmt_r, int had_r, void* codes_r, uint8_t* scales_r,
                                int fmt_c, int had_c, void* codes_c, uint8_t* scales_c,
                                int scale_layout, void* stream);

/* Bytes of an MXQ_SCALES_TC scale buffer (0 on bad arguments). */
size_t mxq_scales_tc_bytes(int64_t lines, int64_t blocked);

/*
 * Ablation quantizer: MX quantization with the randomness that [AMD-FP4] §01
 * sets against its deterministic rotation -- a random Hadamard rotation and
 * stochastic rounding.  Single layout, arguments and preconditions as
 * mxq_quantize, plus:
 *   hadamard   != 0: rotate every block by H_32 * diag(d) before quantizing,
 *              d_i = -1 where bit i of sign_mask is set, else +1 (one random
 *              sign vector drawn by the caller, shared by all blocks; the
 *              butterflies and the normalization are those of
 *              mxq_hadamard_quantize).  sign_mask must be 0 when hadamard
 *              is 0 (MXQ_ERR_ARG otherwise).
 *   stochastic != 0: element codes by stochastic rounding instead of round
 *              to nearest even.  With q the element grid step at |v| (v the
 *              element divided by the block scale), |v| rounds up to the next
 *              grid point iff bits < floor(frac(|v| / q) * 2^32), where bits
 *              is word (i % 4) of Philox4x32-10(counter = (i / 4 low 32 bits,
 *              i / 4 high 32 bits, 0, 0), key = (seed low 32, seed high 32))
 *              and i = input row * cols + input column (the same bits for
 *              either layout).  Saturates at the largest finite element; the
 *              sign is kept.  The block exponent is the deterministic one.
 * hadamard == 0 and stochastic == 0 is mxq_quantize; sign_mask == 0 without
 * stochastic rounding is mxq_hadamard_quantize.  The output depends only on
 * x, sign_mask and seed.
 */
mxq_status mxq_quantize_ablation(const void* x, int64_t rows, int64_t cols, int layout, int fmt,
                                 int hadamard, uint32_t sign_mask, int stochastic, uint64_t seed,
                                 void* codes, uint8_t* scales, void* stream);

/*
 * Dequantization: out[r][c] = dec(code) * 2^(s-127), exact in fp32 (an
 * overflow gives inf; scale 0xFF gives NaN); bf16 output is that fp32 value
 * rounded to nearest even.  OCP MX v1.0 (value of an MX element).
 * rows, cols, layout and fmt describe the tensor as it was quantized
 * (codes laid out as mxq_quantize wrote them); out is always [rows][cols].
 * out_dtype: MXQ_OUT_F32 or MXQ_OUT_BF16.
 */
mxq_status mxq_dequantize(const void* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                          int layout, int fmt, void* out, int out_dtype, void* stream);

/*
 * Block-scaled GEMM C[m][n] = sum_k dec(A[m][k]) * dec(B[n][k]) with fp32
 * accumulation on the tensor cores.
 *   [AMD-FP4] §02-§03: the forward (Y = X W^T), dgrad (dX = dY W) and Wgrad
 *   (dW = dY^T X) products run on MX codes.
 * A: codes [M][K] (E2M1: [M][K/2]), sA [M][K/32]; B: codes [N][K]
 * (E2M1: [N][K/2]), sB [N][K/32] -- both "K-major", as MXQ_ROWWISE (or
 * MXQ_COLWISE_T for the transposed operand) writes them.  Both operands use
 * the same fmt (MXQ_E4M3, MXQ_E5M2 or MXQ_E2M1).  C: [M][N] row-major, fp32 or bf16 (out_dtype).
 * K % 32 == 0, M >= 1, N >= 1; N % 4 == 0 (fp32) / N % 8 == 0 (bf16).
 * workspace: device scratch of at least mxq_gemm_workspace_size() bytes,
 * 256-byte aligned; it receives the scales in the tensor-core layout.
 */
mxq_status mxq_gemm(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB, int fmt,
                    int64_t M, int64_t N, int64_t K, void* C, int out_dtype,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * mxq_gemm whose epilogue writes the product as row-wise MX codes instead of
 * fp32/bf16: the next layer's operand straight from the accumulators, with
 * no bf16 round trip through memory (a GEMM fused with its consumer's
 * quantization, in the spirit of the fused kernels -- fused MLP among them --
 * that [LUMEN] §2 "AITER高性能内核集成" lists).
 * The fp32 accumulators of each output row are split into 32-column blocks;
 * each block gets the shared exponent of its fp32 amax and its elements are
 * rounded to out_fmt by the rules of mxq_quantize (the conventions at the
 * top of this file), without rounding the fp32 values to bf16 first.
 * A, sA, B, sB, fmt, M, N, K, workspace: as mxq_gemm.
 * out_fmt: MXQ_E4M3, MXQ_E5M2 or MXQ_E2M1.  N % 32 == 0 (MXQ_ERR_ARG).
 * out_codes: [M][N] bytes (E2M1: [M][N/2]), 16-byte aligned (MXQ_ERR_ALIGN);
 * out_scales: [M][N/32], any alignment.  The layout is MXQ_ROWWISE's.
 */
mxq_status mxq_gemm_quantize(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                             int fmt, int64_t M, int64_t N, int64_t K, int out_fmt,
                             void* out_codes, uint8_t* out_scales, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * mxq_gemm with sA and sB in the given mxq_scale_layout.  With
 * MXQ_SCALES_TC (sA from an M-line, sB from an N-line quantization with
 * blocked dimension K) the scale re-layout pass is skipped, workspace may be
 * NULL and workspace_bytes 0, and K % 128 == 0 (E4M3, E5M2) or K % 256 == 0
 * (E2M1) is required; sA and sB must be 16-byte aligned.
 * MXQ_SCALES_ROWMAJOR is exactly mxq_gemm.
 */
mxq_status mxq_gemm_ex(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB, int fmt,
                       int64_t M, int64_t N, int64_t K, void* C, int out_dtype, int scale_layout,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * mxq_gemm_quantize with the input scales sA, sB in scale_layout and the
 * output scales in out_scale_layout (mxq_scale_layout).  With
 * out_scale_layout MXQ_SCALES_TC the output (M lines, blocked dimension N)
 * can feed mxq_gemm_ex directly; it needs N % 128 == 0 (E4M3, E5M2) or
 * N % 256 == 0 (E2M1) and a 16-byte aligned out_scales of
 * mxq_scales_tc_bytes(M, N) bytes.  Input-side rules as mxq_gemm_ex.
 */
mxq_status mxq_gemm_quantize_ex(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                                int fmt, int64_t M, int64_t N, int64_t K, int scale_layout,
                                int out_fmt, void* out_codes, uint8_t* out_scales,
                                int out_scale_layout, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * One problem of mxq_gemm_grouped: C[M][N] = dec(A) dec(B)^T as in mxq_gemm,
 * with sA, sB in the tensor cores' chunk layout (MXQ_SCALES_TC), as for
 * mxq_gemm_ex with that layout.  out_dtype: MXQ_OUT_F32 or MXQ_OUT_BF16.
 */
typedef struct {
  const void* A;
  const uint8_t* sA;
  const void* B;
  const uint8_t* sB;
  void* C;
  int64_t M, N, K;
  int out_dtype;
} mxq_gemm_problem;

/*
 * Several independent GEMMs of one element format in one launch: their
 * 256x256 tiles are numbered problem after problem and run by one persistent
 * grid, so a problem with few tiles does not leave most clusters idle in its
 * last wave.  [AMD-FP4] §02 runs a weight-gradient (Wgrad) GEMM per linear
 * layer; the layers' Wgrad GEMMs depend on nothing the others compute, so a
 * backward pass can issue them together.
 *
 * problems: count (1..8) problems in host memory (read during the call), each
 * with the preconditions of mxq_gemm_ex for MXQ_SCALES_TC (K % 128 == 0 for
 * E4M3/E5M2, % 256 for E2M1; 16-byte aligned pointers; chunk-layout scales of
 * mxq_scales_tc_bytes(M, K) and (N, K) bytes).  Each C gets exactly what
 * mxq_gemm_ex would write for its problem, bit for bit.  The caller owns
 * every buffer; no workspace.  Argument errors return before any launch.
 */
mxq_status mxq_gemm_grouped(const mxq_gemm_problem* problems, int count, int fmt, void* stream);

/* Bytes of workspace mxq_gemm needs for this problem (0 on bad arguments). */
size_t mxq_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int fmt);

/*
 * mxq_gemm for callers that cannot allocate device memory when they call:
 * code embedded in a host application that owns the device memory pool and
 * passes a plug-in only its input and output buffers, or code running under a
 * fixed memory budget that forbids per-call allocation.  The pages describe
 * no such entry point; it exists only for these callers.
 *
 * Arguments and results are those of mxq_gemm, without the workspace: the
 * scale scratch is a fixed 16 MiB device buffer inside the library, which
 * every GPU that loads the library keeps until the process exits.  Problems
 * whose mxq_gemm_workspace_size() exceeds 16 MiB are rejected with
 * MXQ_ERR_WORKSPACE before any work is queued.  The call allocates nothing.
 * The first call on each device looks up that device's address of the buffer
 * (with the device current); make that first call before any stream capture.
 * All calls share the buffer: calls that overlap on the GPU (other streams,
 * other host threads) race on it and must be serialized by the caller.
 * The looked-up address is kept for the life of the process: after
 * cudaDeviceReset() (or any teardown of the device's primary context) the
 * entry point must not be called again in that process.
 */
mxq_status mxq_gemm_noalloc(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                            int fmt, int64_t M, int64_t N, int64_t K, void* C, int out_dtype,
                            void* stream);

/*
 * Synchronizes `stream`, then reports and clears device-side errors recorded
 * by earlier calls on any stream (MXQ_ERR_TIMEOUT when a bounded wait inside
 * a kernel gave up), or MXQ_ERR_CUDA when the stream reports a CUDA error.
 */
mxq_status mxq_check(void* stream);

/*
 * Upper bound, in nanoseconds, of every device-side wait (default 2e9).
 * A kernel whose wait runs out records MXQ_ERR_TIMEOUT and returns early.
 */
void mxq_set_wait_timeout_ns(uint64_t ns);

/*
 * Test hook for the failure path: launches one CTA that waits on a barrier
 * no one completes, with the given limit, so that the bounded wait expires
 * and records MXQ_ERR_TIMEOUT for mxq_check() to report.
 */
mxq_status mxq_debug_expire_wait(uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H */
