/*
 * hlq.h -- C ABI of libhlq, the GB300 (sm_103a) kernels of the HLQ/HOT
 * backward pass of one linear layer y = x . w^T (or an im2col'd conv).
 *
 * Method: "HLQ: Fast and Efficient Backpropagation via Hadamard Low-rank
 * Quantization" (Kim & Park), TL;DR: g_x = g_y . w through 4-bit Hadamard
 * quantization (HQ) and g_w = (1/B) gbar_y^T . xbar through the Hadamard
 * low-rank approximation (HLA) with int8 arithmetic, the stored activation
 * compressed at forward time (ACBP); "HOT: Hadamard-based Optimized
 * Training", Approach: the same assignment of HQ / HLA+int8 to the two
 * gradient paths, activation buffer compression, and per-token vs
 * per-tensor quantizer chosen per layer.
 *
 * Shapes: x [T, Cin], w [Cout, Cin], g_y [T, Cout], g_x [T, Cin],
 * g_w [Cout, Cin]; every matrix row-major (last index contiguous).
 * Block B = 16 (Hadamard block, also the 1/B of the g_w formula).
 * T' = T * rank / 16 is the reduced token count of the HLA.
 *
 * Conventions for every entry point:
 *  - Pointers named d_* are device pointers owned by the caller; the library
 *    never allocates or frees device memory.  Scratch goes in a caller
 *    workspace `ws` of at least hlq_workspace_bytes(...) bytes (256-byte
 *    aligned).  Device pointers must be 16-byte aligned.
 *  - All work is enqueued on `stream` (a cudaStream_t passed as void*;
 *    NULL = legacy default stream) and is asynchronous.  The only call that
 *    waits is hlq_read_device_status.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    non-OK status means nothing was launched and no memory was written.
 *    Launch errors return HLQ_ERR_CUDA.  Nothing aborts, throws or traps:
 *    device-side conditions (non-finite input) set a flag that
 *    hlq_read_device_status returns.
 *  - Preconditions: block == 16; rank in {1, 2, 4, 8, 16}; T, Cin, Cout
 *    multiples of 16 (zero allowed: the outputs are then zero-filled);
 *    finite inputs with |v| <= FLT_MAX/16.
 */
#ifndef HLQ_H
#define HLQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HLQ_OK = 0,
    HLQ_ERR_INVALID_ARG = 1, /* null pointer, bad enum, bad block/rank */
    HLQ_ERR_SHAPE = 2,       /* size not a multiple of 16, negative */
    HLQ_ERR_ALIGN = 3,       /* pointer not 16-byte (ws: 256-byte) aligned */
    HLQ_ERR_UNSUPPORTED = 4, /* valid but not implemented (e.g. per-token w) */
    HLQ_ERR_WORKSPACE = 5,   /* ws_bytes below hlq_workspace_bytes() */
    HLQ_ERR_OVERFLOW = 6,    /* an integer accumulator could overflow */
    HLQ_ERR_CUDA = 7         /* a CUDA launch or copy failed */
} hlq_status;

typedef enum { HLQ_F32 = 0, HLQ_BF16 = 1 } hlq_dtype;

/* Layer-wise quantizer selection (HOT, Approach): one scale per tensor, or
 * one scale per token (row of g_y). */
typedef enum { HLQ_PER_TENSOR = 0, HLQ_PER_TOKEN = 1 } hlq_gran;

/* Rounding of the int4 HQ codes: stochastic (Philox4x32-10 keyed on seed and
 * element index) or round-to-nearest-even (for tests). */
typedef enum { HLQ_RNE = 0, HLQ_SR = 1 } hlq_round;

typedef enum {
    HLQ_OP_COMPRESS_ACTIVATION = 0,
    HLQ_OP_BACKWARD_GX = 1,
    HLQ_OP_BACKWARD_GW = 2,
    HLQ_OP_BACKWARD = 3, /* hlq_linear_backward: both gradients */
    HLQ_OP_SELECT_GRANULARITY = 4, /* hlq_select_gy_granularity */
    HLQ_OP_ABLATION_GW_HQ = 5,     /* hlq_ablation_gw_hq */
    HLQ_OP_ABLATION_GX_HLA = 6,    /* hlq_ablation_gx_hla */
    HLQ_OP_BACKWARD_FUSED = 7,     /* hlq_linear_backward_fused */
    HLQ_OP_LAYER_STEP = 8          /* hlq_layer_step */
} hlq_op;

/* Device status flags (hlq_read_device_status). */
#define HLQ_DEV_NONFINITE 0x1u /* a transform input was inf or NaN */
#define HLQ_DEV_TIMEOUT 0x2u   /* a bounded device wait gave up */
#define HLQ_DEV_BADCODE 0x4u   /* an operand code was outside its range */

/*
 * Workspace bytes needed by one call of `op` with these sizes (rank is used
 * by the g_w op only).  The result is a multiple of 256.
 */
size_t hlq_workspace_bytes(int op, int64_t T, int64_t Cin, int64_t Cout,
                           int block, int rank);

/*
 * Format word of the stored activation (xbar_fmt): the code width, 8 or 4,
 * optionally OR'ed with HLQ_XBAR_PER_CHANNEL for one scale per input
 * channel (d_xbar_scale [Cin]) instead of one per tensor (d_xbar_scale [1]).
 * The per-channel scale is the per-layer granularity choice of HOT
 * (Approach) carried to the stored activation: its token dim is the g_w
 * contraction dim, so the scale that still factors out of the integer GEMM
 * is one per channel, i.e. per column of g_w.
 */
#define HLQ_XBAR_INT8 8
#define HLQ_XBAR_INT4 4
#define HLQ_XBAR_PER_CHANNEL 0x100

/*
 * ACBP at forward time (HOT, Approach: stored activations compressed when
 * the forward pass runs; HLQ TL;DR: int4 activation compression, ACBP).
 * x [T, Cin] (dtype dt) -> d_xbar codes (token dim contiguous) and
 * d_xbar_scale fp32 ([1], or [Cin] with HLQ_XBAR_PER_CHANNEL):
 *   Xbar[c, rank*b + k] = RN_f32( sum_j H16[sigma(k)][j] x[16b + j, c] )
 *   s = RN_f32(max|Xbar| / qmax),  code = clamp(rne(RN_f32(Xbar / s)), +-qmax)
 * where sigma(k) is the Sylvester row of sequency k (the rank lowest-
 * sequency Walsh rows are kept) and the max runs over the tensor, or over
 * row c of Xbar for the scale s_c of channel c.  s == 0 gives all-zero codes.
 * Code width 8: qmax 127, d_xbar [Cin, T'] int8 codes.
 * Code width 4: qmax 7, d_xbar [Cin, T'/2] bytes, two's-complement int4 codes
 *   packed two per byte (code 2k in the low nibble, 2k+1 in the high one);
 *   even ranks only (HLQ_ERR_UNSUPPORTED for rank 1).
 * Another width or unknown flag bits: HLQ_ERR_INVALID_ARG.
 * Workspace: hlq_workspace_bytes(HLQ_OP_COMPRESS_ACTIVATION, ...), which
 * grows with Cin (one amax slot per channel).
 */
hlq_status hlq_compress_activation(const void *d_x, int dt, int64_t T,
                                   int64_t Cin, int block, int rank, int xbar_fmt,
                                   int8_t *d_xbar, float *d_xbar_scale,
                                   void *d_ws, size_t ws_bytes, void *stream);

/*
 * Activation gradient g_x = g_y . w with int4 HQ (HLQ TL;DR; HLQ sections
 * "Alternative Optimization Technique: Hadamard Quantization" and "HLQ:
 * Hadamard Low-rank Quantization"):
 *   Y  = g_y transformed by H16 along Cout in blocks of 16 (Sylvester order),
 *   Wt = w   transformed by H16 along Cout,
 *   each rounded once to fp32 from the exact sum;
 *   s_gy = RN(amax/7) per token (gran_gy) or per tensor; s_w per tensor;
 *   codes: x = RN(Y/s), stochastic rounding q = floor(x) + [u < x-floor(x)],
 *   u = (word >> 8) * 2^-24 of Philox4x32-10 with key (seed lo, seed hi) and
 *   counter (e/4 lo, e/4 hi, stream, 0), word e%4, e = row*cols + col of the
 *   transformed tensor, stream 0 for g_y and 1 for w; clamp to [-7, 7];
 *   acc[t, i] = sum_c qY[t, c] qW[i, c]  (exact integer);
 *   g_x[t, i] = acc * s_gy[t] * s_w / 16   (fp32).
 * gran_w must be HLQ_PER_TENSOR.
 */
hlq_status hlq_linear_backward_gx(const void *d_gy, const void *d_w, int dt,
                                  int64_t T, int64_t Cin, int64_t Cout,
                                  int block, int gran_gy, int gran_w, int rnd,
                                  uint64_t seed, float *d_gx, void *d_ws,
                                  size_t ws_bytes, void *stream);

/*
 * Weight gradient g_w = (1/16) gbar_y^T . xbar with HLA + int8 (HLQ TL;DR,
 * with B read as the Hadamard block size; HOT, Approach):
 *   gbar_y = HLA of g_y along tokens as in hlq_compress_activation,
 *   s_g = RN(amax/127) per tensor, int8 codes by round-to-nearest-even,
 *   acc[o, i] = sum_t' qG[o, t'] qX[i, t']  (exact integer),
 *   g_w[o, i] = acc * s_g * s_x / 16   (fp32),
 * s_x the tensor scale, or s_x[i] with HLQ_XBAR_PER_CHANNEL in xbar_fmt.
 * d_xbar / d_xbar_scale come from hlq_compress_activation with the same T,
 * Cin, rank and xbar_fmt (the qX codes are then in [-127, 127] or [-7, 7]).
 * Needs T' * 127 * qmax_x < 2^31.
 */
hlq_status hlq_linear_backward_gw(const void *d_gy, int dt, const int8_t *d_xbar,
                                  const float *d_xbar_scale, int64_t T,
                                  int64_t Cin, int64_t Cout, int block,
                                  int rank, int xbar_fmt, float *d_gw, void *d_ws,
                                  size_t ws_bytes, void *stream);

/*
 * How every g_w GEMM of the library takes its int8 operands (HLQ TL;DR:
 * int8 on the g_w path).  One setting for the process, read by each call
 * when it enqueues its work; results are bit-identical in every mode, only
 * the HBM layout and the kernels differ:
 *   HLQ_GW_WIDEN      the int8 x-bar is widened to fp16 in the workspace by
 *                     a kernel of its own; the HLA codes of g_y are written
 *                     as fp16;
 *   HLQ_GW_INT8_X     the GEMM loads the int8 x-bar itself and widens each
 *                     tile to fp16 in shared memory; g_y codes as fp16;
 *   HLQ_GW_INT8_BOTH  both operands int8 in HBM (the HLA codes of g_y too),
 *                     both widened in shared memory (the fused reader of
 *                     hlq_linear_backward_fused writes fp16 codes and takes
 *                     HLQ_GW_INT8_X there);
 *   HLQ_GW_AUTO       the library's default (the fastest measured).
 * The in-GEMM widening needs int8 x-bar whose rows T' bytes are a multiple
 * of 16 and a 16-byte aligned d_xbar; other calls use HLQ_GW_WIDEN.  The
 * workspace sizes do not depend on the mode.  hlq_set_gw_operands returns
 * HLQ_ERR_INVALID_ARG for an unknown mode; hlq_get_gw_operands returns the
 * setting.
 */
#define HLQ_GW_AUTO 0
#define HLQ_GW_WIDEN 1
#define HLQ_GW_INT8_X 2
#define HLQ_GW_INT8_BOTH 3
hlq_status hlq_set_gw_operands(int mode);
int hlq_get_gw_operands(void);

/*
 * For per-kernel timing: with on = 1, hlq_linear_backward (both readers of
 * g_y) and hlq_layer_step run all their branches on the caller's stream,
 * one after the other, instead of forking the g_w branch and the HQ of w to
 * library streams; the kernels and their results are the same.  on = 0
 * restores the default.  A process-wide setting read when a call enqueues
 * its work; on outside {0, 1} is HLQ_ERR_INVALID_ARG.
 */
hlq_status hlq_debug_serialize_branches(int on);

/*
 * The whole backward pass of the layer: g_x exactly as hlq_linear_backward_gx
 * and g_w exactly as hlq_linear_backward_gw, with the independent branches
 * overlapped on the GPU.  The g_w branch and the HQ of w run on auxiliary
 * streams of the library (per device, created on first use) forked from and
 * joined back into `stream` with events, so all work is still ordered after
 * what precedes the call on `stream` and before what follows it.
 * Workspace: hlq_workspace_bytes(HLQ_OP_BACKWARD, ...).  Arguments are the
 * union of the two calls'.
 */
hlq_status hlq_linear_backward(const void *d_gy, const void *d_w, const int8_t *d_xbar,
                               const float *d_xbar_scale, int dt, int64_t T,
                               int64_t Cin, int64_t Cout, int block, int rank,
                               int xbar_fmt, int gran_gy, int gran_w, int rnd, uint64_t seed,
                               float *d_gx, float *d_gw, void *d_ws, size_t ws_bytes,
                               void *stream);

/*
 * One layer step from device buffers: the ACBP compression of x (as
 * hlq_compress_activation, into d_xbar / d_xbar_scale) and both gradients
 * (as hlq_linear_backward), in one call.  The compression is the first step
 * of the g_w branch, the only one that reads the stored activation, so it
 * runs beside the HQ of g_y and the g_x GEMM instead of before them.  With a
 * per-token g_y scale the HLA of g_y runs on a library stream of its own
 * beside the compression; with a per-tensor one a single fused reader of
 * g_y serves both paths (as hlq_linear_backward_fused).  Every output bit
 * equals the separate calls'.  Arguments as for those two calls; workspace
 * hlq_workspace_bytes(HLQ_OP_LAYER_STEP, ...).
 */
hlq_status hlq_layer_step(const void *d_x, const void *d_gy, const void *d_w, int dt,
                          int64_t T, int64_t Cin, int64_t Cout, int block, int rank,
                          int xbar_fmt, int gran_gy, int gran_w, int rnd, uint64_t seed,
                          float *d_gx, float *d_gw, int8_t *d_xbar, float *d_xbar_scale,
                          void *d_ws, size_t ws_bytes, void *stream);

/*
 * hlq_linear_backward with one fused reader of g_y for both paths: a first
 * pass over g_y takes the HQ maxima (per token or per tensor) and the HLA
 * maximum, a second writes the HQ int4 codes and the HLA int8 codes, each
 * from one TMA-staged 16-token x 256-column tile of g_y per CTA (two full
 * reads of g_y instead of three).  The HQ of w and the widening of the
 * stored activation run on library streams meanwhile; the two GEMMs follow
 * on `stream`.  Every output bit equals hlq_linear_backward's.
 * Arguments as for hlq_linear_backward; workspace
 * hlq_workspace_bytes(HLQ_OP_BACKWARD_FUSED, ...) (that of HLQ_OP_BACKWARD
 * plus one amax slot per token).
 */
hlq_status hlq_linear_backward_fused(const void *d_gy, const void *d_w,
                                     const int8_t *d_xbar, const float *d_xbar_scale,
                                     int dt, int64_t T, int64_t Cin, int64_t Cout,
                                     int block, int rank, int xbar_fmt, int gran_gy,
                                     int gran_w, int rnd, uint64_t seed, float *d_gx,
                                     float *d_gw, void *d_ws, size_t ws_bytes,
                                     void *stream);

/*
 * hlq_linear_backward_gx with its intermediates copied out, for bit-exact
 * checks (same formulas):
 *   d_qgy [T, Cout]  int8 codes of Y,   d_sgy [T] or [1] fp32,
 *   d_qw  [Cin, Cout] int8 codes of Wt (transposed: contraction dim
 *   contiguous),  d_sw [1],  d_acc [T, Cin] int32 accumulators,
 *   d_qgy_packed [T, Cout/2], d_qw_packed [Cin, Cout/2] bytes: the same
 *   codes as packed int4 (two's-complement nibbles, code 2k of a row in
 *   the low nibble of byte k), the layout of the method's int4 operands;
 *   the GEMM itself reads one E4M3 byte per code.
 * Any of the seven may be NULL.  Workspace as for HLQ_OP_BACKWARD_GX.
 */
hlq_status hlq_debug_gx_parts(const void *d_gy, const void *d_w, int dt,
                              int64_t T, int64_t Cin, int64_t Cout, int block,
                              int gran_gy, int gran_w, int rnd, uint64_t seed,
                              float *d_gx, void *d_ws, size_t ws_bytes,
                              int8_t *d_qgy, float *d_sgy, int8_t *d_qw,
                              float *d_sw, int32_t *d_acc, uint8_t *d_qgy_packed,
                              uint8_t *d_qw_packed, void *stream);

/*
 * hlq_linear_backward_gw with its intermediates copied out:
 *   d_qg [Cout, T'] int8 codes of gbar_y, d_sg [1], d_acc [Cout, Cin] int32.
 * Any of the three may be NULL.  Workspace as for HLQ_OP_BACKWARD_GW.
 */
hlq_status hlq_debug_gw_parts(const void *d_gy, int dt, const int8_t *d_xbar,
                              const float *d_xbar_scale, int64_t T, int64_t Cin,
                              int64_t Cout, int block, int rank, int xbar_fmt,
                              float *d_gw, void *d_ws, size_t ws_bytes, int8_t *d_qg,
                              float *d_sg, int32_t *d_acc, void *stream);

/*
 * The exactly rounded Hadamard coefficients alone, for bit-exact checks of
 * the transform ("HLQ ...", section "Hadamard Transform"):
 *   axis 0: src [rows, cols], Y[r, 16b+i] = RN_f32(sum_j H16[i][j] src[r, 16b+j])
 *   axis 1: src [rows, cols], Y[16b+i, c] = RN_f32(sum_j H16[i][j] src[16b+j, c])
 * d_y [rows, cols] fp32.  rows, cols multiples of 16; axis 1 needs
 * rows <= 16 * 65535.
 */
hlq_status hlq_debug_hq_transform(const void *d_src, int dt, int64_t rows,
                                  int64_t cols, int axis, float *d_y,
                                  void *stream);

/*
 * The HLA coefficients alone: src [T, C] -> d_out [C, T'] fp32,
 *   out[c, rank*b + k] = RN_f32(sum_j H16[sigma(k)][j] src[16b + j, c]).
 * T <= 16 * 65535.
 */
hlq_status hlq_debug_hla_transform(const void *d_src, int dt, int64_t T,
                                   int64_t C, int rank, float *d_out,
                                   void *stream);

/*
 * Read (and, if `clear` is non-zero, reset) the device status flags of the
 * current device.  Synchronises `stream` first.  *flags is a host pointer.
 */
hlq_status hlq_read_device_status(uint32_t *flags, int clear, void *stream);

/*
 * Second-opinion integer GEMM on the CUDA cores (dp4a), for checking the
 * tensor-core GEMMs at full size: d_acc[m, n] = sum_k A[m, k] * B[n, k] with
 * A [M, K] and B [N, K] int8 (contraction dim contiguous), int32 sums.
 * `kind` is 0 or 1 (kept for symmetry with the two GEMMs; both read int8).
 */
hlq_status hlq_debug_reference_gemm(int kind, const void *d_a, const void *d_b,
                                    int64_t M, int64_t N, int64_t K,
                                    int32_t *d_acc, void *stream);

/*
 * The tensor-core GEMM alone, with an explicit plan, for checks and tuning:
 *   d_acc[m, n] = sum_k A[m, k] * B[n, k]   (int32, exact)
 * kind 0: A, B hold E4M3 bytes of integers in [-7, 7] (the g_x GEMM);
 * kind 1: A, B hold fp16 values of integers in [-127, 127] (the g_w GEMM);
 * kind 2: A as kind 1, B int8 codes in [-127, 127] widened to fp16 in shared
 *         memory by the GEMM (the g_w GEMM under HLQ_GW_INT8_X);
 * kind 3: A and B int8 codes, both widened (HLQ_GW_INT8_BOTH).
 * lda / ldb: row strides in elements (16-byte multiples).  bn: tile width
 * 96, 128 or 256 (0 = the library's choice); splits: K split count (0 = the
 * library's choice; > 1 needs d_ws of hlq_debug_tc_gemm_ws_bytes(M, N);
 * -1 = stream-K: one CTA per SM, each taking an equal run of the tiles'
 * k-blocks, the partial tiles summed exactly in d_ws; kinds 1-3 only, no
 * pairs; kind 0 runs unsplit); pair: 1 = a CTA pair per 256-row tile (tcgen05
 * cta_group::2; tile widths 128 and 256), 0 = one CTA per 128-row tile,
 * -1 = the library's choice.  M, N, K multiples of 16.  An unsupported
 * plan is HLQ_ERR_INVALID_ARG.
 */
hlq_status hlq_debug_tc_gemm(int kind, const void *d_a, int64_t lda,
                             const void *d_b, int64_t ldb, int64_t M, int64_t N,
                             int64_t K, int bn, int splits, int pair, int32_t *d_acc,
                             void *d_ws, size_t ws_bytes, void *stream);
size_t hlq_debug_tc_gemm_ws_bytes(int64_t M, int64_t N);

/*
 * The failure path of the library's bounded device waits, without a fault:
 * one CTA waits on an mbarrier that nothing arrives at, gives up after
 * limit_ns (0 < limit_ns <= 10^9), writes *d_result = 0 (device int32) and
 * raises HLQ_DEV_TIMEOUT in the status word (hlq_read_device_status).  The
 * context stays usable.
 */
hlq_status hlq_debug_wait_timeout(uint64_t limit_ns, int32_t *d_result, void *stream);

/*
 * The plans the layer entries choose for the two GEMMs of a layer on a GPU
 * with `sms` SMs (host computation only, nothing is launched): tile width
 * and K split of the g_x GEMM (E4M3, M = T, N = Cin, K = Cout) and of the
 * g_w GEMM (fp16, M = Cout, N = Cin, K = T*rank/16; split -1: stream-K, as
 * for hlq_debug_tc_gemm), and whether the g_w
 * GEMM is ordered after the g_x GEMM (1: each has at least one unit per SM,
 * so running them side by side would only delay the later one), and
 * whether each GEMM runs on CTA pairs (1) or one CTA per tile (0).
 */
hlq_status hlq_debug_gemm_plan(int64_t T, int64_t Cin, int64_t Cout, int rank, int sms,
                               int *gx_bn, int *gx_splits, int *gw_bn, int *gw_splits,
                               int *in_sequence, int *gx_pair, int *gw_pair);

/*
 * Layer-wise quantizer selection for the HQ of g_y (HOT summary page,
 * Approach: per-token or per-tensor quantizer chosen per layer; Limitations:
 * the choice comes from calibration data, switching where the two
 * quantizers' errors differ by half).  On a
 * calibration sample d_gy [T, Cout] (dtype dt): Y = the 16-point Hadamard
 * transform along Cout as in hlq_linear_backward_gx, quantized to int4 with
 * round-to-nearest-even codes at both granularities,
 *   d_mse[0] = mean over all T*Cout elements of (q*s - Y)^2, per tensor,
 *   d_mse[1] = the same per token (fp64, each difference exact),
 *   *d_choice = HLQ_PER_TOKEN if d_mse[0] > threshold * d_mse[1] else
 *               HLQ_PER_TENSOR  (threshold 1.5 reads "50 %").
 * d_mse: 2 doubles (8-byte aligned), d_choice: 1 int32, both device memory.
 * Workspace: hlq_workspace_bytes(HLQ_OP_SELECT_GRANULARITY, ...).  The sums
 * are accumulated with atomics, so the last bits of d_mse may differ
 * between runs; the choice differs only within that rounding of the
 * threshold.
 */
hlq_status hlq_select_gy_granularity(const void *d_gy, int dt, int64_t T,
                                     int64_t Cout, int block, double threshold,
                                     double *d_mse, int32_t *d_choice, void *d_ws,
                                     size_t ws_bytes, void *stream);

/*
 * Ablation of the weight-gradient path, for numerical-error studies (HOT
 * summary page, ablation table: Hadamard-transformed 4-bit quantization on
 * one gradient path; as printed the table names the two paths the other way
 * round from the method's own assignment of HQ to g_x and HLA to g_w, so its
 * path labels are read as swapped, and this is that row on the weight-
 * gradient path, in place of HLA + int8): g_y and
 * x are both transformed along tokens in blocks of 16 (the contraction dim
 * of g_w), quantized to int4 per tensor exactly as the HQ of w in
 * hlq_linear_backward_gx (SR on Philox streams 2 for g_y and 3 for x, element
 * e = t*C + c of the transformed [T, C] tensor), and
 *   acc[o, i] = sum_t qG[t, o] qX[t, i]  (exact),  g_w = acc * s_g * s_x / 16.
 * d_gy [T, Cout], d_x [T, Cin] (dtype dt) -> d_gw [Cout, Cin] fp32; d_acc
 * [Cout, Cin] int32 may be NULL (else it receives acc).  Needs 49 * T < 2^24.
 * Workspace: hlq_workspace_bytes(HLQ_OP_ABLATION_GW_HQ, ...).
 */
hlq_status hlq_ablation_gw_hq(const void *d_gy, const void *d_x, int dt, int64_t T,
                              int64_t Cin, int64_t Cout, int block, int rnd,
                              uint64_t seed, float *d_gw, int32_t *d_acc, void *d_ws,
                              size_t ws_bytes, void *stream);

/*
 * Ablation of the activation-gradient path, for numerical-error studies (HOT
 * summary page, ablation table: internal HLA on a gradient path, the path
 * labels read as swapped as for hlq_ablation_gw_hq, i.e. HLA on the g_x
 * contraction; quantized with the int8 rule HLA is paired with on the g_w
 * path): the contraction dim of g_x = g_y . w is Cout, and both operands
 * keep the `rank` lowest-sequency Walsh rows of each 16-block of Cout,
 *   Gb[t, r*b + k] = RN_f32( sum_j H16[sigma(k)][j] g_y[t, 16b + j] ),
 *   Wb[i, r*b + k] = RN_f32( sum_j H16[sigma(k)][j] w[16b + j, i] ),
 *   s = RN(amax/127) per tensor for each, RNE int8 codes,
 *   acc[t, i] = sum_c' qG[t, c'] qW[i, c']  (exact, c' < Cout*rank/16),
 *   g_x = acc * s_g * s_w / 16.
 * d_gy [T, Cout], d_w [Cout, Cin] (dtype dt) -> d_gx [T, Cin] fp32; d_acc
 * [T, Cin] int32 may be NULL (else it receives acc).  Needs
 * Cout*rank/16 * 127^2 < 2^31.  rank in {1, 2, 4, 8, 16}.
 * Workspace: hlq_workspace_bytes(HLQ_OP_ABLATION_GX_HLA, ..., rank).
 */
hlq_status hlq_ablation_gx_hla(const void *d_gy, const void *d_w, int dt, int64_t T,
                               int64_t Cin, int64_t Cout, int block, int rank,
                               float *d_gx, int32_t *d_acc, void *d_ws, size_t ws_bytes,
                               void *stream);

/*
 * One layer step from HOST buffers, every host<->device copy inside the
 * call: the ACBP compression of x (as hlq_compress_activation) and both
 * gradients (as hlq_linear_backward), results copied back to the host.
 * This entry has no counterpart in the pages (they run inside a training
 * framework with device-resident tensors); it serves callers whose data
 * lives in host memory, and it overlaps the copies with the computation:
 * g_y goes up in chunks of `chunk_tokens` rows (a multiple of 128; 0 = the
 * library's choice, ~16 MB of g_y per chunk) on a copy stream, the HQ of
 * each chunk and its g_x GEMM start as soon as it has landed, each g_x chunk
 * goes back to the host on a second copy stream while later chunks compute,
 * and the g_w branch (HLA of g_y, then the compression of x, the widening
 * and the g_w GEMM) runs alongside.  Results are bit-identical to the
 * device entry points on the same inputs.
 *   h_x [T, Cin], h_gy [T, Cout], h_w [Cout, Cin]: host, dtype dt;
 *   h_gx [T, Cin], h_gw [Cout, Cin]: host fp32 outputs;
 *   d_xbar (int8 [Cin, T'] or packed int4 [Cin, T'/2], per xbar_fmt as in
 *   hlq_compress_activation) and d_xbar_scale [1] or [Cin]: device, filled by the
 *   call (the stored activation of the step);
 *   d_ws: device workspace of hlq_layer_step_host_workspace_bytes(...),
 *   which also holds the device copies of the inputs and outputs.
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister):
 * pageable memory works but the copies are then staged and slower.  The call
 * is asynchronous on `stream`: the host buffers must stay valid, and h_gx /
 * h_gw are complete, only once `stream` has reached the end of the call.
 * Arguments are validated as for the device entry points (host pointers
 * non-null when their tensor is non-empty; chunk_tokens >= 0).
 */
hlq_status hlq_layer_step_host(const void *h_x, const void *h_gy, const void *h_w,
                               int dt, int64_t T, int64_t Cin, int64_t Cout,
                               int block, int rank, int xbar_fmt, int gran_gy,
                               int gran_w, int rnd, uint64_t seed, float *h_gx, float *h_gw,
                               int8_t *d_xbar, float *d_xbar_scale,
                               int64_t chunk_tokens, void *d_ws, size_t ws_bytes,
                               void *stream);
size_t hlq_layer_step_host_workspace_bytes(int dt, int64_t T, int64_t Cin,
                                           int64_t Cout, int block, int rank);

/*
 * Launch tracing, for timing without a profiler.  hlq_trace_begin creates
 * 2*capacity CUDA events (host-side objects, no device memory) and turns
 * tracing on: every later kernel launch of this library, on any stream, is
 * bracketed by two events recorded on that stream, up to `capacity` launches
 * (later ones run untraced).  hlq_trace_end turns tracing off, waits for the
 * recorded events and returns how many launches were traced; hlq_trace_get
 * gives launch i's kernel name (static string) and its device time in ms.
 * hlq_trace_free destroys the events.  Not thread-safe: trace from one host
 * thread at a time.  Launches traced while their stream is being captured
 * into a CUDA graph record their events as external event nodes: every
 * replay of the graph re-records them, and hlq_trace_get (after the replay
 * has finished) returns that replay's times.
 */
hlq_status hlq_trace_begin(int capacity);
hlq_status hlq_trace_end(int *n_launches);
hlq_status hlq_trace_get(int i, const char **name, float *ms);
hlq_status hlq_trace_free(void);

/*
 * hlq_linear_backward_gx for callers that cannot allocate device memory:
 * code hosted by another runtime that owns all device memory and gives
 * plugins none, or loops that forbid cudaMalloc/cudaFree (which can
 * synchronize the device) once running.  It computes exactly what
 * hlq_linear_backward_gx computes, with the same arguments minus the
 * workspace, and allocates nothing: its scratch is one fixed device array
 * of this library of hlq_noalloc_scratch_bytes() bytes (40 MiB), held by
 * every GPU that loads the library until the process exits.  The paper has
 * no counterpart to this entry point.
 *  - Sizes whose scratch (the g_x workspace of hlq_workspace_bytes) exceeds
 *    that array are refused with HLQ_ERR_WORKSPACE before anything runs.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the array, which keeps the last call's contents; each
 *    call clears what must start at zero.  Calls whose work overlaps on the
 *    GPU (other streams, other host threads) race on the array: order them
 *    on one stream or synchronize between them.
 *  - The looked-up address is kept for the life of the process, like the
 *    address of the library's device status word: a cudaDeviceReset while
 *    the library is in use unloads its device code and leaves both stale,
 *    and is not supported.
 */
hlq_status hlq_linear_backward_gx_noalloc(const void *d_gy, const void *d_w, int dt,
                                          int64_t T, int64_t Cin, int64_t Cout,
                                          int block, int gran_gy, int gran_w,
                                          int rnd, uint64_t seed, float *d_gx,
                                          void *stream);
size_t hlq_noalloc_scratch_bytes(void);

/* Static text for a status code. */
const char *hlq_status_string(int status);

/* Library version, e.g. 0x000100 for 0.1.0. */
int hlq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HLQ_H */
