// hlq_kernels.h -- host-side launchers of the libhlq kernels (internal).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "hlq.h"

namespace hlq {

// HQ of a [rows, cols] tensor along cols (g_y).  amax_only: per-tensor
// pre-pass into *amax_slot.  Otherwise writes E4M3 codes [rows, cols] and
// scales ([rows] if per_token else [1], from *amax_slot).  The rows may be
// rows row0 .. of a larger tensor (pointers already offset): the random
// words are drawn for their element indices in that tensor.
cudaError_t launch_hq_rows(const void* src, bool bf16, int64_t rows,
                           int64_t cols, bool per_token, bool amax_only,
                           unsigned int* amax_slot, uint8_t* codes,
                           float* scales, int rnd, uint64_t seed,
                           uint32_t stream_id, unsigned int* status,
                           cudaStream_t st, int64_t row0 = 0);

// HQ of a [rows, cols] tensor along rows (w), codes written transposed
// [cols, rows] (E4M3), per-tensor scale from *amax_slot.
// Layer-wise quantizer selection: RNE int4 HQ errors of g_y per tensor
// (scale from *amax_slot) and per token added into sums[0..1] (zeroed by the
// caller), then mse[g] = sums[g] / (rows * cols) and *choice.
cudaError_t launch_hq_mse(const void* src, bool bf16, int64_t rows, int64_t cols,
                          const unsigned int* amax_slot, double* sums, double threshold,
                          double* mse, int32_t* choice, unsigned int* status,
                          cudaStream_t st);

cudaError_t launch_hq_cols(const void* src, bool bf16, int64_t rows,
                           int64_t cols, bool amax_only,
                           unsigned int* amax_slot, uint8_t* codes_t,
                           float* scale, int rnd, uint64_t seed,
                           uint32_t stream_id, unsigned int* status,
                           cudaStream_t st);

// Output formats of launch_hla: int8 codes, their fp16 values, or int4
// codes packed two per byte (even ranks only).
constexpr int kHlaOutI8 = 0, kHlaOutF16 = 1, kHlaOutI4 = 2;

// HLA of src [T, C] along tokens -> codes [C, T*rank/16] in `out_fmt`,
// per-tensor scale RN(amax/qmax) from *amax_slot (qmax 7 for int4, else 127).
// out_ld: row stride of `out` in codes (>= T*rank/16).
// per_col: one amax slot and one scale per column c of src (amax_slot[c],
// scale[c]; the code row of channel c) instead of one for the tensor.
cudaError_t launch_hla(const void* src, bool bf16, int64_t T, int64_t C,
                       int rank, bool amax_only, int out_fmt,
                       unsigned int* amax_slot, void* out, int64_t out_ld,
                       float* scale, unsigned int* status, cudaStream_t st,
                       bool per_col = false);

// HLA along the rows of src [rows, cols]: per 16-block of a row the rank
// lowest-sequency coefficients, per-tensor amax pass (amax_only) or int8 RNE
// codes with s = RN(amax/127) stored as fp16 [rows, out_ld] (column
// rank*b + k), scale[0] = s.
cudaError_t launch_hla_rows(const void* src, bool bf16, int64_t rows, int64_t cols,
                            int rank, bool amax_only, unsigned int* amax_slot, void* out,
                            int64_t out_ld, float* scale, unsigned int* status,
                            cudaStream_t st);

// Fused reader of g_y [T, C] for both paths, one pass per call: amax_only
// gives the HQ maxima (per row into hq_amax[T] when per_token, else one slot)
// and the HLA maximum (hla_amax); otherwise the HQ E4M3 codes qy [T, C] with
// scales sgy ([T] or [1]) and the HLA int8 codes as fp16 qg [C, hla_ld] with
// scale sg[0], exactly as launch_hq_rows and launch_hla produce them.
cudaError_t launch_gy_fused(const void* gy, bool bf16, int64_t T, int64_t C, int rank,
                            bool per_token, bool amax_only, unsigned int* hq_amax,
                            unsigned int* hla_amax, uint8_t* qy, float* sgy, void* qg,
                            int64_t hla_ld, float* sg, int rnd, uint64_t seed,
                            unsigned int* status, cudaStream_t st);

// One CTA waiting on an mbarrier that never completes, for limit_ns: sets
// *result = 0 and raises HLQ_DEV_TIMEOUT in the status word.
// Device address of the library's status word (HLQ_DEV_* flags) on the
// current device; the word lives with the kernels that raise its flags.
cudaError_t status_word_address(unsigned int** out);

cudaError_t launch_wait_timeout_probe(unsigned long long limit_ns, int32_t* result,
                                      unsigned int* status, cudaStream_t st);

// Transform only (fp32 coefficients), for bit-exact checks.
cudaError_t launch_hq_rows_transform(const void* src, bool bf16, int64_t rows,
                                     int64_t cols, float* Y,
                                     unsigned int* status, cudaStream_t st);
cudaError_t launch_hq_cols_transform(const void* src, bool bf16, int64_t rows,
                                     int64_t cols, float* Y,
                                     unsigned int* status, cudaStream_t st);
cudaError_t launch_hla_transform(const void* src, bool bf16, int64_t T,
                                 int64_t C, int rank, float* out,
                                 unsigned int* status, cudaStream_t st);

// in [rows, cols] int8 (row stride cols), or packed int4 -> out [rows, out_ld]
// fp16.
cudaError_t launch_widen_i4_f16(const uint8_t* in, void* out, int64_t rows, int64_t cols,
                                int64_t out_ld, cudaStream_t st);
cudaError_t launch_widen_i8_f16(const int8_t* in, void* out, int64_t rows,
                                int64_t cols, int64_t out_ld, cudaStream_t st);
cudaError_t launch_pack_e4m3_int4(const uint8_t* in, uint8_t* out, int64_t n,
                                  cudaStream_t st);
cudaError_t launch_decode_e4m3(const uint8_t* in, int8_t* out, int64_t n,
                               cudaStream_t st);
cudaError_t launch_decode_f16(const void* in, int8_t* out, int64_t rows,
                              int64_t cols, int64_t ld, cudaStream_t st);

// Operand code formats of the GEMMs.
enum CodeFmt { kFmtE4M3 = 0, kFmtI8 = 1, kFmtF16 = 2 };

// Exact integer GEMM on CUDA cores (dp4a): acc[m, n] = sum_k A[m,k] B[n,k],
// A [M, K], B [N, K] (contraction dim contiguous).  Epilogue:
// out[m, n] = float(acc) * (sa[per_row_a ? m : 0] * sb[0]) * 0.0625f.
// acc_out (nullable) receives the int32 sums.
cudaError_t launch_gemm_simple(const void* A, int fmtA, const void* B,
                               int fmtB, int64_t M, int64_t N, int64_t K,
                               const float* sa, bool per_row_a,
                               const float* sb, float* out, int32_t* acc_out,
                               cudaStream_t st);

// A TMA tensor map over a row-major [rows, cols] bf16 / fp32 matrix with
// boxes of box_rows x box_cols, no swizzle, zero fill outside the matrix.
bool make_tile_map_2d(CUtensorMap* map, const void* ptr, bool bf16, int64_t rows,
                      int64_t cols, int box_cols, int box_rows);

// Tensor-core GEMM (hlq_gemm_tc.cu).  kind 0: E4M3 operands (int4 codes),
// kind 1: fp16 operands (int8 codes).  A [M, K] (row stride lda elements),
// B [N, K] (ldb); out [M, N] fp32 = acc * sa[m or 0] * sb[0] / 16.
// raw (kind 1 only): kRawB / kRawA mark an operand given as int8 codes in
// HBM (row stride in bytes, a multiple of 16, base 16-byte aligned), widened
// to fp16 in shared memory inside the GEMM.
struct GemmPlan {
  int bn = 128;      // tile width (96, 128 or 256)
  int splits = 1;    // K split count (int32 workspace reduction)
  int num_kb = 0;    // k-blocks of 128 bytes
  int chunk_kb = 0;  // k-blocks per exact fp32 accumulation chunk
  int pair = 0;      // 1: a CTA pair per 256-row tile (tcgen05 cta_group::2)
  int stream_k = 0;  // 1: equal k-block runs per SM over all tiles (kind 1,
                     // unsplit, no pairs; partial tiles summed like K splits)
};
GemmPlan plan_gemm_tc(int kind, int64_t M, int64_t N, int64_t K, int num_sms,
                      int max_splits);
size_t gemm_tc_split_ws_bytes(int64_t M, int64_t N);
cudaError_t launch_gemm_tc(int kind, const void* A, int64_t lda, const void* B,
                           int64_t ldb, int64_t M, int64_t N, int64_t K,
                           const GemmPlan& plan, const float* sa, bool per_row_a,
                           const float* sb, float* out, int32_t* acc_out,
                           void* split_ws, unsigned int* status, cudaStream_t st,
                           bool per_col_b = false,  // sb[n] per column (kind 1)
                           int raw = 0);
constexpr int kRawB = 1, kRawA = 2;

// The g_x path with a given workspace (the body of hlq_linear_backward_gx)
// and the workspace it needs.
size_t gx_workspace_bytes(int64_t T, int64_t Cin, int64_t Cout);
hlq_status backward_gx_with_ws(const void* gy, const void* w, int dt, int64_t T,
                               int64_t Cin, int64_t Cout, int block, int gran_gy,
                               int gran_w, int rnd, uint64_t seed, float* gx,
                               void* ws, size_t ws_bytes, void* stream);

}  // namespace hlq
