// hlq_gemm_simple.cu -- exact integer GEMM on the CUDA cores (dp4a).
//
// A deliberately plain second opinion for the tensor-core GEMMs: 64x64
// output tiles, operands decoded to int8 in shared memory, int32 dp4a
// accumulation (exact for every size the API admits), and the same dequant
// epilogue as the tensor-core path.
#include <cstdint>

#include "hlq_device.cuh"
#include "hlq_kernels.h"

namespace hlq {

namespace {

constexpr int kTile = 64;
constexpr int kKStep = 64;          // codes per k-step
constexpr int kWords = kKStep / 4;  // int32 words per row per k-step

__device__ __forceinline__ int decode_code(const void* base, int fmt,
                                           int64_t idx) {
  if (fmt == kFmtE4M3)
    return int_of_e4m3(static_cast<const uint8_t*>(base)[idx]);
  if (fmt == kFmtI8) return static_cast<const int8_t*>(base)[idx];
  return __half2int_rn(static_cast<const __half*>(base)[idx]);
}

// Load 4 consecutive codes (k..k+3, zero past K) as a packed int8x4 word.
__device__ __forceinline__ uint32_t load_word(const void* base, int fmt,
                                              int64_t row, int64_t K,
                                              int64_t k) {
  uint32_t w = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    int v = (k + t < K) ? decode_code(base, fmt, row * K + k + t) : 0;
    w |= (uint32_t)(v & 0xff) << (8 * t);
  }
  return w;
}

__global__ void __launch_bounds__(256) gemm_simple_kernel(
    const void* __restrict__ A, int fmtA, const void* __restrict__ B, int fmtB,
    int64_t M, int64_t N, int64_t K, const float* __restrict__ sa,
    int per_row_a, const float* __restrict__ sb, float* __restrict__ out,
    int32_t* __restrict__ acc_out) {
  __shared__ uint32_t As[kTile][kWords + 1];
  __shared__ uint32_t Bs[kTile][kWords + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t m0 = (int64_t)blockIdx.y * kTile, n0 = (int64_t)blockIdx.x * kTile;
  int acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += kKStep) {
    for (int idx = threadIdx.x; idx < kTile * kWords; idx += blockDim.x) {
      const int r = idx / kWords, w = idx % kWords;
      const int64_t k = k0 + 4 * w;
      As[r][w] = (m0 + r < M) ? load_word(A, fmtA, m0 + r, K, k) : 0u;
      Bs[r][w] = (n0 + r < N) ? load_word(B, fmtB, n0 + r, K, k) : 0u;
    }
    __syncthreads();
#pragma unroll 4
    for (int w = 0; w < kWords; ++w) {
      int a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = (int)As[ty + 16 * i][w];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = (int)Bs[tx + 16 * j][w];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __dp4a(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty + 16 * i;
    if (m >= M) continue;
    const float scale = out ? (per_row_a ? sa[m] : sa[0]) * sb[0] : 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx + 16 * j;
      if (n >= N) continue;
      if (out) out[m * N + n] = (float)acc[i][j] * scale * 0.0625f;
      if (acc_out) acc_out[m * N + n] = acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simple(const void* A, int fmtA, const void* B,
                               int fmtB, int64_t M, int64_t N, int64_t K,
                               const float* sa, bool per_row_a,
                               const float* sb, float* out, int32_t* acc_out,
                               cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  dim3 grid((unsigned)((N + kTile - 1) / kTile), (unsigned)((M + kTile - 1) / kTile));
  gemm_simple_kernel<<<grid, 256, 0, st>>>(A, fmtA, B, fmtB, M, N, K, sa,
                                           per_row_a ? 1 : 0, sb, out, acc_out);
  return cudaGetLastError();
}

}  // namespace hlq
