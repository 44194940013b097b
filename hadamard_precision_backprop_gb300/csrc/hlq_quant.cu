// hlq_quant.cu -- the transform/quantize kernels of the HLQ backward pass.
//
//  hq_rows_kernel : HQ of g_y [T, Cout] along Cout (16-point Walsh-Hadamard
//                   per block of 16 contiguous values, int4 codes with
//                   Philox stochastic rounding, per-token or per-tensor
//                   scale).  "HLQ: Fast and Efficient Backpropagation via
//                   Hadamard Low-rank Quantization", sections "Hadamard
//                   Transform" and "Alternative Optimization Technique:
//                   Hadamard Quantization"; HOT, Approach (layer-wise
//                   quantizer selection).
//  hq_cols_kernel : HQ of w [Cout, Cin] along Cout (blocks of 16 rows),
//                   written transposed [Cin, Cout] so the contraction dim is
//                   contiguous for the GEMM.
//  hla_kernel     : HLA along tokens (16-token blocks, the `rank` lowest-
//                   sequency Walsh rows kept), per-tensor int8 codes with
//                   round-to-nearest-even, written [C, T'] (token dim
//                   contiguous).  "HLQ ...", section "Analysis on Hadamard
//                   Low-rank Approximation for Backpropagation"; HOT,
//                   Approach (HLA + INT8 on the weight-gradient path, and
//                   compression of the stored activation at forward time).
//
// Every kernel has an AMAX mode (the per-tensor pre-pass: transform and
// reduce max|coefficient| into a 32-bit slot) and a QUANT mode.  The
// transform result is the exact sum rounded once to fp32: the fp32 butterfly
// when the block's exponent spread makes it exact, else exact_sum16.
//
// Code formats written here (one byte or one bf16 per code, so that the
// tensor-core GEMMs can read them without any widening):
//   int4 HQ codes  -> E4M3 bytes (integers -7..7 are exact in E4M3)
//   int8 HLA codes -> int8 bytes, or bf16 values (integers up to 256 exact)
#include <cstdint>

#include "hlq_device.cuh"
#include "hlq_kernels.h"

namespace hlq {

enum Mode { kAmax = 0, kQuant = 1 };

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) {
  return a < b ? a : b;
}

// ---------------------------------------------------------------------------
// Row transform: one warp per row, each lane an octet (8 contiguous values);
// lanes 2p and 2p+1 hold the two halves of one 16-block.
// ---------------------------------------------------------------------------
template <bool kBf16>
__device__ __forceinline__ void load_octet(const void* src, int64_t idx,
                                           bool valid, float* v) {
  if (!valid) {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = 0.0f;
    return;
  }
  if (kBf16) {
    uint4 r = __ldg(reinterpret_cast<const uint4*>(
        static_cast<const uint16_t*>(src) + idx));
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x);
    v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
    v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z);
    v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
  } else {
    const float4* p =
        reinterpret_cast<const float4*>(static_cast<const float*>(src) + idx);
    float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// Transform one octet in place (all 32 lanes must call this together).
template <bool kBf16>
__device__ __forceinline__ void transform_octet(float* v, unsigned int* status) {
  const int lane = threadIdx.x & 31;
  const bool upper = (lane & 1) != 0;
  ExpRange er = exp_range_init();
#pragma unroll
  for (int k = 0; k < 8; ++k) exp_range_add(er, v[k]);
  er.emax = max(er.emax, __shfl_xor_sync(0xffffffffu, er.emax, 1));
  er.emin = min(er.emin, __shfl_xor_sync(0xffffffffu, er.emin, 1));
  if (any_nonfinite(er)) raise_flag(status, HLQ_DEV_NONFINITE);
  const bool exact = butterfly_exact<kBf16>(er);
  // When some block of the warp defeats the fp32 butterfly, gather its 16
  // inputs first (shuffles stay warp-uniform), then overwrite below.
  const bool any_slow = !__all_sync(0xffffffffu, exact);
  float full[16];
  if (any_slow) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float o = __shfl_xor_sync(0xffffffffu, v[k], 1);
      full[k] = upper ? o : v[k];
      full[8 + k] = upper ? v[k] : o;
    }
  }
  fwht8(v);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float o = __shfl_xor_sync(0xffffffffu, v[k], 1);
    v[k] = upper ? (o - v[k]) : (v[k] + o);
  }
  if (!exact) {
    const int base = upper ? 8 : 0;
    for (int k = 0; k < 8; ++k) v[k] = exact_sum16(full, hrow_negmask(base + k));
  }
}

// kPerToken: scale per row computed in a first pass over the row.
// Otherwise (per tensor) the amax comes from `amax_slot` (AMAX mode fills it).
template <bool kBf16, int kMode, bool kPerToken>
__global__ void __launch_bounds__(256) hq_rows_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    unsigned int* __restrict__ amax_slot, uint8_t* __restrict__ codes,
    float* __restrict__ scales, int rnd, uint64_t seed, uint32_t stream,
    unsigned int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
  if (row >= rows) return;  // whole warp leaves together
  const int64_t n_oct = cols >> 3;
  const int iters = (int)((n_oct + 31) >> 5);
  const int64_t base = row * cols;

  float amax = 0.0f;
  if (kMode == kAmax || kPerToken) {
    for (int it = 0; it < iters; ++it) {
      const int64_t oct = (int64_t)it * 32 + lane;
      const bool valid = oct < n_oct;
      float v[8];
      load_octet<kBf16>(src, base + oct * 8, valid, v);
      transform_octet<kBf16>(v, status);
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
    }
    amax = warp_max(amax);
    if (kMode == kAmax) {
      if (lane == 0) atomic_max_nonneg(amax_slot, amax);
      return;
    }
  } else {
    amax = __uint_as_float(*amax_slot);
  }
  const float s = __fdiv_rn(amax, 7.0f);
  if (lane == 0) {
    if (kPerToken) scales[row] = s;
    else if (row == 0) scales[0] = s;
  }
  for (int it = 0; it < iters; ++it) {
    const int64_t oct = (int64_t)it * 32 + lane;
    const bool valid = oct < n_oct;
    float v[8];
    load_octet<kBf16>(src, base + oct * 8, valid, v);
    transform_octet<kBf16>(v, status);
    if (!valid) continue;
    const int64_t e0 = base + oct * 8;  // element index of v[0]
    uint32_t word[8];
    if (rnd == HLQ_SR) {
      U4 a = philox_block(seed, stream, (uint64_t)e0 >> 2);
      U4 b = philox_block(seed, stream, ((uint64_t)e0 >> 2) + 1);
      word[0] = a.x; word[1] = a.y; word[2] = a.z; word[3] = a.w;
      word[4] = b.x; word[5] = b.y; word[6] = b.z; word[7] = b.w;
    }
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      int q = (rnd == HLQ_SR) ? quant_sr(v[k], s, word[k], 7) : quant_rne(v[k], s, 7);
      uint32_t b = e4m3_of_int(q);
      if (k < 4) lo |= b << (8 * k);
      else hi |= b << (8 * (k - 4));
    }
    *reinterpret_cast<uint2*>(codes + e0) = make_uint2(lo, hi);
  }
}

// ---------------------------------------------------------------------------
// Column transform (w): one thread per (16-row block, 4 adjacent columns).
// Output codes are written transposed: codes[c * rows + 16b + i].
// ---------------------------------------------------------------------------
template <bool kBf16>
__device__ __forceinline__ void load_quad(const void* src, int64_t idx, float* v) {
  if (kBf16) {
    uint2 r = __ldg(reinterpret_cast<const uint2*>(
        static_cast<const uint16_t*>(src) + idx));
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x);
    v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
  } else {
    float4 a = __ldg(reinterpret_cast<const float4*>(
        static_cast<const float*>(src) + idx));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  }
}

template <bool kBf16>
__device__ __forceinline__ void transform_column16(float* col, unsigned int* status) {
  ExpRange er = exp_range_init();
#pragma unroll
  for (int j = 0; j < 16; ++j) exp_range_add(er, col[j]);
  if (any_nonfinite(er)) raise_flag(status, HLQ_DEV_NONFINITE);
  if (butterfly_exact<kBf16>(er)) {
    fwht16(col);
  } else {
    float in[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) in[j] = col[j];
    for (int i = 0; i < 16; ++i) col[i] = exact_sum16(in, hrow_negmask(i));
  }
}

template <bool kBf16, int kMode>
__global__ void __launch_bounds__(128) hq_cols_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    unsigned int* __restrict__ amax_slot, uint8_t* __restrict__ codes_t,
    float* __restrict__ scale, int rnd, uint64_t seed, uint32_t stream,
    unsigned int* __restrict__ status) {
  const int64_t cq = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // quad
  const int64_t b = blockIdx.y;                                       // block
  const bool valid = cq * 4 < cols;
  float v[4][16];
  if (valid) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float q[4];
      load_quad<kBf16>(src, (16 * b + j) * cols + cq * 4, q);
#pragma unroll
      for (int c = 0; c < 4; ++c) v[c][j] = q[c];
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) transform_column16<kBf16>(v[c], status);
  }
  if (kMode == kAmax) {
    float amax = 0.0f;
    if (valid) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[c][i]));
    }
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) atomic_max_nonneg(amax_slot, amax);
    return;
  }
  const float s = __fdiv_rn(__uint_as_float(*amax_slot), 7.0f);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) scale[0] = s;
  if (!valid) return;
  uint32_t packed[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int w = 0; w < 4; ++w) packed[c][w] = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t e = (uint64_t)((16 * b + i) * cols + cq * 4);
    U4 r = {0, 0, 0, 0};
    if (rnd == HLQ_SR) r = philox_block(seed, stream, e >> 2);
    const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int q = (rnd == HLQ_SR) ? quant_sr(v[c][i], s, words[c], 7)
                              : quant_rne(v[c][i], s, 7);
      packed[c][i >> 2] |= e4m3_of_int(q) << (8 * (i & 3));
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(codes_t + (cq * 4 + c) * rows + 16 * b) =
        make_uint4(packed[c][0], packed[c][1], packed[c][2], packed[c][3]);
}

// ---------------------------------------------------------------------------
// HLA along tokens.  CTA tile: 64 columns x 16 token blocks (256 tokens);
// thread (tx, ty): column pair tx (0..31), token blocks ty and ty + 8.
// Codes are staged in shared memory so each output row [c, T'] is written
// as contiguous 16-byte chunks.
// ---------------------------------------------------------------------------
constexpr int kHlaCols = 64;
constexpr int kHlaTB = 16;

template <bool kBf16>
__device__ __forceinline__ void load_pair(const void* src, int64_t idx, float* v) {
  if (kBf16) {
    uint32_t r = __ldg(reinterpret_cast<const uint32_t*>(
        static_cast<const uint16_t*>(src) + idx));
    v[0] = bf16_lo(r);
    v[1] = bf16_hi(r);
  } else {
    float2 a = __ldg(reinterpret_cast<const float2*>(
        static_cast<const float*>(src) + idx));
    v[0] = a.x;
    v[1] = a.y;
  }
}

// kOut: 0 = int8 codes, 1 = bf16-valued codes
template <bool kBf16, int kMode, int kOut>
__global__ void __launch_bounds__(256) hla_kernel(
    const void* __restrict__ src, int64_t T, int64_t C, int rank,
    unsigned int* __restrict__ amax_slot, void* __restrict__ out, int64_t out_ld,
    float* __restrict__ scale, unsigned int* __restrict__ status) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t n_tb = T >> 4;
  const int64_t Tp = n_tb * rank;
  const int64_t c0 = (int64_t)blockIdx.x * kHlaCols + 2 * tx;
  const int64_t tb0 = (int64_t)blockIdx.y * kHlaTB;
  const bool col_ok = c0 < C;
  constexpr int kBytes = kOut ? 2 : 1;
  const int row_codes = kHlaTB * rank;  // codes per column in this tile

  float s = 0.0f;
  if (kMode == kQuant) s = __fdiv_rn(__uint_as_float(*amax_slot), 127.0f);
  float amax = 0.0f;
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    const int tbl = ty + 8 * half;  // local token block
    const int64_t tb = tb0 + tbl;
    const bool ok = col_ok && tb < n_tb;
    float v[2][16];
    if (ok) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float p[2];
        load_pair<kBf16>(src, (16 * tb + j) * C + c0, p);
        v[0][j] = p[0];
        v[1][j] = p[1];
      }
      transform_column16<kBf16>(v[0], status);
      transform_column16<kBf16>(v[1], status);
    }
    if (kMode == kAmax) {
      if (ok)
        for (int k = 0; k < rank; ++k) {
          const int r = sequency_row(k);
          amax = fmaxf(amax, fmaxf(fabsf(v[0][r]), fabsf(v[1][r])));
        }
    } else if (ok) {
      for (int cc = 0; cc < 2; ++cc) {
        uint8_t* dst = smem + ((2 * tx + cc) * row_codes + tbl * rank) * kBytes;
        for (int k = 0; k < rank; ++k) {
          const int q = quant_rne(v[cc][sequency_row(k)], s, 127);
          if (kOut) {
            reinterpret_cast<__nv_bfloat16*>(dst)[k] = __int2bfloat16_rn(q);
          } else {
            reinterpret_cast<int8_t*>(dst)[k] = (int8_t)q;
          }
        }
      }
    }
  }
  if (kMode == kAmax) {
    amax = warp_max(amax);
    if (tx == 0) atomic_max_nonneg(amax_slot, amax);
    return;
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) scale[0] = s;
  __syncthreads();
  // Write the tile: column c gets codes [tb0*rank, (tb0+valid_tb)*rank).
  const int64_t valid_tb = imin64(kHlaTB, n_tb - tb0);
  const int64_t seg_bytes = valid_tb * rank * kBytes;
  const int64_t row_bytes = out_ld * kBytes;
  const bool vec = (seg_bytes % 16 == 0) && (row_bytes % 16 == 0) &&
                   ((tb0 * rank * kBytes) % 16 == 0);
  uint8_t* outb = static_cast<uint8_t*>(out);
  const int cols_here = (int)imin64(kHlaCols, C - (int64_t)blockIdx.x * kHlaCols);
  if (vec) {
    const int chunks = (int)(seg_bytes / 16);
    for (int idx = threadIdx.x; idx < cols_here * chunks; idx += blockDim.x) {
      const int cl = idx / chunks, ch = idx % chunks;
      const int64_t c = (int64_t)blockIdx.x * kHlaCols + cl;
      uint4 val = *reinterpret_cast<const uint4*>(smem + cl * row_codes * kBytes + ch * 16);
      *reinterpret_cast<uint4*>(outb + c * row_bytes + tb0 * rank * kBytes + ch * 16) = val;
    }
  } else {
    for (int idx = threadIdx.x; idx < cols_here * seg_bytes; idx += blockDim.x) {
      const int cl = (int)(idx / seg_bytes), by = (int)(idx % seg_bytes);
      const int64_t c = (int64_t)blockIdx.x * kHlaCols + cl;
      outb[c * row_bytes + tb0 * rank * kBytes + by] = smem[cl * row_codes * kBytes + by];
    }
  }
}

// ---------------------------------------------------------------------------
// Transform-only kernels (debug read-back of the exactly rounded Hadamard
// coefficients; same device functions as the quantizing kernels).
// ---------------------------------------------------------------------------
template <bool kBf16>
__global__ void __launch_bounds__(256) hq_rows_transform_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    float* __restrict__ Y, unsigned int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int64_t n_oct = cols >> 3;
  const int iters = (int)((n_oct + 31) >> 5);
  for (int it = 0; it < iters; ++it) {
    const int64_t oct = (int64_t)it * 32 + lane;
    const bool valid = oct < n_oct;
    float v[8];
    load_octet<kBf16>(src, row * cols + oct * 8, valid, v);
    transform_octet<kBf16>(v, status);
    if (!valid) continue;
    float4* dst = reinterpret_cast<float4*>(Y + row * cols + oct * 8);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(128) hq_cols_transform_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    float* __restrict__ Y, unsigned int* __restrict__ status) {
  const int64_t cq = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t b = blockIdx.y;
  if (cq * 4 >= cols) return;
  float v[4][16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float q[4];
    load_quad<kBf16>(src, (16 * b + j) * cols + cq * 4, q);
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c][j] = q[c];
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) transform_column16<kBf16>(v[c], status);
  for (int i = 0; i < 16; ++i)
    *reinterpret_cast<float4*>(Y + (16 * b + i) * cols + cq * 4) =
        make_float4(v[0][i], v[1][i], v[2][i], v[3][i]);
}

template <bool kBf16>
__global__ void __launch_bounds__(256) hla_transform_kernel(
    const void* __restrict__ src, int64_t T, int64_t C, int rank,
    float* __restrict__ out, unsigned int* __restrict__ status) {
  const int64_t cp = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // pair
  const int64_t tb = blockIdx.y;
  if (cp * 2 >= C) return;
  const int64_t Tp = (T >> 4) * rank;
  float v[2][16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float p[2];
    load_pair<kBf16>(src, (16 * tb + j) * C + 2 * cp, p);
    v[0][j] = p[0];
    v[1][j] = p[1];
  }
  transform_column16<kBf16>(v[0], status);
  transform_column16<kBf16>(v[1], status);
  for (int cc = 0; cc < 2; ++cc)
    for (int k = 0; k < rank; ++k)
      out[(2 * cp + cc) * Tp + tb * rank + k] = v[cc][sequency_row(k)];
}

// ---------------------------------------------------------------------------
// Format conversions (GEMM operand widening and debug read-back).
// ---------------------------------------------------------------------------
// int8 codes [rows, cols] -> bf16 codes [rows, out_ld]; 8 codes per thread
// (cols is a multiple of 8 on the vector path).
__global__ void widen_i8_to_bf16_kernel(const int8_t* __restrict__ in,
                                        __nv_bfloat16* __restrict__ out,
                                        int64_t rows, int64_t cols,
                                        int64_t out_ld) {
  const int64_t per_row = (cols + 7) / 8;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * per_row) return;
  const int64_t r = idx / per_row, c = (idx % per_row) * 8;
  const int8_t* src = in + r * cols + c;
  __nv_bfloat16* dst = out + r * out_ld + c;
  if (c + 8 <= cols && (cols % 8) == 0) {
    uint2 v = *reinterpret_cast<const uint2*>(src);
    const int8_t* b = reinterpret_cast<const int8_t*>(&v);
    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = __int2bfloat16_rn(b[k]);
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(o);
  } else {
    for (int k = 0; k < 8 && c + k < cols; ++k) dst[k] = __int2bfloat16_rn(src[k]);
  }
}

__global__ void decode_e4m3_kernel(const uint8_t* __restrict__ in,
                                   int8_t* __restrict__ out, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (int8_t)int_of_e4m3(in[i]);
}

__global__ void decode_bf16_kernel(const __nv_bfloat16* __restrict__ in,
                                   int8_t* __restrict__ out, int64_t rows,
                                   int64_t cols, int64_t ld) {
  const int64_t n = rows * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (int8_t)__bfloat162int_rn(in[(i / cols) * ld + i % cols]);
}

// ---------------------------------------------------------------------------
// Host-side launchers.
// ---------------------------------------------------------------------------
static inline unsigned grid1(int64_t n, int per) {
  return (unsigned)((n + per - 1) / per);
}

cudaError_t launch_hq_rows(const void* src, bool bf16, int64_t rows,
                           int64_t cols, bool per_token, bool amax_only,
                           unsigned int* amax_slot, uint8_t* codes,
                           float* scales, int rnd, uint64_t seed,
                           uint32_t stream_id, unsigned int* status,
                           cudaStream_t st) {
  const int threads = 256, warps = threads / 32;
  dim3 grid(grid1(rows, warps));
#define HQR(B, M, P)                                                        \
  hq_rows_kernel<B, M, P><<<grid, threads, 0, st>>>(src, rows, cols,        \
                                                    amax_slot, codes, scales, \
                                                    rnd, seed, stream_id, status)
  if (amax_only) {
    if (bf16) HQR(true, kAmax, false); else HQR(false, kAmax, false);
  } else if (per_token) {
    if (bf16) HQR(true, kQuant, true); else HQR(false, kQuant, true);
  } else {
    if (bf16) HQR(true, kQuant, false); else HQR(false, kQuant, false);
  }
#undef HQR
  return cudaGetLastError();
}

cudaError_t launch_hq_cols(const void* src, bool bf16, int64_t rows,
                           int64_t cols, bool amax_only,
                           unsigned int* amax_slot, uint8_t* codes_t,
                           float* scale, int rnd, uint64_t seed,
                           uint32_t stream_id, unsigned int* status,
                           cudaStream_t st) {
  const int threads = 128;
  dim3 grid(grid1(cols / 4, threads), (unsigned)(rows / 16));
#define HQC(B, M)                                                        \
  hq_cols_kernel<B, M><<<grid, threads, 0, st>>>(src, rows, cols, amax_slot, \
                                                 codes_t, scale, rnd, seed,  \
                                                 stream_id, status)
  if (amax_only) {
    if (bf16) HQC(true, kAmax); else HQC(false, kAmax);
  } else {
    if (bf16) HQC(true, kQuant); else HQC(false, kQuant);
  }
#undef HQC
  return cudaGetLastError();
}

size_t hla_smem_bytes(int rank, bool out_bf16) {
  return (size_t)kHlaCols * kHlaTB * rank * (out_bf16 ? 2 : 1);
}

cudaError_t launch_hla(const void* src, bool bf16, int64_t T, int64_t C,
                       int rank, bool amax_only, bool out_bf16,
                       unsigned int* amax_slot, void* out, int64_t out_ld,
                       float* scale, unsigned int* status, cudaStream_t st) {
  dim3 grid(grid1(C, kHlaCols), grid1(T / 16, kHlaTB));
  const size_t smem = amax_only ? 0 : hla_smem_bytes(rank, out_bf16);
#define HLA(B, M, O)                                                           \
  do {                                                                         \
    if (smem > 48 * 1024)                                                      \
      cudaFuncSetAttribute(hla_kernel<B, M, O>,                                \
                           cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                           (int)smem);                                         \
    hla_kernel<B, M, O><<<grid, 256, smem, st>>>(src, T, C, rank, amax_slot,   \
                                                 out, out_ld, scale, status);  \
  } while (0)
  if (amax_only) {
    if (bf16) HLA(true, kAmax, 0); else HLA(false, kAmax, 0);
  } else if (out_bf16) {
    if (bf16) HLA(true, kQuant, 1); else HLA(false, kQuant, 1);
  } else {
    if (bf16) HLA(true, kQuant, 0); else HLA(false, kQuant, 0);
  }
#undef HLA
  return cudaGetLastError();
}

cudaError_t launch_hq_rows_transform(const void* src, bool bf16, int64_t rows,
                                     int64_t cols, float* Y,
                                     unsigned int* status, cudaStream_t st) {
  dim3 grid(grid1(rows, 8));
  if (bf16) hq_rows_transform_kernel<true><<<grid, 256, 0, st>>>(src, rows, cols, Y, status);
  else hq_rows_transform_kernel<false><<<grid, 256, 0, st>>>(src, rows, cols, Y, status);
  return cudaGetLastError();
}

cudaError_t launch_hq_cols_transform(const void* src, bool bf16, int64_t rows,
                                     int64_t cols, float* Y,
                                     unsigned int* status, cudaStream_t st) {
  dim3 grid(grid1(cols / 4, 128), (unsigned)(rows / 16));
  if (bf16) hq_cols_transform_kernel<true><<<grid, 128, 0, st>>>(src, rows, cols, Y, status);
  else hq_cols_transform_kernel<false><<<grid, 128, 0, st>>>(src, rows, cols, Y, status);
  return cudaGetLastError();
}

cudaError_t launch_hla_transform(const void* src, bool bf16, int64_t T,
                                 int64_t C, int rank, float* out,
                                 unsigned int* status, cudaStream_t st) {
  dim3 grid(grid1(C / 2, 256), (unsigned)(T / 16));
  if (bf16) hla_transform_kernel<true><<<grid, 256, 0, st>>>(src, T, C, rank, out, status);
  else hla_transform_kernel<false><<<grid, 256, 0, st>>>(src, T, C, rank, out, status);
  return cudaGetLastError();
}

cudaError_t launch_widen_i8_bf16(const int8_t* in, void* out, int64_t rows,
                                 int64_t cols, int64_t out_ld, cudaStream_t st) {
  if (rows * cols == 0) return cudaSuccess;
  const int64_t n = rows * ((cols + 7) / 8);
  widen_i8_to_bf16_kernel<<<grid1(n, 256), 256, 0, st>>>(
      in, static_cast<__nv_bfloat16*>(out), rows, cols, out_ld);
  return cudaGetLastError();
}

cudaError_t launch_decode_e4m3(const uint8_t* in, int8_t* out, int64_t n,
                               cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  decode_e4m3_kernel<<<(unsigned)imin64(grid1(n, 256), 4096), 256, 0, st>>>(in, out, n);
  return cudaGetLastError();
}

cudaError_t launch_decode_bf16(const void* in, int8_t* out, int64_t rows,
                               int64_t cols, int64_t ld, cudaStream_t st) {
  const int64_t n = rows * cols;
  if (n == 0) return cudaSuccess;
  decode_bf16_kernel<<<(unsigned)imin64(grid1(n, 256), 4096), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(in), out, rows, cols, ld);
  return cudaGetLastError();
}

}  // namespace hlq
