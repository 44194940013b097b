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
//  col_kernel     : HQ of w [Cout, Cin] along Cout (blocks of 16 rows),
//                   written transposed [Cin, Cout] so the contraction dim is
//                   contiguous for the GEMM.
//  col_kernel     : HLA along tokens (16-token blocks, the `rank` lowest-
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

// The 16 exactly rounded Hadamard coefficients of a block whose exponent
// spread defeats the fp32 butterfly: int64 fixed point when it fits, else
// the wide exact accumulator.  Kept out of line so the common path stays
// small (it is taken by a small fraction of blocks).
__device__ __noinline__ void slow_block16(const float* in, float* out, int bf16) {
  const bool ok = bf16 ? fwht16_fixed<true>(in, out) : fwht16_fixed<false>(in, out);
  if (!ok)
    for (int i = 0; i < 16; ++i) out[i] = exact_sum16(in, hrow_negmask(i));
}

// Butterfly of one octet in place, given whether its 16-block is exact in the
// fp32 butterfly (both lanes of the pair agree).  All 32 lanes call this.
template <bool kBf16>
__device__ __forceinline__ void octet_butterfly(float* v, bool exact) {
  const int lane = threadIdx.x & 31;
  const bool upper = (lane & 1) != 0;
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
    float y[16];
    slow_block16(full, y, kBf16 ? 1 : 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = upper ? y[8 + k] : y[k];
  }
}

// Transform one octet in place (all 32 lanes must call this together).
template <bool kBf16>
__device__ __forceinline__ void transform_octet(float* v, unsigned int* status) {
  ExpRange er = exp_range_init();
#pragma unroll
  for (int k = 0; k < 8; ++k) exp_range_add(er, v[k]);
  er.emax = max(er.emax, __shfl_xor_sync(0xffffffffu, er.emax, 1));
  er.emin = min(er.emin, __shfl_xor_sync(0xffffffffu, er.emin, 1));
  if (any_nonfinite(er)) raise_flag(status, HLQ_DEV_NONFINITE);
  octet_butterfly<kBf16>(v, butterfly_exact<kBf16>(er));
}

// The same for eight packed bf16 values: the exponent range comes from
// two-lane 16-bit SIMD max/min over |bits| (zeros mapped to the largest
// pattern so that they drop out of the minimum), then the values unpack.
__device__ __forceinline__ void transform_octet_bf16(const uint4& raw, float* v,
                                                     unsigned int* status) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t mx = 0u, mn = 0x7fff7fffu;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t a = w[k] & 0x7fff7fffu;
    mx = __vmaxu2(mx, a);
    mn = __vminu2(mn, a | (__vcmpeq2(a, 0u) & 0x7fff7fffu));
  }
  uint32_t hi = max(mx & 0xffffu, mx >> 16);
  uint32_t lo = min(mn & 0xffffu, mn >> 16);
  hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, 1));
  lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, 1));
  const uint32_t emax = hi >> 7;
  if (emax == 255u) raise_flag(status, HLQ_DEV_NONFINITE);
  const bool all_zero = lo == 0x7fffu;
  const uint32_t emin = max(lo >> 7, 1u);
  const bool exact = all_zero || (emax <= 254u && emax - min(emin, emax) <= 12u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = bf16_lo(w[k]);
    v[2 * k + 1] = bf16_hi(w[k]);
  }
  octet_butterfly<true>(v, exact);
}

// Raw octet as loaded from HBM (kept packed while the row sits in registers).
template <bool kBf16>
struct RawOct;
template <>
struct RawOct<true> {
  uint4 a;
};
template <>
struct RawOct<false> {
  float4 a, b;
};

template <bool kBf16>
__device__ __forceinline__ RawOct<kBf16> load_raw(const void* src, int64_t idx,
                                                  bool valid);
template <>
__device__ __forceinline__ RawOct<true> load_raw<true>(const void* src, int64_t idx,
                                                       bool valid) {
  RawOct<true> r;
  r.a = valid ? __ldg(reinterpret_cast<const uint4*>(
                    static_cast<const uint16_t*>(src) + idx))
              : make_uint4(0, 0, 0, 0);
  return r;
}
template <>
__device__ __forceinline__ RawOct<false> load_raw<false>(const void* src, int64_t idx,
                                                         bool valid) {
  RawOct<false> r;
  const float4* p =
      reinterpret_cast<const float4*>(static_cast<const float*>(src) + idx);
  r.a = valid ? __ldg(p) : make_float4(0.f, 0.f, 0.f, 0.f);
  r.b = valid ? __ldg(p + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
  return r;
}

__device__ __forceinline__ void unpack(const RawOct<true>& r, float* v) {
  v[0] = bf16_lo(r.a.x); v[1] = bf16_hi(r.a.x);
  v[2] = bf16_lo(r.a.y); v[3] = bf16_hi(r.a.y);
  v[4] = bf16_lo(r.a.z); v[5] = bf16_hi(r.a.z);
  v[6] = bf16_lo(r.a.w); v[7] = bf16_hi(r.a.w);
}
__device__ __forceinline__ void unpack(const RawOct<false>& r, float* v) {
  v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
  v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
}

// Quantize one transformed octet (elements e0 .. e0+7) to E4M3 int4 codes.
__device__ __forceinline__ void quantize_octet(const float* v, float s, int rnd,
                                               const PhiloxKeys& keys, uint32_t stream,
                                               int64_t e0, uint8_t* codes) {
  float r[8];
  if (rnd == HLQ_SR) {
    const U4 a = philox_block_k(keys, stream, (uint64_t)e0 >> 2);
    const U4 b = philox_block_k(keys, stream, ((uint64_t)e0 >> 2) + 1);
    r[0] = quant_sr_f(v[0], s, a.x, 7.0f);
    r[1] = quant_sr_f(v[1], s, a.y, 7.0f);
    r[2] = quant_sr_f(v[2], s, a.z, 7.0f);
    r[3] = quant_sr_f(v[3], s, a.w, 7.0f);
    r[4] = quant_sr_f(v[4], s, b.x, 7.0f);
    r[5] = quant_sr_f(v[5], s, b.y, 7.0f);
    r[6] = quant_sr_f(v[6], s, b.z, 7.0f);
    r[7] = quant_sr_f(v[7], s, b.w, 7.0f);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) r[k] = quant_rne_f(v[k], s, 7.0f);
  }
  const uint32_t lo = e4m3x2(r[0], r[1]) | (e4m3x2(r[2], r[3]) << 16);
  const uint32_t hi = e4m3x2(r[4], r[5]) | (e4m3x2(r[6], r[7]) << 16);
  *reinterpret_cast<uint2*>(codes + e0) = make_uint2(lo, hi);
}

template <bool kBf16>
__device__ __forceinline__ void transform_raw(const RawOct<kBf16>& r, float* v,
                                              unsigned int* status);
template <>
__device__ __forceinline__ void transform_raw<true>(const RawOct<true>& r, float* v,
                                                    unsigned int* status) {
  transform_octet_bf16(r.a, v, status);
}
template <>
__device__ __forceinline__ void transform_raw<false>(const RawOct<false>& r, float* v,
                                                     unsigned int* status) {
  unpack(r, v);
  transform_octet<false>(v, status);
}

// One warp per row; lane = octet within each 256-value stretch of the row;
// the next octet's load is issued before the current one is transformed.
// kPerToken: the scale of a row comes from a first pass over it; the
// transformed values wait in shared memory (`stage`, when the launch gave
// room: 8 rows per CTA) so the second pass neither re-reads HBM nor
// re-transforms.  Per tensor: one pass, amax from `amax_slot` (which the
// AMAX mode fills).
template <bool kBf16, int kMode, bool kPerToken>
__global__ void __launch_bounds__(256) hq_rows_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    unsigned int* __restrict__ amax_slot, uint8_t* __restrict__ codes,
    float* __restrict__ scales, int rnd, uint64_t seed, uint32_t stream,
    unsigned int* __restrict__ status, int stage) {
  extern __shared__ float4 srow[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int warps = blockDim.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * warps + wid;
  if (row >= rows) return;  // whole warp leaves together
  const int n_oct = (int)(cols >> 3);
  const int iters = (n_oct + 31) >> 5;
  const int64_t base = row * cols;
  // staged octet (it, lane): float4 halves at [(2*it + h) * 32 + lane]
  float4* my = srow + (size_t)wid * iters * 64;

  float amax = 0.0f;
  if (kMode == kAmax || kPerToken) {
    RawOct<kBf16> cur = load_raw<kBf16>(src, base + lane * 8, lane < n_oct);
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
      const int oct = it * 32 + lane;
      const int nx = oct + 32;
      RawOct<kBf16> nxt = load_raw<kBf16>(src, base + (int64_t)nx * 8,
                                          it + 1 < iters && nx < n_oct);
      float v[8];
      transform_raw<kBf16>(cur, v, status);
      if (kPerToken && stage) {
        my[(2 * it) * 32 + lane] = make_float4(v[0], v[1], v[2], v[3]);
        my[(2 * it + 1) * 32 + lane] = make_float4(v[4], v[5], v[6], v[7]);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
      cur = nxt;
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
  const PhiloxKeys keys = philox_keys(seed);
  __syncwarp();
  if (kPerToken && stage) {
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
      const int oct = it * 32 + lane;
      if (oct >= n_oct) break;
      const float4 a = my[(2 * it) * 32 + lane], b = my[(2 * it + 1) * 32 + lane];
      const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      quantize_octet(v, s, rnd, keys, stream, base + (int64_t)oct * 8, codes);
    }
    return;
  }
  RawOct<kBf16> cur = load_raw<kBf16>(src, base + lane * 8, lane < n_oct);
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    const int oct = it * 32 + lane;
    const int nx = oct + 32;
    RawOct<kBf16> nxt = load_raw<kBf16>(src, base + (int64_t)nx * 8,
                                        it + 1 < iters && nx < n_oct);
    float v[8];
    transform_raw<kBf16>(cur, v, status);
    if (oct < n_oct) quantize_octet(v, s, rnd, keys, stream, base + (int64_t)oct * 8, codes);
    cur = nxt;
  }
}

// ---------------------------------------------------------------------------
// Column transforms: w (HQ along Cout, blocks of 16 rows, all 16 Sylvester
// rows, int4 codes) and x / g_y (HLA along tokens, blocks of 16 tokens, the
// `rank` lowest-sequency rows, int8 codes).  Both write [C, X] with the
// transformed dim contiguous (X = Cout for w, T' for HLA).
//
// Thread: kCPT = 2 adjacent columns of one 16-row block (4-byte bf16 /
// 8-byte fp32 loads, a warp reads 128/256 contiguous bytes per row).  CTA:
// 32 x 8 threads = 64 columns x 16 blocks (two per warp), codes staged in
// shared memory so every output row segment leaves as 16-byte stores.
// ---------------------------------------------------------------------------
enum ColOut { kColHqE4M3 = 0, kColI8 = 1, kColBf16 = 2 };
constexpr int kCPT = 2;               // columns per thread
constexpr int kColCols = 32 * kCPT;   // columns per CTA tile
constexpr int kColBlocks = 16;

template <bool kBf16>
__device__ __forceinline__ void load_pair(const void* src, int64_t idx, float* v) {
  if (kBf16) {
    const uint32_t r = __ldg(reinterpret_cast<const uint32_t*>(
        static_cast<const uint16_t*>(src) + idx));
    v[0] = bf16_lo(r);
    v[1] = bf16_hi(r);
  } else {
    const float2 a = __ldg(reinterpret_cast<const float2*>(
        static_cast<const float*>(src) + idx));
    v[0] = a.x;
    v[1] = a.y;
  }
}

// 16 rows x 2 adjacent columns, kept packed until used.
template <bool kBf16>
struct RawPairCol;
template <>
struct RawPairCol<true> {
  uint32_t p[16];
};
template <>
struct RawPairCol<false> {
  float2 p[16];
};

template <bool kBf16>
__device__ __forceinline__ void load_pair_col(const void* src, int64_t idx, int64_t ld,
                                              RawPairCol<kBf16>& r);
template <>
__device__ __forceinline__ void load_pair_col<true>(const void* src, int64_t idx,
                                                    int64_t ld, RawPairCol<true>& r) {
  const uint16_t* p = static_cast<const uint16_t*>(src) + idx;
#pragma unroll
  for (int j = 0; j < 16; ++j) r.p[j] = __ldg(reinterpret_cast<const uint32_t*>(p + j * ld));
}
template <>
__device__ __forceinline__ void load_pair_col<false>(const void* src, int64_t idx,
                                                     int64_t ld, RawPairCol<false>& r) {
  const float* p = static_cast<const float*>(src) + idx;
#pragma unroll
  for (int j = 0; j < 16; ++j) r.p[j] = __ldg(reinterpret_cast<const float2*>(p + j * ld));
}

template <bool kBf16>
__device__ __forceinline__ void unpack_pair_col(const RawPairCol<kBf16>& r, float (*v)[16]);
template <>
__device__ __forceinline__ void unpack_pair_col<true>(const RawPairCol<true>& r,
                                                      float (*v)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    v[0][j] = bf16_lo(r.p[j]);
    v[1][j] = bf16_hi(r.p[j]);
  }
}
template <>
__device__ __forceinline__ void unpack_pair_col<false>(const RawPairCol<false>& r,
                                                       float (*v)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    v[0][j] = r.p[j].x;
    v[1][j] = r.p[j].y;
  }
}

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

// Exactly rounded coefficients of one 16-value column, in place, given
// whether the fp32 butterfly is exact for it: the `rank` kept rows in
// sequency order in x[0..rank), or all 16 in Sylvester order when `natural`.
template <bool kBf16>
__device__ __forceinline__ void column_butterfly(float* x, bool exact, int rank,
                                                 bool natural) {
  if (exact) {
    float t[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = x[j];
    fwht16(t);
    if (natural) {
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = t[i];
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (k < rank) x[k] = t[sequency_row(k)];
    }
  } else {
    // rare: these two arrays live in local memory for the out-of-line call
    float in[16], o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) in[j] = x[j];
    slow_block16(in, o, kBf16 ? 1 : 0);
    if (natural) {
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = o[i];
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (k < rank) x[k] = o[sequency_row(k)];
    }
  }
}

template <bool kBf16>
__device__ __forceinline__ void column_coeffs(float* x, int rank, bool natural,
                                              unsigned int* status) {
  ExpRange er = exp_range_init();
#pragma unroll
  for (int j = 0; j < 16; ++j) exp_range_add(er, x[j]);
  if (any_nonfinite(er)) raise_flag(status, HLQ_DEV_NONFINITE);
  column_butterfly<kBf16>(x, butterfly_exact<kBf16>(er), rank, natural);
}

// Exactness of the two columns of 16 packed bf16 pairs (low half = column
// 0), by 16-bit SIMD max/min of |bits| as in transform_octet_bf16.
__device__ __forceinline__ void pair_col_exact_bf16(const uint32_t (&p)[16], bool* exact,
                                                    unsigned int* status) {
  uint32_t mx = 0u, mn = 0x7fff7fffu;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t a = p[j] & 0x7fff7fffu;
    mx = __vmaxu2(mx, a);
    mn = __vminu2(mn, a | (__vcmpeq2(a, 0u) & 0x7fff7fffu));
  }
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t hi = (mx >> (16 * c)) & 0xffffu, lo = (mn >> (16 * c)) & 0xffffu;
    const uint32_t emax = hi >> 7, emin = max(lo >> 7, 1u);
    if (emax == 255u) raise_flag(status, HLQ_DEV_NONFINITE);
    exact[c] = lo == 0x7fffu || (emax <= 254u && emax - min(emin, emax) <= 12u);
  }
}

// Shared-memory staging of a column tile: local row r = c * 32 + tx holds
// the codes of global column tile_base + kCPT * tx + c; a row is kColBlocks
// chunks of R codes plus one pad chunk (an odd number of chunks), so the 32
// chunk stores of a warp (consecutive rows) fall in distinct banks.
__device__ __forceinline__ int col_tile_col(int r) { return kCPT * (r & 31) + (r >> 5); }

// Store `n` bytes (4, 8, 16 or 32) of packed codes.
__device__ __forceinline__ void store_chunk(uint8_t* dst, const uint32_t* p, int n) {
  if (n >= 16) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(p[0], p[1], p[2], p[3]);
    if (n == 32) *reinterpret_cast<uint4*>(dst + 16) = make_uint4(p[4], p[5], p[6], p[7]);
  } else if (n == 8) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(p[0], p[1]);
  } else if (n == 4) {
    *reinterpret_cast<uint32_t*>(dst) = p[0];
  } else {
    for (int i = 0; i < n; ++i) dst[i] = (uint8_t)(p[i >> 2] >> (8 * (i & 3)));
  }
}

template <bool kBf16, int kMode, int kOut, int kR>
__global__ void __launch_bounds__(256, 2) col_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    unsigned int* __restrict__ amax_slot, void* __restrict__ out, int64_t out_ld,
    float* __restrict__ scale, int rnd, uint64_t seed, uint32_t stream,
    unsigned int* __restrict__ status) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr bool kHq = kOut == kColHqE4M3;
  constexpr int kBytes = kOut == kColBf16 ? 2 : 1;
  constexpr int R = kHq ? 16 : kR;  // codes per block per column
  constexpr int chunk = R * kBytes;   // bytes per block per column
  constexpr int row_stride = (kColBlocks + 1) * chunk;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t n_blk = rows >> 4;
  const int64_t c0 = (int64_t)blockIdx.x * kColCols + kCPT * tx;
  const int64_t b0 = (int64_t)blockIdx.y * kColBlocks;
  const bool col_ok = c0 < cols;

  float s = 0.0f;
  if (kMode == kQuant)
    s = __fdiv_rn(__uint_as_float(*amax_slot), kHq ? 7.0f : 127.0f);
  float amax = 0.0f;
  // both blocks of this thread are fetched before either is transformed
  RawPairCol<kBf16> raw[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int64_t b = b0 + ty + 8 * half;
    if (col_ok && b < n_blk) load_pair_col<kBf16>(src, 16 * b * cols + c0, cols, raw[half]);
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int bl = ty + 8 * half;
    const int64_t b = b0 + bl;
    if (!col_ok || b >= n_blk) continue;
    float v[kCPT][16];
    if constexpr (kBf16) {
      bool exact[2];
      pair_col_exact_bf16(raw[half].p, exact, status);
      unpack_pair_col<kBf16>(raw[half], v);
#pragma unroll
      for (int c = 0; c < kCPT; ++c) column_butterfly<kBf16>(v[c], exact[c], R, kHq);
    } else {
      unpack_pair_col<kBf16>(raw[half], v);
#pragma unroll
      for (int c = 0; c < kCPT; ++c) column_coeffs<kBf16>(v[c], R, kHq, status);
    }
    if (kMode == kAmax) {
#pragma unroll
      for (int c = 0; c < kCPT; ++c)
#pragma unroll
        for (int k = 0; k < 16; ++k)
          if (k < R) amax = fmaxf(amax, fabsf(v[c][k]));
      continue;
    }
    if (kHq) {
      // element (16b+i, c0+c) of the transformed [rows, cols] tensor; the
      // thread's columns lie in one Philox block of four (cols % 4 == 0)
      uint32_t w[kCPT][4];
#pragma unroll
      for (int c = 0; c < kCPT; ++c)
#pragma unroll
        for (int k = 0; k < 4; ++k) w[c][k] = 0u;
      const PhiloxKeys keys = philox_keys(seed);
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        float q[2][kCPT];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          U4 r = {0u, 0u, 0u, 0u};
          if (rnd == HLQ_SR)
            r = philox_block_k(keys, stream, (uint64_t)((16 * b + i + h) * cols + c0) >> 2);
          const bool hi = (c0 & 2) != 0;
          const uint32_t words[2] = {hi ? r.z : r.x, hi ? r.w : r.y};
#pragma unroll
          for (int c = 0; c < kCPT; ++c)
            q[h][c] = (rnd == HLQ_SR) ? quant_sr_f(v[c][i + h], s, words[c], 7.0f)
                                      : quant_rne_f(v[c][i + h], s, 7.0f);
        }
#pragma unroll
        for (int c = 0; c < kCPT; ++c)
          w[c][i >> 2] |= e4m3x2(q[0][c], q[1][c]) << (8 * (i & 3));
      }
#pragma unroll
      for (int c = 0; c < kCPT; ++c)
        *reinterpret_cast<uint4*>(smem + (size_t)(c * 32 + tx) * row_stride + bl * 16) =
            make_uint4(w[c][0], w[c][1], w[c][2], w[c][3]);
    } else {
#pragma unroll
      for (int c = 0; c < kCPT; ++c) {
        uint32_t p[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          if (k < R) {
            const int q = quant_rne(v[c][k], s, 127);
            if (kOut == kColBf16) {
              const uint32_t h = __bfloat16_as_ushort(__int2bfloat16_rn(q));
              p[k >> 1] |= h << (16 * (k & 1));
            } else {
              p[k >> 2] |= ((uint32_t)q & 0xffu) << (8 * (k & 3));
            }
          }
        }
        store_chunk(smem + (size_t)(c * 32 + tx) * row_stride + bl * chunk, p, chunk);
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
  const int64_t valid_b = imin64(kColBlocks, n_blk - b0);
  const int64_t seg_bytes = valid_b * chunk;
  const int64_t row_bytes = out_ld * kBytes;
  const int64_t off = b0 * chunk;
  const bool vec = (seg_bytes % 16 == 0) && (row_bytes % 16 == 0) && (off % 16 == 0) &&
                   (chunk % 16 == 0 || (kColBlocks * chunk) % 16 == 0);
  uint8_t* outb = static_cast<uint8_t*>(out);
  const int64_t col_base = (int64_t)blockIdx.x * kColCols;
  if (vec && chunk >= 16) {
    const int chunks = (int)(seg_bytes / 16);
    for (int idx = threadIdx.x; idx < kColCols * chunks; idx += blockDim.x) {
      const int r = idx / chunks, ch = idx % chunks;
      const int64_t c = col_base + col_tile_col(r);
      if (c < cols)
        *reinterpret_cast<uint4*>(outb + c * row_bytes + off + ch * 16) =
            *reinterpret_cast<const uint4*>(smem + (size_t)r * row_stride + ch * 16);
    }
  } else {
    for (int64_t idx = threadIdx.x; idx < (int64_t)kColCols * seg_bytes; idx += blockDim.x) {
      const int r = (int)(idx / seg_bytes);
      const int by = (int)(idx % seg_bytes);
      const int64_t c = col_base + col_tile_col(r);
      if (c < cols) outb[c * row_bytes + off + by] = smem[(size_t)r * row_stride + by];
    }
  }
}

// ---------------------------------------------------------------------------
// HQ of w [Cout, Cin] along Cout (blocks of 16 rows), codes written
// transposed [Cin, Cout].  w is small next to g_y, so the kernel trades
// redundant transforms for parallelism: thread (tx, ty) owns column pair tx
// (64 columns per CTA), block ty / 2 (4 blocks per CTA) and quantizes half
// of its 16 coefficients (ty % 2), drawing one Philox block per coefficient
// row for the pair.
// ---------------------------------------------------------------------------
constexpr int kWCols = 64;
constexpr int kWBlocks = 4;
constexpr int kWRowStride = kWBlocks * 16 + 8;  // bytes; 9 x 8-byte chunks

template <bool kBf16, int kMode>
__global__ void __launch_bounds__(256) hq_w_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    unsigned int* __restrict__ amax_slot, uint8_t* __restrict__ codes_t,
    float* __restrict__ scale, int rnd, uint64_t seed, uint32_t stream,
    unsigned int* __restrict__ status) {
  __shared__ __align__(16) uint8_t stage[kWCols * kWRowStride];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int bl = ty >> 1, part = ty & 1;
  const int64_t c0 = (int64_t)blockIdx.x * kWCols + 2 * tx;
  const int64_t b = (int64_t)blockIdx.y * kWBlocks + bl;
  const int64_t n_blk = rows >> 4;
  const bool ok = c0 < cols && b < n_blk;
  float v[2][16];
  if (ok) {
    RawPairCol<kBf16> raw;
    load_pair_col<kBf16>(src, 16 * b * cols + c0, cols, raw);
    if constexpr (kBf16) {
      bool exact[2];
      pair_col_exact_bf16(raw.p, exact, status);
      unpack_pair_col<kBf16>(raw, v);
      column_butterfly<kBf16>(v[0], exact[0], 16, true);
      column_butterfly<kBf16>(v[1], exact[1], 16, true);
    } else {
      unpack_pair_col<kBf16>(raw, v);
      column_coeffs<kBf16>(v[0], 16, true, status);
      column_coeffs<kBf16>(v[1], 16, true, status);
    }
  }
  if (kMode == kAmax) {
    float amax = 0.0f;
    if (ok && part == 0) {
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fmaxf(fabsf(v[0][i]), fabsf(v[1][i])));
    }
    amax = warp_max(amax);
    if (tx == 0) atomic_max_nonneg(amax_slot, amax);
    return;
  }
  const float s = __fdiv_rn(__uint_as_float(*amax_slot), 7.0f);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) scale[0] = s;
  if (ok) {
    const PhiloxKeys keys = philox_keys(seed);
    const bool hi = (c0 & 2) != 0;
    float h8[2][8];  // this thread's half of the coefficients (static indexing)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      h8[0][k] = part ? v[0][8 + k] : v[0][k];
      h8[1][k] = part ? v[1][8 + k] : v[1][k];
    }
    uint32_t w[2][2] = {{0u, 0u}, {0u, 0u}};
#pragma unroll
    for (int h = 0; h < 8; h += 2) {
      float q[2][2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = 8 * part + h + u;
        // element (16b+i, c0+c) of the transformed [rows, cols] tensor
        U4 r = {0u, 0u, 0u, 0u};
        if (rnd == HLQ_SR)
          r = philox_block_k(keys, stream, (uint64_t)((16 * b + i) * cols + c0) >> 2);
        const uint32_t w0 = hi ? r.z : r.x, w1 = hi ? r.w : r.y;
        const float y0 = h8[0][h + u], y1 = h8[1][h + u];
        q[u][0] = rnd == HLQ_SR ? quant_sr_f(y0, s, w0, 7.0f) : quant_rne_f(y0, s, 7.0f);
        q[u][1] = rnd == HLQ_SR ? quant_sr_f(y1, s, w1, 7.0f) : quant_rne_f(y1, s, 7.0f);
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) w[c][h >> 2] |= e4m3x2(q[0][c], q[1][c]) << (8 * (h & 3));
    }
#pragma unroll
    for (int c = 0; c < 2; ++c)
      *reinterpret_cast<uint2*>(stage + (c * 32 + tx) * kWRowStride + bl * 16 + part * 8) =
          make_uint2(w[c][0], w[c][1]);
  }
  __syncthreads();
  // row r of the stage = column tile_base + 2 * (r % 32) + r / 32; its
  // valid_b blocks of 16 codes go to codes_t[col, 16 * b0 ...]
  const int64_t b0 = (int64_t)blockIdx.y * kWBlocks;
  const int valid_b = (int)imin64(kWBlocks, n_blk - b0);
  const int chunks = valid_b * 2;  // 8-byte chunks per row
  for (int idx = threadIdx.x; idx < kWCols * chunks; idx += blockDim.x) {
    const int r = idx / chunks, ch = idx % chunks;
    const int64_t c = (int64_t)blockIdx.x * kWCols + 2 * (r & 31) + (r >> 5);
    if (c < cols)
      *reinterpret_cast<uint2*>(codes_t + c * rows + 16 * b0 + ch * 8) =
          *reinterpret_cast<const uint2*>(stage + r * kWRowStride + ch * 8);
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

// Column transforms alone: thread = 4 adjacent columns of one 16-row block;
// natural = all 16 Sylvester rows written [rows, cols]; else the `rank`
// sequency rows written [cols, rows/16*rank].
template <bool kBf16>
__global__ void __launch_bounds__(128) col_transform_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols, int rank, int natural,
    float* __restrict__ out, unsigned int* __restrict__ status) {
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
  const int64_t Tp = (rows >> 4) * rank;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    column_coeffs<kBf16>(v[c], natural ? 16 : rank, natural != 0, status);
    if (natural) {
#pragma unroll
      for (int i = 0; i < 16; ++i) out[(16 * b + i) * cols + cq * 4 + c] = v[c][i];
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (k < rank) out[(cq * 4 + c) * Tp + b * rank + k] = v[c][k];
    }
  }
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
  // per-token rows wait transformed (fp32) in shared memory between the two
  // passes when 8 of them fit in 160 KB (Cout <= 5120), else re-read
  const size_t row_bytes = (size_t)((cols / 8 + 31) / 32) * 64 * 16;
  const bool stage = per_token && !amax_only && row_bytes * warps <= 160 * 1024;
  const size_t smem = stage ? row_bytes * warps : 0;
#define HQR(B, M, P)                                                              \
  do {                                                                            \
    if (smem > 48 * 1024)                                                         \
      cudaFuncSetAttribute(hq_rows_kernel<B, M, P>,                               \
                           cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024); \
    hq_rows_kernel<B, M, P><<<grid, threads, smem, st>>>(                         \
        src, rows, cols, amax_slot, codes, scales, rnd, seed, stream_id, status,  \
        stage ? 1 : 0);                                                           \
  } while (0)
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

template <bool B, int M, int O, int R>
static cudaError_t launch_col_r(const void* src, int64_t rows, int64_t cols,
                                unsigned int* amax_slot, void* out, int64_t out_ld,
                                float* scale, int rnd, uint64_t seed, uint32_t stream_id,
                                unsigned int* status, cudaStream_t st) {
  constexpr int RR = O == kColHqE4M3 ? 16 : R;
  const size_t smem =
      M == kAmax ? 0 : (size_t)kColCols * (kColBlocks + 1) * RR * (O == kColBf16 ? 2 : 1);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(
        col_kernel<B, M, O, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(grid1(cols, kColCols), grid1(rows / 16, kColBlocks));
  col_kernel<B, M, O, R><<<grid, 256, smem, st>>>(src, rows, cols, amax_slot, out,
                                                  out_ld, scale, rnd, seed, stream_id,
                                                  status);
  return cudaGetLastError();
}

template <bool B, int M, int O>
static cudaError_t launch_col(const void* src, int64_t rows, int64_t cols, int rank,
                              unsigned int* amax_slot, void* out, int64_t out_ld,
                              float* scale, int rnd, uint64_t seed, uint32_t stream_id,
                              unsigned int* status, cudaStream_t st) {
#define LCR(R) \
  launch_col_r<B, M, O, R>(src, rows, cols, amax_slot, out, out_ld, scale, rnd, seed, \
                           stream_id, status, st)
  if constexpr (O == kColHqE4M3) {
    return LCR(16);
  } else {
    switch (rank) {
      case 1: return LCR(1);
      case 2: return LCR(2);
      case 4: return LCR(4);
      case 8: return LCR(8);
      default: return LCR(16);
    }
  }
#undef LCR
}

cudaError_t launch_hq_cols(const void* src, bool bf16, int64_t rows,
                           int64_t cols, bool amax_only,
                           unsigned int* amax_slot, uint8_t* codes_t,
                           float* scale, int rnd, uint64_t seed,
                           uint32_t stream_id, unsigned int* status,
                           cudaStream_t st) {
  dim3 grid(grid1(cols, kWCols), grid1(rows / 16, kWBlocks));
#define HQW(B, M)                                                                  \
  hq_w_kernel<B, M><<<grid, 256, 0, st>>>(src, rows, cols, amax_slot, codes_t, scale, \
                                          rnd, seed, stream_id, status)
  if (amax_only) {
    if (bf16) HQW(true, kAmax); else HQW(false, kAmax);
  } else {
    if (bf16) HQW(true, kQuant); else HQW(false, kQuant);
  }
#undef HQW
  return cudaGetLastError();
}

cudaError_t launch_hla(const void* src, bool bf16, int64_t T, int64_t C,
                       int rank, bool amax_only, bool out_bf16,
                       unsigned int* amax_slot, void* out, int64_t out_ld,
                       float* scale, unsigned int* status, cudaStream_t st) {
#define COL(B, M, O)                                                                  \
  launch_col<B, M, O>(src, T, C, rank, amax_slot, out, out_ld, scale, HLQ_RNE, 0, 0, \
                      status, st)
  if (amax_only) return bf16 ? COL(true, kAmax, kColI8) : COL(false, kAmax, kColI8);
  if (out_bf16) return bf16 ? COL(true, kQuant, kColBf16) : COL(false, kQuant, kColBf16);
  return bf16 ? COL(true, kQuant, kColI8) : COL(false, kQuant, kColI8);
#undef COL
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
  if (bf16) col_transform_kernel<true><<<grid, 128, 0, st>>>(src, rows, cols, 16, 1, Y, status);
  else col_transform_kernel<false><<<grid, 128, 0, st>>>(src, rows, cols, 16, 1, Y, status);
  return cudaGetLastError();
}

cudaError_t launch_hla_transform(const void* src, bool bf16, int64_t T,
                                 int64_t C, int rank, float* out,
                                 unsigned int* status, cudaStream_t st) {
  dim3 grid(grid1(C / 4, 128), (unsigned)(T / 16));
  if (bf16) col_transform_kernel<true><<<grid, 128, 0, st>>>(src, T, C, rank, 0, out, status);
  else col_transform_kernel<false><<<grid, 128, 0, st>>>(src, T, C, rank, 0, out, status);
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
