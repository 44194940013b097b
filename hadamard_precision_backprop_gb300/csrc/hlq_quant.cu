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
//  hq_w_kernel    : HQ of w [Cout, Cin] along Cout (blocks of 16 rows),
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
#include "hlq_tma.cuh"

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

// Butterfly of one octet (the lane pair 2p, 2p+1 holds one 16-block): the
// fp32 butterfly over lanes, across the pair with one shuffle stage.
__device__ __forceinline__ void octet_fwht(float* v) {
  // across the pair: lower lane v + o, upper lane o - v, as fma(v, +-1, o)
  // (exact product, one rounding: the same result), two lanes per fma
  const float sg = (threadIdx.x & 1) ? -1.0f : 1.0f;
  const unsigned long long sg2 = f2_pack(sg, sg);
  fwht8(v);
  float o[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) o[k] = __shfl_xor_sync(0xffffffffu, v[k], 1);
#pragma unroll
  for (int k = 0; k < 8; k += 2)
    f2_unpack(f2_fma(f2_pack(v[k], v[k + 1]), sg2, f2_pack(o[k], o[k + 1])), v[k], v[k + 1]);
}

// Exactly rounded transform of one octet in place.  tier (equal on both
// lanes of a pair): 0 = the fp32 butterfly is exact (exponent spread <= 12
// binades for bf16 inputs); 1 = split: values within 12 binades of the
// block's largest exponent `emax` and the rest are transformed separately
// (each part is exact) and the two exact results added with one rounding;
// 2 = out-of-line exact path.  All 32 lanes call this.
template <bool kBf16>
__device__ __forceinline__ void octet_butterfly(float* v, int tier, uint32_t emax) {
  const bool upper = (threadIdx.x & 1) != 0;
  // gather a slow block's 16 inputs first (shuffles stay warp-uniform)
  const bool any_slow = __any_sync(0xffffffffu, tier == 2);
  float full[16];
  if (any_slow) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float o = __shfl_xor_sync(0xffffffffu, v[k], 1);
      full[k] = upper ? o : v[k];
      full[8 + k] = upper ? v[k] : o;
    }
  }
  if (__any_sync(0xffffffffu, tier == 1)) {
    float lo[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t e = max((__float_as_uint(v[k]) >> 23) & 0xffu, 1u);
      const bool high = tier != 1 || e + 12u >= emax;
      lo[k] = high ? 0.0f : v[k];
      v[k] = high ? v[k] : 0.0f;
    }
    octet_fwht(v);
    octet_fwht(lo);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] += lo[k];  // exact + exact, one rounding
  } else {
    octet_fwht(v);
  }
  if (tier == 2) {
    float y[16];
    slow_block16(full, y, kBf16 ? 1 : 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = upper ? y[8 + k] : y[k];
  }
}

// Tier of a block from its exponent range (emax = largest exponent field,
// emin = smallest over non-zero values with subnormals as 1, all_zero).
__device__ __forceinline__ int block_tier_bf16(uint32_t emax, uint32_t emin, bool all_zero) {
  if (all_zero) return 0;
  if (emax == 255u) return 2;
  const uint32_t spread = emax - min(emin, emax);
  return spread <= 12u ? 0 : (spread <= 25u ? 1 : 2);
}

// Split of a column for tier 1: x -> (values within 12 binades of emax,
// the rest).
__device__ __forceinline__ void split_high_low(const float* x, uint32_t emax, float* hi,
                                               float* lo) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t e = max((__float_as_uint(x[j]) >> 23) & 0xffu, 1u);
    const bool high = e + 12u >= emax;
    hi[j] = high ? x[j] : 0.0f;
    lo[j] = high ? 0.0f : x[j];
  }
}

// Transform one octet in place (fp32 inputs: the butterfly is never exact
// for 24-bit significands, so blocks with values take the exact path).
template <bool kBf16>
__device__ __forceinline__ void transform_octet(float* v, unsigned int* status) {
  ExpRange er = exp_range_init();
#pragma unroll
  for (int k = 0; k < 8; ++k) exp_range_add(er, v[k]);
  er.emax = max(er.emax, __shfl_xor_sync(0xffffffffu, er.emax, 1));
  er.emin = min(er.emin, __shfl_xor_sync(0xffffffffu, er.emin, 1));
  if (any_nonfinite(er)) raise_flag(status, HLQ_DEV_NONFINITE);
  octet_butterfly<kBf16>(v, butterfly_exact<kBf16>(er) ? 0 : 2, er.emax);
}

// The same for eight packed bf16 values: the exponent range comes from
// 32-bit integer max/min over |bits| (zeros wrap to the largest value under
// "minus one" and drop out of the minimum), then the values unpack.
__device__ __forceinline__ void transform_octet_bf16(const uint4& raw, float* v,
                                                     unsigned int* status) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  // both 16-bit halves at once: |bits| max, and min of |bits| - 1 (mod 2^16)
  uint32_t hi2 = 0u, lom2 = 0xffffffffu;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t a = w[k] & 0x7fff7fffu;
    hi2 = u16x2_max(hi2, a);
    lom2 = u16x2_min(lom2, u16x2_add(a, 0xffffffffu));
  }
  uint32_t hi = max(hi2 & 0xffffu, hi2 >> 16);
  uint32_t lom1 = min(lom2 & 0xffffu, lom2 >> 16);  // 0xffff: all zero so far
  hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, 1));
  lom1 = min(lom1, __shfl_xor_sync(0xffffffffu, lom1, 1));
  const uint32_t emax = hi >> 7;
  if (emax == 255u) raise_flag(status, HLQ_DEV_NONFINITE);
  const bool all_zero = lom1 == 0xffffu;
  const uint32_t emin = max(((lom1 + 1u) & 0xffffu) >> 7, 1u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = bf16_lo(w[k]);
    v[2 * k + 1] = bf16_hi(w[k]);
  }
  octet_butterfly<true>(v, block_tier_bf16(emax, emin, all_zero), emax);
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

// Quantize one transformed octet (elements e0 .. e0+7 of `codes`) to E4M3
// int4 codes; the random words are those of elements e_off + e0 .. of the
// whole tensor.
// kNonZero: the caller has branched on s == 0 (all-zero codes) already.
template <bool kNonZero = false>
__device__ __forceinline__ void quantize_octet(const float* v, float s, int rnd,
                                               const PhiloxKeys& keys, uint32_t stream,
                                               int64_t e0, int64_t e_off, uint8_t* codes) {
  float r[8];
  if (rnd == HLQ_SR) {
    const uint64_t q = (uint64_t)(e_off + e0) >> 2;
    const U4 a = philox_block_k(keys, stream, q);
    const U4 b = philox_block_k(keys, stream, q + 1);
    const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k)
      r[k] = kNonZero ? quant_sr_nz(v[k], s, wd[k], 7.0f) : quant_sr_f(v[k], s, wd[k], 7.0f);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      r[k] = kNonZero ? quant_rne_nz(v[k], s, 7.0f) : quant_rne_f(v[k], s, 7.0f);
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
    float* __restrict__ scales, int rnd, const PhiloxKeys keys, uint32_t stream,
    unsigned int* __restrict__ status, int stage, int64_t e_off) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float4 srow[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int warps = blockDim.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * warps + wid;
  const int n_oct = (int)(cols >> 3);
  const int iters = (n_oct + 31) >> 5;
  const int64_t base = row * cols;
  if (kMode == kAmax) {  // per-tensor pre-pass: transform, max, one atomic per CTA
    float amax = 0.0f;
    if (row < rows) {  // warp-uniform
      RawOct<kBf16> cur = load_raw<kBf16>(src, base + lane * 8, lane < n_oct);
#pragma unroll 1
      for (int it = 0; it < iters; ++it) {
        const int nx = it * 32 + lane + 32;
        RawOct<kBf16> nxt = load_raw<kBf16>(src, base + (int64_t)nx * 8,
                                            it + 1 < iters && nx < n_oct);
        float v[8];
        transform_raw<kBf16>(cur, v, status);
#pragma unroll
        for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
        cur = nxt;
      }
    }
    cta_max_to_slot(amax, amax_slot);
    return;
  }
  if (row >= rows) return;  // whole warp leaves together
  // staged octet (it, lane): float4 halves at [(2*it + h) * 32 + lane]
  float4* my = srow + (size_t)wid * iters * 64;

  float amax = 0.0f;
  if (kPerToken) {
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
  } else {
    amax = __uint_as_float(ld_dep_u32(amax_slot));
  }
  const float s = __fdiv_rn(amax, 7.0f);
  if (lane == 0) {
    if (kPerToken) scales[row] = s;
    else if (row == 0) scales[0] = s;
  }
  __syncwarp();
  if (s == 0.0f) {  // warp-uniform: an all-zero row (or tensor) has all-zero codes
#pragma unroll 1
    for (int oct = lane; oct < n_oct; oct += 32)
      *reinterpret_cast<uint2*>(codes + base + (int64_t)oct * 8) = make_uint2(0u, 0u);
    return;
  }
  if (kPerToken && stage) {
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
      const int oct = it * 32 + lane;
      if (oct >= n_oct) break;
      const float4 a = my[(2 * it) * 32 + lane], b = my[(2 * it + 1) * 32 + lane];
      const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      quantize_octet<true>(v, s, rnd, keys, stream, base + (int64_t)oct * 8, e_off, codes);
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
    if (oct < n_oct)
      quantize_octet<true>(v, s, rnd, keys, stream, base + (int64_t)oct * 8, e_off, codes);
    cur = nxt;
  }
}

// ---------------------------------------------------------------------------
// Column transforms (the 16 values of a block lie in one column, 16 rows
// apart): helpers shared by the w and HLA kernels and the transform-only
// debug kernel.
// ---------------------------------------------------------------------------
enum ColOut { kColI8 = 1, kColF16 = 2, kColI4 = 3 };

// Code storage of an HLA output format: bytes per code as num / den (int4
// codes are packed two per byte, code 2k in the low nibble), and the
// symmetric code range.
template <int kOut>
struct ColFmt {
  static constexpr int kNum = kOut == kColF16 ? 2 : 1;
  static constexpr int kDen = kOut == kColI4 ? 2 : 1;
  static constexpr float kQmax = kOut == kColI4 ? 7.0f : 127.0f;
};

// Pack code k (an integer-valued float) of a column's block into p.
template <int kOut>
__device__ __forceinline__ void pack_code(uint32_t* p, int k, float q) {
  if (kOut == kColF16)
    p[k >> 1] |= (uint32_t)__half_as_ushort(__float2half_rn(q)) << (16 * (k & 1));
  else if (kOut == kColI4)
    p[k >> 3] |= ((uint32_t)(int)q & 0xfu) << (4 * (k & 7));
  else
    p[k >> 2] |= ((uint32_t)(int)q & 0xffu) << (8 * (k & 3));
}

// Store `n` bytes (1, 2, 4, 8, 16 or 32) of packed codes; dst is aligned to
// min(n, 16) bytes.  Every width is one typed store: a byte-by-byte copy of
// the 2-byte case (rank-1 bf16 codes) wrote wrong low bytes.
__device__ __forceinline__ void store_chunk(uint8_t* dst, const uint32_t* p, int n) {
  if (n >= 16) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(p[0], p[1], p[2], p[3]);
    if (n == 32) *reinterpret_cast<uint4*>(dst + 16) = make_uint4(p[4], p[5], p[6], p[7]);
  } else if (n == 8) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(p[0], p[1]);
  } else if (n == 4) {
    *reinterpret_cast<uint32_t*>(dst) = p[0];
  } else if (n == 2) {
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(p[0] & 0xffffu);
  } else {
    *dst = (uint8_t)(p[0] & 0xffu);
  }
}

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

// Exactly rounded coefficients of one 16-value column, in place, given its
// tier (0 fast, 1 split, 2 out-of-line exact; see octet_butterfly): the
// `rank` kept rows in sequency order in x[0..rank), or all 16 in Sylvester
// order when `natural`.
template <bool kBf16>
__device__ __forceinline__ void column_butterfly(float* x, int tier, uint32_t emax,
                                                 int rank, bool natural) {
  float t[16];
  if (tier == 0) {
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = x[j];
    fwht16(t);
  } else if (tier == 1) {
    float lo[16];
    split_high_low(x, emax, t, lo);
    fwht16(t);
    fwht16(lo);
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] += lo[j];  // exact + exact, one rounding
  } else {
    // rare: these two arrays live in local memory for the out-of-line call
    float in[16], o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) in[j] = x[j];
    slow_block16(in, o, kBf16 ? 1 : 0);
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = o[j];
  }
  if (natural) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = t[i];
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k)
      if (k < rank) x[k] = t[sequency_row(k)];
  }
}

template <bool kBf16>
__device__ __forceinline__ void column_coeffs(float* x, int rank, bool natural,
                                              unsigned int* status) {
  ExpRange er = exp_range_init();
#pragma unroll
  for (int j = 0; j < 16; ++j) exp_range_add(er, x[j]);
  if (any_nonfinite(er)) raise_flag(status, HLQ_DEV_NONFINITE);
  column_butterfly<kBf16>(x, butterfly_exact<kBf16>(er) ? 0 : 2, er.emax, rank, natural);
}

// Tiers (as in octet_butterfly) of the two columns of 16 packed bf16 pairs
// (low half = column 0), from the largest |bits| and the smallest non-zero
// |bits| of each column, kept in place in their half of the word (plain
// 32-bit integer max/min; a zero minus one wraps to the largest value and
// drops out of the minimum).
__device__ __forceinline__ void pair_col_tiers_bf16(const uint32_t (&p)[16], int* tier,
                                                    uint32_t* emax_out,
                                                    unsigned int* status) {
  // the two columns in the two 16-bit lanes: |bits| max, and min of
  // |bits| - 1 (mod 2^16, so a zero becomes 0xffff and drops out)
  uint32_t mx = 0u, mn = 0xffffffffu;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t a = p[j] & 0x7fff7fffu;
    mx = u16x2_max(mx, a);
    mn = u16x2_min(mn, u16x2_add(a, 0xffffffffu));
  }
  const uint32_t hi[2] = {mx & 0xffffu, mx >> 16};
  const uint32_t lo[2] = {((mn & 0xffffu) + 1u) & 0xffffu, ((mn >> 16) + 1u) & 0xffffu};
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t emax = hi[c] >> 7, emin = max(lo[c] >> 7, 1u);
    if (emax == 255u) raise_flag(status, HLQ_DEV_NONFINITE);
    tier[c] = block_tier_bf16(emax, emin, lo[c] == 0u);
    emax_out[c] = emax;
  }
}


// ---------------------------------------------------------------------------
// HLA along tokens (a1, a5, and their amax pre-pass).
//
// The Sylvester rows of sequency < R are H_R applied to sums over runs of
// L = 16/R consecutive tokens (H16[L*i][j] = H_R[i][j/L]), so coefficient k
// is Z[sigma(k)/L] with Z = H_R . (run sums): for R = 8 that is 8 pair sums
// and an 8-point butterfly instead of a 16-point one.  Both are stages of the
// 16-point butterfly, so the fp32 exactness rule applies unchanged; blocks
// that defeat it take the out-of-line exact path on all 16 inputs.
//
// Thread = 2 adjacent columns (one 4-byte bf16 pair per row); a warp holds
// 64 columns; each warp walks kHlaBW consecutive 16-token blocks with the
// next block's 16 loads in flight while the current one is transformed.
// CTA = 8 warps = 64 columns x 8*kHlaBW blocks; codes staged in shared
// memory leave as contiguous row segments of 8*kHlaBW*R codes.
// ---------------------------------------------------------------------------
constexpr int kHlaBW = 4;                 // blocks per warp
constexpr int kHlaBlocks = 8 * kHlaBW;    // blocks per CTA
constexpr int kHlaCols = 64;

// Column c (0: low, 1: high half of each pair) of a raw block, as fp32.
__device__ __forceinline__ float col_val(const RawPairCol<true>& r, int c, int j) {
  return c ? bf16_hi(r.p[j]) : bf16_lo(r.p[j]);
}
__device__ __forceinline__ float col_val(const RawPairCol<false>& r, int c, int j) {
  return c ? r.p[j].y : r.p[j].x;
}

template <int kR>
__device__ __forceinline__ void hla_fast(const float* x, float* coef) {
  constexpr int L = 16 / kR;
  float z[kR];
#pragma unroll
  for (int m = 0; m < kR; ++m) {
    float acc = x[m * L];
#pragma unroll
    for (int t = 1; t < L; ++t) acc += x[m * L + t];
    z[m] = acc;
  }
  // butterfly: the pair sums above are the first log2(L) stages; for the
  // remaining ones the order matches fwht16's on the full block
#pragma unroll
  for (int h = 1; h < kR; h <<= 1)
#pragma unroll
    for (int a = 0; a < kR; ++a)
      if ((a & h) == 0) {
        const float p = z[a], q = z[a + h];
        z[a] = p + q;
        z[a + h] = p - q;
      }
#pragma unroll
  for (int k = 0; k < kR; ++k) coef[k] = z[sequency_row(k) / L];
}

template <bool kBf16, int kMode, int kOut, int kR>
__global__ void __launch_bounds__(256, 2) hla_kernel(
    const void* __restrict__ src, int64_t T, int64_t C,
    unsigned int* __restrict__ amax_slot, void* __restrict__ out, int64_t out_ld,
    float* __restrict__ scale, unsigned int* __restrict__ status, int per_col) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) uint8_t smem[];
  using F = ColFmt<kOut>;
  constexpr int chunk = kR * F::kNum / F::kDen;           // bytes / block / column
  static_assert(chunk >= 1, "int4 codes need an even rank");
  constexpr int row_stride = (kHlaBlocks + 1) * chunk;    // odd number of chunks
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t n_blk = T >> 4;
  const int64_t c0 = (int64_t)blockIdx.x * kHlaCols + 2 * tx;
  const int64_t b_cta = (int64_t)blockIdx.y * kHlaBlocks;
  const int64_t b_first = b_cta + ty * kHlaBW;
  const bool col_ok = c0 < C;
  const int nb = col_ok ? (int)imin64(kHlaBW, n_blk - b_first) : 0;

  // scales: one for the tensor, or (per_col) one per column of the pair
  float sc[2] = {0.0f, 0.0f};
  if (kMode == kQuant) {
    if (!per_col) {
      sc[0] = sc[1] = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot)), F::kQmax);
    } else if (col_ok) {
      sc[0] = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot + c0)), F::kQmax);
      sc[1] = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot + c0 + 1)), F::kQmax);
      if (blockIdx.y == 0 && ty == 0) {
        scale[c0] = sc[0];
        scale[c0 + 1] = sc[1];
      }
    }
  }
  float am[2] = {0.0f, 0.0f};
  RawPairCol<kBf16> cur, nxt;
  if (nb > 0) load_pair_col<kBf16>(src, 16 * b_first * C + c0, C, cur);
#pragma unroll 1
  for (int i = 0; i < nb; ++i) {
    if (i + 1 < nb) load_pair_col<kBf16>(src, 16 * (b_first + i + 1) * C + c0, C, nxt);
    int tier[2];
    uint32_t emax[2];
    if constexpr (kBf16) {
      pair_col_tiers_bf16(cur.p, tier, emax, status);
    } else {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        ExpRange er = exp_range_init();
#pragma unroll
        for (int j = 0; j < 16; ++j) exp_range_add(er, col_val(cur, c, j));
        if (any_nonfinite(er)) raise_flag(status, HLQ_DEV_NONFINITE);
        tier[c] = butterfly_exact<false>(er) ? 0 : 2;
        emax[c] = er.emax;
      }
    }
    const int bl = ty * kHlaBW + i;  // block within the CTA tile
#pragma unroll
    for (int c = 0; c < 2; ++c) {  // one column at a time keeps few values live
      float coef[kR];
      float xv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) xv[j] = col_val(cur, c, j);
      if (tier[c] == 0) {
        hla_fast<kR>(xv, coef);
      } else if (tier[c] == 1) {
        float hi[16], lo[16], ch[kR];
        split_high_low(xv, emax[c], hi, lo);
        hla_fast<kR>(hi, coef);
        hla_fast<kR>(lo, ch);
#pragma unroll
        for (int k = 0; k < kR; ++k) coef[k] += ch[k];  // exact + exact, one rounding
      } else {
        float in[16], o[16];  // rare: local memory for the out-of-line call
#pragma unroll
        for (int j = 0; j < 16; ++j) in[j] = xv[j];
        slow_block16(in, o, kBf16 ? 1 : 0);
#pragma unroll
        for (int k = 0; k < kR; ++k) coef[k] = o[sequency_row(k)];
      }
      if (kMode == kAmax) {
#pragma unroll
        for (int k = 0; k < kR; ++k) am[c] = fmaxf(am[c], fabsf(coef[k]));
      } else {
        uint32_t p[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < kR; ++k)
          pack_code<kOut>(p, k, quant_rne_f(coef[k], sc[c], F::kQmax));
        store_chunk(smem + (size_t)(c * 32 + tx) * row_stride + bl * chunk, p, chunk);
      }
    }
    cur = nxt;
  }
  if (kMode == kAmax) {
    if (!per_col) {
      cta_max_to_slot(fmaxf(am[0], am[1]), amax_slot);
    } else if (nb > 0) {
      atomic_max_nonneg(&amax_slot[c0], am[0]);
      atomic_max_nonneg(&amax_slot[c0 + 1], am[1]);
    }
    return;
  }
  if (!per_col && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) scale[0] = sc[0];
  __syncthreads();
  // stage row r holds column tile_base + 2 * (r % 32) + r / 32
  const int64_t valid_b = imin64(kHlaBlocks, n_blk - b_cta);
  const int64_t seg_bytes = valid_b * chunk;
  const int64_t row_bytes = out_ld * F::kNum / F::kDen;
  const int64_t off = b_cta * chunk;
  uint8_t* outb = static_cast<uint8_t*>(out);
  const int64_t col_base = (int64_t)blockIdx.x * kHlaCols;
  // copy width: the widest that divides the shared row stride (so every
  // shared-memory row start is aligned), the segment, the output row
  // stride and the segment offset
  if (row_stride % 16 == 0 && seg_bytes % 16 == 0 && row_bytes % 16 == 0 && off % 16 == 0) {
    const int chunks = (int)(seg_bytes / 16);
    for (int idx = threadIdx.x; idx < kHlaCols * chunks; idx += blockDim.x) {
      const int r = idx / chunks, ch = idx % chunks;
      const int64_t c = col_base + 2 * (r & 31) + (r >> 5);
      if (c < C)
        *reinterpret_cast<uint4*>(outb + c * row_bytes + off + ch * 16) =
            *reinterpret_cast<const uint4*>(smem + (size_t)r * row_stride + ch * 16);
    }
  } else if (row_stride % 8 == 0 && seg_bytes % 8 == 0 && row_bytes % 8 == 0 &&
             off % 8 == 0) {
    const int chunks = (int)(seg_bytes / 8);
    for (int idx = threadIdx.x; idx < kHlaCols * chunks; idx += blockDim.x) {
      const int r = idx / chunks, ch = idx % chunks;
      const int64_t c = col_base + 2 * (r & 31) + (r >> 5);
      if (c < C)
        *reinterpret_cast<uint2*>(outb + c * row_bytes + off + ch * 8) =
            *reinterpret_cast<const uint2*>(smem + (size_t)r * row_stride + ch * 8);
    }
  } else {
    for (int64_t idx = threadIdx.x; idx < (int64_t)kHlaCols * seg_bytes; idx += blockDim.x) {
      const int r = (int)(idx / seg_bytes);
      const int by = (int)(idx % seg_bytes);
      const int64_t c = col_base + 2 * (r & 31) + (r >> 5);
      if (c < C) outb[c * row_bytes + off + by] = smem[(size_t)r * row_stride + by];
    }
  }
}

// ---------------------------------------------------------------------------
// HLA along the rows of src [rows, cols] (blocks of 16 consecutive values of
// a row; the ablation of the g_x path keeps the low-sequency Walsh rows of
// g_y along Cout): the exactly rounded 16-point transform of each block as
// in hq_rows_kernel (one warp per row, two lanes per block), the kR kept
// coefficients in sequency order, per-tensor amax (kAmax) or RNE int8 codes
// stored as bf16 [rows, out_ld] at column rank*b + k (kQuant).
// ---------------------------------------------------------------------------
template <bool kBf16, int kMode, int kR>
__global__ void __launch_bounds__(256) hla_rows_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    unsigned int* __restrict__ amax_slot, void* __restrict__ out, int64_t out_ld,
    float* __restrict__ scale, unsigned int* __restrict__ status) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int n_oct = (int)(cols >> 3);
  const int iters = (n_oct + 31) >> 5;
  float s = 0.0f;
  if (kMode == kQuant) s = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot)), 127.0f);
  float amax = 0.0f;
  if (row < rows) {  // warp-uniform: every lane of the warp reaches the shuffles
    const int64_t base = row * cols;
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
      const int oct = it * 32 + lane;
      const bool valid = oct < n_oct;
      const RawOct<kBf16> raw = load_raw<kBf16>(src, base + (int64_t)oct * 8, valid);
      float v[8];
      transform_raw<kBf16>(raw, v, status);  // v[k] = Y[8 * (lane & 1) + k]
      float y[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float o = __shfl_xor_sync(0xffffffffu, v[k], 1);
        y[k] = v[k];
        y[8 + k] = o;
      }
      if (valid && (lane & 1) == 0) {  // the lower lane of the pair owns the block
        if (kMode == kAmax) {
#pragma unroll
          for (int k = 0; k < kR; ++k) amax = fmaxf(amax, fabsf(y[sequency_row(k)]));
        } else {
          uint32_t p[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
          for (int k = 0; k < kR; ++k)
            pack_code<kColF16>(p, k, quant_rne_f(y[sequency_row(k)], s, 127.0f));
          const int64_t b = oct >> 1;
          store_chunk(static_cast<uint8_t*>(out) + (row * out_ld + b * kR) * 2, p, 2 * kR);
        }
      }
    }
  }
  if (kMode == kAmax) {
    cta_max_to_slot(amax, amax_slot);
  } else if (blockIdx.x == 0 && threadIdx.x == 0) {
    scale[0] = s;
  }
}

// ---------------------------------------------------------------------------
// HLA through TMA-staged tiles.  A CTA owns 256 columns x kTmaTiles
// consecutive 16-token blocks; thread 0 starts one TMA copy per block (box
// 16 rows x 256 columns) into its own shared-memory stage as soon as the
// barriers exist, so a CTA's whole input is in flight at once; its threads
// then take two columns each and process their blocks in order as they land,
// reading their 16 values per column out of shared memory (one 32-bit word
// per lane per row: conflict-free).  Thread (t, i) takes column pair t of
// the kTmaLoop consecutive blocks i * kTmaLoop .. (its code pieces of one
// row follow each other in memory).  Blocks per thread, measured on Llama
// down_proj (maximum pass, quant pass of the compression): one 118 + 172 us,
// two 103 + 154 us, four 97 + 154 us; ResNet-50 im2col 63 + 88, 56 + 78,
// 54 + 80 us; ViT-B qkv quant 14.2, 14.5, 15.9 us: up to four for the
// maximum pass and two for the quant pass, fewer when the grid would have
// less than two CTAs per SM (a 256-token layer: 17 -> 31 us of compression
// with four).
// ---------------------------------------------------------------------------
constexpr int kTmaCols = 256;
constexpr int kTmaBlocks = 1;  // thread groups of 128
template <int kMode>
struct TmaLoop {
  static constexpr int kMaxLoop = kMode == kAmax ? 4 : 2;  // consecutive blocks per thread
};

template <bool kBf16>
__device__ __forceinline__ void read_pair_col(const uint8_t* stage, int t,
                                              RawPairCol<kBf16>& r) {
  if constexpr (kBf16) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(stage);
#pragma unroll
    for (int j = 0; j < 16; ++j) r.p[j] = p[j * (kTmaCols / 2) + t];
  } else {
    const float2* p = reinterpret_cast<const float2*>(stage);
#pragma unroll
    for (int j = 0; j < 16; ++j) r.p[j] = p[j * (kTmaCols / 2) + t];
  }
}

template <bool kBf16, int kMode, int kOut, int kR>
__global__ void __launch_bounds__(128 * kTmaBlocks) hla_tma_kernel(
    const __grid_constant__ CUtensorMap tm, int64_t T, int64_t C,
    unsigned int* __restrict__ amax_slot, void* __restrict__ out, int64_t out_ld,
    float* __restrict__ scale, unsigned int* __restrict__ status, int per_col, int tok_fast,
    int tma_loop) {
  constexpr int kStage = 16 * kTmaCols * (kBf16 ? 2 : 4);
  using F = ColFmt<kOut>;
  constexpr int kChunk = kR * F::kNum / F::kDen;  // code bytes / block / column
  static_assert(kChunk >= 1, "int4 codes need an even rank");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  // tma_loop (1 .. kMaxLoop) consecutive blocks per thread, as many tiles
  // per CTA (the launch sized the shared memory for them)
  const int kTmaLoop = tma_loop, kTmaTiles = kTmaBlocks * tma_loop;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTmaTiles * kStage);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kTmaTiles);

  // thread (t, i): column pair t of blocks i * kTmaLoop .. of the tile
  const int t = threadIdx.x & 127, i = threadIdx.x >> 7;
  const int64_t n_blk = T >> 4;
  // tok_fast: token blocks along grid x, so that CTAs launched one after the
  // other write neighbouring pieces of the same code rows (whole 32-byte
  // sectors form in L2 before they are written back)
  const int64_t b0 = (int64_t)(tok_fast ? blockIdx.x : blockIdx.y) * kTmaTiles;
  const int nb = (int)imin64(kTmaTiles, n_blk - b0);
  const int64_t col0 = (int64_t)(tok_fast ? blockIdx.y : blockIdx.x) * kTmaCols;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int k = 0; k < kTmaTiles; ++k) mbar_init(&full[k], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_wait();  // the input and the amax slot come from earlier kernels
  if (threadIdx.x == 0) {
    for (int k = 0; k < nb; ++k) {
      mbar_expect_tx(&full[k], kStage);
      tma_load_2d(smem + k * kStage, &tm, &full[k], (int)col0, (int)(16 * (b0 + k)));
    }
  }
  __syncthreads();

  const int64_t c0 = col0 + 2 * t;
  const bool col_ok = c0 < C;
  // scales: one for the tensor, or (per_col) one per column of the pair
  float sc[2] = {0.0f, 0.0f};
  if (kMode == kQuant) {
    if (!per_col) {
      sc[0] = sc[1] = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot)), F::kQmax);
    } else if (col_ok) {
      sc[0] = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot + c0)), F::kQmax);
      sc[1] = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot + c0 + 1)), F::kQmax);
      if (b0 == 0 && i == 0) {  // the CTAs of the first token tile
        scale[c0] = sc[0];
        scale[c0 + 1] = sc[1];
      }
    }
  }
  float am[2] = {0.0f, 0.0f};
  uint8_t* outb = static_cast<uint8_t*>(out);
#pragma unroll 1
  for (int l = 0; l < kTmaLoop; ++l) {
    const int kb = i * kTmaLoop + l;  // stage (block of the tile)
    if (kb >= nb) break;
    if (!mbar_wait(&full[kb], 0u, abort_flag, status)) break;
    if (!col_ok) continue;
    RawPairCol<kBf16> cur;
    read_pair_col<kBf16>(smem + kb * kStage, t, cur);
    int tier[2];
    uint32_t emax[2];
    if constexpr (kBf16) {
      pair_col_tiers_bf16(cur.p, tier, emax, status);
    } else {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        ExpRange er = exp_range_init();
#pragma unroll
        for (int j = 0; j < 16; ++j) exp_range_add(er, col_val(cur, c, j));
        if (any_nonfinite(er)) raise_flag(status, HLQ_DEV_NONFINITE);
        tier[c] = butterfly_exact<false>(er) ? 0 : 2;
        emax[c] = er.emax;
      }
    }
    const int64_t b = b0 + kb;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float coef[kR];
      float xv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) xv[j] = col_val(cur, c, j);
      if (tier[c] == 0) {
        hla_fast<kR>(xv, coef);
      } else if (tier[c] == 1) {
        float hi[16], lo[16], ch[kR];
        split_high_low(xv, emax[c], hi, lo);
        hla_fast<kR>(hi, coef);
        hla_fast<kR>(lo, ch);
#pragma unroll
        for (int k = 0; k < kR; ++k) coef[k] += ch[k];  // exact + exact, one rounding
      } else {
        float in[16], o[16];  // rare: local memory for the out-of-line call
#pragma unroll
        for (int j = 0; j < 16; ++j) in[j] = xv[j];
        slow_block16(in, o, kBf16 ? 1 : 0);
#pragma unroll
        for (int k = 0; k < kR; ++k) coef[k] = o[sequency_row(k)];
      }
      if (kMode == kAmax) {
#pragma unroll
        for (int k = 0; k < kR; ++k) am[c] = fmaxf(am[c], fabsf(coef[k]));
      } else {
        uint32_t p[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < kR; ++k)
          pack_code<kOut>(p, k, quant_rne_f(coef[k], sc[c], F::kQmax));
        store_chunk(outb + ((c0 + c) * out_ld + b * kR) * F::kNum / F::kDen, p, kChunk);
      }
    }
  }
  if (threadIdx.x == 0 && *abort_flag) {  // let every copy land before exit
    for (int k = 0; k < nb; ++k) {
      const unsigned long long t0 = now_ns();
      while (!mbar_test(&full[k], 0u) && now_ns() - t0 < kWaitNs) {
      }
    }
  }
  if (kMode == kAmax) {
    if (!per_col) {
      cta_max_to_slot(fmaxf(am[0], am[1]), amax_slot);
    } else if (col_ok) {
      atomic_max_nonneg(&amax_slot[c0], am[0]);
      atomic_max_nonneg(&amax_slot[c0 + 1], am[1]);
    }
  } else if (!per_col && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    scale[0] = sc[0];
  }
}

// ---------------------------------------------------------------------------
// Fused reader of g_y [T, Cout] for both gradient paths: one 16-token x
// 256-column tile per CTA, loaded once by TMA, gives
//   - the HQ of the tile's 16 rows (16-value blocks along Cout, the exactly
//     rounded transform of hq_rows_kernel; thread t takes row t / 8 and the
//     two blocks at columns 32 * (t % 8) .. of the tile), and
//   - the HLA of its 256 columns (16-token blocks; thread t takes columns
//     2t, 2t + 1 as hla_tma_kernel does).
// kAmax: per-row (kPerToken, one atomicMax per row and tile into amax_rows)
// or per-tensor HQ maxima, and the HLA maximum.  kQuant: E4M3 int4 codes of
// the HQ (Philox SR stream 0, element t * Cout + c) with per-row or tensor
// scales, and the HLA int8 codes as bf16 [Cout, hla_ld].  The two passes
// replace the HQ kernel and the two HLA kernels: two reads of g_y instead
// of three, and no transformed row staged in shared memory.
// ---------------------------------------------------------------------------
template <bool kBf16, int kR>
__device__ __forceinline__ void hla_pair_col_coefs(const RawPairCol<kBf16>& cur, int c, int tier,
                                                   uint32_t emax, float (&coef)[kR]) {
  float xv[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) xv[j] = col_val(cur, c, j);
  if (tier == 0) {
    hla_fast<kR>(xv, coef);
  } else if (tier == 1) {
    float hi[16], lo[16], ch[kR];
    split_high_low(xv, emax, hi, lo);
    hla_fast<kR>(hi, coef);
    hla_fast<kR>(lo, ch);
#pragma unroll
    for (int k = 0; k < kR; ++k) coef[k] += ch[k];  // exact + exact, one rounding
  } else {
    float in[16], o[16];  // rare: local memory for the out-of-line call
#pragma unroll
    for (int j = 0; j < 16; ++j) in[j] = xv[j];
    slow_block16(in, o, kBf16 ? 1 : 0);
#pragma unroll
    for (int k = 0; k < kR; ++k) coef[k] = o[sequency_row(k)];
  }
}

template <bool kBf16>
__device__ __forceinline__ void pair_tiers(const RawPairCol<kBf16>& cur, int (&tier)[2],
                                           uint32_t (&emax)[2], unsigned int* status) {
  if constexpr (kBf16) {
    pair_col_tiers_bf16(cur.p, tier, emax, status);
  } else {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      ExpRange er = exp_range_init();
#pragma unroll
      for (int j = 0; j < 16; ++j) exp_range_add(er, col_val(cur, c, j));
      if (any_nonfinite(er)) raise_flag(status, HLQ_DEV_NONFINITE);
      tier[c] = butterfly_exact<false>(er) ? 0 : 2;
      emax[c] = er.emax;
    }
  }
}

// The 32 consecutive values of one tile row starting at column x0, as the
// "pair" form of two 16-value blocks (low half / .x = block at x0, high
// half / .y = block at x0 + 16), value j of each block in word j.
template <bool kBf16>
__device__ __forceinline__ void read_row_blocks(const uint8_t* stage, int row, int x0,
                                                RawPairCol<kBf16>& r) {
  if constexpr (kBf16) {
    const uint4* q = reinterpret_cast<const uint4*>(stage + (row * kTmaCols + x0) * 2);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a = q[i];
      w[4 * i] = a.x; w[4 * i + 1] = a.y; w[4 * i + 2] = a.z; w[4 * i + 3] = a.w;
    }
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      r.p[j] = __byte_perm(w[j / 2], w[8 + j / 2], 0x5410);      // even columns
      r.p[j + 1] = __byte_perm(w[j / 2], w[8 + j / 2], 0x7632);  // odd columns
    }
  } else {
    const float4* q = reinterpret_cast<const float4*>(stage + (row * kTmaCols + x0) * 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 a = q[i], b = q[4 + i];
      r.p[4 * i] = make_float2(a.x, b.x);
      r.p[4 * i + 1] = make_float2(a.y, b.y);
      r.p[4 * i + 2] = make_float2(a.z, b.z);
      r.p[4 * i + 3] = make_float2(a.w, b.w);
    }
  }
}

constexpr int kFusedTiles = 2;  // 16-token tiles per CTA of the fused reader

template <bool kBf16, int kMode, bool kPerToken, int kR>
__global__ void __launch_bounds__(128) gy_fused_kernel(
    const __grid_constant__ CUtensorMap tm, int64_t T, int64_t C,
    unsigned int* __restrict__ hq_amax, unsigned int* __restrict__ hla_amax,
    uint8_t* __restrict__ qy, float* __restrict__ sgy, void* __restrict__ qg,
    int64_t hla_ld, float* __restrict__ sg, int rnd, const PhiloxKeys keys,
    unsigned int* __restrict__ status, int tiles) {
  // tiles (1 .. 2): consecutive 16-token tiles of the same 256 columns per
  // CTA, all loaded at once, processed in order
  constexpr int kStage = 16 * kTmaCols * (kBf16 ? 2 : 4);
  using F = ColFmt<kColF16>;
  constexpr int kChunk = kR * 2;  // fp16 code bytes per block and column
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + tiles * kStage);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + tiles);
  __shared__ float partial[2][4];

  const int t = threadIdx.x;
  const int64_t n_cc = (C + kTmaCols - 1) / kTmaCols;
  const int64_t n_blk = T >> 4;
  const int64_t u = blockIdx.x;
  const int64_t col0 = (u % n_cc) * kTmaCols, b0 = (u / n_cc) * tiles;
  const int nb = (int)imin64(tiles, n_blk - b0);
  pdl_trigger();
  if (t == 0) {
    for (int k = 0; k < tiles; ++k) mbar_init(&full[k], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_wait();  // g_y and the amax slots come from earlier work
  if (t == 0) {
    for (int k = 0; k < nb; ++k) {
      mbar_expect_tx(&full[k], kStage);
      tma_load_2d(smem + k * kStage, &tm, &full[k], (int)col0, (int)(16 * (b0 + k)));
    }
  }
  __syncthreads();
  const int hq_row = t >> 3;                  // 0..15
  const int x0 = 32 * (t & 7);                // first column of the pair of blocks
  float s_hla = 0.0f;
  if (kMode == kQuant) s_hla = __fdiv_rn(__uint_as_float(ld_dep_u32(hla_amax)), F::kQmax);
  float am_hla = 0.0f, am_hq = 0.0f;
  const int64_t c0 = col0 + 2 * t;
  const int64_t cb = col0 + x0;
  const bool blk_ok[2] = {cb < C, cb + 16 < C};
  bool live = true;
#pragma unroll 1
  for (int l = 0; l < nb && live; ++l) {
    const int64_t b = b0 + l;
    const int64_t tok = 16 * b + hq_row;
    float s_hq = 0.0f;
    if (kMode == kQuant)
      s_hq = __fdiv_rn(__uint_as_float(ld_dep_u32(kPerToken ? hq_amax + tok : hq_amax)), 7.0f);
    live = mbar_wait(&full[l], 0u, abort_flag, status);
    const uint8_t* stage = smem + l * kStage;
    float am_row = 0.0f;  // this tile's HQ maximum of the thread's row part
    // ---- HLA: column pair t ----
    if (live && c0 < C) {
      RawPairCol<kBf16> cur;
      read_pair_col<kBf16>(stage, t, cur);
      int tier[2];
      uint32_t emax[2];
      pair_tiers<kBf16>(cur, tier, emax, status);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float coef[kR];
        hla_pair_col_coefs<kBf16, kR>(cur, c, tier[c], emax[c], coef);
        if (kMode == kAmax) {
#pragma unroll
          for (int k = 0; k < kR; ++k) am_hla = fmaxf(am_hla, fabsf(coef[k]));
        } else {
          uint32_t p[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
          for (int k = 0; k < kR; ++k)
            pack_code<kColF16>(p, k, quant_rne_f(coef[k], s_hla, F::kQmax));
          store_chunk(static_cast<uint8_t*>(qg) + ((c0 + c) * hla_ld + b * kR) * 2, p, kChunk);
        }
      }
    }
    // ---- HQ: row hq_row, blocks at columns x0 and x0 + 16 of the tile ----
    if (live && blk_ok[0]) {
      RawPairCol<kBf16> cur;
      read_row_blocks<kBf16>(stage, hq_row, x0, cur);
      int tier[2];
      uint32_t emax[2];
      pair_tiers<kBf16>(cur, tier, emax, status);
      float v[2][16];
      unpack_pair_col<kBf16>(cur, v);
      column_butterfly<kBf16>(v[0], tier[0], emax[0], 16, true);
      column_butterfly<kBf16>(v[1], tier[1], emax[1], 16, true);
      if (kMode == kAmax) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          am_row = fmaxf(am_row, fabsf(v[0][i]));
          if (blk_ok[1]) am_row = fmaxf(am_row, fabsf(v[1][i]));
        }
      } else {
        const int64_t e = tok * C + cb;
        quantize_octet(v[0], s_hq, rnd, keys, 0u, e, 0, qy);
        quantize_octet(v[0] + 8, s_hq, rnd, keys, 0u, e + 8, 0, qy);
        if (blk_ok[1]) {
          quantize_octet(v[1], s_hq, rnd, keys, 0u, e + 16, 0, qy);
          quantize_octet(v[1] + 8, s_hq, rnd, keys, 0u, e + 24, 0, qy);
        }
      }
    }
    if (kMode == kAmax) {
      if (kPerToken) {  // the 8 threads of a row are consecutive lanes
        am_row = fmaxf(am_row, __shfl_xor_sync(0xffffffffu, am_row, 1));
        am_row = fmaxf(am_row, __shfl_xor_sync(0xffffffffu, am_row, 2));
        am_row = fmaxf(am_row, __shfl_xor_sync(0xffffffffu, am_row, 4));
        if ((t & 7) == 0 && tok < T) atomic_max_nonneg(hq_amax + tok, am_row);
      } else {
        am_hq = fmaxf(am_hq, am_row);
      }
    } else if (kPerToken && col0 == 0 && (t & 7) == 0 && tok < T) {
      sgy[tok] = s_hq;
    }
    live = __all_sync(0xffffffffu, live);  // warp-uniform for the shuffles above
  }
  if (t == 0 && *abort_flag) {  // let the copies land before exit
    for (int k = 0; k < nb; ++k) {
      const unsigned long long t0 = now_ns();
      while (!mbar_test(&full[k], 0u) && now_ns() - t0 < kWaitNs) {
      }
    }
  }
  if (kMode == kAmax) {
    am_hla = warp_max(am_hla);
    if (!kPerToken) am_hq = warp_max(am_hq);
    if ((t & 31) == 0) {
      partial[0][t >> 5] = am_hla;
      partial[1][t >> 5] = am_hq;
    }
    __syncthreads();
    if (t == 0) {
      atomic_max_nonneg(hla_amax, fmaxf(fmaxf(partial[0][0], partial[0][1]),
                                        fmaxf(partial[0][2], partial[0][3])));
      if (!kPerToken)
        atomic_max_nonneg(hq_amax, fmaxf(fmaxf(partial[1][0], partial[1][1]),
                                         fmaxf(partial[1][2], partial[1][3])));
    }
  } else if (u == 0 && t == 0) {
    sg[0] = s_hla;
    if (!kPerToken)
      sgy[0] = __fdiv_rn(__uint_as_float(ld_dep_u32(hq_amax)), 7.0f);
  }
}

// ---------------------------------------------------------------------------
// HQ of w [Cout, Cin] along Cout (blocks of 16 rows), codes written
// transposed [Cin, Cout] (also the along-token HQ of the g_w ablation, with
// rows = tokens).  Thread = (column quad, 16-row block): it loads the 16 x 4
// values (8 or 16 bytes per row; consecutive threads take consecutive quads,
// so a warp reads 256 or 512 contiguous bytes per row), transforms the four
// columns, and quantizes coefficient row i of the quad with the one Philox
// block that covers elements (16b + i) * cols + 4q .. + 3; each column's 16
// codes leave as one 16-byte store into its row of the transposed output.
// ---------------------------------------------------------------------------
template <bool kBf16>
struct RawQuad;
template <>
struct RawQuad<true> {
  RawPairCol<true> lo, hi;  // columns 0, 1 and 2, 3
};
template <>
struct RawQuad<false> {
  RawPairCol<false> lo, hi;
};

template <bool kBf16>
__device__ __forceinline__ void load_quad_col(const void* src, int64_t idx, int64_t ld,
                                              RawQuad<kBf16>& r) {
  if constexpr (kBf16) {
    const uint16_t* p = static_cast<const uint16_t*>(src) + idx;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(p + j * ld));
      r.lo.p[j] = w.x;
      r.hi.p[j] = w.y;
    }
  } else {
    const float* p = static_cast<const float*>(src) + idx;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float4 w = __ldg(reinterpret_cast<const float4*>(p + j * ld));
      r.lo.p[j] = make_float2(w.x, w.y);
      r.hi.p[j] = make_float2(w.z, w.w);
    }
  }
}

// All 16 exactly rounded coefficients (Sylvester order) of the two columns
// of a pair, given their tiers.
template <bool kBf16>
__device__ __forceinline__ void pair_full_coefs(const RawPairCol<kBf16>& r, float (*v)[16],
                                                unsigned int* status) {
  if constexpr (kBf16) {
    int tier[2];
    uint32_t emax[2];
    pair_col_tiers_bf16(r.p, tier, emax, status);
    unpack_pair_col<kBf16>(r, v);
    column_butterfly<kBf16>(v[0], tier[0], emax[0], 16, true);
    column_butterfly<kBf16>(v[1], tier[1], emax[1], 16, true);
  } else {
    unpack_pair_col<kBf16>(r, v);
    column_coeffs<kBf16>(v[0], 16, true, status);
    column_coeffs<kBf16>(v[1], 16, true, status);
  }
}

template <bool kBf16, int kMode>
__global__ void __launch_bounds__(128) hq_w_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    unsigned int* __restrict__ amax_slot, uint8_t* __restrict__ codes_t,
    float* __restrict__ scale, int rnd, const PhiloxKeys keys, uint32_t stream,
    unsigned int* __restrict__ status) {
  pdl_trigger();
  pdl_wait();
  const int64_t n_q = cols >> 2, n_blk = rows >> 4;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool ok = idx < n_q * n_blk;
  const int64_t q = ok ? idx % n_q : 0, b = ok ? idx / n_q : 0;
  float v[4][16];
  if (ok) {
    RawQuad<kBf16> raw;
    load_quad_col<kBf16>(src, 16 * b * cols + 4 * q, cols, raw);
    pair_full_coefs<kBf16>(raw.lo, v, status);
    pair_full_coefs<kBf16>(raw.hi, v + 2, status);
  }
  if (kMode == kAmax) {
    float amax = 0.0f;
    if (ok) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[c][i]));
    }
    cta_max_to_slot(amax, amax_slot);
    return;
  }
  const float s = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot)), 7.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) scale[0] = s;
  if (!ok) return;
  uint32_t w[4][4] = {};  // column c's 16 code bytes (code i in byte i)
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    float qv[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      // elements (16b + i + u) * cols + 4q + c of the transformed tensor
      const uint64_t e = (uint64_t)((16 * b + i + u) * cols + 4 * q);
      U4 r = {0u, 0u, 0u, 0u};
      if (rnd == HLQ_SR) r = philox_block_k(keys, stream, e >> 2);
      const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        qv[u][c] = rnd == HLQ_SR ? quant_sr_f(v[c][i + u], s, wd[c], 7.0f)
                                 : quant_rne_f(v[c][i + u], s, 7.0f);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
      w[c][i >> 2] |= e4m3x2(qv[0][c], qv[1][c]) << (16 * ((i >> 1) & 1));
  }
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(codes_t + (4 * q + c) * rows + 16 * b) =
        make_uint4(w[c][0], w[c][1], w[c][2], w[c][3]);
}

// The same HQ with two threads per column pair and block (each transforms
// the pair and quantizes half of its 16 rows, drawing a Philox block per
// row for the pair): twice the transforms and random words of the quad
// kernel, but eight times its threads, which is what a small tensor (the w
// of a ViT-B layer) needs to fill the GPU: thread (tx, ty) owns column pair
// tx (64 columns per CTA) and block ty / 2 (4 blocks per CTA); the
// transposed codes leave through shared memory in 8-byte chunks.
constexpr int kWCols = 64;
constexpr int kWBlocks = 4;
constexpr int kWRowStride = kWBlocks * 16 + 8;  // bytes; 9 x 8-byte chunks

template <bool kBf16, int kMode>
__global__ void __launch_bounds__(256) hq_w_pair_kernel(
    const void* __restrict__ src, int64_t rows, int64_t cols,
    unsigned int* __restrict__ amax_slot, uint8_t* __restrict__ codes_t,
    float* __restrict__ scale, int rnd, const PhiloxKeys keys, uint32_t stream,
    unsigned int* __restrict__ status) {
  pdl_trigger();
  pdl_wait();
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
      int tier[2];
      uint32_t emax[2];
      pair_col_tiers_bf16(raw.p, tier, emax, status);
      unpack_pair_col<kBf16>(raw, v);
      column_butterfly<kBf16>(v[0], tier[0], emax[0], 16, true);
      column_butterfly<kBf16>(v[1], tier[1], emax[1], 16, true);
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
    cta_max_to_slot(amax, amax_slot);
    return;
  }
  const float s = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot)), 7.0f);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) scale[0] = s;
  if (ok) {
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
// Quantization error of the int4 HQ of g_y with RNE codes, per tensor and
// per token at once (layer-wise quantizer selection): one warp per row; the
// row's transformed values give its amax (per-token scale), then a second
// transform of the row (it is still in L1/L2) gives both errors
// (q * s - Y)^2, exact differences in fp64, summed per warp and added into
// sums[0] (per tensor, scale from *amax_slot) and sums[1] (per token).
// Squared quantization errors of one quantizer, accumulated without fp64
// arithmetic per element (GB300's fp64 rate is a small fraction of its fp32
// rate): with s scaled by 2^-E (E its exponent, so the scaled errors sit
// near 1 and no square underflows) and the element by the same power of
// two (exact), the error q s - y is the exact pair
//   (RN(q s) - y) + (q s - RN(q s)),
// the first difference exact by Sterbenz's lemma (q != 0 means y / s rounds
// to q, so y and q s are within a factor of two; q == 0 gives -y), the
// second the product's exact rounding error from one fused multiply-add.
// Its square is a^2 (split exactly by another FMA) + 2 a b (rounded: a
// correction ~2^-22 of a^2), the tiny b^2 dropped; the running sum is a
// double-float pair updated with an exact two-sum.  About 46 significant
// bits in all: the sums agree with an fp64 evaluation (exact differences,
// rounded squares and sums) to far better than 1e-9 relative.
struct ErrSum {
  float hi = 0.0f, lo = 0.0f;
  __device__ __forceinline__ void add_sq(float q, float s_scaled, float y_scaled) {
    const float p = q * s_scaled;
    const float pe = fmaf(q, s_scaled, -p);   // q s - RN(q s), exact
    const float a = p - y_scaled;             // exact (Sterbenz)
    const float sq = a * a;
    const float sq_e = fmaf(a, a, -sq);       // a^2 - RN(a^2), exact
    const float t = hi + sq;                  // two-sum of hi and sq
    const float bv = t - hi;
    const float err = (hi - (t - bv)) + (sq - bv);
    hi = t;
    lo += err + sq_e + 2.0f * a * pe;
  }
};

// 2^-E for the scale's exponent E, clamped to [-100, 100] (0 for s == 0)
__device__ __forceinline__ int scale_exp(float s) {
  if (!(s > 0.0f)) return 0;
  const int e = (int)((__float_as_uint(s) >> 23) & 0xffu) - 127;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}

template <bool kBf16>
__global__ void __launch_bounds__(256) hq_mse_kernel(const void* __restrict__ src,
                                                     int64_t rows, int64_t cols,
                                                     const unsigned int* __restrict__ amax_slot,
                                                     double* __restrict__ sums,
                                                     unsigned int* __restrict__ status) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;  // whole warp leaves together
  const int n_oct = (int)(cols >> 3);
  const int iters = (n_oct + 31) >> 5;
  const int64_t base = row * cols;
  float amax = 0.0f;
  for (int it = 0; it < iters; ++it) {
    const int oct = it * 32 + lane;
    float v[8];
    transform_raw<kBf16>(load_raw<kBf16>(src, base + (int64_t)oct * 8, oct < n_oct), v, status);
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
  }
  amax = warp_max(amax);
  const float st = __fdiv_rn(amax, 7.0f);
  const float sg = __fdiv_rn(__uint_as_float(ld_dep_u32(amax_slot)), 7.0f);
  const int et = scale_exp(st), eg = scale_exp(sg);
  const float pt = ldexpf(1.0f, -et), pg = ldexpf(1.0f, -eg);
  const float st_s = st * pt, sg_s = sg * pg;
  ErrSum at, ag;
  for (int it = 0; it < iters; ++it) {
    const int oct = it * 32 + lane;
    float v[8];
    transform_raw<kBf16>(load_raw<kBf16>(src, base + (int64_t)oct * 8, oct < n_oct), v, status);
    if (oct >= n_oct) continue;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      at.add_sq(quant_rne_f(v[k], st, 7.0f), st_s, v[k] * pt);
      ag.add_sq(quant_rne_f(v[k], sg, 7.0f), sg_s, v[k] * pg);
    }
  }
  double et_sum = ldexp((double)at.hi + (double)at.lo, 2 * et);
  double eg_sum = ldexp((double)ag.hi + (double)ag.lo, 2 * eg);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    et_sum += __shfl_xor_sync(0xffffffffu, et_sum, o);
    eg_sum += __shfl_xor_sync(0xffffffffu, eg_sum, o);
  }
  if (lane == 0) {
    atomicAdd(&sums[0], eg_sum);
    atomicAdd(&sums[1], et_sum);
  }
}

// mse[g] = sums[g] / n; choice = per-token iff mse[0] > threshold * mse[1].
__global__ void lqs_finalize_kernel(const double* __restrict__ sums, int64_t n,
                                    double threshold, double* __restrict__ mse,
                                    int32_t* __restrict__ choice) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const double mt = n > 0 ? ld_dep_f64(sums) / (double)n : 0.0;
  const double mk = n > 0 ? ld_dep_f64(sums + 1) / (double)n : 0.0;
  mse[0] = mt;
  mse[1] = mk;
  *choice = mt > threshold * mk ? HLQ_PER_TOKEN : HLQ_PER_TENSOR;
}


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
// int8 codes [rows, cols] -> fp16 codes [rows, out_ld]; kWidenCodes codes per
// thread (cols a multiple of kWidenCodes on the vector path).  Llama
// down_proj x-bar (117 MB in, 235 MB out): 8 codes per thread 67.5 us,
// 16 codes 69.5 us, 32 codes 82.1 us.
constexpr int kWidenCodes = 8;
__global__ void widen_i8_to_f16_kernel(const int8_t* __restrict__ in,
                                       __half* __restrict__ out,
                                       int64_t rows, int64_t cols,
                                       int64_t out_ld) {
  pdl_trigger();
  pdl_wait();
  const int64_t per_row = (cols + kWidenCodes - 1) / kWidenCodes;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * per_row) return;
  const int64_t r = idx / per_row, c = (idx % per_row) * kWidenCodes;
  const int8_t* src = in + r * cols + c;
  __half* dst = out + r * out_ld + c;
  if (c + kWidenCodes <= cols && (cols % kWidenCodes) == 0) {
#pragma unroll
    for (int h = 0; h < kWidenCodes / 8; ++h) {
      uint2 v = ld_dep_u2(src + 8 * h);
      const int8_t* b = reinterpret_cast<const int8_t*>(&v);
      __align__(16) __half o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = __int2half_rn(b[k]);
      *reinterpret_cast<uint4*>(dst + 8 * h) = *reinterpret_cast<const uint4*>(o);
    }
  } else {
    for (int k = 0; k < kWidenCodes && c + k < cols; ++k)
      dst[k] = __int2half_rn((int8_t)ld_dep_u8(src + k));
  }
}

__global__ void decode_e4m3_kernel(const uint8_t* __restrict__ in,
                                   int8_t* __restrict__ out, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (int8_t)int_of_e4m3(in[i]);
}

// E4M3 code bytes (integers in [-7, 7]) to packed int4: byte i holds codes
// 2i (low nibble) and 2i + 1 (high nibble), two's complement.
__global__ void pack_e4m3_int4_kernel(const uint8_t* __restrict__ in,
                                      uint8_t* __restrict__ out, int64_t n_bytes) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_bytes;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t lo = (uint32_t)int_of_e4m3(in[2 * i]) & 0xfu;
    const uint32_t hi = (uint32_t)int_of_e4m3(in[2 * i + 1]) & 0xfu;
    out[i] = (uint8_t)(lo | (hi << 4));
  }
}

__global__ void decode_f16_kernel(const __half* __restrict__ in,
                                   int8_t* __restrict__ out, int64_t rows,
                                   int64_t cols, int64_t ld) {
  const int64_t n = rows * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (int8_t)__half2int_rn(in[(i / cols) * ld + i % cols]);
}

// Device status word of this library (HLQ_DEV_* flags): every kernel that
// can detect a device-side condition takes its address.
__device__ unsigned int g_status_word;

cudaError_t status_word_address(unsigned int** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
  *out = static_cast<unsigned int*>(p);
  return e;
}

// ---------------------------------------------------------------------------
// Host-side launchers.
// ---------------------------------------------------------------------------
// Raise a kernel's dynamic shared-memory limit once per device (the call is
// not free, and launches come in the microseconds).
// (one cache per kernel: the kernel is a template argument)
template <auto kKernel>
static cudaError_t ensure_smem_limit(size_t bytes) {
  static int done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev] >= (int)bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kKernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done[dev] = (int)bytes;
  return e;
}

static inline unsigned grid1(int64_t n, int per) {
  return (unsigned)((n + per - 1) / per);
}

cudaError_t launch_hq_rows(const void* src, bool bf16, int64_t rows,
                           int64_t cols, bool per_token, bool amax_only,
                           unsigned int* amax_slot, uint8_t* codes,
                           float* scales, int rnd, uint64_t seed,
                           uint32_t stream_id, unsigned int* status,
                           cudaStream_t st, int64_t row0) {
  if (rows == 0) return cudaSuccess;
  const int threads = 256, warps = threads / 32;
  dim3 grid(grid1(rows, warps));
  // per-token rows wait transformed (fp32) in shared memory between the two
  // passes when the staging leaves room for three CTAs (24 warps) per SM
  // (Cout <= 2304: 72 KB per CTA); longer rows are read again (from L1/L2,
  // right after the first pass) and transformed again instead: with one
  // CTA of 8 staged 4096-value rows per SM (128 KB) the Llama-shaped HQ of
  // g_y took 236 us, issue-bound at 8 warps per SM
  const size_t row_bytes = (size_t)((cols / 8 + 31) / 32) * 64 * 16;
  const bool stage = per_token && !amax_only && row_bytes * warps <= 74 * 1024;
  const size_t smem = stage ? row_bytes * warps : 0;
#define HQR(B, M, P)                                                              \
  do {                                                                            \
    if (smem > 48 * 1024 &&                                                       \
        ensure_smem_limit<hq_rows_kernel<B, M, P>>(160 * 1024) != cudaSuccess)    \
      return cudaGetLastError();                                                  \
    launch_pdl(hq_rows_kernel<B, M, P>, grid, dim3(threads), smem, st, src, rows,  \
               cols, amax_slot, codes, scales, rnd, philox_keys(seed), stream_id, status,       \
               stage ? 1 : 0, row0 * cols);                                       \
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

cudaError_t launch_hla_rows(const void* src, bool bf16, int64_t rows, int64_t cols,
                            int rank, bool amax_only, unsigned int* amax_slot, void* out,
                            int64_t out_ld, float* scale, unsigned int* status,
                            cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const dim3 grid(grid1(rows, 8));
#define HLR(B, M, R)                                                                   \
  launch_pdl(hla_rows_kernel<B, M, R>, grid, dim3(256), 0, st, src, rows, cols, amax_slot, \
             out, out_ld, scale, status)
#define HLR_RANK(B, M)                 \
  switch (rank) {                      \
    case 1: HLR(B, M, 1); break;       \
    case 2: HLR(B, M, 2); break;       \
    case 4: HLR(B, M, 4); break;       \
    case 8: HLR(B, M, 8); break;       \
    case 16: HLR(B, M, 16); break;     \
    default: return cudaErrorInvalidValue; \
  }
  if (amax_only) {
    if (bf16) { HLR_RANK(true, kAmax) } else { HLR_RANK(false, kAmax) }
  } else {
    if (bf16) { HLR_RANK(true, kQuant) } else { HLR_RANK(false, kQuant) }
  }
#undef HLR_RANK
#undef HLR
  return cudaGetLastError();
}

cudaError_t launch_hq_mse(const void* src, bool bf16, int64_t rows, int64_t cols,
                          const unsigned int* amax_slot, double* sums, double threshold,
                          double* mse, int32_t* choice, unsigned int* status,
                          cudaStream_t st) {
  if (rows > 0) {
    if (bf16)
      launch_pdl(hq_mse_kernel<true>, dim3(grid1(rows, 8)), dim3(256), 0, st, src, rows,
                 cols, amax_slot, sums, status);
    else
      launch_pdl(hq_mse_kernel<false>, dim3(grid1(rows, 8)), dim3(256), 0, st, src, rows,
                 cols, amax_slot, sums, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  launch_pdl(lqs_finalize_kernel, dim3(1), dim3(32), 0, st, (const double*)sums,
             rows * cols, threshold, mse, choice);
  return cudaGetLastError();
}

cudaError_t launch_hq_cols(const void* src, bool bf16, int64_t rows,
                           int64_t cols, bool amax_only,
                           unsigned int* amax_slot, uint8_t* codes_t,
                           float* scale, int rnd, uint64_t seed,
                           uint32_t stream_id, unsigned int* status,
                           cudaStream_t st) {
  const int64_t threads = (cols / 4) * (rows / 16);
  if (threads == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  // quad kernel when it has at least 4 CTAs of 128 threads per SM, else the
  // pair kernel's 8x more threads (ViT-B qkv w: 14.7 us pair, 18.7 us quad;
  // Llama down_proj w: 219 us pair, 152 us quad; one thread per column pair
  // with the quad's random words shared by shuffles measured 146 us against
  // the quad kernel's 134 us there)
  if (threads >= (int64_t)sms * 4 * 128) {
    const dim3 grid(grid1(threads, 128));
#define HQW(B, M)                                                                   \
  launch_pdl(hq_w_kernel<B, M>, grid, dim3(128), 0, st, src, rows, cols, amax_slot, \
             codes_t, scale, rnd, philox_keys(seed), stream_id, status)
    if (amax_only) {
      if (bf16) HQW(true, kAmax); else HQW(false, kAmax);
    } else {
      if (bf16) HQW(true, kQuant); else HQW(false, kQuant);
    }
#undef HQW
  } else {
    const dim3 grid(grid1(cols, kWCols), grid1(rows / 16, kWBlocks));
#define HQP(B, M)                                                                        \
  launch_pdl(hq_w_pair_kernel<B, M>, grid, dim3(256), 0, st, src, rows, cols, amax_slot, \
             codes_t, scale, rnd, philox_keys(seed), stream_id, status)
    if (amax_only) {
      if (bf16) HQP(true, kAmax); else HQP(false, kAmax);
    } else {
      if (bf16) HQP(true, kQuant); else HQP(false, kQuant);
    }
#undef HQP
  }
  return cudaGetLastError();
}

template <bool B, int M, int O, int R>
static cudaError_t launch_hla_r(const void* src, int64_t T, int64_t C,
                                unsigned int* amax_slot, void* out, int64_t out_ld,
                                float* scale, unsigned int* status, int per_col,
                                cudaStream_t st) {
  // TMA-staged path: chunk stores of R codes need R-code-aligned rows
  using F = ColFmt<O>;
  const int chunk = R * F::kNum / F::kDen;
  const bool chunk_ok = (chunk == 1 || chunk == 2 || chunk % 4 == 0) &&
                        (out_ld * F::kNum / F::kDen) % (chunk >= 16 ? 16 : chunk) == 0;
  CUtensorMap tm;
  if (chunk_ok && make_tile_map_2d(&tm, src, B, T, C, kTmaCols, 16)) {
    // blocks per thread: the mode's maximum, halved while the grid would
    // have fewer than two CTAs per SM
    static int sms_of[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!sms_of[dev] &&
        cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorInvalidDevice;
    int loop = TmaLoop<M>::kMaxLoop;
    while (loop > 1 && (int64_t)grid1(T / 16, kTmaBlocks * loop) * grid1(C, kTmaCols) <
                           2 * (int64_t)sms_of[dev])
      loop /= 2;
    const int kTmaTiles = kTmaBlocks * loop;
    const size_t smem = 128 + (size_t)kTmaTiles * 16 * kTmaCols * (B ? 2 : 4) +
                        kTmaTiles * 8 + 16;
    cudaError_t e = ensure_smem_limit<hla_tma_kernel<B, M, O, R>>(smem);
    if (e != cudaSuccess) return e;
    const int64_t col_tiles = grid1(C, kTmaCols), tok_tiles = grid1(T / 16, kTmaTiles);
    const int tok_fast = col_tiles <= 65535 ? 1 : 0;  // grid y limit
    const dim3 grid = tok_fast ? dim3((unsigned)tok_tiles, (unsigned)col_tiles)
                               : dim3((unsigned)col_tiles, (unsigned)tok_tiles);
    launch_pdl(hla_tma_kernel<B, M, O, R>, grid, dim3(128 * kTmaBlocks), smem, st, tm, T,
               C, amax_slot, out, out_ld, scale, status, per_col, tok_fast, loop);
    return cudaGetLastError();
  }
  const size_t smem = M == kAmax ? 0 : (size_t)kHlaCols * (kHlaBlocks + 1) * chunk;
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_smem_limit<hla_kernel<B, M, O, R>>(smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(grid1(C, kHlaCols), grid1(T / 16, kHlaBlocks));
  launch_pdl(hla_kernel<B, M, O, R>, grid, dim3(256), smem, st, src, T, C, amax_slot, out, out_ld,
             scale, status, per_col);
  return cudaGetLastError();
}

template <bool B, int M, int O>
static cudaError_t launch_hla_o(const void* src, int64_t T, int64_t C, int rank,
                                unsigned int* amax_slot, void* out, int64_t out_ld,
                                float* scale, unsigned int* status, int per_col,
                                cudaStream_t st) {
#define LHR(R) \
  launch_hla_r<B, M, O, R>(src, T, C, amax_slot, out, out_ld, scale, status, per_col, st)
  if constexpr (O == kColI4) {  // two codes per byte: even ranks only
    switch (rank) {
      case 2: return LHR(2);
      case 4: return LHR(4);
      case 8: return LHR(8);
      case 16: return LHR(16);
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (rank) {
      case 1: return LHR(1);
      case 2: return LHR(2);
      case 4: return LHR(4);
      case 8: return LHR(8);
      default: return LHR(16);
    }
  }
#undef LHR
}

cudaError_t launch_hla(const void* src, bool bf16, int64_t T, int64_t C,
                       int rank, bool amax_only, int out_fmt,
                       unsigned int* amax_slot, void* out, int64_t out_ld,
                       float* scale, unsigned int* status, cudaStream_t st, bool per_col) {
  const int pc = per_col ? 1 : 0;
#define LHO(B, M, O) \
  launch_hla_o<B, M, O>(src, T, C, rank, amax_slot, out, out_ld, scale, status, pc, st)
  if (amax_only) return bf16 ? LHO(true, kAmax, kColI8) : LHO(false, kAmax, kColI8);
  if (out_fmt == kHlaOutF16)
    return bf16 ? LHO(true, kQuant, kColF16) : LHO(false, kQuant, kColF16);
  if (out_fmt == kHlaOutI4) return bf16 ? LHO(true, kQuant, kColI4) : LHO(false, kQuant, kColI4);
  return bf16 ? LHO(true, kQuant, kColI8) : LHO(false, kQuant, kColI8);
#undef LHO
}

cudaError_t launch_gy_fused(const void* gy, bool bf16, int64_t T, int64_t C, int rank,
                            bool per_token, bool amax_only, unsigned int* hq_amax,
                            unsigned int* hla_amax, uint8_t* qy, float* sgy, void* qg,
                            int64_t hla_ld, float* sg, int rnd, uint64_t seed,
                            unsigned int* status, cudaStream_t st) {
  if (T == 0 || C == 0) return cudaSuccess;
  CUtensorMap tm;
  if (!make_tile_map_2d(&tm, gy, bf16, T, C, kTmaCols, 16)) return cudaErrorInvalidValue;
  // two 16-token tiles per CTA, one when that would leave fewer than two CTAs
  // per SM (as for the HLA kernel)
  static int sms_of[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!sms_of[dev] &&
      cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  const int64_t n_cc = grid1(C, kTmaCols);
  int per_cta = kFusedTiles;
  while (per_cta > 1 && n_cc * grid1(T / 16, per_cta) < 2 * (int64_t)sms_of[dev]) per_cta /= 2;
  const size_t smem = 128 + (size_t)per_cta * (16 * kTmaCols * (bf16 ? 2 : 4) + 8) + 16;
  const int64_t tiles = n_cc * grid1(T / 16, per_cta);
#define GYF(B, M, P, R)                                                                  \
  do {                                                                                   \
    cudaError_t e = ensure_smem_limit<gy_fused_kernel<B, M, P, R>>(smem);                \
    if (e != cudaSuccess) return e;                                                      \
    launch_pdl(gy_fused_kernel<B, M, P, R>, dim3((unsigned)tiles), dim3(128), smem, st, tm, \
               T, C, hq_amax, hla_amax, qy, sgy, qg, hla_ld, sg, rnd, philox_keys(seed), status, \
               per_cta);                                                                 \
  } while (0)
#define GYF_R(B, M, P)                         \
  switch (rank) {                              \
    case 1: GYF(B, M, P, 1); break;            \
    case 2: GYF(B, M, P, 2); break;            \
    case 4: GYF(B, M, P, 4); break;            \
    case 8: GYF(B, M, P, 8); break;            \
    case 16: GYF(B, M, P, 16); break;          \
    default: return cudaErrorInvalidValue;     \
  }
#define GYF_P(B, M)                            \
  if (per_token) {                             \
    GYF_R(B, M, true)                          \
  } else {                                     \
    GYF_R(B, M, false)                         \
  }
  if (amax_only) {
    if (bf16) { GYF_P(true, kAmax) } else { GYF_P(false, kAmax) }
  } else {
    if (bf16) { GYF_P(true, kQuant) } else { GYF_P(false, kQuant) }
  }
#undef GYF_P
#undef GYF_R
#undef GYF
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

// Packed int4 codes [rows, cols/2 bytes] (code 2k in the low nibble) to
// fp16 rows with stride out_ld; 8 codes per thread.
__global__ void widen_i4_to_f16_kernel(const uint8_t* __restrict__ in,
                                       __half* __restrict__ out, int64_t rows,
                                        int64_t cols, int64_t out_ld) {
  pdl_trigger();
  pdl_wait();
  const int64_t per_row = (cols + 7) / 8;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * per_row) return;
  const int64_t r = idx / per_row, c = (idx % per_row) * 8;
  const uint8_t* src = in + (r * cols + c) / 2;
  __half* dst = out + r * out_ld + c;
  auto code = [&](int k) {  // sign-extended nibble k of the run
    const int v = (ld_dep_u8(src + (k >> 1)) >> (4 * (k & 1))) & 0xf;
    return v >= 8 ? v - 16 : v;
  };
  if (c + 8 <= cols && (cols % 8) == 0) {
    const uint32_t w = ld_dep_u32(reinterpret_cast<const unsigned int*>(src));
    __align__(16) __half o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int v = (int)((w >> (4 * k)) & 0xfu);
      o[k] = __int2half_rn(v >= 8 ? v - 16 : v);
    }
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(o);
  } else {
    for (int k = 0; k < 8 && c + k < cols; ++k) dst[k] = __int2half_rn(code(k));
  }
}

cudaError_t launch_widen_i4_f16(const uint8_t* in, void* out, int64_t rows, int64_t cols,
                                 int64_t out_ld, cudaStream_t st) {
  if (rows * cols == 0) return cudaSuccess;
  const int64_t n = rows * ((cols + 7) / 8);
  launch_pdl(widen_i4_to_f16_kernel, dim3(grid1(n, 256)), dim3(256), 0, st, in,
             static_cast<__half*>(out), rows, cols, out_ld);
  return cudaGetLastError();
}

cudaError_t launch_widen_i8_f16(const int8_t* in, void* out, int64_t rows,
                                 int64_t cols, int64_t out_ld, cudaStream_t st) {
  if (rows * cols == 0) return cudaSuccess;
  const int64_t n = rows * ((cols + kWidenCodes - 1) / kWidenCodes);
  launch_pdl(widen_i8_to_f16_kernel, dim3(grid1(n, 256)), dim3(256), 0, st, in,
             static_cast<__half*>(out), rows, cols, out_ld);
  return cudaGetLastError();
}

// A bounded wait that runs out: one CTA waits on an mbarrier that nothing
// arrives at, gives up after limit_ns, raises HLQ_DEV_TIMEOUT and returns
// (the failure path of every pipeline wait, exercised without a fault).
__global__ void wait_timeout_probe_kernel(unsigned long long limit_ns, int32_t* result,
                                          unsigned int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool ok = mbar_wait_for(&bar, 0u, &abort_flag, status, limit_ns);
  __syncthreads();
  if (threadIdx.x == 0) *result = ok ? 1 : 0;
}

cudaError_t launch_wait_timeout_probe(unsigned long long limit_ns, int32_t* result,
                                      unsigned int* status, cudaStream_t st) {
  wait_timeout_probe_kernel<<<1, 32, 0, st>>>(limit_ns, result, status);
  return cudaGetLastError();
}

cudaError_t launch_pack_e4m3_int4(const uint8_t* in, uint8_t* out, int64_t n,
                                  cudaStream_t st) {
  const int64_t nb = n / 2;
  if (nb == 0) return cudaSuccess;
  pack_e4m3_int4_kernel<<<(unsigned)imin64(grid1(nb, 256), 4096), 256, 0, st>>>(in, out, nb);
  return cudaGetLastError();
}

cudaError_t launch_decode_e4m3(const uint8_t* in, int8_t* out, int64_t n,
                               cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  decode_e4m3_kernel<<<(unsigned)imin64(grid1(n, 256), 4096), 256, 0, st>>>(in, out, n);
  return cudaGetLastError();
}

cudaError_t launch_decode_f16(const void* in, int8_t* out, int64_t rows,
                               int64_t cols, int64_t ld, cudaStream_t st) {
  const int64_t n = rows * cols;
  if (n == 0) return cudaSuccess;
  decode_f16_kernel<<<(unsigned)imin64(grid1(n, 256), 4096), 256, 0, st>>>(
      static_cast<const __half*>(in), out, rows, cols, ld);
  return cudaGetLastError();
}

}  // namespace hlq
