// hlq_device.cuh -- device building blocks shared by the HLQ kernels:
// input decoding, the exact 16-point Hadamard sums, Philox4x32-10, the
// int4/int8 quantizers and the device status word.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "hlq.h"

namespace hlq {

// Programmatic dependent launch: the hot kernels are launched with the
// programmatic-serialization attribute (launch_pdl), let the next kernel in
// the stream start launching at once (pdl_trigger), and wait for the
// previous kernel's completion and memory (pdl_wait) before they touch
// global memory.  Both are no-ops for a kernel launched without the
// attribute.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Reads of what an earlier kernel of the stream wrote (amax slots, scales,
// sums, stored codes).  Under programmatic dependent launch a kernel runs
// while its predecessor may still be writing, and only pdl_wait() orders it
// after those writes.  The read-only data path (ld.global.nc, which __ldg and
// loads through const __restrict__ pointers may use) is valid only for data
// that nothing writes during the kernel's lifetime, so these reads are
// ordinary coherent loads, written as volatile asm so that they stay after
// the wait.
__device__ __forceinline__ unsigned int ld_dep_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float ld_dep_f32(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ double ld_dep_f64(const double* p) {
  double v;
  asm volatile("ld.relaxed.gpu.global.f64 %0, [%1];" : "=d"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_dep_u2(const void* p) {
  uint2 v;
  asm volatile("ld.relaxed.gpu.global.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint8_t ld_dep_u8(const void* p) {
  unsigned short v;
  asm volatile("ld.relaxed.gpu.global.u8 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
  return (uint8_t)v;
}

template <typename... Exp, typename... Act>
static cudaError_t launch_pdl(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

// Device status word (HLQ_DEV_* flags): every kernel that can detect a
// device-side condition takes its address; hlq_read_device_status reads it.
__device__ __forceinline__ void raise_flag(unsigned int* status, unsigned int f) {
  atomicOr(status, f);
}

// ---------------------------------------------------------------------------
// Input decoding.  bf16 is the top half of an fp32, so widening is exact.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t pair) {
  return __uint_as_float(pair << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t pair) {
  return __uint_as_float(pair & 0xffff0000u);
}

// ---------------------------------------------------------------------------
// Exactness test for the fp32 butterfly.
//
// A 16-point Hadamard sum of values whose largest exponent field is emax and
// whose smallest (non-zero, subnormals counted as field 1) is emin needs
// emax - emin + 24 + 4 bits for fp32 inputs (24-bit significands) and
// emax - emin + 8 + 4 bits for bf16 inputs (8-bit significands).  When that fits in fp32's 24-bit
// significand, every partial sum of the butterfly is exact, so the result is
// the exact sum whatever the order, i.e. the once-rounded value.
// We track, per value, (field, field_for_min) with zeros mapped to
// (0, 255) so that they drop out of both extremes.
// ---------------------------------------------------------------------------
struct ExpRange {
  uint32_t emax;  // max exponent field
  uint32_t emin;  // min exponent field over non-zero values (>= 1)
};

__device__ __forceinline__ void exp_range_add(ExpRange& r, float v) {
  uint32_t b = __float_as_uint(v) & 0x7fffffffu;
  uint32_t e = b >> 23;
  uint32_t emn = (b == 0u) ? 255u : max(e, 1u);
  r.emax = max(r.emax, e);
  r.emin = min(r.emin, emn);
}

__device__ __forceinline__ ExpRange exp_range_init() { return {0u, 255u}; }

// bf16 inputs: exact when emax - emin <= 12; fp32 inputs never qualify.
template <bool kBf16>
__device__ __forceinline__ bool butterfly_exact(const ExpRange& r) {
  if (r.emin == 255u) return true;  // all zero
  if (!kBf16) return false;
  return r.emax - r.emin <= 12u;
}

__device__ __forceinline__ bool any_nonfinite(const ExpRange& r) {
  return r.emax == 255u;
}

// ---------------------------------------------------------------------------
// Exact signed sum of 16 fp32 values, rounded once to fp32 (nearest, ties to
// even).  Fallback for blocks whose exponent spread defeats the fp32
// butterfly.  Each finite fp32 is m * 2^(p - 149) with m < 2^24, p >= 0;
// the sum is held as a signed 320-bit two's-complement integer in units of
// 2^-149 spread over ten 32-bit digits carried in int64 (signed digits, one
// carry pass at the end), then rounded by direct construction of the fp32
// bit pattern.  `neg_mask` bit j negates term j.
// ---------------------------------------------------------------------------
static __device__ __noinline__ float exact_sum16(const float* v, uint32_t neg_mask) {
  long long d[10];
#pragma unroll
  for (int i = 0; i < 10; ++i) d[i] = 0;
  for (int j = 0; j < 16; ++j) {
    uint32_t b = __float_as_uint(v[j]);
    uint32_t e = (b >> 23) & 0xffu;
    uint32_t m = b & 0x7fffffu;
    if (e == 255u) continue;  // non-finite: flagged elsewhere
    if (e != 0u) m |= 0x800000u;
    if (m == 0u) continue;
    int p = (e != 0u) ? int(e) - 1 : 0;
    unsigned long long w = (unsigned long long)m << (p & 31);
    long long lo = (long long)(w & 0xffffffffull), hi = (long long)(w >> 32);
    int li = p >> 5;
    bool neg = ((b >> 31) ^ ((neg_mask >> j) & 1u)) != 0u;
    if (neg) {
      d[li] -= lo;
      d[li + 1] -= hi;
    } else {
      d[li] += lo;
      d[li + 1] += hi;
    }
  }
  // carry pass: digits 0..8 end in [0, 2^32); digit 9 keeps the sign
  for (int i = 0; i < 9; ++i) {
    long long c = d[i] >> 32;  // arithmetic shift: floor division
    d[i] -= c * 4294967296ll;
    d[i + 1] += c;
  }
  bool negative = d[9] < 0;
  uint32_t u[10];
  if (negative) {  // magnitude = two's complement of the 320-bit value
    unsigned long long carry = 1;
    for (int i = 0; i < 10; ++i) {
      unsigned long long t =
          (unsigned long long)(~(uint32_t)(d[i] & 0xffffffffll)) + carry;
      u[i] = (uint32_t)t;
      carry = t >> 32;
    }
  } else {
    for (int i = 0; i < 10; ++i) u[i] = (uint32_t)d[i];
  }
  int top = -1;
  for (int i = 9; i >= 0; --i)
    if (u[i] != 0u) {
      top = i * 32 + 31 - __clz(u[i]);
      break;
    }
  if (top < 0) return 0.0f;
  uint32_t bits;
  if (top <= 23) {
    bits = u[0];  // m * 2^-149 with m < 2^24 is its own fp32 bit pattern
  } else {
    int shift = top - 23;
    int k = shift >> 5, r = shift & 31;
    unsigned long long win =
        (unsigned long long)u[k] | ((unsigned long long)u[k + 1] << 32);
    uint32_t keep = (uint32_t)(win >> r) & 0xffffffu;  // r + 24 <= 56 bits
    // round bit (shift-1) and sticky bits (below shift-1)
    int rb = shift - 1;
    uint32_t round_bit = (u[rb >> 5] >> (rb & 31)) & 1u;
    bool sticky = (u[rb >> 5] & ((1u << (rb & 31)) - 1u)) != 0u;
    for (int i = 0; i < (rb >> 5); ++i) sticky |= (u[i] != 0u);
    if (round_bit && (sticky || (keep & 1u))) ++keep;
    if (keep == (1u << 24)) {
      keep >>= 1;
      ++shift;
    }
    bits = ((uint32_t)shift << 23) + keep;  // exponent field shift+1
  }
  return __uint_as_float(bits | (negative ? 0x80000000u : 0u));
}

// Exact 16-point Hadamard transform of v in 64-bit fixed point: every value
// is m * 2^(p-150) (m its 24-bit significand, p its exponent field, >= 1),
// so with pmin the smallest p of the non-zero values, n_j = m_j << (p_j - pmin)
// are integers and y_i = sum_j H[i][j] n_j * 2^(pmin-150) exactly.  bf16
// inputs have 16 zero low significand bits, which are dropped first.  The
// sums fit in int64 when the exponent spread is at most 51 (bf16) or 35
// (fp32) binades; each y_i is then rounded once by the int64 -> fp32
// conversion and rescaled by an exponent shift.  Returns false (y is then
// garbage) when the spread is larger or a result would be subnormal.
template <bool kBf16>
__device__ __forceinline__ bool fwht16_fixed(const float* v, float* y) {
  constexpr int kDrop = kBf16 ? 16 : 0;
  constexpr int kMaxSpread = kBf16 ? 51 : 35;
  int pmin = 255, pmax = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t b = __float_as_uint(v[j]) & 0x7fffffffu;
    if (b != 0u) {
      const int p = max((int)(b >> 23), 1);
      pmin = min(pmin, p);
      pmax = max(pmax, p);
    }
  }
  if (pmax == 0) {
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = 0.0f;
    return true;
  }
  if (pmax - pmin > kMaxSpread) return false;
  long long n[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t b = __float_as_uint(v[j]);
    const uint32_t e = (b >> 23) & 0xffu;
    uint32_t m = b & 0x7fffffu;
    if (e != 0u) m |= 0x800000u;
    long long mag = 0;
    if (m != 0u) mag = (long long)(m >> kDrop) << (max((int)e, 1) - pmin);
    n[j] = (b >> 31) ? -mag : mag;
  }
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)
#pragma unroll
    for (int a = 0; a < 16; ++a)
      if ((a & h) == 0) {
        const long long p = n[a], q = n[a + h];
        n[a] = p + q;
        n[a + h] = p - q;
      }
  const int L = pmin - 150 + kDrop;  // y_i = n_i * 2^L
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (n[i] == 0) {
      y[i] = 0.0f;
    } else {
      const uint32_t fb = __float_as_uint(__ll2float_rn(n[i]));
      const int E = (int)((fb >> 23) & 0xffu) + L;
      ok &= (E >= 1);
      y[i] = __uint_as_float(fb + ((uint32_t)L << 23));
    }
  }
  return ok;
}

// Sylvester H16 row i as a negate mask: bit j set when popcount(i & j) odd.
__device__ __forceinline__ uint32_t hrow_negmask(int i) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) m |= (uint32_t)(__popc(i & j) & 1) << j;
  return m;
}

// In-place 16-point fast Walsh-Hadamard transform in Sylvester (natural)
// order: y_i = sum_j (-1)^popcount(i&j) x_j.
__device__ __forceinline__ void fwht16(float* x) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)
#pragma unroll
    for (int a = 0; a < 16; ++a)
      if ((a & h) == 0) {
        float p = x[a], q = x[a + h];
        x[a] = p + q;
        x[a + h] = p - q;
      }
}

// Two 16-bit unsigned lanes in one 32-bit register: lane-wise max, min and
// modular add (sm_90+ packed integer instructions).
__device__ __forceinline__ uint32_t u16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t u16x2_min(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t u16x2_add(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two fp32 lanes in one 64-bit register, and the packed IEEE add, subtract
// and fused multiply-add of sm_100+ (each lane rounded to nearest exactly as
// the scalar instruction rounds it).
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// 8-point butterfly (the three within-octet stages of a 16-point one).  The
// stages at distance 2 and 4 pair whole (x[2i], x[2i+1]) lanes and run as
// packed adds; the stage at distance 1 follows as scalar adds.  Stages
// commute, and the callers use this only where every partial sum is exact
// (or on parts that are), so the order leaves the results unchanged.
__device__ __forceinline__ void fwht8(float* x) {
  unsigned long long p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = f2_pack(x[2 * i], x[2 * i + 1]);
#pragma unroll
  for (int h = 1; h < 4; h <<= 1)
#pragma unroll
    for (int a = 0; a < 4; ++a)
      if ((a & h) == 0) {
        const unsigned long long u = p[a], v = p[a + h];
        p[a] = f2_add(u, v);
        p[a + h] = f2_sub(u, v);
      }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a, b;
    f2_unpack(p[i], a, b);
    x[2 * i] = a + b;
    x[2 * i + 1] = a - b;
  }
}

// Sylvester row of sequency k: bit-reversed (4 bits) Gray code of k.
__device__ __forceinline__ int sequency_row(int k) {
  int g = k ^ (k >> 1);
  return ((g & 1) << 3) | ((g & 2) << 1) | ((g & 4) >> 1) | ((g & 8) >> 3);
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2,
// 3", SC'11).  Counter (c0..c3), key (k0, k1).
// ---------------------------------------------------------------------------
struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(uint32_t c0, uint32_t c1,
                                            uint32_t c2, uint32_t c3,
                                            uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    unsigned long long p0 = (unsigned long long)0xD2511F53u * c0;
    unsigned long long p1 = (unsigned long long)0xCD9E8D57u * c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return {c0, c1, c2, c3};
}

// The four words for elements 4q .. 4q+3 of `stream`.
__device__ __forceinline__ U4 philox_block(uint64_t seed, uint32_t stream,
                                           uint64_t q) {
  return philox4x32_10((uint32_t)q, (uint32_t)(q >> 32), stream, 0u,
                       (uint32_t)seed, (uint32_t)(seed >> 32));
}

// The ten round keys of a seed (the key schedule does not depend on the
// counter).  The launchers compute them on the host and pass them by value,
// so the kernels read them from the parameter (constant) bank instead of
// holding twenty registers per thread.
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

__host__ __device__ __forceinline__ PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys k;
  uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = a;
    k.k1[r] = b;
    a += 0x9E3779B9u;
    b += 0xBB67AE85u;
  }
  return k;
}

__device__ __forceinline__ U4 philox_block_k(const PhiloxKeys& k, uint32_t stream,
                                             uint64_t q) {
  uint32_t c0 = (uint32_t)q, c1 = (uint32_t)(q >> 32), c2 = stream, c3 = 0u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const unsigned long long p0 = (unsigned long long)0xD2511F53u * c0;
    const unsigned long long p1 = (unsigned long long)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k.k0[r];
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k.k1[r];
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
  }
  return {c0, c1, c2, c3};
}

// ---------------------------------------------------------------------------
// Quantizers, float-valued (integer-valued results, clamped to +-qmax):
//   SR:  x = RN(y / s), f = floor(x), q = f + [u < x - f], u = (word >> 8) 2^-24
//   RNE: q = rint(RN(y / s))
// Division is IEEE round-to-nearest.  The _nz forms are for a scale known
// to be non-zero (callers that branch on s == 0 once per row or tensor);
// the _f forms give 0 when s == 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float quant_sr_nz(float y, float s, uint32_t word, float qmax) {
  const float x = __fdiv_rn(y, s);
  const float f = floorf(x);
  const float frac = x - f;
  const float u = __uint2float_rn(word >> 8) * 5.9604644775390625e-08f;  // 2^-24
  return fminf(fmaxf(f + ((u < frac) ? 1.0f : 0.0f), -qmax), qmax);
}
__device__ __forceinline__ float quant_rne_nz(float y, float s, float qmax) {
  return fminf(fmaxf(rintf(__fdiv_rn(y, s)), -qmax), qmax);
}

__device__ __forceinline__ float quant_sr_f(float y, float s, uint32_t word, float qmax) {
  const float r = quant_sr_nz(y, s, word, qmax);
  return s == 0.0f ? 0.0f : r;
}

__device__ __forceinline__ float quant_rne_f(float y, float s, float qmax) {
  const float r = quant_rne_nz(y, s, qmax);
  return s == 0.0f ? 0.0f : r;
}

// Two integer-valued floats in [-7, 7] to two E4M3 bytes (exact; a in the
// low byte).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// E4M3 byte of an integer in [-7, 7] (exact): |q| = 1.m * 2^e, bias 7.
__device__ __forceinline__ uint32_t e4m3_of_int(int q) {
  // table for |q| = 0..7: 0x00 0x38 0x40 0x44 0x48 0x4A 0x4C 0x4E
  const uint32_t lo = 0x44403800u, hi = 0x4E4C4A48u;
  int a = q < 0 ? -q : q;
  uint32_t mag = ((a < 4 ? lo : hi) >> (8 * (a & 3))) & 0xffu;
  return mag | (q < 0 ? 0x80u : 0u);
}

// Integer value of an E4M3 byte that encodes an integer in [-7, 7].
__device__ __forceinline__ int int_of_e4m3(uint32_t b) {
  uint32_t mag = b & 0x7fu;
  int v;
  if (mag == 0u) {
    v = 0;
  } else {
    int e = int(mag >> 3) - 7;          // unbiased exponent (0..2 here)
    int m = int(mag & 7u) | 8;          // 1.mmm as 4 bits
    v = (e >= 3) ? (m << (e - 3)) : (m >> (3 - e));
  }
  return (b & 0x80u) ? -v : v;
}

// Max of non-negative floats by their bit patterns (monotone for >= 0).
__device__ __forceinline__ void atomic_max_nonneg(unsigned int* slot, float v) {
  atomicMax(slot, __float_as_uint(v));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Max over the CTA (every thread calls it; blockDim.x a multiple of 32, at
// most 1024), then one atomicMax per CTA into `slot`.
__device__ __forceinline__ void cta_max_to_slot(float v, unsigned int* slot) {
  __shared__ float partial[32];
  v = warp_max(v);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) partial[w] = v;
  __syncthreads();
  if (w == 0) {
    float m = lane < (int)(blockDim.x >> 5) ? partial[lane] : 0.0f;
    m = warp_max(m);
    if (lane == 0) atomic_max_nonneg(slot, m);
  }
}

}  // namespace hlq
