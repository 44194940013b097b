// hlq_gemm_tc.cu -- exact integer GEMMs of the HLQ backward pass on the
// sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
//   acc[m, n] = sum_k A[m, k] * B[n, k]     (A [M, K], B [N, K], K contiguous)
//   out[m, n] = float(acc) * (sa[m or 0] * sb[0] / 16)
//
// sm_103a has no integer MMA kind, so the integer codes ride on float
// operand types that hold them exactly:
//   - g_x path: int4 codes in [-7, 7] as E4M3 bytes, tcgen05.mma kind::f8f6f4;
//   - g_w path: int8 codes in [-127, 127] as fp16, tcgen05.mma kind::f16.
// A g_w operand may also stay int8 in HBM: its tiles are loaded as bytes
// and widened to fp16 in shared memory by the epilogue warps (kCvt).
// Products are integers and the fp32 TMEM accumulator holds every partial
// sum exactly while it stays below 2^24; the K loop is therefore cut into
// chunks of at most `chunk_kb` k-blocks whose accumulators are drained into
// int32 registers (49 * K < 2^24 lets the E4M3 path use one chunk; the bf16
// path uses chunks of 16 k-blocks = 1024 codes, 1024 * 127^2 < 2^24).
//
// Two tile shapes.  One CTA per 128 x BN output tile (cta_group::1), or one
// CTA pair (a cluster of two) per 256 x BN tile (kPair, cta_group::2): CTA r
// of the pair loads rows 128 r .. 128 r + 127 of the tile's A block and rows
// (BN/2) r .. of its B block into its own shared memory, CTA 0 issues the
// M = 256 MMAs, which read both CTAs' shared memory at the same offsets and
// leave each CTA's 128 accumulator rows in its own TMEM.  Each SM then
// receives half the B bytes per k-block of the one-CTA tile of the same
// width, which is what bounds the mainloop (operand delivery from L2).
//
// CTA layout (persistent over output tiles, each optionally split along K
// with an exact int32 reduction through a workspace):
//   warp 0      TMA producer (one lane): A and B k-blocks of 128 bytes per
//               row into a ring of 128B-swizzled smem tiles (4-6 stages);
//   warp 1      TMEM allocator and MMA issuer (one lane), 4 MMAs per k-block
//               into one of two TMEM accumulators (double buffer per chunk);
//   warps 2..   epilogue: drain TMEM (tcgen05.ld) into int32 registers per
//               chunk, then dequantize and store fp32 rows; with int8
//               operands they first widen each stage's tiles.
// Every mbarrier wait is bounded (HLQ_DEV_TIMEOUT, then the CTA winds down).
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "hlq_device.cuh"
#include "hlq_kernels.h"
#include "hlq_tma.cuh"

namespace hlq {
namespace {

constexpr int kBM = 128;
constexpr int kRowBytes = 128;  // bytes of one k-block per row (swizzle span)

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile stored with the 128-byte
// swizzle (rows of 128 bytes, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;        // stride byte offset: 8 rows
  d |= (uint64_t)1 << 46;                  // descriptor version
  d |= (uint64_t)2 << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 accumulator, A/B K-major, shape M x N.
// Operand formats 0: E4M3 under kind::f8f6f4 (kKind 0), fp16 under
// kind::f16 (kKind 1).
__host__ __device__ constexpr uint32_t make_idesc(int kKind, int M, int N) {
  return (void)kKind, (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int kKind, bool kPair = false>
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t a, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  if (kPair) {
    if (kKind == 0) {
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
          "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
          : "memory");
    } else {
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
          "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
          : "memory");
    }
    return;
  }
  if (kKind == 0) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          saddr(bar))
      : "memory");
}

// Pair form: once the MMAs issued so far complete, arrive on the barrier at
// the same shared-memory offset in both CTAs of the pair.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  const uint16_t both = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(saddr(bar)),
      "h"(both)
      : "memory");
}

template <bool kPair>
__device__ __forceinline__ void mma_commit_to(uint64_t* bar) {
  if (kPair) mma_commit_pair(bar);
  else mma_commit(bar);
}

// 32 TMEM lanes x 32 consecutive 32-bit columns; thread i gets lane i.
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 TMEM lanes x 16 consecutive 32-bit columns (the drains of the GEMMs
// that widen int8 operands, which hold more registers between drains).
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The mainloop is bound by the latency of a TMA round trip (L2 -> shared
// memory, MMA, release), so the ring holds as many stages as shared memory
// allows: 7 of 28 KB for 96-wide tiles, 6 of 32 KB for 128-wide ones, 4 of
// 48 KB for 256-wide ones.  A 96-wide tile serves shapes where it needs
// fewer waves than 128-wide ones.
// CTA pairs: 6 stages of 32 KB (16 KB of A, 16 KB of the B half) for 256-wide
// tiles, 8 of 24 KB for 128-wide ones.
// kCvt (kind 1): kRawB / kRawA mark operands that arrive as int8 codes; the
// TMA puts them, unswizzled, in the upper half of their fp16 slot and the
// epilogue warps widen them in place (same stage sizes).
template <int BN, bool kPair = false, int kCvt = 0>
struct TcCfg {
  static_assert(BN == 96 || BN == 128 || BN == 256, "tile widths 96, 128, 256");
  static_assert(!kPair || BN != 96, "CTA pairs take 128- or 256-wide tiles");
  static constexpr int kStages =
      kPair ? (BN == 256 ? 6 : 8) : (BN == 96 ? 7 : (BN == 128 ? 6 : 4));
  static constexpr int kColGroups = BN > 128 ? 2 : 1;     // 128-column halves
  static constexpr int kEpiWarps = 4 * kColGroups;        // 4 TMEM lane quarters each
  static constexpr int kColsPerThread = BN / kColGroups;  // 96 or 128
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kBRows = kPair ? BN / 2 : BN;      // B rows in this CTA
  static constexpr int kTileM = kPair ? 2 * kBM : kBM;    // output rows per tile
  static constexpr uint32_t kABytes = kBM * kRowBytes;
  static constexpr uint32_t kBBytes = kBRows * kRowBytes;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  // bytes the TMA delivers per stage (int8 operands: half their fp16 slot)
  static constexpr uint32_t kLoadBytes =
      ((kCvt & kRawA) ? kABytes / 2 : kABytes) + ((kCvt & kRawB) ? kBBytes / 2 : kBBytes);
  // 16-code pieces of the int8 tiles per converting (epilogue) thread
  static constexpr int kConvThreads = 32 * kEpiWarps;
  static constexpr int kAPieces = (kCvt & kRawA) ? kBM * 4 / kConvThreads : 0;
  static constexpr int kBPieces = (kCvt & kRawB) ? kBRows * 4 / kConvThreads : 0;
  static_assert((kBRows * 4) % kConvThreads == 0 && (kBM * 4) % kConvThreads == 0,
                "whole pieces per converting thread");
  // two accumulators, each starting on a 128-column boundary
  static constexpr uint32_t kAccStride = BN <= 128 ? 128 : 256;
  static constexpr uint32_t kTmemCols = 2 * kAccStride;
  // epilogue staging: one 32 x 32 fp32 box (128B-swizzled) per epilogue warp
  static constexpr uint32_t kStageOutBytes = 32 * 32 * 4;
  static constexpr size_t kSmem =
      1024 + (size_t)kStages * kStageBytes + (size_t)kEpiWarps * kStageOutBytes + 256;
  static_assert(kSmem <= 232448, "227 KB of shared memory per CTA");
  static_assert(3 * kStages * 8 + 4 * 8 + 8 <= 256, "barriers fit their 256 bytes");
};

// Barrier over the `n` epilogue threads (named barrier 1) that also returns
// whether `pred` held in every one of them.
__device__ __forceinline__ bool epi_barrier_all(bool pred, int n) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(n)
      : "memory");
  return r != 0;
}

// Two int8 codes of a word (flipped to c + 128 by the caller) as fp16x2:
// the permute builds the fp16 bit patterns 0x64uu = 1024 + c + 128, exact
// integers, and one fp16x2 subtraction of 1152 (0x6480) leaves c exactly.
__device__ __forceinline__ uint32_t f16x2_of_biased_i8(uint32_t biased, uint32_t sel) {
  uint32_t h, r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(h) : "r"(biased), "r"(0x64646464u), "r"(sel));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
  return r;
}

// Piece q of an int8 tile (16 codes: row q / 4, codes 16 (q % 4) ..) to the
// two 16-byte chunks of its fp16 row in the 128B-swizzled tile layout the
// MMA descriptors expect (chunk c of row r at c ^ (r % 8)).
__device__ __forceinline__ void put_widened_piece(uint8_t* slot, int q, uint4 v) {
  const uint32_t a = v.x ^ 0x80808080u, b = v.y ^ 0x80808080u;
  const uint32_t c = v.z ^ 0x80808080u, d = v.w ^ 0x80808080u;
  const uint4 lo = make_uint4(f16x2_of_biased_i8(a, 0x4140u), f16x2_of_biased_i8(a, 0x4342u),
                              f16x2_of_biased_i8(b, 0x4140u), f16x2_of_biased_i8(b, 0x4342u));
  const uint4 hi = make_uint4(f16x2_of_biased_i8(c, 0x4140u), f16x2_of_biased_i8(c, 0x4342u),
                              f16x2_of_biased_i8(d, 0x4140u), f16x2_of_biased_i8(d, 0x4342u));
  const int row = q >> 2, c0 = (q & 3) * 2;
  uint8_t* rp = slot + row * kRowBytes;
  *reinterpret_cast<uint4*>(rp + ((c0 ^ (row & 7)) << 4)) = lo;
  *reinterpret_cast<uint4*>(rp + (((c0 + 1) ^ (row & 7)) << 4)) = hi;
}

// Persistent: CTA b (CTA pair b with kPair) processes work units b, b + G,
// ... (G = the number of CTAs, or of pairs) where a unit is (output tile,
// K split).  The TMA producer and the MMA issuer run through their units
// without pausing between tiles; a unit's epilogue (stores, or exact int32
// reductions for a split unit) overlaps the next unit's MMAs.
//
// With kPair, CTA 0 of the pair owns the barriers that gate the MMA: the
// full barrier of a stage expects both CTAs' bytes (each CTA's loads signal
// CTA 0's barrier), and the accumulator-empty barrier counts the epilogue
// warps of both CTAs (CTA 1's arrive remotely).  The MMA commits arrive on
// the stage-empty and accumulator-full barriers of both CTAs at once.
//
// With kCvt, each CTA's loads signal its own full barrier; its epilogue
// warps wait there, widen the int8 codes of the stage, and arrive on the
// stage's converted barrier (CTA 0's, for a pair), which gates the MMA.  The
// same warps drain the accumulators, each chunk's drain placed after the
// first few conversions of the next chunk.
template <int kKind, int BN, bool kPair, int kCvt>
__global__ void __launch_bounds__(TcCfg<BN, kPair, kCvt>::kThreads, 1) gemm_tc_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
    const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmAcc,
    const __grid_constant__ CUtensorMap tmSplit,
    int M, int N, int num_kb, int chunk_kb, int kb_per_split, int splits, int tiles_n,
    int tiles_m, int group_m, int num_units, int sk_len, const float* __restrict__ sa,
    int per_row_a,
    const float* __restrict__ sb, int per_col_b, float* __restrict__ out,
    int32_t* __restrict__ acc_out,
    int32_t* __restrict__ split_acc, unsigned int* __restrict__ slab_count,
    unsigned int* __restrict__ status) {
  using C = TcCfg<BN, kPair, kCvt>;
  static_assert(kCvt == 0 || kKind == 1, "int8 operands feed the fp16 GEMM");
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_out = smem + kStages * C::kStageBytes;  // [kEpiWarps][4 KB]
  uint64_t* full = reinterpret_cast<uint64_t*>(stage_out + C::kEpiWarps * C::kStageOutBytes);
  uint64_t* empty = full + kStages;
  uint64_t* conv = empty + kStages;   // [kStages], kCvt only
  uint64_t* tfull = conv + kStages;   // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // rank in the pair (0 without pairs) and this CTA's (or pair's) place in
  // the persistent grid
  const uint32_t rank = kPair ? cluster_rank() : 0u;
  const int first_unit = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int unit_step = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&conv[s], kPair ? 2 * C::kEpiWarps : C::kEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kPair ? 2 * C::kEpiWarps : C::kEpiWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    if (kPair) {  // one warp of each CTA of the pair allocates together
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       saddr(tmem_holder)),
                   "r"(C::kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       saddr(tmem_holder)),
                   "r"(C::kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();  // the peer's barriers exist before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // barriers of CTA 0 that both CTAs of a pair signal
  const uint32_t full_lead = kPair ? cluster_map(saddr(full), 0) : 0u;
  const uint32_t conv_lead = kPair ? cluster_map(saddr(conv), 0) : 0u;
  const uint32_t tempty_lead = kPair ? cluster_map(saddr(tempty), 0) : 0u;
  // the prologue above overlaps the previous kernel; operands, scales and
  // outputs are touched only after it has completed
  pdl_trigger();
  pdl_wait();

  // unit -> (row tile, column tile, first k-block, k-blocks).  Tiles go in
  // groups of group_m row tiles; within a group the row tile changes
  // fastest, so the units in flight at once share their B tiles and the
  // group's A rows stay in L2 while the column tiles go by.
  auto unit_tile = [&](int u, int& tm, int& tn, int& kb0, int& nkb) {
    const int t = u / splits, z = u - t * splits;
    const int g = t / (group_m * tiles_n), r = t - g * (group_m * tiles_n);
    const int gm = min(group_m, tiles_m - g * group_m);  // rows of this group
    tn = r / gm;
    tm = g * group_m + (r - tn * gm);
    kb0 = z * kb_per_split;
    nkb = max(0, min(num_kb, kb0 + kb_per_split) - kb0);
  };
  // The j-th unit of this CTA (pair): its tile, k-block range and how many
  // units share the tile (`parts`; 1: the unit stores the tile itself).
  // Without stream-K the units are u = first_unit + j * unit_step.  With
  // stream-K (sk_len > 0, one CTA per SM, num_units = tiles, no pairs) CTA b
  // takes the k-blocks [b sk_len, (b + 1) sk_len) of the tiles laid end to
  // end, one unit per tile it touches: every SM gets the same share of a
  // GEMM whose tiles fill less than one wave.
  struct Unit {
    int tm, tn, kb0, nkb, parts;
  };
  auto get_unit = [&](int j, Unit& w) -> bool {
    if (sk_len == 0) {
      const int u = first_unit + j * unit_step;
      if (u >= num_units) return false;
      unit_tile(u, w.tm, w.tn, w.kb0, w.nkb);
      w.parts = splits;
      return true;
    }
    const long long total = (long long)num_units * num_kb;
    const long long s0 = (long long)first_unit * sk_len;
    const long long e0 = min(s0 + (long long)sk_len, total);
    const long long t = s0 / num_kb + j;
    const long long ts = t * num_kb, te = ts + num_kb;
    const long long a = max(s0, ts), e = min(e0, te);
    if (a >= e) return false;
    int kb_unused, nkb_unused;
    unit_tile((int)t, w.tm, w.tn, kb_unused, nkb_unused);  // splits == 1 here
    w.kb0 = (int)(a - ts);
    w.nkb = (int)(e - a);
    w.parts = (int)((te - 1) / sk_len - ts / sk_len + 1);
    return true;
  };

  if (warp == 0) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA))
                   : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB))
                   : "memory");
      const int elems = kRowBytes / (kKind == 1 ? 2 : 1);
      int i = 0;  // k-blocks issued by this CTA so far
      Unit w;
      for (int ju = 0; !*abort_flag && get_unit(ju, w); ++ju) {
        const int m0 = w.tm * C::kTileM, n0 = w.tn * BN, kb0 = w.kb0, nkb = w.nkb;
        for (int j = 0; j < nkb; ++j, ++i) {
          const int s = i % kStages;
          const uint32_t ph = (uint32_t)(i / kStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, status)) break;
          uint8_t* a = smem + s * C::kStageBytes;
          const int kx = (kb0 + j) * elems;
          if (kCvt != 0) {
            // this CTA's own barrier; int8 tiles land in the upper half of
            // their slot, where the epilogue warps widen them
            mbar_expect_tx(&full[s], C::kLoadBytes);
            tma_load_2d(a + ((kCvt & kRawA) ? C::kABytes / 2 : 0u), &tmA, &full[s], kx,
                        m0 + (int)rank * kBM);
            tma_load_2d(a + C::kABytes + ((kCvt & kRawB) ? C::kBBytes / 2 : 0u), &tmB,
                        &full[s], kx, n0 + (int)rank * C::kBRows);
          } else if (kPair) {
            // CTA 0 expects both halves; each CTA's copies signal CTA 0
            if (rank == 0) mbar_expect_tx(&full[s], 2 * C::kStageBytes);
            const uint32_t bar = full_lead + (uint32_t)(s * sizeof(uint64_t));
            tma_load_2d_pair(a, &tmA, bar, kx, m0 + (int)rank * kBM);
            tma_load_2d_pair(a + C::kABytes, &tmB, bar, kx, n0 + (int)rank * C::kBRows);
          } else {
            mbar_expect_tx(&full[s], C::kStageBytes);
            tma_load_2d(a, &tmA, &full[s], kx, m0);
            tma_load_2d(a + C::kABytes, &tmB, &full[s], kx, n0);
          }
        }
      }
      if (*abort_flag && (!kPair || kCvt != 0)) {  // let the copies already issued land
        for (int k = max(0, i - kStages); k < i; ++k) {
          const unsigned long long t0 = now_ns();
          while (!mbar_test(&full[k % kStages], (uint32_t)(k / kStages) & 1u) &&
                 now_ns() - t0 < kWaitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {  // the MMA issuer (CTA 0 of a pair)
      const uint32_t idesc = make_idesc(kKind, C::kTileM, BN);
      int i = 0, cc = 0;  // k-blocks and accumulation chunks consumed so far
      bool ok = true;
      Unit w;
      for (int ju = 0; ok && get_unit(ju, w); ++ju) {
        const int nkb = w.nkb;
        const int nch = (nkb + chunk_kb - 1) / chunk_kb;
        for (int c = 0, j = 0; c < nch && ok; ++c, ++cc) {
          const int buf = cc & 1;
          const uint32_t use = (uint32_t)(cc >> 1);
          // CTA 1's epilogue warps arrive here from the other SM of a pair
          if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, status, kPair)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + (uint32_t)(buf * C::kAccStride);
          const int j_end = min(nkb, j + chunk_kb);
          for (int jj = 0; j < j_end; ++j, ++jj, ++i) {
            const int s = i % kStages;
            const uint32_t ph = (uint32_t)(i / kStages) & 1u;
            // loaded (and, for int8 operands, widened by both CTAs)
            const bool ready = kCvt != 0
                                   ? mbar_wait(&conv[s], ph, abort_flag, status, kPair)
                                   : mbar_wait(&full[s], ph, abort_flag, status);
            if (!ready) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a = saddr(smem + s * C::kStageBytes);
            const uint32_t b = a + C::kABytes;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_issue<kKind, kPair>(d, sw128_desc(a + 32 * k), sw128_desc(b + 32 * k), idesc,
                                      (jj > 0 || k > 0) ? 1u : 0u);
            mma_commit_to<kPair>(&empty[s]);
          }
          if (ok) mma_commit_to<kPair>(&tfull[buf]);
        }
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int ew = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int colgrp = ew >> 2;
    const int row = (int)rank * kBM + quarter * 32 + lane;  // row within the tile
    uint8_t* stg = stage_out + ew * C::kStageOutBytes;
    // accumulator buffer drained: tell the MMA issuer (CTA 0 of a pair)
    auto release_acc = [&](int buf) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair && rank != 0)
          mbar_arrive_cluster(tempty_lead + (uint32_t)(buf * sizeof(uint64_t)));
        else
          mbar_arrive(&tempty[buf]);
      }
    };
    // One 32 x 32 box of 32-bit values (this thread's row, 32 columns)
    // through the warp's staging buffer (128B swizzle: 16-byte chunk c of row
    // r at c ^ (r % 8), conflict-free) and a TMA store, which clips rows >= M
    // and columns >= N.
    auto store_box = [&](const CUtensorMap* map, int x, int y, const uint32_t (&v)[32],
                         bool reduce_add = false) {
      if (lane == 0) tma_store_wait_read();  // the previous box has been read
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
            make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (reduce_add)
          tma_reduce_add_2d(map, x, y, stg);
        else
          tma_store_2d(map, x, y, stg);
      }
    };
    auto dequant_scale = [&](int m) {
      return (out && m < M) ? ld_dep_f32(sa + (per_row_a ? m : 0)) * ld_dep_f32(sb) * 0.0625f
                            : 0.0f;
    };
    // per_col_b: the B scale of column n, sb[n], in the same product order
    auto row_scale_a = [&](int m) {
      return (out && m < M) ? ld_dep_f32(sa + (per_row_a ? m : 0)) : 0.0f;
    };
    auto col_scaled = [&](int32_t a, float ra, int n) {
      return __float_as_uint((float)a * (ra * ld_dep_f32(sb + min(n, N - 1)) * 0.0625f));
    };
    int cc = 0;
    bool ok = true;
    if constexpr (kKind == 0) {
      Unit w;
      for (int ju = 0; ok && get_unit(ju, w); ++ju) {
        const int m0 = w.tm * C::kTileM, n0 = w.tn * BN;
        const int m = m0 + row;
        const int nb = n0 + colgrp * C::kColsPerThread;
        const int y = m0 + (int)rank * kBM + quarter * 32;
        // one accumulation chunk, never split: stream each 32-column TMEM
        // slice straight into a store box
        const int buf = cc & 1;
        const uint32_t use = (uint32_t)(cc >> 1);
        ++cc;
        ok = mbar_wait(&tfull[buf], use & 1u, abort_flag, status);
        ok = __all_sync(0xffffffffu, ok);  // also reconverges the warp
        if (!ok) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                               (uint32_t)(buf * C::kAccStride + colgrp * C::kColsPerThread);
        const float scale = dequant_scale(m);
#pragma unroll
        for (int jc = 0; jc < C::kColsPerThread / 32; ++jc) {
          uint32_t r[32];
          tmem_ld_x32(taddr + 32 * jc, r);
          if (jc == C::kColsPerThread / 32 - 1) release_acc(buf);  // read out
          const int x = nb + 32 * jc;
          if (x >= N) continue;
          if (acc_out) {
            uint32_t v[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = (uint32_t)__float2int_rn(__uint_as_float(r[q]));
            store_box(&tmAcc, x, y, v);
          }
          if (out) {
#pragma unroll
            for (int q = 0; q < 32; ++q)
              r[q] = __float_as_uint((float)__float2int_rn(__uint_as_float(r[q])) * scale);
            store_box(&tmOut, x, y, r);
          }
        }
      }
    } else {
      int32_t acc[C::kColsPerThread];
#pragma unroll
      for (int q = 0; q < C::kColsPerThread; ++q) acc[q] = 0;
      // add the next accumulation chunk (in TMEM buffer cc & 1) into acc
      auto drain = [&]() -> bool {
        const int buf = cc & 1;
        const uint32_t use = (uint32_t)(cc >> 1);
        ++cc;
        bool w = mbar_wait(&tfull[buf], use & 1u, abort_flag, status);
        w = __all_sync(0xffffffffu, w);  // also reconverges the warp
        if (!w) return false;
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                               (uint32_t)(buf * C::kAccStride + colgrp * C::kColsPerThread);
        if constexpr (kCvt == 0) {
#pragma unroll
          for (int jc = 0; jc < C::kColsPerThread / 32; ++jc) {
            uint32_t r[32];
            tmem_ld_x32(taddr + 32 * jc, r);
#pragma unroll
            for (int q = 0; q < 32; ++q)
              acc[32 * jc + q] += __float2int_rn(__uint_as_float(r[q]));
          }
        } else {
#pragma unroll
          for (int jc = 0; jc < C::kColsPerThread / 16; ++jc) {
            uint32_t r[16];
            tmem_ld_x16(taddr + 16 * jc, r);
#pragma unroll
            for (int q = 0; q < 16; ++q)
              acc[16 * jc + q] += __float2int_rn(__uint_as_float(r[q]));
          }
        }
        release_acc(buf);
        return true;
      };
      // unit w's sums are complete in acc: store them dequantized, or add
      // them into the split workspace (the last unit of a slab stores)
      auto finish_unit = [&](const Unit& w) {
        const int m0 = w.tm * C::kTileM, n0 = w.tn * BN;
        const int m = m0 + row;
        const int nb = n0 + colgrp * C::kColsPerThread;
        const int y = m0 + (int)rank * kBM + quarter * 32;
        if (w.parts == 1) {
          const float scale = dequant_scale(m);
#pragma unroll
          for (int jc = 0; jc < C::kColsPerThread / 32; ++jc) {
            const int x = nb + 32 * jc;
            if (x >= N) break;
            uint32_t v[32];
            if (acc_out) {
#pragma unroll
              for (int q = 0; q < 32; ++q) v[q] = (uint32_t)acc[32 * jc + q];
              store_box(&tmAcc, x, y, v);
            }
            if (out) {
              if (per_col_b) {
                const float ra = row_scale_a(m);
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = col_scaled(acc[32 * jc + q], ra, x + q);
              } else {
#pragma unroll
                for (int q = 0; q < 32; ++q)
                  v[q] = __float_as_uint((float)acc[32 * jc + q] * scale);
              }
              store_box(&tmOut, x, y, v);
            }
          }
          return;
        }
        // split unit: add the exact partial into split_acc with TMA reduce-add
        // boxes (32 rows x 32 columns, coalesced in L2); the warp that
        // completes a slab (its 32 rows x kColsPerThread columns) last reads
        // the sum back and stores it dequantized
#pragma unroll
        for (int jc = 0; jc < C::kColsPerThread / 32; ++jc) {
          const int x = nb + 32 * jc;
          if (x >= N) break;
          uint32_t v[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] = (uint32_t)acc[32 * jc + q];
          store_box(&tmSplit, x, y, v, true);
        }
        unsigned int last = 0;
        if (lane == 0) {
          tma_store_wait_all();  // the reductions are performed
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          // slab counters per (128-row half tile, epilogue warp)
          const int half = w.tm * (C::kTileM / kBM) + (int)rank;
          const int slab = (half * tiles_n + w.tn) * C::kEpiWarps + ew;
          last = atomicAdd(&slab_count[slab], 1u) == (unsigned int)(w.parts - 1);
          if (last) __threadfence();
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          const float scale = dequant_scale(m);
          const float ra = row_scale_a(m);
#pragma unroll
          for (int jc = 0; jc < C::kColsPerThread / 32; ++jc) {
            const int x = nb + 32 * jc;
            if (x >= N) break;
            int32_t sum[32];
            const int32_t* rowp = split_acc + (size_t)m * N + x;
#pragma unroll
            for (int q = 0; q < 32; q += 4) {
              int4 w4 = make_int4(0, 0, 0, 0);
              if (m < M && x + q < N) w4 = __ldcg(reinterpret_cast<const int4*>(rowp + q));
              sum[q] = w4.x; sum[q + 1] = w4.y; sum[q + 2] = w4.z; sum[q + 3] = w4.w;
            }
            uint32_t v[32];
            if (acc_out) {
#pragma unroll
              for (int q = 0; q < 32; ++q) v[q] = (uint32_t)sum[q];
              store_box(&tmAcc, x, y, v);
            }
            if (out) {
              if (per_col_b) {
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = col_scaled(sum[q], ra, x + q);
              } else {
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = __float_as_uint((float)sum[q] * scale);
              }
              store_box(&tmOut, x, y, v);
            }
          }
        }
      };
      auto zero_acc = [&]() {
#pragma unroll
        for (int q = 0; q < C::kColsPerThread; ++q) acc[q] = 0;
      };
      if constexpr (kCvt == 0) {
        Unit w;
        for (int ju = 0; ok && get_unit(ju, w); ++ju) {
          const int nch = (w.nkb + chunk_kb - 1) / chunk_kb;
          zero_acc();
          for (int c = 0; c < nch && ok; ++c) ok = drain();
          if (!ok) break;
          finish_unit(w);
        }
      } else {
        // widen stage i's int8 tiles in place; false (in every epilogue
        // thread at once) when this or another thread's wait gave up
        const int et = (int)threadIdx.x - 64;  // 0 .. kConvThreads - 1
        int i = 0;
        auto convert = [&]() -> bool {
          const int s = i % kStages;
          const uint32_t ph = (uint32_t)(i / kStages) & 1u;
          ++i;
          const bool w = mbar_wait(&full[s], ph, abort_flag, status);
          uint8_t* a_slot = smem + s * C::kStageBytes;
          uint8_t* b_slot = a_slot + C::kABytes;
          uint4 ra[C::kAPieces > 0 ? C::kAPieces : 1];
          uint4 rb[C::kBPieces > 0 ? C::kBPieces : 1];
#pragma unroll
          for (int p = 0; p < C::kAPieces; ++p)
            ra[p] = *reinterpret_cast<const uint4*>(a_slot + C::kABytes / 2 +
                                                    16 * (et + p * C::kConvThreads));
#pragma unroll
          for (int p = 0; p < C::kBPieces; ++p)
            rb[p] = *reinterpret_cast<const uint4*>(b_slot + C::kBBytes / 2 +
                                                    16 * (et + p * C::kConvThreads));
          // every int8 piece is in registers before any fp16 row lands on it
          __syncwarp();
          if (!epi_barrier_all(ok && w, C::kConvThreads)) return false;
#pragma unroll
          for (int p = 0; p < C::kAPieces; ++p)
            put_widened_piece(a_slot, et + p * C::kConvThreads, ra[p]);
#pragma unroll
          for (int p = 0; p < C::kBPieces; ++p)
            put_widened_piece(b_slot, et + p * C::kConvThreads, rb[p]);
          fence_proxy_async_smem();  // generic writes -> the MMA's reads
          __syncwarp();
          if (lane == 0) {
            if (kPair && rank != 0)
              mbar_arrive_cluster(conv_lead + (uint32_t)(s * sizeof(uint64_t)));
            else
              mbar_arrive(&conv[s]);
          }
          return true;
        };
        // Chunk c - 1 of a unit is drained once the first kLag stages of
        // chunk c are converted (the MMA has finished it by then or soon
        // after, and has converted stages to work on while the drain runs);
        // a unit's last chunk is drained after the first kLag stages of the
        // next unit are converted.  Every unit has k-blocks (the launcher
        // drops empty splits).
        constexpr int kLag = kStages / 2;
        bool live = true;
        int ahead = 0;  // k-blocks of this unit converted during the last one
        Unit w;
        for (int ju = 0; live && get_unit(ju, w); ++ju) {
          const int nkb = w.nkb;
          const int nch = (nkb + chunk_kb - 1) / chunk_kb;
          zero_acc();
          for (int c = 0, j = 0; c < nch && live; ++c) {
            const int len = min(nkb, j + chunk_kb) - j;
            for (int jj = 0; jj < len; ++jj, ++j) {
              if (j >= ahead && !convert()) {
                live = false;
                break;
              }
              if (c > 0 && jj + 1 == min(len, kLag)) ok = drain() && ok;
            }
          }
          if (!live) break;
          ahead = 0;
          Unit w1;
          if (get_unit(ju + 1, w1)) {
            for (; ahead < min(w1.nkb, kLag); ++ahead)
              if (!convert()) {
                live = false;
                break;
              }
          }
          if (!live) break;
          ok = drain() && ok;
          if (ok) finish_unit(w);
        }
        ok = ok && live;
      }
    }
    if (lane == 0) tma_store_wait_all();  // boxes written before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {  // let in-flight copies and tensor-core work finish
    const unsigned long long t0 = now_ns();
    while (now_ns() - t0 < 1000000ull) {
    }
  }
  // a pair leaves together: no remote arrive or copy may target a CTA that
  // has exited, and the peer's TMEM is freed only after CTA 0's MMAs
  if (kPair) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (kPair)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(C::kTmemCols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(C::kTmemCols)
                   : "memory");
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encode() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                       cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// 2-D K-major operand [rows, K] with row stride ld (elements), boxes of
// 128 bytes x box_rows, 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* map, const void* ptr, bool f16, int64_t rows, int64_t K,
              int64_t ld, int box_rows) {
  const int esz = f16 ? 2 : 1;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * esz)};
  cuuint32_t box[2] = {(cuuint32_t)(kRowBytes / esz), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                        2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// int8 operand [rows, K] (row stride ld bytes) for widening in shared
// memory: boxes of 64 codes x box_rows, unswizzled (rows of 64 bytes, read
// back by the converting threads in 16-byte pieces), zero fill outside.
bool make_i8_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int64_t ld,
                 int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {(cuuint32_t)(kRowBytes / 2), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output [rows, cols] of 32-bit elements (fp32 or int32), stored in 32 x 32
// boxes with the 128-byte swizzle of the epilogue's staging buffers.
bool make_out_map(CUtensorMap* map, const void* ptr, bool is_int, int64_t rows,
                  int64_t cols) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * 4)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, is_int ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Persistent grid of one CTA per SM, or of as many CTA pairs as fit at once
// (clusters of two need both SMs of a pair free; the count comes from the
// occupancy query for this kernel, cached per device).
template <int kKind, int BN, bool kPair, int kCvt = 0>
cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& mo,
                      const CUtensorMap& macc, const CUtensorMap& msplit, int64_t M, int64_t N,
                      int num_kb, int chunk_kb,
                      int splits, int num_sms, const float* sa, bool per_row_a,
                      const float* sb, bool per_col_b, float* out, int32_t* acc_out,
                      int32_t* split_acc, unsigned int* slab_count, unsigned int* status,
                      cudaStream_t st, bool stream_k) {
  using C = TcCfg<BN, kPair, kCvt>;
  auto kernel = gemm_tc_kernel<kKind, BN, kPair, kCvt>;
  static bool attr_set[64] = {};
  static int max_pairs[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int kb_per_split = (num_kb + splits - 1) / splits;
  // no empty splits: the last one holds at least one k-block
  if (num_kb > 0) splits = (num_kb + kb_per_split - 1) / kb_per_split;
  const int tiles_n = (int)((N + BN - 1) / BN);
  const int tiles_m = (int)((M + C::kTileM - 1) / C::kTileM);
  const int64_t units = (int64_t)tiles_m * tiles_n * splits;
  if (units > 0x7fffffff) return cudaErrorInvalidValue;
  // row tiles per group: as many as keep the group's A rows within 48 MB of
  // L2 (the Llama down_proj g_w GEMM, A rows of 4 MB per 256-row tile, read
  // 2.9 GB from HBM for 0.3 GB of operands with the column tile changing
  // fastest, 1.0 GB grouped: 564 -> 489 us; its g_x GEMM 553 -> 537 us).
  // Short contractions (< 16 k-blocks) are bound by their fp32 output and
  // keep the row-major tile order, whose stores fill whole output rows
  // together (ResNet-50 im2col g_x, K = 256: 80 us row-major, 92 grouped).
  const int64_t a_tile_bytes = (int64_t)C::kTileM * num_kb * kRowBytes;
  int group_m = (int)((48ll << 20) / (a_tile_bytes > 0 ? a_tile_bytes : 1));
  group_m = group_m < 1 ? 1 : (group_m > tiles_m ? tiles_m : group_m);
  if (num_kb < 16) group_m = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int grid_ctas;
  int sk_len = 0;
  if (stream_k && !kPair && splits == 1 && num_kb > 0) {
    // equal runs of k-blocks over the tiles laid end to end, one CTA per SM
    const int64_t total = units * (int64_t)num_kb;
    const int64_t g = total < num_sms ? total : num_sms;
    const int64_t len = (total + g - 1) / g;
    if (len > 0x7fffffff) return cudaErrorInvalidValue;
    sk_len = (int)len;
    grid_ctas = (int)((total + len - 1) / len);
  } else if (kPair) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    if (!max_pairs[dev]) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(2 * (num_sms / 2));
      q.blockDim = dim3(C::kThreads);
      q.dynamicSmemBytes = C::kSmem;
      q.attrs = &attr[1];
      q.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kernel, &q);
      if (e != cudaSuccess) return e;
      if (n <= 0) return cudaErrorInvalidConfiguration;
      max_pairs[dev] = n;
    }
    const int64_t pairs = units < max_pairs[dev] ? units : max_pairs[dev];
    grid_ctas = (int)(2 * pairs);
  } else {
    grid_ctas = (int)(units < num_sms ? units : num_sms);
  }
  cfg.gridDim = dim3(grid_ctas);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = kPair ? 2 : 1;
  cudaError_t le = cudaLaunchKernelEx(&cfg, kernel, a, b, mo, macc, msplit, (int)M, (int)N,
                                      num_kb, chunk_kb, kb_per_split, splits, tiles_n, tiles_m,
                                      group_m, (int)units, sk_len, sa, per_row_a ? 1 : 0, sb,
                                      per_col_b ? 1 : 0, out, acc_out, split_acc, slab_count,
                                      status);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace

bool make_tile_map_2d(CUtensorMap* map, const void* ptr, bool bf16, int64_t rows,
                      int64_t cols, int box_cols, int box_rows) {
  if (!get_encode()) return false;
  const int esz = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * esz)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Slab counters of a split plan: one per (128-row half tile, epilogue warp);
// pair tiles are 256 rows, so M rounds up to a multiple of 256 there.
static int64_t split_slabs(int64_t M, int64_t N, int bn, bool pair) {
  const int64_t halves = pair ? 2 * ((M + 255) / 256) : (M + kBM - 1) / kBM;
  return halves * ((N + bn - 1) / bn) * (bn > 128 ? 8 : 4);
}

size_t gemm_tc_split_ws_bytes(int64_t M, int64_t N) {
  // int32 partial sums, then the slab counters of whichever tile shape the
  // plan takes
  int64_t slabs = 0;
  for (int bn : {96, 128, 256})
    for (bool pair : {false, true})
      if (!(pair && bn == 96)) {
        const int64_t n = split_slabs(M, N, bn, pair);
        slabs = n > slabs ? n : slabs;
      }
  return (size_t)M * (size_t)N * 4 + (size_t)slabs * 4 + 256;
}

GemmPlan plan_gemm_tc(int kind, int64_t M, int64_t N, int64_t K, int num_sms,
                      int max_splits) {
  GemmPlan p{};
  const int elems = kRowBytes / (kind == 1 ? 2 : 1);
  p.num_kb = (int)((K + elems - 1) / elems);
  p.chunk_kb = (kind == 1) ? 16 : p.num_kb;  // bf16: 1024 codes per exact chunk
  if (p.chunk_kb < 1) p.chunk_kb = 1;
  if (num_sms < 1) num_sms = 1;
  const int64_t tiles_m = (M + kBM - 1) / kBM;
  // Tile width: fewer waves of CTAs, weighted by the measured cost of one
  // tile relative to a 128-wide one: 1.6 for a 256-wide tile, and the same
  // for a 96-wide one (the mainloop waits on k-block round trips, so the
  // g_w GEMM of ViT-B qkv took 38.9 us on 144 SMs with 96-wide tiles and on
  // 108 SMs with 128-wide ones).  A 96-wide tile is therefore taken only
  // when it needs fewer waves, and ties leave SMs to concurrent kernels.
  const int64_t t96 = tiles_m * ((N + 95) / 96);
  const int64_t t128 = tiles_m * ((N + 127) / 128);
  const int64_t t256 = tiles_m * ((N + 255) / 256);
  const double w96 = (double)((t96 + num_sms - 1) / num_sms);
  const double w128 = (double)((t128 + num_sms - 1) / num_sms);
  const double w256 = (double)((t256 + num_sms - 1) / num_sms) * 1.6;
  p.bn = (w256 <= w128 && w256 <= w96) ? 256 : (w96 < w128 ? 96 : 128);
  // K split: only when the tiles fill less than a third of the SMs.  The
  // partial sums are added in L2 by TMA reduce-add boxes (ResNet-50 im2col
  // g_w, 36 tiles x 4 splits: 59 us, against 111 us with per-element
  // atomics), but a split still costs a memset, the reductions and a
  // read-back, and for the ViT-B qkv g_w GEMM 256-wide tiles x 2 splits took
  // 48 us against 39 us unsplit.
  p.splits = 1;
  if (max_splits > 1 && t128 * 3 < num_sms) {
    p.bn = 128;
    int s = (int)(num_sms / t128);
    s = s < max_splits ? s : max_splits;
    while (s > 1 && (p.num_kb + s - 1) / s < 2 * p.chunk_kb) --s;
    p.splits = s > 1 ? s : 1;
  }
  // CTA pairs: the same tile width over 256 rows per pair, i.e. the same
  // output per SM with half the B bytes delivered to each SM.  They pay
  // where the mainloop runs in steady state: at least 16 k-blocks per tile
  // and 4 waves of tiles (Llama down_proj on GB300: g_x 679 -> 552 us,
  // g_w 699 -> 564 us).  Short contractions and single-wave GEMMs ran
  // slower on pairs, whose two epilogues gate each accumulator buffer
  // together (ResNet-50 im2col g_x, K = 256: 80 -> 97 us; ViT-B fc2 g_x,
  // K = 768: 41 -> 45 us; ViT-B qkv g_w, one wave: 41 -> 43 us).
  const int64_t tiles1 = tiles_m * ((N + p.bn - 1) / p.bn);
  p.pair = (p.splits == 1 && p.bn != 96 && M > kBM && p.num_kb >= 16 &&
            tiles1 >= (int64_t)4 * num_sms)
               ? 1
               : 0;
  // Stream-K (equal k-block runs per SM over all tiles, partial tiles summed
  // like K splits) is built but never planned: measured on GB300 it was
  // slower for every g_w shape here -- ViT-B qkv 51.9 us against 39.6 us
  // unsplit on 108 of 152 SMs (each k-block took 0.74 us on 152 SMs against
  // 0.40 us on 108: the operand delivery to the SMs, not the idle SMs,
  // bounds that GEMM), ViT-B fc2 56.5 against 39.6, ResNet-50 im2col 63.6
  // against 58.0 with 4 K splits.
  return p;
}

cudaError_t launch_gemm_tc(int kind, const void* A, int64_t lda, const void* B,
                           int64_t ldb, int64_t M, int64_t N, int64_t K,
                           const GemmPlan& plan, const float* sa, bool per_row_a,
                           const float* sb, float* out, int32_t* acc_out,
                           void* split_ws, unsigned int* status, cudaStream_t st,
                           bool per_col_b, int raw) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (!get_encode()) return cudaErrorNotSupported;
  const bool f16 = kind == 1;
  if ((plan.bn != 96 && plan.bn != 128 && plan.bn != 256) ||
      (plan.splits > 1 && kind == 0) || (per_col_b && kind == 0) ||
      (plan.pair && plan.bn == 96) || (raw & ~(kRawA | kRawB)) || (raw && kind != 1) ||
      (raw && K <= 0) ||
      (plan.stream_k && (kind != 1 || plan.pair || plan.splits > 1)))
    return cudaErrorInvalidValue;
  // int8 operands: TMA rows of 16-byte multiples from a 16-byte aligned base
  auto i8_ok = [](const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ld % 16 == 0;
  };
  if (((raw & kRawA) && !i8_ok(A, lda)) || ((raw & kRawB) && !i8_ok(B, ldb)))
    return cudaErrorInvalidValue;
  const int b_rows = plan.pair ? plan.bn / 2 : plan.bn;
  CUtensorMap ma, mb, mo, macc, msplit;
  if (!((raw & kRawA) ? make_i8_map(&ma, A, M, K, lda, kBM)
                      : make_map(&ma, A, f16, M, K, lda, kBM)))
    return cudaErrorInvalidValue;
  if (!((raw & kRawB) ? make_i8_map(&mb, B, N, K, ldb, b_rows)
                      : make_map(&mb, B, f16, N, K, ldb, b_rows)))
    return cudaErrorInvalidValue;
  memset(&mo, 0, sizeof(mo));
  memset(&macc, 0, sizeof(macc));
  memset(&msplit, 0, sizeof(msplit));
  if (out && !make_out_map(&mo, out, false, M, N)) return cudaErrorInvalidValue;
  if (acc_out && !make_out_map(&macc, acc_out, true, M, N)) return cudaErrorInvalidValue;
  int32_t* split_acc = nullptr;
  unsigned int* slab_count = nullptr;
  if (plan.splits > 1 || plan.stream_k) {
    split_acc = static_cast<int32_t*>(split_ws);
    if (!make_out_map(&msplit, split_acc, true, M, N)) return cudaErrorInvalidValue;
    slab_count = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(split_ws) +
                                                 (size_t)M * (size_t)N * 4);
    const int64_t slabs = split_slabs(M, N, plan.bn, plan.pair != 0);
    cudaError_t e = cudaMemsetAsync(split_ws, 0, (size_t)M * (size_t)N * 4 + (size_t)slabs * 4,
                                    st);
    if (e != cudaSuccess) return e;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    return cudaErrorInvalidDevice;
#define TC(KIND, BN, PAIR, CVT)                                                             \
  launch_tc<KIND, BN, PAIR, CVT>(ma, mb, mo, macc, msplit, M, N, plan.num_kb, plan.chunk_kb,   \
                                 plan.splits, sms, sa, per_row_a, sb, per_col_b, out,         \
                                 acc_out, split_acc, slab_count, status, st,                  \
                                 plan.stream_k != 0)
#define TC_BN(KIND, PAIR, CVT)                                                    \
  (plan.bn == 256 ? TC(KIND, 256, PAIR, CVT)                                      \
                  : (PAIR || plan.bn == 128) ? TC(KIND, 128, PAIR, CVT) : TC(KIND, 96, false, CVT))
  if (kind == 0) return plan.pair ? TC_BN(0, true, 0) : TC_BN(0, false, 0);
  if (raw == kRawB) return plan.pair ? TC_BN(1, true, kRawB) : TC_BN(1, false, kRawB);
  if (raw == (kRawA | kRawB))
    return plan.pair ? TC_BN(1, true, kRawA | kRawB) : TC_BN(1, false, kRawA | kRawB);
  if (raw != 0) return cudaErrorInvalidValue;  // int8 A alone is not built
  return plan.pair ? TC_BN(1, true, 0) : TC_BN(1, false, 0);
#undef TC_BN
#undef TC
}

}  // namespace hlq
