// hlq_api.cu -- the C ABI of libhlq (declared in include/hlq.h): argument
// validation, workspace layout and the launch sequence of each step.
#include <cstdint>
#include <atomic>
#include <mutex>
#include <cstring>
#include <cuda_runtime.h>

#include "hlq.h"
#include "hlq_kernels.h"

namespace hlq {

namespace {

constexpr int kMaxDevices = 64;
unsigned int* g_status_ptr[kMaxDevices] = {};

// Address of the status word on the current device (looked up once).
unsigned int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  if (!g_status_ptr[dev]) {
    unsigned int* p = nullptr;
    if (status_word_address(&p) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = p;
  }
  return g_status_ptr[dev];
}

// ---------------------------------------------------------------------------
// Launch tracing (hlq_trace_*): while enabled, every kernel launch of this
// library is bracketed by two events recorded on its stream, so per-kernel
// device time can be read back without a profiler.
// ---------------------------------------------------------------------------
struct Trace {
  bool on = false;
  int cap = 0, n = 0;
  cudaEvent_t* ev = nullptr;  // 2 * cap events
  const char** name = nullptr;
};
Trace g_trace;

void trace_free() {
  if (g_trace.ev) {
    for (int i = 0; i < 2 * g_trace.cap; ++i) cudaEventDestroy(g_trace.ev[i]);
    delete[] g_trace.ev;
    delete[] g_trace.name;
  }
  g_trace = Trace{};
}

// Inside a stream capture the records are external, so that they become
// event-record nodes of the graph, re-recorded at every replay; outside a
// capture they are plain records (the external flag is refused there).
inline void trace_record(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}
inline void trace_before(cudaStream_t s) {
  if (g_trace.on && g_trace.n < g_trace.cap) trace_record(g_trace.ev[2 * g_trace.n], s);
}
inline void trace_after(const char* what, cudaStream_t s) {
  if (g_trace.on && g_trace.n < g_trace.cap) {
    trace_record(g_trace.ev[2 * g_trace.n + 1], s);
    g_trace.name[g_trace.n] = what;
    ++g_trace.n;
  }
}

// Auxiliary streams per device: 0 runs the g_w branch, 1 the HQ of w, 2 the
// host-to-device and 3 the device-to-host copies of hlq_layer_step_host.
// Created on first use, kept for the process.
constexpr int kAuxStreams = 5;
cudaStream_t g_aux_stream[kMaxDevices][kAuxStreams] = {};
std::mutex g_aux_mutex;

cudaStream_t aux_stream(int which) {
  int dev = 0;
  if (which < 0 || which >= kAuxStreams) return nullptr;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lock(g_aux_mutex);
  if (!g_aux_stream[dev][which]) {
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess)
      return nullptr;
    g_aux_stream[dev][which] = st;
  }
  return g_aux_stream[dev][which];
}

// hlq_debug_serialize_branches: every branch of the device entries on the
// caller's stream, one after the other (for per-kernel timing).
std::atomic<bool> g_serial_branches{false};

// The stream a branch of a device entry runs on: a library stream forked
// from the caller's, or the caller's own when branches are serialised.
cudaStream_t branch_stream(int which, cudaStream_t caller, bool serial) {
  return serial ? caller : aux_stream(which);
}

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

// Workspace layouts (offsets in bytes from ws).
struct GxLayout {
  size_t amax, sgy, sw, qy, qw, total;
};
struct GwLayout {
  size_t amax, sg, qg, xw, split, total;
  int64_t ld;   // row stride (codes) of the fp16 operand buffers
  int64_t ld8;  // row stride of the HLA codes of g_y when they are kept int8
};

GxLayout gx_layout(int64_t T, int64_t Cin, int64_t Cout) {
  GxLayout L{};
  size_t o = 0;
  L.amax = o; o += kAlign;                                   // 2 amax slots
  L.sw = o;   o += kAlign;                                   // s_w
  L.sgy = o;  o += align_up((size_t)(T > 0 ? T : 1) * 4);    // s_gy
  L.qy = o;   o += align_up((size_t)T * (size_t)Cout);       // E4M3 [T, Cout]
  L.qw = o;   o += align_up((size_t)Cin * (size_t)Cout);     // E4M3 [Cin, Cout]
  L.total = o;
  return L;
}

GwLayout gw_layout(int64_t T, int64_t Cin, int64_t Cout, int rank) {
  GwLayout L{};
  const int64_t Tp = T / 16 * rank;
  L.ld = (Tp + 7) / 8 * 8;     // 16-byte rows for the TMA
  L.ld8 = (Tp + 15) / 16 * 16;  // the same for int8 rows (ld8 <= 2 ld)
  size_t o = 0;
  L.amax = o;  o += kAlign;
  L.sg = o;    o += kAlign;
  L.qg = o;    o += align_up((size_t)Cout * (size_t)L.ld * 2);  // fp16 [Cout, ld] or int8 [Cout, ld8]
  L.xw = o;    o += align_up((size_t)Cin * (size_t)L.ld * 2);   // fp16 [Cin, ld]
  L.split = o; o += align_up(gemm_tc_split_ws_bytes(Cout, Cin)); // int32 split-K
  L.total = o;
  return L;
}

// Workspace of the g_x HLA ablation: two amax slots, the two scales, fp16
// codes of g_y [T, ld] and of w [Cin, ld] (ld = Cout' rounded up to 8 codes
// for 16-byte rows).
struct GxHlaLayout {
  size_t amax, s, qg, qw, total;
  int64_t ld;
};
GxHlaLayout gx_hla_layout(int64_t T, int64_t Cin, int64_t Cout, int rank) {
  GxHlaLayout L{};
  const int64_t Kp = Cout / 16 * rank;
  L.ld = (Kp + 7) / 8 * 8;
  size_t o = 0;
  L.amax = o; o += kAlign;
  L.s = o;    o += kAlign;
  L.qg = o;   o += align_up((size_t)T * (size_t)L.ld * 2);
  L.qw = o;   o += align_up((size_t)Cin * (size_t)L.ld * 2);
  L.total = o;
  return L;
}

int device_sm_count() {
  static int count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (!count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    count[dev] = n;
  }
  return count[dev];
}

// amax slot(s): one for the tensor, or one per channel
size_t compress_ws(int64_t, int64_t Cin) {
  return kAlign + align_up((size_t)(Cin > 0 ? Cin : 0) * 4);
}

bool rank_ok(int rank) {
  return rank == 1 || rank == 2 || rank == 4 || rank == 8 || rank == 16;
}

// Format of the ACBP buffer: code bits 8 (int8 codes [Cin, T']) or 4 (int4
// codes packed two per byte [Cin, T'/2], even ranks only), optionally with
// HLQ_XBAR_PER_CHANNEL (scales [Cin] instead of [1]).
inline int xbar_code_bits(int fmt) { return fmt & 0xff; }
inline bool xbar_per_channel(int fmt) { return (fmt & HLQ_XBAR_PER_CHANNEL) != 0; }
hlq_status xbar_fmt_check(int fmt, int rank) {
  if (fmt & ~(0xff | HLQ_XBAR_PER_CHANNEL)) return HLQ_ERR_INVALID_ARG;
  const int bits = xbar_code_bits(fmt);
  if (bits != 8 && bits != 4) return HLQ_ERR_INVALID_ARG;
  if (bits == 4 && rank < 2) return HLQ_ERR_UNSUPPORTED;
  return HLQ_OK;
}

hlq_status check_common(int dt, int64_t T, int64_t Cin, int64_t Cout,
                        int block) {
  if (dt != HLQ_F32 && dt != HLQ_BF16) return HLQ_ERR_INVALID_ARG;
  if (block != 16) return HLQ_ERR_INVALID_ARG;
  if (T < 0 || Cin < 0 || Cout < 0) return HLQ_ERR_SHAPE;
  if (T % 16 || Cin % 16 || Cout % 16) return HLQ_ERR_SHAPE;
  // grid limits of the transform kernels: T/256 and Cout/16 index grid.y
  if (T > (int64_t)256 * 65535 || Cout > (int64_t)16 * 65535 ||
      Cin > ((int64_t)1 << 24))
    return HLQ_ERR_UNSUPPORTED;
  return HLQ_OK;
}


#define HLQ_TRY(expr)                                  \
  do {                                                 \
    cudaError_t _e = (expr);                           \
    if (_e != cudaSuccess) return HLQ_ERR_CUDA;        \
  } while (0)

// A kernel launch: traced when tracing is on.
#define HLQ_LAUNCH(name, s, expr)                      \
  do {                                                 \
    trace_before(s);                                   \
    cudaError_t _e = (expr);                           \
    if (_e != cudaSuccess) return HLQ_ERR_CUDA;        \
    trace_after(name, s);                              \
  } while (0)

// HQ of w (amax pass, then quantization to transposed E4M3 codes).
hlq_status hq_w_launches(const void* w, bool bf16, int64_t Cout, int64_t Cin,
                         unsigned int* amax, uint8_t* qw, float* sw, int rnd, uint64_t seed,
                         unsigned int* status, cudaStream_t s) {
  HLQ_LAUNCH("hq_cols_amax", s,
             launch_hq_cols(w, bf16, Cout, Cin, true, amax, nullptr, nullptr, rnd, seed, 1,
                            status, s));
  HLQ_LAUNCH("hq_cols_quant", s,
             launch_hq_cols(w, bf16, Cout, Cin, false, amax, qw, sw, rnd, seed, 1, status,
                            s));
  return HLQ_OK;
}

// HQ of g_y (an amax pass first for a per-tensor scale).
hlq_status hq_gy_launches(const void* gy, bool bf16, int64_t T, int64_t Cout, bool per_token,
                          unsigned int* amax, uint8_t* qy, float* sgy, int rnd,
                          uint64_t seed, unsigned int* status, cudaStream_t s) {
  if (!per_token)
    HLQ_LAUNCH("hq_rows_amax", s,
               launch_hq_rows(gy, bf16, T, Cout, false, true, amax, nullptr, nullptr, rnd,
                              seed, 0, status, s));
  HLQ_LAUNCH("hq_rows_quant", s,
             launch_hq_rows(gy, bf16, T, Cout, per_token, false, amax, qy, sgy, rnd, seed, 0,
                            status, s));
  return HLQ_OK;
}

hlq_status gx_impl(const void* gy, const void* w, int dt, int64_t T,
                   int64_t Cin, int64_t Cout, int block, int gran_gy,
                   int gran_w, int rnd, uint64_t seed, float* gx, void* ws,
                   size_t ws_bytes, int8_t* dbg_qgy, float* dbg_sgy,
                   int8_t* dbg_qw, float* dbg_sw, int32_t* dbg_acc,
                   void* stream, bool validate_only = false,
                   cudaStream_t w_stream = nullptr, uint8_t* dbg_qgy_packed = nullptr,
                   uint8_t* dbg_qw_packed = nullptr) {
  hlq_status st = check_common(dt, T, Cin, Cout, block);
  if (st != HLQ_OK) return st;
  if (gran_gy != HLQ_PER_TENSOR && gran_gy != HLQ_PER_TOKEN) return HLQ_ERR_INVALID_ARG;
  if (gran_w != HLQ_PER_TENSOR && gran_w != HLQ_PER_TOKEN) return HLQ_ERR_INVALID_ARG;
  if (gran_w != HLQ_PER_TENSOR) return HLQ_ERR_UNSUPPORTED;
  if (rnd != HLQ_RNE && rnd != HLQ_SR) return HLQ_ERR_INVALID_ARG;
  const int64_t n_gx = T * Cin;
  if (n_gx > 0 && !gx) return HLQ_ERR_INVALID_ARG;
  if (T * Cout > 0 && !gy) return HLQ_ERR_INVALID_ARG;
  if (Cout * Cin > 0 && !w) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(gy) || !aligned16(w) || !aligned16(gx)) return HLQ_ERR_ALIGN;
  // |acc| <= 49 * Cout must stay exact through an fp32 accumulator
  if (49 * Cout >= ((int64_t)1 << 24)) return HLQ_ERR_OVERFLOW;
  const GxLayout L = gx_layout(T, Cin, Cout);
  if (!ws || ws_bytes < L.total) return HLQ_ERR_WORKSPACE;
  if (!aligned256(ws)) return HLQ_ERR_ALIGN;
  if (validate_only) return HLQ_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n_gx == 0) return HLQ_OK;
  if (Cout == 0) {  // empty contraction: g_x = 0
    HLQ_TRY(cudaMemsetAsync(gx, 0, (size_t)n_gx * 4, s));
    if (dbg_acc) HLQ_TRY(cudaMemsetAsync(dbg_acc, 0, (size_t)n_gx * 4, s));
    return HLQ_OK;
  }
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(ws);
  unsigned int* amax = reinterpret_cast<unsigned int*>(base + L.amax);
  float* sgy = reinterpret_cast<float*>(base + L.sgy);
  float* sw = reinterpret_cast<float*>(base + L.sw);
  uint8_t* qy = base + L.qy;
  uint8_t* qw = base + L.qw;
  const bool bf16 = dt == HLQ_BF16;
  const bool per_token = gran_gy == HLQ_PER_TOKEN;

  // amax[0]: g_y, amax[1]: w
  HLQ_TRY(cudaMemsetAsync(amax, 0, 8, s));
  // HQ of w: on `w_stream` when given (forked here, joined before the GEMM),
  // so that the small, latency-bound transform of w overlaps the HQ of g_y
  cudaStream_t sw_st = s;
  cudaEvent_t w_fork = nullptr, w_done = nullptr;
  if (w_stream && w_stream != s) {
    if (cudaEventCreateWithFlags(&w_fork, cudaEventDisableTiming) != cudaSuccess)
      return HLQ_ERR_CUDA;
    if (cudaEventCreateWithFlags(&w_done, cudaEventDisableTiming) != cudaSuccess) {
      cudaEventDestroy(w_fork);
      return HLQ_ERR_CUDA;
    }
    sw_st = w_stream;
  }
  hlq_status r = HLQ_OK;
  if (w_fork && (cudaEventRecord(w_fork, s) != cudaSuccess ||
                 cudaStreamWaitEvent(sw_st, w_fork, 0) != cudaSuccess))
    r = HLQ_ERR_CUDA;
  if (r == HLQ_OK)
    r = hq_w_launches(w, bf16, Cout, Cin, amax + 1, qw, sw, rnd, seed, status, sw_st);
  if (r == HLQ_OK)
    r = hq_gy_launches(gy, bf16, T, Cout, per_token, amax, qy, sgy, rnd, seed, status, s);
  if (w_fork) {  // join even after a failure: `s` never runs ahead of `w_stream`
    if (cudaEventRecord(w_done, sw_st) != cudaSuccess ||
        cudaStreamWaitEvent(s, w_done, 0) != cudaSuccess)
      r = HLQ_ERR_CUDA;
    cudaEventDestroy(w_fork);
    cudaEventDestroy(w_done);
  }
  if (r != HLQ_OK) return r;
  const int sms = device_sm_count();
  if (sms <= 0) return HLQ_ERR_CUDA;
  const GemmPlan plan = plan_gemm_tc(0, T, Cin, Cout, sms, 1);
  HLQ_LAUNCH("gemm_gx_tc", s,
             launch_gemm_tc(0, qy, Cout, qw, Cout, T, Cin, Cout, plan, sgy,
                            per_token, sw, gx, dbg_acc, nullptr, status, s));
  if (dbg_qgy) HLQ_TRY(launch_decode_e4m3(qy, dbg_qgy, T * Cout, s));
  if (dbg_qw) HLQ_TRY(launch_decode_e4m3(qw, dbg_qw, Cin * Cout, s));
  if (dbg_qgy_packed) HLQ_TRY(launch_pack_e4m3_int4(qy, dbg_qgy_packed, T * Cout, s));
  if (dbg_qw_packed) HLQ_TRY(launch_pack_e4m3_int4(qw, dbg_qw_packed, Cin * Cout, s));
  if (dbg_sgy)
    HLQ_TRY(cudaMemcpyAsync(dbg_sgy, sgy, (size_t)(per_token ? T : 1) * 4,
                            cudaMemcpyDeviceToDevice, s));
  if (dbg_sw) HLQ_TRY(cudaMemcpyAsync(dbg_sw, sw, 4, cudaMemcpyDeviceToDevice, s));
  return HLQ_OK;
}

// ACBP: HLA of x along tokens, per-tensor amax pass, int8 codes [Cin, T'] or
// packed int4 codes (4 code bits); per-channel scales with HLQ_XBAR_PER_CHANNEL.
hlq_status compress_launches(const void* x, bool bf16, int64_t T, int64_t Cin, int rank,
                             int fmt, int8_t* xbar, float* xscale, unsigned int* amax,
                             unsigned int* status, cudaStream_t s) {
  const int64_t Tp = T / 16 * rank;
  const bool per_ch = xbar_per_channel(fmt);
  const int out = xbar_code_bits(fmt) == 4 ? kHlaOutI4 : kHlaOutI8;
  HLQ_TRY(cudaMemsetAsync(amax, 0, (size_t)(per_ch ? Cin : 1) * 4, s));
  HLQ_LAUNCH("hla_x_amax", s,
             launch_hla(x, bf16, T, Cin, rank, true, kHlaOutI8, amax, nullptr, 0, nullptr,
                        status, s, per_ch));
  HLQ_LAUNCH("hla_x_quant", s,
             launch_hla(x, bf16, T, Cin, rank, false, out, amax, xbar, Tp, xscale, status, s,
                        per_ch));
  return HLQ_OK;
}

// How the g_w GEMM takes its operands (hlq_set_gw_operands): kRawB when it
// reads the int8 x-bar itself, kRawA when the HLA codes of g_y stay int8 too.
// The in-GEMM widening takes int8 x-bar whose rows are whole 16-byte runs
// from a 16-byte aligned base; anything else goes through the widening
// kernel.  The fused reader writes fp16 HLA codes (fused = true).
std::atomic<int> g_gw_operands{HLQ_GW_AUTO};

int gw_raw(int fmt, int64_t Tp, const void* xbar, bool fused) {
  // the default widens x-bar with its own kernel: measured on GB300, the
  // g_w GEMM that widens int8 tiles in shared memory (its epilogue warps
  // convert each stage before the MMA may read it) ran 1669 us at Llama
  // down_proj against 489 + 68 (widening kernel) us, and 62.6 against
  // 41.8 + 9.7 us at ViT-B qkv; both operands int8: 2214 and 73.7 us
  int mode = g_gw_operands.load();
  if (mode == HLQ_GW_AUTO) mode = HLQ_GW_WIDEN;
  if (mode == HLQ_GW_WIDEN || xbar_code_bits(fmt) != 8 || Tp % 16 != 0 || !aligned16(xbar))
    return 0;
  return (mode == HLQ_GW_INT8_BOTH && !fused) ? (kRawA | kRawB) : kRawB;
}

// HLA of g_y: per-tensor amax pass, then int8 codes stored as fp16 [Cout, ld]
// or, with i8, as int8 [Cout, ld8].
hlq_status hla_gy_launches(const void* gy, bool bf16, int64_t T, int64_t Cout, int rank,
                           unsigned int* amax, void* qg, int64_t ld, float* sg,
                           unsigned int* status, cudaStream_t s, bool i8 = false) {
  HLQ_TRY(cudaMemsetAsync(amax, 0, 4, s));
  HLQ_LAUNCH("hla_gy_amax", s,
             launch_hla(gy, bf16, T, Cout, rank, true, kHlaOutF16, amax, nullptr, 0, nullptr,
                        status, s));
  HLQ_LAUNCH("hla_gy_quant", s,
             launch_hla(gy, bf16, T, Cout, rank, false, i8 ? kHlaOutI8 : kHlaOutF16, amax, qg,
                        ld, sg, status, s));
  return HLQ_OK;
}

// ACBP buffer widened to bf16, then the g_w GEMM with its dequantization.
// `after`: an event (the g_x GEMM's end, on another stream) that the GEMM
// must follow, or null.  Both GEMMs are persistent grids of one CTA per SM
// whose tiles are dealt out in advance; run side by side when each fills
// the GPU alone, the later grid's CTAs wait for SMs while their tiles pile
// up (Llama down_proj: 2497 us per step against 2219 us in sequence), while
// smaller ones gain from sharing the SMs (ViT-B qkv: 190.6 us side by side,
// 195.7 in sequence): see gemms_in_sequence.
// Whether the g_w GEMM must follow the g_x GEMM (g_x GEMM over Mx rows):
// only when each one alone has at least one unit per SM, so that running
// them side by side cannot fill idle SMs and only delays the later grid.
bool gemms_in_sequence_on(int64_t Mx, int64_t Cin, int64_t Cout, int64_t Tp, int sms) {
  if (sms <= 0) return false;
  auto units = [](const GemmPlan& p, int64_t M, int64_t N) {  // CTAs' worth of work
    const int64_t tm = p.pair ? 2 * ((M + 255) / 256) : (M + 127) / 128;
    return tm * ((N + p.bn - 1) / p.bn) * p.splits;
  };
  const GemmPlan px = plan_gemm_tc(0, Mx, Cin, Cout, sms, 1);
  const GemmPlan pw = plan_gemm_tc(1, Cout, Cin, Tp, sms, 16);
  return units(px, Mx, Cin) >= sms && units(pw, Cout, Cin) >= sms;
}
bool gemms_in_sequence(int64_t Mx, int64_t Cin, int64_t Cout, int64_t Tp) {
  return gemms_in_sequence_on(Mx, Cin, Cout, Tp, device_sm_count());
}

// The g_w GEMM over the HLA codes of g_y (fp16, or int8 with kRawA in raw)
// and x-bar: read as int8 by the GEMM (kRawB in raw), or first widened to
// fp16 in the workspace.
hlq_status gw_gemm_launches(const int8_t* xbar, int fmt, const float* xscale, int64_t Cin,
                            int64_t Cout, int64_t Tp, const GwLayout& L, uint8_t* base,
                            float* gw, int32_t* dbg_acc, unsigned int* status,
                            cudaStream_t s, cudaEvent_t after, int raw,
                            cudaEvent_t after2 = nullptr) {
  void* xw = base + L.xw;
  const float* sg = reinterpret_cast<const float*>(base + L.sg);
  if (!(raw & kRawB)) {
    if (xbar_code_bits(fmt) == 4)
      HLQ_LAUNCH("widen_xbar", s,
                 launch_widen_i4_f16(reinterpret_cast<const uint8_t*>(xbar), xw, Cin, Tp, L.ld,
                                     s));
    else
      HLQ_LAUNCH("widen_xbar", s, launch_widen_i8_f16(xbar, xw, Cin, Tp, L.ld, s));
  }
  const int sms = device_sm_count();
  if (sms <= 0) return HLQ_ERR_CUDA;
  const GemmPlan plan = plan_gemm_tc(1, Cout, Cin, Tp, sms, 16);
  if (after) HLQ_TRY(cudaStreamWaitEvent(s, after, 0));
  if (after2) HLQ_TRY(cudaStreamWaitEvent(s, after2, 0));
  const void* b = (raw & kRawB) ? static_cast<const void*>(xbar) : xw;
  const int64_t ldb = (raw & kRawB) ? Tp : L.ld;
  const int64_t lda = (raw & kRawA) ? L.ld8 : L.ld;
  HLQ_LAUNCH("gemm_gw_tc", s,
             launch_gemm_tc(1, base + L.qg, lda, b, ldb, Cout, Cin, Tp, plan, sg, false, xscale,
                            gw, dbg_acc, base + L.split, status, s, xbar_per_channel(fmt),
                            raw));
  return HLQ_OK;
}

hlq_status gw_impl(const void* gy, int dt, const int8_t* xbar, int fmt,
                   const float* xscale, int64_t T, int64_t Cin, int64_t Cout,
                   int block, int rank, float* gw, void* ws, size_t ws_bytes,
                   int8_t* dbg_qg, float* dbg_sg, int32_t* dbg_acc,
                   void* stream, bool validate_only = false,
                   cudaEvent_t gemm_after = nullptr, cudaEvent_t hla_ready = nullptr,
                   int raw_given = -1) {
  // hla_ready: the HLA of g_y was enqueued elsewhere (into this workspace, in
  // the format of raw_given, the caller's gw_raw) and completes at that event
  hlq_status st = check_common(dt, T, Cin, Cout, block);
  if (st != HLQ_OK) return st;
  if (!rank_ok(rank)) return HLQ_ERR_INVALID_ARG;
  st = xbar_fmt_check(fmt, rank);
  if (st != HLQ_OK) return st;
  const int64_t Tp = T / 16 * rank;
  const int64_t n_gw = Cout * Cin;
  if (n_gw > 0 && !gw) return HLQ_ERR_INVALID_ARG;
  if (T * Cout > 0 && !gy) return HLQ_ERR_INVALID_ARG;
  if (Cin * Tp > 0 && !xbar) return HLQ_ERR_INVALID_ARG;
  if (!xscale) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(gy) || !aligned16(xbar) || !aligned16(gw)) return HLQ_ERR_ALIGN;
  // |acc| <= T' * 127 * qmax_x must stay below 2^31
  if (Tp * 127 * (xbar_code_bits(fmt) == 4 ? 7 : 127) >= ((int64_t)1 << 31))
    return HLQ_ERR_OVERFLOW;
  const GwLayout L = gw_layout(T, Cin, Cout, rank);
  if (!ws || ws_bytes < L.total) return HLQ_ERR_WORKSPACE;
  if (!aligned256(ws)) return HLQ_ERR_ALIGN;
  if (validate_only) return HLQ_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n_gw == 0) return HLQ_OK;
  if (Tp == 0) {  // no tokens: g_w = 0
    HLQ_TRY(cudaMemsetAsync(gw, 0, (size_t)n_gw * 4, s));
    if (dbg_acc) HLQ_TRY(cudaMemsetAsync(dbg_acc, 0, (size_t)n_gw * 4, s));
    return HLQ_OK;
  }
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(ws);
  unsigned int* amax = reinterpret_cast<unsigned int*>(base + L.amax);
  float* sg = reinterpret_cast<float*>(base + L.sg);
  void* qg = base + L.qg;
  const bool bf16 = dt == HLQ_BF16;

  const int raw = raw_given >= 0 ? raw_given : gw_raw(fmt, Tp, xbar, false);
  const bool qg_i8 = (raw & kRawA) != 0;
  if (!hla_ready) {
    st = hla_gy_launches(gy, bf16, T, Cout, rank, amax, qg, qg_i8 ? L.ld8 : L.ld, sg, status,
                         s, qg_i8);
    if (st != HLQ_OK) return st;
  }
  st = gw_gemm_launches(xbar, fmt, xscale, Cin, Cout, Tp, L, base, gw, dbg_acc, status, s,
                        gemm_after, raw, hla_ready);
  if (st != HLQ_OK) return st;
  if (dbg_qg && qg_i8)
    HLQ_TRY(cudaMemcpy2DAsync(dbg_qg, (size_t)Tp, qg, (size_t)L.ld8, (size_t)Tp, (size_t)Cout,
                              cudaMemcpyDeviceToDevice, s));
  else if (dbg_qg)
    HLQ_TRY(launch_decode_f16(qg, dbg_qg, Cout, Tp, L.ld, s));
  if (dbg_sg) HLQ_TRY(cudaMemcpyAsync(dbg_sg, sg, 4, cudaMemcpyDeviceToDevice, s));
  return HLQ_OK;
}


// Workspace of hlq_layer_step_host: device copies of the inputs and outputs,
// then the workspaces of the compression and of the two gradient branches.
struct StepLayout {
  size_t x, gy, w, gx, gw, cws, gxws, gwws, total;
};

StepLayout step_layout(int dt, int64_t T, int64_t Cin, int64_t Cout, int rank) {
  const size_t esz = dt == HLQ_BF16 ? 2 : 4;
  StepLayout L{};
  size_t o = 0;
  L.x = o;    o += align_up((size_t)T * (size_t)Cin * esz);
  L.gy = o;   o += align_up((size_t)T * (size_t)Cout * esz);
  L.w = o;    o += align_up((size_t)Cout * (size_t)Cin * esz);
  L.gx = o;   o += align_up((size_t)T * (size_t)Cin * 4);
  L.gw = o;   o += align_up((size_t)Cout * (size_t)Cin * 4);
  L.cws = o;  o += align_up(compress_ws(T, Cin));
  L.gxws = o; o += gx_layout(T, Cin, Cout).total;
  L.gwws = o; o += gw_layout(T, Cin, Cout, rank).total;
  L.total = o;
  return L;
}

// At most this many token chunks of g_y per hlq_layer_step_host call.
constexpr int kMaxHostChunks = 64;

// Events of one hlq_layer_step_host call (destroyed when it returns; the
// runtime keeps pending ones alive until they complete): six for the
// streams' hand-offs and two per chunk of g_y.
struct EventSet {
  static constexpr int kCap = 6 + 3 * kMaxHostChunks;
  cudaEvent_t ev[kCap] = {};
  int n = 0;
  cudaEvent_t make() {
    if (n >= kCap) return nullptr;
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    ev[n++] = e;
    return e;
  }
  ~EventSet() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
  }
};

}  // namespace

size_t gx_workspace_bytes(int64_t T, int64_t Cin, int64_t Cout) {
  return gx_layout(T, Cin, Cout).total;
}

hlq_status backward_gx_with_ws(const void* gy, const void* w, int dt, int64_t T,
                               int64_t Cin, int64_t Cout, int block, int gran_gy,
                               int gran_w, int rnd, uint64_t seed, float* gx,
                               void* ws, size_t ws_bytes, void* stream) {
  return gx_impl(gy, w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd, seed, gx, ws,
                 ws_bytes, nullptr, nullptr, nullptr, nullptr, nullptr, stream);
}

}  // namespace hlq

using namespace hlq;

extern "C" {

size_t hlq_workspace_bytes(int op, int64_t T, int64_t Cin, int64_t Cout,
                           int block, int rank) {
  (void)block;
  if (T < 0 || Cin < 0 || Cout < 0) return 0;
  switch (op) {
    case HLQ_OP_COMPRESS_ACTIVATION:
      return compress_ws(T, Cin);
    case HLQ_OP_BACKWARD_GX:
      return gx_layout(T, Cin, Cout).total;
    case HLQ_OP_BACKWARD_GW:
      return gw_layout(T, Cin, Cout, rank_ok(rank) ? rank : 16).total;
    case HLQ_OP_BACKWARD:
      return gx_layout(T, Cin, Cout).total +
             gw_layout(T, Cin, Cout, rank_ok(rank) ? rank : 16).total;
    case HLQ_OP_SELECT_GRANULARITY:
      return kAlign;  // amax slot at 0, two fp64 sums at 16
    case HLQ_OP_ABLATION_GW_HQ:
      // amax slots, the two scales, codes [Cout, T] and [Cin, T]
      return 2 * kAlign + align_up((size_t)Cout * (size_t)T) + align_up((size_t)Cin * (size_t)T);
    case HLQ_OP_ABLATION_GX_HLA:
      return gx_hla_layout(T, Cin, Cout, rank_ok(rank) ? rank : 16).total;
    case HLQ_OP_LAYER_STEP:  // compression, then both layouts
      return compress_ws(T, Cin) + gx_layout(T, Cin, Cout).total +
             gw_layout(T, Cin, Cout, rank_ok(rank) ? rank : 16).total;
    case HLQ_OP_BACKWARD_FUSED:  // both layouts and one amax slot per token
      return gx_layout(T, Cin, Cout).total +
             gw_layout(T, Cin, Cout, rank_ok(rank) ? rank : 16).total +
             align_up((size_t)(T > 0 ? T : 1) * 4);
    default:
      return 0;
  }
}

hlq_status hlq_compress_activation(const void* d_x, int dt, int64_t T,
                                   int64_t Cin, int block, int rank, int xbar_fmt,
                                   int8_t* d_xbar, float* d_xbar_scale,
                                   void* d_ws, size_t ws_bytes, void* stream) {
  hlq_status st = check_common(dt, T, Cin, 16, block);
  if (st != HLQ_OK) return st;
  if (!rank_ok(rank)) return HLQ_ERR_INVALID_ARG;
  st = xbar_fmt_check(xbar_fmt, rank);
  if (st != HLQ_OK) return st;
  const int64_t Tp = T / 16 * rank;
  if (!d_xbar_scale) return HLQ_ERR_INVALID_ARG;
  if (Cin * Tp > 0 && (!d_x || !d_xbar)) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_x) || !aligned16(d_xbar)) return HLQ_ERR_ALIGN;
  if (!d_ws || ws_bytes < compress_ws(T, Cin)) return HLQ_ERR_WORKSPACE;
  if (!aligned256(d_ws)) return HLQ_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Cin * Tp == 0) {
    const int64_t n_scales = xbar_per_channel(xbar_fmt) ? Cin : 1;
    if (n_scales > 0) HLQ_TRY(cudaMemsetAsync(d_xbar_scale, 0, (size_t)n_scales * 4, s));
    return HLQ_OK;
  }
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  return compress_launches(d_x, dt == HLQ_BF16, T, Cin, rank, xbar_fmt, d_xbar,
                           d_xbar_scale, static_cast<unsigned int*>(d_ws), status, s);
}

hlq_status hlq_linear_backward(const void* d_gy, const void* d_w, const int8_t* d_xbar,
                               const float* d_xbar_scale, int dt, int64_t T,
                               int64_t Cin, int64_t Cout, int block, int rank,
                               int xbar_fmt, int gran_gy, int gran_w, int rnd, uint64_t seed,
                               float* d_gx, float* d_gw, void* d_ws, size_t ws_bytes,
                               void* stream) {
  hlq_status st = check_common(dt, T, Cin, Cout, block);
  if (st != HLQ_OK) return st;
  if (!rank_ok(rank)) return HLQ_ERR_INVALID_ARG;
  const size_t gx_bytes = gx_layout(T, Cin, Cout).total;
  const size_t gw_bytes = gw_layout(T, Cin, Cout, rank).total;
  if (!d_ws || ws_bytes < gx_bytes + gw_bytes) return HLQ_ERR_WORKSPACE;
  if (!aligned256(d_ws)) return HLQ_ERR_ALIGN;
  uint8_t* base = static_cast<uint8_t*>(d_ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool serial = g_serial_branches.load();  // one reading per call
  cudaStream_t a = branch_stream(0, s, serial), aw = branch_stream(1, s, serial);
  if (!serial && (!a || !aw)) return HLQ_ERR_CUDA;  // (null: the legacy stream)
  // validate both branches before forking (nothing enqueued on failure)
  st = gw_impl(d_gy, dt, d_xbar, xbar_fmt, d_xbar_scale, T, Cin, Cout, block, rank, d_gw,
               base + gx_bytes, gw_bytes, nullptr, nullptr, nullptr, nullptr,
               /*validate_only=*/true);
  if (st != HLQ_OK) return st;
  st = gx_impl(d_gy, d_w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd, seed, d_gx,
               base, gx_bytes, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
               /*validate_only=*/true);
  if (st != HLQ_OK) return st;
  cudaEvent_t fork = nullptr, join = nullptr;
  if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess)
    return HLQ_ERR_CUDA;
  if (cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
    cudaEventDestroy(fork);
    return HLQ_ERR_CUDA;
  }
  cudaEvent_t gx_done = nullptr;
  if (cudaEventCreateWithFlags(&gx_done, cudaEventDisableTiming) != cudaSuccess) {
    cudaEventDestroy(fork);
    cudaEventDestroy(join);
    return HLQ_ERR_CUDA;
  }
  hlq_status r = HLQ_OK;
  if (cudaEventRecord(fork, s) != cudaSuccess || cudaStreamWaitEvent(a, fork, 0) != cudaSuccess)
    r = HLQ_ERR_CUDA;
  if (r == HLQ_OK)  // g_x branch on the caller's stream, its HQ of w on a third
    r = gx_impl(d_gy, d_w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd, seed, d_gx,
                base, gx_bytes, nullptr, nullptr, nullptr, nullptr, nullptr, stream,
                false, aw);
  if (r == HLQ_OK && cudaEventRecord(gx_done, s) != cudaSuccess) r = HLQ_ERR_CUDA;
  if (r == HLQ_OK)  // g_w branch on the auxiliary stream (its GEMM maybe after g_x's)
    r = gw_impl(d_gy, dt, d_xbar, xbar_fmt, d_xbar_scale, T, Cin, Cout, block, rank, d_gw,
                base + gx_bytes, gw_bytes, nullptr, nullptr, nullptr, a, false,
                gemms_in_sequence(T, Cin, Cout, T / 16 * rank) ? gx_done : nullptr);
  // join even after a failure, so the caller's stream never runs ahead of
  // work already enqueued on the auxiliary stream
  if (cudaEventRecord(join, a) != cudaSuccess || cudaStreamWaitEvent(s, join, 0) != cudaSuccess)
    r = HLQ_ERR_CUDA;
  cudaEventDestroy(fork);
  cudaEventDestroy(join);
  cudaEventDestroy(gx_done);
  return r;
}

// The ACBP compression of x and both gradients in one call, from device
// buffers: the compression runs first on the g_w branch (the only one that
// needs the stored activation), so it overlaps the HQ of g_y and the g_x
// GEMM on the caller's stream; the HQ of w runs on a third stream.  Same
// bits as hlq_compress_activation followed by hlq_linear_backward.
static hlq_status fused_launches(const void* d_gy, const void* d_w, const void* d_x, int8_t* d_xbar,
                          float* d_xbar_scale, int dt, int64_t T, int64_t Cin, int64_t Cout,
                          int rank, int xbar_fmt, int gran_gy, int rnd, uint64_t seed,
                          float* d_gx, float* d_gw, uint8_t* gxb, uint8_t* gwb,
                          unsigned int* amax_rows, unsigned int* x_amax, cudaStream_t s);

hlq_status hlq_layer_step(const void* d_x, const void* d_gy, const void* d_w, int dt,
                          int64_t T, int64_t Cin, int64_t Cout, int block, int rank,
                          int xbar_fmt, int gran_gy, int gran_w, int rnd, uint64_t seed,
                          float* d_gx, float* d_gw, int8_t* d_xbar, float* d_xbar_scale,
                          void* d_ws, size_t ws_bytes, void* stream) {
  hlq_status st = check_common(dt, T, Cin, Cout, block);
  if (st != HLQ_OK) return st;
  if (!rank_ok(rank)) return HLQ_ERR_INVALID_ARG;
  st = xbar_fmt_check(xbar_fmt, rank);
  if (st != HLQ_OK) return st;
  const int64_t Tp = T / 16 * rank;
  if (!d_xbar_scale) return HLQ_ERR_INVALID_ARG;
  if (Cin * Tp > 0 && (!d_x || !d_xbar)) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_x) || !aligned16(d_xbar)) return HLQ_ERR_ALIGN;
  const size_t c_bytes = compress_ws(T, Cin);
  const size_t gx_bytes = gx_layout(T, Cin, Cout).total;
  const size_t gw_bytes = gw_layout(T, Cin, Cout, rank).total;
  if (!d_ws || ws_bytes < c_bytes + gx_bytes + gw_bytes) return HLQ_ERR_WORKSPACE;
  if (!aligned256(d_ws)) return HLQ_ERR_ALIGN;
  uint8_t* base = static_cast<uint8_t*>(d_ws);
  uint8_t* gxb = base + c_bytes;
  uint8_t* gwb = gxb + gx_bytes;
  st = gw_impl(d_gy, dt, d_xbar, xbar_fmt, d_xbar_scale, T, Cin, Cout, block, rank, d_gw, gwb,
               gw_bytes, nullptr, nullptr, nullptr, nullptr, /*validate_only=*/true);
  if (st != HLQ_OK) return st;
  st = gx_impl(d_gy, d_w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd, seed, d_gx, gxb,
               gx_bytes, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
               /*validate_only=*/true);
  if (st != HLQ_OK) return st;
  if (T * Cin * Cout == 0) {  // degenerate sizes: the separate calls, in order
    st = hlq_compress_activation(d_x, dt, T, Cin, block, rank, xbar_fmt, d_xbar,
                                 d_xbar_scale, base, c_bytes, stream);
    if (st != HLQ_OK) return st;
    return hlq_linear_backward(d_gy, d_w, d_xbar, d_xbar_scale, dt, T, Cin, Cout, block, rank,
                               xbar_fmt, gran_gy, gran_w, rnd, seed, d_gx, d_gw, gxb,
                               gx_bytes + gw_bytes, stream);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // a per-tensor scale for g_y: one fused reader of g_y for both paths (two
  // passes over g_y instead of four; ViT-B fc2: 27.7 -> 18.3 us of maxima and
  // 38.4 -> 37.1 us of codes, ResNet-50 im2col: 36.0 -> 22.6 and 48.9 ->
  // 44.7 us; the steps stay at 207 and 366 us, whose critical path is the
  // compression on the g_w branch), the compression on the g_w branch as
  // below.  A per-token scale keeps the two readers: the fused one
  // transforms each row twice there (Llama down_proj step 1820 against
  // 1768 us).
  if (gran_gy == HLQ_PER_TENSOR)
    return fused_launches(d_gy, d_w, d_x, d_xbar, d_xbar_scale, dt, T, Cin, Cout, rank,
                          xbar_fmt, gran_gy, rnd, seed, d_gx, d_gw, gxb, gwb, nullptr,
                          reinterpret_cast<unsigned int*>(base), s);
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  const bool serial = g_serial_branches.load();  // one reading per call
  cudaStream_t a = branch_stream(0, s, serial), aw = branch_stream(1, s, serial);
  if (!serial && (!a || !aw)) return HLQ_ERR_CUDA;  // (null: the legacy stream)
  cudaStream_t ah = branch_stream(4, s, serial);  // the HLA of g_y
  if (!serial && !ah) return HLQ_ERR_CUDA;
  EventSet E;
  cudaEvent_t fork = E.make(), join = E.make(), gx_done = E.make(), hla_done = E.make();
  if (!fork || !join || !gx_done || !hla_done) return HLQ_ERR_CUDA;
  hlq_status r = HLQ_OK;
  if (cudaEventRecord(fork, s) != cudaSuccess || cudaStreamWaitEvent(a, fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(ah, fork, 0) != cudaSuccess)
    r = HLQ_ERR_CUDA;
  // the HLA of g_y on its own stream from the start (it needs only g_y),
  // beside the compression of x; the g_w GEMM waits for both (ViT-B qkv step
  // 191.6 -> 180.6 us, the 256-token layer 52.7 -> 44.5 us; Llama down_proj,
  // whose kernels each fill the GPU, unchanged)
  const int rw = gw_raw(xbar_fmt, Tp, d_xbar, false);
  {
    const GwLayout WL = gw_layout(T, Cin, Cout, rank);
    const bool qg_i8 = (rw & kRawA) != 0;
    if (r == HLQ_OK)
      r = hla_gy_launches(d_gy, dt == HLQ_BF16, T, Cout, rank,
                          reinterpret_cast<unsigned int*>(gwb + WL.amax), gwb + WL.qg,
                          qg_i8 ? WL.ld8 : WL.ld, reinterpret_cast<float*>(gwb + WL.sg), status,
                          ah, qg_i8);
    if (cudaEventRecord(hla_done, ah) != cudaSuccess && r == HLQ_OK) r = HLQ_ERR_CUDA;
  }
  if (r == HLQ_OK)  // g_x branch on the caller's stream, its HQ of w on a third
    r = gx_impl(d_gy, d_w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd, seed, d_gx, gxb,
                gx_bytes, nullptr, nullptr, nullptr, nullptr, nullptr, stream, false, aw);
  if (r == HLQ_OK && cudaEventRecord(gx_done, s) != cudaSuccess) r = HLQ_ERR_CUDA;
  if (r == HLQ_OK)  // g_w branch: compression of x, widening, g_w GEMM
    r = compress_launches(d_x, dt == HLQ_BF16, T, Cin, rank, xbar_fmt, d_xbar, d_xbar_scale,
                          reinterpret_cast<unsigned int*>(base), status, a);
  if (r == HLQ_OK)
    r = gw_impl(d_gy, dt, d_xbar, xbar_fmt, d_xbar_scale, T, Cin, Cout, block, rank, d_gw,
                gwb, gw_bytes, nullptr, nullptr, nullptr, a, false,
                gemms_in_sequence(T, Cin, Cout, Tp) ? gx_done : nullptr, hla_done, rw);
  // join even after a failure (the HLA stream through the g_w branch)
  if (cudaStreamWaitEvent(a, hla_done, 0) != cudaSuccess ||
      cudaEventRecord(join, a) != cudaSuccess || cudaStreamWaitEvent(s, join, 0) != cudaSuccess)
    r = HLQ_ERR_CUDA;
  return r;
}

hlq_status hlq_select_gy_granularity(const void* d_gy, int dt, int64_t T, int64_t Cout,
                                     int block, double threshold, double* d_mse,
                                     int32_t* d_choice, void* d_ws, size_t ws_bytes,
                                     void* stream) {
  hlq_status st = check_common(dt, T, 16, Cout, block);
  if (st != HLQ_OK) return st;
  if (!d_mse || !d_choice || !(threshold >= 0.0)) return HLQ_ERR_INVALID_ARG;
  if (T * Cout > 0 && !d_gy) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_gy) || reinterpret_cast<uintptr_t>(d_mse) % 8 ||
      reinterpret_cast<uintptr_t>(d_choice) % 4)
    return HLQ_ERR_ALIGN;
  if (!d_ws || ws_bytes < kAlign) return HLQ_ERR_WORKSPACE;
  if (!aligned256(d_ws)) return HLQ_ERR_ALIGN;
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(d_ws);
  unsigned int* amax = reinterpret_cast<unsigned int*>(base);
  double* sums = reinterpret_cast<double*>(base + 16);
  const bool bf16 = dt == HLQ_BF16;
  HLQ_TRY(cudaMemsetAsync(base, 0, 32, s));
  if (T * Cout > 0)
    HLQ_LAUNCH("hq_rows_amax", s,
               launch_hq_rows(d_gy, bf16, T, Cout, false, true, amax, nullptr, nullptr,
                              HLQ_RNE, 0, 0, status, s));
  HLQ_LAUNCH("hq_mse", s,
             launch_hq_mse(d_gy, bf16, T, Cout, amax, sums, threshold, d_mse, d_choice,
                           status, s));
  return HLQ_OK;
}

hlq_status hlq_ablation_gw_hq(const void* d_gy, const void* d_x, int dt, int64_t T,
                              int64_t Cin, int64_t Cout, int block, int rnd, uint64_t seed,
                              float* d_gw, int32_t* d_acc, void* d_ws, size_t ws_bytes,
                              void* stream) {
  hlq_status st = check_common(dt, T, Cin, Cout, block);
  if (st != HLQ_OK) return st;
  if (rnd != HLQ_RNE && rnd != HLQ_SR) return HLQ_ERR_INVALID_ARG;
  if ((T * Cout > 0 && !d_gy) || (T * Cin > 0 && !d_x) || (Cout * Cin > 0 && !d_gw))
    return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_gy) || !aligned16(d_x) || !aligned16(d_gw) || !aligned16(d_acc))
    return HLQ_ERR_ALIGN;
  if (49 * T >= ((int64_t)1 << 24)) return HLQ_ERR_OVERFLOW;
  const size_t need = hlq_workspace_bytes(HLQ_OP_ABLATION_GW_HQ, T, Cin, Cout, block, 8);
  if (!d_ws || ws_bytes < need) return HLQ_ERR_WORKSPACE;
  if (!aligned256(d_ws)) return HLQ_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Cout * Cin == 0) return HLQ_OK;
  if (T == 0) {  // empty contraction
    HLQ_TRY(cudaMemsetAsync(d_gw, 0, (size_t)(Cout * Cin) * 4, s));
    if (d_acc) HLQ_TRY(cudaMemsetAsync(d_acc, 0, (size_t)(Cout * Cin) * 4, s));
    return HLQ_OK;
  }
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(d_ws);
  unsigned int* amax = reinterpret_cast<unsigned int*>(base);      // [0] g_y, [1] x
  float* sg = reinterpret_cast<float*>(base + kAlign);
  float* sx = sg + 4;
  uint8_t* qg = base + 2 * kAlign;                                 // [Cout, T]
  uint8_t* qx = qg + align_up((size_t)Cout * (size_t)T);           // [Cin, T]
  const bool bf16 = dt == HLQ_BF16;
  HLQ_TRY(cudaMemsetAsync(amax, 0, 8, s));
  HLQ_LAUNCH("hq_tok_gy_amax", s,
             launch_hq_cols(d_gy, bf16, T, Cout, true, amax, nullptr, nullptr, rnd, seed, 2,
                            status, s));
  HLQ_LAUNCH("hq_tok_gy_quant", s,
             launch_hq_cols(d_gy, bf16, T, Cout, false, amax, qg, sg, rnd, seed, 2, status,
                            s));
  HLQ_LAUNCH("hq_tok_x_amax", s,
             launch_hq_cols(d_x, bf16, T, Cin, true, amax + 1, nullptr, nullptr, rnd, seed, 3,
                            status, s));
  HLQ_LAUNCH("hq_tok_x_quant", s,
             launch_hq_cols(d_x, bf16, T, Cin, false, amax + 1, qx, sx, rnd, seed, 3, status,
                            s));
  const int sms = device_sm_count();
  if (sms <= 0) return HLQ_ERR_CUDA;
  const GemmPlan plan = plan_gemm_tc(0, Cout, Cin, T, sms, 1);
  HLQ_LAUNCH("gemm_gw_hq_tc", s,
             launch_gemm_tc(0, qg, T, qx, T, Cout, Cin, T, plan, sg, false, sx, d_gw, d_acc,
                            nullptr, status, s));
  return HLQ_OK;
}

hlq_status hlq_ablation_gx_hla(const void* d_gy, const void* d_w, int dt, int64_t T,
                               int64_t Cin, int64_t Cout, int block, int rank, float* d_gx,
                               int32_t* d_acc, void* d_ws, size_t ws_bytes, void* stream) {
  hlq_status st = check_common(dt, T, Cin, Cout, block);
  if (st != HLQ_OK) return st;
  if (!rank_ok(rank)) return HLQ_ERR_INVALID_ARG;
  if ((T * Cout > 0 && !d_gy) || (Cout * Cin > 0 && !d_w) || (T * Cin > 0 && !d_gx))
    return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_gy) || !aligned16(d_w) || !aligned16(d_gx) || !aligned16(d_acc))
    return HLQ_ERR_ALIGN;
  const int64_t Kp = Cout / 16 * rank;
  if (Kp * 127 * 127 >= ((int64_t)1 << 31)) return HLQ_ERR_OVERFLOW;
  const GxHlaLayout L = gx_hla_layout(T, Cin, Cout, rank);
  if (!d_ws || ws_bytes < L.total) return HLQ_ERR_WORKSPACE;
  if (!aligned256(d_ws)) return HLQ_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T * Cin == 0) return HLQ_OK;
  if (Kp == 0) {  // empty contraction
    HLQ_TRY(cudaMemsetAsync(d_gx, 0, (size_t)(T * Cin) * 4, s));
    if (d_acc) HLQ_TRY(cudaMemsetAsync(d_acc, 0, (size_t)(T * Cin) * 4, s));
    return HLQ_OK;
  }
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(d_ws);
  unsigned int* amax = reinterpret_cast<unsigned int*>(base + L.amax);  // [0] g_y, [1] w
  float* sg = reinterpret_cast<float*>(base + L.s);
  float* sw = sg + 4;
  void* qg = base + L.qg;
  void* qw = base + L.qw;
  const bool bf16 = dt == HLQ_BF16;
  HLQ_TRY(cudaMemsetAsync(amax, 0, 8, s));
  HLQ_LAUNCH("hla_rows_gy_amax", s,
             launch_hla_rows(d_gy, bf16, T, Cout, rank, true, amax, nullptr, 0, nullptr,
                             status, s));
  HLQ_LAUNCH("hla_rows_gy_quant", s,
             launch_hla_rows(d_gy, bf16, T, Cout, rank, false, amax, qg, L.ld, sg, status, s));
  HLQ_LAUNCH("hla_w_amax", s,
             launch_hla(d_w, bf16, Cout, Cin, rank, true, kHlaOutF16, amax + 1, nullptr, 0,
                        nullptr, status, s));
  HLQ_LAUNCH("hla_w_quant", s,
             launch_hla(d_w, bf16, Cout, Cin, rank, false, kHlaOutF16, amax + 1, qw, L.ld, sw,
                        status, s));
  const int sms = device_sm_count();
  if (sms <= 0) return HLQ_ERR_CUDA;
  const GemmPlan plan = plan_gemm_tc(1, T, Cin, Kp, sms, 1);
  HLQ_LAUNCH("gemm_gx_hla_tc", s,
             launch_gemm_tc(1, qg, L.ld, qw, L.ld, T, Cin, Kp, plan, sg, false, sw, d_gx, d_acc,
                            nullptr, status, s));
  return HLQ_OK;
}

// Both gradients with one fused reader of g_y (gy_fused_kernel): the HQ
// maxima and the HLA maximum in one pass over g_y, then the HQ codes and the
// HLA codes in a second; the HQ of w and the widening of the stored
// activation run on the auxiliary streams meanwhile, and the two GEMMs
// follow the second pass.  Same results as hlq_linear_backward.
// The backward with one fused reader of g_y (two passes: the HQ and HLA
// maxima, then both codes), after validation.  d_x (may be null): compress
// x into d_xbar / d_xbar_scale first, on the g_w branch (x_amax: the
// compression's maximum slots).  amax_rows: per-token HQ maxima [T] (per-token
// g_y only).
static hlq_status fused_launches(const void* d_gy, const void* d_w, const void* d_x, int8_t* d_xbar,
                          float* d_xbar_scale, int dt, int64_t T, int64_t Cin, int64_t Cout,
                          int rank, int xbar_fmt, int gran_gy, int rnd, uint64_t seed,
                          float* d_gx, float* d_gw, uint8_t* gxb, uint8_t* gwb,
                          unsigned int* amax_rows, unsigned int* x_amax, cudaStream_t s) {
  const int64_t Tp = T / 16 * rank;
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return HLQ_ERR_CUDA;
  const bool serial = g_serial_branches.load();  // one reading per call
  cudaStream_t a = branch_stream(0, s, serial), aw = branch_stream(1, s, serial);
  if (!serial && (!a || !aw)) return HLQ_ERR_CUDA;  // (null: the legacy stream)
  const GxLayout GL = gx_layout(T, Cin, Cout);
  const GwLayout WL = gw_layout(T, Cin, Cout, rank);
  unsigned int* gx_amax = reinterpret_cast<unsigned int*>(gxb + GL.amax);
  float* sgy = reinterpret_cast<float*>(gxb + GL.sgy);
  float* sw = reinterpret_cast<float*>(gxb + GL.sw);
  uint8_t* qy = gxb + GL.qy;
  uint8_t* qw = gxb + GL.qw;
  unsigned int* gw_amax = reinterpret_cast<unsigned int*>(gwb + WL.amax);
  float* sg = reinterpret_cast<float*>(gwb + WL.sg);
  const bool bf16 = dt == HLQ_BF16;
  const bool per_token = gran_gy == HLQ_PER_TOKEN;

  EventSet E;
  cudaEvent_t fork = E.make(), w_done = E.make(), gw_done = E.make();
  if (!fork || !w_done || !gw_done) return HLQ_ERR_CUDA;
  hlq_status r = HLQ_OK;
  auto fail = [&](cudaError_t e) {
    if (e != cudaSuccess && r == HLQ_OK) r = HLQ_ERR_CUDA;
  };
  fail(cudaEventRecord(fork, s));
  // HQ of w on its own stream
  fail(cudaStreamWaitEvent(aw, fork, 0));
  fail(cudaMemsetAsync(gx_amax + 1, 0, 4, aw));
  if (r == HLQ_OK) r = hq_w_launches(d_w, bf16, Cout, Cin, gx_amax + 1, qw, sw, rnd, seed, status, aw);
  fail(cudaEventRecord(w_done, aw));
  // the stored activation (compressed here first when x is given) widened
  // to fp16 meanwhile (unless the GEMM reads the int8 codes itself)
  const int gw_rw = gw_raw(xbar_fmt, Tp, d_xbar, true);
  fail(cudaStreamWaitEvent(a, fork, 0));
  if (r == HLQ_OK && d_x)
    r = compress_launches(d_x, bf16, T, Cin, rank, xbar_fmt, d_xbar, d_xbar_scale, x_amax,
                          status, a);
  if (r == HLQ_OK && !(gw_rw & kRawB)) {
    trace_before(a);
    if (xbar_code_bits(xbar_fmt) == 4)
      fail(launch_widen_i4_f16(reinterpret_cast<const uint8_t*>(d_xbar), gwb + WL.xw, Cin, Tp,
                                WL.ld, a));
    else
      fail(launch_widen_i8_f16(d_xbar, gwb + WL.xw, Cin, Tp, WL.ld, a));
    trace_after("widen_xbar", a);
  }
  // the two passes over g_y
  fail(cudaMemsetAsync(gw_amax, 0, 4, s));
  fail(per_token ? cudaMemsetAsync(amax_rows, 0, (size_t)T * 4, s)
                 : cudaMemsetAsync(gx_amax, 0, 4, s));
  unsigned int* hq_slot = per_token ? amax_rows : gx_amax;
  if (r == HLQ_OK) {
    trace_before(s);
    fail(launch_gy_fused(d_gy, bf16, T, Cout, rank, per_token, true, hq_slot, gw_amax, nullptr,
                         nullptr, nullptr, 0, nullptr, rnd, seed, status, s));
    trace_after("gy_fused_amax", s);
    trace_before(s);
    fail(launch_gy_fused(d_gy, bf16, T, Cout, rank, per_token, false, hq_slot, gw_amax, qy,
                         sgy, gwb + WL.qg, WL.ld, sg, rnd, seed, status, s));
    trace_after("gy_fused_quant", s);
  }
  // both GEMMs on the caller's stream, one after the other: each is a
  // persistent grid of one CTA per SM whose tiles are dealt out in advance,
  // so run side by side the later one's CTAs wait for SMs and its tiles
  // finish last (measured on ResNet-50 im2col: 674 us per step instead of
  // 434 us)
  fail(cudaEventRecord(gw_done, a));  // the widened stored activation
  fail(cudaStreamWaitEvent(s, w_done, 0));
  if (r == HLQ_OK) {
    const GemmPlan px = plan_gemm_tc(0, T, Cin, Cout, sms, 1);
    trace_before(s);
    fail(launch_gemm_tc(0, qy, Cout, qw, Cout, T, Cin, Cout, px, sgy, per_token, sw, d_gx,
                        nullptr, nullptr, status, s));
    trace_after("gemm_gx_tc", s);
  }
  fail(cudaStreamWaitEvent(s, gw_done, 0));  // join (also after a failure)
  if (r == HLQ_OK) {
    const GemmPlan pw = plan_gemm_tc(1, Cout, Cin, Tp, sms, 16);
    trace_before(s);
    fail(launch_gemm_tc(1, gwb + WL.qg, WL.ld, (gw_rw & kRawB) ? (const void*)d_xbar : gwb + WL.xw,
                        (gw_rw & kRawB) ? Tp : WL.ld, Cout, Cin, Tp, pw, sg, false,
                        d_xbar_scale, d_gw, nullptr, gwb + WL.split, status, s,
                        xbar_per_channel(xbar_fmt), gw_rw));
    trace_after("gemm_gw_tc", s);
  }
  return r;
}

hlq_status hlq_linear_backward_fused(const void* d_gy, const void* d_w, const int8_t* d_xbar,
                                     const float* d_xbar_scale, int dt, int64_t T,
                                     int64_t Cin, int64_t Cout, int block, int rank,
                                     int xbar_fmt, int gran_gy, int gran_w, int rnd,
                                     uint64_t seed, float* d_gx, float* d_gw, void* d_ws,
                                     size_t ws_bytes, void* stream) {
  hlq_status st = check_common(dt, T, Cin, Cout, block);
  if (st != HLQ_OK) return st;
  if (!rank_ok(rank)) return HLQ_ERR_INVALID_ARG;
  const size_t gx_bytes = gx_layout(T, Cin, Cout).total;
  const size_t gw_bytes = gw_layout(T, Cin, Cout, rank).total;
  const size_t rows_bytes = align_up((size_t)(T > 0 ? T : 1) * 4);
  if (!d_ws || ws_bytes < gx_bytes + gw_bytes + rows_bytes) return HLQ_ERR_WORKSPACE;
  if (!aligned256(d_ws)) return HLQ_ERR_ALIGN;
  uint8_t* base = static_cast<uint8_t*>(d_ws);
  uint8_t* gxb = base;
  uint8_t* gwb = base + gx_bytes;
  unsigned int* amax_rows = reinterpret_cast<unsigned int*>(base + gx_bytes + gw_bytes);
  st = gw_impl(d_gy, dt, d_xbar, xbar_fmt, d_xbar_scale, T, Cin, Cout, block, rank, d_gw, gwb,
               gw_bytes, nullptr, nullptr, nullptr, nullptr, /*validate_only=*/true);
  if (st != HLQ_OK) return st;
  st = gx_impl(d_gy, d_w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd, seed, d_gx, gxb,
               gx_bytes, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
               /*validate_only=*/true);
  if (st != HLQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T * Cin * Cout == 0) {  // degenerate sizes: the separate paths zero-fill
    st = gx_impl(d_gy, d_w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd, seed, d_gx, gxb,
                 gx_bytes, nullptr, nullptr, nullptr, nullptr, nullptr, stream);
    if (st != HLQ_OK) return st;
    return gw_impl(d_gy, dt, d_xbar, xbar_fmt, d_xbar_scale, T, Cin, Cout, block, rank, d_gw,
                   gwb, gw_bytes, nullptr, nullptr, nullptr, stream);
  }
  return fused_launches(d_gy, d_w, nullptr, const_cast<int8_t*>(d_xbar),
                        const_cast<float*>(d_xbar_scale), dt, T, Cin, Cout, rank, xbar_fmt,
                        gran_gy, rnd, seed, d_gx, d_gw, gxb, gwb, amax_rows, nullptr, s);
}

size_t hlq_layer_step_host_workspace_bytes(int dt, int64_t T, int64_t Cin, int64_t Cout,
                                           int block, int rank) {
  (void)block;
  if (T < 0 || Cin < 0 || Cout < 0 || (dt != HLQ_F32 && dt != HLQ_BF16)) return 0;
  return step_layout(dt, T, Cin, Cout, rank_ok(rank) ? rank : 16).total;
}

hlq_status hlq_layer_step_host(const void* h_x, const void* h_gy, const void* h_w, int dt,
                               int64_t T, int64_t Cin, int64_t Cout, int block, int rank,
                               int xbar_fmt, int gran_gy, int gran_w, int rnd, uint64_t seed,
                               float* h_gx,
                               float* h_gw, int8_t* d_xbar, float* d_xbar_scale,
                               int64_t chunk_tokens, void* d_ws, size_t ws_bytes,
                               void* stream) {
  hlq_status st = check_common(dt, T, Cin, Cout, block);
  if (st != HLQ_OK) return st;
  if (!rank_ok(rank) || chunk_tokens < 0) return HLQ_ERR_INVALID_ARG;
  if ((T * Cin > 0 && (!h_x || !h_gx)) || (T * Cout > 0 && !h_gy) ||
      (Cout * Cin > 0 && (!h_w || !h_gw)))
    return HLQ_ERR_INVALID_ARG;
  const StepLayout L = step_layout(dt, T, Cin, Cout, rank);
  if (!d_ws || ws_bytes < L.total) return HLQ_ERR_WORKSPACE;
  if (!aligned256(d_ws)) return HLQ_ERR_ALIGN;
  uint8_t* base = static_cast<uint8_t*>(d_ws);
  void* x = base + L.x;
  void* gy = base + L.gy;
  void* w = base + L.w;
  float* gx = reinterpret_cast<float*>(base + L.gx);
  float* gw = reinterpret_cast<float*>(base + L.gw);
  const size_t gx_bytes = gx_layout(T, Cin, Cout).total;
  const size_t gw_bytes = gw_layout(T, Cin, Cout, rank).total;
  // validate every device step before anything is enqueued
  st = gx_impl(gy, w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd, seed, gx, base + L.gxws,
               gx_bytes, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, true);
  if (st != HLQ_OK) return st;
  st = gw_impl(gy, dt, d_xbar, xbar_fmt, d_xbar_scale, T, Cin, Cout, block, rank, gw,
               base + L.gwws, gw_bytes, nullptr, nullptr, nullptr, nullptr, true);
  if (st != HLQ_OK) return st;
  if (!d_xbar_scale) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_xbar)) return HLQ_ERR_ALIGN;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t esz = dt == HLQ_BF16 ? 2 : 4;
  const int64_t Tp = T / 16 * rank;
  auto h2d = [](void* d, const void* h, size_t n, cudaStream_t q) {
    return n ? cudaMemcpyAsync(d, h, n, cudaMemcpyHostToDevice, q) : cudaSuccess;
  };
  auto d2h = [](void* h, const void* d, size_t n, cudaStream_t q) {
    return n ? cudaMemcpyAsync(h, d, n, cudaMemcpyDeviceToHost, q) : cudaSuccess;
  };
  if (T == 0 || Cin == 0 || Cout == 0) {  // degenerate sizes: one stream, in order
    HLQ_TRY(h2d(x, h_x, (size_t)(T * Cin) * esz, s));
    HLQ_TRY(h2d(gy, h_gy, (size_t)(T * Cout) * esz, s));
    HLQ_TRY(h2d(w, h_w, (size_t)(Cout * Cin) * esz, s));
    st = hlq_compress_activation(x, dt, T, Cin, block, rank, xbar_fmt, d_xbar, d_xbar_scale,
                                 base + L.cws, compress_ws(T, Cin), stream);
    if (st != HLQ_OK) return st;
    st = hlq_linear_backward_gx(gy, w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd, seed,
                                gx, base + L.gxws, gx_bytes, stream);
    if (st != HLQ_OK) return st;
    st = hlq_linear_backward_gw(gy, dt, d_xbar, d_xbar_scale, T, Cin, Cout, block, rank,
                                xbar_fmt, gw,
                                base + L.gwws, gw_bytes, stream);
    if (st != HLQ_OK) return st;
    HLQ_TRY(d2h(h_gx, gx, (size_t)(T * Cin) * 4, s));
    HLQ_TRY(d2h(h_gw, gw, (size_t)(Cout * Cin) * 4, s));
    return HLQ_OK;
  }

  // chunks of g_y rows: multiples of 128 (GEMM tiles), ~16 MB each, at most
  // kMaxHostChunks of them
  int64_t ch = chunk_tokens;
  if (ch == 0) ch = (int64_t)((16u << 20) / ((size_t)Cout * esz));
  ch = (ch + 127) / 128 * 128;
  if (ch < 128) ch = 128;
  if ((T + ch - 1) / ch > kMaxHostChunks)
    ch = ((T + kMaxHostChunks - 1) / kMaxHostChunks + 127) / 128 * 128;
  const int nc = (int)((T + ch - 1) / ch);
  if (nc < 1 || nc > kMaxHostChunks) return HLQ_ERR_INVALID_ARG;

  cudaStream_t a_gw = aux_stream(0), a_w = aux_stream(1), cin = aux_stream(2),
               cout = aux_stream(3);
  if (!a_gw || !a_w || !cin || !cout) return HLQ_ERR_CUDA;
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return HLQ_ERR_CUDA;

  EventSet E;
  cudaEvent_t fork = E.make(), w_in = E.make(), w_done = E.make(), gw_done = E.make(),
              out_done = E.make();
  cudaEvent_t gy_in[kMaxHostChunks], x_in[kMaxHostChunks], gx_done[kMaxHostChunks];
  bool events_ok = fork && w_in && w_done && gw_done && out_done;
  for (int c = 0; c < nc; ++c) {
    gy_in[c] = E.make();
    x_in[c] = E.make();
    gx_done[c] = E.make();
    events_ok = events_ok && gy_in[c] && x_in[c] && gx_done[c];
  }
  if (!events_ok) return HLQ_ERR_CUDA;

  const bool bf16 = dt == HLQ_BF16;
  const bool per_token = gran_gy == HLQ_PER_TOKEN;
  uint8_t* gxb = base + L.gxws;
  const GxLayout GL = gx_layout(T, Cin, Cout);
  unsigned int* gx_amax = reinterpret_cast<unsigned int*>(gxb + GL.amax);
  float* sgy = reinterpret_cast<float*>(gxb + GL.sgy);
  float* sw = reinterpret_cast<float*>(gxb + GL.sw);
  uint8_t* qy = gxb + GL.qy;
  uint8_t* qw = gxb + GL.qw;
  uint8_t* gwb = base + L.gwws;
  const GwLayout WL = gw_layout(T, Cin, Cout, rank);
  unsigned int* gw_amax = reinterpret_cast<unsigned int*>(gwb + WL.amax);
  float* sg = reinterpret_cast<float*>(gwb + WL.sg);

  hlq_status r = HLQ_OK;
  auto fail = [&](cudaError_t e) {
    if (e != cudaSuccess && r == HLQ_OK) r = HLQ_ERR_CUDA;
  };
  fail(cudaEventRecord(fork, s));
  // copy-in stream: w (first needed), the g_y chunks, then the x chunks
  fail(cudaStreamWaitEvent(cin, fork, 0));
  fail(h2d(w, h_w, (size_t)(Cout * Cin) * esz, cin));
  fail(cudaEventRecord(w_in, cin));
  for (int c = 0; c < nc; ++c) {
    const int64_t r0 = c * ch, rows = (r0 + ch <= T ? ch : T - r0);
    fail(h2d(static_cast<uint8_t*>(gy) + (size_t)r0 * Cout * esz,
             static_cast<const uint8_t*>(h_gy) + (size_t)r0 * Cout * esz,
             (size_t)rows * Cout * esz, cin));
    fail(cudaEventRecord(gy_in[c], cin));
  }
  for (int c = 0; c < nc; ++c) {
    const int64_t r0 = c * ch, rows = (r0 + ch <= T ? ch : T - r0);
    fail(h2d(static_cast<uint8_t*>(x) + (size_t)r0 * Cin * esz,
             static_cast<const uint8_t*>(h_x) + (size_t)r0 * Cin * esz,
             (size_t)rows * Cin * esz, cin));
    fail(cudaEventRecord(x_in[c], cin));
  }
  // HQ of w
  fail(cudaStreamWaitEvent(a_w, w_in, 0));
  fail(cudaMemsetAsync(gx_amax + 1, 0, 4, a_w));
  if (r == HLQ_OK) r = hq_w_launches(w, bf16, Cout, Cin, gx_amax + 1, qw, sw, rnd, seed, status, a_w);
  fail(cudaEventRecord(w_done, a_w));
  // g_x branch on the caller's stream, chunk by chunk
  fail(cudaMemsetAsync(gx_amax, 0, 4, s));
  auto gemm_chunk = [&](int c) {
    const int64_t r0 = c * ch, rows = (r0 + ch <= T ? ch : T - r0);
    const GemmPlan plan = plan_gemm_tc(0, rows, Cin, Cout, sms, 1);
    if (r == HLQ_OK) {
      trace_before(s);
      fail(launch_gemm_tc(0, qy + (size_t)r0 * Cout, Cout, qw, Cout, rows, Cin, Cout, plan,
                          per_token ? sgy + r0 : sgy, per_token, sw, gx + (size_t)r0 * Cin,
                          nullptr, nullptr, status, s));
      trace_after("gemm_gx_tc", s);
    }
    fail(cudaEventRecord(gx_done[c], s));
  };
  for (int c = 0; c < nc && r == HLQ_OK; ++c) {
    const int64_t r0 = c * ch, rows = (r0 + ch <= T ? ch : T - r0);
    fail(cudaStreamWaitEvent(s, gy_in[c], 0));
    const uint8_t* gyc = static_cast<const uint8_t*>(gy) + (size_t)r0 * Cout * esz;
    if (per_token) {
      trace_before(s);
      fail(launch_hq_rows(gyc, bf16, rows, Cout, true, false, gx_amax, qy + (size_t)r0 * Cout,
                          sgy + r0, rnd, seed, 0, status, s, r0));
      trace_after("hq_rows_quant", s);
      if (c == 0) fail(cudaStreamWaitEvent(s, w_done, 0));
      gemm_chunk(c);
    } else {
      trace_before(s);
      fail(launch_hq_rows(gyc, bf16, rows, Cout, false, true, gx_amax, nullptr, nullptr, rnd,
                          seed, 0, status, s, r0));
      trace_after("hq_rows_amax", s);
    }
  }
  if (!per_token && r == HLQ_OK) {  // the per-tensor scale needs all of g_y
    trace_before(s);
    fail(launch_hq_rows(gy, bf16, T, Cout, false, false, gx_amax, qy, sgy, rnd, seed, 0,
                        status, s, 0));
    trace_after("hq_rows_quant", s);
    fail(cudaStreamWaitEvent(s, w_done, 0));
    for (int c = 0; c < nc; ++c) gemm_chunk(c);
  }
  // g_w branch.  The per-tensor maxima of the HLA of g_y and of the
  // compression of x are gathered chunk by chunk as the chunks land (16-token
  // blocks never straddle a chunk: chunks are multiples of 128 tokens), so
  // that only the quant passes, the widening of x-bar, the g_w GEMM and its
  // copy-out follow the last byte of x.
  const int gw_rw = gw_raw(xbar_fmt, Tp, d_xbar, false);
  const bool qg_i8 = (gw_rw & kRawA) != 0;
  const bool x_per_ch = xbar_per_channel(xbar_fmt);
  unsigned int* x_amax = reinterpret_cast<unsigned int*>(base + L.cws);
  fail(cudaStreamWaitEvent(a_gw, fork, 0));
  fail(cudaMemsetAsync(gw_amax, 0, 4, a_gw));
  fail(cudaMemsetAsync(x_amax, 0, (size_t)(x_per_ch ? Cin : 1) * 4, a_gw));
  for (int c = 0; c < nc && r == HLQ_OK; ++c) {
    const int64_t r0 = c * ch, rows = (r0 + ch <= T ? ch : T - r0);
    fail(cudaStreamWaitEvent(a_gw, gy_in[c], 0));
    trace_before(a_gw);
    fail(launch_hla(static_cast<const uint8_t*>(gy) + (size_t)r0 * Cout * esz, bf16, rows, Cout,
                    rank, true, kHlaOutF16, gw_amax, nullptr, 0, nullptr, status, a_gw));
    trace_after("hla_gy_amax", a_gw);
  }
  if (r == HLQ_OK) {
    trace_before(a_gw);
    fail(launch_hla(gy, bf16, T, Cout, rank, false, qg_i8 ? kHlaOutI8 : kHlaOutF16, gw_amax,
                    gwb + WL.qg, qg_i8 ? WL.ld8 : WL.ld, sg, status, a_gw));
    trace_after("hla_gy_quant", a_gw);
  }
  for (int c = 0; c < nc && r == HLQ_OK; ++c) {
    const int64_t r0 = c * ch, rows = (r0 + ch <= T ? ch : T - r0);
    fail(cudaStreamWaitEvent(a_gw, x_in[c], 0));
    trace_before(a_gw);
    fail(launch_hla(static_cast<const uint8_t*>(x) + (size_t)r0 * Cin * esz, bf16, rows, Cin,
                    rank, true, kHlaOutI8, x_amax, nullptr, 0, nullptr, status, a_gw, x_per_ch));
    trace_after("hla_x_amax", a_gw);
  }
  if (r == HLQ_OK) {
    trace_before(a_gw);
    fail(launch_hla(x, bf16, T, Cin, rank, false,
                    xbar_code_bits(xbar_fmt) == 4 ? kHlaOutI4 : kHlaOutI8, x_amax, d_xbar, Tp,
                    d_xbar_scale, status, a_gw, x_per_ch));
    trace_after("hla_x_quant", a_gw);
  }
  if (r == HLQ_OK)
    r = gw_gemm_launches(d_xbar, xbar_fmt, d_xbar_scale, Cin, Cout, Tp, WL, gwb, gw, nullptr,
                         status, a_gw,
                         gemms_in_sequence(ch < T ? ch : T, Cin, Cout, Tp) ? gx_done[nc - 1]
                                                                           : nullptr,
                         gw_rw);
  fail(cudaEventRecord(gw_done, a_gw));
  // copy-out stream: g_x chunk by chunk as they finish, then g_w
  for (int c = 0; c < nc; ++c) {
    const int64_t r0 = c * ch, rows = (r0 + ch <= T ? ch : T - r0);
    fail(cudaStreamWaitEvent(cout, gx_done[c], 0));
    fail(d2h(h_gx + (size_t)r0 * Cin, gx + (size_t)r0 * Cin, (size_t)rows * Cin * 4, cout));
  }
  fail(cudaStreamWaitEvent(cout, gw_done, 0));
  fail(d2h(h_gw, gw, (size_t)(Cout * Cin) * 4, cout));
  fail(cudaEventRecord(out_done, cout));
  // join every stream back into the caller's (also after a failure)
  fail(cudaStreamWaitEvent(s, out_done, 0));
  fail(cudaStreamWaitEvent(s, w_done, 0));
  return r;
}

hlq_status hlq_linear_backward_gx(const void* d_gy, const void* d_w, int dt,
                                  int64_t T, int64_t Cin, int64_t Cout,
                                  int block, int gran_gy, int gran_w, int rnd,
                                  uint64_t seed, float* d_gx, void* d_ws,
                                  size_t ws_bytes, void* stream) {
  return gx_impl(d_gy, d_w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd,
                 seed, d_gx, d_ws, ws_bytes, nullptr, nullptr, nullptr,
                 nullptr, nullptr, stream);
}

hlq_status hlq_linear_backward_gw(const void* d_gy, int dt,
                                  const int8_t* d_xbar,
                                  const float* d_xbar_scale, int64_t T,
                                  int64_t Cin, int64_t Cout, int block,
                                  int rank, int xbar_fmt, float* d_gw, void* d_ws,
                                  size_t ws_bytes, void* stream) {
  return gw_impl(d_gy, dt, d_xbar, xbar_fmt, d_xbar_scale, T, Cin, Cout, block, rank,
                 d_gw, d_ws, ws_bytes, nullptr, nullptr, nullptr, stream);
}

hlq_status hlq_debug_gx_parts(const void* d_gy, const void* d_w, int dt,
                              int64_t T, int64_t Cin, int64_t Cout, int block,
                              int gran_gy, int gran_w, int rnd, uint64_t seed,
                              float* d_gx, void* d_ws, size_t ws_bytes,
                              int8_t* d_qgy, float* d_sgy, int8_t* d_qw,
                              float* d_sw, int32_t* d_acc, uint8_t* d_qgy_packed,
                              uint8_t* d_qw_packed, void* stream) {
  return gx_impl(d_gy, d_w, dt, T, Cin, Cout, block, gran_gy, gran_w, rnd,
                 seed, d_gx, d_ws, ws_bytes, d_qgy, d_sgy, d_qw, d_sw, d_acc,
                 stream, false, nullptr, d_qgy_packed, d_qw_packed);
}

hlq_status hlq_debug_gw_parts(const void* d_gy, int dt, const int8_t* d_xbar,
                              const float* d_xbar_scale, int64_t T,
                              int64_t Cin, int64_t Cout, int block, int rank,
                              int xbar_fmt, float* d_gw, void* d_ws, size_t ws_bytes,
                              int8_t* d_qg, float* d_sg, int32_t* d_acc,
                              void* stream) {
  return gw_impl(d_gy, dt, d_xbar, xbar_fmt, d_xbar_scale, T, Cin, Cout, block, rank,
                 d_gw, d_ws, ws_bytes, d_qg, d_sg, d_acc, stream);
}

hlq_status hlq_debug_hq_transform(const void* d_src, int dt, int64_t rows,
                                  int64_t cols, int axis, float* d_y,
                                  void* stream) {
  if (dt != HLQ_F32 && dt != HLQ_BF16) return HLQ_ERR_INVALID_ARG;
  if (axis != 0 && axis != 1) return HLQ_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || rows % 16 || cols % 16) return HLQ_ERR_SHAPE;
  if (rows / 16 > 65535 && axis == 1) return HLQ_ERR_UNSUPPORTED;
  if (rows * cols > 0 && (!d_src || !d_y)) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_src) || !aligned16(d_y)) return HLQ_ERR_ALIGN;
  if (rows * cols == 0) return HLQ_OK;
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = dt == HLQ_BF16;
  if (axis == 0)
    HLQ_TRY(launch_hq_rows_transform(d_src, bf16, rows, cols, d_y, status, s));
  else
    HLQ_TRY(launch_hq_cols_transform(d_src, bf16, rows, cols, d_y, status, s));
  return HLQ_OK;
}

hlq_status hlq_debug_hla_transform(const void* d_src, int dt, int64_t T,
                                   int64_t C, int rank, float* d_out,
                                   void* stream) {
  if (dt != HLQ_F32 && dt != HLQ_BF16) return HLQ_ERR_INVALID_ARG;
  if (!rank_ok(rank)) return HLQ_ERR_INVALID_ARG;
  if (T < 0 || C < 0 || T % 16 || C % 16) return HLQ_ERR_SHAPE;
  if (T / 16 > 65535) return HLQ_ERR_UNSUPPORTED;
  if (T * C > 0 && (!d_src || !d_out)) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_src) || !aligned16(d_out)) return HLQ_ERR_ALIGN;
  if (T * C == 0) return HLQ_OK;
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  HLQ_TRY(launch_hla_transform(d_src, dt == HLQ_BF16, T, C, rank, d_out, status,
                               static_cast<cudaStream_t>(stream)));
  return HLQ_OK;
}

hlq_status hlq_debug_reference_gemm(int kind, const void* d_a, const void* d_b,
                                    int64_t M, int64_t N, int64_t K,
                                    int32_t* d_acc, void* stream) {
  if (kind != 0 && kind != 1) return HLQ_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return HLQ_ERR_SHAPE;
  if (M * N > 0 && (!d_a || !d_b || !d_acc)) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_a) || !aligned16(d_b) || !aligned16(d_acc)) return HLQ_ERR_ALIGN;
  if (M * N == 0) return HLQ_OK;
  HLQ_TRY(launch_gemm_simple(d_a, kFmtI8, d_b, kFmtI8, M, N, K, nullptr, false,
                             nullptr, nullptr, d_acc, static_cast<cudaStream_t>(stream)));
  return HLQ_OK;
}

hlq_status hlq_debug_tc_gemm(int kind, const void* d_a, int64_t lda, const void* d_b,
                             int64_t ldb, int64_t M, int64_t N, int64_t K, int bn,
                             int splits, int pair, int32_t* d_acc, void* d_ws,
                             size_t ws_bytes, void* stream) {
  if (kind < 0 || kind > 3) return HLQ_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || N % 16 || K % 16 || M % 16) return HLQ_ERR_SHAPE;
  if (bn != 0 && bn != 96 && bn != 128 && bn != 256) return HLQ_ERR_INVALID_ARG;
  if (splits < -1 || splits > 64) return HLQ_ERR_INVALID_ARG;  // -1: stream-K
  if (pair < -1 || pair > 1) return HLQ_ERR_INVALID_ARG;
  if (pair == 1 && bn == 96) return HLQ_ERR_INVALID_ARG;    // pairs: 128 or 256 wide
  if (kind == 0 && (splits > 1 || splits == -1)) return HLQ_ERR_INVALID_ARG;  // E4M3: unsplit
  if (splits == -1 && pair == 1) return HLQ_ERR_INVALID_ARG;  // stream-K: one CTA per tile
  // element bytes of A and B: E4M3 (kind 0), fp16 (kind 1; A of kind 2),
  // int8 widened in the GEMM (B of kinds 2 and 3, A of kind 3)
  const int esz_a = (kind == 1 || kind == 2) ? 2 : 1;
  const int esz_b = kind == 1 ? 2 : 1;
  if (lda < K || ldb < K || (lda * esz_a) % 16 || (ldb * esz_b) % 16) return HLQ_ERR_ALIGN;
  if (M * N > 0 && (!d_a || !d_b || !d_acc)) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_a) || !aligned16(d_b) || !aligned16(d_acc)) return HLQ_ERR_ALIGN;
  if (kind == 0 && 49 * K >= ((int64_t)1 << 24)) return HLQ_ERR_OVERFLOW;
  if (kind != 0 && K * 127 * 127 >= ((int64_t)1 << 31)) return HLQ_ERR_OVERFLOW;
  if (M * N == 0) return HLQ_OK;
  if (kind >= 2 && K == 0) return HLQ_ERR_SHAPE;
  const int sms = device_sm_count();
  if (sms <= 0) return HLQ_ERR_CUDA;
  const int gk = kind == 0 ? 0 : 1;  // the GEMM kind
  const int raw = kind == 2 ? kRawB : (kind == 3 ? (kRawA | kRawB) : 0);
  GemmPlan plan = plan_gemm_tc(gk, M, N, K, sms, gk == 1 ? 16 : 1);
  if (bn) plan.bn = bn;
  if (splits > 0) {
    plan.splits = splits;
    plan.stream_k = 0;
  } else if (splits == -1) {
    plan.splits = 1;
    plan.stream_k = 1;
    plan.pair = 0;
  }
  if (pair >= 0) plan.pair = pair;
  if (plan.pair) plan.stream_k = 0;
  if (plan.pair && plan.bn == 96) return HLQ_ERR_INVALID_ARG;
  const bool ws_used = plan.splits > 1 || plan.stream_k;
  if (ws_used && (!d_ws || ws_bytes < gemm_tc_split_ws_bytes(M, N))) return HLQ_ERR_WORKSPACE;
  if (ws_used && !aligned256(d_ws)) return HLQ_ERR_ALIGN;
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  HLQ_LAUNCH(kind == 0 ? "gemm_gx_tc" : "gemm_gw_tc", s,
             launch_gemm_tc(gk, d_a, lda, d_b, ldb, M, N, K, plan, nullptr, false,
                            nullptr, nullptr, d_acc, d_ws, status, s, false, raw));
  return HLQ_OK;
}

hlq_status hlq_set_gw_operands(int mode) {
  if (mode < HLQ_GW_AUTO || mode > HLQ_GW_INT8_BOTH) return HLQ_ERR_INVALID_ARG;
  g_gw_operands.store(mode);
  return HLQ_OK;
}

int hlq_get_gw_operands(void) { return g_gw_operands.load(); }

hlq_status hlq_debug_serialize_branches(int on) {
  if (on != 0 && on != 1) return HLQ_ERR_INVALID_ARG;
  g_serial_branches.store(on != 0);
  return HLQ_OK;
}

hlq_status hlq_debug_gemm_plan(int64_t T, int64_t Cin, int64_t Cout, int rank, int sms,
                               int* gx_bn, int* gx_splits, int* gw_bn, int* gw_splits,
                               int* in_sequence, int* gx_pair, int* gw_pair) {
  if (T < 0 || Cin < 0 || Cout < 0 || !rank_ok(rank) || sms <= 0) return HLQ_ERR_INVALID_ARG;
  if (!gx_bn || !gx_splits || !gw_bn || !gw_splits || !in_sequence || !gx_pair || !gw_pair)
    return HLQ_ERR_INVALID_ARG;
  const int64_t Tp = T / 16 * rank;
  const GemmPlan px = plan_gemm_tc(0, T, Cin, Cout, sms, 1);
  const GemmPlan pw = plan_gemm_tc(1, Cout, Cin, Tp, sms, 16);
  *gx_bn = px.bn;
  *gx_splits = px.splits;
  *gw_bn = pw.bn;
  *gw_splits = pw.stream_k ? -1 : pw.splits;  // -1: stream-K
  *in_sequence = gemms_in_sequence_on(T, Cin, Cout, Tp, sms) ? 1 : 0;
  *gx_pair = px.pair;
  *gw_pair = pw.pair;
  return HLQ_OK;
}

hlq_status hlq_debug_wait_timeout(uint64_t limit_ns, int32_t* d_result, void* stream) {
  if (!d_result || limit_ns == 0 || limit_ns > 1000000000ull) return HLQ_ERR_INVALID_ARG;
  if (!aligned16(d_result)) return HLQ_ERR_ALIGN;
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  HLQ_TRY(launch_wait_timeout_probe(limit_ns, d_result, status,
                                    static_cast<cudaStream_t>(stream)));
  return HLQ_OK;
}

size_t hlq_debug_tc_gemm_ws_bytes(int64_t M, int64_t N) {
  return gemm_tc_split_ws_bytes(M, N);
}

hlq_status hlq_trace_begin(int capacity) {
  if (capacity <= 0 || capacity > (1 << 20)) return HLQ_ERR_INVALID_ARG;
  trace_free();
  g_trace.ev = new cudaEvent_t[2 * (size_t)capacity]();
  g_trace.name = new const char*[capacity]();
  for (int i = 0; i < 2 * capacity; ++i) {
    if (cudaEventCreate(&g_trace.ev[i]) != cudaSuccess) {
      g_trace.cap = i / 2;  // destroy what was created
      for (int j = 0; j < i; ++j) cudaEventDestroy(g_trace.ev[j]);
      delete[] g_trace.ev;
      delete[] g_trace.name;
      g_trace = Trace{};
      return HLQ_ERR_CUDA;
    }
  }
  g_trace.cap = capacity;
  g_trace.n = 0;
  g_trace.on = true;
  return HLQ_OK;
}

hlq_status hlq_trace_end(int* n_launches) {
  if (!n_launches) return HLQ_ERR_INVALID_ARG;
  g_trace.on = false;
  *n_launches = g_trace.n;
  for (int i = 0; i < g_trace.n; ++i)
    if (cudaEventSynchronize(g_trace.ev[2 * i + 1]) != cudaSuccess)
      return HLQ_ERR_CUDA;
  return HLQ_OK;
}

hlq_status hlq_trace_get(int i, const char** name, float* ms) {
  if (!name || !ms || i < 0 || i >= g_trace.n) return HLQ_ERR_INVALID_ARG;
  *name = g_trace.name[i];
  if (cudaEventElapsedTime(ms, g_trace.ev[2 * i], g_trace.ev[2 * i + 1]) !=
      cudaSuccess)
    return HLQ_ERR_CUDA;
  return HLQ_OK;
}

hlq_status hlq_trace_free(void) {
  trace_free();
  return HLQ_OK;
}

hlq_status hlq_read_device_status(uint32_t* flags, int clear, void* stream) {
  if (!flags) return HLQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int* status = device_status_ptr();
  if (!status) return HLQ_ERR_CUDA;
  unsigned int v = 0;
  HLQ_TRY(cudaMemcpyAsync(&v, status, 4, cudaMemcpyDeviceToHost, s));
  if (clear) HLQ_TRY(cudaMemsetAsync(status, 0, 4, s));
  HLQ_TRY(cudaStreamSynchronize(s));
  *flags = v;
  return HLQ_OK;
}

const char* hlq_status_string(int status) {
  switch (status) {
    case HLQ_OK: return "HLQ_OK";
    case HLQ_ERR_INVALID_ARG: return "HLQ_ERR_INVALID_ARG";
    case HLQ_ERR_SHAPE: return "HLQ_ERR_SHAPE";
    case HLQ_ERR_ALIGN: return "HLQ_ERR_ALIGN";
    case HLQ_ERR_UNSUPPORTED: return "HLQ_ERR_UNSUPPORTED";
    case HLQ_ERR_WORKSPACE: return "HLQ_ERR_WORKSPACE";
    case HLQ_ERR_OVERFLOW: return "HLQ_ERR_OVERFLOW";
    case HLQ_ERR_CUDA: return "HLQ_ERR_CUDA";
    default: return "HLQ_UNKNOWN_STATUS";
  }
}

int hlq_version(void) { return 0x000100; }

}  // extern "C"
