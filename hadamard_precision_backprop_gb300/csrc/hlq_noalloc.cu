// hlq_noalloc.cu -- hlq_linear_backward_gx_noalloc: the g_x path of
// hlq_linear_backward_gx for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code hosted inside another
// runtime that owns all device memory and hands none out to plugins, or
// latency-critical loops that forbid cudaMalloc/cudaFree after start-up
// (both can synchronize the device).  This entry point needs neither a
// workspace argument nor any allocation: its scratch (the int4 codes of g_y
// and w, stored one E4M3 byte per code for the tensor-core GEMM, their
// scales and the amax slots) lives in one fixed device array of this
// library, kNoAllocScratchBytes long, which every GPU that loads the library
// holds until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "hlq.h"
#include "hlq_kernels.h"

namespace hlq {
namespace {

// 40 MiB: enough for T * Cout + Cin * Cout code bytes plus the scales of a
// ViT-B-sized layer (T = 12608, Cin = 768, Cout = 2304 needs about 31 MB).
constexpr size_t kNoAllocScratchBytes = (size_t)40 << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device, looked up the
// first time this device calls in (host code only knows the array by a
// host-side stand-in symbol, which must never reach a kernel).
hlq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return HLQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
      return HLQ_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return HLQ_OK;
}

}  // namespace
}  // namespace hlq

extern "C" hlq_status hlq_linear_backward_gx_noalloc(
    const void* d_gy, const void* d_w, int dt, int64_t T, int64_t Cin, int64_t Cout,
    int block, int gran_gy, int gran_w, int rnd, uint64_t seed, float* d_gx,
    void* stream) {
  if (T < 0 || Cin < 0 || Cout < 0) return HLQ_ERR_SHAPE;
  // sizes whose scratch would not fit the fixed array are refused up front
  if (T > ((int64_t)1 << 40) || Cin > ((int64_t)1 << 40) || Cout > ((int64_t)1 << 40) ||
      hlq::gx_workspace_bytes(T, Cin, Cout) > hlq::kNoAllocScratchBytes)
    return HLQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  const hlq_status st = hlq::scratch_address(&scratch);
  if (st != HLQ_OK) return st;
  return hlq::backward_gx_with_ws(d_gy, d_w, dt, T, Cin, Cout, block, gran_gy, gran_w,
                                  rnd, seed, d_gx, scratch, hlq::kNoAllocScratchBytes,
                                  stream);
}

extern "C" size_t hlq_noalloc_scratch_bytes(void) { return hlq::kNoAllocScratchBytes; }
