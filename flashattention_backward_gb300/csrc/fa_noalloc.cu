// fa_backward_static_workspace: the full backward pass (preprocess, main
// kernel, convert) for callers that cannot allocate device memory.
//
// fa_backward needs two scratch buffers besides its inputs and outputs: the
// per-row D = rowsum(O * dO) and the fp32 dQ accumulator.  Some callers cannot
// provide them: code that runs inside a host framework or plugin interface
// that owns all device memory and forbids allocation while it executes, a
// process whose device-memory budget is fixed at start-up, or a latency-bound
// loop that must not pay cudaMalloc's implicit device-wide synchronisation.
// This entry point takes its scratch from two fixed-size arrays defined in
// this file instead.  Every GPU that loads the library holds them (68 MiB)
// until the process exits.
//
// Set-up: the device addresses of the arrays are looked up with
// cudaGetSymbolAddress on the first call on each device, with that device
// current (host code cannot pass the symbols themselves: on the host they only
// name shadow variables).  Make that first call on a device before any stream
// capture on it.
//
// Sharing: every call on a device uses the same arrays, and they keep the last
// call's contents.  The preprocess kernel rewrites D and zeroes the
// accumulator at the start of every call, so nothing carries over from one
// call to the next, but calls whose kernels overlap on the GPU (different
// streams without ordering, or several host threads) race on the arrays and
// produce wrong results.  Order such calls on one stream.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kAccumFloats = size_t(16) << 20;  // 64 MiB of fp32 dQ accumulator
constexpr size_t kRowFloats = size_t(1) << 20;     // 4 MiB of fp32 D

static __device__ __align__(256) float g_static_dq_accum[kAccumFloats];
static __device__ __align__(256) float g_static_D[kRowFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_accum_ptr[kMaxDevices] = {nullptr};
float* g_D_ptr[kMaxDevices] = {nullptr};

// Device addresses of this device's arrays (looked up once per device).
bool static_workspace(float** D, float** accum) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_accum_ptr[dev]) {
    void* a = nullptr;
    void* d = nullptr;
    if (cudaGetSymbolAddress(&a, g_static_dq_accum) != cudaSuccess) return false;
    if (cudaGetSymbolAddress(&d, g_static_D) != cudaSuccess) return false;
    g_accum_ptr[dev] = static_cast<float*>(a);
    g_D_ptr[dev] = static_cast<float*>(d);
  }
  *D = g_D_ptr[dev];
  *accum = g_accum_ptr[dev];
  return true;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_backward_static_workspace(const fa_problem* p, const void* Q, const void* K, const void* V,
                                                  const void* O, const void* dO, const float* L, void* dQ,
                                                  void* dK, void* dV, void* stream) {
  fa::NvtxRange range("fa_backward_static_workspace");
  const size_t acc_elems = fa_dq_accum_elems(p);  // 0 when p is NULL or invalid
  if (acc_elems == 0) {
    // report the same code fa_backward's own validation gives; nothing launches
    return fa_backward(p, Q, K, V, O, dO, L, nullptr, nullptr, dQ, dK, dV, stream);
  }
  const size_t rows = (size_t)p->B * p->H * p->N;
  if (acc_elems > fa::kAccumFloats || rows > fa::kRowFloats) return FA_ERR_UNSUPPORTED;
  float* D = nullptr;
  float* acc = nullptr;
  if (!fa::static_workspace(&D, &acc)) return FA_ERR_CUDA;
  return fa_backward(p, Q, K, V, O, dO, L, D, acc, dQ, dK, dV, stream);
}
