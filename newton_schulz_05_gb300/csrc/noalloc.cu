// muon_step_static: the Muon step with its workspace in a static device
// array, for callers that cannot allocate device memory.
//
// Who needs it: a host runtime that reserves nearly all of the GPU's memory
// for its own pooled allocator at start-up (a serving engine or a training
// framework with a fixed arena) leaves nothing for a library's cudaMalloc,
// and a caller running a latency-bound loop cannot afford cudaMalloc, which
// may block and synchronise the device.  This entry point takes no workspace
// argument and allocates nothing: its scratch is the file-scope array below,
// of a fixed size, held by every GPU that loads the library until exit.
//
// Set-up: the array's name is, in host code, a host-side stand-in and not a
// device address.  The first call on each device, with that device current,
// asks the runtime for the array's device address (cudaGetSymbolAddress)
// and caches it per device.  Make that first call before any stream capture.
// The cache assumes the device is not reset (cudaDeviceReset) afterwards.
//
// Sharing: every call uses the same array and finds the previous call's
// contents there.  The only value that must start at zero (the device error
// word in the header) is cleared on the caller's stream at every call; all
// other scratch is fully written before it is read.  Calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array.  muon_static_error reads the error word a step left behind.
#include <mutex>

#include "internal.h"

namespace {

__device__ __align__(256) unsigned char g_static_workspace[MUON_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
void* g_static_ptr[kMaxDevices];
std::mutex g_static_mu;

// The static array of the current device; `stream` must belong to it.
muon_status static_workspace(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MUON_ERR_CUDA;
  int sdev = dev;
  if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return MUON_ERR_CUDA;
  if (sdev != dev) return MUON_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return MUON_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return MUON_OK;
}

}  // namespace

extern "C" muon_status muon_step_static(const muon_plan_t* plan, void* const* params,
                                        const void* const* grads, float* const* momentum,
                                        float lr, float beta, float wd, int nesterov,
                                        int ns_steps, const float* coeffs, void* stream) {
  if (!plan) return MUON_ERR_INVALID_ARG;
  size_t need = 0;
  muon_status st = muon_plan_workspace_bytes(plan, &need);
  if (st != MUON_OK) return st;
  if (need > (size_t)MUON_STATIC_WORKSPACE_BYTES) return MUON_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  st = static_workspace(s, &ws);
  if (st != MUON_OK) return st;
  if (cudaMemsetAsync(ws, 0, muon::kHeaderBytes, s) != cudaSuccess) return MUON_ERR_CUDA;
  return muon_step(plan, params, grads, momentum, lr, beta, wd, nesterov, ns_steps, coeffs, ws,
                   (size_t)MUON_STATIC_WORKSPACE_BYTES, stream);
}

extern "C" muon_status muon_static_error(void* stream, int clear, int* code) {
  if (!code) return MUON_ERR_INVALID_ARG;
  void* ws = nullptr;
  const muon_status st = static_workspace(static_cast<cudaStream_t>(stream), &ws);
  if (st != MUON_OK) return st;
  return muon_workspace_error(ws, stream, clear, code);
}
