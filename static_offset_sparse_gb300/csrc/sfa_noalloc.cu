// Allocation-free forward: sfa_forward with its scratch in a fixed device array.
//
// Some callers cannot hand the library a workspace: the host program may own
// every byte of device memory through its own pool and forbid raw cudaMalloc
// from plugins, or run under a hard memory budget where a fresh allocation in
// the middle of a step can fail.  For them this entry point keeps the
// forward's scratch (the RoPE-rotated bf16 copy of K used by the tensor-core
// kernel) in a file-scope device array of SFA_STATIC_WS_BYTES that every GPU
// loading the library holds until the process exits.  The caller still
// provides q, k, v, o and lse.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "sfa_internal.h"

namespace {

// The scratch.  In host code this name is only a stand-in for the device
// symbol: its device address comes from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_static_ws[SFA_STATIC_WS_BYTES];

// Device address of g_static_ws on the current device.  It is looked up with
// that device current on the first call there and cached together with the
// context it belongs to; a call from another context of the same device (for
// instance after cudaDeviceReset made a fresh primary context) looks it up
// again, so a cached address never outlives its context.
int static_ws_address(void** out) {
  static std::mutex mu;
  static void* cache[64] = {nullptr};
  static CUcontext owner[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SFA_ERR_CUDA;
  const CUcontext ctx = sfa::current_context();  // nullptr before the first runtime call
  std::lock_guard<std::mutex> lock(mu);
  if (!ctx || !cache[dev] || owner[dev] != ctx) {
    void* p = nullptr;  // the lookup makes the device's primary context current if none was
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return SFA_ERR_CUDA;
    cache[dev] = p;
    owner[dev] = sfa::current_context();
  }
  *out = cache[dev];
  return SFA_OK;
}

}  // namespace

extern "C" int sfa_forward_noalloc(const sfa_desc* d, const void* q, const void* k, const void* v,
                                   void* o, float* lse, void* stream) {
  size_t need = 0;
  int rc = sfa_workspace_size(d, 1, 0, &need);
  if (rc != SFA_OK) return rc;
  if (need > (size_t)SFA_STATIC_WS_BYTES) return SFA_ERR_CAPACITY;
  void* ws = nullptr;
  if ((rc = static_ws_address(&ws)) != SFA_OK) return rc;
  // The scratch needs no clearing: the forward writes every K' row it reads
  // before reading it, on the same stream.
  return sfa_forward(d, q, k, v, o, lse, ws, (size_t)SFA_STATIC_WS_BYTES, stream);
}
