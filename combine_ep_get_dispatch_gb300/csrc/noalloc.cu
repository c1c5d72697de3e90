// Routing layout without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they need
// the layout: code that runs inside a host framework whose caching allocator
// owns the GPU's memory (a raw cudaMalloc would bypass its accounting and can
// fail once the pool has reserved most of HBM), plug-ins that are handed only
// their input and output buffers, and latency-critical loops where a
// cudaMalloc may synchronise the device. For them this file keeps the
// layout's scratch (the per-chunk counters and the grid-barrier word) in a
// fixed file-scope device array and passes it to the same kernel that
// ep_get_dispatch_layout launches.
//
// The array costs every GPU that loads the library kStaticScratchBytes of
// memory until the process exits. Every call shares it and it keeps the last
// call's contents; each call zeroes the barrier words first (the layout's
// own calls leave them zero, but a caller of this entry point cannot clear
// the array after a timed-out call), and the counters are rewritten in full.
// Calls that overlap on the GPU (for example on two streams without ordering
// between them) race on it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "ep.h"
#include "kernels.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_layout_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device. In host code the array's name is only a host-side stand-in, so the
// address must come from the runtime.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || !p) return EP_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return EP_OK;
}

}  // namespace

extern "C" int ep_get_dispatch_layout_noalloc(const ep_layout_t* L, int32_t* status, void* stream) {
  if (!L) return EP_ERR_INVALID_ARG;
  const size_t need =
      ep_layout_workspace_bytes(L->num_tokens, L->num_topk, L->num_experts, L->num_ranks);
  if (need == 0) return EP_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return EP_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != EP_OK) return rc;
  // The same checks as ep_get_dispatch_layout come first, so an argument
  // error enqueues nothing; then the array's 256-byte barrier block is
  // zeroed on the stream, then the layout runs.
  return ep::layout_call(L, scratch, kStaticScratchBytes, status, static_cast<cudaStream_t>(stream), true);
}
