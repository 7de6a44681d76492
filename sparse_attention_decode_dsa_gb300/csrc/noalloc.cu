// The fixed scratch of dsa_indexer_topk_noalloc: one file-scope device array, in a
// translation unit of its own.
//
// Callers that cannot allocate device memory (plugin hosts and serving runtimes that
// give the library no allocator and fix their memory budget up front, request paths
// that must not call cudaMalloc because it can synchronise the device) use this array as
// the indexer's workspace.  Every GPU that loads this module holds the array until the
// process exits.  With lazy module loading (the CUDA default) the module -- and so the
// array -- becomes resident on a device when noalloc_scratch() first looks up its address
// there; with CUDA_MODULE_LOADING=EAGER it is resident from context creation.
//
// In host code the array's name denotes a host-side stand-in, not device memory: a
// kernel handed it would fault or, where the GPU can reach host memory, silently use the
// wrong memory.  Its device address is therefore looked up with cudaGetSymbolAddress,
// once per device with that device current, and passed to the kernels as a pointer.
#include <mutex>

#include "dsa_internal.h"

namespace dsa {

namespace {
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
}  // namespace

cudaError_t noalloc_scratch(void** ptr, int* device) {
  *ptr = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  *device = dev;
  if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *ptr = g_addr[dev];
  return cudaSuccess;
}

}  // namespace dsa
