// ring_noalloc.cu -- cpattn_ring for callers that cannot allocate device
// memory.
//
// cpattn_ring needs a caller-provided fp32 workspace for the running merged
// output and LSE.  Some callers cannot provide one: code that runs where
// cudaMalloc is not allowed or not wanted (inside a framework's memory pool
// that hands out no extra buffers, in a process with a fixed device-memory
// budget, or in a plugin that only receives its input and output pointers).
// This entry point takes its workspace from a fixed array in the library's
// own device memory instead, so the caller passes inputs and outputs only.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// bytes.  Every GPU that loads this library holds it until the process
// exits.  Host code cannot use the array's name as a device address, so on
// the first call on each device this file looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it; that first
// call should therefore happen before any stream capture.  All calls share
// the one array: two calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on it.  The kernel writes every
// workspace element it later reads, so nothing has to be cleared between
// calls.  No call here allocates or frees device memory.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;   // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_ring_scratch[kNoAllocScratchBytes];

std::mutex g_lock;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_ring_scratch on the current device (looked up once per
// device), or nullptr on failure.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_ring_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

size_t cpattn_ring_noalloc_max_workspace_bytes(void) { return kNoAllocScratchBytes; }

cpattn_status cpattn_ring_noalloc(const cpattn_tensor* q, const cpattn_tensor* k,
                                  const cpattn_tensor* v, float scale, int ring_degree,
                                  int ring_anything, cpattn_tensor* out, cpattn_tensor* lse,
                                  void* stream) {
  if (!q) return CPATTN_ERR_NULL;
  const size_t need = cpattn_ring_workspace_bytes(q, ring_degree);
  if (need > kNoAllocScratchBytes) return CPATTN_ERR_WORKSPACE;
  void* scratch = scratch_on_current_device();
  if (scratch == nullptr) return CPATTN_ERR_CUDA;
  return cpattn_ring(q, k, v, scale, ring_degree, ring_anything, out, lse, scratch,
                     kNoAllocScratchBytes, stream);
}

}  // extern "C"
