// spa_noalloc.cu - decode entry point that allocates nothing.
//
// Some callers cannot allocate device memory at the point where they decode: a runtime whose
// allocator is owned by someone else, or an embedded host with no allocator hooks.  For them the
// split-K partials live in a scratch array compiled into this library instead of in a caller
// workspace.
//
// The array is a file-scope __device__ object, so every GPU that loads the library holds it
// until the process exits.  In host code its name is only a host-side stand-in, never a device
// address: the first call on each device, with that device current, asks the runtime for the
// real address (cudaGetSymbolAddress) and keeps it for later calls on that device.
#include <cuda_runtime.h>

#include <mutex>

#include "sparse_attn_paged.h"
#include "spa_launch.h"

namespace {

constexpr size_t kScratchBytes = SPA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device (set up once per device).
int scratch_on_current_device(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return SPA_OK;
}

}  // namespace

extern "C" int sparse_attn_paged_decode_noalloc(const void* q, const spa_pool_t* win,
                                                const spa_pool_t* cmp, const spa_problem_t* prob,
                                                void* out, void* stream) {
  if (!prob) return SPA_ERR_NULL;
  // The partials of this problem must fit the built-in array (with as few as one split); no
  // larger buffer can be had here.
  if (spa::decode_partials_bytes(prob, kScratchBytes) > kScratchBytes) return SPA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_on_current_device(&scratch);
  if (st != SPA_OK) return st;
  return spa::decode_with_partials(q, win, cmp, prob, out, scratch, kScratchBytes, stream);
}
