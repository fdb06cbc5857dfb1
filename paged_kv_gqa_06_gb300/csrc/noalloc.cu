// forge_paged_gqa_decode_noalloc: the paged GQA decode for callers that must
// not allocate device memory.
//
// Some callers cannot allocate device memory at the point where they decode:
// processes that size their device memory once at start-up -- for example a
// serving loop that has handed everything left to its KV-block pool, where a
// later allocation fails or takes memory the pool counts on -- and callers
// that run under a memory manager of their own (an embedding runtime or a
// framework allocator) that forbids allocations it did not make.
// forge_paged_gqa_decode may allocate its split scratch on first use; this
// entry point never does.  Its scratch is the file-scope array below, which
// every GPU that loads this module holds for the life of the process.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/forge_paged.h"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(FORGE_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;
constexpr int kFallbackSplitTokens = 1024;  // largest split: smallest scratch

// Split scratch shared by every call of forge_paged_gqa_decode_noalloc on a
// device.  It is never cleared by this file: its split arrival counters are
// zero at load (static device memory is zero-initialised) and every completed
// decode returns them to zero, and every other value the decode reads from
// it is written earlier in the same call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FORGE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FORGE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FORGE_OK;
}

}  // namespace

extern "C" int forge_paged_gqa_decode_noalloc(const forge_tensor* q, const forge_tensor* k_cache,
                                              const forge_tensor* v_cache, const forge_tensor* block_tables,
                                              const forge_tensor* context_lens, float scale, forge_tensor* out,
                                              void* stream) {
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != FORGE_OK) return rc;
  // The automatic split length first; if its scratch does not fit, the
  // longest split, which needs the least.  Both checks happen on the host
  // before anything is enqueued.
  rc = forge_paged_gqa_decode_ex(q, k_cache, v_cache, block_tables, context_lens, scale, out, scratch,
                                 kScratchBytes, 0, stream);
  if (rc != FORGE_ERR_WORKSPACE) return rc;
  return forge_paged_gqa_decode_ex(q, k_cache, v_cache, block_tables, context_lens, scale, out, scratch,
                                   kScratchBytes, kFallbackSplitTokens, stream);
}
