// bsfa_noalloc.cu -- bsfa_prefill_fwd_noalloc: the gated prefill for callers
// that cannot allocate device memory at call time.
//
// Some callers must not call cudaMalloc (or any allocator) when they run
// attention: code inside a CUDA graph that is being captured, real-time
// serving loops that pre-plan every byte of device memory up front, plugins
// hosted by a framework that owns the allocator, and embedded runtimes with a
// fixed memory map.  bsfa_prefill_fwd asks such callers for a workspace
// buffer; this entry point needs none.  Its scratch (the per-call sequence
// table and the heaviest-first tile schedule written by the scheduling pass)
// lives in a fixed array in device memory that belongs to the library and is
// set aside when the library is loaded, on every GPU that loads it, until the
// process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "bsfa.h"

namespace {

// Fixed scratch: 256 KiB per device.  A call needs
// bsfa_prefill_workspace_size(p) bytes of it (a few bytes per sequence and per
// 128-row query tile); larger requests are rejected.
constexpr size_t kScratchBytes = 256u * 1024u;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name stands for a host-side shadow, not for device memory, so
// the device address is looked up once per device (with that device current)
// and cached.
void* scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" bsfa_status bsfa_prefill_fwd_noalloc(const bsfa_fwd_params* p, bsfa_stream_t stream) {
  if (p == nullptr) return BSFA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSFA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BSFA_ERR_UNSUPPORTED;
  const size_t need = bsfa_prefill_workspace_size(p);
  if (need == 0) return BSFA_ERR_INVALID_ARG;
  if (need > kScratchBytes) return BSFA_ERR_UNSUPPORTED;  // beyond the fixed scratch
  void* scratch = scratch_address(dev);
  if (scratch == nullptr) return BSFA_ERR_CUDA;
  bsfa_fwd_params q = *p;
  q.workspace = scratch;
  q.workspace_bytes = kScratchBytes;
  return bsfa_prefill_fwd(&q, stream);
}
