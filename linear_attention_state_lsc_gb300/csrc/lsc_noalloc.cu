// lsc_noalloc.cu -- lsc_gdn_recurrent_noalloc: the chunked resumed-prefill
// recurrence for callers that cannot allocate device memory.
//
// Who needs it: code that may not allocate device memory at call time -- a
// serving loop that must keep its device-memory footprint fixed after
// start-up, a host framework whose own allocator owns the GPU's memory and
// forbids other allocations, or a latency-critical path that cannot afford
// the synchronisation an allocation may bring.  lsc_gdn_recurrent's chunked order
// needs scratch for the per-chunk records (a caller buffer or a
// stream-ordered allocation); this entry point uses instead a scratch array
// that lives in the library's own device image, so nothing is allocated at
// call time.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes; every
// GPU that loads the library holds it until the process exits.  Host code
// cannot use the variable's name as a device address (in host code it names
// a host-side stand-in), so the first call on each device -- with that device
// current -- asks the runtime for the array's device address
// (cudaGetSymbolAddress) and keeps it; that first call should therefore come
// before any stream capture.  Later calls on the device reuse the address.
//
// Every call shares the one array and finds it as the last call left it.
// Nothing in it has to start at zero: the first kernel of a call writes every
// record the second kernel reads.  Calls whose work overlaps on the GPU (on
// different streams, or different host threads) race on the array and must
// be ordered by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "lsc.h"
#include "lsc_chunk.h"
#include "lsc_internal.h"

namespace lsc {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;  // 64 MiB per device
static_assert(kNoAllocScratchBytes % 256 == 0, "whole 256-byte granules");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device.
class ScratchAddress {
 public:
  cudaError_t get(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (addr_[dev] == nullptr) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      addr_[dev] = p;
    }
    *out = addr_[dev];
    return cudaSuccess;
  }

 private:
  void *addr_[kMaxDevices] = {};
  std::mutex mu_;
};

ScratchAddress g_scratch_address;

}  // namespace
}  // namespace lsc

extern "C" {

int lsc_gdn_recurrent_noalloc(lsc_pool *pool, int32_t layer, const lsc_gdn_recurrent_args *args, void *stream) {
  if (!pool || !args) return LSC_ERR_INVALID_ARG;
  if (args->algorithm != LSC_RECURRENT_AUTO && args->algorithm != LSC_RECURRENT_CHUNKED) return LSC_ERR_INVALID_ARG;
  if (args->workspace != nullptr || args->workspace_bytes != 0) return LSC_ERR_INVALID_ARG;
  if (args->n_seq < 0 || args->total_tokens < 0) return LSC_ERR_INVALID_ARG;
  lsc_gdn_recurrent_args a = *args;
  a.algorithm = LSC_RECURRENT_CHUNKED;
  size_t need = 0;
  int rc = lsc_gdn_recurrent_workspace_bytes(pool, &a, &need);
  if (rc != LSC_OK) return rc;
  if (need > lsc::kNoAllocScratchBytes) return LSC_ERR_NO_MEMORY;  // the call does not fit the array
  void *scratch = nullptr;
  if (lsc::g_scratch_address.get(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_CUDA;
  }
  a.workspace = scratch;
  a.workspace_bytes = lsc::kNoAllocScratchBytes;
  return lsc_gdn_recurrent(pool, layer, &a, stream);  // a caller workspace: no allocation on this path
}

}  // extern "C"
