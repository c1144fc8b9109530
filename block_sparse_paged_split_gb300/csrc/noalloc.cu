// wise_decode_noalloc: the one-call decode for callers that cannot allocate
// device memory.
//
// Some callers may not call cudaMalloc at all: a caller running inside a
// CUDA-graph capture it does not own, a plugin whose host framework forbids
// allocations outside its own pool, or an embedded runtime that sizes every
// allocation up front.  They cannot provide the workspace that wise_decode
// takes, so this entry point runs the same three kernels (compaction, split
// partial, finish) over a scratch area that lives in this library's own
// static device memory instead.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes
// (16 MiB).  Every GPU that loads the library keeps it until the process
// exits.  Host code cannot use the array's name as a device address, so the
// first call on each device looks the address up with cudaGetSymbolAddress
// (with that device current) and caches it; that first call may load this
// module's device code, so make it before any stream capture begins.
//
// Every call on a device shares the one array and it keeps whatever the last
// call left there.  Nothing in it has to start at zero: each call's
// compaction writes every word the later kernels read.  Two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array and corrupt each other's results.
#include <mutex>

#include "internal.h"

namespace wise {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once
// per device).
wise_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_error(WISE_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return record_error(WISE_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return record_error(WISE_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return WISE_OK;
}

}  // namespace
}  // namespace wise

extern "C" wise_status wise_decode_noalloc(const wise_shape* shape, const void* q,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* page_table, const int32_t* seq_lens,
                                           const int8_t* modes, uint32_t* support, void* out,
                                           float* lse, wise_stream_t stream) {
  size_t need = 0;
  wise_status st = wise_workspace_bytes(shape, &need);
  if (st != WISE_OK) return st;
  if (need > wise::kNoAllocScratchBytes)
    return wise::record_error(WISE_ERR_WORKSPACE,
                              "this shape needs a %zu-byte workspace; the static scratch of "
                              "wise_decode_noalloc holds %zu bytes (use wise_decode)",
                              need, wise::kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((st = wise::scratch_address(&scratch)) != WISE_OK) return st;
  return wise_decode(shape, q, k_cache, v_cache, page_table, seq_lens, modes, support, out, lse,
                     scratch, wise::kNoAllocScratchBytes, stream);
}
