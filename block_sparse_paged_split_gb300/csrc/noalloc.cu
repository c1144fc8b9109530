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
// first call in each CUDA context looks the address up with
// cudaGetSymbolAddress (with that context's device current) and caches it
// under the context handle; that first call may load this module's device
// code, so make it before any stream capture begins.  A cudaDeviceReset
// destroys the context the cached address belongs to: make no call between
// the reset and the next first call in the new context (a new context
// normally gets a new handle; if the driver hands back the same handle the
// stale address would be used, so re-create state after a reset before
// calling again).
//
// Every call on a device shares the one array and it keeps whatever the last
// call left there.  Nothing in it has to start at zero: each call's
// compaction writes every word the later kernels read.  Two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array and corrupt each other's results.  The kernels report device-side
// conditions (a bounded wait that gave up, a clamped sequence length) in the
// array's status word; wise_noalloc_status copies it to the host, since a
// caller of this entry point has no workspace of its own to read it from.
#include <mutex>

#include "internal.h"

namespace wise {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Cached scratch addresses, one per CUDA context that has called in.
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mu;
struct ScratchEntry {
  CUcontext ctx;
  void* ptr;
};
ScratchEntry g_scratch[kMaxContexts] = {};
int g_scratch_used = 0;
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_get_current = nullptr;

// Device address of the scratch array in the current context (looked up once
// per context).
wise_status scratch_address(void** out) {
  cudaError_t e;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_ctx_get_current) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return record_error(WISE_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS)
    return record_error(WISE_ERR_CUDA, "cuCtxGetCurrent failed");
  if (ctx)
    for (int i = 0; i < g_scratch_used; ++i)
      if (g_scratch[i].ctx == ctx) {
        *out = g_scratch[i].ptr;
        return WISE_OK;
      }
  if (g_scratch_used == kMaxContexts)
    return record_error(WISE_ERR_UNSUPPORTED, "more than %d CUDA contexts", kMaxContexts);
  // With no context current yet, this runtime call makes the current
  // device's primary context current, and the address belongs to it.
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr)
    return record_error(WISE_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
  if (!ctx && (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx))
    return record_error(WISE_ERR_CUDA, "no current CUDA context");
  g_scratch[g_scratch_used++] = ScratchEntry{ctx, p};
  *out = p;
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

extern "C" wise_status wise_noalloc_status(int32_t* host_status, wise_stream_t stream) {
  if (!host_status) return wise::record_error(WISE_ERR_INVALID_ARG, "host_status is NULL");
  void* scratch = nullptr;
  wise_status st = wise::scratch_address(&scratch);
  if (st != WISE_OK) return st;
  // The status word is the first int32 of the workspace layout.
  cudaError_t e = cudaMemcpyAsync(host_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return wise::record_error(WISE_ERR_CUDA, "status copy: %s", cudaGetErrorString(e));
  return WISE_OK;
}
