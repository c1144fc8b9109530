// Self-test of the failure path without a fault.
//
// Every wait of the library's kernels on an mbarrier (a producer's copies, a
// consumer's release) is bounded by %globaltimer: a wait that runs out sets
// WISE_DEVERR_WAIT_TIMEOUT in a status word and lets the kernel return,
// instead of hanging the GPU.  This entry point runs that mechanism on a
// barrier nothing ever arrives on, so a caller can check on its own device
// that the wait gives up, that the status reaches the host, and that the
// context stays usable afterwards.  The pages have no counterpart; it
// computes nothing of the method.
#include "internal.h"

namespace wise {

__global__ void wait_timeout_kernel(int32_t* __restrict__ status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // No thread arrives and no copy completes on `bar`: the wait for its first
  // phase runs out after the library's wait limit.  Nothing is in flight.
  const bool done = mbar_wait(b, 0);
  if (!done && threadIdx.x == 0) flag_error(status, WISE_DEVERR_WAIT_TIMEOUT);
}

}  // namespace wise

extern "C" wise_status wise_selftest_wait_timeout(int32_t* status_word, wise_stream_t stream) {
  if (!status_word || (reinterpret_cast<uintptr_t>(status_word) & 3) != 0)
    return wise::record_error(WISE_ERR_INVALID_ARG, "status_word must be a 4-byte aligned device pointer");
  wise::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status_word);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return wise::record_error(WISE_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return WISE_OK;
}
