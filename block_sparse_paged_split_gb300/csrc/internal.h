// Host-side declarations shared by the library's translation units.
#pragma once

#include "common.cuh"

namespace wise {

// Launchers (host).  Each enqueues one kernel on `stream` and returns the
// launch status; none allocates or synchronises.
cudaError_t launch_compact(const KParams& kp, const int8_t* modes, const int32_t* seq_lens,
                           const uint32_t* support, const WsView& ws, cudaStream_t stream);

cudaError_t launch_partial_bf16(const KParams& kp, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const void* q, const int32_t* page_table, const int32_t* seq_lens,
                                const int8_t* modes, const WsView& ws, cudaStream_t stream);
cudaError_t launch_partial_f32(const KParams& kp, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const void* q, const int32_t* page_table, const int32_t* seq_lens,
                               const int8_t* modes, const WsView& ws, cudaStream_t stream);

cudaError_t launch_finish(int dtype, const KParams& kp, const int8_t* modes,
                          const int32_t* seq_lens, const WsView& ws, uint32_t* support,
                          void* out, float* lse, cudaStream_t stream);

cudaError_t launch_union(uint32_t* dst, const uint32_t* src, int64_t n_words,
                         cudaStream_t stream);

cudaError_t launch_validate(const KParams& kp, const int32_t* page_table,
                            const int32_t* seq_lens, const int8_t* modes,
                            const uint32_t* support, int32_t* err_word, cudaStream_t stream);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Records a printf-style reason for wise_last_error() and returns `status`.
wise_status record_error(wise_status status, const char* fmt, ...);

}  // namespace wise
