// Host-side declarations shared by the library's translation units.
#pragma once

#include <utility>

#include "common.cuh"

namespace wise {

// Launchers (host).  Each enqueues one kernel on `stream` and returns the
// launch status; none allocates or synchronises.
cudaError_t launch_compact(const KParams& kp, const int8_t* modes, const int32_t* seq_lens,
                           const MaskView& mv, const WsView& ws, cudaStream_t stream);

// Where the finish pass writes when it is folded into the partial pass
// (out == nullptr: not folded).
struct FoldArgs {
  uint32_t* support;  // [R, Hkv, W] (the folded finish takes flat masks only)
  void* out;
  float* lse;
};

// The folded finish handles rows of at most 64 blocks and 8 split slots.
inline bool can_fold_finish(const KParams& kp) { return kp.S_max <= 8 && kp.max_blocks <= 64; }

cudaError_t launch_partial_bf16(const KParams& kp, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const void* q, const int32_t* page_table, const int32_t* seq_lens,
                                const int8_t* modes, const WsView& ws, const FoldArgs& fa,
                                cudaStream_t stream);
cudaError_t launch_partial_f32(const KParams& kp, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const void* q, const int32_t* page_table, const int32_t* seq_lens,
                               const int8_t* modes, const WsView& ws, const FoldArgs& fa,
                               cudaStream_t stream);

cudaError_t launch_finish(int dtype, const KParams& kp, const int8_t* modes,
                          const int32_t* seq_lens, const WsView& ws, const MaskView& mv,
                          void* out, float* lse, cudaStream_t stream);

cudaError_t launch_union(uint32_t* dst, const uint32_t* src, int64_t n_words,
                         cudaStream_t stream);

cudaError_t launch_head_union(const KParams& kp, uint32_t* support, cudaStream_t stream);

cudaError_t launch_block_mass(int dtype, const KParams& kp, const void* q, const void* k_cache,
                              const int32_t* page_table, const int32_t* seq_lens,
                              const int8_t* modes, const float* lse, const WsView& ws,
                              cudaStream_t stream);

cudaError_t launch_validate(const KParams& kp, const int32_t* page_table,
                            const int32_t* seq_lens, const int8_t* modes, const MaskView& mv,
                            int32_t* err_word, cudaStream_t stream);

// Launches `kern` as a programmatic dependent of the previous kernel in the
// stream: its CTAs may start while that kernel finishes, and every kernel of
// this library calls grid_dependency_wait() before it reads anything an
// earlier kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Records a printf-style reason for wise_last_error() and returns `status`.
wise_status record_error(wise_status status, const char* fmt, ...);

}  // namespace wise
