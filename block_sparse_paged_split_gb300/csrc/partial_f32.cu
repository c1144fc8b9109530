// Instantiations of the split partial kernel for f32 K/V (head dim 64
// and 128, query heads per KV head 1, 2, 4, 8).
#include "partial_kernel.cuh"

namespace wise {

cudaError_t launch_partial_f32(const KParams& kp, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                  const void* q, const int32_t* page_table, const int32_t* seq_lens,
                                  const int8_t* modes, const WsView& ws, const FoldArgs& fa,
                                  cudaStream_t stream) {
  if (kp.D == 128)
    return launch_partial_d<float, 128>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, fa, stream);
  return launch_partial_d<float, 64>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, fa, stream);
}

}  // namespace wise
