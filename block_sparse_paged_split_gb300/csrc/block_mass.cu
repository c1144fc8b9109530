// Block masses rebuilt from the LSE by a second read of K: the discovery of
// the FlashAttention decode path, kept as an ablation of the in-pass tile
// statistics.
//
// [WISE PR, "What changes", FlashAttention decode bullet]: discovery rereads
// K once to rebuild block mass from the attention's LSE.  For every
// discovery row r, query head h and block b:
//
//   l_b = sum_{j in b, j < L_r} 2^(s_j - lse2_h),  s_j = scale log2(e) <q_h, k_j>,
//
// written to the tile statistics as (lse2_h, l_b), so the finish pass's
// p_b = l_b 2^(m_b - lse2) is the block's softmax mass and its selection
// runs unchanged.  One warp per (row, KV head, block): the warp reads each of
// the block's 32 key rows with one coalesced load (lane: its slice; all 32
// loads in flight together, kept in registers for every query head of the
// group), the partial dot products are transposed through shared memory so
// lane t sums token t's score, then a warp sum per query head.
#include <type_traits>

#include "internal.h"

namespace wise {

constexpr int kMassWarps = 8;

// A lane's DPL consecutive elements of a row, as loaded (one vector load:
// the row slices are 8- or 16-byte aligned) and widened to float.
template <typename T, int DPL>
struct Slice;

template <int DPL>
struct Slice<__nv_bfloat16, DPL> {
  using Raw = typename std::conditional<DPL == 4, uint2, uint32_t>::type;
  static __device__ __forceinline__ Raw load(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const Raw*>(p));
  }
  static __device__ __forceinline__ void widen(const Raw& v, float (&x)[DPL]) {
    if constexpr (DPL == 4) {
      x[0] = Elem<__nv_bfloat16>::lo(v.x); x[1] = Elem<__nv_bfloat16>::hi(v.x);
      x[2] = Elem<__nv_bfloat16>::lo(v.y); x[3] = Elem<__nv_bfloat16>::hi(v.y);
    } else {
      x[0] = Elem<__nv_bfloat16>::lo(v); x[1] = Elem<__nv_bfloat16>::hi(v);
    }
  }
};

template <int DPL>
struct Slice<float, DPL> {
  using Raw = typename std::conditional<DPL == 4, float4, float2>::type;
  static __device__ __forceinline__ Raw load(const float* p) {
    return __ldg(reinterpret_cast<const Raw*>(p));
  }
  static __device__ __forceinline__ void widen(const Raw& v, float (&x)[DPL]) {
    if constexpr (DPL == 4) {
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
      x[0] = v.x; x[1] = v.y;
    }
  }
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kMassWarps * 32)
    block_mass_kernel(const T* __restrict__ q, const T* __restrict__ k_cache,
                      const int32_t* __restrict__ page_table, const int32_t* __restrict__ seq_lens,
                      const int8_t* __restrict__ modes, const float* __restrict__ lse,
                      const WsView ws, const KParams kp) {
  constexpr int DPL = D / 32;
  __shared__ float part_all[kMassWarps][kTile * 33];
  grid_dependency_wait();  // the LSE from the previous finish pass
  grid_dependents_launch();
  const int lane = threadIdx.x & 31;
  float* part = part_all[threadIdx.x >> 5];
  const int64_t n_units = (int64_t)kp.R * kp.Hkv * kp.max_blocks;
  const int64_t stride = (int64_t)gridDim.x * kMassWarps;
  for (int64_t u = (int64_t)blockIdx.x * kMassWarps + (threadIdx.x >> 5); u < n_units; u += stride) {
    const int b = (int)(u % kp.max_blocks);
    const int rg = (int)(u / kp.max_blocks);
    const int r = rg / kp.Hkv, g = rg - r * kp.Hkv;
    const int mode = modes[r];
    if (mode != WISE_MODE_DISCOVER && mode != WISE_MODE_DISCOVER_UNION) continue;
    const int L = clamp_len(seq_lens[r], kp.cap_tokens);
    const int tok0 = b * kTile;
    if (tok0 >= L) continue;
    const int n_valid = min(kTile, L - tok0);
    // The block spans one or two pages; a page id outside the pool reads
    // zeros, as do tokens past the row's length.
    const int32_t* pt = page_table + (size_t)r * kp.max_pages + tok0 / kp.P;
    const int pg0 = pt[0];
    const int pg1 = (kp.P * 2 == kTile && tok0 + kp.P < L) ? pt[1] : -1;
    // All 32 key rows of the block are loaded before any is used (the lane
    // keeps its slices in registers for every query head of the group).
    using S = Slice<T, DPL>;
    typename S::Raw raw[kTile];
#pragma unroll
    for (int i = 0; i < kTile; ++i) {
      const int page = i < kp.P ? pg0 : pg1;
      raw[i] = typename S::Raw{};
      if (i < n_valid && page >= 0 && page < kp.num_pages)
        raw[i] = S::load(k_cache + (((size_t)page * kp.P + (i % kp.P)) * kp.Hkv + g) * D + lane * DPL);
    }
#pragma unroll 1
    for (int hl = 0; hl < G; ++hl) {
      const int h = g * G + hl;
      float qv[DPL];
      S::widen(S::load(q + ((size_t)r * kp.Hq + h) * D + lane * DPL), qv);
      // Token i's partial dot over this lane's elements goes to part[i][lane].
#pragma unroll
      for (int i = 0; i < kTile; ++i) {
        float kx[DPL];
        S::widen(raw[i], kx);
        float a = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) a = fmaf(qv[d], kx[d], a);
        part[i * 33 + lane] = a;
      }
      __syncwarp();
      // Lane t sums token t's 32 partials (row stride 33: no bank conflict).
      float st = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) st += part[lane * 33 + k];
      __syncwarp();
      const float lse2 = lse[(size_t)r * kp.Hq + h] * kLog2e;
      const float e = (lane < n_valid && lse2 > -INFINITY) ? fast_exp2(st * kp.scale_log2 - lse2) : 0.f;
      const float lb = warp_sum(e);
      if (lane == 0) ws.tile_stats[((size_t)r * kp.Hq + h) * kp.max_blocks + b] = make_float2(lse2, lb);
    }
  }
}

template <typename T, int D>
static cudaError_t launch_mass_d(const KParams& kp, const void* q, const void* k_cache,
                                 const int32_t* page_table, const int32_t* seq_lens,
                                 const int8_t* modes, const float* lse, const WsView& ws,
                                 cudaStream_t stream) {
  const int grid = sm_count() * 8;  // grid-stride over the blocks
  const T* qt = static_cast<const T*>(q);
  const T* kt = static_cast<const T*>(k_cache);
  switch (kp.G) {
    case 1: return launch_pdl(block_mass_kernel<T, D, 1>, dim3(grid), dim3(kMassWarps * 32), 0, stream, qt, kt, page_table, seq_lens, modes, lse, ws, kp);
    case 2: return launch_pdl(block_mass_kernel<T, D, 2>, dim3(grid), dim3(kMassWarps * 32), 0, stream, qt, kt, page_table, seq_lens, modes, lse, ws, kp);
    case 4: return launch_pdl(block_mass_kernel<T, D, 4>, dim3(grid), dim3(kMassWarps * 32), 0, stream, qt, kt, page_table, seq_lens, modes, lse, ws, kp);
    case 8: return launch_pdl(block_mass_kernel<T, D, 8>, dim3(grid), dim3(kMassWarps * 32), 0, stream, qt, kt, page_table, seq_lens, modes, lse, ws, kp);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
static cudaError_t launch_mass_t(const KParams& kp, const void* q, const void* k_cache,
                                 const int32_t* page_table, const int32_t* seq_lens,
                                 const int8_t* modes, const float* lse, const WsView& ws,
                                 cudaStream_t stream) {
  if (kp.D == 128)
    return launch_mass_d<T, 128>(kp, q, k_cache, page_table, seq_lens, modes, lse, ws, stream);
  return launch_mass_d<T, 64>(kp, q, k_cache, page_table, seq_lens, modes, lse, ws, stream);
}

cudaError_t launch_block_mass(int dtype, const KParams& kp, const void* q, const void* k_cache,
                              const int32_t* page_table, const int32_t* seq_lens,
                              const int8_t* modes, const float* lse, const WsView& ws,
                              cudaStream_t stream) {
  if (kp.R == 0) return cudaSuccess;
  if (dtype == WISE_DTYPE_BF16)
    return launch_mass_t<__nv_bfloat16>(kp, q, k_cache, page_table, seq_lens, modes, lse, ws, stream);
  return launch_mass_t<float>(kp, q, k_cache, page_table, seq_lens, modes, lse, ws, stream);
}

}  // namespace wise
