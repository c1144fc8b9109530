// Compaction of support masks into tile lists and a balanced work list,
// the standalone support union, and the batch validator.
//
// [WISE PR, "What changes"]: sparse rows walk only their selected tiles,
// compacted first so the loop has no branch; programs cover about eight
// tiles, so one long dense row does not set the latency of a launch whose
// other rows are sparse.  The work list cuts every (row, KV head)'s tile list
// in order into items of at most tiles_per_item tiles; the cut depends only
// on that row's own mode, length and mask, so a row's result does not depend
// on the rest of the batch.
#include "internal.h"

namespace wise {

constexpr int kCompactThreads = 1024;

// Block-wide exclusive scan of one int per thread; returns the block total
// through *total.  Uses `warp_tot` (32 ints of shared memory).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int nw = blockDim.x >> 5;
    int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, t, o);
      if (lane >= o) t += y;
    }
    if (lane < nw) warp_tot[lane] = t;
  }
  __syncthreads();
  const int base = wid ? warp_tot[wid - 1] : 0;
  *total = warp_tot[(blockDim.x >> 5) - 1];
  __syncthreads();
  return base + incl - v;
}

__global__ void __launch_bounds__(kCompactThreads)
    compact_kernel(const int8_t* __restrict__ modes, const int32_t* __restrict__ seq_lens,
                   const uint32_t* __restrict__ support, const WsView ws, const KParams kp) {
  __shared__ int warp_tot[32];
  if (threadIdx.x == 0) *ws.status = 0;
  __syncthreads();
  const int npair = kp.R * kp.Hkv;
  int carry = 0;
  for (int base = 0; base < npair; base += kCompactThreads) {
    const int idx = base + threadIdx.x;
    int count = 0, nitems = 0, r = 0, g = 0, nb = 0;
    bool sparse = false;
    if (idx < npair) {
      r = idx / kp.Hkv;
      g = idx - r * kp.Hkv;
      const int raw = seq_lens[r];
      const int L = clamp_len(raw, kp.cap_tokens);
      if (raw > kp.cap_tokens && g == 0) flag_error(ws.status, WISE_DEVERR_SEQ_LEN_CLAMPED);
      nb = (L + kTile - 1) / kTile;
      sparse = modes[r] == WISE_MODE_SPARSE;
      if (sparse) {
        if (support != nullptr) {
          const uint32_t* words = support + (size_t)idx * kp.W;
          for (int w = 0; w * 32 < nb; ++w) {
            const int lo = w * 32;
            const uint32_t valid = lo + 32 <= nb ? 0xffffffffu : (1u << (nb - lo)) - 1u;
            count += __popc(words[w] & valid);
          }
        }
      } else {
        count = nb;
      }
      nitems = (count + kp.T - 1) / kp.T;
    }
    int total = 0;
    const int first = carry + block_exclusive_scan(nitems, warp_tot, &total);
    if (idx < npair) {
      ws.head_info[idx] = make_int4(first, nitems, count, 0);
      for (int s = 0; s < nitems; ++s) {
        const int t0 = s * kp.T;
        ws.items[first + s] = make_int4(r, g, t0, min(kp.T, count - t0));
      }
      if (sparse && count > 0) {
        const uint32_t* words = support + (size_t)idx * kp.W;
        int32_t* list = ws.tile_list + (size_t)idx * kp.max_blocks;
        int k = 0;
        for (int w = 0; w * 32 < nb; ++w) {
          const int lo = w * 32;
          uint32_t bits = words[w] & (lo + 32 <= nb ? 0xffffffffu : (1u << (nb - lo)) - 1u);
          while (bits) {
            list[k++] = lo + __ffs(bits) - 1;
            bits &= bits - 1;
          }
        }
      }
    }
    carry += total;
  }
  if (threadIdx.x == 0) *ws.num_items = carry;
}

cudaError_t launch_compact(const KParams& kp, const int8_t* modes, const int32_t* seq_lens,
                           const uint32_t* support, const WsView& ws, cudaStream_t stream) {
  compact_kernel<<<1, kCompactThreads, 0, stream>>>(modes, seq_lens, support, ws, kp);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ union
__global__ void union_kernel(uint32_t* __restrict__ dst, const uint32_t* __restrict__ src,
                             int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15) == 0;
  if (vec) {
    const int64_t n4 = n / 4;
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (int64_t j = i; j < n4; j += stride) {
      uint4 a = d4[j];
      const uint4 b = s4[j];
      a.x |= b.x; a.y |= b.y; a.z |= b.z; a.w |= b.w;
      d4[j] = a;
    }
    for (int64_t j = n4 * 4 + i; j < n; j += stride) dst[j] |= src[j];
  } else {
    for (int64_t j = i; j < n; j += stride) dst[j] |= src[j];
  }
}

cudaError_t launch_union(uint32_t* dst, const uint32_t* src, int64_t n_words, cudaStream_t stream) {
  if (n_words <= 0) return cudaSuccess;
  const int64_t work = (n_words + 3) / 4;
  int grid = (int)((work + 255) / 256);
  const int cap = sm_count() * 8;
  if (grid > cap) grid = cap;
  union_kernel<<<grid, 256, 0, stream>>>(dst, src, n_words);
  return cudaGetLastError();
}

// --------------------------------------------------------------- validate
__global__ void validate_kernel(const int32_t* __restrict__ page_table,
                                const int32_t* __restrict__ seq_lens,
                                const int8_t* __restrict__ modes,
                                const uint32_t* __restrict__ support, int32_t* err,
                                const KParams kp) {
  const int r = blockIdx.x;
  const int raw = seq_lens[r];
  const int mode = modes[r];
  if (threadIdx.x == 0) {
    if (mode < 0 || mode > 3) atomicOr(err, WISE_BAD_MODE);
    if (raw < 0 || raw > kp.cap_tokens) atomicOr(err, WISE_BAD_SEQ_LEN);
  }
  const int L = clamp_len(raw, kp.cap_tokens);
  const int npg = (L + kp.P - 1) / kp.P;
  const int32_t* pt = page_table + (size_t)r * kp.max_pages;
  for (int i = threadIdx.x; i < npg; i += blockDim.x) {
    const int p = pt[i];
    if (p < 0 || p >= kp.num_pages) atomicOr(err, WISE_BAD_PAGE);
  }
  if (mode == WISE_MODE_SPARSE && L > 0) {
    const int nb = (L + kTile - 1) / kTile;
    for (int g = threadIdx.x; g < kp.Hkv; g += blockDim.x) {
      bool any = false;
      if (support != nullptr) {
        const uint32_t* words = support + ((size_t)r * kp.Hkv + g) * kp.W;
        for (int w = 0; w * 32 < nb; ++w) {
          const int lo = w * 32;
          any |= (words[w] & (lo + 32 <= nb ? 0xffffffffu : (1u << (nb - lo)) - 1u)) != 0;
        }
      }
      if (!any) atomicOr(err, WISE_EMPTY_SPARSE_SUPPORT);
    }
  }
}

cudaError_t launch_validate(const KParams& kp, const int32_t* page_table,
                            const int32_t* seq_lens, const int8_t* modes,
                            const uint32_t* support, int32_t* err_word, cudaStream_t stream) {
  if (kp.R == 0) return cudaSuccess;
  validate_kernel<<<kp.R, 128, 0, stream>>>(page_table, seq_lens, modes, support, err_word, kp);
  return cudaGetLastError();
}

}  // namespace wise
