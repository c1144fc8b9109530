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

// Work items are block ranges: item (rg, s) holds the tiles of (row, KV head)
// rg that lie in blocks [s*T, s*T + T) -- all of them for dense and discover
// rows, the selected ones for sparse rows (skipped when none is).  A row's
// split therefore depends only on its own length, mode and mask, and a
// sparse row with every block selected splits exactly like a dense row.
// Item (rg, s) writes its partial output to slot rg * S_max + s.
//
// Compaction writes the items already in schedule order, which is the order
// the partial pass hands them out (through an atomic counter): tile count
// descending, so the last warps do not finish long items alone.  Each record
// is self-contained: x = rg, y = first index in the tile list (sparse) or
// first block (otherwise), z = tiles | flags | s << 8, w = row length.
//
// Phase A, a thread per (row, KV head): item and tile counts and a
// histogram of item sizes (warp-aggregated shared-memory atomics).
// Phase B, the same thread: its item records at their schedule slots,
// empty-range markers for sparse rows, and its tile list.
__device__ __forceinline__ int range_count(bool sparse, const uint32_t* words, int s, int T,
                                           int nb) {
  const int lo = s * T;
  if (lo >= nb) return 0;
  const int n = min(T, nb - lo);
  if (!sparse) return n;
  if (!words) return 0;
  // T is at most 16 and a power of two here, so a range never straddles words.
  const uint32_t w = words[lo >> 5] >> (lo & 31);
  return __popc(w & ((1u << n) - 1u));
}

__global__ void __launch_bounds__(kCompactThreads)
    compact_kernel(const int8_t* __restrict__ modes, const int32_t* __restrict__ seq_lens,
                   const uint32_t* __restrict__ support, const int32_t* __restrict__ page_table,
                   const WsView ws, const KParams kp) {
  grid_dependency_wait();
  grid_dependents_launch();  // the partial pass may start its prologue now
  __shared__ int warp_tot[32];
  __shared__ int size_slot[17];  // items per size (1..T), then the next schedule slot
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    *ws.status = 0;
    *ws.queue = 0;
    *ws.queue_done = 0;
  }
  for (int i = threadIdx.x; i <= 16; i += blockDim.x) size_slot[i] = 0;
  __syncthreads();
  const int npair = kp.R * kp.Hkv;
  const int T = kp.T;
  const int S = kp.S_max;

  // Phase A: counts and the size histogram.
  int carry_items = 0;
  for (int base = 0; base < npair; base += kCompactThreads) {
    const int idx = base + threadIdx.x;
    const bool valid = idx < npair;
    int nb = 0, nitems = 0, count = 0;
    bool sparse = false;
    const uint32_t* words = nullptr;
    if (valid) {
      const int r = idx / kp.Hkv;
      const int raw = seq_lens[r];
      const int L = clamp_len(raw, kp.cap_tokens);
      if (raw > kp.cap_tokens && idx % kp.Hkv == 0) flag_error(ws.status, WISE_DEVERR_SEQ_LEN_CLAMPED);
      nb = (L + kTile - 1) / kTile;
      sparse = modes[r] == WISE_MODE_SPARSE;
      words = (sparse && support) ? support + (size_t)idx * kp.W : nullptr;
    }
    for (int s = 0; s < S; ++s) {
      const int n = valid ? range_count(sparse, words, s, T, nb) : 0;
      count += n;
      nitems += n > 0;
      const unsigned same = __match_any_sync(kFull, n);
      if (n > 0 && lane == __ffs(same) - 1) atomicAdd(&size_slot[n], __popc(same));
    }
    if (valid) ws.head_info[idx] = make_int4(idx * S, (nb + T - 1) / T, count, nitems);
    int tot = 0;
    block_exclusive_scan(nitems, warp_tot, &tot);
    carry_items += tot;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    *ws.num_items = carry_items;
    int run = 0;
    for (int sz = T; sz >= 1; --sz) {
      const int n = size_slot[sz];
      size_slot[sz] = run;
      run += n;
    }
  }
  __syncthreads();

  // Phase B: item records at their schedule slots, empty-range markers,
  // tile lists.
  for (int base = 0; base < npair; base += kCompactThreads) {
    const int idx = base + threadIdx.x;
    const bool valid = idx < npair;
    int r = 0, nb = 0, L = 0, flags = 0;
    bool sparse = false;
    const uint32_t* words = nullptr;
    if (valid) {
      r = idx / kp.Hkv;
      L = clamp_len(seq_lens[r], kp.cap_tokens);
      nb = (L + kTile - 1) / kTile;
      const int mode = modes[r];
      sparse = mode == WISE_MODE_SPARSE;
      words = (sparse && support) ? support + (size_t)idx * kp.W : nullptr;
      flags = (sparse ? kItemSparse : 0) |
              (mode == WISE_MODE_DISCOVER || mode == WISE_MODE_DISCOVER_UNION ? kItemDiscover : 0);
    }
    int first = 0;  // index into this pair's tile list (sparse rows)
    for (int s = 0; s < S; ++s) {
      const int n = valid ? range_count(sparse, words, s, T, nb) : 0;
      const unsigned same = __match_any_sync(kFull, n);
      const int leader = __ffs(same) - 1;
      int slot = 0;
      if (n > 0 && lane == leader) slot = atomicAdd(&size_slot[n], __popc(same));
      slot = __shfl_sync(kFull, slot, leader);
      if (n > 0) {
        ws.items[slot + __popc(same & ((1u << lane) - 1u))] =
            make_int4(idx, sparse ? first : s * T, n | flags | (s << 8), L);
      } else if (sparse && s * T < nb) {
        // An empty range of a sparse row: mark its partial slot so the
        // finish pass skips it.
        for (int h = 0; h < kp.G; ++h)
          ws.partial_ml[((size_t)idx * S + s) * kp.G + h] = make_float2(-INFINITY, 0.f);
      }
      first += n;
    }
    if (sparse && words) {
      // Each selected tile with its page ids, so the partial pass needs one
      // load per tile (pages past the row's length are never read: 0).
      const int32_t* pt = page_table + (size_t)r * kp.max_pages;
      const int ppt = kTile / kp.P;  // pages per tile: 2 or 1
      int4* list = ws.tile_list + (size_t)idx * kp.max_blocks;
      int k = 0;
      for (int w = 0; w * 32 < nb; ++w) {
        const int lo = w * 32;
        uint32_t bits = words[w] & (lo + 32 <= nb ? 0xffffffffu : (1u << (nb - lo)) - 1u);
        while (bits) {
          const int b = lo + __ffs(bits) - 1;
          const int pg = b * ppt;
          const bool two = ppt == 2 && b * kTile + kp.P < L;
          list[k++] = make_int4(b, pt[pg], two ? pt[pg + 1] : 0, 0);
          bits &= bits - 1;
        }
      }
    }
  }
}

cudaError_t launch_compact(const KParams& kp, const int8_t* modes, const int32_t* seq_lens,
                           const uint32_t* support, const int32_t* page_table, const WsView& ws,
                           cudaStream_t stream) {
  return launch_pdl(compact_kernel, dim3(1), dim3(kCompactThreads), 0, stream, modes, seq_lens,
                    support, page_table, ws, kp);
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
