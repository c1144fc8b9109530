// Compaction of support masks into a balanced list of work items, the
// support unions (across depths and across a row's KV heads), and the batch
// validator.
//
// [WISE PR, "What changes"]: sparse rows walk only their selected tiles,
// compacted first so the loop has no branch; programs cover about eight
// tiles, so one long dense row does not set the latency of a launch whose
// other rows are sparse.  Every (row, KV head)'s blocks are cut into ranges
// of tiles_per_item blocks; a range's tiles (all of them, or the selected
// ones for a sparse row) form one work item.  The cut depends only on that
// row's own mode, length and mask, so a row's result does not depend on the
// rest of the batch.
#include "internal.h"
#include "list1.cuh"

namespace wise {

constexpr int kCompactThreads = 1024;
constexpr int kCompactCluster = 8;  // CTAs of the one cluster the kernel runs as

// Work items are block ranges: item (rg, s) holds the tiles of (row, KV head)
// rg that lie in blocks [s*T, s*T + T) -- all of them for dense and discover
// rows, the selected ones for sparse rows (no item when none is).  A row's
// split therefore depends only on its own length, mode and mask, and a
// sparse row with every block selected splits exactly like a dense row.
// Item (rg, s) writes its partial output to slot rg * S_max + s.
//
// An item record carries its compacted tiles as a bitmap over its range:
// x = rg, y = s | s << 16 (range, and the partial slot it writes), z = tile
// bitmap (bit i: block s*T + i) | tile count << 16, w = row length | sparse
// << 24 | discover << 25.  The partial pass walks the
// set bits in order (the k-th tile is the k-th set bit), so its inner loop
// has no branch and needs no list in memory.
//
// Compaction writes the items already in schedule order, which is the order
// the partial pass hands them out (through an atomic counter): tile count
// descending, so the last warps do not finish long items alone.
//
// Work is flattened to one unit per (row, KV head, range) and spread over
// the threads of one thread-block cluster (8 CTAs of 1024 threads).  Every
// global load a unit needs (the row's mode and length, the range's mask word)
// goes out at once, so the kernel makes one memory round trip.  Phase A
// counts each unit's tiles into its CTA's histogram of item sizes
// (warp-aggregated shared-memory atomics), and the thread of a pair's range 0
// writes the pair's head info (a sparse pair's tile and item counts start at
// 0).  After a cluster barrier every CTA reads the others' histograms through
// distributed shared memory and works out where its items of each size start
// in the schedule (larger sizes first, then lower CTA ranks), so no counter
// in global memory has to be reset between calls.  Phase B writes each item
// at its schedule slot, adds a sparse range's tiles to its pair's counts and
// marks the partial slots of a sparse row's empty ranges.
struct UnitInfo {
  uint32_t bits;  // tiles of the range (bit i: block s*T + i)
  int L, flags;
  bool sparse;
  int raw;        // the row's length before clamping
};

// The loads of one unit (issued together; nothing here waits on them), all
// after the dependency wait: the row's mode, length and mask slot (the
// caller's inputs, possibly written by the kernel before this one), then the
// mask word (possibly written by the previous call's finish pass).
struct UnitLoad {
  int mode, raw, slot;
  uint32_t word;
};

__device__ __forceinline__ void unit_load_inputs(UnitLoad& l, int u, int nunits,
                                                 const int8_t* __restrict__ modes,
                                                 const int32_t* __restrict__ seq_lens,
                                                 const MaskView& mv, const KParams& kp) {
  l = UnitLoad{-1, 0, -1, 0u};
  if (u < nunits) {
    const int r = u / kp.S_max / kp.Hkv;
    l.mode = modes[r];
    l.raw = seq_lens[r];
    l.slot = mask_slot(mv, r);
  }
}

__device__ __forceinline__ void unit_load_mask(UnitLoad& l, int u, int nunits,
                                               const MaskView& mv, const KParams& kp) {
  if (u < nunits && l.slot >= 0) {
    const int pair = u / kp.S_max, s = u - pair * kp.S_max;
    // s * T < max_blocks <= 32 W: the word is inside the pair's mask.
    l.word = mask_of(mv, l.slot, pair % kp.Hkv, kp.W)[(s * kp.T) >> 5];
  }
}

__device__ __forceinline__ UnitLoad unit_load(int u, int nunits, const int8_t* __restrict__ modes,
                                              const int32_t* __restrict__ seq_lens,
                                              const MaskView& mv, const KParams& kp) {
  UnitLoad l;
  unit_load_inputs(l, u, nunits, modes, seq_lens, mv, kp);
  unit_load_mask(l, u, nunits, mv, kp);
  return l;
}

__device__ __forceinline__ UnitInfo unit_info(int u, const UnitLoad& l, const KParams& kp) {
  UnitInfo ui{0u, 0, 0, false, 0};
  if (l.mode < 0) return ui;  // past the last unit
  const int s = u % kp.S_max;
  ui.raw = l.raw;
  ui.L = clamp_len(l.raw, kp.cap_tokens);
  ui.sparse = l.mode == WISE_MODE_SPARSE;
  ui.flags = (ui.sparse ? kItemSparse : 0) |
             (l.mode == WISE_MODE_DISCOVER || l.mode == WISE_MODE_DISCOVER_UNION ? kItemDiscover : 0);
  const int nb = (ui.L + kTile - 1) / kTile;
  const int lo = s * kp.T;
  if (lo < nb) {
    const int n = min(kp.T, nb - lo);
    const uint32_t full = n >= 32 ? 0xffffffffu : (1u << n) - 1u;
    // T is a power of two up to 16, so a range never straddles mask words.
    ui.bits = ui.sparse ? (l.word >> (lo & 31)) & full : full;
  }
  return ui;
}

__global__ void __cluster_dims__(kCompactCluster, 1, 1) __launch_bounds__(kCompactThreads)
    compact_kernel(const int8_t* __restrict__ modes, const int32_t* __restrict__ seq_lens,
                   const MaskView mv, const WsView ws, const KParams kp) {
  __shared__ int hist[kMaxT + 1];                     // this CTA's items of each size
  __shared__ int next[kMaxT + 1];                     // its next schedule slot of each size
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();
  const int nthreads = kCompactCluster * kCompactThreads;
  const int gt = (int)crank * kCompactThreads + threadIdx.x;
  const int S = kp.S_max;
  const int nunits = kp.R * kp.Hkv * S;

  // The thread's units are u = gt + i * nthreads; the first kCached stay in
  // registers between the two phases (more are looked up again in phase B).
  constexpr int kCached = 4;
  const int rounds = (nunits + nthreads - 1) / nthreads;
  UnitLoad ld[kCached];
  // Everything is read after the dependency wait: the mask comes from the
  // previous call, and the caller's inputs may come from the kernel before
  // this one (its writes are only certain to be visible past the wait).
  grid_dependency_wait();
  grid_dependents_launch();  // the partial pass may start its prologue now
#pragma unroll
  for (int c = 0; c < kCached; ++c) {
    ld[c] = UnitLoad{-1, 0, -1, 0u};
    if (c < rounds) unit_load_inputs(ld[c], c * nthreads + gt, nunits, modes, seq_lens, mv, kp);
  }
#pragma unroll
  for (int c = 0; c < kCached; ++c)
    if (c < rounds) unit_load_mask(ld[c], c * nthreads + gt, nunits, mv, kp);
  if (gt == 0) {
    *ws.status = 0;
    *ws.queue = 0;
    *ws.queue_done = 0;
  }
  if (gt < kMaxT) ws.l1_counter[gt] = 0;  // a finish building list 1 appends from 0
  if (threadIdx.x <= kMaxT) hist[threadIdx.x] = 0;
  __syncthreads();
  auto unit = [&](int i, int u) {
    if (i < kCached) {
      UnitLoad l{-1, 0, -1, 0u};
#pragma unroll
      for (int c = 0; c < kCached; ++c)
        if (c == i) l = ld[c];
      return unit_info(u, l, kp);
    }
    return unit_info(u, unit_load(u, nunits, modes, seq_lens, mv, kp), kp);
  };

  // Phase A: this CTA's histogram of item sizes; head info from each pair's
  // range 0.
  for (int i = 0; i < rounds; ++i) {
    const int u = i * nthreads + gt;
    const UnitInfo ui = unit(i, u);
    const int n = __popc(ui.bits);
    const unsigned same = __match_any_sync(kFull, n);
    if (n > 0 && lane == __ffs(same) - 1) atomicAdd(&hist[n], __popc(same));
    if (u < nunits && u % S == 0) {
      const int pair = u / S;
      const int nb = (ui.L + kTile - 1) / kTile;
      const int nr = (nb + kp.T - 1) / kp.T;
      ws.head_info[pair] = ui.sparse ? make_int4(pair * S, nr, 0, 0) : make_int4(pair * S, nr, nb, nr);
      ws.tickets[pair] = 0;
    }
  }
  cluster_arrive();  // histograms complete; head info and the resets above visible
  cluster_wait();
  // Warp 0: lane sz reads every CTA's count of items of size sz (distributed
  // shared memory, all loads in flight together), then a suffix sum over the
  // lanes gives the items of larger sizes.  Schedule: sizes T..1; within a
  // size, CTA 0's items first.
  if (threadIdx.x < 32) {
    const int sz = lane;
    int cnt[kCompactCluster];
#pragma unroll
    for (int c = 0; c < kCompactCluster; ++c)
      cnt[c] = (sz >= 1 && sz <= kp.T) ? load_peer(&hist[sz], c) : 0;
    int tot = 0, mine_before = 0;
#pragma unroll
    for (int c = 0; c < kCompactCluster; ++c) {
      tot += cnt[c];
      if (c < (int)crank) mine_before += cnt[c];
    }
    int suffix = tot;  // items of size >= sz
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(kFull, suffix, o);
      if (lane + o < 32) suffix += y;
    }
    if (sz >= 1 && sz <= kp.T) next[sz] = suffix - tot + mine_before;
    if (gt == 0) *ws.num_items = suffix;  // lane 0 (size 0 holds nothing)
  }
  cluster_arrive();  // this CTA is done reading the others' shared memory
  __syncthreads();

  // Phase B: item records at their schedule slots, sparse pairs' counts,
  // empty-range markers.
  for (int i = 0; i < rounds; ++i) {
    const int u = i * nthreads + gt;
    const int pair = u / S, s = u - pair * S;
    const UnitInfo ui = unit(i, u);
    const int n = __popc(ui.bits);
    const unsigned same = __match_any_sync(kFull, n);
    const int leader = __ffs(same) - 1;
    int slot = 0;
    if (n > 0 && lane == leader) slot = atomicAdd(&next[n], __popc(same));
    slot = __shfl_sync(kFull, slot, leader);
    if (n > 0) {
      ws.items[slot + __popc(same & ((1u << lane) - 1u))] =
          make_int4(pair, s | (s << 16), (int)(ui.bits | ((uint32_t)n << 16)), ui.L | ui.flags);
      if (ui.sparse) {
        atomicAdd(&ws.head_info[pair].z, n);
        atomicAdd(&ws.head_info[pair].w, 1);
      }
    } else if (u < nunits && ui.sparse && s * kp.T < (ui.L + kTile - 1) / kTile) {
      // An empty range of a sparse row: mark its partial slot so the finish
      // pass skips it.
      for (int h = 0; h < kp.G; ++h) {
        ws.partial_ml[((size_t)pair * S + s) * kp.G + h] = make_float2(-INFINITY, 0.f);
        ws.partial_ml_other[((size_t)pair * S + s) * kp.G + h] = make_float2(-INFINITY, 0.f);
      }
    }
    if (u < nunits && s == 0 && pair % kp.Hkv == 0 && ui.raw > kp.cap_tokens)
      flag_error(ws.status, WISE_DEVERR_SEQ_LEN_CLAMPED);
  }
  cluster_wait();  // no CTA leaves while another may still read its histogram
}

cudaError_t launch_compact(const KParams& kp, const int8_t* modes, const int32_t* seq_lens,
                           const MaskView& mv, const WsView& ws, cudaStream_t stream) {
  return launch_pdl(compact_kernel, dim3(kCompactCluster), dim3(kCompactThreads), 0, stream, modes,
                    seq_lens, mv, ws, kp);
}

// ------------------------------------------------------------------ list 1 from the modes and masks
// The work list of a call built from its rows' modes, lengths and masks alone:
// one CTA per (row, KV head) appends the pair's items to list 1 (compact
// slots, one bucket per tile count: the list a finish with
// WISE_FLAG_BUILD_SPARSE_LIST writes) -- a sparse row's selected ranges, from
// its mask words copied to shared memory, or every range of a dense or
// discover row.  modes null: every row sparse.  The work is the pair's W words
// and its ranges with a tile to attend, so an all-sparse call's cost follows
// the selection, where compaction visits every block range of every row.
constexpr int kBuildThreads = 128;

__global__ void __launch_bounds__(kBuildThreads)
    build_list_kernel(const int8_t* __restrict__ modes, const int32_t* __restrict__ seq_lens,
                      const MaskView mv, const WsView ws, const KParams kp) {
  __shared__ uint32_t words[WISE_MAX_BLOCKS / 32];
  __shared__ List1Smem sm;
  const int rg = blockIdx.x;
  const int r = rg / kp.Hkv, g = rg - r * kp.Hkv;
  grid_dependency_wait();  // the inputs and the mask may come from the kernel before
  grid_dependents_launch();  // the partial pass may start its prologue now
  const int raw = seq_lens[r];
  const int L = clamp_len(raw, kp.cap_tokens);
  const int mode = modes ? (int)modes[r] : (int)WISE_MODE_SPARSE;
  const bool sparse = mode == WISE_MODE_SPARSE;
  const uint32_t* mw = sparse ? mask_of(mv, mask_slot(mv, r), g, kp.W) : nullptr;
  if (threadIdx.x == 0 && g == 0 && raw > kp.cap_tokens)
    flag_error(ws.status, WISE_DEVERR_SEQ_LEN_CLAMPED);
  if (L == 0 || (sparse && mw == nullptr)) {  // nothing to attend: no item
    if (threadIdx.x == 0) list1_empty_pair(ws, kp, rg);
    return;
  }
  if (sparse) {
    for (int i = threadIdx.x; i < kp.W; i += blockDim.x) words[i] = mw[i];
    __syncthreads();
  }
  const int flags = sparse ? kItemSparse
                           : (mode == WISE_MODE_DISCOVER || mode == WISE_MODE_DISCOVER_UNION
                                  ? kItemDiscover : 0);
  list1_build_pair(ws, kp, rg, L, words, !sparse, flags, sm);
}

cudaError_t launch_build_list(const KParams& kp, const int8_t* modes, const int32_t* seq_lens,
                              const MaskView& mv, const WsView& ws, cudaStream_t stream) {
  if (kp.R == 0) return cudaSuccess;
  // A pair's ranges in one pass of the CTA's threads: one warp (its barriers
  // are then a warp's) up to 32 ranges, four warps beyond.
  const int threads = kp.S_max <= 32 ? 32 : kBuildThreads;
  return launch_pdl(build_list_kernel, dim3(kp.R * kp.Hkv), dim3(threads), 0, stream, modes,
                    seq_lens, mv, ws, kp);
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

// ------------------------------------------------------------- head union
// [WISE PR, "What changes", FlashAttention decode bullet]: sparse rows attend
// the head union of their support.  One thread per (row, mask word): the OR
// of the row's KV heads' words, written back to every head.
__global__ void head_union_kernel(uint32_t* __restrict__ support, int R, int Hkv, int W) {
  grid_dependency_wait();  // the mask from the previous kernel
  grid_dependents_launch();
  const int64_t n = (int64_t)R * W;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / W, w = i - r * W;
    uint32_t* base = support + r * Hkv * W + w;
    uint32_t u = 0u;
    for (int g = 0; g < Hkv; ++g) u |= base[(int64_t)g * W];
    for (int g = 0; g < Hkv; ++g) base[(int64_t)g * W] = u;
  }
}

cudaError_t launch_head_union(const KParams& kp, uint32_t* support, cudaStream_t stream) {
  const int64_t n = (int64_t)kp.R * kp.W;
  if (n == 0) return cudaSuccess;
  int grid = (int)((n + 255) / 256);
  const int cap = sm_count() * 4;
  if (grid > cap) grid = cap;
  return launch_pdl(head_union_kernel, dim3(grid), dim3(256), 0, stream, support, kp.R, kp.Hkv,
                    kp.W);
}

// --------------------------------------------------------------- validate
__global__ void validate_kernel(const int32_t* __restrict__ page_table,
                                const int32_t* __restrict__ seq_lens,
                                const int8_t* __restrict__ modes, const MaskView mv,
                                int32_t* err, const KParams kp) {
  const int r = blockIdx.x;
  const int raw = seq_lens[r];
  const int mode = modes[r];
  if (threadIdx.x == 0) {
    if (mode < 0 || mode > 3) atomicOr(err, WISE_BAD_MODE);
    if (raw < 0 || raw > kp.cap_tokens) atomicOr(err, WISE_BAD_SEQ_LEN);
    if (mv.row_slot) {
      const int sl = mv.row_slot[r];
      if (sl < -1 || (mv.num_slots > 0 && sl >= mv.num_slots)) atomicOr(err, WISE_BAD_SLOT);
    }
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
    const int slot = mask_slot(mv, r);
    for (int g = threadIdx.x; g < kp.Hkv; g += blockDim.x) {
      bool any = false;
      if (slot >= 0) {
        const uint32_t* words = mask_of(mv, slot, g, kp.W);
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
                            const int32_t* seq_lens, const int8_t* modes, const MaskView& mv,
                            int32_t* err_word, cudaStream_t stream) {
  if (kp.R == 0) return cudaSuccess;
  validate_kernel<<<kp.R, 128, 0, stream>>>(page_table, seq_lens, modes, mv, err_word, kp);
  return cudaGetLastError();
}

}  // namespace wise
