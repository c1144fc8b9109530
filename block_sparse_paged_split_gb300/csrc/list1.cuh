// List 1: the work list of a following all-sparse call, written by the finish
// pass that leaves the mask (WISE_FLAG_BUILD_SPARSE_LIST), so that call needs
// no compaction launch.
//
// [WISE PR, "What changes"]: sparse rows walk only their selected tiles,
// compacted first so the loop has no branch.  The finish of a discovery depth
// already holds every (row, KV head)'s final mask, so it cuts the pair's
// selected tiles into work items itself: item k of the pair holds the
// selected blocks of the k-th non-empty range [s*T, s*T + T) as a bitmap over
// the range and writes its split to partial slot rg * S_max + k (compact
// slots, so the finish that merges them needs no marker for empty ranges).
//
// Items go to one bucket per tile count (bucket n-1 at items_1 + (n-1) *
// max_items), each pair taking its positions with one atomicAdd per size it
// has.  The counters start at 0: compaction zeroes them, and so does the last
// CTA of every partial pass that is not itself on list 1 -- the finish that
// builds the list waits for its own call's partial pass to complete.  The
// partial pass on list 1 reads the counters and schedules larger items first
// (the order compaction writes), mapping a schedule position to its bucket.
#pragma once

#include "common.cuh"

namespace wise {

// Shared memory of one pair's list build.
struct List1Smem {
  int hist[kMaxT];   // the pair's items with j + 1 tiles
  int gbase[kMaxT];  // their first position in bucket j
  int cur[kMaxT];    // items of bucket j placed so far
  int wcnt[32];      // per-warp counts of one scan chunk
};

// The selected blocks of range s (blocks [s*T, s*T + T) below nb) as a bitmap
// over the range; mw holds the pair's mask words.  T <= 16 is a power of two,
// so a range never straddles a word.
__device__ __forceinline__ uint32_t list1_range_bits(const uint32_t* mw, int s, int T, int nb) {
  const int lo = s * T;
  if (lo >= nb) return 0u;
  const int n = min(T, nb - lo);
  const uint32_t full = n >= 32 ? 0xffffffffu : (1u << n) - 1u;
  return (mw[lo >> 5] >> (lo & 31)) & full;
}

// A pair with no item in list 1 (padding rows, masks selecting nothing).
__device__ __forceinline__ void list1_empty_pair(const WsView& ws, const KParams& kp, int rg) {
  ws.head_info_1[rg] = make_int4(rg * kp.S_max, 0, 0, 0);
}

// Every blocks of range s below nb (a row that attends all its blocks).
__device__ __forceinline__ uint32_t list1_range_full(int s, int T, int nb) {
  const int lo = s * T;
  if (lo >= nb) return 0u;
  const int n = min(T, nb - lo);
  return n >= 32 ? 0xffffffffu : (1u << n) - 1u;
}

// Every thread of the CTA calls this (blockDim.x a multiple of 32): the items
// of (row, KV head) rg, whose row holds L tokens, appended to list 1, and the
// pair's head info.  full: every block of the row (a dense or discover row);
// otherwise the blocks selected in the mask words mw (shared memory).  flags:
// the row's mode flags for the records (kItemSparse, kItemDiscover).
static __device__ __noinline__ void list1_build_pair(const WsView& ws, const KParams& kp, int rg,
                                                        int L, const uint32_t* mw, bool full,
                                                        int flags, List1Smem& sm) {
  const int th = threadIdx.x, nt = blockDim.x;
  const int lane = th & 31, warp = th >> 5, nw = nt >> 5;
  const int T = kp.T;
  const int nb = (L + kTile - 1) / kTile;
  const int nr = (nb + T - 1) / T;
  if (th < kMaxT) {
    sm.hist[th] = 0;
    sm.cur[th] = 0;
  }
  __syncthreads();
  for (int s = th; s < nr; s += nt) {
    const int n = __popc(full ? list1_range_full(s, T, nb) : list1_range_bits(mw, s, T, nb));
    if (n) atomicAdd(&sm.hist[n - 1], 1);
  }
  __syncthreads();
  if (th < T) {
    const int c = sm.hist[th];
    sm.gbase[th] = c ? atomicAdd(ws.l1_counter + th, c) : 0;
  }
  if (th == 0) {
    int items = 0, tiles = 0;
    for (int j = 0; j < T; ++j) {
      items += sm.hist[j];
      tiles += (j + 1) * sm.hist[j];
    }
    ws.head_info_1[rg] = make_int4(rg * kp.S_max, items, tiles, items);
  }
  __syncthreads();
  // Item k of the pair is its k-th non-empty range: a CTA-wide exclusive
  // count of the non-empty ranges before each, chunk by chunk.
  int carry = 0;
  for (int base = 0; base < nr; base += nt) {
    const int s = base + th;
    const uint32_t bits =
        s >= nr ? 0u : (full ? list1_range_full(s, T, nb) : list1_range_bits(mw, s, T, nb));
    const int n = __popc(bits);
    const unsigned bal = __ballot_sync(kFull, n > 0);
    if (lane == 0) sm.wcnt[warp] = __popc(bal);
    __syncthreads();
    int before = 0, tot = 0;
    for (int w2 = 0; w2 < nw; ++w2) {
      const int c = sm.wcnt[w2];
      before += w2 < warp ? c : 0;
      tot += c;
    }
    __syncthreads();
    if (n) {
      const int k = carry + before + __popc(bal & ((1u << lane) - 1u));
      const int pos = sm.gbase[n - 1] + atomicAdd(&sm.cur[n - 1], 1);
      // The counters start at 0 after any compaction of the workspace, so a
      // bucket never holds more than max_items; a position past it means the
      // call came out of order and the item is dropped.
      if (pos >= 0 && pos < ws.max_items)
        ws.items_1[(size_t)(n - 1) * ws.max_items + pos] =
            make_int4(rg, s | (k << 16), (int)(bits | ((uint32_t)n << 16)), L | flags);
      else
        flag_error(ws.status, WISE_DEVERR_BAD_WORK_LIST);
    }
    carry += tot;
  }
}

// List 1 straight from the rows' modes, lengths and masks (wise_build_list;
// modes null: every row sparse, wise_build_sparse_list): one CTA per (row, KV
// head) runs list1_build_pair on the pair's mask words or its whole length.
// Its counters must be 0 when the kernel starts (the caller resets the
// workspace header first).  Defined in compact.cu.
cudaError_t launch_build_list(const KParams& kp, const int8_t* modes, const int32_t* seq_lens,
                              const MaskView& mv, const WsView& ws, cudaStream_t stream);

}  // namespace wise
