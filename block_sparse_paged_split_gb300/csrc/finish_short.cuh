// Finish of short rows (at most 64 blocks and 8 split slots), shared by the
// finish kernel and by the partial pass when the finish is folded into it.
//
// [WISE PR, "What changes"]: the splits of a (row, KV head) are merged by
// their log-sum-exp, and a discovery row keeps the shortest prefix of its
// blocks, by mass descending (ties to the lower block index), whose mass
// reaches eta; the mask is [row, head, block] with the query heads of a KV
// group ORed.
//
//   merge    M = max_i m_i, Lambda = sum_i l_i 2^(m_i - M),
//            out = sum_i acc_i 2^(m_i - M) / Lambda, lse = (M + log2 Lambda) ln 2
//            (m_i in log2 units of the scaled score).  An empty range of a
//            sparse row holds (-inf, 0) and contributes nothing.
//   select   p_b = l_b 2^(m_b - lse2); 64-bit keys (~bits(p_b) << 32 | b) are
//            sorted ascending by a bitonic network in registers (E keys a
//            lane, block lane * E + e); the block at sorted position k is kept
//            iff the mass before it is below eta (eta >= 1 keeps every block).
#pragma once

#include "common.cuh"

namespace wise {

constexpr int kShortSlots = 8;    // split slots of a short row, at most

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int o) {
  uint32_t lo = __shfl_xor_sync(kFull, (uint32_t)v, o);
  uint32_t hi = __shfl_xor_sync(kFull, (uint32_t)(v >> 32), o);
  return ((uint64_t)hi << 32) | lo;
}

// Loads that bypass L1 when the data was written by other SMs during the
// same launch (the folded finish); plain loads otherwise.
template <bool kL2, typename V>
__device__ __forceinline__ V ld_ws(const V* p) {
  if constexpr (kL2) return __ldcg(p);
  else return *p;
}

// Sorts the warp's 32*E keys ascending; key i lives in lane i / E, slot i % E.
template <int E>
__device__ __forceinline__ void warp_bitonic_sort(uint64_t (&key)[E], int lane) {
  constexpr int N = 32 * E;
#pragma unroll
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= E) {
        const int lj = j / E;  // partner lane distance
        const bool lower = (lane & lj) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = lane * E + e;
          const bool up = (i & k) == 0;
          const uint64_t other = shfl_xor_u64(key[e], lj);
          const uint64_t mn = key[e] < other ? key[e] : other;
          const uint64_t mx = key[e] < other ? other : key[e];
          key[e] = (lower == up) ? mn : mx;
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & j) == 0) {
            const int i = lane * E + e;
            const bool up = (i & k) == 0;
            const uint64_t a = key[e], b = key[e ^ j];
            const bool swap = up ? (a > b) : (a < b);
            key[e] = swap ? b : a;
            key[e ^ j] = swap ? a : b;
          }
        }
      }
    }
  }
}

// Selection over the warp's blocks (st[e]: the statistics of block
// lane * E + e); returns the kept blocks as mask words 0 and 1, the same in
// every lane.
template <int E>
__device__ __forceinline__ uint2 warp_select_words(const float2 (&st)[2], int nb, float lse2,
                                                   float eta, int lane) {
  constexpr uint64_t kPad = ~0ull;
  uint64_t key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane * E + e;
    if (i < nb) {
      const float2 t = st[e];
      const float p = t.y * exp2f(t.x - lse2);
      key[e] = ((uint64_t)(~__float_as_uint(p)) << 32) | (uint32_t)i;
    } else {
      key[e] = kPad;
    }
  }
  warp_bitonic_sort<E>(key, lane);
  float pm[E];
  float tot = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    pm[e] = key[e] == kPad ? 0.f : __uint_as_float(~(uint32_t)(key[e] >> 32));
    tot += pm[e];
  }
  float incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  float before = __shfl_up_sync(kFull, incl, 1);
  if (lane == 0) before = 0.f;
  const bool all = eta >= 1.f;
  uint32_t w0 = 0u, w1 = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (key[e] != kPad && (all || before < eta)) {
      const uint32_t b = (uint32_t)key[e];
      if (b < 32) w0 |= 1u << b;
      else w1 |= 1u << (b - 32);
    }
    before += pm[e];
  }
  return make_uint2(__reduce_or_sync(kFull, w0), __reduce_or_sync(kFull, w1));
}

// Merges query head h's split slots of (row, KV head) rg (slot i at
// rg * S_max + i, i < nslots) in every lane, writes the head's output row and
// LSE, and returns the LSE in log2 units (or -inf when no slot holds mass).
template <typename T, bool kL2>
__device__ __forceinline__ float short_merge_head(const WsView& ws, const KParams& kp, int rg,
                                                  int h_in_group, int nslots, T* out_row,
                                                  float* lse_out, int lane) {
  const int G = kp.G, D = kp.D;
  const int dpl = D >> 5;
  const size_t slot0 = (size_t)rg * kp.S_max;
  float2 t[kShortSlots];
  float4 a[kShortSlots];
#pragma unroll
  for (int i = 0; i < kShortSlots; ++i) {
    const bool in = i < nslots;
    const size_t idx = (slot0 + (in ? i : 0)) * G + h_in_group;
    t[i] = in ? ld_ws<kL2>(ws.partial_ml + idx) : make_float2(-INFINITY, 0.f);
    const float* ap = ws.partial_acc + idx * D + lane * dpl;
    if (dpl == 4) {
      a[i] = ld_ws<kL2>(reinterpret_cast<const float4*>(ap));
    } else {
      const float2 v = ld_ws<kL2>(reinterpret_cast<const float2*>(ap));
      a[i] = make_float4(v.x, v.y, 0.f, 0.f);
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kShortSlots; ++i)
    if (t[i].y > 0.f) M = fmaxf(M, t[i].x);
  float lam = 0.f;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kShortSlots; ++i) {
    const bool used = t[i].y > 0.f;  // an empty range's accumulator is never used
    const float w = used ? exp2f(t[i].x - M) : 0.f;
    lam = fmaf(t[i].y, w, lam);
    o[0] += used ? a[i].x * w : 0.f;
    o[1] += used ? a[i].y * w : 0.f;
    o[2] += used ? a[i].z * w : 0.f;
    o[3] += used ? a[i].w * w : 0.f;
  }
  T* orow = out_row + lane * dpl;
  if (!(lam > 0.f)) {  // nothing selected: output 0, LSE -inf
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = 0.f;
    if (dpl == 4) Elem<T>::template store_global<4>(orow, o);
    else Elem<T>::template store_global<2>(orow, reinterpret_cast<const float(&)[2]>(o));
    if (lane == 0) *lse_out = -INFINITY;
    return -INFINITY;
  }
  const float inv = 1.f / lam;
#pragma unroll
  for (int j = 0; j < 4; ++j) o[j] *= inv;
  if (dpl == 4) Elem<T>::template store_global<4>(orow, o);
  else Elem<T>::template store_global<2>(orow, reinterpret_cast<const float(&)[2]>(o));
  const float lse2 = M + log2f(lam);
  if (lane == 0) *lse_out = lse2 * kLn2;
  return lse2;
}

// Tile statistics of query head h (global index) in the layout of the
// selection: block lane * E + e, E = 1 for rows of up to 32 blocks, 2 up to 64.
template <bool kL2>
__device__ __forceinline__ void short_load_stats(const WsView& ws, const KParams& kp, int r, int h,
                                                 int nb, int lane, float2 (&st)[2]) {
  const float2* ts = ws.tile_stats + (size_t)(r * kp.Hq + h) * kp.max_blocks;
  const int E = nb > 32 ? 2 : 1;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int i = lane * E + e;
    st[e] = e < E && i < nb ? ld_ws<kL2>(ts + i) : make_float2(0.f, 0.f);
  }
}

// The whole finish of (row, KV head) rg by one warp, inside the partial pass
// (its slots and statistics were written by other SMs of the same launch):
// every query head of the group merged and written, then, for discovery rows,
// the group's selections ORed and the mask written (DISCOVER) or ORed into
// (DISCOVER_UNION), bits at or past the row's block count cleared.
template <typename T>
__device__ __forceinline__ void short_finish_pair_warp(const WsView& ws, const KParams& kp, int rg,
                                                       int L, int mode, uint32_t* support, T* out,
                                                       float* lse, int lane) {
  const int r = rg / kp.Hkv, g = rg - r * kp.Hkv;
  const int nb = (L + kTile - 1) / kTile;
  uint32_t* const mw = support ? support + (size_t)rg * kp.W : nullptr;
  // Written by compaction, before this launch; within the pair's slots.
  const int nslots = min(max(ws.head_info[rg].y, 0), min(kp.S_max, kShortSlots));
  const bool disc = (mode == WISE_MODE_DISCOVER || mode == WISE_MODE_DISCOVER_UNION) && mw != nullptr;
  uint32_t w0 = 0u, w1 = 0u;
  for (int hl = 0; hl < kp.G; ++hl) {
    const int h = g * kp.G + hl;
    float2 st[2];
    if (disc) short_load_stats<true>(ws, kp, r, h, nb, lane, st);
    const float lse2 = short_merge_head<T, true>(ws, kp, rg, hl, nslots,
                                                 out + ((size_t)r * kp.Hq + h) * kp.D,
                                                 lse + (size_t)r * kp.Hq + h, lane);
    if (disc && lse2 > -INFINITY) {
      const uint2 w = nb > 32 ? warp_select_words<2>(st, nb, lse2, kp.eta, lane)
                              : warp_select_words<1>(st, nb, lse2, kp.eta, lane);
      w0 |= w.x;
      w1 |= w.y;
    }
  }
  if (disc && lane < kp.W) {
    const int lo = lane * 32;
    const uint32_t valid = lo + 32 <= nb ? 0xffffffffu : (lo < nb ? (1u << (nb - lo)) - 1u : 0u);
    uint32_t* word = mw + lane;
    uint32_t w = (lane == 0 ? w0 : w1) & valid;
    if (mode == WISE_MODE_DISCOVER_UNION) w |= ld_ws<true>(word) & valid;
    *word = w;
  }
}

}  // namespace wise
