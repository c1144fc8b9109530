// Finish pass of WISE paged decode attention.
//
// [WISE PR, "What changes"]: a finish kernel merges the splits and runs the
// selection for discovery rows.  Rows of up to 64 blocks: one CTA per (row,
// KV head), one warp per query head (finish_short_kernel).  Longer rows: one
// CTA of 8 warps per (row, query head), the G CTAs of a KV head forming a
// thread-block cluster whose first CTA ORs the group's selections through
// distributed shared memory (finish_kernel).
//
//   merge    M = max_i m_i, Lambda = sum_i l_i 2^(m_i - M),
//            out = sum_i acc_i 2^(m_i - M) / Lambda, lse = (M + log2 Lambda) ln 2
//            (m_i in log2 units of the scaled score).  Slot i is block range
//            i of the row; an empty range of a sparse row holds (-inf, 0) and
//            contributes nothing (its accumulator is never read into the sum).
//   select   for discover rows: p_b = l_b 2^(m_b - lse2) per block; 64-bit
//            keys (~bits(p_b) << 32 | b) are sorted ascending -- mass
//            descending, ties to the lower block index -- by a bitonic
//            network; the block at sorted position k is kept iff the mass
//            before it is below eta, which is exactly the shortest prefix
//            reaching eta (eta >= 1 keeps every block).  The group's query
//            heads OR their choices in shared memory; the mask is written
//            (DISCOVER) or ORed into (DISCOVER_UNION), with bits at or past
//            the row's block count cleared.
#include "finish_short.cuh"
#include "internal.h"
#include "list1.cuh"

namespace wise {

constexpr int kMaxW = WISE_MAX_BLOCKS / 32;  // mask words of a (row, KV head), at most

__device__ __forceinline__ void group_sync(int id, int threads) {
  if (threads == 32) {
    __syncwarp();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
  }
}

// Exclusive prefix over the group's threads (thread th contributes v);
// `scratch` holds one float per warp of the group.
__device__ __forceinline__ float group_exclusive_scan(float v, int th, int wph, float* scratch,
                                                      int bar_id) {
  const int lane = th & 31, wsub = th >> 5;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (wph == 1) return incl - v;
  if (lane == 31) scratch[wsub] = incl;
  group_sync(bar_id, wph * 32);
  float before = 0.f;
  for (int w = 0; w < wsub; ++w) before += scratch[w];
  group_sync(bar_id, wph * 32);
  return before + incl - v;
}

// One bitonic stage whose partner distance J (< E) stays within a thread's
// registers; `base` is the group-wide index of the thread's key 0.
template <int E, int J>
__device__ __forceinline__ void bitonic_reg_stage(uint64_t (&key)[E], int base, int k) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if ((e & J) == 0) {
      const bool up = ((base + e) & k) == 0;
      const uint64_t a = key[e], b = key[e + J];
      const bool swap = up ? (a > b) : (a < b);
      key[e] = swap ? b : a;
      key[e + J] = swap ? a : b;
    }
  }
}

// Ascending bitonic sort of a group's npad = 32 * E * wph keys: key i
// (i = wsub * 32E + lane * E + e) lives in register e of lane `lane` of the
// group's warp wsub.  Stages whose partner lies in another warp exchange
// through shared memory (`xbuf`, npad keys, one named barrier each side);
// stages within a warp use shuffles, stages within a thread its registers.
template <int E>
__device__ __forceinline__ void group_bitonic_sort(uint64_t (&key)[E], int lane, int wsub, int wph,
                                                   uint64_t* xbuf, int bar_id) {
  const int npad = 32 * E * wph;
  const int base = wsub * 32 * E + lane * E;
  for (int k = 2; k <= npad; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32 * E) {
#pragma unroll
        for (int e = 0; e < E; ++e) xbuf[base + e] = key[e];
        group_sync(bar_id, wph * 32);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = base + e;
          const uint64_t other = xbuf[i ^ j];
          const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
          key[e] = keep_min ? (key[e] < other ? key[e] : other) : (key[e] < other ? other : key[e]);
        }
        group_sync(bar_id, wph * 32);
      } else if (j >= E) {
        const int lj = j / E;  // partner lane distance
        const bool lower = (lane & lj) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const bool up = ((base + e) & k) == 0;
          const uint64_t other = shfl_xor_u64(key[e], lj);
          const uint64_t mn = key[e] < other ? key[e] : other;
          const uint64_t mx = key[e] < other ? other : key[e];
          key[e] = (lower == up) ? mn : mx;
        }
      } else if (j == 4) {
        if constexpr (E > 4) bitonic_reg_stage<E, 4>(key, base, k);
      } else if (j == 2) {
        if constexpr (E > 2) bitonic_reg_stage<E, 2>(key, base, k);
      } else {
        if constexpr (E > 1) bitonic_reg_stage<E, 1>(key, base, k);
      }
    }
  }
}

// Selection for one query head by its group of wph warps: keys from the
// (prefetched) tile statistics st[e] of block wsub * 32E + lane * E + e,
// sorted, then each kept block ORed into smask.
template <int E>
__device__ __forceinline__ void group_select(const float2 (&st)[E], int nb, float lse2, float eta,
                                             int lane, int wsub, int wph, uint64_t* xbuf,
                                             float* scratch, int bar_id, uint32_t* smask) {
  constexpr uint64_t kPad = ~0ull;
  const int base = wsub * 32 * E + lane * E;
  uint64_t key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = base + e;
    if (i < nb) {
      const float p = st[e].y * exp2f(st[e].x - lse2);
      key[e] = ((uint64_t)(~__float_as_uint(p)) << 32) | (uint32_t)i;
    } else {
      key[e] = kPad;
    }
  }
  group_bitonic_sort<E>(key, lane, wsub, wph, xbuf, bar_id);
  float pm[E];
  float mine = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    pm[e] = key[e] == kPad ? 0.f : __uint_as_float(~(uint32_t)(key[e] >> 32));
    mine += pm[e];
  }
  float before = group_exclusive_scan(mine, wsub * 32 + lane, wph, scratch, bar_id);
  const bool all = eta >= 1.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (key[e] != kPad && (all || before < eta)) {
      const uint32_t b = (uint32_t)key[e];
      atomicOr(&smask[b >> 5], 1u << (b & 31));
    }
    before += pm[e];
  }
}

// Sums over the group's threads of N unsigned integers at once: one warp
// reduction instruction each, the warps' sums through shared memory, one named
// barrier.  `buf` holds two sets of wph * N sums used alternately (by
// `parity`), so a warp that races ahead to the next call never overwrites a set
// another warp is still reading.
template <int N>
__device__ __forceinline__ void group_sums_u32(const uint32_t (&v)[N], uint32_t (&out)[N],
                                               int lane, int wsub, int wph, uint32_t* buf,
                                               int& parity, int bar_id) {
  uint32_t* b = buf + (parity & 1) * wph * N;
#pragma unroll
  for (int n = 0; n < N; ++n) {
    const uint32_t w = __reduce_add_sync(kFull, v[n]);
    if (lane == 0) b[wsub * N + n] = w;
  }
  group_sync(bar_id, wph * 32);
#pragma unroll
  for (int n = 0; n < N; ++n) out[n] = 0u;
  for (int w = 0; w < wph; ++w) {
#pragma unroll
    for (int n = 0; n < N; ++n) out[n] += b[w * N + n];
  }
  ++parity;
}

// Selection for one query head without sorting (rows of 512 or more padded
// blocks).  The rule -- order blocks by mass descending, equal masses by the
// lower block index, keep the shortest prefix reaching eta -- keeps every
// block whose mass exceeds some threshold value v, plus the blocks of mass
// exactly v in index order until the sum reaches eta.  The masses become
// fixed-point integers (p * 2^31, truncated: every sum is exact, so the result
// does not depend on the order of addition; the masses sum to about 1, so
// every sum fits in 32 bits), and v is the largest float bit pattern whose
// blocks of mass >= v sum to eta or more, found two bits at a time from the
// top (three group sums a step).  The truncation moves a sum by less than
// 4096 * 2^-31 = 1.9e-6, so the cutoff can differ from an exact prefix sum
// only where the cumulative mass lies that close to eta.  Block i = wsub * 32E
// + lane * E + e stays in index order, so the kept blocks become mask words by
// shuffles (each word written once, no atomics).
template <int E>
__device__ __forceinline__ void group_select_threshold(const float2 (&st)[E], int nb, float lse2,
                                                       float eta, int lane, int wsub, int wph,
                                                       uint32_t* buf, int* cnt, int bar_id,
                                                       uint32_t* smask) {
  constexpr float kFix = 2147483648.0f;  // 2^31
  const int base = wsub * 32 * E + lane * E;
  uint32_t key[E], m[E];
  uint32_t mine[1] = {0u};
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (base + e < nb) {
      const float p = st[e].y * exp2f(st[e].x - lse2);
      key[e] = __float_as_uint(p);
      m[e] = __float2uint_rz(p * kFix);
    } else {
      key[e] = 0u;
      m[e] = 0u;
    }
    mine[0] += m[e];
  }
  int parity = 0;
  uint32_t total[1];
  group_sums_u32<1>(mine, total, lane, wsub, wph, buf, parity, bar_id);
  // At least one fixed-point unit: the rule always keeps a block.
  const uint32_t eta_fix = max(__double2uint_rn(fmin((double)eta, 1.0) * 2147483648.0), 1u);
  bool keep[E];
  if (eta >= 1.f || total[0] < eta_fix) {
    // eta >= 1 keeps every block; so does a sum that never reaches eta.
#pragma unroll
    for (int e = 0; e < E; ++e) keep[e] = base + e < nb;
  } else {
    uint32_t v = 0u;
    // Masses are below 2 (bit 30 clear): bits 29..0, two a step.
    for (int b = 28; b >= 0; b -= 2) {
      uint32_t sm[3] = {0u, 0u, 0u}, tot[3];
#pragma unroll
      for (int e = 0; e < E; ++e)
#pragma unroll
        for (int c = 0; c < 3; ++c) sm[c] += key[e] >= (v | ((uint32_t)(c + 1) << b)) ? m[e] : 0u;
      group_sums_u32<3>(sm, tot, lane, wsub, wph, buf, parity, bar_id);
      v |= (tot[2] >= eta_fix ? 3u : tot[1] >= eta_fix ? 2u : tot[0] >= eta_fix ? 1u : 0u) << b;
    }
    uint32_t a[1] = {0u}, above[1];
    int ties = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      a[0] += key[e] > v ? m[e] : 0u;
      ties += (key[e] == v && base + e < nb) ? 1 : 0;
    }
    group_sums_u32<1>(a, above, lane, wsub, wph, buf, parity, bar_id);
    // Every tied block has mass v, hence the same fixed-point mass.
    const uint32_t mt = __float2uint_rz(__uint_as_float(v) * kFix);
    const uint32_t need = eta_fix - above[0];  // > 0 by the choice of v
    const uint32_t take = mt ? (need + mt - 1u) / mt : 0xffffffffu;
    // Ties before this thread's first block, in block order.
    int incl = ties;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) cnt[wsub] = incl;
    group_sync(bar_id, wph * 32);
    uint32_t rank = (uint32_t)(incl - ties);
    for (int w = 0; w < wsub; ++w) rank += (uint32_t)cnt[w];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const bool tied = key[e] == v && base + e < nb;
      keep[e] = (key[e] > v && base + e < nb) || (tied && rank < take);
      rank += tied ? 1u : 0u;
    }
  }
  // 32 / E consecutive lanes hold one mask word.
  constexpr int kLanesPerWord = 32 / E;
  uint32_t nib = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) nib |= keep[e] ? (1u << e) : 0u;
  uint32_t word = nib << ((lane % kLanesPerWord) * E);
#pragma unroll
  for (int o = 1; o < kLanesPerWord; o <<= 1) word |= __shfl_xor_sync(kFull, word, o);
  if (lane % kLanesPerWord == 0) smask[base >> 5] = word;
}

// Long rows: one CTA of W warps per (row, query head); the G CTAs of
// a KV head's group form one thread-block cluster, so their selections are
// ORed through distributed shared memory (every SM of the group sorts one
// head's keys, instead of one SM sorting all of them).
//   merge   the warps take the split slots round-robin, four loads in flight
//           per lane, with an online rescale; the warps' (m, l, acc) are then
//           combined through shared memory.
//   select  npad = 32 * E * W keys (npad >= max_blocks, a power of
//           two; blocks past the row's n_b are padding) are sorted mostly in
//           registers (see group_bitonic_sort).
// W = 4 warps a head for up to 512 keys, 8 for 1024, 16 for 2048 and 4096
// (rows past 32K tokens; same-box A/B: 4 warps made the 4K finish 18.7 ->
// 12.6 us, 8 warps stay best at 1024 keys).

template <typename T, int E, int W, bool kBuild>
__global__ void __launch_bounds__(W * 32)
    finish_kernel(const int8_t* __restrict__ modes, const int32_t* __restrict__ seq_lens,
                  const WsView ws, const KParams kp, const MaskView mv,
                  T* __restrict__ out, float* __restrict__ lse) {
  constexpr int wph = W;
  extern __shared__ __align__(16) uint8_t fsm[];
  __shared__ uint32_t smask[kMaxW];
  __shared__ uint32_t fwords[kMaxW];  // the mask the call leaves (list 1 is built from it)
  __shared__ List1Smem l1sm;
  static_assert(E * W <= kMaxW, "smask holds a word for every 32 padded keys");
  const int G = kp.G, D = kp.D;
  const int gs = wph * 32;
  const int th = threadIdx.x;
  const int lane = th & 31, wsub = th >> 5;
  const int bar_id = 1;
  // Shared memory: keys [npad] u64 | scratch [wph][D + 2] f32.
  uint64_t* xbuf = reinterpret_cast<uint64_t*>(fsm);
  float* scratch = reinterpret_cast<float*>(fsm + (size_t)32 * E * wph * 8);

  const int hgrp = (int)cluster_rank();  // query head within the KV group
  const int rg = blockIdx.x / G;
  const int r = rg / kp.Hkv, g = rg - r * kp.Hkv;
  const int h = g * G + hgrp;
  const int L = clamp_len(seq_lens[r], kp.cap_tokens);
  // On list 1 every row is sparse, unless the list was built for the call's
  // modes (wise_build_list; the modes are then passed).
  const int mode = (kp.list1 && !modes) ? (int)WISE_MODE_SPARSE : (int)modes[r];
  const int nb = (L + kTile - 1) / kTile;
  uint32_t* const mw = mask_of(mv, mask_slot(mv, r), g, kp.W);  // the pair's mask, or null
  const bool disc = (mode == WISE_MODE_DISCOVER || mode == WISE_MODE_DISCOVER_UNION) && mw != nullptr;
  const int dpl = D >> 5;  // 2 or 4 dims per lane
  T* orow = out + ((size_t)r * kp.Hq + h) * D + lane * dpl;
  float o[4] = {0.f, 0.f, 0.f, 0.f};

  // Read before the dependency wait: the caller's inputs and the head info
  // (written by compaction or by the finish that built list 1).  The kernel
  // before this one is the call's partial pass, which triggers this launch
  // only after its own dependency wait, so all of them are complete (and the
  // partial pass does not write them).
  int4 hi;
  if (kp.dense_list) {  // every range of the row is one item
    const int nr = (nb + kp.T - 1) / kp.T;
    hi = make_int4(rg * kp.S_max, nr, nb, nr);
  } else {
    hi = (kp.list1 ? ws.head_info_1 : ws.head_info)[rg];
  }
  // The next kernel may start launching now: its CTAs take the SMs the
  // partial pass frees in its tail and wait there (a pass whose inputs are
  // ready issues its first copies meanwhile); every kernel of the library
  // waits for this one before it touches the workspace or the mask.
  grid_dependents_launch();
  grid_dependency_wait();    // the partial pass's results
  // The mask words the call starts from (the group's first CTA): union-discover
  // rows OR into them, and a list build takes them as they are for rows this
  // call does not select.
  const bool need_old = (disc && mode == WISE_MODE_DISCOVER_UNION) || (kBuild && !disc);
  const uint32_t old_word = (need_old && mw && hgrp == 0 && th < kp.W) ? mw[th] : 0u;
  float2 st[E];
  const float2* ts = ws.tile_stats + (size_t)(r * kp.Hq + h) * kp.max_blocks;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = wsub * 32 * E + lane * E + e;
    st[e] = disc && i < nb ? ts[i] : make_float2(0.f, 0.f);
  }
  // Padding rows and sparse rows selecting nothing: the whole cluster (one
  // row and KV head) leaves here, before any cluster barrier.  Their masks
  // select nothing, so a list build gives them no item.
  if (L == 0 || hi.z == 0) {
    if (wsub == 0) {
      if (dpl == 4) Elem<T>::template store_global<4>(orow, o);
      else Elem<T>::template store_global<2>(orow, reinterpret_cast<const float(&)[2]>(o));
      if (lane == 0) lse[(size_t)r * kp.Hq + h] = -INFINITY;
    }
    if (kBuild && hgrp == 0 && th == 0) list1_empty_pair(ws, kp, rg);
    return;
  }

  // ---- merge the pair's split slots (hi.y of them from hi.x)
  const size_t slot0 = (size_t)rg * kp.S_max;  // = hi.x
  const float2* ml = ws.partial_ml + slot0 * G + hgrp;  // slot s at ml[s * G]
  const float* acc = ws.partial_acc + (slot0 * G + hgrp) * D + lane * dpl;
  const int n = min(max(hi.y, 0), kp.S_max);
  float m_w = -INFINITY, lam = 0.f;
  // Slots in flight per lane (8 for 1024-key rows measured no faster at 32K:
  // 13.3 vs 13.4 us, ncu, with 102 instead of 64 registers).
  constexpr int U = 4;
  for (int s0 = wsub; s0 < n; s0 += U * wph) {
    float2 t[U];
    float4 a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int s = s0 + u * wph;
      const bool in = s < n;
      t[u] = in ? ml[(size_t)s * G] : make_float2(-INFINITY, 0.f);
      const float* ap = acc + (size_t)(in ? s : 0) * G * D;
      a[u] = dpl == 4 ? *reinterpret_cast<const float4*>(ap) : make_float4(ap[0], ap[1], 0.f, 0.f);
    }
    float mb = m_w;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (t[u].y > 0.f) mb = fmaxf(mb, t[u].x);
    if (mb > m_w) {  // rescale what this warp has summed so far
      const float sc = exp2f(m_w - mb);
      lam *= sc;
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] *= sc;
      m_w = mb;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool used = t[u].y > 0.f;  // an empty range's accumulator is never used
      const float w = used ? exp2f(t[u].x - m_w) : 0.f;
      lam = fmaf(t[u].y, w, lam);
      o[0] += used ? a[u].x * w : 0.f;
      o[1] += used ? a[u].y * w : 0.f;
      o[2] += used ? a[u].z * w : 0.f;
      o[3] += used ? a[u].w * w : 0.f;
    }
  }
  // Combine the warps: every warp forms M and Lambda, warp 0 the output.
  {
    float* mine = scratch + wsub * (D + 2);
    if (lane == 0) {
      mine[D] = m_w;
      mine[D + 1] = lam;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < dpl) mine[lane * dpl + j] = o[j];
    group_sync(bar_id, gs);
    float M = -INFINITY;
    for (int w = 0; w < wph; ++w) M = fmaxf(M, scratch[w * (D + 2) + D]);
    lam = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = 0.f;
    for (int w = 0; w < wph; ++w) {
      const float* part = scratch + w * (D + 2);
      const float sc = part[D + 1] > 0.f ? exp2f(part[D] - M) : 0.f;
      lam = fmaf(part[D + 1], sc, lam);
      if (wsub == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < dpl) o[j] = fmaf(part[lane * dpl + j], sc, o[j]);
      }
    }
    m_w = M;
    group_sync(bar_id, gs);
  }
  const float lse2 = m_w + log2f(lam);
  if (wsub == 0) {
    const float inv = 1.f / lam;
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] *= inv;
    if (dpl == 4) Elem<T>::template store_global<4>(orow, o);
    else Elem<T>::template store_global<2>(orow, reinterpret_cast<const float(&)[2]>(o));
    if (lane == 0) lse[(size_t)r * kp.Hq + h] = lse2 * kLn2;
  }

  if (!disc) {  // the whole cluster
    if (kBuild && hgrp == 0) {
      if (th < kp.W) fwords[th] = old_word;
      __syncthreads();
      list1_build_pair(ws, kp, rg, L, fwords, false, kItemSparse, l1sm);
    }
    return;
  }

  // ---- eta selection for this query head, then the group's OR
  for (int i = th; i < kp.W; i += gs) smask[i] = 0u;
  __syncthreads();
  if constexpr (32 * E * W >= 512) {
    // 512 keys or more: the threshold search (the bitonic sort of 1024 keys
    // took 10 us of a 19 us finish at 32K, %globaltimer stamps per CTA).
    group_select_threshold<E>(st, nb, lse2, kp.eta, lane, wsub, wph,
                              reinterpret_cast<uint32_t*>(xbuf), reinterpret_cast<int*>(scratch),
                              bar_id, smask);
  } else {
    group_select<E>(st, nb, lse2, kp.eta, lane, wsub, wph, xbuf, scratch, bar_id, smask);
  }
  __syncthreads();
  cluster_arrive();  // every head's choice is in its CTA's smask
  cluster_wait();
  if (hgrp == 0 && th < kp.W) {
    const int lo = th * 32;
    const uint32_t valid = lo + 32 <= nb ? 0xffffffffu : (lo < nb ? (1u << (nb - lo)) - 1u : 0u);
    uint32_t w = 0u;
    for (int c = 0; c < G; ++c) w |= (uint32_t)load_peer(reinterpret_cast<const int*>(&smask[th]), c);
    w &= valid;
    if (mode == WISE_MODE_DISCOVER_UNION) w |= old_word & valid;
    mw[th] = w;
    fwords[th] = w;
  }
  cluster_arrive();  // no CTA leaves while the group's first CTA may still read it
  cluster_wait();
  if (kBuild && hgrp == 0) list1_build_pair(ws, kp, rg, L, fwords, false, kItemSparse, l1sm);
}

// ------------------------------------------------------------------ short rows
// Rows of at most 64 blocks and 8 split slots: one warp per query head, the
// merge in each lane over all slots, the sort in registers with shuffles
// (finish_short.cuh); the group's selections are ORed in shared memory.
template <typename T, bool kBuild>
__global__ void __launch_bounds__(256)
    finish_short_kernel(const int8_t* __restrict__ modes, const int32_t* __restrict__ seq_lens,
                        const WsView ws, const KParams kp, const MaskView mv,
                        T* __restrict__ out, float* __restrict__ lse) {
  __shared__ uint32_t smask[2];
  __shared__ uint32_t fwords[2];  // the mask the call leaves (list 1 is built from it)
  __shared__ List1Smem l1sm;
  const int rg = blockIdx.x;
  const int r = rg / kp.Hkv, g = rg - r * kp.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = g * kp.G + warp;
  const int L = clamp_len(seq_lens[r], kp.cap_tokens);
  // On list 1 every row is sparse, unless the list was built for the call's
  // modes (wise_build_list; the modes are then passed).
  const int mode = (kp.list1 && !modes) ? (int)WISE_MODE_SPARSE : (int)modes[r];
  const int nb = (L + kTile - 1) / kTile;
  uint32_t* const mw = mask_of(mv, mask_slot(mv, r), g, kp.W);  // the pair's mask, or null
  const bool disc = (mode == WISE_MODE_DISCOVER || mode == WISE_MODE_DISCOVER_UNION) && mw != nullptr;
  // Read before the dependency wait: the head info (written by compaction or
  // by the finish that built list 1).  The kernel before this one is the
  // call's partial pass, which triggers this launch only after its own
  // dependency wait, so it is complete.
  int4 hi;
  if (kp.dense_list) {  // every range of the row is one item
    const int nr = (nb + kp.T - 1) / kp.T;
    hi = make_int4(rg * kp.S_max, nr, nb, nr);
  } else {
    hi = (kp.list1 ? ws.head_info_1 : ws.head_info)[rg];
  }
  if (threadIdx.x < 2) smask[threadIdx.x] = 0u;
  // The next kernel may start launching now: its CTAs take the SMs the
  // partial pass frees in its tail and wait there (a pass whose inputs are
  // ready issues its first copies meanwhile); every kernel of the library
  // waits for this one before it touches the workspace or the mask.
  grid_dependents_launch();
  grid_dependency_wait();    // the partial pass's results
  // The mask words the call starts from: union-discover rows OR into them, and
  // a list build takes them as they are for the rows this call does not select.
  const bool need_old = (disc && mode == WISE_MODE_DISCOVER_UNION) || (kBuild && !disc);
  const uint32_t old_word = (need_old && mw && (int)threadIdx.x < kp.W) ? mw[threadIdx.x] : 0u;
  float2 st[2];
  if (disc) short_load_stats<false>(ws, kp, r, h, nb, lane, st);
  // Slot count from the head info, within the pair's S_max slots.
  const int nslots = hi.z == 0 ? 0 : min(max(hi.y, 0), kp.S_max);
  const float lse2 = short_merge_head<T, false>(ws, kp, rg, warp, nslots,
                                                out + ((size_t)r * kp.Hq + h) * kp.D,
                                                lse + (size_t)r * kp.Hq + h, lane);
  if (!kBuild && (!disc || L == 0)) return;  // a padding row's mask is left as it is
  __syncthreads();
  if (disc && L > 0 && lse2 > -INFINITY) {
    const uint2 w = nb > 32 ? warp_select_words<2>(st, nb, lse2, kp.eta, lane)
                            : warp_select_words<1>(st, nb, lse2, kp.eta, lane);
    if (lane == 0) {
      atomicOr(&smask[0], w.x);
      atomicOr(&smask[1], w.y);
    }
  }
  __syncthreads();
  if ((int)threadIdx.x < kp.W) {
    const int tw = threadIdx.x;
    uint32_t w = old_word;
    if (disc && L > 0) {
      const int lo = tw * 32;
      const uint32_t valid = lo + 32 <= nb ? 0xffffffffu : (lo < nb ? (1u << (nb - lo)) - 1u : 0u);
      w = smask[tw] & valid;
      if (mode == WISE_MODE_DISCOVER_UNION) w |= old_word & valid;
      mw[tw] = w;
    }
    fwords[tw] = w;
  }
  if (!kBuild) return;
  __syncthreads();
  list1_build_pair(ws, kp, rg, L, fwords, false, kItemSparse, l1sm);
}

// Rows of at most 64 blocks and 8 split slots (can_fold_finish) take the
// short kernel (one warp per query head); longer ones a CTA of W warps per
// query head, clustered by KV head (E = npad / (32 W) keys a thread).
static int finish_warps(const KParams& kp) {
  return kp.max_blocks <= 512 ? 4 : kp.max_blocks <= 1024 ? 8 : 16;
}

static int finish_npad(const KParams& kp) {
  int n = 32 * finish_warps(kp);
  while (n < kp.max_blocks) n <<= 1;
  return n;
}

template <typename T, int E, int W, bool kBuild>
static cudaError_t launch_long(const KParams& kp, const int8_t* modes, const int32_t* seq_lens,
                               const WsView& ws, const MaskView& mv, void* out, float* lse,
                               cudaStream_t stream) {
  const size_t smem = (size_t)32 * E * W * 8 + (size_t)W * (kp.D + 2) * 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kp.R * kp.Hkv * kp.G);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kp.G;  // the KV head's query heads (at most 8: portable)
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, finish_kernel<T, E, W, kBuild>, modes, seq_lens, ws, kp, mv,
                            static_cast<T*>(out), lse);
}

// The list build (WISE_FLAG_BUILD_SPARSE_LIST) is a separate instantiation,
// so the other calls run kernels without its code (with it inlined, the
// compiler gave the short finish 61 instead of 76 registers and issued its
// split loads in two rounds: 1.5 us slower per launch, ncu launch list).
template <typename T, bool kBuild>
static cudaError_t launch_finish_b(const KParams& kp, const int8_t* modes,
                                   const int32_t* seq_lens, const WsView& ws, const MaskView& mv,
                                   void* out, float* lse, cudaStream_t stream) {
  if (can_fold_finish(kp))
    return launch_pdl(finish_short_kernel<T, kBuild>, dim3(kp.R * kp.Hkv), dim3(32 * kp.G), 0,
                      stream, modes, seq_lens, ws, kp, mv, static_cast<T*>(out), lse);
  if (kp.list1 && !modes) {
    // Every row sparse: no selection, so no sort keys -- the warps only take
    // the pair's split slots (at most S_max).  Sized by the row length (16
    // warps and 4096 keys at 128K) the CTAs held 82 registers x 512 threads,
    // one CTA an SM, and the finish of a 64-row sparse call grew from 8 to
    // 30 us with the context at a fixed selection.
    if (kp.S_max <= 32) return launch_long<T, 1, 4, kBuild>(kp, modes, seq_lens, ws, mv, out, lse, stream);
    return launch_long<T, 1, 8, kBuild>(kp, modes, seq_lens, ws, mv, out, lse, stream);
  }
  const int w = finish_warps(kp);
  const int e = finish_npad(kp) / (32 * w);
  if (w == 4) {
    switch (e) {  // npad <= 512: e <= 4
      case 1: return launch_long<T, 1, 4, kBuild>(kp, modes, seq_lens, ws, mv, out, lse, stream);
      case 2: return launch_long<T, 2, 4, kBuild>(kp, modes, seq_lens, ws, mv, out, lse, stream);
      default: return launch_long<T, 4, 4, kBuild>(kp, modes, seq_lens, ws, mv, out, lse, stream);
    }
  }
  if (w == 8) return launch_long<T, 4, 8, kBuild>(kp, modes, seq_lens, ws, mv, out, lse, stream);
  // npad 2048 or 4096 with 16 warps: e = 4 or 8
  if (e == 4) return launch_long<T, 4, 16, kBuild>(kp, modes, seq_lens, ws, mv, out, lse, stream);
  return launch_long<T, 8, 16, kBuild>(kp, modes, seq_lens, ws, mv, out, lse, stream);
}

template <typename T>
static cudaError_t launch_finish_t(const KParams& kp, const int8_t* modes,
                                   const int32_t* seq_lens, const WsView& ws, const MaskView& mv,
                                   void* out, float* lse, cudaStream_t stream) {
  return kp.build ? launch_finish_b<T, true>(kp, modes, seq_lens, ws, mv, out, lse, stream)
                  : launch_finish_b<T, false>(kp, modes, seq_lens, ws, mv, out, lse, stream);
}

cudaError_t launch_finish(int dtype, const KParams& kp, const int8_t* modes,
                          const int32_t* seq_lens, const WsView& ws, const MaskView& mv,
                          void* out, float* lse, cudaStream_t stream) {
  if (kp.R == 0) return cudaSuccess;
  if (dtype == WISE_DTYPE_BF16)
    return launch_finish_t<__nv_bfloat16>(kp, modes, seq_lens, ws, mv, out, lse, stream);
  return launch_finish_t<float>(kp, modes, seq_lens, ws, mv, out, lse, stream);
}

}  // namespace wise
