// Finish pass of WISE paged decode attention.
//
// [WISE PR, "What changes"]: a finish kernel merges the splits and runs the
// selection for discovery rows.  One CTA per (row, KV head), one warp per
// query head of the group.
//
//   merge    M = max_i m_i, Lambda = sum_i l_i 2^(m_i - M),
//            out = sum_i acc_i 2^(m_i - M) / Lambda, lse = (M + log2 Lambda) ln 2
//            (m_i in log2 units of the scaled score).
//   select   for discover rows: p_b = l_b 2^(m_b - lse2) per block; the warp
//            sorts 64-bit keys (~bits(p_b) << 32 | b) ascending, i.e. mass
//            descending with ties to the lower block index, with a bitonic
//            network held in registers (E keys per lane, lane-major blocks);
//            block at sorted position k is kept iff the mass before it is
//            below eta, which is exactly the shortest prefix reaching eta
//            (eta >= 1 keeps every block).  The group's query heads OR their
//            choices in shared memory; the mask is written (DISCOVER) or ORed
//            into (DISCOVER_UNION), with bits at or past the row's block
//            count cleared.
#include "internal.h"

namespace wise {

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int o) {
  uint32_t lo = __shfl_xor_sync(kFull, (uint32_t)v, o);
  uint32_t hi = __shfl_xor_sync(kFull, (uint32_t)(v >> 32), o);
  return ((uint64_t)hi << 32) | lo;
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

// Eta selection of one (row, query head): marks the kept blocks in smask.
// Not inlined: the unrolled network is large and does not depend on the
// element type, head dim or group size of the calling kernel.
template <int E>
__device__ __noinline__ void select_blocks(const float2* __restrict__ ts, int nb, float lse2,
                                              float eta, uint32_t* smask, int lane) {
  constexpr uint64_t kPad = ~0ull;
  uint64_t key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane * E + e;
    if (i < nb) {
      const float2 t = ts[i];
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
  // Exclusive scan of the lane totals: mass of every earlier lane's keys.
  float incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  float before = __shfl_up_sync(kFull, incl, 1);
  if (lane == 0) before = 0.f;
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

// One CTA per (row, KV head) with one warp per query head of the group; the
// head dim (64 or 128) and group size are runtime values: the merge is a few
// loads per item, so only the element type is a template parameter.
template <typename T>
__global__ void __launch_bounds__(256)
    finish_kernel(const int8_t* __restrict__ modes, const int32_t* __restrict__ seq_lens,
                  const WsView ws, const KParams kp, uint32_t* __restrict__ support,
                  T* __restrict__ out, float* __restrict__ lse) {
  __shared__ uint32_t smask[32];
  grid_dependency_wait();    // the partial pass's results
  grid_dependents_launch();  // the next call's compaction may start launching
  const int rg = blockIdx.x;
  const int r = rg / kp.Hkv, g = rg - r * kp.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = kp.G, D = kp.D;
  const int dpl = D >> 5;  // 2 or 4 dims per lane
  const int h = g * G + warp;
  const int L = clamp_len(seq_lens[r], kp.cap_tokens);
  const int mode = modes[r];
  T* orow = out + ((size_t)r * kp.Hq + h) * D + lane * dpl;
  float o[4] = {0.f, 0.f, 0.f, 0.f};

  const int4 hi = ws.head_info[rg];
  if (L == 0 || hi.z == 0) {  // padding row, or a sparse row selecting nothing
    if (dpl == 4) Elem<T>::template store_global<4>(orow, o);
    else Elem<T>::template store_global<2>(orow, reinterpret_cast<const float(&)[2]>(o));
    if (lane == 0) lse[(size_t)r * kp.Hq + h] = -INFINITY;
    return;
  }

  const float2* ml = ws.partial_ml;
  float M = -INFINITY;
  // hi.x = first partial slot of this (row, KV head) (rg * S_max); its hi.y
  // block ranges occupy the next slots (an empty range of a sparse row
  // holds (-inf, 0) and is skipped).
  for (int i = 0; i < hi.y; ++i) M = fmaxf(M, ml[(size_t)(hi.x + i) * G + warp].x);
  float lam = 0.f;
  for (int i = 0; i < hi.y; ++i) {
    const size_t idx = (size_t)(hi.x + i) * G + warp;
    const float2 t = ml[idx];
    if (!(t.y > 0.f)) continue;
    const float w = exp2f(t.x - M);
    lam = fmaf(t.y, w, lam);
    const float* a = ws.partial_acc + idx * D + lane * dpl;
    if (dpl == 4) {
      const float4 v = *reinterpret_cast<const float4*>(a);
      o[0] = fmaf(v.x, w, o[0]); o[1] = fmaf(v.y, w, o[1]);
      o[2] = fmaf(v.z, w, o[2]); o[3] = fmaf(v.w, w, o[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(a);
      o[0] = fmaf(v.x, w, o[0]); o[1] = fmaf(v.y, w, o[1]);
    }
  }
  const float inv = 1.f / lam;
#pragma unroll
  for (int j = 0; j < 4; ++j) o[j] *= inv;
  if (dpl == 4) Elem<T>::template store_global<4>(orow, o);
  else Elem<T>::template store_global<2>(orow, reinterpret_cast<const float(&)[2]>(o));
  const float lse2 = M + log2f(lam);
  if (lane == 0) lse[(size_t)r * kp.Hq + h] = lse2 * kLn2;

  if ((mode != WISE_MODE_DISCOVER && mode != WISE_MODE_DISCOVER_UNION) || support == nullptr) return;

  if (threadIdx.x < 32) smask[threadIdx.x] = 0u;
  __syncthreads();
  const int nb = (L + kTile - 1) / kTile;
  const float2* ts = ws.tile_stats + (size_t)(r * kp.Hq + h) * kp.max_blocks;
  if (nb <= 32) select_blocks<1>(ts, nb, lse2, kp.eta, smask, lane);
  else if (nb <= 64) select_blocks<2>(ts, nb, lse2, kp.eta, smask, lane);
  else if (nb <= 128) select_blocks<4>(ts, nb, lse2, kp.eta, smask, lane);
  else if (nb <= 256) select_blocks<8>(ts, nb, lse2, kp.eta, smask, lane);
  else if (nb <= 512) select_blocks<16>(ts, nb, lse2, kp.eta, smask, lane);
  else select_blocks<32>(ts, nb, lse2, kp.eta, smask, lane);
  __syncthreads();
  if ((int)threadIdx.x < kp.W) {
    const int t = threadIdx.x;
    const int lo = t * 32;
    const uint32_t valid = lo + 32 <= nb ? 0xffffffffu : (lo < nb ? (1u << (nb - lo)) - 1u : 0u);
    uint32_t* word = support + (size_t)rg * kp.W + t;
    uint32_t w = smask[t] & valid;
    if (mode == WISE_MODE_DISCOVER_UNION) w |= *word & valid;
    *word = w;
  }
}

cudaError_t launch_finish(int dtype, const KParams& kp, const int8_t* modes,
                          const int32_t* seq_lens, const WsView& ws, uint32_t* support,
                          void* out, float* lse, cudaStream_t stream) {
  if (kp.R == 0) return cudaSuccess;
  const int grid = kp.R * kp.Hkv;
  const int threads = 32 * kp.G;
  if (dtype == WISE_DTYPE_BF16)
    return launch_pdl(finish_kernel<__nv_bfloat16>, dim3(grid), dim3(threads), 0, stream, modes,
                      seq_lens, ws, kp, support, static_cast<__nv_bfloat16*>(out), lse);
  return launch_pdl(finish_kernel<float>, dim3(grid), dim3(threads), 0, stream, modes, seq_lens,
                    ws, kp, support, static_cast<float*>(out), lse);
}

}  // namespace wise
