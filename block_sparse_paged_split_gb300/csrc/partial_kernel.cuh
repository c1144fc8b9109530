// Split partial pass of WISE paged decode attention (one launch per call).
//
// [WISE PR, "What changes"]: split-KV paged decode with per-row modes; dense
// rows attend every tile, discover rows also record each 32-token tile's max
// and exp-sum, sparse rows walk their compacted tile list; programs cover
// about eight tiles with one warp each.
//
// GB300 design:
//   * Persistent grid: every SM holds one CTA of WARPS independent warps; warp
//     w takes work items w, w + NW, w + 2 NW, ... (NW = warps in the grid).
//     Items come from the compaction kernel, so dense and sparse rows cost
//     the same per item and no row sets the latency of the launch.
//   * Each warp owns a STAGES-deep ring of shared-memory stages; one stage is
//     one 32-token tile of K and of V.  Lane 0 fetches a tile with one TMA
//     bulk-tensor copy per page and per cache (box = one page of one KV head:
//     page_size rows of head_dim elements), completing on the stage's
//     mbarrier.  The fetch stream runs STAGES tiles ahead of the math and
//     crosses item boundaries, so HBM stays busy across items.
//   * Math is FP32 FMA (multi-head decode reads every K/V element once: about
//     one FMA per byte, far below the tensor-core ridge).  Lane l holds dims
//     [l*DPL, (l+1)*DPL) of the query; the 32 per-token partial dot products
//     are reduced with a 31-shuffle transpose reduction so lane j ends with
//     token j's score.  Scores are kept in log2 units (scale * log2 e folded
//     in) and exponentiated with ex2.approx.
//   * Online softmax per item: running max m, per-lane exp-sum, accumulator
//     rescaled once per tile.  The item's unnormalised output, max and
//     exp-sum go to the workspace; the finish kernel merges the items.
#pragma once

#include "internal.h"

namespace wise {

template <typename T, int D, int G, int WARPS, int STAGES>
struct PartialCfg {
  static constexpr int DPL = D / 32;
  static constexpr int ROW_BYTES = D * (int)sizeof(T);
  static constexpr int TILE_BYTES = kTile * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
  static constexpr int PBUF_BYTES = G * kTile * 4;
  static constexpr int BAR_BYTES = ((8 * STAGES + 127) / 128) * 128;
  static constexpr int WARP_BYTES = STAGES * STAGE_BYTES + PBUF_BYTES + BAR_BYTES;
  static constexpr int SMEM_BYTES = WARPS * WARP_BYTES;
};

// Launch shape per element type and head dim: three stages per warp and as
// many warps as fit in ~192 KB of shared memory (one CTA per SM).
template <typename T, int D>
struct PartialTune {
  static constexpr int STAGES = 3;
  static constexpr int STAGE_BYTES = 2 * kTile * D * (int)sizeof(T);
  static constexpr int WARPS_RAW = (192 * 1024) / (STAGES * STAGE_BYTES);
  static constexpr int WARPS = WARPS_RAW > 8 ? 8 : (WARPS_RAW < 1 ? 1 : WARPS_RAW);
};

struct ItemRef {
  int4 rec;     // row, kv head, first index in the tile list, tile count
  int L;        // clamped sequence length of the row
  int sparse;   // row is in sparse mode (tile list is explicit)
};

__device__ __forceinline__ ItemRef load_item(const WsView& ws, const KParams& kp,
                                             const int32_t* __restrict__ seq_lens,
                                             const int8_t* __restrict__ modes, int item) {
  ItemRef it;
  it.rec = ws.items[item];
  it.L = clamp_len(seq_lens[it.rec.x], kp.cap_tokens);
  it.sparse = modes[it.rec.x] == WISE_MODE_SPARSE;
  return it;
}

__device__ __forceinline__ int tile_index(const WsView& ws, const KParams& kp, const ItemRef& it,
                                          int k) {
  return it.sparse
             ? ws.tile_list[(size_t)(it.rec.x * kp.Hkv + it.rec.y) * kp.max_blocks + it.rec.z + k]
             : it.rec.z + k;
}

template <typename T, int D, int G, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32, 1)
    partial_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const T* __restrict__ q, const int32_t* __restrict__ page_table,
                   const int32_t* __restrict__ seq_lens, const int8_t* __restrict__ modes,
                   const WsView ws, const KParams kp) {
  using C = PartialCfg<T, D, G, WARPS, STAGES>;
  constexpr int DPL = C::DPL;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t* wbase = smem + warp * C::WARP_BYTES;
  float* pbuf = reinterpret_cast<float*>(wbase + STAGES * C::STAGE_BYTES);
  const uint32_t stage0 = smem_u32(wbase);
  const uint32_t bar0 = smem_u32(wbase + STAGES * C::STAGE_BYTES + C::PBUF_BYTES);

  if (lane == 0) {
    if (warp == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int n_items = *ws.num_items;
  const int NW = gridDim.x * WARPS;
  const int first = blockIdx.x * WARPS + warp;

  // ---- fetch side (warp-uniform cursor; lane 0 issues the copies)
  int p_item = first, p_k = 0;
  ItemRef p_it{};
  if (p_item < n_items) p_it = load_item(ws, kp, seq_lens, modes, p_item);
  uint32_t seq_p = 0, seq_c = 0;

  auto issue_next = [&]() {
    if (p_item >= n_items) return;
    const int b = tile_index(ws, kp, p_it, p_k);
    const int stage = seq_p % STAGES;
    if (lane == 0) {
      const int tok0 = b * kTile;
      const int pages_in_tile = kTile / kp.P;
      int npg = (p_it.L - tok0 + kp.P - 1) / kp.P;  // pages holding a valid token
      npg = npg < pages_in_tile ? npg : pages_in_tile;
      const uint32_t bar = bar0 + 8 * stage;
      mbar_arrive_expect_tx(bar, (uint32_t)(2 * npg * kp.P * C::ROW_BYTES));
      const uint32_t kdst = stage0 + stage * C::STAGE_BYTES;
      const int32_t* pt = page_table + (size_t)p_it.rec.x * kp.max_pages + tok0 / kp.P;
      for (int pp = 0; pp < npg; ++pp) {
        const int page = pt[pp];
        // A page id outside the pool reads the tensor's out-of-bounds fill (zeros).
        const int tok = (page >= 0 && page < kp.num_pages) ? page * kp.P : kp.num_pages * kp.P;
        const uint32_t off = pp * kp.P * C::ROW_BYTES;
        tma_load_3d(kdst + off, &tmK, 0, p_it.rec.y, tok, bar);
        tma_load_3d(kdst + C::TILE_BYTES + off, &tmV, 0, p_it.rec.y, tok, bar);
      }
    }
    ++seq_p;
    if (++p_k == p_it.rec.w) {
      p_k = 0;
      p_item += NW;
      if (p_item < n_items) p_it = load_item(ws, kp, seq_lens, modes, p_item);
    }
  };

  // Waits out every fetch still in flight (bounded), so no copy lands in
  // shared memory after the CTA exits.
  auto drain = [&]() {
    while (seq_c < seq_p) {
      mbar_wait(bar0 + 8 * (seq_c % STAGES), (seq_c / STAGES) & 1);
      ++seq_c;
    }
  };

#pragma unroll
  for (int s = 0; s < STAGES; ++s) issue_next();

  for (int item = first; item < n_items; item += NW) {
    const ItemRef it = load_item(ws, kp, seq_lens, modes, item);
    const int r = it.rec.x, g = it.rec.y;
    const int mode = modes[r];
    const bool disc = (mode == WISE_MODE_DISCOVER) || (mode == WISE_MODE_DISCOVER_UNION);

    float qf[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
      Elem<T>::template load_global<DPL>(q + ((size_t)r * kp.Hq + g * G + h) * D + lane * DPL, qf[h]);

    float m_run[G], l_lane[G], acc[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_run[h] = -INFINITY;
      l_lane[h] = 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) acc[h][i] = 0.f;
    }

    for (int k = 0; k < it.rec.w; ++k) {
      const int b = tile_index(ws, kp, it, k);
      const int rem = it.L - b * kTile;
      const int n_valid = rem < kTile ? rem : kTile;
      const int stage = seq_c % STAGES;
      if (!mbar_wait(bar0 + 8 * stage, (seq_c / STAGES) & 1)) {
        if (lane == 0) flag_error(ws.status, WISE_DEVERR_WAIT_TIMEOUT);
        drain();
        return;
      }
      const uint8_t* kt = wbase + stage * C::STAGE_BYTES;
      const uint8_t* vt = kt + C::TILE_BYTES;

#pragma unroll
      for (int h = 0; h < G; ++h) {
        // s_j partial dot products over this lane's dims, one per token.
        float part[kTile];
#pragma unroll
        for (int j = 0; j < kTile; ++j) {
          float kx[DPL];
          Elem<T>::template load<DPL>(kt + j * C::ROW_BYTES, lane, kx);
          float a = qf[h][0] * kx[0];
#pragma unroll
          for (int i = 1; i < DPL; ++i) a = fmaf(qf[h][i], kx[i], a);
          part[j] = a;
        }
        // Transpose reduction: after the level with offset o, lanes with bit o
        // set hold the upper half of the remaining tokens; lane j ends with
        // the complete dot product of token j.
#pragma unroll
        for (int o = 16, n = 16; o > 0; o >>= 1, n >>= 1) {
          const bool upper = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < n; ++i) {
            const float send = upper ? part[i] : part[i + n];
            const float keep = upper ? part[i + n] : part[i];
            part[i] = keep + __shfl_xor_sync(kFull, send, o);
          }
        }
        const float s = lane < n_valid ? part[0] * kp.scale_log2 : -INFINITY;
        const float mt = warp_max(s);
        if (disc) {
          const float lb = warp_sum(fast_exp2(s - mt));
          if (lane == 0)
            ws.tile_stats[(size_t)(r * kp.Hq + g * G + h) * kp.max_blocks + b] = make_float2(mt, lb);
        }
        const float m_new = fmaxf(m_run[h], mt);
        const float alpha = fast_exp2(m_run[h] - m_new);
        const float pj = fast_exp2(s - m_new);
        l_lane[h] = fmaf(l_lane[h], alpha, pj);
        m_run[h] = m_new;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[h][i] *= alpha;

        float* pb = pbuf + h * kTile;
        pb[lane] = pj;
        __syncwarp();
        if (n_valid == kTile) {
#pragma unroll
          for (int j = 0; j < kTile; j += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(pb + j);
            const float pw[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float vx[DPL];
              Elem<T>::template load<DPL>(vt + (j + u) * C::ROW_BYTES, lane, vx);
#pragma unroll
              for (int i = 0; i < DPL; ++i) acc[h][i] = fmaf(pw[u], vx[i], acc[h][i]);
            }
          }
        } else {
          // Last tile of the row: tokens past the length may hold anything
          // (even NaN) and are never touched.
          for (int j = 0; j < n_valid; ++j) {
            const float pw = pb[j];
            float vx[DPL];
            Elem<T>::template load<DPL>(vt + j * C::ROW_BYTES, lane, vx);
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[h][i] = fmaf(pw, vx[i], acc[h][i]);
          }
        }
        __syncwarp();
      }
      ++seq_c;
      issue_next();  // refill the stage just consumed
    }

#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float l_tot = warp_sum(l_lane[h]);
      const size_t o = (size_t)item * G + h;
      float* dst = ws.partial_acc + o * D + lane * DPL;
      if constexpr (DPL == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(acc[h][0], acc[h][1]);
      }
      if (lane == 0) ws.partial_ml[o] = make_float2(m_run[h], l_tot);
    }
  }
  drain();
}

template <typename T, int D, int G>
inline cudaError_t launch_partial_t(const KParams& kp, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const void* q,
                                    const int32_t* page_table, const int32_t* seq_lens,
                                    const int8_t* modes, const WsView& ws, cudaStream_t stream) {
  constexpr int WARPS = PartialTune<T, D>::WARPS;
  constexpr int STAGES = PartialTune<T, D>::STAGES;
  using C = PartialCfg<T, D, G, WARPS, STAGES>;
  static_assert(C::SMEM_BYTES <= 227 * 1024, "partial kernel shared memory");
  auto kern = partial_kernel<T, D, G, WARPS, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, WARPS * 32, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int grid = sm_count() * per_sm;
  kern<<<grid, WARPS * 32, C::SMEM_BYTES, stream>>>(tmK, tmV, static_cast<const T*>(q),
                                                    page_table, seq_lens, modes, ws, kp);
  return cudaGetLastError();
}

template <typename T, int D>
inline cudaError_t launch_partial_d(const KParams& kp, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const void* q,
                                    const int32_t* page_table, const int32_t* seq_lens,
                                    const int8_t* modes, const WsView& ws, cudaStream_t stream) {
  switch (kp.G) {
    case 1: return launch_partial_t<T, D, 1>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, stream);
    case 2: return launch_partial_t<T, D, 2>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, stream);
    case 4: return launch_partial_t<T, D, 4>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, stream);
    case 8: return launch_partial_t<T, D, 8>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace wise
