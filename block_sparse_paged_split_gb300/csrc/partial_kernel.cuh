// Split partial pass of WISE paged decode attention (one launch per call).
//
// [WISE PR, "What changes"]: split-KV paged decode with per-row modes; dense
// rows attend every tile, discover rows also record each 32-token tile's max
// and exp-sum, sparse rows walk their compacted tile list; programs cover
// about eight tiles, so one long dense row does not set the latency of a
// launch whose other rows are sparse.
//
// GB300 design (persistent, one CTA per SM, warp-specialised):
//   * C consumer warps, each owning an S-deep ring of shared-memory stages;
//     one stage holds one 32-token tile of K and of V (and, for the first tile
//     of a work item, the item's query rows).
//   * One producer warp.  Its lane c feeds consumer c: it takes the next work
//     item from the largest-first schedule through an atomic counter (one
//     self-contained record per item, fetched an item ahead), reads the tile
//     list and page table two tiles ahead, writes a small descriptor into the stage,
//     and issues one TMA bulk-tensor copy per page and cache (box = one page of
//     one KV head) plus a bulk copy of q, all completing on the stage's "full"
//     mbarrier.  Consumers release a stage through its "empty" mbarrier.  The
//     producer polls with non-blocking tests, so one lane's wait never holds
//     another consumer's refill; consumers never wait on a global load.
//   * Math is FP32 FMA: multi-head decode reads each K/V element once (about
//     one FMA per byte, far below the tensor-core ridge).  Lane l holds dims
//     [l*DPL, (l+1)*DPL) of the query; lane l computes token (i XOR l) at
//     step i, which makes the 31-shuffle transpose reduction select-free and
//     leaves lane j with token j's score.  bf16 operands go straight into
//     fma.rn.f32.bf16 (exact products, one rounding: the same result as
//     widening first).  Scores are kept in log2 units (scale * log2 e folded
//     in) and exponentiated with ex2.approx.
//   * Online softmax per item: running max m, per-lane exp-sum, accumulator
//     rescaled once per tile.  The item's unnormalised output, max and
//     exp-sum go to the workspace; the finish kernel merges the items.
#pragma once

#include <mutex>

#include "internal.h"

namespace wise {

// Descriptor of one stage, written by the producer lane.
struct StageDesc {
  int item;   // partial-output slot of the work item, or -1: no more work
  int tile;   // block index b within the row
  int info;   // n_valid (bits 0-7) | first tile of item (bit 8) | last (bit 9) | discover (bit 10)
  int rg;     // row * Hkv + kv head
};

// A tile the producer lane has prepared: its stage descriptor, the page ids
// of its (one or two) pages, and where its query rows live.
struct Prepared {
  StageDesc d;
  int pages[2];
  int npg, row, head;
  bool ok;
};

template <typename T, int D, int G, int C, int S>
struct PartialCfg {
  static constexpr int DPL = D / 32;
  static constexpr int ROW_BYTES = D * (int)sizeof(T);
  static constexpr int TILE_BYTES = kTile * ROW_BYTES;
  static constexpr int Q_BYTES = G * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES + ((Q_BYTES + 127) / 128) * 128;
  static constexpr int RING_BYTES = S * STAGE_BYTES;
  static constexpr int DESC_BYTES = S * (int)sizeof(StageDesc);
  static constexpr int BAR_BYTES = 2 * S * 8;  // full[S], empty[S]
  static constexpr int PBUF_BYTES = G * kTile * 4;
  static constexpr int EXTRA_BYTES = ((DESC_BYTES + BAR_BYTES + PBUF_BYTES + 127) / 128) * 128;
  static constexpr int CONSUMER_BYTES = RING_BYTES + EXTRA_BYTES;
  static constexpr int SMEM_BYTES = C * CONSUMER_BYTES;
  static constexpr int THREADS = (C + 1) * 32;
};

// Launch shape per element type and head dim: two stages per consumer and as
// many consumers as fit in ~200 KB of shared memory (one CTA per SM); six
// consumers with two stages measured faster than four with three.
template <typename T, int D, int G>
struct PartialTune {
  static constexpr int S = 2;
  static constexpr int STAGE_BYTES = PartialCfg<T, D, G, 1, S>::CONSUMER_BYTES;
  static constexpr int C_RAW = (200 * 1024) / STAGE_BYTES;
  static constexpr int C = C_RAW > 12 ? 12 : (C_RAW < 1 ? 1 : C_RAW);
};

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// d = a * b + c with bf16 a, b (packed in the low/high half of a 32-bit word)
// and an fp32 accumulator.
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

// Query rows of one head, as the consumer keeps them: bf16 stays packed (the
// q.k products use fma.rn.f32.bf16), fp32 stays fp32.
template <typename T, int DPL>
struct QRegs;

template <int DPL>
struct QRegs<__nv_bfloat16, DPL> {
  uint32_t w[DPL / 2];
  __device__ __forceinline__ void load(const uint8_t* row, int lane) {
    if constexpr (DPL == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(row + lane * 8);
      w[0] = v.x; w[1] = v.y;
    } else {
      w[0] = *reinterpret_cast<const uint32_t*>(row + lane * 4);
    }
  }
  // <q, k> over this lane's dims, k read from a shared-memory row.
  __device__ __forceinline__ float dot(const uint8_t* krow, int lane) const {
    if constexpr (DPL == 4) {
      const uint2 k = *reinterpret_cast<const uint2*>(krow + lane * 8);
      float a = fma_bf16_lo(w[0], k.x, 0.f);
      a = fma_bf16_hi(w[0], k.x, a);
      a = fma_bf16_lo(w[1], k.y, a);
      return fma_bf16_hi(w[1], k.y, a);
    } else {
      const uint32_t k = *reinterpret_cast<const uint32_t*>(krow + lane * 4);
      return fma_bf16_hi(w[0], k, fma_bf16_lo(w[0], k, 0.f));
    }
  }
};

template <int DPL>
struct QRegs<float, DPL> {
  float x[DPL];
  __device__ __forceinline__ void load(const uint8_t* row, int lane) {
    Elem<float>::template load<DPL>(row, lane, x);
  }
  __device__ __forceinline__ float dot(const uint8_t* krow, int lane) const {
    float k[DPL];
    Elem<float>::template load<DPL>(krow, lane, k);
    float a = x[0] * k[0];
#pragma unroll
    for (int i = 1; i < DPL; ++i) a = fmaf(x[i], k[i], a);
    return a;
  }
};

template <typename T, int D, int G, int C, int S>
__global__ void __launch_bounds__((C + 1) * 32, 1)
    partial_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const T* __restrict__ q, const int32_t* __restrict__ page_table,
                   const int32_t* __restrict__ seq_lens, const int8_t* __restrict__ modes,
                   const WsView ws, const KParams kp) {
  using Cfg = PartialCfg<T, D, G, C, S>;
  constexpr int DPL = Cfg::DPL;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  // Per-consumer regions: ring | descriptors | full[S] | empty[S] | pbuf.
  auto ring = [&](int c) { return smem + c * Cfg::CONSUMER_BYTES; };
  auto descs = [&](int c) {
    return reinterpret_cast<StageDesc*>(ring(c) + Cfg::RING_BYTES);
  };
  auto full_bar = [&](int c, int s) {
    return smem_u32(ring(c) + Cfg::RING_BYTES + Cfg::DESC_BYTES) + 8 * s;
  };
  auto empty_bar = [&](int c, int s) { return full_bar(c, 0) + 8 * (S + s); };

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    for (int c = 0; c < C; ++c)
      for (int s = 0; s < S; ++s) {
        mbar_init(full_bar(c, s), 1);
        mbar_init(empty_bar(c, s), 1);
      }
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();  // compaction's items, schedule and counters

  const int n_items = *ws.num_items;

  if (warp == C) {
    // ------------------------------------------------------------ producer
    // Lane c serves consumer c.  It holds the next work item's record (loaded
    // as soon as the current item starts) and up to two tiles prepared ahead
    // (descriptor and page ids, whose loads overlap the wait for a free
    // stage), so a stage that frees gets its copies issued at once.
    const bool active = lane < C;
    const int c = lane;
    uint32_t seq = 0;
    bool exhausted = !active, posted_done = !active;
    int4 nxt = make_int4(0, 0, 0, 0), cur = make_int4(0, 0, 0, 0);
    bool nxt_ok = false, cur_ok = false;
    int k = 0;
    Prepared p0{}, p1{};
    uint64_t idle_since = 0;
    // Each consumer's first item is its own schedule slot (no atomic on the
    // launch's critical path); later ones come from the counter, offset by
    // the number of consumers in the grid.
    const int n_consumers = gridDim.x * C;
    bool first_claim = true;
    while (true) {
      bool progressed = false;
      if (!posted_done) {
        if (!cur_ok && nxt_ok) {
          cur = nxt;
          cur_ok = true;
          nxt_ok = false;
          k = 0;
        }
        // Claim the next item only when the current one is about to run out
        // (two tiles left to prepare): claiming earlier would hoard items
        // other consumers could start sooner.
        if (!nxt_ok && !exhausted && (!cur_ok || (cur.z & 0xff) - k <= 2)) {
          const int slot = first_claim ? blockIdx.x * C + c : n_consumers + atomicAdd(ws.queue, 1);
          first_claim = false;
          if (slot < n_items) {
            nxt = ws.items[slot];
            nxt_ok = true;
          } else {
            exhausted = true;
          }
        }
        if (cur_ok && !p1.ok) {
          // Prepare tile k of the current item into p1.
          const int rg = cur.x;
          const int ntiles = cur.z & 0xff;
          const int row = rg / kp.Hkv;
          int b;
          if (cur.z & kItemSparse) {
            // One load: the compacted tile with its page ids.
            const int4 t = ws.tile_list[(size_t)rg * kp.max_blocks + cur.y + k];
            b = t.x;
            p1.pages[0] = t.y;
            p1.pages[1] = t.z;
          } else {
            b = cur.y + k;
            const int32_t* pt = page_table + (size_t)row * kp.max_pages + b * (kTile / kp.P);
            const bool two = kp.P * 2 == kTile && b * kTile + kp.P < cur.w;
            p1.pages[0] = pt[0];
            p1.pages[1] = two ? pt[1] : 0;
          }
          const int tok0 = b * kTile;
          const int rem = cur.w - tok0;
          const int pages_in_tile = kTile / kp.P;
          int npg = (rem + kp.P - 1) / kp.P;
          npg = npg < pages_in_tile ? npg : pages_in_tile;
          p1.npg = npg;
          p1.row = row;
          p1.head = rg - row * kp.Hkv;
          p1.d.item = rg * kp.S_max + ((cur.z >> 8) & 0xffff);
          p1.d.tile = b;
          p1.d.info = (rem < kTile ? rem : kTile) | (k == 0 ? 256 : 0) | (k + 1 == ntiles ? 512 : 0) |
                      ((cur.z & kItemDiscover) ? 1024 : 0);
          p1.d.rg = rg;
          p1.ok = true;
          if (++k == ntiles) cur_ok = false;
          if (!p0.ok) {
            p0 = p1;
            p1.ok = false;
          }
        }
        const bool all_out = !p0.ok && !cur_ok && !nxt_ok && exhausted;
        if (p0.ok || all_out) {
          const int stage = seq % S;
          if (mbar_test_wait(empty_bar(c, stage), ((seq / S) & 1) ^ 1)) {
            StageDesc* d = descs(c) + stage;
            const uint32_t fb = full_bar(c, stage);
            if (p0.ok) {
              *d = p0.d;
              const bool first = (p0.d.info & 256) != 0;
              mbar_arrive_expect_tx(fb, (uint32_t)(2 * p0.npg * kp.P * Cfg::ROW_BYTES) +
                                            (first ? (uint32_t)Cfg::Q_BYTES : 0u));
              const uint32_t kdst = smem_u32(ring(c) + stage * Cfg::STAGE_BYTES);
#pragma unroll
              for (int pp = 0; pp < 2; ++pp) {
                if (pp < p0.npg) {
                  const int page = p0.pages[pp];
                  // A page id outside the pool reads the out-of-bounds fill (zeros).
                  const int tok = (page >= 0 && page < kp.num_pages) ? page * kp.P : kp.num_pages * kp.P;
                  const uint32_t off = pp * kp.P * Cfg::ROW_BYTES;
                  tma_load_3d(kdst + off, &tmK, 0, p0.head, tok, fb);
                  tma_load_3d(kdst + Cfg::TILE_BYTES + off, &tmV, 0, p0.head, tok, fb);
                }
              }
              if (first)
                bulk_load(kdst + 2 * Cfg::TILE_BYTES, q + ((size_t)p0.row * kp.Hq + p0.head * G) * D,
                          Cfg::Q_BYTES, fb);
              ++seq;
              p0 = p1;
              p1.ok = false;
            } else {
              d->item = -1;
              mbar_arrive(fb);
              posted_done = true;
            }
            progressed = true;
          }
        }
      }
      if (__all_sync(kFull, posted_done)) {
        // Every lane of this CTA is past the queue.  The last CTA to get here
        // puts the counter back to 0, so a later partial launch over the
        // same compaction (the next depth reusing a mask) starts afresh.
        if (lane == 0) {
          grid_dependents_launch();  // the finish pass may start launching
          __threadfence();
          if (atomicAdd(ws.queue_done, 1) == (int)gridDim.x - 1) {
            __threadfence();
            atomicExch(ws.queue, 0);
            atomicExch(ws.queue_done, 0);
          }
        }
        break;
      }
      if (__any_sync(kFull, progressed)) {
        idle_since = 0;
      } else {
        const uint64_t now = global_ns();
        if (idle_since == 0) idle_since = now;
        if (now - idle_since > kWaitLimitNs) {
          flag_error(ws.status, WISE_DEVERR_WAIT_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int c = warp;
  float* pbuf = reinterpret_cast<float*>(ring(c) + Cfg::RING_BYTES + Cfg::DESC_BYTES + Cfg::BAR_BYTES);
  QRegs<T, DPL> qr[G];
  float m_run[G], l_lane[G], acc[G][DPL];
  uint32_t seq = 0;
  while (true) {
    const int stage = seq % S;
    if (!mbar_wait(full_bar(c, stage), (seq / S) & 1)) {
      if (lane == 0) flag_error(ws.status, WISE_DEVERR_WAIT_TIMEOUT);
      break;
    }
    const StageDesc d = descs(c)[stage];
    if (d.item < 0) break;
    const uint8_t* kt = ring(c) + stage * Cfg::STAGE_BYTES;
    const uint8_t* vt = kt + Cfg::TILE_BYTES;
    const int n_valid = d.info & 255;
    const bool disc = (d.info & 1024) != 0;
    if (d.info & 256) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        qr[h].load(kt + 2 * Cfg::TILE_BYTES + h * Cfg::ROW_BYTES, lane);
        m_run[h] = -INFINITY;
        l_lane[h] = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[h][i] = 0.f;
      }
    }

#pragma unroll
    for (int h = 0; h < G; ++h) {
      // Lane computes token (i ^ lane) at step i.
      float part[kTile];
#pragma unroll
      for (int i = 0; i < kTile; ++i) part[i] = qr[h].dot(kt + (i ^ lane) * Cfg::ROW_BYTES, lane);
      // Select-free transpose reduction: keep the low half, add the
      // partner's high half (which holds the same tokens).
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int i = 0; i < o; ++i) part[i] += __shfl_xor_sync(kFull, part[i + o], o);
      }
      const float s = lane < n_valid ? part[0] * kp.scale_log2 : -INFINITY;
      const float mt = warp_max(s);
      if (disc) {
        const float lb = warp_sum(fast_exp2(s - mt));
        if (lane == 0)
          ws.tile_stats[(size_t)(d.rg * G + h) * kp.max_blocks + d.tile] = make_float2(mt, lb);
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
            Elem<T>::template load<DPL>(vt + (j + u) * Cfg::ROW_BYTES, lane, vx);
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[h][i] = fmaf(pw[u], vx[i], acc[h][i]);
          }
        }
      } else {
        // Last tile of the row: slots past the length may hold anything
        // (even NaN) and are never touched.
        for (int j = 0; j < n_valid; ++j) {
          const float pw = pb[j];
          float vx[DPL];
          Elem<T>::template load<DPL>(vt + j * Cfg::ROW_BYTES, lane, vx);
#pragma unroll
          for (int i = 0; i < DPL; ++i) acc[h][i] = fmaf(pw, vx[i], acc[h][i]);
        }
      }
      __syncwarp();
    }

    if (d.info & 512) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float l_tot = warp_sum(l_lane[h]);
        const size_t o = (size_t)d.item * G + h;
        float* dst = ws.partial_acc + o * D + lane * DPL;
        if constexpr (DPL == 4) {
          *reinterpret_cast<float4*>(dst) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
        } else {
          *reinterpret_cast<float2*>(dst) = make_float2(acc[h][0], acc[h][1]);
        }
        if (lane == 0) ws.partial_ml[o] = make_float2(m_run[h], l_tot);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(c, stage));
    ++seq;
  }
}

template <typename T, int D, int G>
inline cudaError_t launch_partial_t(const KParams& kp, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const void* q,
                                    const int32_t* page_table, const int32_t* seq_lens,
                                    const int8_t* modes, const WsView& ws, cudaStream_t stream) {
  constexpr int C = PartialTune<T, D, G>::C;
  constexpr int S = PartialTune<T, D, G>::S;
  using Cfg = PartialCfg<T, D, G, C, S>;
  static_assert(Cfg::SMEM_BYTES <= 227 * 1024, "partial kernel shared memory");
  static_assert(Cfg::Q_BYTES % 16 == 0, "bulk copy of q needs a multiple of 16 bytes");
  auto kern = partial_kernel<T, D, G, C, S>;
  // Kernel attributes and occupancy are set up once per device (so a call
  // inside a stream capture issues only the launch).
  static std::mutex mu;
  static int grid_of_device[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int grid;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!grid_of_device[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::THREADS, Cfg::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      grid_of_device[dev] = sm_count() * (per_sm < 1 ? 1 : per_sm);
    }
    grid = grid_of_device[dev];
  }
  return launch_pdl(kern, dim3(grid), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, stream, tmK, tmV,
                    static_cast<const T*>(q), page_table, seq_lens, modes, ws, kp);
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
