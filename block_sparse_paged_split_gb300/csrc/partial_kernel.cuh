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
//   * One producer warp per consumer (one active lane).  It takes the next
//     work item through an atomic counter from one of three lists: the
//     largest-first schedule compaction wrote, list 1 (a sparse call's items,
//     written by the previous depth's finish), or the dense list (every range
//     of every row, mapped from the row lengths through a shared-memory table,
//     no record load).  One self-contained record per item, its tiles as a
//     bitmap over its block range, claimed shortly before it is needed; the
//     producer reads the page table a tile ahead, writes a small
//     descriptor into the stage, and issues one TMA bulk-tensor copy per page
//     and cache (box = one page of one KV head) plus a bulk copy of q, all
//     completing on the stage's "full" mbarrier.  Consumers release a stage
//     through its "empty" mbarrier; the producer waits on it with a
//     suspending try_wait, so it costs no issue slots while idle and
//     consumers never wait on a global load.
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
//   * Programmatic dependent launch: the CTAs start while the previous kernel
//     drains and wait before touching the workspace; with
//     WISE_FLAG_INPUTS_READY a dense-list pass, or a pass on a list built
//     before the previous kernel, issues its first copies before that wait.
#pragma once

#include <mutex>
#include <type_traits>

#include "finish_short.cuh"
#include "internal.h"

namespace wise {

// Descriptor of one stage, written by the producer lane.
struct StageDesc {
  int item;   // partial-output slot of the work item, or -1: no more work
  int tile;   // block index b within the row
  int info;   // n_valid (bits 0-7) | first tile of item (bit 8) | last (bit 9) | discover (bit 10)
  int rg;     // row * Hkv + kv head
};

// A tile the producer has prepared: its stage descriptor, the page ids of
// its (one or two) pages, and where its query rows live.
struct Prepared {
  StageDesc d;
  int pages[2];
  int npg, row, head;
  bool ok;
};

// The tensor-core path (bf16 K/V with 2, 4 or 8 query heads per KV head).
template <typename T, int G>
struct UseMma {
  static constexpr bool value = std::is_same<T, __nv_bfloat16>::value && G >= 2;
};

template <typename T, int D, int G, int C, int S>
struct PartialCfg {
  static constexpr bool MMA = UseMma<T, G>::value;
  static constexpr int DPL = D / 32;
  static constexpr int ROW_BYTES = D * (int)sizeof(T);
  static constexpr int TILE_BYTES = kTile * ROW_BYTES;
  static constexpr int Q_BYTES = G * ROW_BYTES;
  // Stages are 1024-byte aligned on the tensor-core path (the 128-byte TMA
  // swizzle repeats every 1024 bytes).
  static constexpr int STAGE_ALIGN = MMA ? 1024 : 128;
  static constexpr int STAGE_BYTES =
      ((2 * TILE_BYTES + Q_BYTES + STAGE_ALIGN - 1) / STAGE_ALIGN) * STAGE_ALIGN;
  static constexpr int RING_BYTES = S * STAGE_BYTES;
  static constexpr int DESC_BYTES = S * (int)sizeof(StageDesc);
  static constexpr int BAR_BYTES = 2 * S * 8;  // full[S], empty[S]
  // FMA path: fp32 probabilities per head; tensor-core path: bf16 P[8][32].
  static constexpr int PBUF_BYTES = MMA ? 8 * kTile * 2 : G * kTile * 4;
  static constexpr int EXTRA_BYTES =
      ((DESC_BYTES + BAR_BYTES + PBUF_BYTES + STAGE_ALIGN - 1) / STAGE_ALIGN) * STAGE_ALIGN;
  static constexpr int CONSUMER_BYTES = RING_BYTES + EXTRA_BYTES;
  // The dense list's per-row table (WISE_FLAG_DENSE_LIST): first item and
  // length | mode flags of every row, after the consumers' regions.
  static constexpr int TAB_OFF = C * CONSUMER_BYTES;
  static constexpr int TAB_BYTES = ((2 * kMaxDenseRows + 1) * 4 + 127) / 128 * 128;
  static constexpr int SMEM_BYTES = TAB_OFF + TAB_BYTES;
  static constexpr int THREADS = 2 * C * 32;  // C consumer warps, C producer warps
};

// Launch shape per element type, head dim and group: as many consumers as fit
// in ~222 KB of shared memory (one CTA per SM), with three stages each on the
// FMA path and two on the tensor-core path (measured on one box, back to
// back: three stages made the MHA steps 0.5-0.7% faster and the grouped-query
// step 7% slower, where they leave room for only three consumers; four
// stages, three consumers, made the 1K step 7% slower; the 222 KB budget,
// six tensor-core consumers instead of five, made the GQA step 2.2% faster).
template <typename T, int D, int G>
struct PartialTune {
  static constexpr int S = UseMma<T, G>::value ? 2 : 3;
  static constexpr int STAGE_BYTES = PartialCfg<T, D, G, 1, S>::CONSUMER_BYTES;
  static constexpr int C_RAW = (222 * 1024) / STAGE_BYTES;
  // At most 8 tensor-core consumers (their 2 x C warps keep ~128 registers
  // a thread), 12 FMA ones.
  static constexpr int C_MAX = UseMma<T, G>::value ? 8 : 12;
  static constexpr int C = C_RAW > C_MAX ? C_MAX : (C_RAW < 1 ? 1 : C_RAW);
};

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

// ---------------------------------------------------------------- tensor cores
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// c += a * b, m16n8k16, bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared-memory address of the 16-byte chunk `chunk` (0..7) of token row
// `tok` in 128-byte half row `half` of a swizzled tile (the TMA 128-byte
// swizzle XORs the chunk index with the row index modulo 8).
__device__ __forceinline__ uint32_t swz(uint32_t tile, int half, int tok, int chunk) {
  return tile + half * (kTile * 128) + tok * 128 + ((chunk ^ (tok & 7)) << 4);
}

// Consumer of the tensor-core path: a query-head group (G = 2, 4 or 8)
// against one 32-token tile is a small dense contraction.  Scores are
// S^T = K Q^T (m16n8k16: 16 tokens x 8 head columns x 16 dims; tokens as M
// so the group of G <= 8 heads fills N), the output is O^T = V^T P^T with
// P rounded to bf16 in shared memory (fp32 accumulators throughout; the
// exp-sums and per-tile statistics use the fp32 probabilities).  Lane
// (g8, q4) = (lane / 4, lane % 4) holds heads 2 q4 and 2 q4 + 1 of tokens
// g8 (+8) of each 16-token half, and dims g8 (+8) of each 16-dim block of O^T.
// The finish pass folded into the partial pass (rows of at most 64 blocks
// and 8 split slots): where the caller's mask, output and LSE go.  out ==
// nullptr: not folded (a separate finish launch follows).
template <typename T>
struct Fold {
  uint32_t* support;
  T* out;
  float* lse;
};

// Called by a consumer warp after it has written item `d`'s partial result:
// the item is counted on its (row, KV head)'s ticket, and the warp that
// completes the pair's last item finishes the pair (merge, output, LSE,
// selection and mask), then puts the ticket back to 0 so a later launch over
// the same compaction starts afresh.  nit: the pair's item count.
template <typename T>
__device__ __forceinline__ void fold_item_done(const WsView& ws, const KParams& kp, const Fold<T>& fold,
                                               const int32_t* __restrict__ seq_lens,
                                               const int8_t* __restrict__ modes, int rg, int nit,
                                               int lane) {
  __threadfence();  // this warp's partial result and tile statistics, before the ticket
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(ws.tickets + rg, 1) + 1 == nit;
  last = __shfl_sync(kFull, last, 0);
  if (!last) return;
  __threadfence();  // every other item of the pair is visible past the ticket
  const int row = rg / kp.Hkv;
  short_finish_pair_warp<T>(ws, kp, rg, clamp_len(seq_lens[row], kp.cap_tokens), modes[row],
                            fold.support, fold.out, fold.lse, lane);
  if (lane == 0) ws.tickets[rg] = 0;
}

// Pairs without any work item (padding rows, sparse rows selecting nothing)
// are never finished by a ticket: the consumer warps write their output (0)
// and LSE (-inf) at the start, 32 pairs a warp at a time.
template <typename T>
__device__ __forceinline__ void fold_empty_pairs(const WsView& ws, const KParams& kp,
                                                 const Fold<T>& fold, int warp_id, int n_warps,
                                                 int lane) {
  const int npair = kp.R * kp.Hkv;
  const int dpl = kp.D >> 5;
  for (int base = warp_id * 32; base < npair; base += n_warps * 32) {
    const int pr = base + lane;
    const bool empty = pr < npair && ws.head_info[pr].w == 0;
    unsigned todo = __ballot_sync(kFull, empty);
    while (todo) {
      const int e = base + __ffs(todo) - 1;
      todo &= todo - 1;
      const int r = e / kp.Hkv, g = e - r * kp.Hkv;
      const float z[4] = {0.f, 0.f, 0.f, 0.f};
      for (int hl = 0; hl < kp.G; ++hl) {
        const size_t h = (size_t)r * kp.Hq + g * kp.G + hl;
        T* orow = fold.out + h * kp.D + lane * dpl;
        if (dpl == 4) Elem<T>::template store_global<4>(orow, z);
        else Elem<T>::template store_global<2>(orow, reinterpret_cast<const float(&)[2]>(z));
        if (lane == 0) fold.lse[h] = -INFINITY;
      }
    }
  }
}

template <int D, int G, int S, typename Cfg>
__device__ __forceinline__ void mma_consume(const WsView& ws, const KParams& kp, uint8_t* ring_base,
                                            const StageDesc* descs, uint32_t full0,
                                            uint32_t empty0, uint16_t* ps, int lane,
                                            const Fold<__nv_bfloat16>& fold,
                                            const int32_t* __restrict__ seq_lens,
                                            const int8_t* __restrict__ modes) {
  const bool folded = fold.out != nullptr;
  int nit = 0;  // the current item's pair: its item count (folded finish)
  constexpr int KS = D / 16;  // 16-dim blocks: k-steps of S^T, m-tiles of O^T
  const int g8 = lane >> 2, q4 = lane & 3;
  const bool hv[2] = {2 * q4 < G, 2 * q4 + 1 < G};
  uint32_t qb[KS][2];
  float o[KS][4];
  float m_run[2] = {-INFINITY, -INFINITY}, l_lane[2] = {0.f, 0.f};
  for (int i = lane; i < 8 * kTile; i += 32) ps[i] = 0;  // padding heads stay 0
  __syncwarp();
  uint32_t seq = 0;
  while (true) {
    const int stage = seq % S;
    if (!mbar_wait(full0 + 8 * stage, (seq / S) & 1)) {
      if (lane == 0) flag_error(ws.status, WISE_DEVERR_WAIT_TIMEOUT);
      break;
    }
    const StageDesc d = descs[stage];
    if (d.item < 0) break;
    uint8_t* kt = ring_base + stage * Cfg::STAGE_BYTES;
    const uint32_t kb = smem_u32(kt);
    const uint32_t vb = kb + Cfg::TILE_BYTES;
    const int n_valid = d.info & 255;
    const bool disc = (d.info & 1024) != 0;
    if (d.info & 256) {
      if (folded) nit = ws.head_info[d.rg].w;
      const uint8_t* qrow = kt + 2 * Cfg::TILE_BYTES + g8 * Cfg::ROW_BYTES;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[ks][0] = g8 < G ? *reinterpret_cast<const uint32_t*>(qrow + (16 * ks + 2 * q4) * 2) : 0u;
        qb[ks][1] = g8 < G ? *reinterpret_cast<const uint32_t*>(qrow + (16 * ks + 8 + 2 * q4) * 2) : 0u;
#pragma unroll
        for (int v = 0; v < 4; ++v) o[ks][v] = 0.f;
      }
      m_run[0] = m_run[1] = -INFINITY;
      l_lane[0] = l_lane[1] = 0.f;
    }
    if (n_valid < kTile) {
      // Last tile of the row: V rows past the length may hold anything (even
      // NaN) and P . V multiplies every row, so zero them.
      for (int i = lane; i < (kTile - n_valid) * (D / 8); i += 32) {
        const int tok = n_valid + i / (D / 8), c = i % (D / 8);
        *reinterpret_cast<uint4*>(kt + Cfg::TILE_BYTES + (c >> 3) * (kTile * 128) + tok * 128 + (c & 7) * 16) =
            make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }

    // S^T = K Q^T
    float sc[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int v = 0; v < 4; ++v) sc[mt][v] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int m = lane >> 3;
        const int tok = 16 * mt + (m & 1) * 8 + (lane & 7);
        uint32_t a[4];
        ldsm_x4(swz(kb, ks >> 2, tok, (ks & 3) * 2 + (m >> 1)), a);
        mma_bf16(sc[mt], a, qb[ks][0], qb[ks][1]);
      }
    }

    // Online softmax per head column (all lanes shuffle; padding heads do
    // not update any state).
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float sv[4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int tok = 16 * mt + g8 + 8 * i;
          sv[2 * mt + i] = tok < n_valid ? sc[mt][2 * i + j] * kp.scale_log2 : -INFINITY;
        }
      float lm = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) lm = fmaxf(lm, __shfl_xor_sync(kFull, lm, o2));
      if (disc) {
        float e = fast_exp2(sv[0] - lm) + fast_exp2(sv[1] - lm) + fast_exp2(sv[2] - lm) +
                  fast_exp2(sv[3] - lm);
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) e += __shfl_xor_sync(kFull, e, o2);
        if (g8 == 0 && hv[j])
          ws.tile_stats[(size_t)(d.rg * G + 2 * q4 + j) * kp.max_blocks + d.tile] = make_float2(lm, e);
      }
      uint16_t* prow = ps + (2 * q4 + j) * kTile;
      if (hv[j]) {
        const float m_new = fmaxf(m_run[j], lm);
        const float alpha = fast_exp2(m_run[j] - m_new);
        float lsum = 0.f;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float pv = fast_exp2(sv[2 * mt + i] - m_new);
            lsum += pv;
            prow[16 * mt + g8 + 8 * i] = __bfloat16_as_ushort(__float2bfloat16_rn(pv));
          }
        l_lane[j] = fmaf(l_lane[j], alpha, lsum);
        m_run[j] = m_new;
#pragma unroll
        for (int md = 0; md < KS; ++md) {
          o[md][j] *= alpha;
          o[md][2 + j] *= alpha;
        }
      }
    }
    __syncwarp();

    // O^T += V^T P^T
    uint32_t pb[2][2];
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      pb[k2][0] = *reinterpret_cast<const uint32_t*>(ps + g8 * kTile + 16 * k2 + 2 * q4);
      pb[k2][1] = *reinterpret_cast<const uint32_t*>(ps + g8 * kTile + 16 * k2 + 8 + 2 * q4);
    }
#pragma unroll
    for (int md = 0; md < KS; ++md) {
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int m = lane >> 3;
        const int tok = 16 * k2 + 8 * (m >> 1) + (lane & 7);
        const int d0 = 16 * md + 8 * (m & 1);
        uint32_t a[4];
        ldsm_x4_trans(swz(vb, d0 >> 6, tok, (d0 & 63) >> 3), a);
        mma_bf16(o[md], a, pb[k2][0], pb[k2][1]);
      }
    }

    if (d.info & 512) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float l_tot = l_lane[j];
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) l_tot += __shfl_xor_sync(kFull, l_tot, o2);
        if (g8 == 0 && hv[j]) ws.partial_ml[(size_t)d.item * G + 2 * q4 + j] = make_float2(m_run[j], l_tot);
      }
#pragma unroll
      for (int md = 0; md < KS; ++md)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int hh = 2 * q4 + (v & 1);
          if (hh < G)
            ws.partial_acc[((size_t)d.item * G + hh) * D + 16 * md + g8 + (v >= 2 ? 8 : 0)] = o[md][v];
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
    ++seq;
    if (folded && (d.info & 512))
      fold_item_done<__nv_bfloat16>(ws, kp, fold, seq_lens, modes, d.rg, nit, lane);
  }
}

template <typename T, int D, int G, int C, int S>
__global__ void __launch_bounds__(2 * C * 32, 1)
    partial_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const T* __restrict__ q, const int32_t* __restrict__ page_table,
                   const int32_t* __restrict__ seq_lens, const int8_t* __restrict__ modes,
                   const WsView ws, const KParams kp, const Fold<T> fold) {
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

  __shared__ int cta_done;  // producers of this CTA past the queue
  if (threadIdx.x == 0) {
    cta_done = 0;
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    for (int c = 0; c < C; ++c)
      for (int s = 0; s < S; ++s) {
        mbar_init(full_bar(c, s), 1);
        mbar_init(empty_bar(c, s), 1);
      }
    fence_mbar_init();
  }
  // The caller's inputs that every item reads first -- the page table and the
  // query rows -- are pulled into L2 while the previous kernel finishes (a
  // prefetch returns no data, so it may run before the dependency wait).
  prefetch_l2(page_table, (size_t)kp.R * kp.max_pages * sizeof(int32_t));
  prefetch_l2(q, (size_t)kp.R * kp.Hq * D * sizeof(T));
  // The dense list: every range of T blocks of every row is an item, ordered
  // by row, then KV head, then range; warp 0 tabulates each row's first item
  // (a prefix over the rows' Hkv * ceil(ceil(L / 32) / T) items) and its
  // length and mode flags, so a claim maps to its item with no record load.
  // Every row's two loads go out at once.
  int* tab_start = reinterpret_cast<int*>(smem + Cfg::TAB_OFF);  // [R + 1]
  int* tab_w = tab_start + kMaxDenseRows + 1;                      // [R]
  bool clamped = false;
  auto build_table = [&]() {
    constexpr int kChunks = kMaxDenseRows / 32;
    int raw[kChunks], md[kChunks];
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      const int r = j * 32 + lane;
      raw[j] = r < kp.R ? __ldcg(seq_lens + r) : 0;
      md[j] = r < kp.R ? (int)__ldcg(modes + r) : 0;
    }
    int carry = 0;
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      if (j * 32 < kp.R) {
        const int r = j * 32 + lane;
        const int L = clamp_len(raw[j], kp.cap_tokens);
        const int nb = (L + kTile - 1) / kTile;
        const int items = r < kp.R ? kp.Hkv * ((nb + kp.T - 1) / kp.T) : 0;
        clamped |= raw[j] > kp.cap_tokens;
        int incl = items;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += y;
        }
        if (r < kp.R) {
          tab_start[r] = carry + incl - items;
          tab_w[r] = L | ((md[j] == WISE_MODE_DISCOVER || md[j] == WISE_MODE_DISCOVER_UNION)
                              ? kItemDiscover : 0);
        }
        carry += __shfl_sync(kFull, incl, 31);
      }
    }
    if (lane == 0) tab_start[kp.R] = carry;
  };
  // With everything the pass reads complete before the previous kernel began
  // (WISE_FLAG_INPUTS_READY: the caller's inputs, and on list 1 the list),
  // the table is built before the dependency wait, and the producers take
  // their first item (from the table, or list 1's counters and records) and
  // issue its copies (page table, K and V) while that kernel still runs,
  // waiting only before the queue claims and the first reuse of a stage; the
  // consumers wait here, before they write.  Those early reads bypass L1.
  const bool early_reads = (kp.dense_list || kp.list1) && kp.inputs_ready;
  if (early_reads && kp.dense_list && warp == 0) build_table();
  __syncthreads();
  // Compaction's items, schedule and counters.  An early-start launch (the
  // previous kernel writes nothing it reads and reads nothing it writes; the
  // compaction it uses completed before that kernel began) skips the wait
  // here and waits before it exits instead, so its completion still implies
  // the previous kernel's.  Its producers, like those of an early-reading
  // pass, still wait before their first queue claim: the kernel ahead may
  // have started before the partial pass that last used the queue had put
  // it back to 0.
  const bool producer_defers = (kp.early || early_reads) && warp >= C;
  if (!kp.early && !producer_defers) grid_dependency_wait();
  if (kp.dense_list && !kp.inputs_ready) {
    if (warp == 0) build_table();
    __syncthreads();
  }
  // A dense-list pass has no compaction to clear the status word: block 0
  // clears it once the previous kernel (which may flag into it) is done, then
  // flags a clamped length.  An early-start pass runs beside that kernel, so
  // it leaves the word as it is and only adds its own flag.
  if (kp.dense_list && blockIdx.x == 0 && warp == 0) {
    if (lane == 0 && !kp.early) *ws.status = 0;
    __syncwarp();
    if (__any_sync(kFull, clamped) && lane == 0) flag_error(ws.status, WISE_DEVERR_SEQ_LEN_CLAMPED);
  }

  if (warp >= C) {
    // ------------------------------------------------------------ producers
    // Warp C + c feeds consumer c; one lane does the work.  It holds the next
    // work item's record (claimed when the current item is about to run out)
    // and the next tile prepared (descriptor and page ids), so a stage that
    // frees gets its copies issued at once.  It waits for a free stage with a
    // suspending try_wait, so an idle producer takes no issue slots.
    if (lane != 0) return;
    const int c = warp - C;
    uint32_t seq = 0;
    bool exhausted = false, first_claim = true;
    int4 nxt = make_int4(0, 0, 0, 0), cur = make_int4(0, 0, 0, 0);
    bool nxt_ok = false, cur_ok = false;
    int k = 0;
    Prepared p{};
    int ahead[2] = {0, 0};  // page ids of the current item's tile k (when ahead_ok)
    bool ahead_ok = false;
    // Each consumer's first item is its own schedule slot (no atomic on the
    // launch's critical path); later ones come from the counter, offset by
    // the number of consumers in the grid.
    const int n_consumers = gridDim.x * C;
    // The item count and the first item's record are loaded together (the
    // record's slot is inside the item array whatever the count).  List 1
    // keeps its items in one bucket per tile count (larger counts first in
    // the schedule): the buckets' schedule positions come first, then the
    // record.
    const int first_slot = blockIdx.x * C + c;
    int l1s[kMaxT];  // list 1: schedule position of the first item with j + 1 tiles
    auto record_at = [&](int slot) -> int4 {
      if (kp.dense_list) {
        // The row: the last one whose first item is at or before the slot
        // (an empty row shares its start with the next row, which wins).
        int lo = 0, hi = kp.R - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (tab_start[mid] <= slot) lo = mid;
          else hi = mid - 1;
        }
        const int w = tab_w[lo];
        const int nb = ((w & kItemLenMask) + kTile - 1) / kTile;
        const int nr = (nb + kp.T - 1) / kp.T;
        const int local = slot - tab_start[lo];
        const int g = local / nr, s_rng = local - g * nr;
        const int n = min(kp.T, nb - s_rng * kp.T);
        return make_int4(lo * kp.Hkv + g, s_rng | (s_rng << 16),
                         (int)(((1u << n) - 1u) | ((unsigned)n << 16)), w);
      }
      if (!kp.list1) return ws.items[slot];
      // Bucket j holds schedule positions [l1s[j], l1s[j - 1]) (l1s is
      // non-increasing in j and l1s[T - 1] = 0): the smallest j with
      // l1s[j] <= slot.
      int jsel = kp.T - 1, base = 0;
#pragma unroll
      for (int j = kMaxT - 1; j >= 0; --j)
        if (j < kp.T && l1s[j] <= slot) {
          jsel = j;
          base = l1s[j];
        }
      const int idx = slot - base;
      if (idx < 0 || idx >= ws.max_items) return make_int4(-1, 0, 0, 0);  // rejected below
      return __ldcg(ws.items_1 + (size_t)jsel * ws.max_items + idx);
    };
    // A record the library did not write for this shape (a call out of
    // order on the workspace) is flagged and skipped, never followed.
    // Only what keeps every access in bounds is checked: the pair, the range
    // and the slot, a non-empty bitmap inside the range, and its last tile
    // below the row's length.  (The producer counts an item's tiles from the
    // bitmap, so the record's count field is never trusted.)
    auto record_ok = [&](const int4& rec) {
      const unsigned bits = (unsigned)rec.z & 0xffffu;
      const unsigned s_rng = (unsigned)rec.y & 0xffffu, slot = (unsigned)rec.y >> 16;
      const int L = rec.w & kItemLenMask;
      const int last = (int)s_rng * kp.T + 31 - __clz(bits | 1u);
      const bool ok = (unsigned)rec.x < (unsigned)(kp.R * kp.Hkv) &&
                      max(s_rng, slot) < (unsigned)kp.S_max && bits - 1u < (1u << kp.T) - 1u &&
                      L <= kp.cap_tokens && last * kTile < L;
      if (!ok) flag_error(ws.status, WISE_DEVERR_BAD_WORK_LIST);
      return ok;
    };
    int n_items;
    int4 first_rec = make_int4(0, 0, 0, 0);
    if (kp.dense_list) {
      n_items = tab_start[kp.R];
      if (first_slot < n_items) first_rec = record_at(first_slot);
    } else if (kp.list1) {
      // Schedule position of each bucket: the items of larger buckets first.
      int cnt[kMaxT];
#pragma unroll
      for (int j = 0; j < kMaxT; ++j) cnt[j] = j < kp.T ? __ldcg(ws.l1_counter + j) : 0;
      int pos = 0;
#pragma unroll
      for (int j = kMaxT - 1; j >= 0; --j) {
        l1s[j] = pos;
        pos += min(max(cnt[j], 0), ws.max_items);
      }
      n_items = pos;
      if (first_slot < n_items) first_rec = record_at(first_slot);
    } else {
      first_rec = first_slot < ws.max_items ? ws.items[first_slot] : make_int4(0, 0, 0, 0);
      n_items = min(*ws.num_items, ws.max_items);
    }
    bool timed_out = false;
    bool waited = !producer_defers;  // the dependency wait is behind this lane
    while (true) {
      if (!cur_ok && nxt_ok) {
        cur = nxt;
        cur_ok = true;
        nxt_ok = false;
        k = 0;
      }
      // Claim the next item only when the current one is about to run out
      // (one tile left to prepare): claiming earlier would hoard items other
      // consumers could start sooner (measured: claiming at four tiles left
      // is 0.9% slower, at one 0.5% faster than at two).  Small items of
      // list 1 (a few selected tiles each) need their claim, record and
      // page-table round trips started earlier than one tile covers: there
      // the claim goes out two tiles ahead (measured at 1K: sparse partial
      // 22.9 vs 23.6 µs, step -0.35%).
      const int cur_tiles = __popc((unsigned)cur.z & 0xffffu);
      if (!nxt_ok && !exhausted &&
          (!cur_ok || cur_tiles - k <= (kp.list1 && cur_tiles <= 4 ? 2 : 1))) {
        if (!first_claim && !waited) {
          grid_dependency_wait();
          waited = true;
        }
        const int slot = first_claim ? first_slot : n_consumers + atomicAdd(ws.queue, 1);
        if (slot < n_items) {
          nxt = first_claim ? first_rec : record_at(slot);
          nxt_ok = record_ok(nxt);
        } else {
          exhausted = true;
        }
        first_claim = false;
        if (!cur_ok && nxt_ok) continue;  // start on it right away
      }
      if (cur_ok && !p.ok) {
        // Prepare tile k of the current item: the k-th set bit of its range
        // bitmap, and the page ids of its one or two pages.
        const int rg = cur.x;
        const int ntiles = __popc((unsigned)cur.z & 0xffffu);
        const int L = cur.w & kItemLenMask;
        const int row = rg / kp.Hkv;
        const int range0 = (cur.y & 0xffff) * kp.T;
        const int b = range0 + (int)__fns((unsigned)cur.z & 0xffffu, 0, k + 1);
        // A tile's page ids are loaded one tile ahead (with the previous
        // tile's), so two tiles' copies go out back to back at an item's start.
        auto load_pages = [&](int blk, int (&pg)[2]) {
          const int32_t* pt = page_table + (size_t)row * kp.max_pages + blk * (kTile / kp.P);
          const bool two = kp.P * 2 == kTile && blk * kTile + kp.P < L;
          pg[0] = __ldcg(pt);
          pg[1] = two ? __ldcg(pt + 1) : 0;
        };
        if (ahead_ok) {
          p.pages[0] = ahead[0];
          p.pages[1] = ahead[1];
        } else {
          load_pages(b, p.pages);
        }
        ahead_ok = k + 1 < ntiles;
        if (ahead_ok) load_pages(range0 + (int)__fns((unsigned)cur.z & 0xffffu, 0, k + 2), ahead);
        const int tok0 = b * kTile;
        const int rem = L - tok0;
        const int pages_in_tile = kTile / kp.P;
        int npg = (rem + kp.P - 1) / kp.P;
        p.npg = npg < pages_in_tile ? npg : pages_in_tile;
        p.row = row;
        p.head = rg - row * kp.Hkv;
        p.d.item = rg * kp.S_max + (cur.y >> 16);
        p.d.tile = b;
        p.d.info = (rem < kTile ? rem : kTile) | (k == 0 ? 256 : 0) | (k + 1 == ntiles ? 512 : 0) |
                   ((cur.w & kItemDiscover) ? 1024 : 0);
        p.d.rg = rg;
        p.ok = true;
        if (++k == ntiles) cur_ok = false;
      }
      if (!p.ok && (cur_ok || nxt_ok || !exhausted)) continue;
      // Wait for the stage (bounded), then issue the prepared tile or, with
      // nothing left, the end marker.  A stage is reused only once the
      // consumer frees it, which it does past its dependency wait: a deferring
      // producer takes that wait first, so the bounded wait below never
      // counts the previous kernel's run time.
      const int stage = seq % S;
      if (seq >= (uint32_t)S && !waited && !kp.early) {
        grid_dependency_wait();
        waited = true;
      }
      if (!mbar_wait(empty_bar(c, stage), ((seq / S) & 1) ^ 1)) {
        flag_error(ws.status, WISE_DEVERR_WAIT_TIMEOUT);
        timed_out = true;
        // Copies already issued into the ring may still be landing: wait
        // (bounded) for the last phase of every stage issued before leaving,
        // so the CTA never exits with a bulk copy writing its shared memory.
        for (uint32_t i = seq > (uint32_t)S ? seq - S : 0u; i < seq; ++i)
          mbar_wait(full_bar(c, i % S), (i / S) & 1);
        break;
      }
      StageDesc* d = descs(c) + stage;
      const uint32_t fb = full_bar(c, stage);
      if (!p.ok) {
        d->item = -1;
        mbar_arrive(fb);
        break;
      }
      *d = p.d;
      const bool first = (p.d.info & 256) != 0;
      mbar_arrive_expect_tx(fb, (uint32_t)(2 * p.npg * kp.P * Cfg::ROW_BYTES) +
                                    (first ? (uint32_t)Cfg::Q_BYTES : 0u));
      const uint32_t kdst = smem_u32(ring(c) + stage * Cfg::STAGE_BYTES);
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        if (pp < p.npg) {
          const int page = p.pages[pp];
          // A page id outside the pool reads the out-of-bounds fill (zeros).
          const int tok = (page >= 0 && page < kp.num_pages) ? page * kp.P : kp.num_pages * kp.P;
          if constexpr (Cfg::MMA) {
            // 64-element half rows with the 128-byte swizzle: half h of the
            // tile is [32 tokens][128 B] at h * 4 KB.
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
              const uint32_t off = h * (kTile * 128) + pp * kp.P * 128;
              tma_load_3d(kdst + off, &tmK, h * 64, p.head, tok, fb);
              tma_load_3d(kdst + Cfg::TILE_BYTES + off, &tmV, h * 64, p.head, tok, fb);
            }
          } else {
            const uint32_t off = pp * kp.P * Cfg::ROW_BYTES;
            tma_load_3d(kdst + off, &tmK, 0, p.head, tok, fb);
            tma_load_3d(kdst + Cfg::TILE_BYTES + off, &tmV, 0, p.head, tok, fb);
          }
        }
      }
      if (first)
        bulk_load(kdst + 2 * Cfg::TILE_BYTES, q + ((size_t)p.row * kp.Hq + p.head * G) * D,
                  Cfg::Q_BYTES, fb);
      ++seq;
      p.ok = false;
    }
    if (!waited) grid_dependency_wait();  // before the counters below
    // This CTA's last producer past the queue tells the grid; the last CTA
    // puts the counter back to 0, so a later partial launch over the same
    // compaction (the next depth reusing a mask) starts afresh.
    if (!timed_out && atomicAdd(&cta_done, 1) == C - 1) {
      grid_dependents_launch();  // the finish pass may start launching
      __threadfence();
      if (atomicAdd(ws.queue_done, 1) == (int)gridDim.x - 1) {
        __threadfence();
        atomicExch(ws.queue, 0);
        atomicExch(ws.queue_done, 0);
        // A finish of this call may build list 1: its counters start at 0.
        // (A pass on list 1 leaves them: the next call may reuse the list.)
        if (!kp.list1)
          for (int j = 0; j < kMaxT; ++j) ws.l1_counter[j] = 0;
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  if (fold.out != nullptr) fold_empty_pairs<T>(ws, kp, fold, blockIdx.x * C + warp, gridDim.x * C, lane);
  if constexpr (Cfg::MMA) {
    mma_consume<D, G, S, Cfg>(
        ws, kp, ring(warp), descs(warp), full_bar(warp, 0), empty_bar(warp, 0),
        reinterpret_cast<uint16_t*>(ring(warp) + Cfg::RING_BYTES + Cfg::DESC_BYTES + Cfg::BAR_BYTES),
        lane, fold, seq_lens, modes);
  } else {
  const int c = warp;
  float* pbuf = reinterpret_cast<float*>(ring(c) + Cfg::RING_BYTES + Cfg::DESC_BYTES + Cfg::BAR_BYTES);
  QRegs<T, DPL> qr[G];
  float m_run[G], l_lane[G], acc[G][DPL];
  uint32_t seq = 0;
  const bool folded = fold.out != nullptr;
  int nit = 0;  // the current item's pair: its item count (folded finish)
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
      if (folded) nit = ws.head_info[d.rg].w;
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
    if (folded && (d.info & 512)) fold_item_done<T>(ws, kp, fold, seq_lens, modes, d.rg, nit, lane);
  }
  }
  if (kp.early && threadIdx.x == 0) grid_dependency_wait();  // see the prologue
}

template <typename T, int D, int G>
inline cudaError_t launch_partial_t(const KParams& kp, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const void* q,
                                    const int32_t* page_table, const int32_t* seq_lens,
                                    const int8_t* modes, const WsView& ws, const FoldArgs& fa,
                                    cudaStream_t stream) {
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
  const Fold<T> fold{fa.support, static_cast<T*>(fa.out), fa.lse};
  return launch_pdl(kern, dim3(grid), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, stream, tmK, tmV,
                    static_cast<const T*>(q), page_table, seq_lens, modes, ws, kp, fold);
}

template <typename T, int D>
inline cudaError_t launch_partial_d(const KParams& kp, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const void* q,
                                    const int32_t* page_table, const int32_t* seq_lens,
                                    const int8_t* modes, const WsView& ws, const FoldArgs& fa,
                                    cudaStream_t stream) {
  switch (kp.G) {
    case 1: return launch_partial_t<T, D, 1>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, fa, stream);
    case 2: return launch_partial_t<T, D, 2>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, fa, stream);
    case 4: return launch_partial_t<T, D, 4>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, fa, stream);
    case 8: return launch_partial_t<T, D, 8>(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, fa, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace wise
