// Device helpers shared by the WISE kernels: inline PTX for mbarriers and TMA
// bulk-tensor copies (sm_90+ forms, compiled for sm_103a), bounded waits, and
// warp-level reductions.  Nothing here depends on torch.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wise.h"

namespace wise {

constexpr int kTile = 32;             // block / tile size B in tokens
constexpr int kMaxT = 16;             // largest tiles_per_item
constexpr int kMaxDenseRows = WISE_DENSE_LIST_MAX_ROWS;  // rows of a call on the dense list
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Wall-clock limit of every mbarrier wait (nanoseconds of %globaltimer); a
// wait that runs out sets WISE_DEVERR_WAIT_TIMEOUT instead of hanging.
constexpr uint64_t kWaitLimitNs = 500ull * 1000 * 1000;

// Per-call constants every kernel needs.
struct KParams {
  int R, Hq, Hkv, G, D, P, max_pages, num_pages, max_blocks, W, T;
  int S_max;         // splits per (row, KV head) at most: ceil(max_blocks / T)
  int cap_tokens;    // min(max_blocks * 32, max_pages * P)
  float scale_log2;  // softmax scale * log2(e): scores are kept in log2 units
  float eta;
  int early;         // partial pass: start before the previous kernel has completed
  int list1;         // partial and finish: the work list is list 1 (built by an
                     // earlier finish), every row sparse
  int build;         // finish: also build list 1 from the mask this call leaves
  int dense_list;    // partial and finish: every block of every row, items derived from
                     // the row lengths (no compaction)
  int inputs_ready;  // partial: the caller's inputs were complete before the previous
                     // kernel began (a dense-list pass may read them before its wait)
};

// Device view of the caller's workspace (offsets from wise_workspace_layout).
struct WsView {
  int32_t* status;
  int32_t* num_items;
  int32_t* queue;      // next schedule slot; zeroed by compaction and again by
                       // the last CTA of every partial launch
  int32_t* queue_done; // CTAs of the running partial launch past the queue
  int4* head_info;     // [R*Hkv]: first item, item count, tile count, 0
  int4* items;         // [max_items] in schedule order: rg, range, bitmap | count << 16, L | flags
  float2* partial_ml;  // [max_items, G], split s of rg in slot rg * S_max + s
  float2* partial_ml_other;  // the other slot set's (compaction marks empty ranges in both)
  float* partial_acc;  // [max_items, G, D]
  float2* tile_stats;  // [R*Hq, max_blocks]
  int32_t* tickets;    // [R*Hkv]: items of the pair completed in the running partial
                       // pass (zeroed by compaction and by the pair's finisher)
  int32_t max_items;
  // List 1: the work list of a following all-sparse call, written by a finish
  // (its items bucketed by tile count, bucket n-1 at items_1 + (n-1) * max_items).
  int32_t* l1_counter;  // [kMaxT]: items of list 1 with n tiles at [n-1]
  int4* head_info_1;    // [R*Hkv]: as head_info, for list 1
  int4* items_1;        // [kMaxT * max_items]
};

__device__ __forceinline__ int clamp_len(int L, int cap) { return L < 0 ? 0 : (L > cap ? cap : L); }

// Where each row's support mask lives [WISE PR, "What changes", wise.py
// bullet: per-request slots hold a [slot, layer, head, block] bitmask]: the W
// words of (row r, KV head g) are at words + slot(r) * slot_stride + g * W,
// with slot(r) = row_slot[r], or r itself when row_slot is null.  A row whose
// slot is negative (or >= num_slots when num_slots > 0) has no mask.
struct MaskView {
  uint32_t* words;          // slot 0's mask at the call's layer; null: no mask at all
  const int32_t* row_slot;  // [R] or null
  long long slot_stride;    // words from one slot's mask to the next
  int num_slots;            // 0: not checked
};

__device__ __forceinline__ int mask_slot(const MaskView& m, int r) {
  if (!m.words) return -1;
  if (!m.row_slot) return r;
  const int s = m.row_slot[r];
  return (s < 0 || (m.num_slots > 0 && s >= m.num_slots)) ? -1 : s;
}

__device__ __forceinline__ uint32_t* mask_of(const MaskView& m, int slot, int g, int W) {
  return slot < 0 ? nullptr : m.words + (long long)slot * m.slot_stride + (long long)g * W;
}

// Work item record: x = row * Hkv + KV head, y = block range s | partial slot
// k << 16 (the item writes its split to slot rg * S_max + k), z = tile bitmap
// over the range | tile count << 16, w = row length (bits 0-23) | mode flags.
constexpr int kItemSparse = 1 << 24;
constexpr int kItemDiscover = 1 << 25;
constexpr int kItemLenMask = (1 << 24) - 1;

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ----------------------------------------------------------------------- TMA
// 3-D tiled bulk-tensor load global -> shared, completing on an mbarrier.
// Coordinates are innermost first: (element within the row, KV head, token).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ math
// 2^x via the SFU instruction (ex2.approx.ftz: ~2 ulp, 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ void flag_error(int32_t* status, int bit) { atomicOr(status, bit); }

// Programmatic dependent launch: wait until the previous kernel in the stream
// has completed and its writes are visible (a no-op when the kernel was not
// launched as a programmatic dependent).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel in the stream start launching (its CTAs then wait in
// grid_dependency_wait until this grid has completed).
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- clusters
// Rank of this CTA in its thread-block cluster, the cluster barrier (every
// thread of every CTA arrives; release/acquire at cluster scope), and a load
// from another CTA's shared memory (distributed shared memory).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// An int in CTA `rank`'s shared memory at the address of `p` in this CTA's.
__device__ __forceinline__ int load_peer(const int* p, uint32_t rank) {
  uint32_t remote;
  int v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

// Spreads L2 prefetches of the first `bytes` (at most 4 MiB) of a buffer over
// every thread of the grid, one 128-byte line each.
__device__ __forceinline__ void prefetch_l2(const void* base, size_t bytes) {
  constexpr size_t kCap = size_t(4) << 20;
  if (bytes > kCap) bytes = kCap;
  const size_t lines = (bytes + 127) / 128;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < lines; i += stride)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(base) + i * 128));
}

// Element-type traits: how a lane loads its DPL = D/32 consecutive elements of
// one K or V row from shared memory and widens them to float.
template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
  static constexpr CUtensorMapDataType kMapType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
  template <int DPL>
  static __device__ __forceinline__ void load(const uint8_t* row, int lane, float (&x)[DPL]) {
    if constexpr (DPL == 4) {
      uint2 w = *reinterpret_cast<const uint2*>(row + lane * 8);
      x[0] = lo(w.x); x[1] = hi(w.x); x[2] = lo(w.y); x[3] = hi(w.y);
    } else {
      uint32_t w = *reinterpret_cast<const uint32_t*>(row + lane * 4);
      x[0] = lo(w); x[1] = hi(w);
    }
  }
  template <int DPL>
  static __device__ __forceinline__ void load_global(const __nv_bfloat16* p, float (&x)[DPL]) {
#pragma unroll
    for (int i = 0; i < DPL; ++i) x[i] = __bfloat162float(p[i]);
  }
  template <int DPL>
  static __device__ __forceinline__ void store_global(__nv_bfloat16* p, const float (&x)[DPL]) {
#pragma unroll
    for (int i = 0; i < DPL; i += 2)
      *reinterpret_cast<__nv_bfloat162*>(p + i) = __floats2bfloat162_rn(x[i], x[i + 1]);
  }
};

template <>
struct Elem<float> {
  static constexpr CUtensorMapDataType kMapType = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  template <int DPL>
  static __device__ __forceinline__ void load(const uint8_t* row, int lane, float (&x)[DPL]) {
    if constexpr (DPL == 4) {
      float4 v = *reinterpret_cast<const float4*>(row + lane * 16);
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
      float2 v = *reinterpret_cast<const float2*>(row + lane * 8);
      x[0] = v.x; x[1] = v.y;
    }
  }
  template <int DPL>
  static __device__ __forceinline__ void load_global(const float* p, float (&x)[DPL]) {
#pragma unroll
    for (int i = 0; i < DPL; ++i) x[i] = p[i];
  }
  template <int DPL>
  static __device__ __forceinline__ void store_global(float* p, const float (&x)[DPL]) {
#pragma unroll
    for (int i = 0; i < DPL; ++i) p[i] = x[i];
  }
};

}  // namespace wise
