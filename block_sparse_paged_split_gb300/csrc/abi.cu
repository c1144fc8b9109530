// The extern "C" entry points of libwise.so (declared in include/wise.h):
// host-side argument checks, workspace layout, TMA tensor-map construction
// (cached), and launch sequencing.  No entry point allocates device memory or
// synchronises a stream.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "list1.cuh"

namespace wise {
namespace {

thread_local char g_last_error[320] = "";

wise_status fail(wise_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

wise_status cuda_fail(cudaError_t e, const char* what) {
  return fail(WISE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

wise_status check_shape(const wise_shape* s) {
  if (!s) return fail(WISE_ERR_INVALID_ARG, "shape is NULL");
  if (s->num_rows < 0) return fail(WISE_ERR_INVALID_ARG, "num_rows < 0");
  if (s->num_q_heads < 1 || s->num_kv_heads < 1)
    return fail(WISE_ERR_INVALID_ARG, "head counts must be >= 1");
  if (s->num_q_heads % s->num_kv_heads)
    return fail(WISE_ERR_INVALID_ARG, "num_q_heads %% num_kv_heads != 0");
  const int G = s->num_q_heads / s->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(WISE_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", G);
  if (s->head_dim != 64 && s->head_dim != 128)
    return fail(WISE_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", s->head_dim);
  if (s->page_size != 16 && s->page_size != 32)
    return fail(WISE_ERR_UNSUPPORTED, "page_size must be 16 or 32 (got %d)", s->page_size);
  if (s->tile_tokens != kTile)
    return fail(WISE_ERR_UNSUPPORTED, "tile_tokens must be 32 (got %d)", s->tile_tokens);
  if (s->max_pages_per_row < 1 || s->num_pages < 1)
    return fail(WISE_ERR_INVALID_ARG, "max_pages_per_row and num_pages must be >= 1");
  if ((int64_t)s->num_pages * s->page_size > INT32_MAX / 2)
    return fail(WISE_ERR_UNSUPPORTED, "num_pages * page_size too large");
  if (s->max_blocks < 1 || s->max_blocks > WISE_MAX_BLOCKS)
    return fail(WISE_ERR_UNSUPPORTED, "max_blocks must be in [1, %d] (got %d)", WISE_MAX_BLOCKS,
                s->max_blocks);
  if (s->tiles_per_item < 0 || s->tiles_per_item > 16 ||
      (s->tiles_per_item & (s->tiles_per_item - 1)) != 0)
    return fail(WISE_ERR_INVALID_ARG, "tiles_per_item must be 0, 1, 2, 4, 8 or 16");
  if (s->dtype != WISE_DTYPE_BF16 && s->dtype != WISE_DTYPE_F32)
    return fail(WISE_ERR_INVALID_ARG, "unknown dtype %d", s->dtype);
  if (!std::isfinite(s->scale) || s->scale < 0.f)
    return fail(WISE_ERR_INVALID_ARG, "scale must be finite and >= 0");
  if (!std::isfinite(s->eta) || !(s->eta > 0.f))
    return fail(WISE_ERR_INVALID_ARG, "eta must be finite and > 0");
  const int64_t heads = (int64_t)s->num_rows * s->num_q_heads;
  if (heads * s->max_blocks > INT32_MAX / 2 || heads * s->head_dim > INT32_MAX / 2)
    return fail(WISE_ERR_UNSUPPORTED, "batch too large");
  return WISE_OK;
}

KParams make_params(const wise_shape* s) {
  KParams kp;
  kp.R = s->num_rows;
  kp.Hq = s->num_q_heads;
  kp.Hkv = s->num_kv_heads;
  kp.G = s->num_q_heads / s->num_kv_heads;
  kp.D = s->head_dim;
  kp.P = s->page_size;
  kp.max_pages = s->max_pages_per_row;
  kp.num_pages = s->num_pages;
  kp.max_blocks = s->max_blocks;
  kp.W = (s->max_blocks + 31) / 32;
  // Default split: 8 tiles; 16 when rows can exceed 64 blocks and the batch
  // still gives ~4 items of 16 tiles per consumer of a GB300 (fewer claims
  // and split slots: measured faster at 4K-32K tokens over 8-64 rows; with
  // fewer items the longer ones leave consumers idle at the end).
  if (s->tiles_per_item) {
    kp.T = s->tiles_per_item;
  } else {
    const int64_t items16 = (int64_t)s->num_rows * s->num_kv_heads * ((s->max_blocks + 15) / 16);
    kp.T = (s->max_blocks > 64 && items16 >= 4096) ? 16 : 8;
  }
  kp.S_max = (s->max_blocks + kp.T - 1) / kp.T;
  const int64_t cap_a = (int64_t)s->max_blocks * kTile;
  const int64_t cap_b = (int64_t)s->max_pages_per_row * s->page_size;
  kp.cap_tokens = (int)(cap_a < cap_b ? cap_a : cap_b);
  const float scale = s->scale > 0.f ? s->scale : 1.f / std::sqrt((float)s->head_dim);
  kp.scale_log2 = scale * kLog2e;
  kp.eta = s->eta;
  kp.early = 0;
  kp.list1 = 0;
  kp.build = 0;
  kp.dense_list = 0;
  kp.inputs_ready = 0;
  return kp;
}

void compute_layout(const wise_shape* s, wise_layout* l) {
  const KParams kp = make_params(s);
  const size_t pairs = (size_t)kp.R * kp.Hkv;
  const size_t max_items = pairs * (size_t)((kp.max_blocks + kp.T - 1) / kp.T);
  size_t off = 0;
  l->status_word = 0;
  l->num_items = 4;
  l->queue = 8;
  off = 256;
  l->head_info = off;   off = up256(off + pairs * sizeof(int4));
  l->items = off;       off = up256(off + max_items * sizeof(int4));
  l->partial_ml = off;  off = up256(off + max_items * kp.G * sizeof(float2));
  l->partial_acc = off; off = up256(off + max_items * kp.G * kp.D * sizeof(float));
  l->tile_stats = off;  off = up256(off + (size_t)kp.R * kp.Hq * kp.max_blocks * sizeof(float2));
  l->tickets = off;     off = up256(off + pairs * sizeof(int32_t));
  l->partial_ml_1 = off;  off = up256(off + max_items * kp.G * sizeof(float2));
  l->partial_acc_1 = off; off = up256(off + max_items * kp.G * kp.D * sizeof(float));
  l->tile_stats_1 = off;  off = up256(off + (size_t)kp.R * kp.Hq * kp.max_blocks * sizeof(float2));
  l->head_info_1 = off;   off = up256(off + pairs * sizeof(int4));
  l->items_1 = off;       off = up256(off + (size_t)kp.T * max_items * sizeof(int4));
  l->list1 = 128;
  l->max_items = max_items;
  l->total_bytes = off;
}

// slot_set: which of the two sets of split results and tile statistics the
// view's partial_ml / partial_acc / tile_stats point at.
wise_status make_view(const wise_shape* s, void* ws, size_t ws_bytes, WsView* v, int slot_set = 0) {
  wise_layout l;
  compute_layout(s, &l);
  if (!ws) return fail(WISE_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(WISE_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < l.total_bytes)
    return fail(WISE_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, l.total_bytes);
  uint8_t* b = static_cast<uint8_t*>(ws);
  v->status = reinterpret_cast<int32_t*>(b + l.status_word);
  v->num_items = reinterpret_cast<int32_t*>(b + l.num_items);
  v->queue = reinterpret_cast<int32_t*>(b + l.queue);
  v->queue_done = reinterpret_cast<int32_t*>(b + l.queue + 4);
  v->head_info = reinterpret_cast<int4*>(b + l.head_info);
  v->items = reinterpret_cast<int4*>(b + l.items);
  v->partial_ml = reinterpret_cast<float2*>(b + (slot_set ? l.partial_ml_1 : l.partial_ml));
  v->partial_acc = reinterpret_cast<float*>(b + (slot_set ? l.partial_acc_1 : l.partial_acc));
  v->tile_stats = reinterpret_cast<float2*>(b + (slot_set ? l.tile_stats_1 : l.tile_stats));
  v->partial_ml_other = reinterpret_cast<float2*>(b + (slot_set ? l.partial_ml : l.partial_ml_1));
  v->tickets = reinterpret_cast<int32_t*>(b + l.tickets);
  v->max_items = (int32_t)l.max_items;
  v->l1_counter = reinterpret_cast<int32_t*>(b + l.list1);
  v->head_info_1 = reinterpret_cast<int4*>(b + l.head_info_1);
  v->items_1 = reinterpret_cast<int4*>(b + l.items_1);
  return WISE_OK;
}

wise_status mask_view(const wise_shape* s, const wise_mask* m, MaskView* v) {
  if (!m) return fail(WISE_ERR_INVALID_ARG, "mask descriptor is NULL");
  const int64_t head_words = (int64_t)s->num_kv_heads * ((s->max_blocks + 31) / 32);
  if (m->words && !aligned(m->words, 4)) return fail(WISE_ERR_INVALID_ARG, "mask words misaligned");
  if (m->row_slot && !aligned(m->row_slot, 4))
    return fail(WISE_ERR_INVALID_ARG, "row_slot misaligned");
  if (m->num_slots < 0) return fail(WISE_ERR_INVALID_ARG, "num_slots < 0");
  if (m->slot_stride < 0 || (m->slot_stride != 0 && m->slot_stride < head_words))
    return fail(WISE_ERR_INVALID_ARG, "slot_stride must be 0 or at least num_kv_heads * W = %lld",
                (long long)head_words);
  *v = MaskView{m->words, m->row_slot, (long long)(m->slot_stride ? m->slot_stride : head_words),
                m->num_slots};
  return WISE_OK;
}

// ------------------------------------------------------------ tensor maps
struct MapKey {
  const void* ptr;
  int device, num_pages, page_size, kv_heads, head_dim, dtype, swizzled;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && device == o.device && num_pages == o.num_pages &&
           page_size == o.page_size && kv_heads == o.kv_heads && head_dim == o.head_dim &&
           dtype == o.dtype && swizzled == o.swizzled;
  }
};

// The tensor-core path (bf16 with grouped query heads) loads half rows of 64
// elements with the 128-byte shared-memory swizzle; the FMA path loads whole
// rows unswizzled.
bool uses_tensor_cores(const wise_shape* s) {
  return s->dtype == WISE_DTYPE_BF16 && s->num_q_heads > s->num_kv_heads;
}

constexpr int kMapCache = 32;
std::mutex g_map_mu;
MapKey g_map_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_used = 0, g_map_next = 0;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

wise_status tensor_map(const wise_shape* s, const void* base, CUtensorMap* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const int swizzled = uses_tensor_cores(s) ? 1 : 0;
  const MapKey key{base, dev, s->num_pages, s->page_size, s->num_kv_heads, s->head_dim, s->dtype,
                   swizzled};
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (int i = 0; i < g_map_used; ++i)
    if (g_map_keys[i] == key) {
      *out = g_maps[i];
      return WISE_OK;
    }
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return fail(WISE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const size_t es = s->dtype == WISE_DTYPE_BF16 ? 2 : 4;
  // View of a pool as [tokens = num_pages * page_size][KV head][element];
  // one box is one page of one KV head.
  const cuuint64_t dims[3] = {(cuuint64_t)s->head_dim, (cuuint64_t)s->num_kv_heads,
                              (cuuint64_t)s->num_pages * s->page_size};
  const cuuint64_t strides[2] = {(cuuint64_t)s->head_dim * es,
                                 (cuuint64_t)s->num_kv_heads * s->head_dim * es};
  const cuuint32_t box[3] = {(cuuint32_t)(swizzled ? 64 : s->head_dim), 1u,
                             (cuuint32_t)s->page_size};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUtensorMap m;
  CUresult r = g_encode(&m,
                        s->dtype == WISE_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzled ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WISE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  const int slot = g_map_used < kMapCache ? g_map_used++ : (g_map_next++ % kMapCache);
  g_map_keys[slot] = key;
  g_maps[slot] = m;
  *out = m;
  return WISE_OK;
}

}  // namespace

wise_status record_error(wise_status status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

// ---------------------------------------------------------------- devices
int sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

}  // namespace wise

using namespace wise;

extern "C" {

const char* wise_status_string(wise_status s) {
  switch (s) {
    case WISE_OK: return "WISE_OK";
    case WISE_ERR_INVALID_ARG: return "WISE_ERR_INVALID_ARG";
    case WISE_ERR_UNSUPPORTED: return "WISE_ERR_UNSUPPORTED";
    case WISE_ERR_WORKSPACE: return "WISE_ERR_WORKSPACE";
    case WISE_ERR_CUDA: return "WISE_ERR_CUDA";
  }
  return "WISE_ERR_UNKNOWN";
}

const char* wise_last_error(void) { return g_last_error; }

wise_status wise_workspace_bytes(const wise_shape* shape, size_t* bytes) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (!bytes) return fail(WISE_ERR_INVALID_ARG, "bytes is NULL");
  wise_layout l;
  compute_layout(shape, &l);
  *bytes = l.total_bytes;
  return WISE_OK;
}

wise_status wise_workspace_reset(const wise_shape* shape, void* workspace, size_t workspace_bytes,
                                 wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  WsView ws;
  if ((st = make_view(shape, workspace, workspace_bytes, &ws)) != WISE_OK) return st;
  cudaError_t e = cudaMemsetAsync(workspace, 0, 256, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : cuda_fail(e, "workspace header reset");
}

wise_status wise_workspace_layout(const wise_shape* shape, wise_layout* layout) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (!layout) return fail(WISE_ERR_INVALID_ARG, "layout is NULL");
  compute_layout(shape, layout);
  return WISE_OK;
}

wise_status wise_compact_tiles_m(const wise_shape* shape, const int8_t* modes,
                                 const int32_t* seq_lens, const wise_mask* mask,
                                 void* workspace, size_t workspace_bytes, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  WsView ws;
  if ((st = make_view(shape, workspace, workspace_bytes, &ws)) != WISE_OK) return st;
  if (shape->num_rows > 0 && (!modes || !seq_lens))
    return fail(WISE_ERR_INVALID_ARG, "modes and seq_lens must not be NULL");
  MaskView mv;
  if ((st = mask_view(shape, mask, &mv)) != WISE_OK) return st;
  cudaError_t e = launch_compact(make_params(shape), modes, seq_lens, mv, ws,
                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : cuda_fail(e, "compact launch");
}

wise_status wise_compact_tiles(const wise_shape* shape, const int8_t* modes,
                               const int32_t* seq_lens, const uint32_t* support,
                               void* workspace, size_t workspace_bytes, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (support && !aligned(support, 4)) return fail(WISE_ERR_INVALID_ARG, "support misaligned");
  const wise_mask m{const_cast<uint32_t*>(support), nullptr, 0, 0};
  return wise_compact_tiles_m(shape, modes, seq_lens, &m, workspace, workspace_bytes, stream);
}

wise_status wise_build_list_m(const wise_shape* shape, const int8_t* modes,
                              const int32_t* seq_lens, const wise_mask* mask, void* workspace,
                              size_t workspace_bytes, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  WsView ws;
  if ((st = make_view(shape, workspace, workspace_bytes, &ws)) != WISE_OK) return st;
  if (shape->num_rows > 0 && !seq_lens) return fail(WISE_ERR_INVALID_ARG, "seq_lens is NULL");
  MaskView mv;
  if ((st = mask_view(shape, mask, &mv)) != WISE_OK) return st;
  if (!modes && !mv.words)
    return fail(WISE_ERR_INVALID_ARG, "an all-sparse list is built from the support mask");
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // A new call: status word and queue counters back to 0, list 1's bucket
  // counters too (the build appends to them).
  cudaError_t e = cudaMemsetAsync(workspace, 0, 256, s);
  if (e != cudaSuccess) return cuda_fail(e, "workspace header reset");
  e = launch_build_list(make_params(shape), modes, seq_lens, mv, ws, s);
  return e == cudaSuccess ? WISE_OK : cuda_fail(e, "list build launch");
}

wise_status wise_build_list(const wise_shape* shape, const int8_t* modes, const int32_t* seq_lens,
                            const uint32_t* support, void* workspace, size_t workspace_bytes,
                            wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (shape->num_rows > 0 && !modes) return fail(WISE_ERR_INVALID_ARG, "modes is NULL");
  if (support && !aligned(support, 4)) return fail(WISE_ERR_INVALID_ARG, "support misaligned");
  const wise_mask m{const_cast<uint32_t*>(support), nullptr, 0, 0};
  return wise_build_list_m(shape, modes, seq_lens, &m, workspace, workspace_bytes, stream);
}

wise_status wise_build_sparse_list_m(const wise_shape* shape, const int32_t* seq_lens,
                                     const wise_mask* mask, void* workspace,
                                     size_t workspace_bytes, wise_stream_t stream) {
  return wise_build_list_m(shape, nullptr, seq_lens, mask, workspace, workspace_bytes, stream);
}

wise_status wise_build_sparse_list(const wise_shape* shape, const int32_t* seq_lens,
                                   const uint32_t* support, void* workspace,
                                   size_t workspace_bytes, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (support && !aligned(support, 4)) return fail(WISE_ERR_INVALID_ARG, "support misaligned");
  const wise_mask m{const_cast<uint32_t*>(support), nullptr, 0, 0};
  return wise_build_list_m(shape, nullptr, seq_lens, &m, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// The partial pass, with the finish folded in when `fa.out` is set.
wise_status partial_pass(const wise_shape* shape, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* page_table, const int32_t* seq_lens,
                         const int8_t* modes, void* workspace, size_t workspace_bytes,
                         const FoldArgs& fa, uint32_t flags, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (flags & ~(uint32_t)(WISE_FLAG_SLOT_SET_1 | WISE_FLAG_EARLY_START | WISE_FLAG_SPARSE_LIST |
                          WISE_FLAG_DENSE_LIST | WISE_FLAG_INPUTS_READY | WISE_FLAG_LIST_MODES))
    return fail(WISE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  if ((flags & WISE_FLAG_LIST_MODES) && !(flags & WISE_FLAG_SPARSE_LIST))
    return fail(WISE_ERR_INVALID_ARG, "WISE_FLAG_LIST_MODES goes with WISE_FLAG_SPARSE_LIST");
  if ((flags & (WISE_FLAG_SPARSE_LIST | WISE_FLAG_DENSE_LIST)) && fa.out)
    return fail(WISE_ERR_INVALID_ARG, "the folded finish takes neither list flag");
  if ((flags & WISE_FLAG_SPARSE_LIST) && (flags & WISE_FLAG_DENSE_LIST))
    return fail(WISE_ERR_INVALID_ARG, "WISE_FLAG_SPARSE_LIST and WISE_FLAG_DENSE_LIST exclude each other");
  if ((flags & WISE_FLAG_DENSE_LIST) && shape->num_rows > WISE_DENSE_LIST_MAX_ROWS)
    return fail(WISE_ERR_UNSUPPORTED, "WISE_FLAG_DENSE_LIST takes at most %d rows (got %d)",
                WISE_DENSE_LIST_MAX_ROWS, shape->num_rows);
  if ((flags & (WISE_FLAG_DENSE_LIST | WISE_FLAG_SPARSE_LIST)) && (flags & WISE_FLAG_EARLY_START) &&
      !(flags & WISE_FLAG_INPUTS_READY))
    return fail(WISE_ERR_INVALID_ARG,
                "an early start on the dense list or list 1 needs WISE_FLAG_INPUTS_READY");
  WsView ws;
  if ((st = make_view(shape, workspace, workspace_bytes, &ws, (flags & WISE_FLAG_SLOT_SET_1) ? 1 : 0)) != WISE_OK)
    return st;
  if (shape->num_rows == 0) return WISE_OK;
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens ||
      (!modes && !(flags & WISE_FLAG_SPARSE_LIST)))
    return fail(WISE_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(WISE_ERR_INVALID_ARG, "q, k_cache and v_cache must be 16-byte aligned");
  CUtensorMap tmK, tmV;
  if ((st = tensor_map(shape, k_cache, &tmK)) != WISE_OK) return st;
  if ((st = tensor_map(shape, v_cache, &tmV)) != WISE_OK) return st;
  KParams kp = make_params(shape);
  kp.early = (flags & WISE_FLAG_EARLY_START) ? 1 : 0;
  kp.list1 = (flags & WISE_FLAG_SPARSE_LIST) ? 1 : 0;
  kp.dense_list = (flags & WISE_FLAG_DENSE_LIST) ? 1 : 0;
  kp.inputs_ready = (flags & WISE_FLAG_INPUTS_READY) ? 1 : 0;
  cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = shape->dtype == WISE_DTYPE_BF16
                      ? launch_partial_bf16(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, fa, st_)
                      : launch_partial_f32(kp, tmK, tmV, q, page_table, seq_lens, modes, ws, fa, st_);
  return e == cudaSuccess ? WISE_OK : cuda_fail(e, "partial launch");
}

}  // namespace

extern "C" {

wise_status wise_decode_partial(const wise_shape* shape, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* page_table,
                                const int32_t* seq_lens, const int8_t* modes, void* workspace,
                                size_t workspace_bytes, wise_stream_t stream) {
  return partial_pass(shape, q, k_cache, v_cache, page_table, seq_lens, modes, workspace,
                      workspace_bytes, FoldArgs{nullptr, nullptr, nullptr}, 0u, stream);
}

wise_status wise_decode_partial_ex(const wise_shape* shape, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* page_table,
                                   const int32_t* seq_lens, const int8_t* modes, void* workspace,
                                   size_t workspace_bytes, uint32_t flags, wise_stream_t stream) {
  return partial_pass(shape, q, k_cache, v_cache, page_table, seq_lens, modes, workspace,
                      workspace_bytes, FoldArgs{nullptr, nullptr, nullptr}, flags, stream);
}

wise_status wise_decode_partial_finish(const wise_shape* shape, const void* q,
                                       const void* k_cache, const void* v_cache,
                                       const int32_t* page_table, const int32_t* seq_lens,
                                       const int8_t* modes, void* workspace,
                                       size_t workspace_bytes, uint32_t* support, void* out,
                                       float* lse, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (!can_fold_finish(make_params(shape))) {
    // Long rows: the two passes as separate launches.
    st = wise_decode_partial(shape, q, k_cache, v_cache, page_table, seq_lens, modes, workspace,
                             workspace_bytes, stream);
    if (st != WISE_OK) return st;
    return wise_decode_finish(shape, modes, seq_lens, workspace, workspace_bytes, support, out,
                              lse, stream);
  }
  if (shape->num_rows > 0 && (!out || !lse))
    return fail(WISE_ERR_INVALID_ARG, "a required pointer is NULL");
  if (shape->num_rows > 0 &&
      (!aligned(out, 16) || !aligned(lse, 4) || (support && !aligned(support, 4))))
    return fail(WISE_ERR_INVALID_ARG, "out must be 16-byte aligned, lse and support 4-byte");
  return partial_pass(shape, q, k_cache, v_cache, page_table, seq_lens, modes, workspace,
                      workspace_bytes, FoldArgs{support, out, lse}, 0u, stream);
}

wise_status wise_decode_finish_m(const wise_shape* shape, const int8_t* modes,
                                 const int32_t* seq_lens, void* workspace,
                                 size_t workspace_bytes, uint32_t flags, const wise_mask* mask,
                                 void* out, float* lse, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (flags & ~(uint32_t)(WISE_FLAG_SLOT_SET_1 | WISE_FLAG_BUILD_SPARSE_LIST | WISE_FLAG_SPARSE_LIST |
                          WISE_FLAG_DENSE_LIST | WISE_FLAG_LIST_MODES))
    return fail(WISE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  if ((flags & WISE_FLAG_LIST_MODES) && !(flags & WISE_FLAG_SPARSE_LIST))
    return fail(WISE_ERR_INVALID_ARG, "WISE_FLAG_LIST_MODES goes with WISE_FLAG_SPARSE_LIST");
  if ((flags & WISE_FLAG_SPARSE_LIST) && (flags & WISE_FLAG_DENSE_LIST))
    return fail(WISE_ERR_INVALID_ARG, "WISE_FLAG_SPARSE_LIST and WISE_FLAG_DENSE_LIST exclude each other");
  if ((flags & WISE_FLAG_DENSE_LIST) && shape->num_rows > WISE_DENSE_LIST_MAX_ROWS)
    return fail(WISE_ERR_UNSUPPORTED, "WISE_FLAG_DENSE_LIST takes at most %d rows (got %d)",
                WISE_DENSE_LIST_MAX_ROWS, shape->num_rows);
  WsView ws;
  if ((st = make_view(shape, workspace, workspace_bytes, &ws, (flags & WISE_FLAG_SLOT_SET_1) ? 1 : 0)) != WISE_OK)
    return st;
  if (shape->num_rows == 0) return WISE_OK;
  const bool list_modes = (flags & WISE_FLAG_LIST_MODES) != 0;
  if ((!modes && (list_modes || !(flags & WISE_FLAG_SPARSE_LIST))) || !seq_lens || !out || !lse)
    return fail(WISE_ERR_INVALID_ARG, "a required pointer is NULL");
  MaskView mv;
  if ((st = mask_view(shape, mask, &mv)) != WISE_OK) return st;
  if ((flags & WISE_FLAG_BUILD_SPARSE_LIST) && !mv.words)
    return fail(WISE_ERR_INVALID_ARG, "WISE_FLAG_BUILD_SPARSE_LIST needs the support mask");
  if ((flags & WISE_FLAG_BUILD_SPARSE_LIST) && (flags & WISE_FLAG_SPARSE_LIST))
    return fail(WISE_ERR_INVALID_ARG,
                "a call on list 1 leaves the mask as it is; it cannot build list 1 again");
  if (!aligned(out, 16) || !aligned(lse, 4))
    return fail(WISE_ERR_INVALID_ARG, "out must be 16-byte aligned, lse 4-byte");
  KParams kp = make_params(shape);
  kp.build = (flags & WISE_FLAG_BUILD_SPARSE_LIST) ? 1 : 0;
  kp.list1 = (flags & WISE_FLAG_SPARSE_LIST) ? 1 : 0;
  kp.dense_list = (flags & WISE_FLAG_DENSE_LIST) ? 1 : 0;
  // On list 1 the finish sees the modes only when the list was built for
  // them; without them every row is sparse.
  const int8_t* kmodes = (kp.list1 && !list_modes) ? nullptr : modes;
  cudaError_t e = launch_finish(shape->dtype, kp, kmodes, seq_lens, ws, mv, out, lse,
                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : cuda_fail(e, "finish launch");
}

wise_status wise_decode_finish_ex(const wise_shape* shape, const int8_t* modes,
                                  const int32_t* seq_lens, void* workspace,
                                  size_t workspace_bytes, uint32_t flags, uint32_t* support,
                                  void* out, float* lse, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (support && !aligned(support, 4))
    return fail(WISE_ERR_INVALID_ARG, "out must be 16-byte aligned, lse and support 4-byte");
  const wise_mask m{support, nullptr, 0, 0};
  return wise_decode_finish_m(shape, modes, seq_lens, workspace, workspace_bytes, flags, &m, out,
                              lse, stream);
}

wise_status wise_decode_finish(const wise_shape* shape, const int8_t* modes,
                               const int32_t* seq_lens, void* workspace, size_t workspace_bytes,
                               uint32_t* support, void* out, float* lse, wise_stream_t stream) {
  return wise_decode_finish_ex(shape, modes, seq_lens, workspace, workspace_bytes, 0u, support,
                               out, lse, stream);
}

wise_status wise_decode_m(const wise_shape* shape, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* page_table, const int32_t* seq_lens,
                          const int8_t* modes, const wise_mask* mask, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, wise_stream_t stream) {
  wise_status st = wise_compact_tiles_m(shape, modes, seq_lens, mask, workspace, workspace_bytes,
                                        stream);
  if (st != WISE_OK) return st;
  st = wise_decode_partial(shape, q, k_cache, v_cache, page_table, seq_lens, modes, workspace,
                           workspace_bytes, stream);
  if (st != WISE_OK) return st;
  return wise_decode_finish_m(shape, modes, seq_lens, workspace, workspace_bytes, 0u, mask, out,
                              lse, stream);
}

wise_status wise_decode(const wise_shape* shape, const void* q, const void* k_cache,
                        const void* v_cache, const int32_t* page_table, const int32_t* seq_lens,
                        const int8_t* modes, uint32_t* support, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (support && !aligned(support, 4)) return fail(WISE_ERR_INVALID_ARG, "support misaligned");
  const wise_mask m{support, nullptr, 0, 0};
  return wise_decode_m(shape, q, k_cache, v_cache, page_table, seq_lens, modes, &m, out, lse,
                       workspace, workspace_bytes, stream);
}

wise_status wise_support_union(uint32_t* dst, const uint32_t* src, int64_t n_words,
                               wise_stream_t stream) {
  if (n_words < 0) return fail(WISE_ERR_INVALID_ARG, "n_words < 0");
  if (n_words == 0) return WISE_OK;
  if (!dst || !src) return fail(WISE_ERR_INVALID_ARG, "dst and src must not be NULL");
  if (!aligned(dst, 4) || !aligned(src, 4)) return fail(WISE_ERR_INVALID_ARG, "misaligned mask");
  cudaError_t e = launch_union(dst, src, n_words, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : cuda_fail(e, "union launch");
}

wise_status wise_block_mass(const wise_shape* shape, const void* q, const void* k_cache,
                            const int32_t* page_table, const int32_t* seq_lens,
                            const int8_t* modes, const float* lse, void* workspace,
                            size_t workspace_bytes, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  WsView ws;
  if ((st = make_view(shape, workspace, workspace_bytes, &ws)) != WISE_OK) return st;
  if (shape->num_rows == 0) return WISE_OK;
  if (!q || !k_cache || !page_table || !seq_lens || !modes || !lse)
    return fail(WISE_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(lse, 4))
    return fail(WISE_ERR_INVALID_ARG, "q and k_cache must be 16-byte aligned, lse 4-byte");
  cudaError_t e = launch_block_mass(shape->dtype, make_params(shape), q, k_cache, page_table,
                                    seq_lens, modes, lse, ws, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : cuda_fail(e, "block mass launch");
}

wise_status wise_support_head_union(const wise_shape* shape, uint32_t* support,
                                    wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (shape->num_rows == 0) return WISE_OK;
  if (!support) return fail(WISE_ERR_INVALID_ARG, "support is NULL");
  if (!aligned(support, 4)) return fail(WISE_ERR_INVALID_ARG, "support misaligned");
  cudaError_t e = launch_head_union(make_params(shape), support, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : cuda_fail(e, "head union launch");
}

wise_status wise_validate_m(const wise_shape* shape, const int32_t* page_table,
                            const int32_t* seq_lens, const int8_t* modes, const wise_mask* mask,
                            int32_t* err_word, wise_stream_t stream) {
  wise_status st = check_shape(shape);
  if (st != WISE_OK) return st;
  if (!err_word) return fail(WISE_ERR_INVALID_ARG, "err_word is NULL");
  MaskView mv;
  if ((st = mask_view(shape, mask, &mv)) != WISE_OK) return st;
  if (shape->num_rows == 0) return WISE_OK;
  if (!page_table || !seq_lens || !modes)
    return fail(WISE_ERR_INVALID_ARG, "a required pointer is NULL");
  cudaError_t e = launch_validate(make_params(shape), page_table, seq_lens, modes, mv, err_word,
                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : cuda_fail(e, "validate launch");
}

wise_status wise_validate(const wise_shape* shape, const int32_t* page_table,
                          const int32_t* seq_lens, const int8_t* modes, const uint32_t* support,
                          int32_t* err_word, wise_stream_t stream) {
  const wise_mask m{const_cast<uint32_t*>(support), nullptr, 0, 0};
  return wise_validate_m(shape, page_table, seq_lens, modes, &m, err_word, stream);
}

}  // extern "C"
