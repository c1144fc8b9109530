/*
 * wise.h - C ABI of the WISE working-set paged decode attention library
 * (libwise.so, CUDA kernels for sm_103a).
 *
 * The operation (vllm-rlt pull request "WISE working-set decode", PR #143,
 * sections "Summary" and "What changes"): one decode call attends, for every
 * row of a batch and every query head, over that row's paged K/V cache.  Each
 * row runs in one of three modes:
 *   dense     ordinary paged decode attention over all of the row's tokens;
 *   discover  dense, and it also records every 32-token tile's max and
 *             exp-sum; the finish step turns them into per-block softmax
 *             masses and applies the eta selection (B = 32, eta = 0.95 by
 *             default) into a [row, KV head, block] support bitmask;
 *             DISCOVER overwrites the mask, DISCOVER_UNION ORs the new choice
 *             into it (review comment "[P2] Distinguish discovery density
 *             from reused union density");
 *   sparse    attends only the row's selected tiles, compacted first so the
 *             inner loop has no branch; the softmax is renormalised over the
 *             selected tokens ("Tests": sparse output matches masked
 *             attention).
 * The split-KV structure (a partial pass over work items of about eight
 * tiles, then a finish pass that merges the splits by log-sum-exp) follows
 * the same section: one long dense row must not set the latency of a launch
 * whose other rows are sparse.
 *
 * One call of the path, on one CUDA stream:
 *     wise_compact_tiles -> wise_decode_partial -> wise_decode_finish
 * (wise_decode runs all three); a call may take its work list from
 * wise_build_list (wise_build_sparse_list when every row is sparse) instead
 * of the compaction.  wise_support_union ORs masks kept per depth.
 * Variants from the pages' FlashAttention decode path, built for comparison:
 * wise_support_head_union (head-union masks) and wise_block_mass (block
 * masses from the LSE by a second read of K); wise_decode_partial_finish
 * folds the finish into the partial pass; the _ex calls take a second set of
 * split slots and an early start, so consecutive calls can overlap.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     caller owns every buffer, including the workspace.  The library never
 *     allocates device memory, never synchronises the stream and never
 *     blocks; all work is enqueued on `stream` (NULL = legacy default stream).
 *   - Arguments the host can check (null pointers, alignment, shape limits,
 *     workspace size) are checked before anything is enqueued; on failure the
 *     call returns a status and enqueues nothing.  A failed launch returns
 *     WISE_ERR_CUDA.  wise_last_error() gives a one-line reason for the
 *     calling thread's last non-OK status.
 *   - Device data is never trusted to be in range and never traps: a page id
 *     outside [0, num_pages) reads zeros, a seq_len above the row's capacity
 *     is clamped to it and flagged in the workspace status word; use
 *     wise_validate to check a batch explicitly.
 *
 * Layouts (row-major, no padding):
 *   q, out       [num_rows, num_q_heads, head_dim], dtype of the shape
 *   k_cache,
 *   v_cache      [num_pages, page_size, num_kv_heads, head_dim] (paged, the
 *                token-major layout of FlashAttention's paged KV cache)
 *   page_table   int32 [num_rows, max_pages_per_row]; token j of row r lives
 *                in page page_table[r][j / page_size], slot j % page_size
 *   seq_lens     int32 [num_rows]; 0 marks a padding row
 *   modes        int8  [num_rows], WISE_MODE_*
 *   support      uint32 [num_rows, num_kv_heads, W], W = ceil(max_blocks/32);
 *                block b of a (row, KV head) is bit (b % 32) of word b / 32.
 *                Block b covers tokens [32 b, 32 b + 32) of the row.
 *   lse          float32 [num_rows, num_q_heads]: natural log of the softmax
 *                normaliser sum_j exp(scale * q . k_j) over attended tokens.
 * Query head h reads KV head h / (num_q_heads / num_kv_heads).  For grouped
 * query heads each query head selects blocks with its own eta rule and the
 * KV head's mask is the OR over its group, so sparse rows attend the group's
 * union.  Padding rows (seq_len 0) get out = 0 and lse = -inf and leave the
 * mask untouched; a sparse row whose mask selects nothing gets the same.
 */
#ifndef WISE_H_
#define WISE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st *wise_stream_t;

typedef enum {
  WISE_OK = 0,
  WISE_ERR_INVALID_ARG = 1, /* null pointer, misalignment, bad shape field */
  WISE_ERR_UNSUPPORTED = 2, /* valid but not built (e.g. head_dim 96)      */
  WISE_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small  */
  WISE_ERR_CUDA = 4         /* a CUDA runtime call or launch failed        */
} wise_status;

enum {
  WISE_MODE_DENSE = 0,
  WISE_MODE_DISCOVER = 1,
  WISE_MODE_DISCOVER_UNION = 2,
  WISE_MODE_SPARSE = 3
};

enum { WISE_DTYPE_BF16 = 0, WISE_DTYPE_F32 = 1 };

/* Bits of the workspace status word (set by the kernels, read by the caller
 * from the workspace after the stream has run; see wise_workspace_layout).
 * After WISE_DEVERR_WAIT_TIMEOUT the out, lse and support a call wrote are
 * undefined (some work items were not computed). */
enum {
  WISE_DEVERR_SEQ_LEN_CLAMPED = 1, /* a seq_len exceeded the row's capacity */
  WISE_DEVERR_WAIT_TIMEOUT = 2,    /* a bounded wait gave up (no hang)      */
  WISE_DEVERR_BAD_WORK_LIST = 4    /* the workspace's work list was not one
                                      the library wrote for this shape (a
                                      call out of order); bad items skipped */
};

/* Bits of the word written by wise_validate. */
enum {
  WISE_BAD_MODE = 1,           /* mode outside 0..3                          */
  WISE_BAD_SEQ_LEN = 2,        /* seq_len < 0 or above the row's capacity    */
  WISE_BAD_PAGE = 4,           /* a page id the row uses is outside the pool */
  WISE_EMPTY_SPARSE_SUPPORT = 8, /* a sparse (row, KV head) selects nothing  */
  WISE_BAD_SLOT = 16            /* a row slot below -1 or past num_slots     */
};

/* Largest max_blocks: 4096 blocks of 32 tokens, rows of up to 128K tokens
 * (a (row, KV head) mask of 128 words). */
#define WISE_MAX_BLOCKS 4096

typedef struct {
  int32_t num_rows;          /* R >= 0 (0: every call is a no-op)              */
  int32_t num_q_heads;       /* Hq >= 1                                         */
  int32_t num_kv_heads;      /* Hkv >= 1, Hq % Hkv == 0, Hq/Hkv in {1,2,4,8}    */
  int32_t head_dim;          /* D in {64, 128}                                  */
  int32_t page_size;         /* tokens per page: 16 or 32                       */
  int32_t tile_tokens;       /* block size B; must be 32                        */
  int32_t max_pages_per_row; /* page_table row stride, >= 1                     */
  int32_t num_pages;         /* pages in the K/V pools, >= 1                    */
  int32_t max_blocks;        /* mask capacity per (row, KV head),
                                1..WISE_MAX_BLOCKS; a row's capacity
                                is min(max_blocks * 32,
                                max_pages_per_row * page_size) tokens          */
  int32_t tiles_per_item;    /* blocks per split range T: 1, 2, 4, 8 or 16;
                                0 means 8, or 16 when max_blocks > 64 and
                                num_rows * num_kv_heads * ceil(max_blocks /
                                16) >= 4096.
                                Work item s of a (row, KV head)
                                holds its tiles in blocks [s*T, s*T + T)   */
  int32_t dtype;             /* WISE_DTYPE_* of q, k_cache, v_cache and out     */
  float scale;               /* softmax scale; 0 means 1/sqrt(head_dim)         */
  float eta;                 /* selection threshold, > 0; >= 1 selects all      */
} wise_shape;

/* Where the rows' support masks live, for the _m calls [WISE PR, "What
 * changes", wise.py bullet: the engine keeps a [slot, layer, head, block]
 * support bitmask of per-request slots, freed with the request's
 * allocation].  The W = ceil(max_blocks / 32) words of (row r, KV head g)
 * are at words + slot(r) * slot_stride + g * W, where slot(r) = row_slot[r]
 * (or r when row_slot is NULL).  For a pool [slots, layers, num_kv_heads, W]
 * and layer l: words = pool + l * num_kv_heads * W, slot_stride = layers *
 * num_kv_heads * W, num_slots = slots.  A row whose slot is negative (or
 * >= num_slots when num_slots > 0) has no mask: sparse rows attend nothing
 * (out 0, lse -inf), discover rows select as usual but store nothing, and a
 * list build gives them no item; wise_validate_m flags slots below -1 or
 * past num_slots.  Rows whose slots coincide share one mask: two such rows
 * that discover in the same call race on it. */
typedef struct {
  uint32_t *words;          /* device; 4-byte aligned                            */
  const int32_t *row_slot;  /* device int32 [num_rows], or NULL: slot = row      */
  int64_t slot_stride;      /* uint32 words between slots; 0 means num_kv_heads
                               * W; with row_slot, at least num_kv_heads * W     */
  int32_t num_slots;        /* slots in the pool, >= 0 (0: slots not checked)    */
} wise_mask;

/* Offsets (bytes from the workspace base) of the workspace regions, for
 * callers that inspect intermediate results.  All offsets are 256-aligned. */
typedef struct {
  size_t status_word;   /* int32: WISE_DEVERR_* bits, cleared by compaction   */
  size_t num_items;     /* int32: work items written by compaction            */
  size_t queue;         /* int32 x2: next schedule slot and finished CTAs of
                           the partial pass (both back to 0 after each pass) */
  size_t head_info;     /* int32x4 [R*Hkv]: first partial slot (rg * S),
                           block ranges, tiles, non-empty items                */
  size_t items;         /* int32x4 [max_items], in schedule order (tile count
                           descending): row*Hkv + KV head, block range s,
                           tile bitmap (bit i: block s*T + i) | tile count
                           << 16, sequence length | sparse << 24 |
                           discover << 25                                      */
  size_t partial_ml;    /* float32x2 [max_items, G]: running max (log2 units)
                           and exp-sum per item and query head; range s of
                           (row, KV head) rg lives in slot rg * S + s, with
                           S = ceil(max_blocks / tiles_per_item); an empty
                           range of a sparse row holds (-inf, 0)              */
  size_t partial_acc;   /* float32 [max_items, G, D]: unnormalised outputs     */
  size_t tile_stats;    /* float32x2 [R*Hq, max_blocks]: per tile max (log2
                           units of the scaled score) and exp-sum (discover)  */
  size_t tickets;       /* int32 [R*Hkv]: items of each (row, KV head) the
                           running wise_decode_partial_finish has completed;
                           0 between calls                                    */
  size_t partial_ml_1;  /* slot set 1 (WISE_FLAG_SLOT_SET_1): the same three   */
  size_t partial_acc_1; /* regions again, so a partial pass can write its      */
  size_t tile_stats_1;  /* splits while the previous call's finish reads set 0 */
  size_t max_items;     /* capacity of the item arrays                         */
  size_t total_bytes;   /* = wise_workspace_bytes                              */
  size_t list1;         /* int32 [16]: list 1's items with n tiles at [n - 1]
                           (WISE_FLAG_BUILD_SPARSE_LIST)                      */
  size_t head_info_1;   /* int32x4 [R*Hkv]: head info of list 1 (first slot,
                           slots = items, tiles, items)                       */
  size_t items_1;       /* int32x4 [tiles_per_item * max_items]: list 1's
                           items with n tiles at items_1 + (n - 1) * max_items;
                           slots are compact (item k of a pair writes slot
                           rg * S + k)                                          */
} wise_layout;

/* Bytes of device workspace one call sequence needs for this shape.  Host
 * only; enqueues nothing.  `bytes` is a host pointer. */
wise_status wise_workspace_bytes(const wise_shape *shape, size_t *bytes);

/* Zeroes the workspace header (status word, item count, queue counters,
 * list-1 counters): asynchronously on `stream`, allocating nothing.  A new
 * workspace needs it (or a wise_compact_tiles) before its first call with
 * WISE_FLAG_DENSE_LIST. */
wise_status wise_workspace_reset(const wise_shape *shape, void *workspace,
                                 size_t workspace_bytes, wise_stream_t stream);

/* Region offsets for this shape (host only). `layout` is a host pointer. */
wise_status wise_workspace_layout(const wise_shape *shape,
                                  wise_layout *layout);

/* Compaction [WISE PR, "What changes": sparse rows are compacted first so
 * the loop has no branch; programs cover about eight tiles].  For each
 * (row, KV head) and each range s of T = tiles_per_item blocks: a work item
 * holding the range's tiles (every block below the row's block count for
 * dense and discover rows, the selected ones for sparse rows; no item for an
 * empty range) as a bitmap over the range, written in schedule order (tile
 * count descending).  Reads modes, seq_lens and, for sparse rows, support;
 * writes the workspace (items, head info) and clears its status word.  The
 * workspace must be 256-byte aligned and at least wise_workspace_bytes
 * long. */
wise_status wise_compact_tiles(const wise_shape *shape, const int8_t *modes,
                               const int32_t *seq_lens, const uint32_t *support,
                               void *workspace, size_t workspace_bytes,
                               wise_stream_t stream);

/* The work list of a call in which every row is sparse, built from the mask
 * alone [WISE PR, "What changes": sparse rows are compacted first]: list 1
 * of the workspace, as a finish with WISE_FLAG_BUILD_SPARSE_LIST writes it
 * (per (row, KV head): its k-th block range holding a selected tile is item
 * k, a bitmap of the selected blocks of that range; items bucketed by tile
 * count), for a partial pass and finish with WISE_FLAG_SPARSE_LIST.  Where
 * compaction visits every block range of every row, this reads each (row,
 * KV head)'s W mask words and writes one record per selected range, so the
 * sparse call's cost follows its selection, not its rows' lengths.  Resets
 * the workspace header (status word, counters), then writes list 1 and its
 * head info; padding rows and masks selecting nothing get no item, and a
 * length above the row's capacity is clamped and flagged.  support must not
 * be NULL. */
wise_status wise_build_sparse_list(const wise_shape *shape, const int32_t *seq_lens,
                                   const uint32_t *support, void *workspace,
                                   size_t workspace_bytes, wise_stream_t stream);

/* The work list of a call of any modes, built from the rows' modes, lengths
 * and masks as wise_build_sparse_list builds an all-sparse one: each sparse
 * row's selected ranges, every block range of a dense or discover row (with
 * the discover flag, so the partial pass records tile statistics); padding
 * rows and sparse rows without a selected block get no item.  The call then
 * runs its partial pass and finish with WISE_FLAG_SPARSE_LIST |
 * WISE_FLAG_LIST_MODES and the same modes: a mixed batch, or a batch past
 * WISE_DENSE_LIST_MAX_ROWS, without wise_compact_tiles.  modes must not be
 * NULL; support may be NULL (sparse rows then get no item). */
wise_status wise_build_list(const wise_shape *shape, const int8_t *modes,
                            const int32_t *seq_lens, const uint32_t *support, void *workspace,
                            size_t workspace_bytes, wise_stream_t stream);

/* Split partial pass [WISE PR, "What changes": split-KV paged decode with
 * per-row modes].  For every work item written by wise_compact_tiles and
 * every query head of its KV head: online softmax over the item's tiles,
 * writing the unnormalised output, running max and exp-sum to the
 * workspace; discover and discover-union rows also write each tile's max and
 * exp-sum.  q, k_cache and v_cache must be 16-byte aligned. */
wise_status wise_decode_partial(const wise_shape *shape, const void *q,
                                const void *k_cache, const void *v_cache,
                                const int32_t *page_table, const int32_t *seq_lens,
                                const int8_t *modes, void *workspace,
                                size_t workspace_bytes, wise_stream_t stream);

/* Finish [WISE PR, "What changes": a finish kernel merges the splits and runs
 * the selection for discovery rows].  Merges each (row, query head)'s splits
 * by log-sum-exp into out and lse; for discover rows computes the block
 * masses p_b = exp-sum_b * exp(max_b - lse), orders them by mass descending
 * (ties: lower block index), keeps the shortest prefix whose cumulative mass
 * reaches eta, ORs the selections of the KV head's query-head group and
 * writes (DISCOVER) or ORs (DISCOVER_UNION) it into support, clearing bits at
 * or past the row's block count.  Sparse and dense rows leave support alone.
 * out must be 16-byte aligned; support may be NULL if no row discovers. */
wise_status wise_decode_finish(const wise_shape *shape, const int8_t *modes,
                               const int32_t *seq_lens, void *workspace,
                               size_t workspace_bytes, uint32_t *support,
                               void *out, float *lse, wise_stream_t stream);

/* Flags of the _ex calls. */
enum {
  /* Use the workspace's second set of split results and tile statistics
   * (partial_ml_1, partial_acc_1, tile_stats_1).  A partial pass and the
   * finish that reads it must use the same set. */
  WISE_FLAG_SLOT_SET_1 = 1u,
  /* Partial pass only: start streaming without waiting for the previous
   * kernel in the stream to complete (the launch still completes after it).
   * Legal when that kernel writes nothing this call reads and reads nothing
   * it writes, and the compaction this call uses completed before that
   * kernel began: for instance the finish of the previous depth, on the other
   * slot set, when both calls share one compaction, or -- with
   * WISE_FLAG_INPUTS_READY, which a pass on the dense list or on list 1
   * then needs -- a call on the dense list or on a list built before that
   * finish.  The queue claims still wait for the previous kernel.  An
   * early dense-list pass leaves the status word as it is. */
  WISE_FLAG_EARLY_START = 2u,
  /* Finish only: also write the work list of a following call in which every
   * row is sparse on the mask as this call leaves it ("list 1" of the
   * workspace: head info, items bucketed by tile count, and their schedule
   * positions), so that call needs no wise_compact_tiles launch [WISE PR,
   * "What changes": sparse rows are compacted first; the finish of a
   * discovery depth already holds each (row, KV head)'s final mask].  Rows of
   * every mode get their list from the mask after the call; padding rows and
   * masks selecting nothing get no item.  support must not be NULL, and the
   * call's partial pass must not be on list 1 (that pass, or a compaction,
   * empties list 1 for this finish to fill).  List 1 stays valid until the
   * next partial pass that is not on it, the next compaction or the next
   * wise_build_sparse_list. */
  WISE_FLAG_BUILD_SPARSE_LIST = 4u,
  /* Partial pass and finish: every row is sparse and the work list is list 1
   * (written by an earlier finish with WISE_FLAG_BUILD_SPARSE_LIST over the
   * same rows and lengths, or by wise_build_sparse_list); modes is ignored
   * and may be NULL (see WISE_FLAG_LIST_MODES for a list of any modes).
   * Both passes of the call take the flag.  Not with
   * wise_decode_partial_finish. */
  WISE_FLAG_SPARSE_LIST = 8u,
  /* Partial pass and finish: every row attends every block below its length
   * (sparse rows too), discover and discover-union rows (by modes) also
   * record and select; the work list is derived from seq_lens by the passes
   * themselves, so no wise_compact_tiles runs [WISE PR, "What changes": the
   * compaction only matters to sparse rows; a dense row's tiles are all of
   * them].  At most WISE_DENSE_LIST_MAX_ROWS rows (else
   * WISE_ERR_UNSUPPORTED).  Both passes of the call take the flag; the
   * partial pass clears the workspace status word.  The workspace's queue
   * counters must be 0, as every compaction and every completed partial pass
   * leave them (wise_workspace_reset zeroes a new workspace).  Not with
   * WISE_FLAG_SPARSE_LIST or wise_decode_partial_finish; with
   * WISE_FLAG_EARLY_START only together with WISE_FLAG_INPUTS_READY. */
  WISE_FLAG_DENSE_LIST = 16u,
  /* Partial pass: everything the pass reads was complete before the kernel
   * ahead of this launch in the stream began: the caller's inputs (q, the
   * K/V pools, the page table, lengths and modes) -- as when that kernel is
   * a pass of this library -- and, with WISE_FLAG_SPARSE_LIST, list 1 (the
   * call is not the first on the list since the finish that built it).  A
   * pass on the dense list or on list 1 then takes its first items and
   * issues their copies while that kernel still runs.  Without the flag
   * every read waits for the previous kernel (a programmatic dependent
   * launch sees that kernel's writes only past its dependency wait).  Other
   * passes accept and ignore it. */
  WISE_FLAG_INPUTS_READY = 32u,
  /* With WISE_FLAG_SPARSE_LIST: list 1 was built by wise_build_list for the
   * modes this call passes, so the rows keep them -- the finish merges every
   * row and, for discover rows, selects and writes (DISCOVER) or ORs
   * (DISCOVER_UNION) the mask; modes must not be NULL.  The partial pass
   * accepts and ignores it (the items carry their rows' flags). */
  WISE_FLAG_LIST_MODES = 64u
};

/* Rows a call with WISE_FLAG_DENSE_LIST takes (its table lives in the
 * partial pass's shared memory). */
#define WISE_DENSE_LIST_MAX_ROWS 256

/* wise_decode_partial with flags (WISE_FLAG_SLOT_SET_1, WISE_FLAG_EARLY_START,
 * WISE_FLAG_SPARSE_LIST, WISE_FLAG_DENSE_LIST, WISE_FLAG_INPUTS_READY); flags = 0
 * is wise_decode_partial.  Unknown flags: WISE_ERR_INVALID_ARG. */
wise_status wise_decode_partial_ex(const wise_shape *shape, const void *q,
                                   const void *k_cache, const void *v_cache,
                                   const int32_t *page_table, const int32_t *seq_lens,
                                   const int8_t *modes, void *workspace,
                                   size_t workspace_bytes, uint32_t flags,
                                   wise_stream_t stream);

/* wise_decode_finish with flags (WISE_FLAG_SLOT_SET_1,
 * WISE_FLAG_BUILD_SPARSE_LIST, WISE_FLAG_SPARSE_LIST, WISE_FLAG_DENSE_LIST);
 * flags = 0 is wise_decode_finish. */
wise_status wise_decode_finish_ex(const wise_shape *shape, const int8_t *modes,
                                  const int32_t *seq_lens, void *workspace,
                                  size_t workspace_bytes, uint32_t flags,
                                  uint32_t *support, void *out, float *lse,
                                  wise_stream_t stream);

/* The partial pass with the finish folded in [WISE PR, "What changes": split
 * partials, then the merge and the selection for discovery rows]: the same
 * results as wise_decode_partial followed by wise_decode_finish, bit for
 * bit, in one launch when every row is short (max_blocks <= 64 and
 * ceil(max_blocks / tiles_per_item) <= 8).  Each work item is counted on
 * its (row, KV head)'s ticket in the workspace once its partial result is
 * written; the warp that completes a pair's last item merges the pair's
 * splits, writes out and lse and, for discover rows, the mask.  Pairs with
 * no item (padding rows, sparse rows selecting nothing) get out 0 and lse
 * -inf.  Nothing waits on a ticket.  Tickets are zeroed by
 * wise_compact_tiles and by the finishing warp, so several calls may reuse
 * one compaction.  For longer rows the two passes are launched one after the
 * other.  Arguments as for the two calls; out must be 16-byte aligned. */
wise_status wise_decode_partial_finish(const wise_shape *shape, const void *q,
                                       const void *k_cache, const void *v_cache,
                                       const int32_t *page_table,
                                       const int32_t *seq_lens, const int8_t *modes,
                                       void *workspace, size_t workspace_bytes,
                                       uint32_t *support, void *out, float *lse,
                                       wise_stream_t stream);

/* The calls that read or write the mask, with the mask addressed through a
 * wise_mask (per-request slots and a layer of a mask pool) instead of a
 * [num_rows, num_kv_heads, W] array; otherwise as wise_compact_tiles,
 * wise_build_sparse_list, wise_build_list, wise_decode_finish_ex,
 * wise_decode and wise_validate (a sparse row without a mask slot gets no
 * item in list 1).  `mask` is a HOST
 * pointer to the descriptor (its words and row_slot are device pointers);
 * mask->words may be NULL where the flat call's support may be NULL.  The
 * compaction reads each row's slot with its mode and length. */
wise_status wise_compact_tiles_m(const wise_shape *shape, const int8_t *modes,
                                 const int32_t *seq_lens, const wise_mask *mask,
                                 void *workspace, size_t workspace_bytes,
                                 wise_stream_t stream);
wise_status wise_build_sparse_list_m(const wise_shape *shape, const int32_t *seq_lens,
                                     const wise_mask *mask, void *workspace,
                                     size_t workspace_bytes, wise_stream_t stream);
wise_status wise_build_list_m(const wise_shape *shape, const int8_t *modes,
                              const int32_t *seq_lens, const wise_mask *mask, void *workspace,
                              size_t workspace_bytes, wise_stream_t stream);
wise_status wise_decode_finish_m(const wise_shape *shape, const int8_t *modes,
                                 const int32_t *seq_lens, void *workspace,
                                 size_t workspace_bytes, uint32_t flags,
                                 const wise_mask *mask, void *out, float *lse,
                                 wise_stream_t stream);
wise_status wise_decode_m(const wise_shape *shape, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *page_table,
                          const int32_t *seq_lens, const int8_t *modes,
                          const wise_mask *mask, void *out, float *lse, void *workspace,
                          size_t workspace_bytes, wise_stream_t stream);
wise_status wise_validate_m(const wise_shape *shape, const int32_t *page_table,
                            const int32_t *seq_lens, const int8_t *modes,
                            const wise_mask *mask, int32_t *err_word, wise_stream_t stream);

/* compact + partial + finish, in that order, on one stream. */
wise_status wise_decode(const wise_shape *shape, const void *q,
                        const void *k_cache, const void *v_cache,
                        const int32_t *page_table, const int32_t *seq_lens,
                        const int8_t *modes, uint32_t *support, void *out,
                        float *lse, void *workspace, size_t workspace_bytes,
                        wise_stream_t stream);

/* dst[i] |= src[i] for i < n_words [review "[P2] Distinguish discovery density
 * from reused union density": the reused support is the union of the
 * discovery depths' choices].  For callers that keep one mask per depth. */
wise_status wise_support_union(uint32_t *dst, const uint32_t *src,
                               int64_t n_words, wise_stream_t stream);

/* Block masses from the LSE by a second read of K [WISE PR, "What changes",
 * FlashAttention decode bullet: discovery rereads K once to rebuild block
 * mass from the attention's LSE].  For every discover or discover-union row
 * r (by `modes`), query head h and block b below the row's block count:
 * tile_stats[r, h, b] = (lse2, sum over the block's tokens j of
 * 2^(scale log2(e) <q_h, k_j> - lse2)), with lse2 = lse[r, h] / ln 2, so a
 * following wise_decode_finish with the same modes selects from these
 * masses.  lse [num_rows, num_q_heads] is the natural-log LSE of a previous
 * finish over the same q and K (a dense call, for instance).  Reads K only;
 * V is not touched.  Other rows are skipped.  q and k_cache must be 16-byte
 * aligned.  The in-pass statistics of the partial pass make this pass
 * unnecessary; it exists to measure what they save. */
wise_status wise_block_mass(const wise_shape *shape, const void *q,
                            const void *k_cache, const int32_t *page_table,
                            const int32_t *seq_lens, const int8_t *modes,
                            const float *lse, void *workspace,
                            size_t workspace_bytes, wise_stream_t stream);

/* Head union of the mask [WISE PR, "What changes", FlashAttention decode
 * bullet: sparse rows attend the per-layer head union of their support]: for
 * every row, each KV head's mask words become the OR of all the row's KV
 * heads' words (support [num_rows, num_kv_heads, ceil(max_blocks / 32)],
 * in place).  A sparse call on the result reads every selected block for
 * every head: the page-granular variant of sparse decode, for comparison
 * with per-head masks. */
wise_status wise_support_head_union(const wise_shape *shape, uint32_t *support,
                                    wise_stream_t stream);

/* Checks a batch's device data and ORs WISE_BAD_* / WISE_EMPTY_SPARSE_SUPPORT
 * bits into *err_word (device int32; the caller zeroes it first).  support
 * may be NULL when no row is sparse.  Never traps; reading only. */
wise_status wise_validate(const wise_shape *shape, const int32_t *page_table,
                          const int32_t *seq_lens, const int8_t *modes,
                          const uint32_t *support, int32_t *err_word,
                          wise_stream_t stream);

/* The same call as wise_decode, for callers that cannot allocate device
 * memory (no counterpart in the paper; it exists for integration only).
 * Instead of a caller-provided workspace it uses a 16 MiB scratch array that
 * lives in the library's static device memory, held by every GPU that loads
 * the library until the process exits.  A shape whose workspace
 * (wise_workspace_bytes) exceeds 16 MiB is rejected with WISE_ERR_WORKSPACE
 * and nothing is enqueued.  The first call in each CUDA context looks up the
 * array's device address (cudaGetSymbolAddress, with that context current)
 * and caches it under the context handle; the lookup may load device code,
 * so make that first call before any stream capture.  The cached address
 * does not survive cudaDeviceReset: after a reset, the first call in the new
 * context looks it up again only if the driver gives that context a new
 * handle.  No call allocates or frees device memory.  All calls on a device
 * share the one array and it keeps the last call's contents (nothing in it
 * needs to start at zero); calls whose GPU work overlaps (different streams
 * without ordering) race on it.  Device-side conditions (WISE_DEVERR_*) land
 * in the array's status word: read them with wise_noalloc_status. */
wise_status wise_decode_noalloc(const wise_shape *shape, const void *q,
                                const void *k_cache, const void *v_cache,
                                const int32_t *page_table, const int32_t *seq_lens,
                                const int8_t *modes, uint32_t *support, void *out,
                                float *lse, wise_stream_t stream);

/* The WISE_DEVERR_* status word of the last wise_decode_noalloc call in the
 * current context (0: no condition), copied into *host_status (a HOST
 * pointer) by a 4-byte device-to-host copy enqueued on `stream`: order the
 * stream after the decode call, then synchronise it before reading
 * *host_status.  After WISE_DEVERR_WAIT_TIMEOUT the call's out, lse and
 * support are undefined.  Allocates nothing.  NULL host_status:
 * WISE_ERR_INVALID_ARG. */
wise_status wise_noalloc_status(int32_t *host_status, wise_stream_t stream);

/* Self-test of the failure path (the pages have no counterpart; it computes
 * nothing of the method).  Every mbarrier wait in this library's kernels is
 * bounded by %globaltimer (500 ms) and, when it runs out, sets
 * WISE_DEVERR_WAIT_TIMEOUT in a status word and returns instead of hanging.
 * This call launches one CTA that waits, through the same bounded wait, on a
 * barrier nothing ever arrives on: after about 500 ms it ORs
 * WISE_DEVERR_WAIT_TIMEOUT into *status_word and returns, with nothing in
 * flight and the context usable.  status_word: a 4-byte aligned device
 * int32 the caller owns (zero it first to read the bit).  Asynchronous on
 * `stream`; a NULL or misaligned pointer returns WISE_ERR_INVALID_ARG. */
wise_status wise_selftest_wait_timeout(int32_t *status_word, wise_stream_t stream);

/* Static name of a status code. */
const char *wise_status_string(wise_status status);

/* One-line reason for the calling thread's last non-OK status ("" if none). */
const char *wise_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* WISE_H_ */
