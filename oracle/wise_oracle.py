"""CPU oracle for WISE working-set paged decode attention.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow definition that the
CUDA library is checked against.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the library never does, and it
imports nothing from the library.  Arithmetic is numpy float64.  Its sibling
wise_oracle.cpp states the same definition in plain C++ with fp32 math; the
same pins check both.

Source: the vllm-rlt pull request "WISE working-set decode" (PR #143),
cited below as [WISE PR, <section>].  What it fixes:

  * Each decode row runs in one of three modes ("What changes"): dense
    (ordinary paged decode attention), discover (dense, recording each
    32-token tile's max and sum), sparse (only the row's selected tiles).
  * A finish step merges the splits and, for discovery rows, runs the
    selection ("What changes"), with B=32 blocks and eta=0.95 ("Summary"),
    into a [slot, layer, head, block] support bitmask ("What changes",
    wise.py bullet); MODE_DISCOVER_UNION ORs the new choice into the previous
    support (review comment "[P2] Distinguish discovery density from reused
    union density").
  * Tests section: sparse output matches masked attention; LSE-derived block
    mass matches softmax block sums; compaction with every block selected is
    bitwise dense.

Readings where the pages are silent (each also listed in the design notes):

  * Block = tile = 32 consecutive token positions counted from token 0; the
    last block of a row holds only its valid tokens.
  * Softmax scale 1/sqrt(D); LSE is the natural log of sum exp(scale q.k).
  * Selection rule ("the reference rule"): order blocks by mass descending,
    equal masses by lower block index; take the smallest prefix whose
    cumulative mass reaches eta; eta >= 1 selects every block; at least one
    block is always taken.  The order and the cutoff are decided on masses
    rounded to float32, the precision the kernel decides in; cumulative sums
    are float64.
  * GQA: each query head selects with its own rule and the KV head's mask is
    the OR over its query-head group, so sparse rows attend the group union.
  * Sparse mode is attention renormalised over the selected tiles (a mask).
  * Padding rows (seq_len 0) produce output 0 and LSE -inf and leave the mask
    untouched, whatever their mode.  A sparse row with no selected block
    attends the empty set: output 0, LSE -inf.
  * Writing a mask clears bits at or past the row's block count.

Parity of every function here is pinned in tests/ against library routines
(torch scaled_dot_product_attention, softmax, logsumexp in float64), brute
force over subsets, closed-form cases and the pages' density example.
"""
from __future__ import annotations

import math
from typing import Dict, List, Tuple

import numpy as np

MODE_DENSE = 0
MODE_DISCOVER = 1
MODE_DISCOVER_UNION = 2
MODE_SPARSE = 3


# --------------------------------------------------------------------------- storage
def to_f64(x: np.ndarray) -> np.ndarray:
    """Stored values as float64.  uint16 arrays hold bfloat16 bit patterns
    (the upper half of an IEEE float32); float32 arrays are taken as is."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def row_kv(cache: np.ndarray, page_row: np.ndarray, L: int, g: int) -> np.ndarray:
    """Token-ordered [L, D] keys (or values) of KV head g for one row.

    The cache is paged [num_pages, page_size, Hkv, D]; token j of the row sits in
    page page_row[j // page_size] at slot j % page_size [WISE PR, "What changes":
    paged decode]."""
    P = cache.shape[1]
    j = np.arange(L)
    return to_f64(cache[np.asarray(page_row)[j // P], j % P, g])


# --------------------------------------------------------------------------- attention
def scores(q: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """s_j = scale * <q, k_j> for every token j."""
    return scale * (K @ q)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, active: np.ndarray,
           scale: float) -> Tuple[np.ndarray, float, np.ndarray]:
    """Softmax attention of one query over the active tokens.

    Returns (o [D], lse, s [L]).  Inactive tokens do not enter the softmax at
    all, which is attention under a mask [WISE PR, "Tests": sparse output
    matches masked attention].  With no active token the result is o = 0,
    lse = -inf."""
    s = scores(q, K, scale)
    if not active.any():
        return np.zeros(V.shape[1]), -math.inf, s
    m = s[active].max()
    e = np.where(active, np.exp(s - m), 0.0)
    Z = e.sum()
    o = (e @ V) / Z
    return o, m + math.log(Z), s


def tile_stats(s: np.ndarray, B: int) -> Tuple[np.ndarray, np.ndarray]:
    """Per 32-token tile b: m_b = max of s over the tile, l_b = sum exp(s - m_b)
    over the tile [WISE PR, "What changes": discover records each 32-token
    tile's max and sum]."""
    L = s.shape[0]
    nb = -(-L // B)
    m = np.empty(nb)
    l = np.empty(nb)
    for b in range(nb):
        t = s[b * B:min((b + 1) * B, L)]
        m[b] = t.max()
        l[b] = np.exp(t - m[b]).sum()
    return m, l


def block_masses(s: np.ndarray, lse: float, B: int) -> np.ndarray:
    """p_b = sum over the tile's tokens of exp(s_j - lse): the softmax mass of
    each block, summed explicitly token by token."""
    L = s.shape[0]
    nb = -(-L // B)
    p = np.empty(nb)
    for b in range(nb):
        p[b] = np.exp(s[b * B:min((b + 1) * B, L)] - lse).sum()
    return p


def select_blocks(p: np.ndarray, eta: float) -> Dict[str, object]:
    """The eta rule over block masses [WISE PR, "Summary": B=32 blocks and the
    eta=0.95 selection rule].

    Blocks are ordered by float32 mass descending, equal masses by lower block
    index; C_k is the cumulative mass of the first k; k* is the smallest k with
    C_k >= eta (all blocks if eta >= 1 or if C never reaches eta).

    Returns dict(sel=bool[n], k=k*, order=int[n], margin, gap) where
    margin = min(C_k* - eta, eta - C_(k*-1)) (C_0 = 0; +inf when eta >= 1) and
    gap = p_(k*) - p_(k*+1) in the sorted order (+inf when k* = n)."""
    n = p.shape[0]
    p32 = p.astype(np.float32).astype(np.float64)
    order = np.lexsort((np.arange(n), -p32))
    C = np.cumsum(p32[order])
    if eta >= 1.0:
        k = n
    else:
        reach = np.nonzero(C >= eta)[0]
        k = int(reach[0]) + 1 if reach.size else n
    sel = np.zeros(n, dtype=bool)
    sel[order[:k]] = True
    if eta >= 1.0:
        margin = math.inf
    else:
        prev = C[k - 2] if k >= 2 else 0.0
        margin = min(C[k - 1] - eta, eta - prev)
    gap = p32[order[k - 1]] - p32[order[k]] if k < n else math.inf
    return {"sel": sel, "k": k, "order": order, "margin": float(margin), "gap": float(gap)}


# --------------------------------------------------------------------------- masks
def mask_bits(support_words: np.ndarray, nb: int) -> np.ndarray:
    """bool[nb]: bit b of a (row, KV head) mask is word[b // 32] >> (b % 32) & 1."""
    b = np.arange(nb)
    w = np.asarray(support_words, dtype=np.uint32)[b // 32]
    return ((w >> (b % 32).astype(np.uint32)) & np.uint32(1)) == 1


def bits_to_words(bits: np.ndarray, W: int) -> np.ndarray:
    words = np.zeros(W, dtype=np.uint32)
    for b in np.nonzero(bits)[0]:
        words[b // 32] |= np.uint32(1) << np.uint32(b % 32)
    return words


def support_union(dst: np.ndarray, src: np.ndarray) -> np.ndarray:
    """Word-wise OR of two support masks [review "[P2] Distinguish discovery
    density from reused union density": chosen is ORed with the previous
    support]."""
    return (np.asarray(dst, np.uint32) | np.asarray(src, np.uint32)).astype(np.uint32)


def support_head_union(support: np.ndarray) -> np.ndarray:
    """[WISE PR, "What changes", FlashAttention decode bullet: sparse rows
    attend the per-layer head union of their support]: every KV head of a row
    gets each block that any KV head of the row selected.  Bit by bit, over
    all mask words."""
    sup = np.asarray(support, dtype=np.uint32)
    R, Hkv, W = sup.shape
    out = np.zeros_like(sup)
    for r in range(R):
        for b in range(32 * W):
            word, bit = b // 32, np.uint32(b % 32)
            if any((int(sup[r, g, word]) >> int(bit)) & 1 for g in range(Hkv)):
                out[r, :, word] |= np.uint32(1) << bit
    return out


def union_density(support: np.ndarray, seq_lens: np.ndarray, B: int) -> float:
    """Selected blocks of the final union over causal blocks, summed over every
    (row, KV head) with a non-empty row [author reply to the review, item 4:
    the first discovery depth adds its selection and the causal blocks, a
    union depth adds only newly set blocks]."""
    sel = 0
    causal = 0
    R, Hkv, _ = support.shape
    for r in range(R):
        nb = -(-int(seq_lens[r]) // B)
        for g in range(Hkv):
            sel += int(mask_bits(support[r, g], nb).sum())
            causal += nb
    return sel / causal if causal else 0.0


# --------------------------------------------------------------------------- compaction
def compact_tiles(support: np.ndarray, modes: np.ndarray, seq_lens: np.ndarray,
                  B: int) -> Dict[str, object]:
    """The compacted tile lists [WISE PR, "What changes": sparse rows attend
    only their selected tiles, compacted first so the loop has no branch].

    Per (row, KV head): the ascending block indices b < n_b whose mask bit is
    set for sparse rows, and every block 0..n_b-1 for the other modes.  How a
    list is cut into work items for the GPU's programs ("about eight tiles"
    each) is a scheduling choice the pages leave open, so it is not defined
    here; the tests check the kernel's items against these lists by their
    properties.  Returns dict(lists=[R][Hkv] int32 arrays, counts=int32
    [R, Hkv])."""
    R, Hkv, _ = support.shape
    lists: List[List[np.ndarray]] = []
    counts = np.zeros((R, Hkv), dtype=np.int32)
    for r in range(R):
        nb = -(-int(seq_lens[r]) // B)
        per = []
        for g in range(Hkv):
            if int(modes[r]) == MODE_SPARSE:
                lst = np.nonzero(mask_bits(support[r, g], nb))[0].astype(np.int32)
            else:
                lst = np.arange(nb, dtype=np.int32)
            per.append(lst)
            counts[r, g] = lst.shape[0]
        lists.append(per)
    return {"lists": lists, "counts": counts}


# --------------------------------------------------------------------------- mask pool
def gather_slot_masks(pool: np.ndarray, row_slot: np.ndarray, layer: int) -> np.ndarray:
    """The masks a batch's rows use, read from a [slot, layer, KV head, word]
    pool [WISE PR, "What changes", wise.py bullet: per-request slots hold a
    [slot, layer, head, block] support bitmask]: row r takes
    pool[row_slot[r], layer]; a row whose slot is -1 has no mask (all zero)."""
    pool = np.asarray(pool, np.uint32)
    R = len(row_slot)
    out = np.zeros((R,) + pool.shape[2:], np.uint32)
    for r in range(R):
        if int(row_slot[r]) >= 0:
            out[r] = pool[int(row_slot[r]), layer]
    return out


def decode_layer_slots(q, k_cache, v_cache, page_table, seq_lens, modes, pool, row_slot,
                       layer: int, decode=None, **kw) -> Dict[str, object]:
    """decode_layer with each row's mask addressed through its slot and the
    layer: the masks are gathered by index, the call runs, and every row
    whose mode writes its mask (discover, discover-union) and that has a
    slot gets its new mask stored back at pool[slot, layer].  Rows without a
    slot attend and discover as with an empty mask and store nothing.
    Returns decode_layer's result with "pool" (the pool after the call) in
    place of "support".  `decode` is the decode_layer to run (this module's
    by default; the C++ oracle passes its own)."""
    sup = gather_slot_masks(pool, row_slot, layer)
    res = (decode or decode_layer)(q, k_cache, v_cache, page_table, seq_lens, modes, sup, **kw)
    new_pool = np.array(pool, dtype=np.uint32, copy=True)
    for r in range(len(row_slot)):
        if int(row_slot[r]) >= 0 and int(modes[r]) in (MODE_DISCOVER, MODE_DISCOVER_UNION) \
                and int(seq_lens[r]) > 0:
            new_pool[int(row_slot[r]), layer] = res["support"][r]
    res["pool"] = new_pool
    return res


# --------------------------------------------------------------------------- one call
def decode_layer(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                 page_table: np.ndarray, seq_lens: np.ndarray, modes: np.ndarray,
                 support: np.ndarray, *, eta: float = 0.95, tile_tokens: int = 32,
                 scale: float = 0.0) -> Dict[str, object]:
    """One WISE decode call for a batch of rows (one layer at one depth).

    q [R, Hq, D]; k_cache, v_cache [num_pages, page_size, Hkv, D] (uint16 bf16
    bits or float32); page_table int32 [R, max_pages]; seq_lens int32 [R];
    modes int8 [R]; support uint32 [R, Hkv, W] (the mask before the call).

    Returns out [R, Hq, D] float64, lse [R, Hq] float64, support (after the
    call), and per (row, query head) diagnostics: tile stats, block masses,
    selections with their margin and gap (discover rows only)."""
    q64 = to_f64(q)
    R, Hq, D = q64.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    B = tile_tokens
    W = support.shape[2]
    if scale == 0.0:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((R, Hq, D))
    lse = np.full((R, Hq), -math.inf)
    new_support = np.array(support, dtype=np.uint32, copy=True)
    diag: Dict[Tuple[int, int], Dict[str, object]] = {}
    for r in range(R):
        L = int(seq_lens[r])
        if L == 0:
            continue
        nb = -(-L // B)
        mode = int(modes[r])
        block_of = np.arange(L) // B
        for g in range(Hkv):
            K = row_kv(k_cache, page_table[r], L, g)
            V = row_kv(v_cache, page_table[r], L, g)
            if mode == MODE_SPARSE:
                active = mask_bits(support[r, g], nb)[block_of]
            else:
                active = np.ones(L, dtype=bool)
            group_sel = np.zeros(nb, dtype=bool)
            for h in range(g * G, (g + 1) * G):
                o, lse_h, s = attend(q64[r, h], K, V, active, scale)
                out[r, h] = o
                lse[r, h] = lse_h
                if mode in (MODE_DISCOVER, MODE_DISCOVER_UNION):
                    m_b, l_b = tile_stats(s, B)
                    p = block_masses(s, lse_h, B)
                    pick = select_blocks(p, eta)
                    group_sel |= pick["sel"]
                    diag[(r, h)] = {"m_b": m_b, "l_b": l_b, "p": p, **pick}
            if mode == MODE_DISCOVER:
                new_support[r, g] = bits_to_words(group_sel, W)
            elif mode == MODE_DISCOVER_UNION:
                previous = bits_to_words(mask_bits(support[r, g], nb), W)
                new_support[r, g] = support_union(previous, bits_to_words(group_sel, W))
    return {"out": out, "lse": lse, "support": new_support, "diag": diag, "scale": scale}
