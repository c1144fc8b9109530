"""wise_build_sparse_list: list 1 of an all-sparse call built from the mask
alone (no compaction, no finish before it); wise_build_list: the same for a
call of any modes (run with WISE_FLAG_LIST_MODES).  Its items equal those a finish
with WISE_FLAG_BUILD_SPARSE_LIST writes for the same mask, they partition the
oracle's compacted tile lists, the sparse call on them equals the compaction's
call bit for bit where the finish merges the same slots in the same order
(rows of at most 64 blocks), and agrees with the oracle everywhere (rows up
to 128K tokens); slot-addressed masks, rows without a mask and clamped
lengths included."""
import numpy as np
import pytest
import torch

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300.workload import custom_workload
from oracle import wise_oracle as O
from tests.gpu_harness import (Batch, compare_masks, compare_outputs, dev_support, gpu_call, item_fields,
                               item_invariant_fails, list1_schedule, np_support, oracle_call,
                               shape_for, words)

pytestmark = pytest.mark.gpu

RAGGED = np.array([1, 31, 32, 33, 300, 517, 0, 1024], np.int32)
CASES = [(4, 4, 128, "bf16"), (8, 2, 128, "bf16"), (4, 1, 64, "bf16"), (4, 2, 128, "f32")]


def _wl(Hq, Hkv, D, dtype, lens=RAGGED, seed=61, page_size=16):
    R = len(lens)
    return custom_workload("sparse_list", R=R, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, depths=2,
                           n_planted=3, seq_lens=lens, pool_factor=2, seed=seed,
                           depth_modes=[np.full(R, W.MODE_SPARSE, np.int8)] * 2,
                           page_size=page_size)


def _random_mask(w, density, seed):
    rng = np.random.default_rng(seed)
    bits = rng.random((w.num_rows, w.num_kv_heads, words(w) * 32)) < density
    sup = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(
        w.num_rows, w.num_kv_heads, -1).copy()
    sup[0, 0] = 0  # a (row, KV head) selecting nothing
    return sup


def _views(shape, ws):
    return {k: t.cpu() for k, t in W.workspace_views(shape, ws).items()}


def _sparse_on_list(b, shape, ws, depth=0):
    """Partial pass and finish on list 1 (every row sparse)."""
    w = b.w
    d = b.dev(depth)
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.num_rows, w.num_q_heads), dtype=torch.float32, device="cuda")
    W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                             None, ws, W.FLAG_SPARSE_LIST)
    W.wise_decode_finish_ex(shape, None, b.seq_lens, ws, None, out, lse, W.FLAG_SPARSE_LIST)
    torch.cuda.synchronize()
    return out, lse


def _items_by_pair(v, T):
    """Each (row, KV head)'s list-1 records, sorted (the order within a bucket
    follows the pairs' atomics, so only the sets are defined)."""
    recs = list1_schedule(v, T)
    f = item_fields(recs)
    out = {}
    for rg in np.unique(f["rg"]):
        sel = recs[f["rg"] == rg]
        out[int(rg)] = sel[np.lexsort(sel.T[::-1])]
    return out


@pytest.mark.parametrize("T", [0, 2, 16])
@pytest.mark.parametrize("Hq,Hkv,lens", [(4, 4, RAGGED), (8, 2, np.array([10000, 5000, 1, 33, 0], np.int32))])
def test_built_list_equals_the_finish_built_list(Hq, Hkv, lens, T):
    w = _wl(Hq, Hkv, 128, "bf16", lens=lens)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w, tiles_per_item=T)
    Tr = W.wise._tiles_per_item(shape)
    sup_np = _random_mask(w, 0.3, seed=67)
    # the finish-built list: a dense call (its mask is left as it is) with
    # WISE_FLAG_BUILD_SPARSE_LIST
    ws_a = W.alloc_workspace(shape)
    sup = dev_support(sup_np)
    dense = torch.zeros(R, dtype=torch.int8, device="cuda")
    d = b.dev(0)
    out = torch.empty_like(d["q"])
    lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    W.wise_compact_tiles(shape, dense, b.seq_lens, sup, ws_a)
    W.wise_decode_partial(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                          dense, ws_a)
    W.wise_decode_finish_ex(shape, dense, b.seq_lens, ws_a, sup, out, lse, W.FLAG_BUILD_SPARSE_LIST)
    # the standalone build, on a workspace that held another call's state
    ws_b = W.alloc_workspace(shape)
    ws_b.fill_(0x5A)
    W.wise_build_sparse_list(shape, b.seq_lens, sup, ws_b)
    torch.cuda.synchronize()
    va, vb = _views(shape, ws_a), _views(shape, ws_b)
    assert int(vb["status"][0]) == 0 and int(vb["queue"][0]) == 0
    assert np.array_equal(va["list1_counter"].numpy()[:Tr], vb["list1_counter"].numpy()[:Tr])
    assert np.array_equal(va["head_info_1"].numpy(), vb["head_info_1"].numpy())
    ia, ib = _items_by_pair(va, Tr), _items_by_pair(vb, Tr)
    assert ia.keys() == ib.keys()
    for rg in ia:
        assert np.array_equal(ia[rg], ib[rg]), rg
    ref = O.compact_tiles(sup_np, np.full(R, W.MODE_SPARSE, np.int8), w.seq_lens, 32)
    fails = item_invariant_fails(list1_schedule(vb, Tr), vb["head_info_1"].numpy(), ref["lists"], Tr,
                                 -(-shape.max_blocks // Tr), w.seq_lens, None, Hkv, compact_slots=True)
    assert not fails, fails[:5]
    assert np.array_equal(np_support(sup), sup_np)  # the build only reads the mask


@pytest.mark.parametrize("Hq,Hkv,D,dtype", CASES)
def test_sparse_call_on_built_list(Hq, Hkv, D, dtype):
    """Rows of at most 64 blocks: the call on the built list equals the
    compaction's sparse call bitwise (twice on one workspace: the second
    build resets what the first call left); against the oracle too."""
    w = _wl(Hq, Hkv, D, dtype)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    sup_np = _random_mask(w, 0.25, seed=71)
    sup = dev_support(sup_np)
    ws = W.alloc_workspace(shape)
    g = gpu_call(b, 1, np.full(R, W.MODE_SPARSE, np.int8), sup_np)
    for _ in range(2):
        W.wise_build_sparse_list(shape, b.seq_lens, sup, ws)
        out, lse = _sparse_on_list(b, shape, ws, depth=1)
        assert torch.equal(out.cpu(), g["out_raw"]) and np.array_equal(lse.cpu().numpy(), g["lse"])
        assert int(_views(shape, ws)["status"][0]) == 0
    o = oracle_call(b, 1, np.full(R, W.MODE_SPARSE, np.int8), sup_np)
    assert not compare_outputs(w, {"out": out.double().cpu().numpy(), "lse": lse.cpu().numpy()}, o)
    # the (row, KV head) selecting nothing: output 0, LSE -inf for its heads
    G = Hq // Hkv
    assert torch.all(out[0, :G] == 0) and torch.all(torch.isneginf(lse[0, :G]))


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 1)])
def test_built_list_long_rows(Hq, Hkv):
    """Rows up to 128K tokens (4096 blocks, 512 ranges of 8 a pair): the call
    on the built list against the oracle, its items against the oracle's
    lists."""
    lens = np.array([131072, 20000, 0, 4097], np.int32)
    w = _wl(Hq, Hkv, 128, "bf16", lens=lens)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    T = W.wise._tiles_per_item(shape)
    sup_np = _random_mask(w, 0.02, seed=73)
    sup = dev_support(sup_np)
    ws = W.alloc_workspace(shape)
    W.wise_build_sparse_list(shape, b.seq_lens, sup, ws)
    out, lse = _sparse_on_list(b, shape, ws)
    v = _views(shape, ws)
    assert int(v["status"][0]) == 0
    o = oracle_call(b, 0, np.full(R, W.MODE_SPARSE, np.int8), sup_np)
    assert not compare_outputs(w, {"out": out.double().cpu().numpy(), "lse": lse.cpu().numpy()}, o)
    ref = O.compact_tiles(sup_np, np.full(R, W.MODE_SPARSE, np.int8), w.seq_lens, 32)
    fails = item_invariant_fails(list1_schedule(v, T), v["head_info_1"].numpy(), ref["lists"], T,
                                 -(-shape.max_blocks // T), w.seq_lens, None, Hkv, compact_slots=True)
    assert not fails, fails[:5]


def test_built_list_from_a_slot_pool():
    """Masks addressed per request slot (wise_build_sparse_list_m): the same
    items as the flat build on the gathered masks; a row without a slot gets
    no item, and its output is 0 with LSE -inf."""
    w = _wl(4, 4, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    T = W.wise._tiles_per_item(shape)
    slots, layers, layer = 11, 3, 2
    rng = np.random.default_rng(79)
    bits = rng.random((slots, layers, 4, words(w) * 32)) < 0.3
    pool_np = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(
        slots, layers, 4, -1).copy()
    row_slot = rng.permutation(slots)[:R].astype(np.int32)
    row_slot[3] = -1
    pool = dev_support(pool_np)
    slots_t = torch.from_numpy(row_slot).cuda()  # the descriptor holds its address
    ws_a = W.alloc_workspace(shape)
    W.wise_build_sparse_list_m(shape, b.seq_lens, W.make_mask(pool, slots_t, layer), ws_a)
    out, lse = _sparse_on_list(b, shape, ws_a)
    gathered = O.gather_slot_masks(pool_np, row_slot, layer)
    ws_b = W.alloc_workspace(shape)
    W.wise_build_sparse_list(shape, b.seq_lens, dev_support(gathered), ws_b)
    torch.cuda.synchronize()
    va, vb = _views(shape, ws_a), _views(shape, ws_b)
    ia, ib = _items_by_pair(va, T), _items_by_pair(vb, T)
    assert ia.keys() == ib.keys() and all(np.array_equal(ia[k], ib[k]) for k in ia)
    assert not any(rg // 4 == 3 for rg in ia)
    assert np.array_equal(np_support(pool), pool_np)
    assert torch.all(out[3] == 0) and torch.all(torch.isneginf(lse[3]))
    o = oracle_call(b, 0, np.full(R, W.MODE_SPARSE, np.int8), gathered)
    assert not compare_outputs(w, {"out": out.double().cpu().numpy(), "lse": lse.cpu().numpy()}, o)


def test_built_list_clamps_and_flags_long_lengths():
    w = _wl(4, 4, 64, "bf16", lens=np.array([64, 100, 40, 33], np.int32))
    b = Batch(w)
    shape = shape_for(w)
    cap = min(w.max_blocks * 32, w.max_pages_per_row * w.page_size)
    lens = w.seq_lens.copy()
    lens[0] = cap + 1000
    full = np.full((4, 4, words(w)), 0xFFFFFFFF, np.uint32)
    ws = W.alloc_workspace(shape)
    W.wise_build_sparse_list(shape, torch.from_numpy(lens).cuda(), dev_support(full), ws)
    torch.cuda.synchronize()
    v = _views(shape, ws)
    assert int(v["status"][0]) & W.wise.DEVERR_SEQ_LEN_CLAMPED
    assert int(v["head_info_1"][0, 0, 2]) == -(-cap // 32)  # every block below the capacity


# ---------------------------------------------------------------- any modes
MIXED = np.array([1, 2, 0, 3, 1, 2, 3, 3], np.int8)  # discover, union, dense, sparse


def _mixed_on_built_list(b, shape, modes_np, sup, depth=0, ws=None):
    """wise_build_list, then the partial pass and finish on list 1 with the
    rows' modes (WISE_FLAG_SPARSE_LIST | WISE_FLAG_LIST_MODES)."""
    w = b.w
    d = b.dev(depth)
    ws = W.alloc_workspace(shape) if ws is None else ws
    modes = torch.from_numpy(modes_np).cuda()
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.num_rows, w.num_q_heads), dtype=torch.float32, device="cuda")
    f = W.FLAG_SPARSE_LIST | W.FLAG_LIST_MODES
    W.wise_build_list(shape, modes, b.seq_lens, sup, ws)
    W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                             modes, ws, f)
    W.wise_decode_finish_ex(shape, modes, b.seq_lens, ws, sup, out, lse, f)
    torch.cuda.synchronize()
    return out, lse, ws


@pytest.mark.parametrize("Hq,Hkv,D,dtype,page_size", [c + (16,) for c in CASES] +
                         [(8, 1, 128, "bf16", 16), (4, 4, 128, "bf16", 32), (8, 2, 64, "f32", 32)])
def test_mixed_call_on_built_list_equals_compaction(Hq, Hkv, D, dtype, page_size):
    """Rows of every mode in one call: on the list built for the modes it
    equals the compaction's call bit for bit (outputs, LSEs and the mask the
    discover rows leave), its items partition the oracle's lists for the same
    modes, and it agrees with the oracle.  Eight query heads a KV head, and
    pages of 32 tokens (one page a tile) too."""
    w = _wl(Hq, Hkv, D, dtype, page_size=page_size)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    T = W.wise._tiles_per_item(shape)
    sup_np = _random_mask(w, 0.3, seed=83)
    g = gpu_call(b, 0, MIXED, sup_np)
    sup = dev_support(sup_np)
    ws = None
    for _ in range(2):  # the second call reuses the workspace
        sup.copy_(dev_support(sup_np))
        out, lse, ws = _mixed_on_built_list(b, shape, MIXED, sup, ws=ws)
        assert torch.equal(out.cpu(), g["out_raw"]) and np.array_equal(lse.cpu().numpy(), g["lse"])
        assert np.array_equal(np_support(sup), g["support"])
        v = _views(shape, ws)
        assert int(v["status"][0]) == 0
    ref = O.compact_tiles(sup_np, MIXED, w.seq_lens, 32)
    fails = item_invariant_fails(list1_schedule(v, T), v["head_info_1"].numpy(), ref["lists"], T,
                                 -(-shape.max_blocks // T), w.seq_lens, MIXED, Hkv, compact_slots=True)
    assert not fails, fails[:5]
    o = oracle_call(b, 0, MIXED, sup_np)
    assert not compare_outputs(w, {"out": out.double().cpu().numpy(), "lse": lse.cpu().numpy()}, o)


@pytest.mark.parametrize("Hq,Hkv,lens", [(2, 2, np.array([20000, 3000, 0, 700, 17000], np.int32)),
                                         (8, 2, np.array([40000, 33, 9000, 0, 131072], np.int32))])
def test_mixed_long_rows_on_built_list(Hq, Hkv, lens):
    """Long rows of every mode (the clustered finish selects on list 1): the
    outputs and the masks against the oracle on the same input mask."""
    w = _wl(Hq, Hkv, 128, "bf16", lens=lens)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    modes_np = np.array([1, 3, 2, 3, 0], np.int8)[:R]
    sup_np = _random_mask(w, 0.05, seed=89)
    sup = dev_support(sup_np)
    out, lse, ws = _mixed_on_built_list(b, shape, modes_np, sup)
    assert int(_views(shape, ws)["status"][0]) == 0
    g = {"out": out.double().cpu().numpy(), "lse": lse.cpu().numpy(), "support": np_support(sup)}
    o = oracle_call(b, 0, modes_np, sup_np)
    fails = compare_outputs(w, g, o)
    fails += compare_masks(w, g["support"], o, modes_np, support_in=sup_np)["fails"]
    assert not fails, fails[:5]


def test_large_mixed_batch_on_built_list():
    """300 rows (past the dense list's limit) of every mode, no compaction:
    sampled rows against the oracle."""
    rng = np.random.default_rng(97)
    lens = rng.integers(0, 1500, size=300).astype(np.int32)
    w = _wl(4, 2, 128, "bf16", lens=lens)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    modes_np = rng.integers(0, 4, size=R).astype(np.int8)
    sup_np = _random_mask(w, 0.2, seed=101)
    sup = dev_support(sup_np)
    out, lse, ws = _mixed_on_built_list(b, shape, modes_np, sup)
    assert int(_views(shape, ws)["status"][0]) == 0
    rows = np.unique(np.concatenate([[0, R - 1], rng.choice(R, size=22, replace=False)]))
    g = {"out": out.double().cpu().numpy(), "lse": lse.cpu().numpy(), "support": np_support(sup)}
    o = oracle_call(b, 0, modes_np, sup_np, rows=rows)
    fails = compare_outputs(w, g, o, rows=rows)
    fails += compare_masks(w, g["support"], o, modes_np, rows=rows, support_in=sup_np)["fails"]
    assert not fails, fails[:5]


def test_mixed_list_on_a_slot_pool():
    """A call of every mode on a list built from a slot pool
    (wise_build_list_m, then the finish through the same descriptor): equal,
    bit for bit, to the same call on the gathered masks, and the discover
    rows write their selections into their own slots only."""
    w = _wl(4, 4, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    slots, layers, layer = 11, 3, 1
    rng = np.random.default_rng(103)
    bits = rng.random((slots, layers, 4, words(w) * 32)) < 0.3
    pool_np = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(
        slots, layers, 4, -1).copy()
    row_slot = rng.permutation(slots)[:R].astype(np.int32)
    row_slot[6] = -1  # a sparse row (MIXED[6] == 3) without a mask
    modes = torch.from_numpy(MIXED).cuda()
    f = W.FLAG_SPARSE_LIST | W.FLAG_LIST_MODES
    d = b.dev(0)
    # on the pool
    pool = dev_support(pool_np)
    slots_t = torch.from_numpy(row_slot).cuda()  # alive while the descriptor is used
    mask = W.make_mask(pool, slots_t, layer)
    ws = W.alloc_workspace(shape)
    out_a = torch.empty_like(d["q"])
    lse_a = torch.empty((R, 4), dtype=torch.float32, device="cuda")
    W.wise_build_list_m(shape, modes, b.seq_lens, mask, ws)
    W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                             modes, ws, f)
    W.wise_decode_finish_m(shape, modes, b.seq_lens, ws, mask, out_a, lse_a, f)
    # on the gathered masks
    gathered = O.gather_slot_masks(pool_np, row_slot, layer)
    sup = dev_support(gathered)
    out_b, lse_b, _ = _mixed_on_built_list(b, shape, MIXED, sup)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)
    after = np_support(pool)
    g_after = np_support(sup)
    for r, sl in enumerate(row_slot):
        if sl >= 0:
            assert np.array_equal(after[sl, layer], g_after[r]), r
    touched = {(int(sl), layer) for sl in row_slot if sl >= 0}
    for sl in range(slots):
        for ly in range(layers):
            if (sl, ly) not in touched:
                assert np.array_equal(after[sl, ly], pool_np[sl, ly]), (sl, ly)
    assert torch.all(out_a[6] == 0) and torch.all(torch.isneginf(lse_a[6]))
