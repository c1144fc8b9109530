"""GPU parity against the CPU oracle at sizes the oracle finishes in seconds:
several tiles per row, ragged tails, padding rows, NaN-filled pool pages and
slots no row owns.  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300.workload import custom_workload, make_workload
from oracle import wise_oracle as O
from tests.gpu_harness import (Batch, compare_masks, compare_outputs, dev_support, gpu_call,
                               item_invariant_fails, list1_schedule, np_support, oracle_call,
                               shape_for, words)
from tests.gpu_harness import oracle_call as _oracle_call

pytestmark = pytest.mark.gpu

RAGGED = np.array([1, 31, 32, 33, 300, 517, 0, 1024], np.int32)


def _wl(Hq, Hkv, D, dtype, lens=RAGGED, seed=3, n_planted=3, page_size=16):
    R = len(lens)
    return custom_workload("parity", R=R, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, depths=3,
                           n_planted=n_planted, seq_lens=lens, pool_factor=2, seed=seed,
                           depth_modes=[np.zeros(R, np.int8)] * 3, page_size=page_size)


CASES = [(4, 4, 128, "bf16"), (4, 4, 64, "bf16"), (8, 2, 128, "bf16"), (4, 1, 64, "bf16"),
         (2, 2, 64, "f32"), (4, 2, 128, "f32")]


@pytest.mark.parametrize("oracle", ["f32", "f64"])
@pytest.mark.parametrize("Hq,Hkv,D,dtype", CASES)
def test_modes_match_oracle(Hq, Hkv, D, dtype, oracle):
    w = _wl(Hq, Hkv, D, dtype)
    b = Batch(w)
    R = w.num_rows
    zero = np.zeros((R, Hkv, words(w)), np.uint32)
    oracle_call = lambda *a, **k: _oracle_call(*a, oracle=oracle, **k)  # noqa: E731
    # dense
    m = np.full(R, W.MODE_DENSE, np.int8)
    g, o = gpu_call(b, 0, m, zero), oracle_call(b, 0, m, zero)
    assert not compare_outputs(w, g, o)
    assert np.array_equal(g["support"], zero)  # dense leaves the mask alone
    # discover at depth 0 (overwrites a garbage mask), union-discover at depth 1
    junk = np.random.default_rng(1).integers(0, 2**32, size=zero.shape, dtype=np.uint32)
    m = np.full(R, W.MODE_DISCOVER, np.int8)
    g, o = gpu_call(b, 0, m, junk), oracle_call(b, 0, m, junk)
    assert not compare_outputs(w, g, o)
    cm = compare_masks(w, g["support"], o, m)
    assert not cm["fails"] and cm["checked"] >= cm["excluded"], cm
    s0 = o["support"]
    m = np.full(R, W.MODE_DISCOVER_UNION, np.int8)
    g, o = gpu_call(b, 1, m, s0), oracle_call(b, 1, m, s0)
    assert not compare_outputs(w, g, o)
    cm = compare_masks(w, g["support"], o, m, support_in=s0)
    assert not cm["fails"], cm
    # sparse on the oracle's union mask (the same mask on both sides)
    s1 = o["support"]
    m = np.full(R, W.MODE_SPARSE, np.int8)
    g, o = gpu_call(b, 2, m, s1), oracle_call(b, 2, m, s1)
    assert not compare_outputs(w, g, o)
    assert np.array_equal(g["support"], s1)  # sparse leaves the mask alone


@pytest.mark.parametrize("eta", [0.5, 0.8, 0.9, 0.99, 1.0])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4)])
def test_eta_range(Hq, Hkv, eta):
    """The selection across the threshold range of the GQA long-context
    workload (0.8-0.99) and its ends: eta = 1 keeps every causal block."""
    w = _wl(Hq, Hkv, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    zero = np.zeros((R, Hkv, words(w)), np.uint32)
    m = np.full(R, W.MODE_DISCOVER, np.int8)
    g, o = gpu_call(b, 0, m, zero, eta=eta), oracle_call(b, 0, m, zero, eta=eta)
    assert not compare_outputs(w, g, o)
    cm = compare_masks(w, g["support"], o, m)
    assert not cm["fails"] and cm["checked"] >= cm["excluded"], cm
    if eta >= 1.0:
        full = np.zeros_like(zero)
        for r in range(R):
            nb = -(-int(w.seq_lens[r]) // 32)
            for blk in range(nb):
                full[r, :, blk >> 5] |= np.uint32(1 << (blk & 31))
        assert np.array_equal(g["support"], full)
    m = np.full(R, W.MODE_SPARSE, np.int8)
    g, o = gpu_call(b, 1, m, o["support"], eta=eta), oracle_call(b, 1, m, o["support"], eta=eta)
    assert not compare_outputs(w, g, o)


@pytest.mark.parametrize("lens", [RAGGED, np.array([16384, 3000, 0, 9000], np.int32)],
                         ids=["short", "long"])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4)])
def test_tiny_eta_keeps_each_heads_top_block(Hq, Hkv, lens):
    """The small end of the threshold: with eta below every block's mass the
    shortest prefix reaching it is one block, so each query head keeps exactly
    its heaviest block (equal masses: the lower index) and a KV head's mask is
    the OR of its group's choices.  Checked against the oracle's block masses
    wherever the two heaviest blocks differ by more than a relative 1e-5 (the
    rest must still keep one to G blocks); rows of 512 blocks and more take the
    finish's threshold search instead of the sort.  Then a sparse call on that
    mask (one tile per query head) against the oracle."""
    eta = 1e-6
    w = _wl(Hq, Hkv, 128, "bf16", lens=lens)
    b = Batch(w)
    R, G = w.num_rows, w.group
    zero = np.zeros((R, Hkv, words(w)), np.uint32)
    m = np.full(R, W.MODE_DISCOVER, np.int8)
    g, o = gpu_call(b, 0, m, zero, eta=eta), oracle_call(b, 0, m, zero, eta=eta)
    assert not compare_outputs(w, g, o)
    checked = 0
    for r in range(R):
        nb = -(-int(w.seq_lens[r]) // 32)
        if nb == 0:
            assert not g["support"][r].any()
            continue
        for kv in range(Hkv):
            want = np.zeros(nb, bool)
            clear = True
            for h in range(kv * G, (kv + 1) * G):
                dg = o["diag"][(r, h)]
                ps = np.asarray(dg["p"], np.float64)[dg["order"]]
                want[dg["order"][0]] = True
                clear &= nb == 1 or ps[0] - ps[1] > 1e-5 * ps[0]
            got = O.mask_bits(g["support"][r, kv], nb)
            assert 1 <= got.sum() <= G, (r, kv)
            if clear:
                checked += 1
                assert np.array_equal(got, want), (r, kv)
    assert checked > 0
    m = np.full(R, W.MODE_SPARSE, np.int8)
    g2, o2 = gpu_call(b, 1, m, g["support"], eta=eta), oracle_call(b, 1, m, g["support"], eta=eta)
    assert not compare_outputs(w, g2, o2)


def test_tile_stats_match_oracle():
    """Discover rows' per-tile max and exp-sum (the workspace intermediates)."""
    w = _wl(4, 4, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    zero = np.zeros((R, 4, words(w)), np.uint32)
    m = np.full(R, W.MODE_DISCOVER, np.int8)
    g, o = gpu_call(b, 0, m, zero), oracle_call(b, 0, m, zero)
    ts = g["ws"]["tile_stats"].numpy()
    for (r, h), dg in o["diag"].items():
        nb = dg["m_b"].shape[0]
        m_gpu = ts[r, h, :nb, 0] / W.wise.LOG2E
        assert np.max(np.abs(m_gpu - dg["m_b"])) < 1e-4
        assert np.max(np.abs(ts[r, h, :nb, 1] / dg["l_b"] - 1)) < 1e-4


def test_tiny_schedule_f32():
    """The 4-row fp32 D=64 workload: rows [dense, discover, sparse, sparse] over
    two depths; sparse rows use a support from a prior discovery of the same
    inputs (depth 0 discover, depth 1 union)."""
    w = make_workload("tiny")
    b = Batch(w)
    R = w.num_rows
    zero = np.zeros((R, w.num_kv_heads, words(w)), np.uint32)
    d0 = np.full(R, W.MODE_DISCOVER, np.int8)
    prior = oracle_call(b, 0, d0, zero)["support"]
    prior = oracle_call(b, 1, np.full(R, W.MODE_DISCOVER_UNION, np.int8), prior)["support"]
    sup = prior.copy()
    sup[w.depth_modes[0] == W.MODE_DISCOVER] = 0
    for depth in range(2):
        m = w.depth_modes[depth]
        g, o = gpu_call(b, depth, m, sup), oracle_call(b, depth, m, sup)
        assert not compare_outputs(w, g, o)
        assert not compare_masks(w, g["support"], o, m, support_in=sup)["fails"]
        sup = o["support"]


def _compact(w, T, modes, sup, lens=None):
    """wise_compact_tiles alone; returns the workspace views on the host."""
    lens = w.seq_lens if lens is None else lens
    shape = shape_for(w, tiles_per_item=T)
    ws = W.alloc_workspace(shape)
    W.wise_compact_tiles(shape, torch.from_numpy(np.asarray(modes, np.int8)).cuda(),
                         torch.from_numpy(np.asarray(lens, np.int32)).cuda(), dev_support(sup), ws)
    torch.cuda.synchronize()
    return shape, {k: t.cpu().numpy() for k, t in W.workspace_views(shape, ws).items()}


def test_compaction_items_partition_the_oracle_lists():
    """The compaction's work items against the oracle's compacted tile lists,
    by properties (the pages fix the lists, the cut into items is the
    kernel's): each item a run of 1..T tiles inside one range, a pair's items
    partitioning its list, slots equal to ranges, schedule non-increasing in
    tile count, head info and record fields right; empty ranges of sparse
    rows marked in both slot sets so the finish skips them."""
    rng = np.random.default_rng(5)
    for T in (1, 2, 4, 8, 16):
        lens = rng.integers(0, 4000, size=9).astype(np.int32)
        w = _wl(4, 2, 64, "bf16", lens=lens, seed=9)
        R = w.num_rows
        bits = rng.random((R, 2, words(w) * 32)) < 0.3
        sup = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(R, 2, -1).copy()
        modes = rng.choice([0, 1, 2, 3], size=R).astype(np.int8)
        shape, v = _compact(w, T, modes, sup)
        ref = O.compact_tiles(sup, modes, lens, 32)
        n = int(v["num_items"][0])
        S_max = -(-shape.max_blocks // T)
        fails = item_invariant_fails(v["items"][:n], v["head_info"], ref["lists"], T, S_max, lens,
                                     modes, 2, compact_slots=False)
        assert not fails, fails[:5]
        assert int(v["queue"][0]) == 0 and int(v["status"][0]) == 0
        for r in range(R):
            nb = -(-int(lens[r]) // 32)
            for g in range(2):
                hi = v["head_info"][r, g]
                assert hi[1] == -(-nb // T)  # one slot per range
                if modes[r] == W.MODE_SPARSE:
                    lst = ref["lists"][r][g]
                    for key in ("partial_ml", "partial_ml_1"):
                        ml = v[key][hi[0]:hi[0] + hi[1]]
                        for s_ in range(hi[1]):
                            if not np.any(lst // T == s_):
                                assert np.all(np.isneginf(ml[s_, :, 0])) and np.all(ml[s_, :, 1] == 0)


def test_compaction_items_depend_only_on_their_row():
    """A pair's items (as (range, slot, bitmap, count, length, flags)) are the
    same in a mixed batch as when its row is compacted alone."""
    rng = np.random.default_rng(15)
    lens = rng.integers(0, 3000, size=7).astype(np.int32)
    w = _wl(4, 2, 64, "bf16", lens=lens, seed=19)
    R = w.num_rows
    bits = rng.random((R, 2, words(w) * 32)) < 0.25
    sup = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(R, 2, -1).copy()
    modes = np.array([3, 0, 1, 3, 2, 3, 0], np.int8)
    for T in (2, 8):
        _, v = _compact(w, T, modes, sup)
        allrec = v["items"][:int(v["num_items"][0])]
        for r in range(R):
            # the same batch with every other row padding (length 0)
            solo = np.zeros_like(lens)
            solo[r] = lens[r]
            _, vs = _compact(w, T, modes, sup, lens=solo)
            one = vs["items"][:int(vs["num_items"][0])]
            for g in range(2):
                a = allrec[allrec[:, 0] == r * 2 + g]
                b = one[one[:, 0] == r * 2 + g]
                key = lambda x: x[np.lexsort((x[:, 1],))]
                assert np.array_equal(key(a), key(b)), (T, r, g)
                assert np.array_equal(v["head_info"][r, g], vs["head_info"][r, g])


def _list1_views(shape, ws):
    return {k: t.cpu() for k, t in W.workspace_views(shape, ws).items()}


@pytest.mark.parametrize("Hq,Hkv,lens", [(4, 4, RAGGED), (8, 2, RAGGED),
                                         (4, 2, np.array([10000, 5000, 1, 33, 0], np.int32))])
def test_finish_built_list_partitions_the_oracle_lists(Hq, Hkv, lens):
    """A finish with WISE_FLAG_BUILD_SPARSE_LIST writes list 1: for every row
    (discover rows from the mask the call writes, the other rows from the
    mask as it is) the items partition the oracle's compacted list of an
    all-sparse call on that mask, with compact slots, bucketed by tile count,
    taken in schedule order (larger buckets first)."""
    w = _wl(Hq, Hkv, 128, "bf16", lens=lens, seed=41)
    b = Batch(w)
    R = w.num_rows
    rng = np.random.default_rng(43)
    bits = rng.random((R, Hkv, words(w) * 32)) < 0.3
    sup_np = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(R, Hkv, -1).copy()
    modes_np = np.array([1, 2, 0, 3, 1, 2, 3, 1] * 2, np.int8)[:R]
    for T in (0, 2, 16):
        shape = shape_for(w, tiles_per_item=T)
        Tr = W.wise._tiles_per_item(shape)
        ws = W.alloc_workspace(shape)
        sup = dev_support(sup_np)
        modes = torch.from_numpy(modes_np).cuda()
        d = b.dev(0)
        out = torch.empty_like(d["q"])
        lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        W.wise_compact_tiles(shape, modes, b.seq_lens, sup, ws)
        W.wise_decode_partial(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                              modes, ws)
        W.wise_decode_finish_ex(shape, modes, b.seq_lens, ws, sup, out, lse,
                                flags=W.FLAG_BUILD_SPARSE_LIST)
        torch.cuda.synchronize()
        v = _list1_views(shape, ws)
        after = np_support(sup)
        ref = O.compact_tiles(after, np.full(R, W.MODE_SPARSE, np.int8), w.seq_lens, 32)
        sched = list1_schedule(v, Tr)
        S_max = -(-shape.max_blocks // Tr)
        fails = item_invariant_fails(sched, v["head_info_1"].numpy(), ref["lists"], Tr, S_max,
                                     w.seq_lens, None, Hkv, compact_slots=True)
        assert not fails, fails[:5]
        assert not v["list1_counter"][Tr:].any()
        # the call itself is unchanged by the flag
        g = gpu_call(b, 0, modes_np, sup_np, tiles_per_item=T)
        assert torch.equal(out.cpu(), g["out_raw"]) and np.array_equal(after, g["support"])


@pytest.mark.parametrize("Hq,Hkv,D,dtype", CASES)
def test_sparse_on_finish_built_list(Hq, Hkv, D, dtype):
    """The four-depth step the benchmark runs -- discover, union-discover
    building list 1, then two sparse depths on list 1 with no compaction --
    against the same calls each with its own compaction (bitwise: rows of at
    most 64 blocks merge their splits in the same order) and against the
    oracle."""
    w = _wl(Hq, Hkv, D, dtype)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    ws = W.alloc_workspace(shape)
    sup = dev_support(np.zeros((R, Hkv, words(w)), np.uint32))
    disc = torch.full((R,), W.MODE_DISCOVER, dtype=torch.int8, device="cuda")
    union = torch.full((R,), W.MODE_DISCOVER_UNION, dtype=torch.int8, device="cuda")
    sparse = torch.full((R,), W.MODE_SPARSE, dtype=torch.int8, device="cuda")
    outs = []
    for rep in range(2):  # the second step reuses the workspace as the benchmark does
        sup.zero_()
        outs = []
        for depth, m, flags, compact in ((0, disc, 0, True), (1, union, W.FLAG_BUILD_SPARSE_LIST, False),
                                         (2, sparse, W.FLAG_SPARSE_LIST, False),
                                         (0, sparse, W.FLAG_SPARSE_LIST, False)):
            d = b.dev(depth)
            out = torch.empty_like(d["q"])
            lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
            if compact:
                W.wise_compact_tiles(shape, m, b.seq_lens, sup, ws)
            pflags = flags & W.FLAG_SPARSE_LIST
            W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                     b.seq_lens, None if pflags else m, ws, pflags)
            W.wise_decode_finish_ex(shape, None if pflags else m, b.seq_lens, ws, sup, out, lse,
                                    flags=flags)
            torch.cuda.synchronize()
            outs.append((out.cpu(), lse.cpu().numpy(), np_support(sup)))
        assert int(W.workspace_views(shape, ws)["queue"].item()) == 0
    s0 = np.zeros((R, Hkv, words(w)), np.uint32)
    g0 = gpu_call(b, 0, np.full(R, 1, np.int8), s0)
    g1 = gpu_call(b, 1, np.full(R, 2, np.int8), g0["support"])
    g2 = gpu_call(b, 2, np.full(R, 3, np.int8), g1["support"])
    g3 = gpu_call(b, 0, np.full(R, 3, np.int8), g1["support"])
    for (out, lse, s_), g in zip(outs, (g0, g1, g2, g3)):
        assert torch.equal(out, g["out_raw"]) and np.array_equal(lse, g["lse"])
        assert np.array_equal(s_, g["support"])
    o = oracle_call(b, 2, np.full(R, 3, np.int8), g1["support"])
    assert not compare_outputs(w, g2, o)


def test_finish_built_list_long_rows_match_oracle():
    """Long rows (the clustered finish) through list 1: a union-discover
    finish builds it, a sparse call runs on it, against the oracle on the
    same mask, for a split of 16 tiles and of 1 (1024 ranges a pair)."""
    lens = np.array([20000, 3000, 0, 700, 17000], np.int32)
    w = _wl(8, 2, 128, "bf16", lens=lens, seed=47, n_planted=6)
    b = Batch(w)
    R = w.num_rows
    for T in (16, 1):
        shape = shape_for(w, tiles_per_item=T)
        ws = W.alloc_workspace(shape)
        g0 = gpu_call(b, 0, np.full(R, 1, np.int8), np.zeros((R, 2, words(w)), np.uint32))
        sup = dev_support(g0["support"])
        union = torch.full((R,), W.MODE_DISCOVER_UNION, dtype=torch.int8, device="cuda")
        d1, d2 = b.dev(1), b.dev(2)
        out = torch.empty_like(d1["q"])
        lse = torch.empty((R, 8), dtype=torch.float32, device="cuda")
        W.wise_compact_tiles(shape, union, b.seq_lens, sup, ws)
        W.wise_decode_partial(shape, d1["q"], d1["k_cache"], d1["v_cache"], b.page_table,
                              b.seq_lens, union, ws)
        W.wise_decode_finish_ex(shape, union, b.seq_lens, ws, sup, out, lse,
                                flags=W.FLAG_BUILD_SPARSE_LIST)
        out2 = torch.empty_like(d2["q"])
        lse2 = torch.empty_like(lse)
        W.wise_decode_partial_ex(shape, d2["q"], d2["k_cache"], d2["v_cache"], b.page_table,
                                 b.seq_lens, None, ws, W.FLAG_SPARSE_LIST)
        W.wise_decode_finish_ex(shape, None, b.seq_lens, ws, None, out2, lse2,
                                flags=W.FLAG_SPARSE_LIST)
        torch.cuda.synchronize()
        mask = np_support(sup)
        g = {"out": out2.double().cpu().numpy(), "lse": lse2.cpu().numpy()}
        o = oracle_call(b, 2, np.full(R, W.MODE_SPARSE, np.int8), mask)
        assert not compare_outputs(w, g, o)
        v = _list1_views(shape, ws)
        ref = O.compact_tiles(mask, np.full(R, 3, np.int8), w.seq_lens, 32)
        fails = item_invariant_fails(list1_schedule(v, T), v["head_info_1"].numpy(), ref["lists"],
                                     T, -(-shape.max_blocks // T), w.seq_lens, None, 2,
                                     compact_slots=True)
        assert not fails, fails[:5]


def test_all_selected_sparse_is_dense_bitwise():
    """[WISE PR, Tests]: with every block selected, sparse is bitwise dense."""
    w = _wl(4, 4, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    full = np.full((R, 4, words(w)), 0xFFFFFFFF, np.uint32)
    gd = gpu_call(b, 0, np.full(R, W.MODE_DENSE, np.int8), full)
    gs = gpu_call(b, 0, np.full(R, W.MODE_SPARSE, np.int8), full)
    gx = gpu_call(b, 0, np.full(R, W.MODE_DISCOVER, np.int8), full.copy())
    assert torch.equal(gd["out_raw"], gs["out_raw"]) and np.array_equal(gd["lse"], gs["lse"])
    assert torch.equal(gd["out_raw"], gx["out_raw"]) and np.array_equal(gd["lse"], gx["lse"])


def test_mixed_launch_equals_uniform_launches_bitwise():
    """One mixed-mode launch equals the uniform launches row for row, bitwise."""
    w = _wl(8, 2, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    rng = np.random.default_rng(11)
    bits = rng.random((R, 2, words(w) * 32)) < 0.4
    sup = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(R, 2, -1).copy()
    mixed = np.array([0, 3, 1, 2, 3, 0, 1, 3], np.int8)
    gm = gpu_call(b, 0, mixed, sup)
    for mode in (0, 1, 2, 3):
        gu = gpu_call(b, 0, np.full(R, mode, np.int8), sup)
        rows = np.nonzero(mixed == mode)[0]
        assert torch.equal(gm["out_raw"][rows], gu["out_raw"][rows])
        assert np.array_equal(gm["lse"][rows], gu["lse"][rows])
        assert np.array_equal(gm["support"][rows], gu["support"][rows])


def test_split_size_invariance():
    """Changing the work-item size only reorders fp32 sums."""
    w = _wl(4, 4, 128, "f32")
    b = Batch(w)
    R = w.num_rows
    zero = np.zeros((R, 4, words(w)), np.uint32)
    m = np.full(R, W.MODE_DENSE, np.int8)
    ref = gpu_call(b, 0, m, zero, tiles_per_item=8)
    for T in (1, 2, 16):
        g = gpu_call(b, 0, m, zero, tiles_per_item=T)
        assert np.max(np.abs(g["out"] - ref["out"])) < 1e-5
        fin = np.isfinite(ref["lse"])
        assert np.max(np.abs(g["lse"][fin] - ref["lse"][fin])) < 1e-5


def test_partial_reuses_a_compaction():
    """Two partial + finish passes over one compaction (the next depth reusing
    the same mask) give the same results as separate compactions."""
    w = _wl(4, 4, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    rng = np.random.default_rng(4)
    bits = rng.random((R, 4, words(w) * 32)) < 0.3
    sup = dev_support(np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(R, 4, -1))
    shape = shape_for(w)
    ws = W.alloc_workspace(shape)
    modes = torch.full((R,), W.MODE_SPARSE, dtype=torch.int8, device="cuda")
    W.wise_compact_tiles(shape, modes, b.seq_lens, sup, ws)
    outs = []
    for depth in (0, 1, 1):
        d = b.dev(depth)
        out = torch.empty_like(d["q"])
        lse = torch.empty((R, 4), dtype=torch.float32, device="cuda")
        W.wise_decode_partial(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                              modes, ws)
        W.wise_decode_finish(shape, modes, b.seq_lens, ws, sup, out, lse)
        outs.append((out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert int(W.workspace_views(shape, ws)["queue"].item()) == 0
    sup_np = np_support(sup)
    for depth, (out, lse) in zip((0, 1, 1), outs):
        ref = gpu_call(b, depth, np.full(R, W.MODE_SPARSE, np.int8), sup_np)
        assert torch.equal(out.cpu(), ref["out_raw"])
        assert np.array_equal(lse.cpu().numpy(), ref["lse"])


def test_one_call_entry_point_matches_stepwise():
    w = _wl(4, 4, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    zero = np.zeros((R, 4, words(w)), np.uint32)
    m = np.array([1, 1, 3, 0, 2, 1, 3, 1], np.int8)
    a = gpu_call(b, 0, m, zero, stepwise=True)
    c = gpu_call(b, 0, m, zero, stepwise=False)
    assert torch.equal(a["out_raw"], c["out_raw"]) and np.array_equal(a["support"], c["support"])


def test_padding_rows_and_empty_sparse_support():
    w = _wl(4, 4, 128, "bf16", lens=np.array([0, 64, 0, 100], np.int32))
    b = Batch(w)
    sup = np.zeros((4, 4, words(w)), np.uint32)
    sup[0] = 0xFFFFFFFF  # padding row: mask must stay untouched even when discovering
    sup[3, 1] = 0         # sparse row 3 head 1 selects nothing
    sup[3, [0, 2, 3]] = 0b101
    m = np.array([W.MODE_DISCOVER, W.MODE_SPARSE, W.MODE_DENSE, W.MODE_SPARSE], np.int8)
    g, o = gpu_call(b, 0, m, sup), oracle_call(b, 0, m, sup)
    assert not compare_outputs(w, g, o)
    assert np.all(g["out"][[0, 2]] == 0) and np.all(np.isneginf(g["lse"][[0, 2]]))
    assert np.all(g["out"][3, 1] == 0) and np.isneginf(g["lse"][3, 1])
    assert np.array_equal(g["support"][0], sup[0])


def test_support_union_kernel():
    rng = np.random.default_rng(2)
    for n in (1, 7, 4096 + 3):
        a = rng.integers(0, 2**32, size=n, dtype=np.uint32)
        c = rng.integers(0, 2**32, size=n, dtype=np.uint32)
        da, dc = dev_support(a), dev_support(c)
        W.wise_support_union(da, dc)
        torch.cuda.synchronize()
        assert np.array_equal(np_support(da), a | c)
    # the union of two discovery depths equals union-discover mode
    w = _wl(4, 4, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    zero = np.zeros((R, 4, words(w)), np.uint32)
    s0 = gpu_call(b, 0, np.full(R, 1, np.int8), zero)["support"]
    s1 = gpu_call(b, 1, np.full(R, 1, np.int8), zero)["support"]
    su = gpu_call(b, 1, np.full(R, 2, np.int8), s0)["support"]
    d0 = dev_support(s0)
    W.wise_support_union(d0, dev_support(s1))
    torch.cuda.synchronize()
    assert np.array_equal(np_support(d0), su)


def test_validate_reports_bad_batches():
    w = _wl(4, 4, 64, "bf16", lens=np.array([64, 100, 40, 33], np.int32))
    shape = shape_for(w)
    pt = w.page_table.copy()
    pt[1, 2] = w.num_pages + 5          # a page outside the pool
    lens = w.seq_lens.copy()
    lens[2] = 10**6                     # above the row capacity
    modes = np.array([0, 0, 0, 3], np.int8)
    sup = np.zeros((4, 4, words(w)), np.uint32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    W.wise_validate(shape, torch.from_numpy(pt).cuda(), torch.from_numpy(lens).cuda(),
                    torch.from_numpy(modes).cuda(), dev_support(sup), err)
    modes_bad = modes.copy()
    modes_bad[0] = 9
    W.wise_validate(shape, torch.from_numpy(w.page_table).cuda(), torch.from_numpy(w.seq_lens).cuda(),
                    torch.from_numpy(modes_bad).cuda(), dev_support(sup), err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & W.wise.BAD_PAGE and e & W.wise.BAD_SEQ_LEN and e & W.wise.EMPTY_SPARSE_SUPPORT
    assert e & W.wise.BAD_MODE


def test_seq_len_above_capacity_is_clamped_and_flagged():
    w = _wl(4, 4, 64, "bf16", lens=np.array([64, 100, 40, 33], np.int32))
    b = Batch(w)
    shape = shape_for(w)
    lens = w.seq_lens.copy()
    cap = min(w.max_blocks * 32, w.max_pages_per_row * w.page_size)
    lens[0] = cap + 1000
    ws = W.alloc_workspace(shape)
    modes = torch.zeros(4, dtype=torch.int8, device="cuda")
    W.wise_compact_tiles(shape, modes, torch.from_numpy(lens).cuda(), None, ws)
    torch.cuda.synchronize()
    v = W.workspace_views(shape, ws)
    assert int(v["status"].item()) & W.wise.DEVERR_SEQ_LEN_CLAMPED
    assert int(v["head_info"][0, 0, 2].item()) == -(-cap // 32)


# Long rows take the multi-warp finish kernel: one CTA of W warps per query
# head (4 up to 512 blocks, 8 up to 1024, 16 beyond), the KV head's query heads as one
# thread-block cluster; its sort keeps E = (padded block count) / (32 W) keys
# per thread.  One case per layout and cluster size.
LONG_CASES = [
    (2, 2, np.array([3000, 100, 0, 2049], np.int32)),         # G=1, 94 blocks: W=4, E=1
    (4, 2, np.array([10000, 5000, 1, 33], np.int32)),         # G=2, 313 blocks: W=4, E=4
    (4, 1, np.array([20000, 700, 9999], np.int32)),           # G=4, 625 blocks: W=8, E=4
    (8, 1, np.array([20000, 3000, 700, 100, 17000], np.int32)),  # G=8 (cluster of 8): W=8, E=4
]


@pytest.mark.parametrize("Hq,Hkv,lens", LONG_CASES)
def test_long_rows_match_oracle(Hq, Hkv, lens):
    w = _wl(Hq, Hkv, 128, "bf16", lens=lens, seed=11, n_planted=6)
    b = Batch(w)
    R = w.num_rows
    junk = np.random.default_rng(2).integers(0, 2**32, size=(R, Hkv, words(w)), dtype=np.uint32)
    m = np.full(R, W.MODE_DISCOVER, np.int8)
    g, o = gpu_call(b, 0, m, junk), oracle_call(b, 0, m, junk)
    assert not compare_outputs(w, g, o)
    cm = compare_masks(w, g["support"], o, m)
    assert not cm["fails"] and cm["checked"] > 0, cm
    s0 = o["support"]
    m = np.full(R, W.MODE_DISCOVER_UNION, np.int8)
    g, o = gpu_call(b, 1, m, s0), oracle_call(b, 1, m, s0)
    assert not compare_outputs(w, g, o)
    assert not compare_masks(w, g["support"], o, m, support_in=s0)["fails"]
    s1 = o["support"]
    m = np.array([W.MODE_SPARSE, W.MODE_DENSE] * R, np.int8)[:R]
    g, o = gpu_call(b, 2, m, s1), oracle_call(b, 2, m, s1)
    assert not compare_outputs(w, g, o)


@pytest.mark.parametrize("eta", [1e-13, 0.3, 0.95, 0.999, 1.0])
def test_long_row_selection_across_eta(eta):
    """Rows of 512 and more padded blocks select by the threshold search (no
    sort): against the oracle at every threshold, including the ends -- a
    vanishing eta keeps each query head's heaviest block only (the group's
    union of argmaxes), eta = 1 keeps every causal block."""
    lens = np.array([20000, 17000, 9000, 700], np.int32)
    w = _wl(8, 2, 128, "bf16", lens=lens, seed=53, n_planted=6)
    b = Batch(w)
    R = w.num_rows
    zero = np.zeros((R, 2, words(w)), np.uint32)
    m = np.full(R, W.MODE_DISCOVER, np.int8)
    g, o = gpu_call(b, 0, m, zero, eta=eta), oracle_call(b, 0, m, zero, eta=eta)
    assert not compare_outputs(w, g, o)
    cm = compare_masks(w, g["support"], o, m)
    assert not cm["fails"], cm
    for r in range(R):
        nb = -(-int(lens[r]) // 32)
        for g_ in range(2):
            bits = O.mask_bits(g["support"][r, g_], nb)
            if eta >= 1.0:
                assert bits.all()
            elif eta < 1e-9:
                # at most one block per query head, each within rounding of its head's maximum
                assert 1 <= bits.sum() <= 4
                heavy = np.zeros(nb, bool)
                for h in range(4 * g_, 4 * g_ + 4):
                    p = o["diag"][(r, h)]["p"]
                    heavy |= p >= p.max() * (1 - 1e-5)
                assert not np.any(bits & ~heavy)


@pytest.mark.parametrize("Hq,Hkv,D,dtype", CASES)
def test_folded_finish_matches_two_passes_bitwise(Hq, Hkv, D, dtype):
    """The partial pass with the finish folded in gives the partial + finish
    results bit for bit in every mode (padding rows, a garbage mask under
    discover, a sparse head selecting nothing), and leaves every ticket at 0."""
    w = _wl(Hq, Hkv, D, dtype)
    b = Batch(w)
    R = w.num_rows
    rng = np.random.default_rng(8)
    bits = rng.random((R, Hkv, words(w) * 32)) < 0.3
    sup = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(R, Hkv, -1).copy()
    sup[1, 0] = 0  # a sparse (row, KV head) selecting nothing
    mixed = np.array([W.MODE_SPARSE, W.MODE_DISCOVER, W.MODE_DENSE, W.MODE_DISCOVER_UNION] * 2,
                     np.int8)[:R]
    for m in [np.full(R, x, np.int8) for x in (0, 1, 2, 3)] + [mixed]:
        a = gpu_call(b, 0, m, sup, stepwise=True)
        f = gpu_call(b, 0, m, sup, fused=True)
        assert torch.equal(a["out_raw"], f["out_raw"]), m
        assert np.array_equal(a["lse"], f["lse"]), m
        assert np.array_equal(a["support"], f["support"]), m
        assert not f["ws"]["tickets"].any()
        assert int(f["ws"]["status"][0]) == 0


def test_folded_finish_reuses_a_compaction():
    """Three folded calls over one compaction (tickets back to 0 after each)
    match separate calls."""
    w = _wl(8, 2, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    rng = np.random.default_rng(6)
    bits = rng.random((R, 2, words(w) * 32)) < 0.4
    sup_np = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(R, 2, -1).copy()
    sup = dev_support(sup_np)
    shape = shape_for(w)
    ws = W.alloc_workspace(shape)
    modes = torch.full((R,), W.MODE_SPARSE, dtype=torch.int8, device="cuda")
    W.wise_compact_tiles(shape, modes, b.seq_lens, sup, ws)
    outs = []
    for depth in (0, 1, 2):
        d = b.dev(depth)
        out = torch.empty_like(d["q"])
        lse = torch.empty((R, 8), dtype=torch.float32, device="cuda")
        W.wise_decode_partial_finish(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                     b.seq_lens, modes, ws, sup, out, lse)
        outs.append((out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert not W.workspace_views(shape, ws)["tickets"].any()
    for depth, (out, lse) in zip((0, 1, 2), outs):
        ref = gpu_call(b, depth, np.full(R, W.MODE_SPARSE, np.int8), sup_np)
        assert torch.equal(out.cpu(), ref["out_raw"])
        assert np.array_equal(lse.cpu().numpy(), ref["lse"])


def test_folded_finish_matches_oracle():
    """Discover, union-discover and sparse through the folded path against the
    oracle (8 query heads per KV head: the tensor-core consumer folds too)."""
    for Hq, Hkv in ((4, 4), (8, 1)):
        w = _wl(Hq, Hkv, 128, "bf16", seed=21)
        b = Batch(w)
        R = w.num_rows
        sup = np.zeros((R, Hkv, words(w)), np.uint32)
        for depth, mode in enumerate((W.MODE_DISCOVER, W.MODE_DISCOVER_UNION, W.MODE_SPARSE)):
            m = np.full(R, mode, np.int8)
            g, o = gpu_call(b, depth, m, sup, fused=True), oracle_call(b, depth, m, sup)
            assert not compare_outputs(w, g, o)
            assert not compare_masks(w, g["support"], o, m, support_in=sup)["fails"]
            sup = o["support"]


def test_head_union_kernel_and_sparse_on_it():
    """The head union of a row's masks (bit-exact against the oracle), then a
    sparse call on the union against the oracle on the same mask."""
    rng = np.random.default_rng(12)
    for Hq, Hkv, lens in ((4, 4, RAGGED), (8, 2, np.array([3000, 100, 0, 2049], np.int32))):
        w = _wl(Hq, Hkv, 128, "bf16", lens=lens, seed=13)
        b = Batch(w)
        R = w.num_rows
        bits = rng.random((R, Hkv, words(w) * 32)) < 0.15
        sup_np = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(R, Hkv, -1).copy()
        sup = dev_support(sup_np)
        W.wise_support_head_union(shape_for(w), sup)
        torch.cuda.synchronize()
        u = np_support(sup)
        assert np.array_equal(u, O.support_head_union(sup_np))
        m = np.full(R, W.MODE_SPARSE, np.int8)
        g, o = gpu_call(b, 0, m, u), oracle_call(b, 0, m, u)
        assert not compare_outputs(w, g, o)


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(4, 4, 128, "bf16"), (8, 2, 128, "bf16"),
                                            (4, 1, 64, "bf16"), (2, 2, 64, "f32")])
def test_block_mass_from_lse_matches_oracle(Hq, Hkv, D, dtype):
    """Discovery without in-pass statistics: a dense call, the block masses
    rebuilt from its LSE by a second read of K, then the finish's selection;
    masses and masks against the oracle, outputs bitwise the dense call's."""
    w = _wl(Hq, Hkv, D, dtype)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    ws = W.alloc_workspace(shape)
    d = b.dev(0)
    sup = dev_support(np.zeros((R, Hkv, words(w)), np.uint32))
    dense = torch.zeros(R, dtype=torch.int8, device="cuda")
    disc_np = np.full(R, W.MODE_DISCOVER, np.int8)
    disc = torch.from_numpy(disc_np).cuda()
    out, out2 = torch.empty_like(d["q"]), torch.empty_like(d["q"])
    lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    lse2 = torch.empty_like(lse)
    W.wise_compact_tiles(shape, dense, b.seq_lens, sup, ws)
    W.wise_decode_partial(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens, dense, ws)
    W.wise_decode_finish(shape, dense, b.seq_lens, ws, sup, out, lse)
    W.wise_block_mass(shape, d["q"], d["k_cache"], b.page_table, b.seq_lens, disc, lse, ws)
    W.wise_decode_finish(shape, disc, b.seq_lens, ws, sup, out2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), out2.cpu()) and torch.equal(lse.cpu(), lse2.cpu())
    o = oracle_call(b, 0, disc_np, np.zeros((R, Hkv, words(w)), np.uint32))
    ts = W.workspace_views(shape, ws)["tile_stats"].cpu().numpy()
    lse_np = lse.cpu().numpy()
    for (r, h), dg in o["diag"].items():
        nb = dg["p"].shape[0]
        p_gpu = ts[r, h, :nb, 1] * np.exp2(ts[r, h, :nb, 0] - lse_np[r, h] / np.log(2.0))
        assert np.max(np.abs(p_gpu - dg["p"])) < 1e-5, (r, h)
    g = {"support": np_support(sup)}
    assert not compare_masks(w, g["support"], o, disc_np)["fails"]


def test_union_depth_reuses_the_discover_compaction():
    """A union-discover call over the discover call's compaction (the same
    work list: same lengths, no sparse row, statistics recorded in both)
    gives the results of its own compaction, bitwise."""
    w = _wl(4, 4, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    ws = W.alloc_workspace(shape)
    zero = np.zeros((R, 4, words(w)), np.uint32)
    sup = dev_support(zero)
    disc = torch.full((R,), W.MODE_DISCOVER, dtype=torch.int8, device="cuda")
    union = torch.full((R,), W.MODE_DISCOVER_UNION, dtype=torch.int8, device="cuda")
    W.wise_compact_tiles(shape, disc, b.seq_lens, sup, ws)
    res = []
    for depth, m in ((0, disc), (1, union)):
        d = b.dev(depth)
        out = torch.empty_like(d["q"])
        lse = torch.empty((R, 4), dtype=torch.float32, device="cuda")
        W.wise_decode_partial(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens, m, ws)
        W.wise_decode_finish(shape, m, b.seq_lens, ws, sup, out, lse)
        torch.cuda.synchronize()
        res.append((out.cpu(), lse.cpu().numpy(), np_support(sup)))
    g0 = gpu_call(b, 0, np.full(R, W.MODE_DISCOVER, np.int8), zero)
    g1 = gpu_call(b, 1, np.full(R, W.MODE_DISCOVER_UNION, np.int8), g0["support"])
    for (out, lse, s_), g in zip(res, (g0, g1)):
        assert torch.equal(out, g["out_raw"]) and np.array_equal(lse, g["lse"])
        assert np.array_equal(s_, g["support"])


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(4, 4, 128, "bf16"), (4, 4, 64, "bf16"),
                                            (8, 2, 128, "bf16"), (2, 2, 64, "f32")])
def test_page_size_32(Hq, Hkv, D, dtype):
    """32-token pages (one page per tile): every mode against the oracle, the
    ragged lengths, padding row and NaN-filled pool included."""
    w = _wl(Hq, Hkv, D, dtype, page_size=32, seed=31)
    b = Batch(w)
    R = w.num_rows
    sup = np.zeros((R, Hkv, words(w)), np.uint32)
    for depth, mode in enumerate((W.MODE_DISCOVER, W.MODE_DISCOVER_UNION, W.MODE_SPARSE)):
        m = np.full(R, mode, np.int8)
        g, o = gpu_call(b, depth, m, sup), oracle_call(b, depth, m, sup)
        assert not compare_outputs(w, g, o)
        assert not compare_masks(w, g["support"], o, m, support_in=sup)["fails"]
        sup = o["support"]
    m = np.zeros(R, np.int8)
    g, o = gpu_call(b, 0, m, sup), oracle_call(b, 0, m, sup)
    assert not compare_outputs(w, g, o)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_overlapped_depths_match_serial_calls(Hq, Hkv):
    """The benchmark's overlapped schedule -- alternating slot sets, the union
    and the second sparse depth reusing the previous compaction and starting
    while the previous finish runs -- gives the serial calls' results
    bitwise, every time over several back-to-back repetitions."""
    w = _wl(Hq, Hkv, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    ws = W.alloc_workspace(shape)
    modes = [W.MODE_DISCOVER, W.MODE_DISCOVER_UNION, W.MODE_SPARSE, W.MODE_SPARSE]
    mt = [torch.full((R,), m, dtype=torch.int8, device="cuda") for m in modes]
    # serial reference
    sup = np.zeros((R, Hkv, words(w)), np.uint32)
    ref = []
    for depth, m in enumerate(modes):
        g = gpu_call(b, depth % 3, np.full(R, m, np.int8), sup)
        ref.append(g)
        sup = g["support"]
    sup_t = dev_support(np.zeros((R, Hkv, words(w)), np.uint32))
    outs = [torch.empty_like(b.dev(depth % 3)["q"]) for depth in range(4)]
    lses = [torch.empty((R, Hq), dtype=torch.float32, device="cuda") for _ in range(4)]
    for rep in range(5):
        sup_t.zero_()
        for depth in range(4):
            d = b.dev(depth % 3)
            reuse = depth in (1, 3)
            flags = W.FLAG_SLOT_SET_1 if depth % 2 else 0
            if not reuse:
                W.wise_compact_tiles(shape, mt[depth], b.seq_lens, sup_t, ws)
            W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                     b.seq_lens, mt[depth], ws,
                                     flags | (W.FLAG_EARLY_START if reuse else 0))
            W.wise_decode_finish_ex(shape, mt[depth], b.seq_lens, ws, sup_t, outs[depth],
                                    lses[depth], flags)
        torch.cuda.synchronize()
        for depth in range(4):
            assert torch.equal(outs[depth].cpu(), ref[depth]["out_raw"]), (rep, depth)
            assert np.array_equal(lses[depth].cpu().numpy(), ref[depth]["lse"]), (rep, depth)
        assert np.array_equal(np_support(sup_t), ref[3]["support"])
    assert int(W.workspace_views(shape, ws)["queue"].item()) == 0


def test_compaction_beyond_cached_rounds():
    """More work units than the compaction keeps in registers (40 rows x 1024
    ranges of one block = 40,960 > 4 x 8192): the units past the cached rounds
    are looked up again; items, masks and outputs against the oracle."""
    rng = np.random.default_rng(23)
    lens = np.concatenate([[32768], rng.integers(0, 500, size=39)]).astype(np.int32)
    R = len(lens)
    w = custom_workload("units", R=R, Hq=1, Hkv=1, D=128, dtype="bf16", depths=2, n_planted=3,
                        seq_lens=lens, pool_factor=1, seed=29,
                        depth_modes=[np.zeros(R, np.int8)] * 2)
    assert w.max_blocks == 1024
    b = Batch(w)
    zero = np.zeros((R, 1, words(w)), np.uint32)
    m = np.array([W.MODE_DISCOVER, W.MODE_DENSE, W.MODE_DISCOVER_UNION, W.MODE_SPARSE] * 10, np.int8)
    prior = oracle_call(b, 1, np.full(R, W.MODE_DISCOVER, np.int8), zero)["support"]
    sup = np.where((m == W.MODE_SPARSE)[:, None, None], prior, zero)
    g, o = gpu_call(b, 0, m, sup, tiles_per_item=1), oracle_call(b, 0, m, sup)
    assert not compare_outputs(w, g, o)
    assert not compare_masks(w, g["support"], o, m, support_in=sup)["fails"]
    ref = O.compact_tiles(sup, m, lens, 32)
    v = {k: t.numpy() for k, t in g["ws"].items()}
    n = int(v["num_items"][0])
    fails = item_invariant_fails(v["items"][:n], v["head_info"], ref["lists"], 1, 1024, lens, m, 1,
                                 compact_slots=False)
    assert not fails, fails[:5]
