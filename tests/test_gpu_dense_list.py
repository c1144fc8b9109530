"""WISE_FLAG_DENSE_LIST: dense and discovery calls whose work list the passes
derive from the row lengths, with no compaction launch.

[WISE PR, "What changes"]: compaction exists for sparse rows; a row that
attends every block below its length has the ranges [s*T, s*T + T) of all its
blocks as its items.  So a call on the dense list must equal, bit for bit, the
same call after a compaction with every row dense or discovering (rows of at
most 64 blocks merge their splits in one order on both paths; longer rows too,
the slots being the same), and through it the oracle."""
import numpy as np
import pytest
import torch

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300.workload import custom_workload
from tests.gpu_harness import (Batch, compare_outputs, dev_support, gpu_call, np_support,
                               oracle_call, shape_for, words)

pytestmark = pytest.mark.gpu

RAGGED = np.array([1, 31, 32, 33, 300, 517, 0, 1024], np.int32)
CASES = [(4, 4, 128, "bf16"), (8, 2, 128, "bf16"), (4, 1, 64, "bf16"), (4, 2, 128, "f32")]


def _wl(Hq, Hkv, D, dtype, lens=RAGGED, seed=5, n_planted=3, page_size=16):
    R = len(lens)
    return custom_workload("dense-list", R=R, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, depths=3,
                           n_planted=n_planted, seq_lens=lens, pool_factor=2, seed=seed,
                           depth_modes=[np.zeros(R, np.int8)] * 3, page_size=page_size)


def _dense_call(b, depth, modes_np, sup, shape, ws, flags=0, finish_flags=0):
    """One call on the dense list (partial and finish); returns out and lse on
    the device."""
    w = b.w
    d = b.dev(depth)
    modes = torch.from_numpy(np.asarray(modes_np, np.int8)).cuda()
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.num_rows, w.num_q_heads), dtype=torch.float32, device="cuda")
    W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                             modes, ws, W.FLAG_DENSE_LIST | flags)
    W.wise_decode_finish_ex(shape, modes, b.seq_lens, ws, sup, out, lse,
                            flags=W.FLAG_DENSE_LIST | (flags & ~W.FLAG_INPUTS_READY) | finish_flags)
    return out, lse


def _fresh(shape):
    ws = W.alloc_workspace(shape)
    W.wise_workspace_reset(shape, ws)
    return ws


def _status(shape, ws):
    return int(W.workspace_views(shape, ws)["status"].item())


@pytest.mark.parametrize("ready", [False, True])
@pytest.mark.parametrize("T", [0, 1, 2, 16])
@pytest.mark.parametrize("Hq,Hkv,D,dtype", CASES)
def test_dense_list_equals_compaction_bitwise(Hq, Hkv, D, dtype, T, ready):
    """Every mode in one call: dense, discover and union rows as after a
    compaction; a sparse row on the dense list attends all its blocks, so it
    equals the same row in dense mode, and its mask is left as it is.  With
    WISE_FLAG_INPUTS_READY the pass reads its inputs before the dependency
    wait; the result is the same."""
    w = _wl(Hq, Hkv, D, dtype)
    b = Batch(w)
    R = w.num_rows
    rng = np.random.default_rng(7)
    sup_np = rng.integers(0, 2**32, size=(R, Hkv, words(w)), dtype=np.uint32)
    modes_np = np.array([1, 2, 0, 3, 1, 2, 3, 1], np.int8)
    shape = shape_for(w, tiles_per_item=T)
    ws = _fresh(shape)
    sup = dev_support(sup_np)
    for rep in range(2):  # a reused workspace: the pass leaves its queue counters at 0
        sup.copy_(dev_support(sup_np))
        out, lse = _dense_call(b, 0, modes_np, sup, shape, ws,
                               flags=W.FLAG_INPUTS_READY if ready else 0)
        torch.cuda.synchronize()
        as_dense = np.where(modes_np == W.MODE_SPARSE, W.MODE_DENSE, modes_np).astype(np.int8)
        g = gpu_call(b, 0, as_dense, sup_np, tiles_per_item=T)
        assert torch.equal(out.cpu(), g["out_raw"]), rep
        assert np.array_equal(lse.cpu().numpy(), g["lse"]), rep
        assert np.array_equal(np_support(sup), g["support"]), rep
        v = W.workspace_views(shape, ws)
        assert int(v["queue"].item()) == 0 and _status(shape, ws) == 0


@pytest.mark.parametrize("Hq,Hkv,D,dtype", CASES)
def test_step_without_compaction(Hq, Hkv, D, dtype):
    """The benchmark's WISE step with no compaction launch: discover on the
    dense list, union-discover on the dense list building list 1, two sparse
    depths on list 1 (the second reading early); twice on one workspace.
    Bitwise against the same calls each after its own compaction, and depth 2
    against the oracle."""
    w = _wl(Hq, Hkv, D, dtype)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    ws = _fresh(shape)
    sup = dev_support(np.zeros((R, Hkv, words(w)), np.uint32))
    outs = []
    for rep in range(2):
        sup.zero_()
        outs = []
        # The second call on list 1 reads the list and its inputs before the
        # dependency wait (both complete before the kernel ahead of it began).
        for depth, mode, kind in ((0, W.MODE_DISCOVER, "dense"), (1, W.MODE_DISCOVER_UNION, "build"),
                                  (2, W.MODE_SPARSE, "list1"), (0, W.MODE_SPARSE, "list1-ready")):
            m = np.full(R, mode, np.int8)
            if kind.startswith("list1"):
                d = b.dev(depth)
                out = torch.empty_like(d["q"])
                lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
                pf = W.FLAG_SPARSE_LIST | (W.FLAG_INPUTS_READY if kind == "list1-ready" else 0)
                W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                         b.seq_lens, None, ws, pf)
                W.wise_decode_finish_ex(shape, None, b.seq_lens, ws, sup, out, lse,
                                        flags=W.FLAG_SPARSE_LIST)
            else:
                out, lse = _dense_call(b, depth, m, sup, shape, ws, flags=W.FLAG_INPUTS_READY,
                                       finish_flags=W.FLAG_BUILD_SPARSE_LIST if kind == "build" else 0)
            torch.cuda.synchronize()
            outs.append((out.cpu(), lse.cpu().numpy(), np_support(sup)))
        v = W.workspace_views(shape, ws)
        assert int(v["queue"].item()) == 0 and _status(shape, ws) == 0
    s0 = np.zeros((R, Hkv, words(w)), np.uint32)
    g0 = gpu_call(b, 0, np.full(R, 1, np.int8), s0)
    g1 = gpu_call(b, 1, np.full(R, 2, np.int8), g0["support"])
    g2 = gpu_call(b, 2, np.full(R, 3, np.int8), g1["support"])
    g3 = gpu_call(b, 0, np.full(R, 3, np.int8), g1["support"])
    for i, ((out, lse, s_), g) in enumerate(zip(outs, (g0, g1, g2, g3))):
        assert torch.equal(out, g["out_raw"]) and np.array_equal(lse, g["lse"]), i
        assert np.array_equal(s_, g["support"]), i
    o = oracle_call(b, 2, np.full(R, 3, np.int8), g1["support"])
    assert not compare_outputs(w, g2, o)


def test_dense_step_on_one_workspace():
    """The dense baseline's four depths on the dense list, one after another
    on one workspace, against the oracle."""
    w = _wl(8, 2, 128, "bf16", seed=9)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    ws = _fresh(shape)
    zero = np.zeros((R, 2, words(w)), np.uint32)
    dense = np.zeros(R, np.int8)
    for depth in (0, 1, 2, 0):
        out, lse = _dense_call(b, depth, dense, None, shape, ws, flags=W.FLAG_INPUTS_READY)
        torch.cuda.synchronize()
        g = {"out": out.double().cpu().numpy(), "lse": lse.cpu().numpy()}
        assert not compare_outputs(w, g, oracle_call(b, depth, dense, zero)), depth


@pytest.mark.parametrize("R", [33, 97, 256])
def test_row_table_many_rows(R):
    """The pass tabulates each row's first item in chunks of 32 rows: row
    counts across several chunks up to the maximum, with empty rows leading,
    trailing and in runs (an empty row shares its first item with the next
    row).  Bitwise against the compaction path; sampled rows against the
    oracle."""
    rng = np.random.default_rng(R)
    lens = rng.integers(1, 700, size=R).astype(np.int32)
    lens[:3] = 0
    lens[-4:] = 0
    lens[R // 2:R // 2 + 5] = 0
    lens[R // 3] = 2048
    w = _wl(4, 2, 64, "bf16", lens=lens, seed=R + 1)
    b = Batch(w)
    modes_np = rng.choice(np.array([0, 1, 2], np.int8), size=R)
    sup_np = np.zeros((R, 2, words(w)), np.uint32)
    for T in (0, 1):
        shape = shape_for(w, tiles_per_item=T)
        ws = _fresh(shape)
        sup = dev_support(sup_np)
        out, lse = _dense_call(b, 1, modes_np, sup, shape, ws)
        torch.cuda.synchronize()
        g = gpu_call(b, 1, modes_np, sup_np, tiles_per_item=T)
        assert torch.equal(out.cpu(), g["out_raw"]) and np.array_equal(lse.cpu().numpy(), g["lse"])
        assert np.array_equal(np_support(sup), g["support"])
    rows = np.unique(np.concatenate([[0, 3, R // 3, R // 2 + 5, R - 5, R - 1],
                                     rng.choice(R, size=10, replace=False)]))
    o = oracle_call(b, 1, modes_np, sup_np, rows=rows)
    assert not compare_outputs(w, g, o, rows=rows)


def test_all_rows_empty():
    """No row holds a token: the list is empty, every output 0 with LSE -inf,
    and the masks of discovering rows are left as they are."""
    lens = np.zeros(5, np.int32)
    w = _wl(4, 4, 128, "bf16", lens=lens)
    b = Batch(w)
    shape = shape_for(w)
    ws = _fresh(shape)
    sup_np = np.full((5, 4, words(w)), 0xA5A5A5A5, np.uint32)
    sup = dev_support(sup_np)
    out, lse = _dense_call(b, 0, np.array([1, 2, 0, 1, 2], np.int8), sup, shape, ws)
    torch.cuda.synchronize()
    assert not out.float().abs().sum().item()
    assert np.all(np.isneginf(lse.cpu().numpy()))
    assert np.array_equal(np_support(sup), sup_np)
    assert int(W.workspace_views(shape, ws)["queue"].item()) == 0


def test_status_is_cleared_and_clamping_flagged():
    """The dense-list pass clears the status word (compaction does that on
    the other path), and flags a length above the row capacity, which it
    clamps as compaction does."""
    w = _wl(4, 4, 64, "bf16", lens=np.array([64, 100, 40, 33], np.int32))
    b = Batch(w)
    shape = shape_for(w)
    ws = _fresh(shape)
    cap = min(w.max_blocks * 32, w.max_pages_per_row * w.page_size)
    lens = w.seq_lens.copy()
    lens[0] = cap + 1000
    modes = np.zeros(4, np.int8)
    W.wise_compact_tiles(shape, torch.from_numpy(modes).cuda(), torch.from_numpy(lens).cuda(),
                         None, ws)
    torch.cuda.synchronize()
    assert _status(shape, ws) & W.wise.DEVERR_SEQ_LEN_CLAMPED
    _dense_call(b, 0, modes, None, shape, ws)
    torch.cuda.synchronize()
    assert _status(shape, ws) == 0
    d = b.dev(0)
    out = torch.empty_like(d["q"])
    lse = torch.empty((4, 4), dtype=torch.float32, device="cuda")
    lt = torch.from_numpy(lens).cuda()
    mt = torch.from_numpy(modes).cuda()
    # row 0 reads up to its capacity: every page-table entry a pool page
    pt = w.page_table.copy()
    pt[0] = np.arange(pt.shape[1]) % w.num_pages
    W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], torch.from_numpy(pt).cuda(),
                             lt, mt, ws, W.FLAG_DENSE_LIST)
    W.wise_decode_finish_ex(shape, mt, lt, ws, None, out, lse, flags=W.FLAG_DENSE_LIST)
    torch.cuda.synchronize()
    assert _status(shape, ws) & W.wise.DEVERR_SEQ_LEN_CLAMPED
    # the clamped row is the row at capacity: its rows 1..3 unchanged
    ref, _ = _dense_call(b, 0, modes, None, shape, _fresh(shape))
    torch.cuda.synchronize()
    assert torch.equal(out[1:].cpu(), ref[1:].cpu())
    assert torch.isfinite(out[0].float()).all()


def test_slot_set_1():
    """The dense list with the workspace's second slot set."""
    w = _wl(4, 2, 128, "bf16")
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    ws = _fresh(shape)
    sup_np = np.zeros((R, 2, words(w)), np.uint32)
    sup = dev_support(sup_np)
    m = np.full(R, W.MODE_DISCOVER, np.int8)
    out, lse = _dense_call(b, 0, m, sup, shape, ws, flags=W.FLAG_SLOT_SET_1)
    torch.cuda.synchronize()
    g = gpu_call(b, 0, m, sup_np)
    assert torch.equal(out.cpu(), g["out_raw"]) and np.array_equal(lse.cpu().numpy(), g["lse"])
    assert np.array_equal(np_support(sup), g["support"])


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(4, 4, 128, "bf16"), (8, 2, 128, "bf16"),
                                           (2, 2, 64, "f32")])
def test_page_size_32(Hq, Hkv, D, dtype):
    """32-token pages (one page per tile): the compaction-free step (dense list
    with early reads, list 1 built by the union finish, a sparse depth on it)
    against the same calls after their own compaction, bit for bit, and the
    sparse depth against the oracle."""
    w = _wl(Hq, Hkv, D, dtype, page_size=32, seed=33)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    ws = _fresh(shape)
    sup = dev_support(np.zeros((R, Hkv, words(w)), np.uint32))
    got = []
    for depth, mode in ((0, W.MODE_DISCOVER), (1, W.MODE_DISCOVER_UNION), (2, W.MODE_SPARSE)):
        m = np.full(R, mode, np.int8)
        if mode == W.MODE_SPARSE:
            d = b.dev(depth)
            out = torch.empty_like(d["q"])
            lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
            W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                     b.seq_lens, None, ws, W.FLAG_SPARSE_LIST)
            W.wise_decode_finish_ex(shape, None, b.seq_lens, ws, sup, out, lse,
                                    flags=W.FLAG_SPARSE_LIST)
        else:
            out, lse = _dense_call(b, depth, m, sup, shape, ws, flags=W.FLAG_INPUTS_READY,
                                   finish_flags=W.FLAG_BUILD_SPARSE_LIST if depth == 1 else 0)
        torch.cuda.synchronize()
        got.append((out.cpu(), lse.cpu().numpy(), np_support(sup)))
    s0 = np.zeros((R, Hkv, words(w)), np.uint32)
    g0 = gpu_call(b, 0, np.full(R, 1, np.int8), s0)
    g1 = gpu_call(b, 1, np.full(R, 2, np.int8), g0["support"])
    g2 = gpu_call(b, 2, np.full(R, 3, np.int8), g1["support"])
    for i, ((out, lse, s_), g) in enumerate(zip(got, (g0, g1, g2))):
        assert torch.equal(out, g["out_raw"]) and np.array_equal(lse, g["lse"]), i
        assert np.array_equal(s_, g["support"]), i
    o = oracle_call(b, 2, np.full(R, 3, np.int8), g1["support"])
    assert not compare_outputs(w, g2, o)
    assert _status(shape, ws) == 0


def test_workspace_state_across_call_kinds():
    """One workspace through a sequence of every kind of call -- dense list,
    compaction, list 1 built and used (also read early), the dense list again,
    a compaction-based sparse call between -- each output and mask bit for bit
    the same as that call made alone on a fresh workspace after its own
    compaction: no queue, counter or list state leaks from one call into the
    next."""
    w = _wl(4, 2, 128, "bf16", seed=35)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    ws = _fresh(shape)
    sup = dev_support(np.zeros((R, 2, words(w)), np.uint32))
    D_, DU, DS, SP = W.MODE_DISCOVER, W.MODE_DISCOVER_UNION, W.MODE_DENSE, W.MODE_SPARSE

    def step(depth, mode, kind):
        m = np.full(R, mode, np.int8)
        mt = torch.from_numpy(m).cuda()
        d = b.dev(depth)
        out = torch.empty_like(d["q"])
        lse = torch.empty((R, 4), dtype=torch.float32, device="cuda")
        sup_in = np_support(sup)
        if kind.startswith("dense"):
            fflags = W.FLAG_BUILD_SPARSE_LIST if kind == "dense+build" else 0
            out, lse = _dense_call(b, depth, m, sup, shape, ws, flags=W.FLAG_INPUTS_READY,
                                   finish_flags=fflags)
        elif kind.startswith("list1"):
            pf = W.FLAG_SPARSE_LIST | (W.FLAG_INPUTS_READY if kind == "list1-ready" else 0)
            W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                     b.seq_lens, None, ws, pf)
            W.wise_decode_finish_ex(shape, None, b.seq_lens, ws, sup, out, lse,
                                    flags=W.FLAG_SPARSE_LIST)
        else:  # compaction, then the two passes (the finish may build list 1)
            W.wise_compact_tiles(shape, mt, b.seq_lens, sup, ws)
            W.wise_decode_partial(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                  b.seq_lens, mt, ws)
            W.wise_decode_finish_ex(shape, mt, b.seq_lens, ws, sup, out, lse,
                                    flags=W.FLAG_BUILD_SPARSE_LIST if kind == "compact+build" else 0)
        torch.cuda.synchronize()
        g = gpu_call(b, depth, m, sup_in)  # alone, on a fresh workspace
        assert torch.equal(out.cpu(), g["out_raw"]), (depth, mode, kind)
        assert np.array_equal(lse.cpu().numpy(), g["lse"]), (depth, mode, kind)
        assert np.array_equal(np_support(sup), g["support"]), (depth, mode, kind)

    for depth, mode, kind in ((0, D_, "dense"), (1, DU, "compact+build"), (2, SP, "list1"),
                              (0, DS, "dense"), (1, SP, "compact"), (2, DU, "dense+build"),
                              (0, SP, "list1"), (1, SP, "list1-ready"), (2, D_, "compact"),
                              (0, DU, "dense")):
        step(depth, mode, kind)
        v = W.workspace_views(shape, ws)
        assert int(v["queue"].item()) == 0 and _status(shape, ws) == 0, (depth, mode, kind)


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(4, 4, 128, "bf16"), (8, 2, 128, "bf16"),
                                           (4, 2, 128, "f32")])
def test_early_start_on_alternate_slot_sets(Hq, Hkv, D, dtype):
    """The step as the benchmark overlaps it: depths on alternate slot sets,
    the dense-list depths and the second list-1 depth starting beside the
    previous finish (WISE_FLAG_EARLY_START with WISE_FLAG_INPUTS_READY), three
    steps queued back to back with no synchronisation: every depth's output,
    LSE and mask bit for bit those of the serial step."""
    w = _wl(Hq, Hkv, D, dtype, seed=37)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    plan = ((0, W.MODE_DISCOVER, "dense"), (1, W.MODE_DISCOVER_UNION, "build"),
            (2, W.MODE_SPARSE, "list1"), (0, W.MODE_SPARSE, "list1-ready"))
    modes = {mode: torch.full((R,), mode, dtype=torch.int8, device="cuda") for _, mode, _ in plan}

    def run_step(ws, sup, early):
        outs = []
        for t, (depth, mode, kind) in enumerate(plan):
            sset = W.FLAG_SLOT_SET_1 if (early and t % 2) else 0
            e = W.FLAG_EARLY_START if early else 0
            d = b.dev(depth)
            out = torch.empty_like(d["q"])
            lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
            m = modes[mode]
            if kind.startswith("list1"):
                pf = W.FLAG_SPARSE_LIST | sset
                if kind == "list1-ready":
                    pf |= W.FLAG_INPUTS_READY | e
                W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                         b.seq_lens, None, ws, pf)
                W.wise_decode_finish_ex(shape, None, b.seq_lens, ws, sup, out, lse,
                                        flags=W.FLAG_SPARSE_LIST | sset)
            else:
                W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                         b.seq_lens, m, ws,
                                         W.FLAG_DENSE_LIST | W.FLAG_INPUTS_READY | sset | e)
                ff = W.FLAG_DENSE_LIST | sset | (W.FLAG_BUILD_SPARSE_LIST if kind == "build" else 0)
                W.wise_decode_finish_ex(shape, m, b.seq_lens, ws, sup, out, lse, flags=ff)
            if not early:
                torch.cuda.synchronize()
            outs.append((out, lse))
        return outs

    ref_ws = _fresh(shape)
    ref_sup = dev_support(np.zeros((R, Hkv, words(w)), np.uint32))
    ref = run_step(ref_ws, ref_sup, early=False)
    torch.cuda.synchronize()
    ws = _fresh(shape)
    sup = dev_support(np.zeros((R, Hkv, words(w)), np.uint32))
    for _ in range(3):
        got = run_step(ws, sup, early=True)
    torch.cuda.synchronize()
    for i, ((o, l), (ro, rl)) in enumerate(zip(got, ref)):
        assert torch.equal(o.cpu(), ro.cpu()) and torch.equal(l.cpu(), rl.cpu()), i
    assert np.array_equal(np_support(sup), np_support(ref_sup))
    assert int(W.workspace_views(shape, ws)["queue"].item()) == 0 and _status(shape, ws) == 0
