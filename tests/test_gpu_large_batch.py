"""Batches past the dense list's row limit (600 rows, more than
WISE_DENSE_LIST_MAX_ROWS): the three depths of a recurrent step as an engine
runs them at that size -- discover on a compaction, union-discover whose
finish also builds the sparse depths' work list over every (row, KV head),
sparse on that list -- with ragged lengths (empty rows among them), grouped
query heads, and a variant with one long row, so the finish takes its
clustered long-row kernel.  Sampled rows of every depth against the oracle
(each depth given the mask the GPU left before it), list 1 against the
oracle's compacted tile lists, and the dense list refused for such a batch
before anything launches."""
import numpy as np
import pytest
import torch

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300.workload import custom_workload
from oracle import wise_oracle as O
from tests.gpu_harness import (Batch, compare_masks, compare_outputs, dev_support,
                               item_invariant_fails, list1_schedule, np_support, oracle_call,
                               shape_for, words)

pytestmark = pytest.mark.gpu

R, HQ, HKV, D = 600, 4, 2, 64


def _workload(long_row: bool):
    rng = np.random.default_rng(41)
    lens = rng.integers(1, 700, size=R).astype(np.int32)
    lens[::13] = 0  # padding rows
    lens[5] = 32    # exactly one block
    if long_row:
        lens[7] = 4096  # 128 blocks: every row then goes through the long-row finish
    modes = [np.full(R, m, np.int8) for m in (W.MODE_DISCOVER, W.MODE_DISCOVER_UNION, W.MODE_SPARSE)]
    w = custom_workload("large_batch", R=R, Hq=HQ, Hkv=HKV, D=D, dtype="bf16", depths=3,
                        n_planted=3, seq_lens=lens, pool_factor=1, seed=43, depth_modes=modes)
    rows = np.unique(np.concatenate([[0, 5, 7, 13, R - 1], rng.choice(R, size=19, replace=False)]))
    return w, rows


@pytest.mark.parametrize("long_row", [False, True])
def test_large_batch_step(long_row):
    w, rows = _workload(long_row)
    assert w.num_rows > W.DENSE_LIST_MAX_ROWS
    b = Batch(w)
    shape = shape_for(w)
    T = W.wise._tiles_per_item(shape)
    ws = W.alloc_workspace(shape)
    W.wise_workspace_reset(shape, ws)
    sup = dev_support(np.zeros((R, HKV, words(w)), np.uint32))
    snaps = []
    for depth, flags in ((0, 0), (1, W.FLAG_BUILD_SPARSE_LIST), (2, W.FLAG_SPARSE_LIST)):
        d = b.dev(depth)
        modes = torch.from_numpy(w.depth_modes[depth]).cuda()
        before = np_support(sup)
        out = torch.empty_like(d["q"])
        lse = torch.empty((R, HQ), dtype=torch.float32, device="cuda")
        if depth < 2:
            W.wise_compact_tiles(shape, modes, b.seq_lens, sup, ws)
        W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                                 modes, ws, flags & W.FLAG_SPARSE_LIST)
        W.wise_decode_finish_ex(shape, modes, b.seq_lens, ws, sup, out, lse, flags)
        torch.cuda.synchronize()
        views = {k: v.cpu() for k, v in W.workspace_views(shape, ws).items()}
        assert int(views["status"][0]) == 0, depth
        snaps.append({"sup_in": before, "out": out.double().cpu().numpy(), "lse": lse.cpu().numpy(),
                      "support": np_support(sup), "ws": views})
    # every depth's sampled rows against the oracle on the same input mask
    checked = 0
    for depth, s in enumerate(snaps):
        modes = w.depth_modes[depth]
        o = oracle_call(b, depth, modes, s["sup_in"], rows=rows)
        fails = compare_outputs(w, s, o, rows=rows)
        cm = compare_masks(w, s["support"], o, modes, rows=rows, support_in=s["sup_in"])
        fails += cm["fails"]
        assert not fails, (depth, fails[:5])
        checked += cm["checked"]
    assert checked > 0
    # padding rows: output 0, LSE -inf, mask untouched (all zero)
    pad = w.seq_lens == 0
    for s in snaps:
        assert np.all(s["out"][pad] == 0) and np.all(np.isneginf(s["lse"][pad]))
    assert not snaps[-1]["support"][pad].any()
    # list 1, built by the union depth's finish, partitions the oracle's
    # compacted tile lists of the mask it left, for every (row, KV head)
    v = snaps[1]["ws"]
    ref = O.compact_tiles(snaps[1]["support"], np.full(R, W.MODE_SPARSE, np.int8), w.seq_lens, 32)
    fails = item_invariant_fails(list1_schedule(v, T), v["head_info_1"].numpy(), ref["lists"], T,
                                 -(-shape.max_blocks // T), w.seq_lens, None, HKV,
                                 compact_slots=True)
    assert not fails, fails[:5]


def test_large_batch_refuses_the_dense_list():
    """The dense list's row table holds at most DENSE_LIST_MAX_ROWS rows: a
    larger batch is refused (unsupported) before any launch, and the
    workspace is left as it was."""
    w, _ = _workload(False)
    b = Batch(w)
    shape = shape_for(w)
    ws = W.alloc_workspace(shape)
    W.wise_workspace_reset(shape, ws)
    torch.cuda.synchronize()
    snapshot = ws.clone()
    d = b.dev(0)
    modes = torch.from_numpy(w.depth_modes[0]).cuda()
    with pytest.raises(W.wise.WiseError) as err:
        W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                                 modes, ws, W.FLAG_DENSE_LIST)
    assert err.value.status == 2  # WISE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.equal(ws, snapshot)
