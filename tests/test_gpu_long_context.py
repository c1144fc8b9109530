"""Rows past 32K tokens, up to the 4096-block (128K-token) limit: mask rows of
up to 128 words, up to 512 split slots a (row, KV head), and the finish's
16-warp selection (2048 and 4096 padded keys, by the threshold search).
Both consumer paths (FMA for one query head a KV head, tensor cores for four),
the three depths of a recurrent step (discover on a compaction,
union-discover building list 1, sparse on list 1) against the oracle on
every row, and all-blocks sparse bitwise equal to dense."""
import numpy as np
import pytest
import torch

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300.workload import custom_workload
from oracle import wise_oracle as O
from tests.gpu_harness import (Batch, compare_masks, compare_outputs, dev_support, gpu_call,
                               item_invariant_fails, list1_schedule, np_support, oracle_call,
                               shape_for, words)

pytestmark = pytest.mark.gpu

# lengths and eta: 4096 blocks (4096 padded keys) at eta 0.95; 1536 blocks
# (2048 padded keys) at eta 0.5, so the sparse depth reads a real subset
CASES = {"128k": (np.array([131072, 65553, 0, 40001], np.int32), 0.95),
         "48k": (np.array([49152, 1, 33000], np.int32), 0.5)}


def _workload(Hq, Hkv, which, seed=53):
    lens, eta = CASES[which]
    R = len(lens)
    modes = [np.full(R, m, np.int8) for m in (W.MODE_DISCOVER, W.MODE_DISCOVER_UNION, W.MODE_SPARSE)]
    return custom_workload("long_context", R=R, Hq=Hq, Hkv=Hkv, D=128, dtype="bf16", depths=3,
                           n_planted=16, seq_lens=lens, pool_factor=1, seed=seed, depth_modes=modes,
                           eta=eta)


@pytest.mark.parametrize("which", ["128k", "48k"])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 1)])
def test_long_rows_step(Hq, Hkv, which):
    w = _workload(Hq, Hkv, which)
    assert w.max_blocks > 1024
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    T = W.wise._tiles_per_item(shape)
    ws = W.alloc_workspace(shape)
    W.wise_workspace_reset(shape, ws)
    sup = dev_support(np.zeros((R, Hkv, words(w)), np.uint32))
    union_views = None
    for depth, flags in ((0, 0), (1, W.FLAG_BUILD_SPARSE_LIST), (2, W.FLAG_SPARSE_LIST)):
        d = b.dev(depth)
        modes_np = w.depth_modes[depth]
        modes = torch.from_numpy(modes_np).cuda()
        before = np_support(sup)
        out = torch.empty_like(d["q"])
        lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        if depth < 2:
            W.wise_compact_tiles(shape, modes, b.seq_lens, sup, ws)
        W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                                 modes, ws, flags & W.FLAG_SPARSE_LIST)
        W.wise_decode_finish_ex(shape, modes, b.seq_lens, ws, sup, out, lse, flags)
        torch.cuda.synchronize()
        views = {k: v.cpu() for k, v in W.workspace_views(shape, ws).items()}
        assert int(views["status"][0]) == 0, depth
        g = {"out": out.double().cpu().numpy(), "lse": lse.cpu().numpy(), "support": np_support(sup)}
        o = oracle_call(b, depth, modes_np, before)
        fails = compare_outputs(w, g, o)
        fails += compare_masks(w, g["support"], o, modes_np, support_in=before)["fails"]
        assert not fails, (depth, fails[:5])
        if depth == 1:
            union_views = views
            union_mask = g["support"]
    # list 1 partitions the oracle's compacted tile lists of the union mask
    ref = O.compact_tiles(union_mask, np.full(R, W.MODE_SPARSE, np.int8), w.seq_lens, 32)
    fails = item_invariant_fails(list1_schedule(union_views, T), union_views["head_info_1"].numpy(),
                                 ref["lists"], T, -(-shape.max_blocks // T), w.seq_lens, None, Hkv,
                                 compact_slots=True)
    assert not fails, fails[:5]


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 1)])
def test_long_rows_all_selected_sparse_is_dense(Hq, Hkv):
    """Every block selected: the sparse call's items, slots and arithmetic are
    the dense call's, so outputs and LSEs are equal bit for bit."""
    w = _workload(Hq, Hkv, "128k")
    b = Batch(w)
    R = w.num_rows
    full = np.zeros((R, Hkv, words(w)), np.uint32)
    for r in range(R):
        nb = -(-int(w.seq_lens[r]) // 32)
        for blk in range(nb):
            full[r, :, blk >> 5] |= np.uint32(1 << (blk & 31))
    dense = gpu_call(b, 0, np.full(R, W.MODE_DENSE, np.int8), full)
    sparse = gpu_call(b, 0, np.full(R, W.MODE_SPARSE, np.int8), full)
    assert torch.equal(dense["out_raw"], sparse["out_raw"])
    assert np.array_equal(dense["lse"], sparse["lse"])
    assert np.array_equal(sparse["support"], full)  # sparse leaves the mask alone
