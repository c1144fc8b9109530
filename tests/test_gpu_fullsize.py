"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (default split size, the four-depth schedule), against the
oracle on every row or on a sample of rows it computes one by one.

Masks are chained the way an engine chains them: each depth's GPU call gets
the GPU's own mask from the previous depth, and the oracle is run on the same
input mask, so every comparison is like for like."""
import numpy as np
import pytest

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300.workload import make_workload
from oracle import wise_oracle as O
from tests.gpu_harness import (Batch, compare_masks, compare_outputs, gpu_call, oracle_call,
                               words)

pytestmark = pytest.mark.gpu


def _check_depth(b, depth, modes, sup_in, rows=None, eta=None):
    w = b.w
    g = gpu_call(b, depth, modes, sup_in, eta=eta)
    o = oracle_call(b, depth, modes, sup_in, eta=eta, rows=rows)
    fails = compare_outputs(w, g, o, rows=rows)
    cm = compare_masks(w, g["support"], o, modes, rows=rows, support_in=sup_in)
    fails += cm["fails"]
    assert not fails, fails[:5]
    assert int(g["ws"]["status"][0]) == 0
    return g, o, cm


def _pipeline(name, rows=None):
    w = make_workload(name)
    b = Batch(w)
    sup = np.zeros((w.num_rows, w.num_kv_heads, words(w)), np.uint32)
    stats = []
    for depth in range(w.num_depths):
        modes = w.depth_modes[depth]
        g, o, cm = _check_depth(b, depth, modes, sup, rows=rows)
        print(f"{name} depth {depth}: masks bit-exact {cm['checked']}, bounds-checked near the "
              f"margin {cm['excluded_margin']}, near a mass tie {cm['excluded_gap']}")
        stats.append(cm)
        sup = g["support"]
    return w, sup, stats


def test_ouro_1k_full_pipeline():
    """64 rows x 1024 tokens, 16 heads, four depths, every row checked."""
    w, sup, stats = _pipeline("ouro1.4b_1k")
    assert stats[0]["checked"] >= 0.95 * (stats[0]["checked"] + stats[0]["excluded"])
    dens = O.union_density(sup, w.seq_lens, 32)
    assert 0.1 < dens < 0.3
    # the planted blocks are in the reused union
    hits = np.mean([set(w.planted[r][h]).issubset(np.nonzero(O.mask_bits(sup[r, h], 32))[0].tolist())
                    for r in range(w.num_rows) for h in range(w.num_kv_heads)])
    assert hits >= 0.99


def test_ouro_4k_full_pipeline_sampled():
    """64 rows x 4096 tokens over a 2x oversized shuffled pool; the GPU runs
    every row, the oracle checks 12 of them."""
    w = make_workload("ouro1.4b_4k")
    b = Batch(w)
    rows = np.array([0, 5, 11, 17, 23, 29, 35, 41, 47, 53, 59, 63])
    sup = np.zeros((w.num_rows, w.num_kv_heads, words(w)), np.uint32)
    for depth in range(3):
        g, _, _ = _check_depth(b, depth, w.depth_modes[depth], sup, rows=rows)
        sup = g["support"]


def test_mixed_8k_full():
    """32 ragged rows up to 8192 tokens, per-row modes; sparse rows use the
    support of a prior discovery of the same inputs."""
    w = make_workload("mixed_8k")
    b = Batch(w)
    zero = np.zeros((w.num_rows, w.num_kv_heads, words(w)), np.uint32)
    prior = gpu_call(b, 0, np.full(w.num_rows, W.MODE_DISCOVER, np.int8), zero)["support"]
    modes = w.depth_modes[0]
    assert set(np.unique(modes)) == {W.MODE_DENSE, W.MODE_DISCOVER, W.MODE_SPARSE}
    _check_depth(b, 0, modes, prior)


@pytest.mark.parametrize("eta", [0.8, 0.9, 0.95, 0.99])
def test_gqa_32k_discover_eta_sweep(eta):
    """8 rows x 32768 tokens, 32 query / 8 KV heads (1024 blocks per mask)."""
    w = make_workload("gqa_32k", eta=eta)
    b = Batch(w)
    zero = np.zeros((w.num_rows, w.num_kv_heads, words(w)), np.uint32)
    g, o, cm = _check_depth(b, 0, w.depth_modes[0], zero, eta=eta)
    print(f"gqa_32k eta {eta}: masks bit-exact {cm['checked']}, bounds-checked near the margin "
          f"{cm['excluded_margin']}, near a mass tie {cm['excluded_gap']}")
    assert cm["checked"] > 0


def test_gqa_32k_pipeline():
    w = make_workload("gqa_32k")
    b = Batch(w)
    sup = np.zeros((w.num_rows, w.num_kv_heads, words(w)), np.uint32)
    for depth in range(3):
        g, _, _ = _check_depth(b, depth, w.depth_modes[depth], sup)
        sup = g["support"]
