"""Sanity of the synthetic recipe (not parity): at the Ouro-1.4B 1K shape the
oracle's eta=0.95 discovery recovers the planted blocks, and the support is
sparse, as the recipe intends."""
import numpy as np
import torch

from block_sparse_paged_split_gb300.workload import make_workload
from oracle import wise_oracle as O
from tests.oracle_pins import as_oracle_array


def test_planted_blocks_are_discovered():
    w = make_workload("ouro1.4b_1k", num_rows=4)
    d = w.depth_inputs(0)
    sup = np.zeros((w.num_rows, w.num_kv_heads, -(-w.max_blocks // 32)), np.uint32)
    res = O.decode_layer(as_oracle_array(d["q"]), as_oracle_array(d["k_cache"]),
                         as_oracle_array(d["v_cache"]), w.page_table, w.seq_lens,
                         w.depth_modes[0], sup, eta=w.eta)
    hits = [set(w.planted[r][h]).issubset(np.nonzero(dg["sel"])[0].tolist())
            for (r, h), dg in res["diag"].items()]
    assert np.mean(hits) >= 0.99
    dens = O.union_density(res["support"], w.seq_lens, w.tile_tokens)
    assert 0.1 < dens < 0.3


def test_workload_is_deterministic_and_poisoned_outside_rows():
    a = make_workload("mixed_8k", num_rows=3, context=2048)
    b = make_workload("mixed_8k", num_rows=3, context=2048)
    assert np.array_equal(a.page_table, b.page_table) and np.array_equal(a.seq_lens, b.seq_lens)
    da, db = a.depth_inputs(0), b.depth_inputs(0)
    assert da["k_cache"].view(torch.int16).equal(db["k_cache"].view(torch.int16))
    # token slots past each row's length hold NaN
    P = a.page_size
    for r, L in enumerate(a.seq_lens):
        if L % P:
            last = a.page_table[r, L // P]
            assert da["k_cache"][last, L % P:].float().isnan().all()


def test_sparse_scaling_inputs():
    """The sparse-scaling inputs: every (row, head) mask holds exactly k
    distinct blocks below the row's block count, the page table is a
    permutation of the pool, and a seed fixes the draw."""
    from block_sparse_paged_split_gb300.workload import sparse_scaling_inputs
    for L, k in ((1000, 5), (4096, 8), (2048, 64), (96, 9)):
        d = sparse_scaling_inputs(3, 2, 64, L, k, seed=11, device="cpu")
        nb = -(-L // 32)
        words = d["support"].numpy().view(np.uint32)
        bits = np.unpackbits(words.view(np.uint8), axis=-1, bitorder="little")
        assert np.all(bits.sum(-1) == min(k, nb))
        assert not bits[..., nb:].any()
        pt = d["page_table"].numpy().ravel()
        assert np.array_equal(np.sort(pt), np.arange(d["num_pages"]))
        assert d["max_blocks"] == nb and d["k_cache"].shape[0] == d["num_pages"]
        again = sparse_scaling_inputs(3, 2, 64, L, k, seed=11, device="cpu")
        assert torch.equal(again["support"], d["support"]) and torch.equal(again["k_cache"], d["k_cache"])
