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
