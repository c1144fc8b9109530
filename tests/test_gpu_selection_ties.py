"""Exact ties in block mass at the cutoff, on long rows (the threshold
selection of rows with 512 or more padded blocks) and on short ones: inputs
are built so that whole groups of blocks hold the same keys, hence the same
tile statistics and the same mass to the last bit.  The eta rule orders equal
masses by the lower block index [WISE PR, Tests: "the reference rule"], so
the kept blocks are known in closed form; the oracle agrees, and so must the
kernel, bit for bit."""
import math

import numpy as np
import pytest
import torch

import block_sparse_paged_split_gb300 as W
from oracle import wise_oracle as O

pytestmark = pytest.mark.gpu


def _case(nb, G, heavy_every, seed):
    """One row of nb blocks (32 tokens each), G query heads on one KV head
    (all with the same query, so every head ties at the same places),
    D=128, bf16: every block repeats the same 32 keys, except that blocks with
    index % heavy_every == 0 (heavy_every > 0) repeat a second set of keys
    pulled towards the query."""
    rng = np.random.default_rng(seed)
    D, P, L = 128, 16, nb * 32
    q = np.repeat(rng.standard_normal((1, 1, D)).astype(np.float32), G, axis=1)
    base = rng.standard_normal((32, D)).astype(np.float32)
    boost = base + 0.5 * q[0].mean(axis=0)
    K = np.tile(base, (nb, 1))
    if heavy_every:
        for b in range(0, nb, heavy_every):
            K[b * 32:(b + 1) * 32] = boost
    V = rng.standard_normal((L, D)).astype(np.float32)
    npg = L // P
    perm = rng.permutation(npg).astype(np.int32)
    k_cache = np.zeros((npg, P, 1, D), np.float32)
    v_cache = np.zeros((npg, P, 1, D), np.float32)
    k_cache[perm] = K.reshape(npg, P, 1, D)
    v_cache[perm] = V.reshape(npg, P, 1, D)
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)  # noqa: E731
    return {"q": bf(q), "k": bf(k_cache), "v": bf(v_cache), "page_table": perm[None, :].copy(),
            "seq_lens": np.array([L], np.int32), "G": G, "nb": nb}


def _run(c, eta):
    G, nb = c["G"], c["nb"]
    shape = W.make_shape(num_rows=1, num_q_heads=G, num_kv_heads=1, head_dim=128, page_size=16,
                         max_pages_per_row=c["page_table"].shape[1], num_pages=c["k"].shape[0],
                         max_blocks=nb, eta=eta)
    Wd = -(-nb // 32)
    sup = torch.zeros((1, 1, Wd), dtype=torch.int32, device="cuda")
    out = torch.empty((1, G, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, G), dtype=torch.float32, device="cuda")
    W.wise_decode(shape, c["q"].cuda(), c["k"].cuda(), c["v"].cuda(),
                  torch.from_numpy(c["page_table"]).cuda(), torch.from_numpy(c["seq_lens"]).cuda(),
                  torch.full((1,), W.MODE_DISCOVER, dtype=torch.int8, device="cuda"), sup, out, lse,
                  W.alloc_workspace(shape))
    torch.cuda.synchronize()
    got = O.mask_bits(sup.cpu().numpy().view(np.uint32)[0, 0], nb)
    as_u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    ref = O.decode_layer(as_u16(c["q"]), as_u16(c["k"]), as_u16(c["v"]), c["page_table"],
                         c["seq_lens"], np.array([W.MODE_DISCOVER], np.int8),
                         np.zeros((1, 1, Wd), np.uint32), eta=eta)
    return got, O.mask_bits(ref["support"][0, 0], nb), ref


@pytest.mark.parametrize("nb,G", [(1000, 1), (1000, 4), (600, 2), (60, 1)])
def test_all_masses_tied(nb, G):
    """Every block has the same mass 1/nb: the rule keeps the first
    ceil(eta * nb) blocks by index (eta chosen away from a multiple of 1/nb)."""
    c = _case(nb, G, 0, seed=nb + G)
    k = int(0.4 * nb) + 1
    eta = (k - 0.5) / nb
    got, ref, _ = _run(c, eta)
    want = np.zeros(nb, bool)
    want[:k] = True
    assert np.array_equal(ref, want)
    assert np.array_equal(got, want), (np.nonzero(got ^ want)[0][:10])


@pytest.mark.parametrize("nb,G", [(1000, 4), (800, 1), (50, 2)])
def test_cutoff_inside_a_tie_group(nb, G):
    """Heavy blocks (every 7th) all tie, light blocks all tie; eta falls
    inside the light group: every heavy block is kept, then light blocks in
    index order, exactly as many as the masses require."""
    c = _case(nb, G, 7, seed=3 * nb + G)
    _, ref_bits, ref = _run(c, 0.5)
    p = ref["diag"][(0, 0)]["p"]
    heavy = np.arange(nb) % 7 == 0
    ph, pl = p[heavy][0], p[~heavy][0]
    assert np.allclose(p[heavy], ph) and np.allclose(p[~heavy], pl) and ph > pl
    # eta half a light block past the middle of the light group
    n_light = int((~heavy).sum()) // 2
    eta = float(heavy.sum() * ph + (n_light - 0.5) * pl)
    got, ref_bits, _ = _run(c, eta)
    want = heavy.copy()
    want[np.nonzero(~heavy)[0][:n_light]] = True
    assert np.array_equal(ref_bits, want)
    assert np.array_equal(got, want), (np.nonzero(got ^ want)[0][:10])
