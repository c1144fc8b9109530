"""Checks that pin the CPU oracle to things other than itself.

Each `pin_*` function takes the oracle *module* and returns a list of failure
messages (empty = the pin holds).  Taking the module lets the mutation tests
plant a mistake in a private copy of the oracle and confirm some pin catches it.

What the pins compare against:
  * library routines in float64 (torch scaled_dot_product_attention, softmax,
    logsumexp, amax; numpy unpackbits);
  * attention written out token by token in plain Python floats (tiny inputs);
  * brute force over every subset of block masses;
  * exact closed-form selections (tests/golden/selection_cases.json);
  * the pages' density example (tests/golden/union_density_example.json);
  * a hand-worked head-union example (tests/golden/head_union_example.json);
  * invariances the pages state: all-blocks sparse is dense bitwise, block
    masses from the LSE equal softmax block sums, the union equals the OR of
    per-depth selections; and the page layout and the page size cannot matter.

An oracle that computes in float32 carries its own TOLERANCES (see
F32_TOLERANCES); the float64 oracles use the module's.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from typing import List

import numpy as np
import torch
import torch.nn.functional as F

from block_sparse_paged_split_gb300.workload import (MODE_DENSE, MODE_DISCOVER,
                                                     MODE_DISCOVER_UNION, MODE_SPARSE,
                                                     custom_workload)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def as_oracle_array(t: torch.Tensor) -> np.ndarray:
    """torch CPU tensor -> the array form the oracle takes (bf16 as uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.contiguous().numpy()


def make_case(Hq, Hkv, D, dtype, lens, seed, pool_factor=2, n_planted=2):
    lens = np.asarray(lens, np.int32)
    w = custom_workload(R=len(lens), Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, depths=1,
                        n_planted=n_planted, seq_lens=lens, pool_factor=pool_factor,
                        seed=seed, depth_modes=[np.zeros(len(lens), np.int8)])
    return w, w.depth_inputs(0, logical=True)


def run(O, w, d, modes, support, eta=0.95, page_table=None, k_cache=None, v_cache=None):
    return O.decode_layer(as_oracle_array(d["q"]),
                          as_oracle_array(d["k_cache"] if k_cache is None else k_cache),
                          as_oracle_array(d["v_cache"] if v_cache is None else v_cache),
                          w.page_table if page_table is None else page_table,
                          w.seq_lens, np.asarray(modes, np.int8), support, eta=eta,
                          tile_tokens=w.tile_tokens)


def empty_support(w) -> np.ndarray:
    return np.zeros((w.num_rows, w.num_kv_heads, -(-w.max_blocks // 32)), np.uint32)


def random_support(w, seed, density=0.4) -> np.ndarray:
    rng = np.random.default_rng(seed)
    W = -(-w.max_blocks // 32)
    bits = rng.random((w.num_rows, w.num_kv_heads, W * 32)) < density
    return np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(
        w.num_rows, w.num_kv_heads, W).copy()


# Float64 tolerances.  An oracle that computes in float32 carries its own
# `TOLERANCES` (the same keys), derived from its measured distance to float64.
TOLERANCES = {"out_rtol": 1e-10, "out_atol": 1e-12, "lse": 1e-10, "mass": 1e-12,
              "tile_max": 1e-12, "mass_sum": 1e-12, "tile_lse": 1e-10, "cutoff_band": 1e-9}


# For the fp32 oracle: measured against the float64 oracle on MHA and GQA
# batches up to 4096 tokens, its worst errors are 1.4e-6 (output), 2.4e-6 (LSE),
# 9e-7 (block mass), 2.2e-6 (tile max), 1.9e-6 (sum of masses - 1); each bound
# below leaves about ten times that.  A cumulative fp32 sum of masses carries
# up to ~1e-6, so selections whose cutoff lies that close to eta are skipped.
F32_TOLERANCES = {"out_rtol": 1e-5, "out_atol": 2e-5, "lse": 2e-5, "mass": 1e-5,
                  "tile_max": 2e-5, "mass_sum": 2e-5, "tile_lse": 2e-5, "cutoff_band": 2e-6}


def tol(O, key: str) -> float:
    return getattr(O, "TOLERANCES", TOLERANCES)[key]


def library_bits(words: np.ndarray, nb: int) -> np.ndarray:
    """Mask bits decoded by numpy's unpackbits (little-endian words)."""
    return np.unpackbits(np.ascontiguousarray(words, dtype="<u4").view(np.uint8),
                         bitorder="little")[:nb].astype(bool)


def _ref_row(d, r, g, h):
    K = d["k_rows"][r][:, g, :].double()
    V = d["v_rows"][r][:, g, :].double()
    q = d["q"][r, h].double()
    return q, K, V


def _sdpa(q, K, V, scale, mask=None):
    am = None if mask is None else torch.as_tensor(mask)[None, None, None, :]
    return F.scaled_dot_product_attention(q[None, None, None, :], K[None, None], V[None, None],
                                          attn_mask=am, scale=scale)[0, 0, 0]


# ----------------------------------------------------------------------------------- pins
def pin_dense_sdpa(O) -> List[str]:
    """Dense output equals torch SDPA (float64), LSE equals torch.logsumexp of the
    scaled scores; MHA and GQA, fp32 and bf16 storage, ragged lengths."""
    fails = []
    for (Hq, Hkv, D, dt, lens, seed) in [(2, 2, 64, "f32", [70, 33, 96, 1, 0], 11),
                                         (4, 2, 128, "bf16", [100, 31, 64], 12)]:
        w, d = make_case(Hq, Hkv, D, dt, lens, seed)
        res = run(O, w, d, [MODE_DENSE] * len(lens), empty_support(w))
        scale = 1.0 / math.sqrt(D)
        G = Hq // Hkv
        for r, L in enumerate(lens):
            for h in range(Hq):
                if L == 0:
                    if not (np.all(res["out"][r, h] == 0) and res["lse"][r, h] == -math.inf):
                        fails.append(f"padding row {r} head {h} not zero/-inf")
                    continue
                q, K, V = _ref_row(d, r, h // G, h)
                o = _sdpa(q, K, V, scale).numpy()
                lse = torch.logsumexp(scale * torch.mv(K, q), 0).item()
                if not np.allclose(res["out"][r, h], o, rtol=tol(O, "out_rtol"),
                                   atol=tol(O, "out_atol")):
                    fails.append(f"dense out differs r={r} h={h}")
                if abs(res["lse"][r, h] - lse) > tol(O, "lse"):
                    fails.append(f"dense lse differs r={r} h={h}")
    return fails


def pin_sparse_masked_sdpa(O) -> List[str]:
    """Sparse output equals SDPA under the boolean tile mask [WISE PR, Tests:
    sparse output matches masked attention]; an empty support gives 0/-inf."""
    fails = []
    for (Hq, Hkv, D, dt, lens, seed) in [(2, 2, 64, "f32", [200, 65, 130, 31], 21),
                                         (4, 2, 128, "bf16", [250, 96], 22)]:
        w, d = make_case(Hq, Hkv, D, dt, lens, seed)
        sup = random_support(w, seed)
        sup[0, 0, :] = 0  # one (row, head) with nothing selected
        res = run(O, w, d, [MODE_SPARSE] * len(lens), sup)
        scale = 1.0 / math.sqrt(D)
        G = Hq // Hkv
        for r, L in enumerate(lens):
            nb = -(-L // w.tile_tokens)
            for h in range(Hq):
                g = h // G
                blocks = library_bits(sup[r, g], nb)
                mask = np.repeat(blocks, w.tile_tokens)[:L]
                if not mask.any():
                    if not (np.all(res["out"][r, h] == 0) and res["lse"][r, h] == -math.inf):
                        fails.append(f"empty support r={r} h={h} not zero/-inf")
                    continue
                q, K, V = _ref_row(d, r, g, h)
                o = _sdpa(q, K, V, scale, mask).numpy()
                s = scale * torch.mv(K, q)
                lse = torch.logsumexp(s[torch.from_numpy(mask)], 0).item()
                if not np.allclose(res["out"][r, h], o, rtol=tol(O, "out_rtol"),
                                   atol=tol(O, "out_atol")):
                    fails.append(f"sparse out differs r={r} h={h}")
                if abs(res["lse"][r, h] - lse) > tol(O, "lse"):
                    fails.append(f"sparse lse differs r={r} h={h}")
    return fails


def pin_sparse_bruteforce_loops(O) -> List[str]:
    """Sparse (and dense) attention written out token by token in plain
    Python floats on tiny inputs: s_j = scale * sum_d q_d k_jd over the
    tokens of the selected blocks only, m = max s_j, Z = sum exp(s_j - m),
    o_d = sum exp(s_j - m) v_jd / Z, lse = m + log Z [WISE PR, Tests: sparse
    output matches masked attention]."""
    fails = []
    lens = [70, 33, 96]
    w, d = make_case(2, 1, 16, "f32", lens, 27)
    sup = random_support(w, 3, density=0.5)
    for mode in (MODE_SPARSE, MODE_DENSE):
        res = run(O, w, d, [mode] * len(lens), sup)
        scale = 1.0 / math.sqrt(16)
        for r, L in enumerate(lens):
            K = d["k_rows"][r][:, 0, :].tolist()
            V = d["v_rows"][r][:, 0, :].tolist()
            words = [int(x) for x in sup[r, 0]]
            active = [mode == MODE_DENSE or (words[(j // 32) // 32] >> ((j // 32) % 32)) & 1
                      for j in range(L)]
            for h in range(2):
                q = d["q"][r, h].tolist()
                s = [scale * sum(q[i] * K[j][i] for i in range(16)) for j in range(L)]
                act = [j for j in range(L) if active[j]]
                if not act:
                    if res["lse"][r, h] != -math.inf:
                        fails.append(f"empty selection r={r} h={h} has an LSE")
                    continue
                m = max(s[j] for j in act)
                e = {j: math.exp(s[j] - m) for j in act}
                Z = sum(e[j] for j in act)
                o = [sum(e[j] * V[j][i] for j in act) / Z for i in range(16)]
                lse = m + math.log(Z)
                if max(abs(a - b) for a, b in zip(o, res["out"][r, h])) > tol(O, "out_atol") + \
                        tol(O, "out_rtol") * max(abs(x) for x in o):
                    fails.append(f"mode {mode} out differs from the loops r={r} h={h}")
                if abs(lse - res["lse"][r, h]) > tol(O, "lse"):
                    fails.append(f"mode {mode} lse differs from the loops r={r} h={h}")
    return fails


def pin_all_blocks_sparse_is_dense(O) -> List[str]:
    """Every block selected: sparse equals dense bitwise [WISE PR, Tests:
    compaction with every block selected is bitwise dense]."""
    w, d = make_case(4, 2, 128, "bf16", [130, 64, 33], 31)
    full = np.full_like(empty_support(w), 0xFFFFFFFF)
    dense = run(O, w, d, [MODE_DENSE] * 3, empty_support(w))
    sparse = run(O, w, d, [MODE_SPARSE] * 3, full)
    if not (np.array_equal(dense["out"], sparse["out"]) and np.array_equal(dense["lse"], sparse["lse"])):
        return ["all-blocks sparse differs from dense"]
    return []


def pin_paging_invariance(O) -> List[str]:
    """Moving pages around the pool (and adding NaN-filled pages no row
    references) leaves every output bitwise unchanged."""
    w, d = make_case(2, 2, 64, "f32", [90, 17, 48], 41, pool_factor=1)
    base = run(O, w, d, [MODE_DENSE, MODE_DISCOVER, MODE_DENSE], empty_support(w))
    rng = np.random.default_rng(5)
    n = w.num_pages
    new_n = 3 * n
    where = rng.permutation(new_n)[:n]          # old page p -> new page where[p]
    kc = torch.full((new_n,) + tuple(d["k_cache"].shape[1:]), float("nan"), dtype=d["k_cache"].dtype)
    vc = kc.clone()
    kc[torch.from_numpy(where)] = d["k_cache"]
    vc[torch.from_numpy(where)] = d["v_cache"]
    pt = np.where(w.page_table >= 0, where[np.maximum(w.page_table, 0)], -1).astype(np.int32)
    moved = run(O, w, d, [MODE_DENSE, MODE_DISCOVER, MODE_DENSE], empty_support(w),
                page_table=pt, k_cache=kc, v_cache=vc)
    fails = []
    for key in ("out", "lse", "support"):
        if not np.array_equal(base[key], moved[key]):
            fails.append(f"page layout changed {key}")
    return fails


def pin_page_size_invariance(O) -> List[str]:
    """The same logical rows paged in 16-token and in 32-token pages (each a
    seeded permutation of its own pool) give bitwise the same outputs, LSEs
    and masks in every mode: the page size only changes where a token is
    stored, never the arithmetic."""
    fails = []
    lens = np.array([70, 33, 96, 1, 0, 64], np.int32)
    modes = np.array([MODE_DENSE, MODE_DISCOVER, MODE_SPARSE, MODE_DISCOVER_UNION, MODE_SPARSE,
                      MODE_DISCOVER], np.int8)
    res = []
    for P in (16, 32):
        w = custom_workload(R=len(lens), Hq=4, Hkv=2, D=64, dtype="f32", depths=1, n_planted=1,
                            seq_lens=lens, pool_factor=2, seed=43, page_size=P,
                            depth_modes=[modes])
        d = w.depth_inputs(0)
        sup = random_support(w, 7, density=0.5)
        res.append(O.decode_layer(as_oracle_array(d["q"]), as_oracle_array(d["k_cache"]),
                                  as_oracle_array(d["v_cache"]), w.page_table, w.seq_lens, modes,
                                  sup, eta=0.9, tile_tokens=32))
    for key in ("out", "lse", "support"):
        if not np.array_equal(res[0][key], res[1][key]):
            fails.append(f"page size 16 vs 32 changed {key}")
    return fails


def pin_block_masses(O) -> List[str]:
    """Per-tile stats and block masses against library softmax/logsumexp:
    m_b = amax over the tile; p_b = sum of the tile's softmax probabilities;
    sum_b p_b = 1; logsumexp_b(m_b + log l_b) = LSE; and the LSE-derived mass
    l_b * exp(m_b - LSE) equals p_b [WISE PR, Tests: LSE-derived block mass
    matches softmax block sums]."""
    fails = []
    w, d = make_case(4, 2, 64, "f32", [200, 47, 32, 1], 51)
    res = run(O, w, d, [MODE_DISCOVER] * 4, empty_support(w))
    scale = 1.0 / math.sqrt(w.head_dim)
    B = w.tile_tokens
    for (r, h), dg in res["diag"].items():
        L = int(w.seq_lens[r])
        q, K, _ = _ref_row(d, r, h // w.group, h)
        s = scale * torch.mv(K, q)
        prob = torch.softmax(s, 0)
        nb = -(-L // B)
        for b in range(nb):
            blk = slice(b * B, min((b + 1) * B, L))
            if abs(dg["p"][b] - prob[blk].sum().item()) > tol(O, "mass"):
                fails.append(f"p_b != softmax block sum r={r} h={h} b={b}")
            if abs(dg["m_b"][b] - torch.amax(s[blk]).item()) > tol(O, "tile_max"):
                fails.append(f"m_b != amax r={r} h={h} b={b}")
            lse_mass = dg["l_b"][b] * math.exp(dg["m_b"][b] - res["lse"][r, h])
            if abs(lse_mass - dg["p"][b]) > tol(O, "mass"):
                fails.append(f"LSE-derived mass differs r={r} h={h} b={b}")
        if abs(dg["p"].sum() - 1.0) > tol(O, "mass_sum"):
            fails.append(f"masses do not sum to 1 r={r} h={h}")
        blk_lse = torch.logsumexp(torch.tensor(dg["m_b"] + np.log(dg["l_b"])), 0).item()
        if abs(blk_lse - res["lse"][r, h]) > tol(O, "tile_lse"):
            fails.append(f"logsumexp of tile stats != lse r={r} h={h}")
    return fails


def _brute_force_k(p: np.ndarray, eta: float):
    n = p.shape[0]
    for k in range(1, n + 1):
        best = max(sum(p[list(c)]) for c in itertools.combinations(range(n), k))
        if best >= eta:
            return k, best
    return n, p.sum()


def pin_selection_bruteforce(O) -> List[str]:
    """Over every subset: k* is the least size of any block set whose mass
    reaches eta, and the chosen set has the largest mass of that size."""
    fails = []
    rng = np.random.default_rng(61)
    for trial in range(150):
        n = int(rng.integers(1, 11))
        p = rng.dirichlet(np.full(n, rng.uniform(0.2, 3.0))).astype(np.float32).astype(np.float64)
        eta = float(rng.uniform(0.05, 0.999))
        C = np.cumsum(np.sort(p)[::-1])
        if np.any(np.abs(C - eta) < tol(O, "cutoff_band")):
            continue
        k, best = _brute_force_k(p, eta)
        got = O.select_blocks(p, eta)
        if got["k"] != k or int(got["sel"].sum()) != k:
            fails.append(f"trial {trial}: k*={got['k']} brute force {k}")
        elif abs(p[got["sel"]].sum() - best) > 1e-12:
            fails.append(f"trial {trial}: chosen mass {p[got['sel']].sum()} < best {best}")
    return fails


def pin_selection_golden(O) -> List[str]:
    with open(os.path.join(GOLDEN, "selection_cases.json")) as f:
        cases = json.load(f)["cases"]
    fails = []
    for c in cases:
        got = O.select_blocks(np.array(c["p"], np.float64), c["eta"])
        if sorted(np.nonzero(got["sel"])[0].tolist()) != c["selected"]:
            fails.append(f"golden p={c['p']} eta={c['eta']}: got {np.nonzero(got['sel'])[0].tolist()}")
    return fails


def pin_selection_limits(O) -> List[str]:
    """eta = 1 takes every block; a tiny eta takes exactly the arg-max block
    (lowest index among equal maxima); a larger eta never takes fewer blocks."""
    fails = []
    rng = np.random.default_rng(71)
    for trial in range(100):
        n = int(rng.integers(1, 40))
        p = rng.dirichlet(np.ones(n)).astype(np.float32).astype(np.float64)
        if not O.select_blocks(p, 1.0)["sel"].all():
            fails.append("eta=1 did not select every block")
        tiny = O.select_blocks(p, 1e-9)["sel"]
        if np.nonzero(tiny)[0].tolist() != [int(np.argmax(p))]:
            fails.append("tiny eta did not select exactly the arg-max")
        prev = np.zeros(n, bool)
        for eta in np.linspace(0.05, 0.99, 12):
            sel = O.select_blocks(p, float(eta))["sel"]
            if np.any(prev & ~sel):
                fails.append("selection not monotone in eta")
                break
            prev = sel
    return fails


def pin_union(O) -> List[str]:
    """Discover at depth 0, then union-discover at depth 1, equals the OR of the
    two depths' own selections [WISE PR, Tests: the fused selection matches
    the union across discovery depths]."""
    fails = []
    w = custom_workload(R=3, Hq=2, Hkv=2, D=64, dtype="f32", depths=2, n_planted=2,
                        seq_lens=np.array([256, 100, 64], np.int32), pool_factor=1, seed=81,
                        depth_modes=[np.zeros(3, np.int8)] * 2)
    d0, d1 = w.depth_inputs(0, logical=True), w.depth_inputs(1, logical=True)
    z = empty_support(w)
    s0 = run(O, w, d0, [MODE_DISCOVER] * 3, z)["support"]
    s1 = run(O, w, d1, [MODE_DISCOVER] * 3, z)["support"]
    u = run(O, w, d1, [MODE_DISCOVER_UNION] * 3, s0)["support"]
    if not np.array_equal(u, s0 | s1):
        fails.append("union-discover != OR of per-depth selections")
    if not np.array_equal(O.support_union(s0, s1), s0 | s1):
        fails.append("support_union != bitwise OR")
    # The union mask really contains both selections (no overwrite).
    for r in range(3):
        for g in range(2):
            nb = -(-int(w.seq_lens[r]) // 32)
            a, b, c = (library_bits(x[r, g], nb) for x in (s0, s1, u))
            if not np.array_equal(c, a | b):
                fails.append(f"union bits differ r={r} g={g}")
    return fails


def pin_head_union(O) -> List[str]:
    """Head union of a row's masks [WISE PR, "What changes", FlashAttention
    decode bullet]: a hand-worked example (tests/golden/head_union_example.json),
    then on random masks every head's blocks are kept and every kept block
    has a head that selected it, row by row."""
    with open(os.path.join(GOLDEN, "head_union_example.json")) as f:
        gold = json.load(f)
    fails = []
    got = O.support_head_union(np.array(gold["support"], np.uint32))
    if not np.array_equal(got, np.array(gold["expected"], np.uint32)):
        fails.append(f"head union example: {got.tolist()}")
    rng = np.random.default_rng(17)
    sup = (rng.random((4, 3, 2 * 32)) < 0.2)
    words = np.packbits(sup, axis=-1, bitorder="little").view(np.uint32).reshape(4, 3, 2)
    u = O.support_head_union(words)
    for r in range(4):
        ub = library_bits(u[r, 0], 64)
        if any(not np.array_equal(library_bits(u[r, g], 64), ub) for g in range(3)):
            fails.append(f"row {r}: heads differ after the union")
        if not np.array_equal(ub, sup[r].any(axis=0)):
            fails.append(f"row {r}: union bits are not the blocks some head selected")
    return fails


def _two_block_input(hot_block: int):
    """One row, one head, D=64, 64 tokens (two causal blocks): every key of the
    hot block equals q, every other key is zero, so the hot block carries all
    but e^-8 of the mass."""
    D, L, P = 64, 64, 16
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 8.0
    k = np.zeros((L // P, P, 1, D), np.float32)
    v = np.random.default_rng(hot_block).standard_normal((L // P, P, 1, D)).astype(np.float32)
    for j in range(hot_block * 32, hot_block * 32 + 32):
        k[j // P, j % P, 0, 0] = 8.0
    return q, k, v, np.arange(L // P, dtype=np.int32)[None, :], np.array([L], np.int32)


def pin_density_example(O) -> List[str]:
    """The pages' worked example: two disjoint one-block selections over two
    causal blocks give a reused-union density of 1.0 (per-selection 0.5)."""
    with open(os.path.join(GOLDEN, "union_density_example.json")) as f:
        gold = json.load(f)
    fails = []
    sup = np.zeros((1, 1, 1), np.uint32)
    sels = []
    for depth, hot in enumerate((0, 1)):
        q, k, v, pt, lens = _two_block_input(hot)
        mode = MODE_DISCOVER if depth == 0 else MODE_DISCOVER_UNION
        res = O.decode_layer(q, k, v, pt, lens, np.array([mode], np.int8), sup, eta=0.95)
        sels.append(np.nonzero(res["diag"][(0, 0)]["sel"])[0].tolist())
        sup = res["support"]
    if sels != gold["depth_selections"]:
        fails.append(f"per-depth selections {sels}")
    if np.nonzero(library_bits(sup[0, 0], 2))[0].tolist() != gold["union_blocks"]:
        fails.append("union blocks differ")
    dens = O.union_density(sup, np.array([64]), 32)
    if dens != gold["union_density"]:
        fails.append(f"union density {dens}")
    per_sel = np.mean([len(s) for s in sels]) / gold["causal_blocks"]
    if per_sel != gold["per_selection_density"]:
        fails.append(f"per-selection density {per_sel}")
    return fails


def pin_compaction(O) -> List[str]:
    """The compacted tile lists, against numpy.unpackbits of the mask: for a
    sparse row the ascending set bits below the row's block count, for any
    other mode every block; counts equal the list lengths."""
    fails = []
    rng = np.random.default_rng(91)
    for trial in range(20):
        R, H = int(rng.integers(1, 5)), int(rng.integers(1, 4))
        lens = rng.integers(0, 300, size=R).astype(np.int32)
        W = max(1, -(-int(-(-lens.max() // 32)) // 32)) + int(rng.integers(0, 2))
        bits = rng.random((R, H, W * 32)) < rng.uniform(0, 1)
        sup = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(R, H, W).copy()
        modes = rng.choice([MODE_DENSE, MODE_DISCOVER, MODE_DISCOVER_UNION, MODE_SPARSE], size=R).astype(np.int8)
        res = O.compact_tiles(sup, modes, lens, 32)
        for r in range(R):
            nb = -(-int(lens[r]) // 32)
            for g in range(H):
                want = (np.nonzero(library_bits(sup[r, g], nb))[0] if modes[r] == MODE_SPARSE
                        else np.arange(nb))
                lst = res["lists"][r][g]
                if not np.array_equal(lst, want):
                    fails.append(f"trial {trial} list r={r} g={g}")
                if int(res["counts"][r, g]) != want.shape[0]:
                    fails.append(f"trial {trial} count r={r} g={g}")
    return fails


def pin_slot_masks(O) -> List[str]:
    """Masks kept per request slot and layer [WISE PR, "What changes",
    wise.py bullet: a [slot, layer, head, block] support bitmask], addressed
    through each row's slot: (a) identity slots on a one-layer pool give
    decode_layer's results exactly; (b) on a pool of 6 slots x 3 layers whose
    (slot, layer, KV head) mask selects exactly block (slot + 2 layer + KV
    head) mod 4, rows with slots [4, 1, -1, 3] at layer 1 attend in sparse mode
    exactly that block of their own slot -- torch SDPA over its keys -- and the
    row without a slot outputs 0 with LSE -inf; (c) a discover call stores
    each row's new mask at (its slot, layer 1) and leaves every other pool
    entry, and the slot-less row's, bitwise unchanged."""
    fails = []
    w, d = make_case(2, 2, 64, "f32", [128, 128, 128, 128], 61)
    q, kc, vc = (as_oracle_array(d[k]) for k in ("q", "k_cache", "v_cache"))
    R, B = 4, w.tile_tokens
    # (a)
    sup = random_support(w, 62)
    plain = O.decode_layer(q, kc, vc, w.page_table, w.seq_lens, np.full(R, MODE_SPARSE, np.int8),
                           sup, tile_tokens=B)
    viaslots = O.decode_layer_slots(q, kc, vc, w.page_table, w.seq_lens,
                                    np.full(R, MODE_SPARSE, np.int8), sup[:, None], np.arange(R),
                                    0, tile_tokens=B)
    if not (np.array_equal(plain["out"], viaslots["out"]) and
            np.array_equal(plain["lse"], viaslots["lse"])):
        fails.append("identity slots differ from decode_layer")
    # (b)
    S, Lyr, layer = 6, 3, 1
    pool = np.zeros((S, Lyr, 2, 1), np.uint32)
    for sl in range(S):
        for ly in range(Lyr):
            for g in range(2):
                pool[sl, ly, g, 0] = np.uint32(1) << np.uint32((sl + 2 * ly + g) % 4)
    row_slot = np.array([4, 1, -1, 3])
    res = O.decode_layer_slots(q, kc, vc, w.page_table, w.seq_lens,
                               np.full(R, MODE_SPARSE, np.int8), pool, row_slot, layer,
                               tile_tokens=B)
    scale = 1.0 / math.sqrt(64)
    for r in range(R):
        for h in range(2):
            if row_slot[r] < 0:
                if not (np.all(res["out"][r, h] == 0) and res["lse"][r, h] == -math.inf):
                    fails.append(f"slot-less row {r} head {h} not zero/-inf")
                continue
            blk = (int(row_slot[r]) + 2 * layer + h) % 4
            mask = np.zeros(128, bool)
            mask[blk * B:(blk + 1) * B] = True
            qq, K, V = _ref_row(d, r, h, h)
            o = _sdpa(qq, K, V, scale, mask).numpy()
            if not np.allclose(res["out"][r, h], o, rtol=tol(O, "out_rtol"), atol=tol(O, "out_atol")):
                fails.append(f"row {r} head {h} does not attend its slot's block {blk}")
    if not np.array_equal(res["pool"], pool):
        fails.append("a sparse call changed the pool")
    # (c)
    res = O.decode_layer_slots(q, kc, vc, w.page_table, w.seq_lens,
                               np.full(R, MODE_DISCOVER, np.int8), pool, row_slot, layer,
                               tile_tokens=B)
    own = O.decode_layer(q, kc, vc, w.page_table, w.seq_lens, np.full(R, MODE_DISCOVER, np.int8),
                         np.zeros((R, 2, 1), np.uint32), tile_tokens=B)["support"]
    want = pool.copy()
    for r in range(R):
        if row_slot[r] >= 0:
            want[row_slot[r], layer] = own[r]
    if not np.array_equal(res["pool"], want):
        fails.append("discover stored masks at the wrong place or touched other entries")
    return fails


ALL_PINS = [pin_dense_sdpa, pin_sparse_masked_sdpa, pin_sparse_bruteforce_loops,
            pin_all_blocks_sparse_is_dense,
            pin_paging_invariance, pin_page_size_invariance, pin_block_masses, pin_selection_bruteforce,
            pin_selection_golden, pin_selection_limits, pin_union, pin_density_example,
            pin_compaction, pin_head_union, pin_slot_masks]
