"""Shared helpers of the GPU parity tests: run one decode call through the C ABI
and through the CPU oracle on the same seeded inputs, and compare.  The oracle
is the C++ one in fp32 unless a test asks for the float64 numpy one (both
are pinned by the CPU tests; the main per-mode test runs against both).

Tolerances (from the arithmetic; the acceptance bar of this library):
  * bf16 output: max |out_gpu - out_oracle| <= 1e-2, against the oracle's
    float64 output (one bf16 ulp at |o| in [2, 4) is 1.6e-2, so a bf16-vs-bf16
    comparison would flag correct roundings; half an ulp at |o| < 4 is 7.8e-3).
  * fp32 output: <= 1e-4 (fp32 accumulation over <= 1e3 terms plus a 2-ulp
    exp2 leaves errors near 1e-6).
  * LSE (natural log, fp32): <= 1e-4 absolute.
  * Support mask: bit-exact for every (row, KV head) whose query heads all have
    an oracle cumulative-mass margin > 1e-4 at the cutoff and a relative mass
    gap > 1e-5 between the last kept and the first dropped block.  The kernel's
    block masses carry relative errors below ~1.5e-6 (2-ulp ex2 terms summed
    over a tile, an accurate exp2 of the max minus an fp32 LSE), so masses
    closer than that may legally swap order; such masks are checked against
    bounds instead: every block the oracle keeps with margin and gap to spare
    must be kept, and nothing outside the cutoff's tolerance band may be.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

import block_sparse_paged_split_gb300 as W
from oracle import wise_oracle as O
from oracle.cpp_oracle import CppOracle
from tests.oracle_pins import as_oracle_array

OUT_TOL = {"bf16": 1e-2, "f32": 1e-4}
LSE_TOL = 1e-4
MARGIN = 1e-4
GAP_REL = 1e-5


def shape_for(w, eta: Optional[float] = None, tiles_per_item: int = 0) -> W.wise_shape:
    return W.make_shape(num_rows=w.num_rows, num_q_heads=w.num_q_heads,
                        num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                        page_size=w.page_size, max_pages_per_row=w.max_pages_per_row,
                        num_pages=w.num_pages, max_blocks=w.max_blocks,
                        dtype=W.DTYPE_BF16 if w.dtype == "bf16" else W.DTYPE_F32,
                        eta=w.eta if eta is None else eta, tiles_per_item=tiles_per_item)


def words(w) -> int:
    return -(-w.max_blocks // 32)


def np_support(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32).copy()


def dev_support(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).cuda()


class Batch:
    """A workload's metadata on the device, plus per-depth inputs on demand."""

    def __init__(self, w):
        self.w = w
        self.page_table = torch.from_numpy(w.page_table).cuda()
        self.seq_lens = torch.from_numpy(w.seq_lens).cuda()
        self._cpu: Dict[int, dict] = {}
        self._dev: Dict[int, dict] = {}

    def cpu(self, depth: int) -> dict:
        if depth not in self._cpu:
            self._cpu[depth] = self.w.depth_inputs(depth)
        return self._cpu[depth]

    def dev(self, depth: int) -> dict:
        if depth not in self._dev:
            self._dev[depth] = {k: v.cuda() for k, v in self.cpu(depth).items()}
        return self._dev[depth]


def gpu_call(b: Batch, depth: int, modes: np.ndarray, support: np.ndarray,
             eta: Optional[float] = None, tiles_per_item: int = 0, stepwise: bool = True,
             fused: bool = False):
    """One decode call through the C ABI; returns out (float64 numpy), lse,
    the support after the call and the workspace views.  stepwise: compact,
    partial and finish as three calls; fused: compact, then the partial pass
    with the finish folded in (the benchmark's launch sequence); otherwise the
    one-call entry point."""
    w = b.w
    shape = shape_for(w, eta, tiles_per_item)
    d = b.dev(depth)
    ws = W.alloc_workspace(shape)
    modes_t = torch.from_numpy(np.asarray(modes, np.int8)).cuda()
    sup = dev_support(support)
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.num_rows, w.num_q_heads), dtype=torch.float32, device="cuda")
    if fused:
        W.wise_compact_tiles(shape, modes_t, b.seq_lens, sup, ws)
        W.wise_decode_partial_finish(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                     b.seq_lens, modes_t, ws, sup, out, lse)
    elif stepwise:
        W.wise_compact_tiles(shape, modes_t, b.seq_lens, sup, ws)
        W.wise_decode_partial(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens,
                              modes_t, ws)
        W.wise_decode_finish(shape, modes_t, b.seq_lens, ws, sup, out, lse)
    else:
        W.wise_decode(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens, modes_t,
                      sup, out, lse, ws)
    torch.cuda.synchronize()
    views = {k: v.cpu() for k, v in W.workspace_views(shape, ws).items()}
    return {"out": out.double().cpu().numpy(), "out_raw": out.cpu(), "lse": lse.cpu().numpy(),
            "support": np_support(sup), "ws": views}


_CPP = {}


def oracle_module(which: str):
    """The oracle a comparison runs against: "f32" is the C++ oracle in fp32
    (the acceptance oracle: plain loops, fp32 math, a sort-based eta prefix),
    "f64" the numpy oracle in float64.  Both are pinned by the CPU tests."""
    if which == "f64":
        return O
    if which not in _CPP:
        _CPP[which] = CppOracle(which.replace("cpp-", ""))
    return _CPP[which]


def oracle_call(b: Batch, depth: int, modes: np.ndarray, support: np.ndarray,
                eta: Optional[float] = None, rows=None, oracle: str = "f32"):
    """The oracle on the same inputs (optionally on a subset of rows)."""
    w = b.w
    c = b.cpu(depth)
    q = as_oracle_array(c["q"])
    pt, sl, md, sup = w.page_table, w.seq_lens, np.asarray(modes, np.int8), support
    if rows is not None:
        rows = np.asarray(rows)
        q, pt, sl, md, sup = q[rows], pt[rows], sl[rows], md[rows], sup[rows]
    e = w.eta if eta is None else eta
    res = oracle_module(oracle).decode_layer(q, as_oracle_array(c["k_cache"]),
                                             as_oracle_array(c["v_cache"]), pt, sl, md, sup, eta=e,
                                             tile_tokens=w.tile_tokens)
    res["eta"] = e
    return res


def o_eta(o, w) -> float:
    return float(o.get("eta", w.eta))


def compare_outputs(w, g, o, rows=None) -> list:
    fails = []
    tol = OUT_TOL[w.dtype]
    go, gl = g["out"], g["lse"]
    if rows is not None:
        go, gl = go[rows], gl[rows]
    err = np.abs(go - o["out"])
    if not np.all(np.isfinite(go)):
        fails.append("non-finite GPU output")
    elif err.max() > tol:
        r, h, _ = np.unravel_index(np.argmax(err), err.shape)
        fails.append(f"out max err {err.max():.3g} > {tol} at row {r} head {h}")
    both_inf = np.isneginf(gl) & np.isneginf(o["lse"])
    with np.errstate(invalid="ignore"):
        lerr = np.where(both_inf, 0.0, np.abs(gl - o["lse"]))
    if not np.all(np.isfinite(lerr)) or lerr.max() > LSE_TOL:
        fails.append(f"lse max err {np.nanmax(lerr):.3g} > {LSE_TOL}")
    return fails


def mask_bounds(dg: dict, eta: float, nb: int):
    """Blocks any valid fp32 evaluation must keep, and blocks it may keep, for
    one query head whose decision is near a tie: a block is certain when the
    mass before it is below eta - MARGIN and it outweighs the first dropped
    block by more than the relative gap GAP_REL; it is possible when the mass
    before it is below eta + MARGIN or it is within GAP_REL of the last kept
    block."""
    if eta >= 1.0:
        allb = np.ones(nb, bool)
        return allb, allb
    p32 = dg["p"].astype(np.float32).astype(np.float64)
    order = dg["order"]
    ps = p32[order]
    before = np.cumsum(ps) - ps
    k = dg["k"]
    p_next = ps[k] if k < nb else -np.inf
    p_last = ps[k - 1]
    must = np.zeros(nb, bool)
    may = np.zeros(nb, bool)
    must[order] = (before < eta - MARGIN) & (ps > p_next + GAP_REL * abs(p_next))
    may[order] = (before < eta + MARGIN) | (ps >= p_last * (1 - GAP_REL))
    return must, may


def decision_is_clear(dg: dict) -> bool:
    """Margin > 1e-4 at the cutoff and a relative gap > 1e-5 to the next block."""
    if dg["margin"] <= MARGIN:
        return False
    if not np.isfinite(dg["gap"]):
        return True
    p_last = float(dg["p"].astype(np.float32)[dg["order"][dg["k"] - 1]])
    return dg["gap"] > GAP_REL * p_last


def compare_masks(w, g_support, o, modes, rows=None, support_in=None) -> Dict[str, object]:
    """Bit-exact comparison where the oracle's decision is unambiguous; for the
    rest, bounds from the oracle's masses (plus, for union-discover rows, the
    bits the mask held before the call, which the union always keeps)."""
    G = w.group
    sup_g = g_support if rows is None else g_support[rows]
    rows_idx = range(sup_g.shape[0])
    checked = excluded_margin = excluded_gap = 0
    fails = []
    for r in rows_idx:
        if int(np.asarray(modes)[r if rows is None else rows[r]]) not in (W.MODE_DISCOVER, W.MODE_DISCOVER_UNION):
            continue
        L = int(w.seq_lens[r if rows is None else rows[r]])
        if L == 0:
            continue
        nb = -(-L // w.tile_tokens)
        for g in range(w.num_kv_heads):
            diags = [o["diag"][(r, h)] for h in range(g * G, (g + 1) * G)]
            clear = all(decision_is_clear(dg) for dg in diags)
            near_margin = any(dg["margin"] <= MARGIN for dg in diags)
            gb = O.mask_bits(sup_g[r, g], nb)
            ob = O.mask_bits(o["support"][r, g], nb)
            if clear:
                checked += 1
                if not np.array_equal(gb, ob):
                    fails.append(f"mask differs row {r} kv head {g}")
            else:
                if near_margin:
                    excluded_margin += 1
                else:
                    excluded_gap += 1
                must = np.zeros(nb, bool)
                may = np.zeros(nb, bool)
                mode_r = int(np.asarray(modes)[r if rows is None else rows[r]])
                if mode_r == W.MODE_DISCOVER_UNION:
                    if support_in is None:
                        raise ValueError("union masks need the input mask")
                    old = O.mask_bits((support_in if rows is None else support_in[rows])[r, g], nb)
                    must |= old
                    may |= old
                for dg in diags:
                    a, c = mask_bounds(dg, o_eta(o, w), nb)
                    must |= a
                    may |= c
                if np.any(must & ~gb) or np.any(gb & ~may):
                    fails.append(f"ambiguous mask outside its bounds row {r} kv head {g}")
            # never any bit at or past the block count
            if np.any(np.unpackbits(sup_g[r, g].view(np.uint8), bitorder="little")[nb:32 * sup_g.shape[2]]):
                fails.append(f"bits past the row end row {r} kv head {g}")
    return {"fails": fails, "checked": checked, "excluded": excluded_margin + excluded_gap,
            "excluded_margin": excluded_margin, "excluded_gap": excluded_gap}


def item_fields(rec: np.ndarray):
    """Fields of work-item records int32 [n, 4]: pair rg, block range s,
    partial slot k, tile bitmap over the range, tile count, row length,
    sparse flag, discover flag."""
    rec = np.asarray(rec, np.int64)
    return {"rg": rec[:, 0], "s": rec[:, 1] & 0xFFFF, "k": rec[:, 1] >> 16,
            "bits": rec[:, 2] & 0xFFFF, "count": (rec[:, 2] >> 16) & 0xFF,
            "L": rec[:, 3] & 0xFFFFFF, "sparse": (rec[:, 3] >> 24) & 1,
            "discover": (rec[:, 3] >> 25) & 1}


def list1_schedule(views: dict, T: int) -> np.ndarray:
    """List 1's items in the order the partial pass hands them out: bucket j
    holds the items of j + 1 tiles (counter[j] of them), larger buckets
    first."""
    cnt = views["list1_counter"].cpu().numpy()[:T].astype(np.int64)
    items = views["items_1"].cpu().numpy()
    out = [items[j, :int(cnt[j])] for j in range(T - 1, -1, -1)]
    return np.concatenate(out) if out else np.zeros((0, 4), np.int32)


def item_invariant_fails(recs: np.ndarray, head_info: np.ndarray, lists, T: int, S_max: int,
                         lens: np.ndarray, modes, Hkv: int, compact_slots: bool) -> list:
    """A work list against the oracle's compacted tile lists, by properties
    (the pages fix the lists; how they are cut into items is the kernel's
    choice): every item holds 1..T tiles, all inside one range [s*T, s*T+T)
    of its pair, as a bitmap whose popcount is its count; a pair's items,
    taken by range, concatenate to exactly its list (so each item is a
    contiguous, strictly ascending run and together they partition it); slots
    are distinct and below the pair's slot count (equal to the range, or
    compact 0..items-1 in range order); the schedule is non-increasing in
    tile count; head info agrees; the record carries the row's length and
    mode flags (modes None: every row sparse)."""
    fails = []
    f = item_fields(recs)
    if recs.shape[0] and np.any(np.diff(f["count"]) > 0):
        fails.append("schedule not in non-increasing tile count")
    pc = np.array([bin(int(b)).count("1") for b in f["bits"]], np.int64)
    if np.any(pc != f["count"]) or np.any(f["count"] < 1) or np.any(f["count"] > T):
        fails.append("item counts do not match bitmaps or exceed T")
    if recs.shape[0] and np.any(f["bits"] >> T):
        fails.append("bitmap bits at or past T")
    R = len(lens)
    for r in range(R):
        for g in range(Hkv):
            rg = r * Hkv + g
            sel = np.nonzero(f["rg"] == rg)[0]
            order = sel[np.argsort(f["s"][sel], kind="stable")]
            tiles = []
            for i in order:
                tiles += [int(f["s"][i]) * T + b for b in range(T) if (int(f["bits"][i]) >> b) & 1]
            want = np.asarray(lists[r][g]).tolist()
            if tiles != want:
                fails.append(f"items of pair ({r},{g}) do not partition its list")
            if len(set(f["s"][order].tolist())) != len(order):
                fails.append(f"pair ({r},{g}) has two items in one range")
            ks = f["k"][order].tolist()
            want_k = list(range(len(order))) if compact_slots else f["s"][order].tolist()
            if ks != want_k:
                fails.append(f"pair ({r},{g}) slots {ks[:8]} != {want_k[:8]}")
            hi = head_info[r, g]
            if int(hi[0]) != rg * S_max or int(hi[2]) != len(want) or int(hi[3]) != len(order):
                fails.append(f"head info of pair ({r},{g}): {hi.tolist()}")
            if len(order) and int(hi[1]) <= max(ks):
                fails.append(f"pair ({r},{g}) slot count {int(hi[1])} too small")
            for i in order:
                if int(f["L"][i]) != int(lens[r]):
                    fails.append(f"item of pair ({r},{g}) has length {int(f['L'][i])}")
                m = 3 if modes is None else int(np.asarray(modes)[r])
                if int(f["sparse"][i]) != (m == 3) or int(f["discover"][i]) != (m in (1, 2)):
                    fails.append(f"item of pair ({r},{g}) has wrong mode flags")
    return fails
