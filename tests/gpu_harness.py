"""Shared helpers of the GPU parity tests: run one decode call through the C ABI
and through the CPU oracle on the same seeded inputs, and compare.

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


def oracle_call(b: Batch, depth: int, modes: np.ndarray, support: np.ndarray,
                eta: Optional[float] = None, rows=None):
    """The oracle on the same inputs (optionally on a subset of rows)."""
    w = b.w
    c = b.cpu(depth)
    q = as_oracle_array(c["q"])
    pt, sl, md, sup = w.page_table, w.seq_lens, np.asarray(modes, np.int8), support
    if rows is not None:
        rows = np.asarray(rows)
        q, pt, sl, md, sup = q[rows], pt[rows], sl[rows], md[rows], sup[rows]
    e = w.eta if eta is None else eta
    res = O.decode_layer(q, as_oracle_array(c["k_cache"]), as_oracle_array(c["v_cache"]), pt, sl,
                         md, sup, eta=e, tile_tokens=w.tile_tokens)
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
    checked = excluded = 0
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
            gb = O.mask_bits(sup_g[r, g], nb)
            ob = O.mask_bits(o["support"][r, g], nb)
            if clear:
                checked += 1
                if not np.array_equal(gb, ob):
                    fails.append(f"mask differs row {r} kv head {g}")
            else:
                excluded += 1
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
    return {"fails": fails, "checked": checked, "excluded": excluded}
