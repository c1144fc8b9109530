"""Seeded synthetic decode workloads shaped like Ouro-1.4B recurrent-depth decode.

This module only *generates inputs*.  It holds none of the attention or
selection arithmetic; the CPU oracle and the CUDA library both consume what it
produces, so it is the one piece of code the two sides share.

Workloads (named by what they are, sizes from the WISE working-set decode PR,
"Results" section: Ouro-1.4B, bf16, always 4 loops; Ouro-1.4B has 16 KV heads
of head dim 128):

  tiny         4 rows x 256 tokens, 2 heads MHA, D=64, fp32, 2 planted blocks
               per (row, head), 2 depths, rows run [dense, discover, sparse,
               sparse].
  ouro1.4b_1k  64 rows x 1024 tokens, 16 heads MHA, D=128, bf16, 4 depths
               each with its own K/V, 4 planted blocks per (row, head).
  ouro1.4b_4k  as above at 4096 tokens, 8 planted blocks, page tables
               shuffled over a page pool twice the size the rows need.
  mixed_8k     32 rows with lengths uniform in [1024, 8192], 8 planted
               blocks, per-row mode 25% dense / 25% discover / 50% sparse.
  gqa_32k      8 rows x 32768 tokens, 32 query / 8 KV heads, 16 planted
               blocks per (row, KV-head group).

Recipe (all draws seeded; every tensor stream is keyed by
(base seed, depth, tensor, row) through numpy's SeedSequence):

  * q_0 ~ N(0,1) [R, Hq, D]; q_t = q_0 + 0.3 * N(0,1) for depth t >= 1.
  * Each row's logical K and V (token-major, [L_r, Hkv, D]) ~ N(0,1), drawn
    independently per depth.
  * Planted support: per (row, head) (MHA) or (row, KV head) (GQA) a set of
    block indices drawn without replacement from the row's valid 32-token
    blocks, identical at every depth.  Every valid key in a planted block gets
    += 0.5 * q_t (the query of that depth for that head; for GQA the mean of
    the group's queries), before rounding to the storage dtype.
  * Paging: the row's tokens are cut into pages of `page_size`; pages are
    placed at a seeded random permutation of the pool.  Pool pages no row
    references, and the token slots past a row's length in its last page, are
    filled with NaN so that any stray read poisons the result.
  * Storage is bf16 (round-to-nearest-even, done by torch's CPU cast) or fp32.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

# Per-row mode codes (the library's int8 mode vocabulary).
MODE_DENSE = 0
MODE_DISCOVER = 1
MODE_DISCOVER_UNION = 2
MODE_SPARSE = 3

_TENSOR_IDS = {"q0": 1, "qnoise": 2, "k": 3, "v": 4, "plant": 5, "pages": 6,
               "lens": 7, "modes": 8}

BASE_SEEDS = {"tiny": 1000, "ouro1.4b_1k": 1001, "ouro1.4b_4k": 1002,
              "mixed_8k": 1003, "gqa_32k": 1004}


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


@dataclasses.dataclass
class Workload:
    name: str
    num_rows: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    tile_tokens: int
    dtype: str                    # "bf16" or "f32"
    eta: float
    num_depths: int
    seq_lens: np.ndarray          # int32 [R]
    page_table: np.ndarray        # int32 [R, max_pages_per_row], -1 past the row
    num_pages: int
    planted: List[List[np.ndarray]]   # [R][plant head] -> block indices
    depth_modes: List[np.ndarray]     # per depth: int8 [R]
    seed: int
    n_planted: int

    @property
    def max_pages_per_row(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def max_blocks(self) -> int:
        return -(-self.max_pages_per_row * self.page_size // self.tile_tokens)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def queries_f32(self, depth: int) -> np.ndarray:
        R, Hq, D = self.num_rows, self.num_q_heads, self.head_dim
        q0 = _rng(self.seed, 0, _TENSOR_IDS["q0"]).standard_normal((R, Hq, D), dtype=np.float32)
        if depth == 0:
            return q0
        noise = _rng(self.seed, depth, _TENSOR_IDS["qnoise"]).standard_normal((R, Hq, D), dtype=np.float32)
        return q0 + np.float32(0.3) * noise

    def depth_inputs(self, depth: int, logical: bool = False) -> Dict[str, object]:
        """q [R,Hq,D], k_cache and v_cache [num_pages, page_size, Hkv, D] on the CPU.

        With `logical=True` also returns "k_rows"/"v_rows": per row the
        token-ordered [L_r, Hkv, D] tensors before paging (same values)."""
        R, Hkv, D, P = self.num_rows, self.num_kv_heads, self.head_dim, self.page_size
        G = self.group
        qf = self.queries_f32(depth)
        # Planting direction per (row, plant head): the head's own query (MHA)
        # or the mean over the query heads of its KV group (GQA).
        plant_dir = qf.reshape(R, Hkv, G, D).mean(axis=2) if G > 1 else qf
        tdt = self.torch_dtype
        nan = float("nan")
        k_pool = torch.full((self.num_pages, P, Hkv, D), nan, dtype=tdt)
        v_pool = torch.full((self.num_pages, P, Hkv, D), nan, dtype=tdt)
        k_rows, v_rows = [], []
        for r in range(R):
            L = int(self.seq_lens[r])
            if L == 0:
                k_rows.append(torch.zeros((0, Hkv, D), dtype=tdt))
                v_rows.append(torch.zeros((0, Hkv, D), dtype=tdt))
                continue
            npg = -(-L // P)
            kr = _rng(self.seed, depth, _TENSOR_IDS["k"], r).standard_normal((npg * P, Hkv, D), dtype=np.float32)
            vr = _rng(self.seed, depth, _TENSOR_IDS["v"], r).standard_normal((npg * P, Hkv, D), dtype=np.float32)
            B = self.tile_tokens
            for h in range(Hkv):
                for b in self.planted[r][h]:
                    lo, hi = int(b) * B, min((int(b) + 1) * B, L)
                    kr[lo:hi, h, :] += np.float32(0.5) * plant_dir[r, h]
            kr[L:] = np.nan
            vr[L:] = np.nan
            pages = torch.from_numpy(self.page_table[r, :npg].astype(np.int64))
            kt = torch.from_numpy(kr).to(tdt)
            vt = torch.from_numpy(vr).to(tdt)
            k_pool[pages] = kt.view(npg, P, Hkv, D)
            v_pool[pages] = vt.view(npg, P, Hkv, D)
            if logical:
                k_rows.append(kt[:L].clone())
                v_rows.append(vt[:L].clone())
        q = torch.from_numpy(qf).to(tdt)
        out = {"q": q, "k_cache": k_pool, "v_cache": v_pool}
        if logical:
            out["k_rows"], out["v_rows"] = k_rows, v_rows
        return out


    def depth_inputs_device(self, depth: int, device="cuda") -> Dict[str, object]:
        """The same recipe with K and V drawn on the device, for timing runs
        whose oracle check is elsewhere: q is the host draw of
        `queries_f32` (so the planted directions are the same), K and V ~
        N(0,1) come from a torch generator on `device` seeded by (seed,
        depth, tensor), planted keys get += 0.5 * the planting direction,
        pool pages no row references and slots past a row's length hold NaN,
        and the values are rounded to the storage dtype.  Same shapes,
        distributions and structure as depth_inputs; other values."""
        R, Hkv, D, P, B = self.num_rows, self.num_kv_heads, self.head_dim, self.page_size, self.tile_tokens
        G = self.group
        qf = self.queries_f32(depth)
        plant_dir = qf.reshape(R, Hkv, G, D).mean(axis=2) if G > 1 else qf
        used = np.zeros((self.num_pages, P), dtype=bool)
        plant_pg, plant_sl, plant_h, plant_row = [], [], [], []
        for r in range(R):
            L = int(self.seq_lens[r])
            if L == 0:
                continue
            tok = np.arange(L)
            pages = self.page_table[r, tok // P]
            used[pages, tok % P] = True
            for h in range(Hkv):
                for b in self.planted[r][h]:
                    t = np.arange(int(b) * B, min((int(b) + 1) * B, L))
                    plant_pg.append(self.page_table[r, t // P])
                    plant_sl.append(t % P)
                    plant_h.append(np.full(t.shape, h))
                    plant_row.append(np.full(t.shape, r))
        cat = lambda xs: torch.from_numpy(np.concatenate(xs).astype(np.int64)).to(device) \
            if xs else torch.zeros(0, dtype=torch.int64, device=device)  # noqa: E731
        pg, sl, hh, rr = cat(plant_pg), cat(plant_sl), cat(plant_h), cat(plant_row)
        unused = torch.from_numpy(~used).to(device)
        dirs = torch.from_numpy(np.ascontiguousarray(plant_dir)).to(device)
        out = {"q": torch.from_numpy(qf).to(self.torch_dtype)}
        for name in ("k", "v"):
            gen = torch.Generator(device=device)
            gen.manual_seed(int(np.random.SeedSequence([self.seed, depth, _TENSOR_IDS[name]])
                                .generate_state(1)[0]))
            pool = torch.randn((self.num_pages, P, Hkv, D), generator=gen, device=device,
                               dtype=torch.float32)
            if name == "k" and pg.numel():
                pool[pg, sl, hh] += 0.5 * dirs[rr, hh]
            pool[unused] = float("nan")
            out[name + "_cache"] = pool.to(self.torch_dtype)
            del pool
        return out


def custom_workload(name: str = "custom", **kw) -> Workload:
    """A workload of any shape built with the same recipe (see `_build`)."""
    return _build(name, **kw)


def _build(name: str, *, R: int, Hq: int, Hkv: int, D: int, dtype: str, depths: int,
           n_planted: int, seq_lens: np.ndarray, pool_factor: int, seed: int,
           depth_modes: List[np.ndarray], eta: float = 0.95, page_size: int = 16,
           tile_tokens: int = 32) -> Workload:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    P, B = page_size, tile_tokens
    n_pages = [-(-int(L) // P) for L in seq_lens]
    max_pages = max(max(n_pages), 1)
    needed = sum(n_pages)
    num_pages = max(pool_factor * needed, 1)
    perm = _rng(seed, 0, _TENSOR_IDS["pages"]).permutation(num_pages).astype(np.int32)
    page_table = np.full((R, max_pages), -1, dtype=np.int32)
    off = 0
    for r in range(R):
        page_table[r, :n_pages[r]] = perm[off:off + n_pages[r]]
        off += n_pages[r]
    prng = _rng(seed, 0, _TENSOR_IDS["plant"])
    planted = []
    for r in range(R):
        nb = -(-int(seq_lens[r]) // B)
        per_head = []
        for _h in range(Hkv):
            k = min(n_planted, nb)
            per_head.append(np.sort(prng.choice(nb, size=k, replace=False)).astype(np.int32)
                            if k > 0 else np.zeros(0, np.int32))
        planted.append(per_head)
    return Workload(name=name, num_rows=R, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                    page_size=P, tile_tokens=B, dtype=dtype, eta=eta, num_depths=depths,
                    seq_lens=seq_lens, page_table=page_table, num_pages=num_pages,
                    planted=planted, depth_modes=[np.asarray(m, np.int8) for m in depth_modes],
                    seed=seed, n_planted=n_planted)


def _recurrent_schedule(R: int, depths: int) -> List[np.ndarray]:
    """Discover at depth 0, union-discover at depth 1, reuse (sparse) after."""
    out = []
    for t in range(depths):
        m = MODE_DISCOVER if t == 0 else (MODE_DISCOVER_UNION if t == 1 else MODE_SPARSE)
        out.append(np.full(R, m, np.int8))
    return out


def make_workload(name: str, *, num_rows: Optional[int] = None, context: Optional[int] = None,
                  seq_lens: Optional[np.ndarray] = None, seed: Optional[int] = None,
                  eta: float = 0.95) -> Workload:
    """Build one of the named workloads; `num_rows`/`context`/`seq_lens` shrink it
    (for parity tests the oracle finishes in seconds) without changing its recipe."""
    base = BASE_SEEDS[name] if seed is None else seed
    if name == "tiny":
        R = num_rows or 4
        L = context or 256
        lens = np.full(R, L, np.int32) if seq_lens is None else seq_lens
        row_modes = [MODE_DENSE, MODE_DISCOVER, MODE_SPARSE, MODE_SPARSE]
        d0 = np.array([row_modes[r % 4] for r in range(R)], np.int8)
        d1 = d0.copy()
        d1[d0 == MODE_DISCOVER] = MODE_DISCOVER_UNION
        return _build(name, R=R, Hq=2, Hkv=2, D=64, dtype="f32", depths=2, n_planted=2,
                      seq_lens=lens, pool_factor=1, seed=base, depth_modes=[d0, d1], eta=eta)
    if name in ("ouro1.4b_1k", "ouro1.4b_4k"):
        R = num_rows or 64
        L = context or (1024 if name.endswith("1k") else 4096)
        lens = np.full(R, L, np.int32) if seq_lens is None else seq_lens
        return _build(name, R=R, Hq=16, Hkv=16, D=128, dtype="bf16", depths=4,
                      n_planted=4 if name.endswith("1k") else 8, seq_lens=lens,
                      pool_factor=1 if name.endswith("1k") else 2, seed=base,
                      depth_modes=_recurrent_schedule(R, 4), eta=eta)
    if name == "mixed_8k":
        R = num_rows or 32
        hi = context or 8192
        lo = min(1024, hi)
        lens = (_rng(base, 0, _TENSOR_IDS["lens"]).integers(lo, hi + 1, size=R).astype(np.int32)
                if seq_lens is None else seq_lens)
        modes = _rng(base, 0, _TENSOR_IDS["modes"]).choice(
            np.array([MODE_DENSE, MODE_DISCOVER, MODE_SPARSE], np.int8), size=R, p=[0.25, 0.25, 0.5])
        return _build(name, R=R, Hq=16, Hkv=16, D=128, dtype="bf16", depths=1, n_planted=8,
                      seq_lens=lens, pool_factor=1, seed=base, depth_modes=[modes], eta=eta)
    if name == "gqa_32k":
        R = num_rows or 8
        L = context or 32768
        lens = np.full(R, L, np.int32) if seq_lens is None else seq_lens
        return _build(name, R=R, Hq=32, Hkv=8, D=128, dtype="bf16", depths=4, n_planted=16,
                      seq_lens=lens, pool_factor=1, seed=base,
                      depth_modes=_recurrent_schedule(R, 4), eta=eta)
    raise KeyError(name)


WORKLOADS = tuple(BASE_SEEDS)


def sparse_scaling_inputs(R: int, H: int, D: int, L: int, k: int, seed: int,
                          device="cuda", page_size: int = 16, tile_tokens: int = 32,
                          shared_blocks: bool = False, num_q_heads: Optional[int] = None):
    """Inputs of the sparse-scaling measurement, drawn on the device (timing
    only; no parity check reads them): R rows of L tokens, H KV heads (and
    num_q_heads query heads, H by default: MHA), bf16 q/K/V ~ N(0,1) from a
    seeded device generator, each row's pages at a seeded permutation of a
    pool exactly the batch's size, and per (row, KV head) k distinct blocks
    drawn uniformly without replacement from the row's L / tile_tokens
    blocks (a seeded host draw; with shared_blocks, one draw per row that all
    its heads share).  Returns q, k_cache, v_cache, page_table, seq_lens and
    the mask [R, H, W] (int32 words)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    npg = -(-L // page_size)
    num_pages = R * npg
    q = torch.randn((R, num_q_heads or H, D), generator=gen, device=device).to(torch.bfloat16)
    k_cache = torch.randn((num_pages, page_size, H, D), generator=gen, device=device,
                          dtype=torch.bfloat16)
    v_cache = torch.randn((num_pages, page_size, H, D), generator=gen, device=device,
                          dtype=torch.bfloat16)
    perm = torch.randperm(num_pages, generator=gen, device=device).to(torch.int32)
    page_table = perm.view(R, npg).contiguous()
    seq_lens = torch.full((R,), L, dtype=torch.int32, device=device)
    nb = -(-L // tile_tokens)
    W = -(-nb // 32)
    rng = _rng(seed, 0, _TENSOR_IDS["plant"])
    draws = rng.random((R, 1 if shared_blocks else H, nb))
    chosen = np.broadcast_to(np.argsort(draws, axis=-1)[..., :min(k, nb)], (R, H, min(k, nb)))
    bits = np.zeros((R, H, 32 * W), dtype=bool)
    np.put_along_axis(bits, chosen, True, axis=-1)
    words = np.packbits(bits, axis=-1, bitorder="little").view(np.int32).reshape(R, H, W)
    support = torch.from_numpy(words.copy()).to(device)
    return {"q": q, "k_cache": k_cache, "v_cache": v_cache, "page_table": page_table,
            "seq_lens": seq_lens, "support": support, "num_pages": num_pages, "max_blocks": nb}
