"""Python handle on the C++ oracle (oracle/wise_oracle.cpp).

TEST INFRASTRUCTURE ONLY, like the rest of this folder: the tests, the smoke
check and the benchmark's CPU-baseline leg use it; the library never does.

`CppOracle("f32")` is the fp32 oracle (fp32 arithmetic throughout);
`CppOracle("f64")` runs the same C++ code in double.  Both expose the numpy
oracle's function names and return forms (decode_layer, select_blocks,
support_union, support_head_union, union_density, compact_tiles), so the same
pins run on all three.  The shared library is compiled here with g++ on first
use (or by the build entry point), with floating-point contraction off so
that x86 and Arm builds round alike.
"""
from __future__ import annotations

import ctypes
import hashlib
import math
import os
import subprocess
import threading
from typing import Dict, Tuple

import numpy as np

from . import wise_oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "wise_oracle.cpp")
LIBDIR = os.path.join(HERE, "lib")
LIBRARY = os.path.join(LIBDIR, "libwise_oracle.so")
CXXFLAGS = ["-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-ffp-contract=off"]

_lock = threading.Lock()
_lib = None


def _source_stamp(source: str = SOURCE, flags=CXXFLAGS) -> str:
    h = hashlib.sha256()
    with open(source, "rb") as f:
        h.update(f.read())
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def compile_oracle(source: str = SOURCE, output: str = LIBRARY) -> str:
    """g++ the oracle into a shared library (skipped when the stamp matches)."""
    stamp_file = output + ".stamp"
    stamp = _source_stamp(source)
    if os.path.exists(output) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return output
    os.makedirs(os.path.dirname(output), exist_ok=True)
    tmp = output + f".{os.getpid()}.tmp"
    cxx = os.environ.get("CXX", "g++")
    res = subprocess.run([cxx] + CXXFLAGS + [source, "-o", tmp], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"g++ failed on {source}:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, output)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return output


class _Problem(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("q_heads", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
                ("max_pages_per_row", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("mask_words", ctypes.c_int32), ("bf16_storage", ctypes.c_int32),
                ("scale", ctypes.c_double), ("eta", ctypes.c_double)]


class _Results(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("out", "lse", "support", "tile_max", "tile_sum", "mass", "selected", "order",
                 "k_star", "margin", "gap")]


def load(path: str = None) -> ctypes.CDLL:
    """The oracle library (compiled if missing or stale).  `path` loads another
    build of it (the mutation tests compile patched copies)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(compile_oracle()))
        return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    for prec in ("f32", "f64"):
        fn = getattr(lib, f"wise_oracle_decode_{prec}")
        fn.argtypes = [ctypes.POINTER(_Problem), vp, vp, vp, vp, vp, vp, vp,
                       ctypes.POINTER(_Results), i32]
        fn.restype = i32
        fn = getattr(lib, f"wise_oracle_select_{prec}")
        fn.argtypes = [vp, i32, dbl, vp, vp, vp, vp]
        fn.restype = i32
    lib.wise_oracle_support_union.argtypes = [vp, vp, vp, i64]
    lib.wise_oracle_support_union.restype = None
    lib.wise_oracle_head_union.argtypes = [vp, i32, i32, i32, vp]
    lib.wise_oracle_head_union.restype = None
    lib.wise_oracle_union_density.argtypes = [vp, vp, i32, i32, i32, i32]
    lib.wise_oracle_union_density.restype = dbl
    lib.wise_oracle_compact.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp]
    lib.wise_oracle_compact.restype = None
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class CppOracle:
    """The C++ oracle in one precision ("f32" or "f64"), with the numpy
    oracle's call forms.  `threads` <= 0 uses every hardware thread."""

    def __init__(self, precision: str = "f32", threads: int = 0, library: str = None):
        if precision not in ("f32", "f64"):
            raise ValueError(precision)
        self.precision = precision
        self.threads = threads
        self.lib = load(library)
        self.last_threads = 0

    # ------------------------------------------------------------------ decode
    def decode_layer(self, q, k_cache, v_cache, page_table, seq_lens, modes, support, *,
                     eta: float = 0.95, tile_tokens: int = 32, scale: float = 0.0,
                     diagnostics: bool = True) -> Dict[str, object]:
        q, k_cache, v_cache = (np.ascontiguousarray(x) for x in (q, k_cache, v_cache))
        kinds = {x.dtype for x in (q, k_cache, v_cache)}
        if kinds == {np.dtype(np.uint16)}:
            bf16 = 1
        elif kinds == {np.dtype(np.float32)}:
            bf16 = 0
        else:
            raise TypeError(f"q, K and V must all be bf16 bits (uint16) or all float32: {kinds}")
        R, Hq, D = q.shape
        num_pages, P, Hkv, D2 = k_cache.shape
        assert D2 == D and v_cache.shape == k_cache.shape
        page_table = np.ascontiguousarray(page_table, np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, np.int32)
        modes = np.ascontiguousarray(modes, np.int8)
        support = np.ascontiguousarray(support, np.uint32)
        W = support.shape[2]
        NB = 32 * W
        # The C++ code trusts its indices: check them here so a bad input
        # raises instead of reading out of bounds.
        if page_table.shape[0] != R or seq_lens.shape[0] != R or modes.shape[0] != R or \
                support.shape[:2] != (R, Hkv) or Hq % Hkv:
            raise ValueError("inconsistent batch shapes")
        for r in range(R):
            L = int(seq_lens[r])
            if L < 0 or L > page_table.shape[1] * P or -(-L // tile_tokens) > NB:
                raise ValueError(f"row {r}: length {L} exceeds its pages or its mask")
            used = page_table[r, :-(-L // P)]
            if used.size and (used.min() < 0 or used.max() >= num_pages):
                raise ValueError(f"row {r}: page id outside the pool")
        prob = _Problem(R, Hq, Hkv, D, P, tile_tokens, page_table.shape[1], num_pages, W, bf16,
                        float(scale), float(eta))
        out = np.zeros((R, Hq, D))
        lse = np.zeros((R, Hq))
        new_support = np.zeros_like(support)
        tmax = np.zeros((R, Hq, NB))
        tsum = np.zeros((R, Hq, NB))
        mass = np.zeros((R, Hq, NB))
        sel = np.zeros((R, Hq, NB), np.uint8)
        order = np.zeros((R, Hq, NB), np.int32)
        kst = np.zeros((R, Hq), np.int32)
        margin = np.zeros((R, Hq))
        gap = np.zeros((R, Hq))
        res = _Results(*(_ptr(a) for a in (out, lse, new_support, tmax, tsum, mass, sel, order,
                                           kst, margin, gap)))
        fn = getattr(self.lib, f"wise_oracle_decode_{self.precision}")
        used = fn(ctypes.byref(prob), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                  _ptr(seq_lens), _ptr(modes), _ptr(support), ctypes.byref(res), self.threads)
        if used < 0:
            raise ValueError("the oracle rejected the shape")
        self.last_threads = used
        if scale == 0.0:
            scale = 1.0 / math.sqrt(D)
        diag: Dict[Tuple[int, int], Dict[str, object]] = {}
        if diagnostics:
            for r in range(R):
                L = int(seq_lens[r])
                if L == 0 or int(modes[r]) not in (1, 2):
                    continue
                nb = -(-L // tile_tokens)
                for h in range(Hq):
                    diag[(r, h)] = {"m_b": tmax[r, h, :nb].copy(), "l_b": tsum[r, h, :nb].copy(),
                                    "p": mass[r, h, :nb].copy(), "sel": sel[r, h, :nb] == 1,
                                    "k": int(kst[r, h]), "order": order[r, h, :nb].copy(),
                                    "margin": float(margin[r, h]), "gap": float(gap[r, h])}
        return {"out": out, "lse": lse, "support": new_support, "diag": diag, "scale": scale}

    def decode_layer_slots(self, q, k_cache, v_cache, page_table, seq_lens, modes, pool,
                           row_slot, layer: int, **kw) -> Dict[str, object]:
        """decode_layer with masks addressed by slot and layer: the index
        layer is the numpy oracle's (gather, call, store back; no arithmetic),
        the call is this oracle's."""
        return wise_oracle.decode_layer_slots(q, k_cache, v_cache, page_table, seq_lens, modes,
                                              pool, row_slot, layer, decode=self.decode_layer,
                                              **kw)

    # ------------------------------------------------------------------ selection
    def select_blocks(self, p, eta: float) -> Dict[str, object]:
        p = np.ascontiguousarray(p, np.float64)
        n = p.shape[0]
        order = np.zeros(n, np.int32)
        sel = np.zeros(n, np.uint8)
        margin = np.zeros(1)
        gap = np.zeros(1)
        fn = getattr(self.lib, f"wise_oracle_select_{self.precision}")
        k = fn(_ptr(p), n, float(eta), _ptr(order), _ptr(sel), _ptr(margin), _ptr(gap))
        return {"sel": sel == 1, "k": int(k), "order": order, "margin": float(margin[0]),
                "gap": float(gap[0])}

    # ------------------------------------------------------------------ masks
    def support_union(self, dst, src) -> np.ndarray:
        a = np.ascontiguousarray(dst, np.uint32)
        b = np.ascontiguousarray(src, np.uint32)
        assert a.shape == b.shape
        out = np.zeros_like(a)
        self.lib.wise_oracle_support_union(_ptr(a), _ptr(b), _ptr(out), a.size)
        return out

    def support_head_union(self, support) -> np.ndarray:
        sup = np.ascontiguousarray(support, np.uint32)
        R, Hkv, W = sup.shape
        out = np.zeros_like(sup)
        self.lib.wise_oracle_head_union(_ptr(sup), R, Hkv, W, _ptr(out))
        return out

    def union_density(self, support, seq_lens, B: int) -> float:
        sup = np.ascontiguousarray(support, np.uint32)
        lens = np.ascontiguousarray(seq_lens, np.int32)
        R, Hkv, W = sup.shape
        return float(self.lib.wise_oracle_union_density(_ptr(sup), _ptr(lens), R, Hkv, W, B))

    # ------------------------------------------------------------------ compaction
    def compact_tiles(self, support, modes, seq_lens, B: int):
        sup = np.ascontiguousarray(support, np.uint32)
        modes = np.ascontiguousarray(modes, np.int8)
        lens = np.ascontiguousarray(seq_lens, np.int32)
        R, Hkv, W = sup.shape
        NB = 32 * W
        lists = np.zeros((R, Hkv, NB), np.int32)
        counts = np.zeros((R, Hkv), np.int32)
        self.lib.wise_oracle_compact(_ptr(sup), _ptr(modes), _ptr(lens), R, Hkv, W, B,
                                     _ptr(lists), _ptr(counts))
        return {"lists": [[lists[r, g, :counts[r, g]].copy() for g in range(Hkv)]
                          for r in range(R)],
                "counts": counts}
