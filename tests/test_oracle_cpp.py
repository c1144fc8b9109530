"""The C++ oracle (fp32, and the same code in double) against its pins (no GPU).

* Every pin the numpy oracle answers to (library routines in float64, brute
  force, closed forms, the pages' density example) also holds for the C++
  oracle: with float64 tolerances in double, and in fp32 with the bounds in
  `oracle_pins.F32_TOLERANCES`.
* The fp32 oracle agrees with the float64 numpy oracle on Ouro-1.4B-shaped
  and grouped-query batches within those bounds, and its masks are bit-exact
  wherever the float64 cutoff has margin (> 1e-4) and a mass gap (> 1e-5).
* The thread count never changes a result.
* Plausible mistakes planted in a patched copy of the C++ source (compiled on
  the CPU into a private library) are each caught by some pin.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest

from block_sparse_paged_split_gb300.workload import (MODE_DISCOVER, MODE_DISCOVER_UNION,
                                                     MODE_SPARSE, custom_workload, make_workload)
from oracle import cpp_oracle
from oracle import wise_oracle as numpy_oracle
from tests import oracle_pins


def f32_oracle(**kw):
    O = cpp_oracle.CppOracle("f32", **kw)
    O.TOLERANCES = oracle_pins.F32_TOLERANCES
    return O


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
@pytest.mark.parametrize("precision", ["f64", "f32"])
def test_cpp_oracle_pin(pin, precision):
    O = cpp_oracle.CppOracle("f64") if precision == "f64" else f32_oracle()
    fails = pin(O)
    assert not fails, "\n".join(fails[:20])


def _schedule_case(name):
    if name == "tiny":
        # 4 x 256 tokens, 2 heads, D=64, fp32 storage; rows run [dense,
        # discover, sparse, sparse] then [dense, union-discover, sparse, sparse]
        return make_workload("tiny")
    if name == "mha_1k":
        lens = np.array([1024, 1024, 1000, 0], np.int32)
        w = custom_workload(R=4, Hq=16, Hkv=16, D=128, dtype="bf16", depths=4, n_planted=4,
                            seq_lens=lens, pool_factor=2, seed=1001,
                            depth_modes=[np.full(4, m, np.int8) for m in
                                         (MODE_DISCOVER, MODE_DISCOVER_UNION, MODE_SPARSE,
                                          MODE_SPARSE)])
    else:
        lens = np.array([4096, 2500], np.int32)
        w = custom_workload(R=2, Hq=8, Hkv=2, D=128, dtype="bf16", depths=4, n_planted=16,
                            seq_lens=lens, pool_factor=1, seed=1004,
                            depth_modes=[np.full(2, m, np.int8) for m in
                                         (MODE_DISCOVER, MODE_DISCOVER_UNION, MODE_SPARSE,
                                          MODE_SPARSE)])
    return w


@pytest.mark.parametrize("case", ["tiny", "mha_1k", "gqa_4k"])
def test_f32_against_float64_oracle(case):
    """The 4-depth schedule; both oracles start every depth from the float64
    oracle's mask (sparse parity is checked on the same mask)."""
    w = _schedule_case(case)
    O32, O64 = f32_oracle(), cpp_oracle.CppOracle("f64")
    T = oracle_pins.F32_TOLERANCES
    sup = oracle_pins.empty_support(w)
    checked = 0
    for t in range(w.num_depths):
        d = w.depth_inputs(t)
        args = [oracle_pins.as_oracle_array(d[k]) for k in ("q", "k_cache", "v_cache")]
        modes = w.depth_modes[t]
        ref = numpy_oracle.decode_layer(*args, w.page_table, w.seq_lens, modes, sup, eta=w.eta)
        a = O32.decode_layer(*args, w.page_table, w.seq_lens, modes, sup, eta=w.eta)
        b = O64.decode_layer(*args, w.page_table, w.seq_lens, modes, sup, eta=w.eta)
        fin = np.isfinite(ref["lse"])
        assert np.array_equal(np.isfinite(a["lse"]), fin)
        assert np.abs(a["out"] - ref["out"]).max() <= T["out_atol"]
        assert np.abs(a["lse"][fin] - ref["lse"][fin]).max() <= T["lse"]
        assert np.abs(b["out"] - ref["out"]).max() <= 1e-12
        assert np.abs(b["lse"][fin] - ref["lse"][fin]).max() <= 1e-12
        for (r, h), dg in ref["diag"].items():
            assert np.abs(a["diag"][(r, h)]["p"] - dg["p"]).max() <= T["mass"]
            last_kept = dg["p"][dg["order"][dg["k"] - 1]]
            if dg["margin"] > 1e-4 and dg["gap"] > 1e-5 * last_kept:
                assert np.array_equal(a["diag"][(r, h)]["sel"], dg["sel"]), (t, r, h)
                checked += 1
        sup = ref["support"]
    assert checked > 0


def test_thread_count_never_changes_results():
    w = _schedule_case("mha_1k")
    d = w.depth_inputs(0)
    args = [oracle_pins.as_oracle_array(d[k]) for k in ("q", "k_cache", "v_cache")]
    sup = oracle_pins.empty_support(w)
    runs = []
    for threads in (1, 3, 8):
        O = cpp_oracle.CppOracle("f32", threads=threads)
        runs.append(O.decode_layer(*args, w.page_table, w.seq_lens, w.depth_modes[0], sup))
        assert O.last_threads == threads
    for other in runs[1:]:
        for key in ("out", "lse", "support"):
            assert np.array_equal(runs[0][key], other[key]), key


# ----------------------------------------------------------------------------- mutants
# (name, text in wise_oracle.cpp, replacement); each text occurs exactly once.
# Every mutant keeps its memory accesses inside the arrays it is given: a
# mutant library that read out of bounds could take the test process down
# instead of failing a pin.
MUTANTS = [
    ("scale_squared", "s[j] = scale * dot;", "s[j] = scale * scale * dot;"),
    ("slot_off_by_one", "const size_t krow = ((size_t(page) * PS + j % PS) * Hkv + g) * D;",
     "const size_t krow = ((size_t(page) * PS + (j + 1) % PS) * Hkv + g) * D;"),
    ("value_of_wrong_kv_head", "const size_t vrow = ((size_t(page) * PS + j % PS) * Hkv + g) * D;",
     "const size_t vrow = ((size_t(page) * PS + j % PS) * Hkv + (g + 1) % Hkv) * D;"),
    ("query_of_wrong_head", "static_cast<T>(stored(q, bf16, pair * D + d))",
     "static_cast<T>(stored(q, bf16, (size_t(r) * Hq + (h + 1) % Hq) * D + d))"),
    ("tile_sum_without_max", "lb += std::exp(s[j] - mb);", "lb += std::exp(s[j]);"),
    ("mass_not_normalised", "pm[b] = eb / Z;", "pm[b] = eb;"),
    ("last_token_dropped", "for (int j = lo; j < hi; ++j) {", "for (int j = lo; j + 1 < hi; ++j) {"),
    ("ties_to_higher_index", "(p[a] == p[b] && a < b)", "(p[a] == p[b] && a > b)"),
    ("strict_cutoff", "if (C[i] >= eta_t) {", "if (C[i] > eta_t) {"),
    ("one_extra_block", "k = i + 1;", "k = std::min(n, i + 2);"),
    ("union_overwrites", "bool bit = modes[r] == DISCOVER_UNION && mask_bit(before, b);",
     "bool bit = false;"),
    ("sparse_ignores_mask", "return mode != SPARSE || mask_bit(words, j / B);", "return true;"),
    ("bit_order_reversed", "return (words[b >> 5] >> (b & 31)) & 1u;",
     "return (words[b >> 5] >> (31 - (b & 31))) & 1u;"),
    ("compaction_drops_last_block", "if (modes[r] != SPARSE || mask_bit(w, b)) lst[c++] = b;",
     "if ((modes[r] != SPARSE || mask_bit(w, b)) && b + 1 < nb) lst[c++] = b;"),
    ("head_union_skips_last_head", "for (int g = 0; g < kv_heads; ++g)\n        any = any ||",
     "for (int g = 0; g + 1 < kv_heads; ++g)\n        any = any ||"),
    ("slot_ignores_page_size", "const size_t krow = ((size_t(page) * PS + j % PS) * Hkv + g) * D;",
     "const size_t krow = ((size_t(page) * PS + (j % PS) % 16) * Hkv + g) * D;"),
    ("padding_row_gets_output", "if (L <= 0) return;  // padding row",
     "if (L <= 0) { out[0] = 1.0; return; }"),
]


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name,text,replacement", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_some_pin_catches_cpp_mutant(name, text, replacement, mutant_dir):
    with open(cpp_oracle.SOURCE) as f:
        src = f.read()
    assert src.count(text) == 1, f"mutation site of {name} not unique"
    path = os.path.join(mutant_dir, f"{name}.cpp")
    with open(path, "w") as f:
        f.write(src.replace(text, replacement))
    lib = os.path.join(mutant_dir, f"lib{name}.so")
    subprocess.run(["g++"] + cpp_oracle.CXXFLAGS + [path, "-o", lib], check=True)
    caught = []
    for precision in ("f64", "f32"):
        O = cpp_oracle.CppOracle(precision, library=lib)
        if precision == "f32":
            O.TOLERANCES = oracle_pins.F32_TOLERANCES
        for pin in oracle_pins.ALL_PINS:
            try:
                fails = pin(O)
            except Exception as e:  # a crash is also a catch
                fails = [repr(e)]
            if fails:
                caught.append(f"{precision}:{pin.__name__}")
    assert any(c.startswith("f64") for c in caught) and any(c.startswith("f32") for c in caught), \
        f"{name} caught only by {caught}"


def test_build_entry_compiles_the_same_oracle():
    """build() compiles this oracle with the loader's own flags, to the path
    the loader reads, so the library it leaves is the one the tests load."""
    import __graft_entry__ as entry
    assert entry.ORACLE_CXXFLAGS == cpp_oracle.CXXFLAGS
    assert os.path.samefile(entry.ORACLE_SOURCE, cpp_oracle.SOURCE)
    assert os.path.abspath(entry.ORACLE_LIBRARY) == os.path.abspath(cpp_oracle.LIBRARY)
