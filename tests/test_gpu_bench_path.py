"""The benchmark's own launch configuration at the full workload sizes.

bench.py's `Pipeline` builds the WISE step the headline times: discover and
union-discover on work lists derived from the row lengths, the union depth's
finish writing the sparse depths' work list, the second sparse depth reading
its list before the dependency wait, no compaction launch (a mixed batch's
list is built for its modes).  Here that same step runs depth by depth (each
depth's output and the mask it leaves snapshotted) and as one replay of its
CUDA graph (bitwise equal
to the depth-by-depth run), and every depth is checked against the oracle on
the inputs the step actually used: every row at 1K, sampled rows beyond (the
oracle computes them one by one from the rows' own pages, gathered from the
device pool).  Each depth's oracle call gets the mask the GPU left before it,
so every comparison is like for like."""
import numpy as np
import pytest
import torch

import bench
import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300.workload import make_workload
from tests.gpu_harness import compare_masks, compare_outputs, oracle_module
from tests.oracle_pins import as_oracle_array

pytestmark = pytest.mark.gpu


def _oracle_rows(pipe, t, modes, sup_in, rows, oracle="f32"):
    """The oracle on depth t's inputs for the given rows, from those rows'
    pages only."""
    w = pipe.w
    d = pipe.depth[t]
    rows = np.asarray(rows)
    pt, sl = w.page_table[rows], w.seq_lens[rows]
    npg = -(-sl // w.page_size)
    used = np.unique(np.concatenate([pt[i, :npg[i]] for i in range(len(rows))] + [np.zeros(1, np.int32)]))
    pt_sub = np.full_like(pt, -1)
    for i in range(len(rows)):
        pt_sub[i, :npg[i]] = np.searchsorted(used, pt[i, :npg[i]])
    idx = torch.from_numpy(used.astype(np.int64)).cuda()
    k = d["k_cache"].index_select(0, idx).cpu()
    v = d["v_cache"].index_select(0, idx).cpu()
    q = d["q"][torch.from_numpy(rows.astype(np.int64)).cuda()].cpu()
    res = oracle_module(oracle).decode_layer(as_oracle_array(q), as_oracle_array(k),
                                             as_oracle_array(v), pt_sub, sl,
                                             np.asarray(modes, np.int8)[rows], sup_in[rows],
                                             eta=w.eta, tile_tokens=w.tile_tokens)
    res["eta"] = w.eta
    return res


def _sup(t):
    return t.cpu().numpy().view(np.uint32).copy()


def _depthwise(pipe, step):
    """Runs the step one depth at a time; per depth: the mask before it, its
    out (float64), out (raw), lse, and the mask after it."""
    snaps = []
    for entry in step:
        t = entry[0]
        before = _sup(pipe.support)
        pipe.run([entry])
        torch.cuda.synchronize()
        snaps.append({"t": t, "sup_in": before, "out": pipe.out[t].double().cpu().numpy(),
                      "out_raw": pipe.out[t].cpu(), "lse": pipe.lse[t].cpu().numpy(),
                      "support": _sup(pipe.support)})
    return snaps


def _status(pipe):
    return int(W.workspace_views(pipe.shape, pipe.ws)["status"].item())


def _check_step(name, rows=None, device_inputs=False, early=False, mixed_list=True):
    w = make_workload(name)
    pipe = bench.Pipeline(w, device_inputs=device_inputs, early_lists=early, mixed_list=mixed_list)
    for _ in range(2):  # the step as the benchmark replays it, on a used workspace
        pipe.run(pipe.wise_step)
    torch.cuda.synchronize()
    assert not any(c[0] == "compact" for _, m, calls in pipe.wise_step for c in calls
                   if mixed_list or "mixed" not in m), "a compaction launch in a compaction-free step"
    snaps = _depthwise(pipe, pipe.wise_step)
    assert _status(pipe) == 0
    # one graph replay of the whole step gives the same bits
    g = pipe.graph(pipe.wise_step)
    pipe.support.copy_(torch.from_numpy(snaps[0]["sup_in"].view(np.int32)).cuda())
    g.replay()
    torch.cuda.synchronize()
    for s in snaps:
        assert torch.equal(pipe.out[s["t"]].cpu(), s["out_raw"]), s["t"]
        assert np.array_equal(pipe.lse[s["t"]].cpu().numpy(), s["lse"]), s["t"]
    assert np.array_equal(_sup(pipe.support), snaps[-1]["support"])
    if isinstance(rows, str):  # "by_mode": the first three rows of each mode of the (single) depth
        m0 = w.depth_modes[0]
        rows = np.sort(np.concatenate([np.nonzero(m0 == m)[0][:3] for m in np.unique(m0)]))
    rows = np.arange(w.num_rows) if rows is None else np.asarray(rows)
    report = []
    for s in snaps:
        t = s["t"]
        modes = w.depth_modes[t]
        o = _oracle_rows(pipe, t, modes, s["sup_in"], rows)
        fails = compare_outputs(w, s, o, rows=rows)
        cm = compare_masks(w, s["support"], o, modes, rows=rows, support_in=s["sup_in"])
        fails += cm["fails"]
        assert not fails, (name, t, fails[:5])
        report.append((t, cm["checked"], cm["excluded_margin"], cm["excluded_gap"]))
        print(f"{name} depth {t}: masks bit-exact {cm['checked']}, near the margin "
              f"{cm['excluded_margin']}, near a mass tie {cm['excluded_gap']}")
    # the dense baseline step (dense list at every depth) against the oracle's dense
    dense = np.zeros(w.num_rows, np.int8)
    zero = np.zeros_like(snaps[0]["sup_in"])
    pipe.run(pipe.dense_step)
    torch.cuda.synchronize()
    for t in range(w.num_depths):
        o = _oracle_rows(pipe, t, dense, zero, rows)
        gd = {"out": pipe.out[t].double().cpu().numpy(), "lse": pipe.lse[t].cpu().numpy()}
        assert not compare_outputs(w, gd, o, rows=rows), (name, "dense", t)
    return report


def test_bench_step_1k_every_row():
    """64 rows x 1024 tokens, 16 heads: every row of every depth."""
    report = _check_step("ouro1.4b_1k")
    assert all(c > 0 for t, c, _, _ in report if t < 2)


def test_bench_step_1k_early_start():
    """The same with `bench.py --early`: consecutive depths on alternate slot
    sets, the dense-list depths and the second list-1 depth starting beside
    the previous finish; the graph replay then overlaps them, and still gives
    the depth-by-depth bits."""
    _check_step("ouro1.4b_1k", rows=np.arange(0, 64, 7), early=True)


def test_bench_step_4k_sampled():
    """64 rows x 4096 tokens (16-tile items), eight sampled rows."""
    _check_step("ouro1.4b_4k", rows=[0, 9, 17, 26, 38, 45, 54, 63], device_inputs=True)


def test_bench_step_mixed_8k_sampled():
    """32 ragged rows up to 8K in one mixed call on the work list built for
    its modes and masks (no compaction), the first three rows of each mode."""
    report = _check_step("mixed_8k", rows="by_mode", device_inputs=True)
    assert sum(c + m + g for _, c, m, g in report) > 0  # discover rows were among them


def test_bench_step_mixed_8k_on_a_compaction():
    """The same mixed call with `bench.py --no-mixed-list`: a compaction
    instead of the work list built for the modes."""
    report = _check_step("mixed_8k", rows="by_mode", device_inputs=True, mixed_list=False)
    assert sum(c + m + g for _, c, m, g in report) > 0


def test_bench_step_gqa_32k_sampled():
    """8 rows x 32K, 32 query / 8 KV heads (tensor-core path), three rows."""
    report = _check_step("gqa_32k", rows=[0, 3, 7], device_inputs=True)
    assert sum(c for _, c, _, _ in report) > 0
