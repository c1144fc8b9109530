"""The benchmark's one-line JSON contract: the CPU reference arm (the oracle
on a bounded sample) and, on a GPU, a short run of the GPU arm."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=600):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=timeout, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    return json.loads(lines[0])


BASE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config")


def test_reference_arm_line():
    out = _run("--impl", "reference", "--steps", "1", "--warmup", "1")
    for k in BASE_KEYS + ("impl", "cpu_baseline", "e2e"):
        assert k in out, k
    assert out["impl"] == "reference" and out["value"] > 0 and out["higher_is_better"]
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["value"] == out["value"]
    assert "workload" in out["config"]


@pytest.mark.gpu
def test_gpu_arm_line():
    out = _run("--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    for k in BASE_KEYS + ("roofline", "e2e", "gpu_launches", "clocks", "modes"):
        assert k in out, k
    assert out["n_gpus"] == 1 and out["steps"] == 3 and out["warmup"] == 3
    assert out["value"] > 0 and out["ms_per_step"] > 0 and out["scaling"] == "weak"
    roof = out["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in roof, k
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert 0 < roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-3)
    e2e = out["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["value"] < out["value"] * 1.05  # the copies cost something
    assert out["gpu_launches"] > 0
    assert set(out["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert out["config"]["workload"].startswith("ouro1.4b_1k")
    assert 0 < out["config"]["support_density_blocks"] <= 1
    # the default run also covers the 4K, mixed 8K and 32K grouped-query workloads
    sweep = out["modes_by_workload"]
    assert set(sweep) == {"ouro1.4b_4k", "mixed_8k", "gqa_32k"}
    for name, res in sweep.items():
        assert res["step_ms"] > 0 and res["rows_per_s"] > 0 and res["dense_step_ms"] > 0, name
        for mode, row in res["modes"].items():
            assert row["call_us"] >= row["partial_us"] > 0, (name, mode)
            assert 0 < row["call_frac_of_measured_hbm"] <= row["partial_frac_of_measured_hbm"]
    # the grouped-query workload over the selection threshold: a lower eta
    # leaves the sparse depths fewer blocks
    pts = sweep["gqa_32k"]["eta_sweep"]
    assert [p["eta"] for p in pts] == [0.8, 0.9, 0.95, 0.99]
    dens = [p["support_density_blocks"] for p in pts]
    assert all(0 < d <= 1 for d in dens) and dens == sorted(dens)
    assert all(p["step_ms"] > 0 and p["dense_step_ms"] > 0 for p in pts)
    # no depth of any workload's step launches a compaction: the sparse
    # depths run on the list the union depth built, the dense and discover
    # depths on the dense list, the mixed call on a list built for its modes
    assert "no compaction launch" in out["config"]["workload"]
    for mode, row in out["modes"].items():
        if mode.startswith("depth"):
            assert "compact" not in row["kernels_us"], mode
    for name, res in sweep.items():
        for mode, row in res["modes"].items():
            if mode.startswith("depth"):
                assert "compact" not in row["kernels_us"], (name, mode)
    assert "build_list" in sweep["mixed_8k"]["modes"]["depth0_mixed"]["kernels_us"]


@pytest.mark.gpu
def test_sparse_scaling_point():
    """One point of the sparse-scaling measurement (8 rows, 4K context, 8
    selected tiles per head): per-kernel times that add up to the call, on the
    list built from the mask and on a compaction, and selected bytes equal to
    rows x heads x tiles x 32 tokens x 512 B."""
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--sparse-scaling",
                          "--point", "4096:8", "--rows", "8"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    out = json.loads([l for l in res.stdout.splitlines() if l.startswith("{")][-1])
    (pt,) = out["sparse_scaling"]
    assert pt["context"] == 4096 and pt["selected_tiles_per_head"] == 8 and out["rows"] == 8
    assert pt["selected_kv_bytes"] == 8 * 16 * 8 * 32 * 512
    parts = pt["sparse_build_us"] + pt["sparse_partial_us"] + pt["sparse_finish_us"]
    assert 0 < parts <= pt["sparse_call_us"] * 1.01
    parts = pt["compaction_us"] + pt["compaction_partial_us"] + pt["compaction_finish_us"]
    assert 0 < parts <= pt["compaction_call_us"] * 1.01
    assert 0 < pt["partial_frac"] < 1.5 and 0 < pt["call_frac"] <= pt["partial_frac"]


@pytest.mark.gpu
def test_sparse_scaling_point_grouped_query():
    """The same measurement on the tensor-core path: 32 query / 8 KV heads,
    4 rows at 8K context, 16 selected tiles per (row, KV head): the selected
    bytes count each KV tile once for its four query heads."""
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--sparse-scaling",
                          "--gqa", "--point", "8192:16", "--rows", "4"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    out = json.loads([l for l in res.stdout.splitlines() if l.startswith("{")][-1])
    (pt,) = out["sparse_scaling"]
    assert out["heads"] == 8 and out["q_heads"] == 32 and out["rows"] == 4
    assert pt["selected_kv_bytes"] == 4 * 8 * 16 * 32 * 512
    assert 0 < pt["sparse_partial_us"] <= pt["sparse_call_us"] * 1.01


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun only rank 0 runs the reference arm; the others print
    nothing and exit 0."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    assert not [l for l in res.stdout.splitlines() if l.startswith("{")]


def test_traffic_record_round_trip(tmp_path, monkeypatch):
    """An ncu '--page raw --csv' export (header row, units row, one row per
    launch) becomes per-launch DRAM bytes keyed by the kernel's source hash;
    the bench scales them to its own rows and drops them once the kernel's
    source or the workload differs."""
    import bench
    raw = tmp_path / "raw.csv"
    raw.write_text(
        '"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum"\n'
        '"","","Mbyte","Kbyte"\n'
        '"0","void wise::partial_kernel<...>(...)","100","500"\n'
        '"1","void wise::finish_short_kernel<...>(...)","7","7"\n'
        '"2","void wise::partial_kernel<...>(...)","1,000","0"\n')
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "traffic.json"))
    bench.record_traffic(str(raw), 32, "ouro1.4b_1k")
    rec = json.loads((tmp_path / "traffic.json").read_text())
    assert rec["per_launch_bytes"] == [100.5e6, 1000e6]
    assert rec["kernel_source_sha256"] == bench.kernel_source_hash()
    assert bench.recorded_traffic(64, "ouro1.4b_1k") == pytest.approx((100.5e6 + 1000e6) / 2 * 2)
    assert bench.recorded_traffic(64, "gqa_32k") is None
    rec["kernel_source_sha256"] = "0" * 64
    (tmp_path / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic(64, "ouro1.4b_1k") is None
