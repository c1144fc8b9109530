"""The benchmark's multi-rank path on the CPU: two gloo ranks, each with its
own batch of the same shape (rows are independent; the data path has no
collective), timings reduced by maximum over ranks, and the whole-job rate
counted over every rank's rows."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

import bench
from block_sparse_paged_split_gb300.workload import make_workload


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank)})
    w_size, r, local = bench.rank_env()
    assert (w_size, r, local) == (world, rank, rank)
    tdist.init_process_group("gloo", rank=r, world_size=w_size)
    try:
        w = make_workload("ouro1.4b_1k", num_rows=2, context=64, seed=bench.rank_seed(r))
        q0 = w.depth_inputs(0)["q"].float()
        # Shapes agree across ranks; the rows themselves differ.
        meta = torch.tensor([w.num_rows, w.num_q_heads, w.num_kv_heads, w.head_dim,
                             int(w.seq_lens.sum())], dtype=torch.int64)
        metas = [torch.zeros_like(meta) for _ in range(world)]
        tdist.all_gather(metas, meta)
        sums = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        tdist.all_gather(sums, q0.double().sum().reshape(1))
        # Per-rank "timings": the slower rank sets the job's time.
        ms = [10.0 + 5.0 * r, 3.0 - r]
        red = bench.max_over_ranks(ms, tdist, "cpu")
        rate = bench.whole_job_rate(w_size, w.num_rows * w.num_depths, 7, red[0])
        with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
            json.dump({"metas": [m.tolist() for m in metas], "sums": [float(x) for x in sums],
                       "red": red, "rate": rate}, f)
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        with open(tmp_path / f"rank{r}.json") as f:
            res = json.load(f)
        metas = res["metas"]
        assert all(m == metas[0] for m in metas), "ranks disagree on the batch shape"
        assert res["sums"][0] != res["sums"][1], "both ranks drew the same rows"
        assert res["red"] == [15.0, 3.0]
        # 2 ranks x (2 rows x 4 depths) x 7 steps over the slowest rank's 15 ms
        assert res["rate"] == pytest.approx(2 * 8 * 7 / 15e-3)


def test_single_rank_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.rank_env() == (1, 0, 0)
    assert bench.rank_seed(0) is None and bench.rank_seed(1) != bench.rank_seed(2)
    assert bench.max_over_ranks([1.5, 2.5], None, "cpu") == [1.5, 2.5]
