#!/usr/bin/env python3
"""Benchmark of WISE working-set paged decode attention on GB300.

One step = one decode step of one layer over the Ouro-1.4B-shaped batch
(64 rows x 1024 tokens, 16 heads MHA, head dim 128, bf16, page 16, B=32)
through its four recurrent depths, each with its own K/V pool:

    depth 0  discover         partial + finish, on the work list the partial
                              pass derives from the row lengths (dense list)
    depth 1  union-discover   the same; its finish also writes the sparse
                              depths' work list (list 1)
    depth 2  sparse           partial + finish on list 1
    depth 3  sparse           partial + finish on list 1 (read before the
                              dependency wait)

No depth launches a compaction; a depth that mixes sparse rows with others
(the mixed 8K batch) takes a work list built for its modes (wise_build_list).
`value` is decode attention rows per second over the whole step (4 x 64
row-calls per step), timed over CUDA-graph replays of the step.  The same K
steps launched eagerly, every launch bracketed by CUDA events on the
launching stream, give the per-mode times and the roofline of the dominant
kernel (the split partial pass); `e2e` adds each step's host copies.  The
dense baseline runs the same launches with every row dense.  Inputs per step
are 2.1 GB of K/V (larger than the 129 MB L2).  The other workloads (4K,
mixed 8K, GQA 32K) follow in `modes_by_workload`.

`--impl reference` times the CPU oracle (the definition the kernels are
checked against) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "ouro1.4b_1k"

# The pages' own end-to-end figures for the same shapes, quoted beside ours as
# context (WISE over the best dense decode, Ouro-1.4B in a full serving engine
# on one GH200, two repeats each) [WISE PR, "Results"].  Another machine and a
# whole engine step (attention is only part of it): context, not a target.
PAGES_SPEEDUP = {
    "ouro1.4b_1k": "1.08-1.19x decode throughput over dense (1K context x 64 requests, GH200)",
    "ouro1.4b_4k": "1.16-1.39x decode throughput over dense (4K context x 20 requests, GH200)",
    "mixed_8k": "1.23-1.41x decode throughput over dense (8K context x 10 requests, GH200)",
}
METRIC = "decode attention rows/s (WISE 4-depth step: discover, union, sparse, sparse)"
UNIT = "rows/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--rows", type=int, default=None,
                   help="fewer rows of the same workload (small profiling case)")
    p.add_argument("--eta", type=float, default=None,
                   help="selection threshold (default: the workload's, 0.95)")
    p.add_argument("--tiles-per-item", type=int, default=0,
                   help="split work-item size (0: the library default)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--lse-discover", action="store_true",
                   help="discover depths rebuild block masses from the LSE by a second read "
                        "of K instead of recording tile statistics in the partial pass")
    p.add_argument("--head-union", action="store_true",
                   help="sparse depths attend the head union of each row's mask")
    p.add_argument("--overlap", action="store_true",
                   help="alternate the two slot sets and start a depth that reuses the previous "
                        "compaction while the previous finish runs (measured: no gain at 1K)")
    p.add_argument("--no-sweep", action="store_true",
                   help="measure only the headline workload (the default run also measures "
                        "the 4K, mixed 8K and 32K grouped-query workloads)")
    p.add_argument("--early", action="store_true",
                   help="depths on the dense list or a ready list 1 start beside the previous "
                        "finish on the other slot set (measured: no gain; off by default)")
    p.add_argument("--no-dense-list", action="store_true",
                   help="dense and discover depths get a compaction instead of deriving their "
                        "work list from the row lengths")
    p.add_argument("--no-sparse-list", action="store_true",
                   help="sparse depths get their own compaction instead of the work list the "
                        "previous depth's finish builds")
    p.add_argument("--no-mixed-list", action="store_true",
                   help="depths that mix sparse rows with others get a compaction instead of "
                        "the work list wise_build_list builds for their modes (measured: the "
                        "same step time at 8K; the built list stays flat past it)")
    p.add_argument("--fold", action="store_true",
                   help="fold the finish into the partial pass (rows of at most 64 blocks)")
    p.add_argument("--sparse-scaling", action="store_true",
                   help="time one sparse call (64 rows, 16 heads MHA, D=128) at contexts "
                        "1K-128K with 8 selected tiles per (row, head), and at 8K with 1-256 "
                        "selected tiles; prints one JSON line with the table")
    p.add_argument("--point", default=None, metavar="CONTEXT:TILES",
                   help="with --sparse-scaling: time only this point (e.g. 8192:1)")
    p.add_argument("--gqa", action="store_true",
                   help="with --sparse-scaling: 32 query / 8 KV heads (the tensor-core path), "
                        "16 rows, contexts 4K-128K")
    p.add_argument("--shared-blocks", action="store_true",
                   help="with --sparse-scaling: every head of a row selects the same blocks")
    p.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    p.add_argument("--record-traffic", default=None, metavar="RAW_CSV",
                   help="store the DRAM bytes of the partial-kernel launches in an ncu "
                        "'--page raw --csv' export (one WISE step of --rows rows) with the "
                        "kernel's source hash, and exit")
    return p.parse_args()


# ----------------------------------------------------------------------------- oracle leg
def oracle_sample_main(spec_json: str) -> None:
    """Runs in a child process (no CUDA context): times the C++ fp32 oracle on
    `rows` rows of the workload through the 4-depth schedule, on every host
    thread and on one, each for at least its target seconds (or a fixed number
    of passes when `reps` is given)."""
    import numpy as np
    from block_sparse_paged_split_gb300.workload import make_workload
    from oracle.cpp_oracle import CppOracle

    spec = json.loads(spec_json)
    w = make_workload(spec["workload"], num_rows=spec["rows"], **eta_kw(spec.get("eta")))
    inputs = []
    for t in range(w.num_depths):
        d = w.depth_inputs(t)
        conv = {}
        for k, v in d.items():
            conv[k] = v.view(torch_int16()).numpy().view(np.uint16) if v.dtype == bf16() else v.numpy()
        inputs.append(conv)
    sup = np.zeros((w.num_rows, w.num_kv_heads, -(-w.max_blocks // 32)), np.uint32)

    mode_names = {0: "dense", 1: "discover", 2: "discover_union", 3: "sparse"}

    def depth_name(m):
        u = {int(x) for x in m}
        return mode_names[u.pop()] if len(u) == 1 else "mixed"

    per_depth = [0.0] * w.num_depths

    def one_pass(O):
        s = sup
        for t in range(w.num_depths):
            d = inputs[t]
            t0 = time.perf_counter()
            s = O.decode_layer(d["q"], d["k_cache"], d["v_cache"], w.page_table, w.seq_lens,
                               w.depth_modes[t], s, eta=w.eta, tile_tokens=w.tile_tokens,
                               diagnostics=False)["support"]
            per_depth[t] += time.perf_counter() - t0

    report = {"row_calls_per_pass": w.num_rows * w.num_depths}
    for key, threads, target in (("all", 0, spec["seconds"]), ("one", 1, spec["seconds_1t"])):
        if target <= 0:
            continue
        O = CppOracle("f32", threads=threads)
        for _ in range(max(1, spec.get("warmup", 1))):  # untimed: page-in, thread start
            one_pass(O)
        per_depth[:] = [0.0] * w.num_depths
        passes, t0 = 0, time.perf_counter()
        while True:
            one_pass(O)
            passes += 1
            el = time.perf_counter() - t0
            if (spec.get("reps") and passes >= spec["reps"]) or (not spec.get("reps") and el >= target):
                break
        report[key] = {"seconds": el, "passes": passes, "threads": O.last_threads,
                       "per_mode": {f"depth{t}_{depth_name(w.depth_modes[t])}":
                                    round(w.num_rows * passes / per_depth[t], 1)
                                    for t in range(w.num_depths)}}
    print(json.dumps(report))


def eta_kw(eta) -> dict:
    return {} if eta is None else {"eta": eta}


def torch_int16():
    import torch
    return torch.int16


def bf16():
    import torch
    return torch.bfloat16


def run_oracle_sample(workload: str, rows: int, seconds: float = 10.0, seconds_1t: float = 3.0,
                      reps: int = 0, warmup: int = 1, eta=None) -> dict:
    """The CPU baseline: the C++ fp32 oracle (the definition the kernels are
    checked against, untuned) on `rows` rows of the workload, in a child
    process with no GPU visible."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    spec = json.dumps({"workload": workload, "rows": rows, "seconds": seconds,
                       "seconds_1t": seconds_1t, "reps": reps, "warmup": warmup, "eta": eta})
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", spec],
                         capture_output=True, text=True, env=env, check=True)
    out = json.loads(res.stdout.strip().splitlines()[-1])
    per = out["row_calls_per_pass"]
    a = out["all"]
    value = per * a["passes"] / a["seconds"]
    sample = (f"{rows} rows of {workload} (same recipe), {a['passes']}x the 4-depth schedule "
              f"through the C++ fp32 oracle on {a['threads']} host threads ({a['seconds']:.1f} s)")
    result = {"value": value, "unit": UNIT, "cores": a["threads"], "kind": "oracle",
              "per_mode_rows_per_s": a["per_mode"]}
    if "one" in out:
        o = out["one"]
        result["value_1_thread"] = round(per * o["passes"] / o["seconds"], 3)
        sample += f"; 1 thread: {o['passes']}x ({o['seconds']:.1f} s)"
    result["sample"] = sample
    return result


# ----------------------------------------------------------------------------- traffic
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "partial_kernel_traffic.json")
KERNEL_SOURCES = ("partial_kernel.cuh", "partial_bf16.cu", "finish_short.cuh", "common.cuh", "internal.h")


def _code_only(text: str) -> str:
    """C++/CUDA source without comments and with whitespace collapsed, so the
    hash follows the code, not its commentary."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "block_sparse_paged_split_gb300", "csrc", n)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def record_traffic(raw_csv: str, rows: int, workload: str) -> None:
    """Per-launch dram__bytes_read.sum + dram__bytes_write.sum of the
    partial-kernel launches in an ncu raw CSV, in launch order (the four
    depths of one step), saved with the kernel's source hash."""
    import csv
    with open(raw_csv) as f:
        table = list(csv.reader(f))
    head = table[0]
    col = {n: i for i, n in enumerate(head)}
    units = table[1]
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    launches = []
    for row in table[2:]:
        if "partial_kernel" not in row[col["Kernel Name"]]:
            continue
        total = 0.0
        for m in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            total += float(row[col[m]].replace(",", "")) * scale[units[col[m]]]
        launches.append(total)
    out = {"kernel_source_sha256": kernel_source_hash(), "workload": workload,
           "captured_rows": rows, "per_launch_bytes": launches,
           "note": "one WISE step (depths 0-3) of the captured rows; scaled to the bench's "
                   "rows by rows/captured_rows (traffic grows in proportion to rows)"}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out))


def recorded_traffic(rows: int, workload: str):
    """Average per-launch DRAM bytes of the partial pass, or None when no
    capture exists for the current kernel source and this workload."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f)
    if (rec.get("kernel_source_sha256") != kernel_source_hash() or not rec.get("per_launch_bytes")
            or rec.get("workload") != workload):
        return None
    per = rec["per_launch_bytes"][:4]
    return sum(per) / len(per) * rows / rec["captured_rows"]


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm
def pack(tensors, device):
    """One byte buffer holding the tensors back to back (each at a 256-byte
    aligned offset) and views of it with the tensors' shapes and dtypes (on
    the CPU the buffer is pinned and the views hold the tensors' values)."""
    import torch
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off = (off + t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8, device=device, pin_memory=device.type == "cpu")
    views = []
    for t, o in zip(tensors, offs):
        v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        if device.type == "cpu":
            v.copy_(t)
        views.append(v)
    return buf, views


class Pipeline:
    """The 4-depth WISE step with all ctypes arguments bound once."""

    def __init__(self, w, tiles_per_item: int = 0, fold: bool = False, head_union: bool = False,
                 lse_discover: bool = False, overlap: bool = False, share=None,
                 sparse_list: bool = True, device_inputs: bool = False, dense_list: bool = True,
                 early_lists: bool = False, mixed_list: bool = True):
        import numpy as np
        import torch
        import block_sparse_paged_split_gb300 as W
        from block_sparse_paged_split_gb300 import wise

        self.W, self.np, self.torch = W, np, torch
        self.w = w
        lib = wise.library()
        self.lib = lib
        self.shape = W.make_shape(num_rows=w.num_rows, num_q_heads=w.num_q_heads,
                                  num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                                  page_size=w.page_size, max_pages_per_row=w.max_pages_per_row,
                                  num_pages=w.num_pages, max_blocks=w.max_blocks,
                                  dtype=W.DTYPE_BF16 if w.dtype == "bf16" else W.DTYPE_F32,
                                  eta=w.eta, tiles_per_item=tiles_per_item)
        dev = torch.device("cuda")
        if share is None and device_inputs:
            # K/V drawn on the device with the same recipe (Workload.
            # depth_inputs_device): the long workloads' host draws take
            # minutes, and timing does not depend on the values.
            drawn = [w.depth_inputs_device(t) for t in range(w.num_depths)]
            self.host = [{"q": d["q"]} for d in drawn]
            self.depth = [{k: v for k, v in d.items() if k != "q"} for d in drawn]
            del drawn
        elif share is None:
            self.host = [w.depth_inputs(t) for t in range(w.num_depths)]
            self.depth = [{k: v.to(dev) for k, v in d.items() if k != "q"} for d in self.host]
        else:
            # A second buffer set over the same resident K/V (the pipelined
            # end-to-end region alternates two): its own step inputs, outputs,
            # mask and workspace.
            self.host = share.host
            self.depth = [{k: v for k, v in d.items() if k != "q"} for d in share.depth]
        # The per-step inputs (every depth's q, the page table, the lengths,
        # every depth's modes) live in one device buffer and the per-step
        # outputs (every depth's out and lse, the mask) in another, so a step
        # moves its inputs and results with one copy each way.
        ins = ([d["q"] for d in self.host] + [torch.from_numpy(w.page_table),
               torch.from_numpy(w.seq_lens)] + [torch.from_numpy(m) for m in w.depth_modes])
        self.in_host, in_views = pack(ins, torch.device("cpu"))
        self.in_dev, in_dev_views = pack(ins, dev)
        self.in_dev.copy_(self.in_host)
        nd = w.num_depths
        for t in range(nd):
            self.depth[t]["q"] = in_dev_views[t]
        self.page_table, self.seq_lens = in_dev_views[nd], in_dev_views[nd + 1]
        self.modes = in_dev_views[nd + 2:]
        self.dense_modes = torch.zeros(w.num_rows, dtype=torch.int8, device=dev)
        outs = ([torch.empty(d["q"].shape, dtype=d["q"].dtype) for d in self.host] +
                [torch.empty((w.num_rows, w.num_q_heads), dtype=torch.float32) for _ in self.host] +
                [torch.zeros((w.num_rows, w.num_kv_heads, W.mask_words(self.shape)), dtype=torch.int32)])
        self.out_dev, out_views = pack(outs, dev)
        self.out_dev.zero_()
        self.out = out_views[:nd]
        self.lse = out_views[nd:2 * nd]
        self.support = out_views[2 * nd]
        self.ws = W.alloc_workspace(self.shape)
        self.stream = torch.cuda.current_stream()
        S = ctypes.byref(self.shape)
        st = self.stream.cuda_stream
        ws, nws = self.ws.data_ptr(), self.ws.numel()
        sup = self.support.data_ptr()
        pt, sl = self.page_table.data_ptr(), self.seq_lens.data_ptr()

        # fold=True: the partial pass with the finish folded in
        # (wise_decode_partial_finish; one launch for rows of at most 64 blocks
        # and 8 splits).  Measured slower than the two launches (every item
        # then pays a device-wide release and a ticket round trip), so the
        # step keeps them apart by default.
        T = tiles_per_item or 8
        self.folded = fold and w.max_blocks <= 64 and -(-w.max_blocks // T) <= 8

        # overlap=True: consecutive depths alternate the workspace's two slot
        # sets, and a depth that reuses the previous depth's compaction starts
        # its partial pass while that depth's finish still runs
        # (WISE_FLAG_EARLY_START: the partial reads nothing the finish writes).
        # Measured: no gain at 1K -- the partial's CTAs need a whole SM, so
        # they start only as the finish's CTAs leave -- hence off by default.
        self.overlap = overlap and not fold and not lse_discover

        # sparse_list=True: the finish of the depth before a run of all-sparse
        # depths also writes their work list (WISE_FLAG_BUILD_SPARSE_LIST), and
        # those depths run on it (WISE_FLAG_SPARSE_LIST) with no compaction
        # launch.  The variants above keep a compaction per sparse depth.
        self.sparse_list = sparse_list and not (fold or overlap or head_union or lse_discover)
        # dense_list=True: depths with no sparse row derive their work list
        # from the row lengths in the partial pass (WISE_FLAG_DENSE_LIST), so
        # with the sparse list the step launches no compaction at all.
        self.dense_list = (dense_list and w.num_rows <= W.DENSE_LIST_MAX_ROWS and
                           not (fold or overlap or head_union or lse_discover))
        # mixed_list=True: a depth that mixes sparse rows with others (and is
        # not itself building or on list 1) gets its work list from
        # wise_build_list for its modes instead of a compaction.
        self.mixed_list = mixed_list and not (fold or overlap or head_union or lse_discover)
        # A list-derived pass needs the workspace's queue counters at 0.
        W.wise_workspace_reset(self.shape, self.ws)

        def calls(modes_t, t, compact=True, early=False, build=False, on_list=False, dense=False,
                  list_ready=False, alt=False, list_modes=False):
            d = self.depth[t]
            m = modes_t.data_ptr()
            c = []
            if list_modes:
                f = W.FLAG_SPARSE_LIST | W.FLAG_LIST_MODES
                c.append(("build_list", lib.wise_build_list, (S, m, sl, sup, ws, nws, st)))
                c.append(("partial", lib.wise_decode_partial_ex,
                          (S, d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                           pt, sl, m, ws, nws, f, st)))
                c.append(("finish", lib.wise_decode_finish_ex,
                          (S, m, sl, ws, nws, f, sup, self.out[t].data_ptr(),
                           self.lse[t].data_ptr(), st)))
                return c
            # alt: consecutive depths take the workspace's two slot sets in
            # turn, so a depth on the dense list, or on a list built before
            # the previous finish, starts while that finish still runs
            # (WISE_FLAG_EARLY_START); the first depth of a step only when the
            # step's depth count is even (the previous step's last depth then
            # used the other set).
            sset = W.FLAG_SLOT_SET_1 if (alt and t % 2) else 0
            may_early = alt and (t > 0 or w.num_depths % 2 == 0)
            if dense:
                # Every kernel ahead of it in the step is a pass of the library.
                pf = (W.FLAG_DENSE_LIST | W.FLAG_INPUTS_READY | sset |
                      (W.FLAG_EARLY_START if may_early else 0))
                ff = W.FLAG_DENSE_LIST | (W.FLAG_BUILD_SPARSE_LIST if build else 0) | sset
                c.append(("partial", lib.wise_decode_partial_ex,
                          (S, d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                           pt, sl, m, ws, nws, pf, st)))
                c.append(("finish", lib.wise_decode_finish_ex,
                          (S, m, sl, ws, nws, ff, sup, self.out[t].data_ptr(),
                           self.lse[t].data_ptr(), st)))
                return c
            if on_list:
                f = W.FLAG_SPARSE_LIST | sset
                # A call after the first on the list reads a list built two or
                # more kernels back, and inputs no kernel of the step writes.
                pf = f | ((W.FLAG_INPUTS_READY | (W.FLAG_EARLY_START if may_early else 0))
                          if list_ready else 0)
                c.append(("partial", lib.wise_decode_partial_ex,
                          (S, d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                           pt, sl, m, ws, nws, pf, st)))
                c.append(("finish", lib.wise_decode_finish_ex,
                          (S, m, sl, ws, nws, f, sup, self.out[t].data_ptr(),
                           self.lse[t].data_ptr(), st)))
                return c
            if compact:
                c.append(("compact", lib.wise_compact_tiles, (S, m, sl, sup, ws, nws, st)))
            if build:
                c.append(("partial", lib.wise_decode_partial,
                          (S, d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                           pt, sl, m, ws, nws, st)))
                c.append(("finish", lib.wise_decode_finish_ex,
                          (S, m, sl, ws, nws, W.FLAG_BUILD_SPARSE_LIST, sup,
                           self.out[t].data_ptr(), self.lse[t].data_ptr(), st)))
                return c
            if self.overlap:
                flags = (W.FLAG_SLOT_SET_1 if t % 2 else 0)
                c.append(("partial", lib.wise_decode_partial_ex,
                          (S, d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                           pt, sl, m, ws, nws, flags | (W.FLAG_EARLY_START if early else 0), st)))
                c.append(("finish", lib.wise_decode_finish_ex,
                          (S, m, sl, ws, nws, flags, sup, self.out[t].data_ptr(),
                           self.lse[t].data_ptr(), st)))
                return c
            if self.folded:
                c.append(("partial", lib.wise_decode_partial_finish,
                          (S, d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                           pt, sl, m, ws, nws, sup, self.out[t].data_ptr(),
                           self.lse[t].data_ptr(), st)))
                return c
            c.append(("partial", lib.wise_decode_partial,
                      (S, d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                       pt, sl, m, ws, nws, st)))
            c.append(("finish", lib.wise_decode_finish,
                      (S, m, sl, ws, nws, sup, self.out[t].data_ptr(), self.lse[t].data_ptr(), st)))
            return c

        mode_name = {W.MODE_DENSE: "dense", W.MODE_DISCOVER: "discover",
                     W.MODE_DISCOVER_UNION: "discover_union", W.MODE_SPARSE: "sparse"}
        def depth_name(m):
            u = set(int(x) for x in m)
            return mode_name[u.pop()] if len(u) == 1 else "mixed"

        def all_sparse(m):
            return all(int(x) == W.MODE_SPARSE for x in m)

        def same_work_list(a, b):
            # A compaction depends on each row's length (the same at every
            # depth of a step), whether the row is sparse (then its mask) and
            # whether it records tile statistics (discover or union-discover).
            # Depths whose rows agree on both, with no sparse row, or whose
            # rows are all sparse on a mask no depth between them rewrote,
            # share one work list.
            kind = lambda x: {W.MODE_DENSE: 0, W.MODE_DISCOVER: 1, W.MODE_DISCOVER_UNION: 1,
                              W.MODE_SPARSE: 2}[int(x)]
            ka, kb = [kind(x) for x in a], [kind(x) for x in b]
            return ka == kb and (all(k != 2 for k in ka) or all(k == 2 for k in ka))

        def lse_discover_calls(modes_t, t):
            # Discovery the FlashAttention way: a dense call, the block masses
            # rebuilt from its LSE by a second read of K, then the finish's
            # selection (it merges the dense call's splits again).
            d = self.depth[t]
            c = calls(self.dense_modes, t)
            c.append(("mass", lib.wise_block_mass,
                      (S, d["q"].data_ptr(), d["k_cache"].data_ptr(), pt, sl, modes_t.data_ptr(),
                       self.lse[t].data_ptr(), ws, nws, st)))
            c.append(("select", lib.wise_decode_finish,
                      (S, modes_t.data_ptr(), sl, ws, nws, sup, self.out[t].data_ptr(),
                       self.lse[t].data_ptr(), st)))
            return c

        def all_discover(m):
            return all(int(x) in (W.MODE_DISCOVER, W.MODE_DISCOVER_UNION) for x in m)

        def compaction_free():
            # Every depth of the step on the dense list or on list 1.
            listed = False
            for t in range(w.num_depths):
                dm = w.depth_modes
                if lse_discover and all_discover(dm[t]):
                    return False
                on_list = self.sparse_list and listed and all_sparse(dm[t])
                build = (self.sparse_list and not all_sparse(dm[t]) and t + 1 < w.num_depths and
                         all_sparse(dm[t + 1]))
                dense = self.dense_list and not any(int(x) == W.MODE_SPARSE for x in dm[t])
                listed = build or on_list
                if not (on_list or dense):
                    return False
            return True

        self.early_lists = early_lists and self.dense_list and compaction_free()
        self.early_dense = early_lists and self.dense_list
        self.wise_step = []
        listed = False  # list 1 holds the work list of an all-sparse depth on the current mask
        list0 = False   # the compacted list holds the previous depth's work list
        prev_on_list = False  # the previous depth ran on list 1
        for t in range(w.num_depths):
            dm = w.depth_modes
            reuse = list0 and same_work_list(dm[t], dm[t - 1])
            list0 = False
            if lse_discover and all_discover(dm[t]):
                self.wise_step.append((t, depth_name(dm[t]), lse_discover_calls(self.modes[t], t)))
                continue
            on_list = self.sparse_list and listed and all_sparse(dm[t])
            build = (self.sparse_list and not all_sparse(dm[t]) and t + 1 < w.num_depths and
                     all_sparse(dm[t + 1]))
            dense = self.dense_list and not any(int(x) == W.MODE_SPARSE for x in dm[t])
            list_ready = on_list and prev_on_list
            prev_on_list = on_list
            listed = build or on_list
            if on_list or build or dense:
                self.wise_step.append((t, depth_name(dm[t]),
                                       calls(self.modes[t], t, compact=not reuse and not dense,
                                             build=build, on_list=on_list, dense=dense,
                                             list_ready=list_ready, alt=self.early_lists)))
                list0 = build and not dense
                continue
            if self.mixed_list and any(int(x) == W.MODE_SPARSE for x in dm[t]):
                self.wise_step.append((t, depth_name(dm[t]),
                                       calls(self.modes[t], t, list_modes=True)))
                listed = False  # list 1 now holds this depth's list, not an all-sparse one
                continue
            list0 = True
            c = calls(self.modes[t], t, compact=not reuse, early=reuse)
            if head_union and all_sparse(w.depth_modes[t]) and not reuse:
                # The page-granular variant: sparse depths attend the head
                # union of the row's mask.
                c.insert(0, ("head_union", lib.wise_support_head_union, (S, sup, st)))
            self.wise_step.append((t, depth_name(w.depth_modes[t]), c))
        # The dense baseline gets the same call sequence: one compaction for
        # its four depths (they share the work list) and the same overlap.
        if self.dense_list:
            self.dense_step = [(t, "dense", calls(self.dense_modes, t, dense=True,
                                                  alt=self.early_dense))
                               for t in range(w.num_depths)]
        else:
            self.dense_step = [(t, "dense", calls(self.dense_modes, t, compact=(t == 0),
                                                  early=(t > 0)))
                               for t in range(w.num_depths)]
        # Sparse rows of a depth that no earlier depth discovers (a mixed
        # batch) use the support of a prior discovery of the same inputs.
        if any(int(x) == W.MODE_SPARSE for x in w.depth_modes[0]):
            disc = torch.full((w.num_rows,), W.MODE_DISCOVER, dtype=torch.int8, device=dev)
            for kind, fn, args in calls(disc, 0):
                fn(*args)
            torch.cuda.synchronize()

    def graph(self, step):
        """The step captured once as a CUDA graph (its launches bound to the
        capture stream)."""
        torch = self.torch
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        rebound = []
        for t, mode, calls in step:
            rb = []
            for kind, fn, args in calls:
                rb.append((kind, fn, tuple(side.cuda_stream if i == len(args) - 1 else a
                                           for i, a in enumerate(args))))
            rebound.append((t, mode, rb))
        with torch.cuda.stream(side):
            self.run(rebound)  # one eager pass on the side stream before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            self.run(rebound)
        torch.cuda.synchronize()
        return g

    def run(self, step, events=None):
        for t, mode, calls in step:
            for kind, fn, args in calls:
                if events is not None:
                    e0 = self.torch.cuda.Event(enable_timing=True)
                    e1 = self.torch.cuda.Event(enable_timing=True)
                    e0.record(self.stream)
                rc = fn(*args)
                if rc != 0:
                    raise RuntimeError(f"{kind} failed: {self.lib.wise_last_error().decode()}")
                if events is not None:
                    e1.record(self.stream)
                    events.append((t, mode, kind, e0, e1))

    def launches_per_step(self, step) -> int:
        return sum(len(calls) for _, _, calls in step)

    def kv_bytes(self, modes) -> int:
        """Algorithmic K+V bytes one partial launch must read for these row
        modes: every token of dense and discover rows, the selected tiles'
        tokens of sparse rows (from the current mask)."""
        np, w, W = self.np, self.w, self.W
        per_head_token = w.head_dim * (2 if w.dtype == "bf16" else 4) * 2
        sup = self.support.cpu().numpy().view(np.uint32)
        total = 0
        for r in range(w.num_rows):
            L = int(w.seq_lens[r])
            if int(modes[r]) != W.MODE_SPARSE:
                total += L * w.num_kv_heads * per_head_token
                continue
            nb = -(-L // 32)
            bits = np.unpackbits(sup[r].view(np.uint8).reshape(w.num_kv_heads, -1), axis=1,
                                 bitorder="little")[:, :nb]
            valid = np.minimum(32, L - 32 * np.arange(nb))
            total += int((bits * valid[None, :]).sum()) * per_head_token
        return total

    def support_density(self, modes) -> float:
        """Block density of the mask the sparse rows attend: set bits over
        the causal blocks, summed over the sparse rows' (row, KV head) pairs
        (the reused-union density of [WISE PR, "Response to review", item 4])."""
        np, w, W = self.np, self.w, self.W
        sup = self.support.cpu().numpy().view(np.uint32)
        kept = causal = 0
        for r in range(w.num_rows):
            if int(modes[r]) != W.MODE_SPARSE:
                continue
            nb = -(-int(w.seq_lens[r]) // 32)
            bits = np.unpackbits(sup[r].view(np.uint8).reshape(w.num_kv_heads, -1), axis=1,
                                 bitorder="little")[:, :nb]
            kept += int(bits.sum())
            causal += nb * w.num_kv_heads
        return kept / causal if causal else 0.0

    def small_bytes(self) -> int:
        w = self.w
        es = 2 if w.dtype == "bf16" else 4
        return w.num_rows * w.num_q_heads * w.head_dim * es  # q read


# Eager launches go out one ctypes call at a time, slower than the GPU runs
# them, so without a lead every event bracket would also hold the host's
# submission of the launch.  Each eager step therefore starts behind a spin
# kernel long enough for the host to queue the whole step first; the events
# then see only the GPU, and the step's time is taken from the end of the spin.
LEAD_CYCLES = 4_000_000  # about 2 ms at the GB300's 2.07 GHz maximum SM clock


def timed_region(pipe, step, K, dist, with_events=True):
    import torch
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    events = [] if with_events else None
    marks = []
    spin = getattr(torch.cuda, "_sleep", None)  # torch's spin kernel (present in 2.9 and 2.11)
    for _ in range(K):
        if spin is not None:
            spin(LEAD_CYCLES)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(pipe.stream)
        pipe.run(step, events)
        end.record(pipe.stream)
        marks.append((start, end))
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    return sum(s.elapsed_time(e) for s, e in marks), events


def graph_region(pipe, graph, K, dist):
    import torch
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(K):
        graph.replay()
    e.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    return s.elapsed_time(e)


def e2e_region(pipe, K, graph=None):
    """The same step through the C ABI from pinned host memory: every step
    copies its inputs (q of each depth, page table, lengths, modes: one
    packed buffer) host -> device and reads its results (out and lse of each
    depth, the mask: one packed buffer) back, inside the timed region.  The
    step's ABI calls run from `graph` (their capture, as an engine replays
    its decode step) or, without one, one by one."""
    import torch
    h_out = torch.empty(pipe.out_dev.shape, dtype=pipe.out_dev.dtype).pin_memory()
    h2d = pipe.in_host.numel() * pipe.in_host.element_size()
    d2h = h_out.numel() * h_out.element_size()

    def one():
        pipe.in_dev.copy_(pipe.in_host, non_blocking=True)
        if graph is not None:
            graph.replay()
        else:
            pipe.run(pipe.wise_step)
        h_out.copy_(pipe.out_dev, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(pipe.stream)
    for _ in range(K):
        one()
    e.record(pipe.stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e), h2d, d2h


def partial_in_step_ms(pipe, base_ms, depth, K, dist):
    """What one partial launch of `depth` costs inside the captured step: the
    step is captured again with one more launch of that depth's partial just
    before it, and the extra time per replay over the plain step is the
    answer.  The extra launch reads a private copy of the depth's K/V pool
    (same values, same items, its own addresses; nothing else reads it), so
    neither it nor the real launch finds the other's tiles in L2, and the
    real launch then rewrites the same splits.  Unlike the eager per-launch
    events, this keeps the programmatic-dependent-launch overlap with the
    neighbouring kernels that the step itself has."""
    torch = pipe.torch
    cold = [pipe.depth[depth]["k_cache"].clone(), pipe.depth[depth]["v_cache"].clone()]
    step = []
    for t, mode, calls in pipe.wise_step:
        if t == depth:
            doubled = []
            for c in calls:
                if c[0] == "partial":
                    args = list(c[2])
                    args[2], args[3] = cold[0].data_ptr(), cold[1].data_ptr()
                    doubled.append(("partial", c[1], tuple(args)))
                doubled.append(c)
            calls = doubled
        step.append((t, mode, calls))
    g = pipe.graph(step)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    extra = (graph_region(pipe, g, K, dist) - base_ms) / K
    del g, cold
    return extra


def e2e_pipelined(pipes, graphs, K):
    """The end-to-end region as an engine runs it: two buffer sets over the
    same resident K/V, so step i+1's host->device input copy and step i-1's
    device->host result copy (each on its own copy stream) run while step i
    computes.  Every step still moves its own inputs from pinned host memory
    and its own results back; the region runs from before the first input
    copy to after the last result copy."""
    import torch
    compute = pipes[0].stream
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    h_out = [torch.empty(p.out_dev.shape, dtype=p.out_dev.dtype).pin_memory() for p in pipes]
    h2d = pipes[0].in_host.numel() * pipes[0].in_host.element_size()
    d2h = h_out[0].numel() * h_out[0].element_size()
    ev = lambda: torch.cuda.Event()

    def run(n, timed):
        computed = [None, None]   # compute of the set's last step done
        read_back = [None, None]  # result copy of the set's last step done
        start = torch.cuda.Event(enable_timing=True) if timed else None
        end = torch.cuda.Event(enable_timing=True) if timed else None
        if timed:
            start.record(compute)
        up.wait_stream(compute)
        down.wait_stream(compute)
        for i in range(n):
            j = i % 2
            p = pipes[j]
            with torch.cuda.stream(up):
                if computed[j] is not None:
                    up.wait_event(computed[j])     # the set's inputs are consumed
                p.in_dev.copy_(p.in_host, non_blocking=True)
                landed = ev()
                landed.record(up)
            compute.wait_event(landed)
            if read_back[j] is not None:
                compute.wait_event(read_back[j])   # the set's results are read
            graphs[j].replay()
            computed[j] = ev()
            computed[j].record(compute)
            with torch.cuda.stream(down):
                down.wait_event(computed[j])
                h_out[j].copy_(p.out_dev, non_blocking=True)
                read_back[j] = ev()
                read_back[j].record(down)
        compute.wait_stream(up)
        compute.wait_stream(down)
        if timed:
            end.record(compute)
        torch.cuda.synchronize()
        return start.elapsed_time(end) if timed else None

    run(4, False)
    return run(K, True), h2d, d2h


# ----------------------------------------------------------------------------- ranks
def rank_env():
    """(world size, rank, local rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(rank: int):
    """Seed of a rank's own batch: every rank decodes different rows of the
    same shape (weak scaling; rows are independent, so nothing is exchanged
    on the data path).  Rank 0 keeps the workload's own seed."""
    return None if rank == 0 else 100000 + rank


def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank timings (the job takes as long as its
    slowest rank)."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_rate(world: int, units_per_step: int, steps: int, ms: float) -> float:
    """Units all ranks processed per second, over the slowest rank's time."""
    return world * units_per_step * steps / (ms * 1e-3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def summarize_events(evts):
    """Mean duration (ms) of each (depth, mode, kernel) over the timed steps."""
    per = {}
    for (tt, mode, kind, e0, e1) in evts:
        per.setdefault((tt, mode, kind), []).append(e0.elapsed_time(e1))
    return {k: statistics.mean(v) for k, v in per.items()}


def mode_table(per, per_dense, kv, R, num_depths, peak):
    """Per depth of the WISE step: call time (every launch of the depth) and
    its partial launch, each as GB/s over the bytes the depth's partial pass
    must read and as a fraction of the measured and of the nominal 8 TB/s HBM
    bandwidth; then the dense baseline's mean call."""
    def rates(nbytes, ms):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return round(gbs, 1), round(gbs / peak, 3), round(gbs / 8000.0, 3)

    modes = {}
    for (tt, m, k) in sorted(per):
        if k != "partial":
            continue
        call_ms = sum(v for (t2, m2, k2), v in per.items() if t2 == tt)
        p_gbs, p_frac, p_nom = rates(kv[(tt, m)], per[(tt, m, k)])
        c_gbs, c_frac, c_nom = rates(kv[(tt, m)], call_ms)
        modes[f"depth{tt}_{m}"] = {
            "call_us": round(call_ms * 1e3, 2), "partial_us": round(per[(tt, m, k)] * 1e3, 2),
            "kernels_us": {k2: round(v * 1e3, 2) for (t2, m2, k2), v in per.items() if t2 == tt},
            "rows_per_s": round(R / (call_ms * 1e-3), 1),
            "partial_gbs": p_gbs, "partial_frac_of_measured_hbm": p_frac,
            "partial_frac_of_nominal_8000_gbs": p_nom,
            "call_gbs": c_gbs, "call_frac_of_measured_hbm": c_frac,
            "call_frac_of_nominal_8000_gbs": c_nom,
            "algorithmic_bytes": kv[(tt, m)]}
    dense_call = sum(per_dense.values()) / num_depths
    dense_part = statistics.mean(v for (tt, m, k), v in per_dense.items() if k == "partial")
    p_gbs, p_frac, p_nom = rates(kv[(0, "dense")], dense_part)
    c_gbs, c_frac, c_nom = rates(kv[(0, "dense")], dense_call)
    modes["dense"] = {"call_us": round(dense_call * 1e3, 2), "partial_us": round(dense_part * 1e3, 2),
                      "rows_per_s": round(R / (dense_call * 1e-3), 1),
                      "partial_gbs": p_gbs, "partial_frac_of_measured_hbm": p_frac,
                      "partial_frac_of_nominal_8000_gbs": p_nom,
                      "call_gbs": c_gbs, "call_frac_of_measured_hbm": c_frac,
                      "call_frac_of_nominal_8000_gbs": c_nom,
                      "algorithmic_bytes": kv[(0, "dense")]}
    return modes


def algorithmic_bytes(pipe, w):
    import numpy as np
    kv = {}
    for t, mode, _ in pipe.wise_step:
        kv[(t, mode)] = pipe.kv_bytes(w.depth_modes[t]) + pipe.small_bytes()
    for t, mode, _ in pipe.dense_step:
        kv[(t, mode)] = pipe.kv_bytes(np.zeros(w.num_rows, np.int8)) + pipe.small_bytes()
    return kv


# Workloads the default run measures after its headline, each on its own
# K/V drawn on the device: the metric is quoted per mode at 1K, 4K and 8K
# context, and the 32K grouped-query workload exercises the tensor-core path.
SWEEP = ("ouro1.4b_4k", "mixed_8k", "gqa_32k")


def sweep_workload(name, args, steps, peak):
    """One workload of the default run's sweep: the WISE step and the dense
    step, each captured as a CUDA graph and replayed `steps` times (CUDA
    events around the replays), then launched eagerly with events around
    every launch for the per-mode table."""
    import numpy as np
    import torch
    from block_sparse_paged_split_gb300.workload import make_workload
    t0 = time.time()
    w = make_workload(name, **eta_kw(args.eta))
    pipe = Pipeline(w, tiles_per_item=args.tiles_per_item, sparse_list=not args.no_sparse_list,
                    device_inputs=True, dense_list=not args.no_dense_list,
                    early_lists=args.early, mixed_list=not args.no_mixed_list)
    for _ in range(3):
        pipe.run(pipe.wise_step)
        pipe.run(pipe.dense_step)
    torch.cuda.synchronize()
    kv = algorithmic_bytes(pipe, w)
    sparse_t = [t for t in range(w.num_depths) if any(int(x) == 3 for x in w.depth_modes[t])]
    density = pipe.support_density(w.depth_modes[sparse_t[0]]) if sparse_t else None
    g, gd = pipe.graph(pipe.wise_step), pipe.graph(pipe.dense_step)
    for _ in range(3):
        g.replay()
        gd.replay()
    ms = graph_region(pipe, g, steps, None)
    ms_dense = graph_region(pipe, gd, steps, None)
    _, ev = timed_region(pipe, pipe.wise_step, steps, None)
    _, ev_dense = timed_region(pipe, pipe.dense_step, steps, None)
    R = w.num_rows
    rows_per_step = R * w.num_depths
    out = {"workload": f"{R} rows x {int(w.seq_lens.min())}-{int(w.seq_lens.max())} tokens, "
                       f"{w.num_q_heads} q / {w.num_kv_heads} kv heads, D={w.head_dim}, "
                       f"{w.num_depths} depth(s): " +
                       ", ".join(pipe_depth_names(pipe)),
           "step_ms": round(ms / steps, 4),
           "rows_per_s": round(rows_per_step * steps / (ms * 1e-3), 1),
           "dense_step_ms": round(ms_dense / steps, 4),
           "speedup_vs_dense": round(ms_dense / ms, 3),
           "support_density_blocks": round(density, 4) if density is not None else None,
           "modes": mode_table(summarize_events(ev), summarize_events(ev_dense), kv, R,
                               w.num_depths, peak),
           "launches_per_step": pipe.launches_per_step(pipe.wise_step),
           "dense_launches_per_step": pipe.launches_per_step(pipe.dense_step),
           "steps": steps, "inputs": "K/V drawn on the device (same recipe, seeded)",
           "wall_s": None}
    del g, gd, pipe
    torch.cuda.empty_cache()
    out["wall_s"] = round(time.time() - t0, 1)
    return out


ETA_SWEEP = (0.8, 0.9, 0.95, 0.99)


def eta_point(name, eta, args, steps):
    """One point of the eta sweep: the WISE step's and the dense step's
    graph-replay times and the reused-union density the sparse depths
    attend, for one selection threshold."""
    import torch
    from block_sparse_paged_split_gb300.workload import make_workload
    w = make_workload(name, eta=eta)
    pipe = Pipeline(w, tiles_per_item=args.tiles_per_item, sparse_list=not args.no_sparse_list,
                    device_inputs=True, dense_list=not args.no_dense_list,
                    early_lists=args.early, mixed_list=not args.no_mixed_list)
    for _ in range(3):
        pipe.run(pipe.wise_step)
    torch.cuda.synchronize()
    sparse_t = [t for t in range(w.num_depths) if any(int(x) == 3 for x in w.depth_modes[t])]
    density = pipe.support_density(w.depth_modes[sparse_t[0]]) if sparse_t else None
    g, gd = pipe.graph(pipe.wise_step), pipe.graph(pipe.dense_step)
    for _ in range(3):
        g.replay()
        gd.replay()
    ms = graph_region(pipe, g, steps, None)
    ms_dense = graph_region(pipe, gd, steps, None)
    out = {"eta": eta, "support_density_blocks": round(density, 4) if density is not None else None,
           "step_ms": round(ms / steps, 4), "dense_step_ms": round(ms_dense / steps, 4),
           "speedup_vs_dense": round(ms_dense / ms, 3),
           "launches": steps * (pipe.launches_per_step(pipe.wise_step) +
                                pipe.launches_per_step(pipe.dense_step))}
    del g, gd, pipe
    torch.cuda.empty_cache()
    return out


def pipe_depth_names(pipe):
    return [f"{mode}" + ("" if not any(c[0] == "compact" for c in calls) else "+compact")
            for _, mode, calls in pipe.wise_step]


def main_ours(args):
    import numpy as np
    import torch
    import torch.distributed as tdist

    world, rank, local = rank_env()
    dist = None
    if world > 1:
        tdist.init_process_group("nccl")
        dist = tdist
    torch.cuda.set_device(local)

    from block_sparse_paged_split_gb300.build import build_library
    from block_sparse_paged_split_gb300.workload import make_workload
    build_library()
    # Weak scaling: every rank decodes its own batch (rows are independent).
    w = make_workload(args.workload, num_rows=args.rows, seed=rank_seed(rank), **eta_kw(args.eta))
    pipe = Pipeline(w, tiles_per_item=args.tiles_per_item, fold=args.fold, head_union=args.head_union,
                    lse_discover=args.lse_discover, overlap=args.overlap,
                    sparse_list=not args.no_sparse_list, dense_list=not args.no_dense_list,
                    early_lists=args.early, mixed_list=not args.no_mixed_list)

    for _ in range(max(args.warmup, 3)):
        pipe.run(pipe.wise_step)
        pipe.run(pipe.dense_step)
    torch.cuda.synchronize()

    # Algorithmic bytes of each depth's partial launch (the mask is the same
    # every step: the inputs do not change).
    kv = algorithmic_bytes(pipe, w)
    sparse_depths = [t for t, mode, _ in pipe.wise_step if mode == "sparse"]
    density = (pipe.kv_bytes(w.depth_modes[sparse_depths[0]]) /
               pipe.kv_bytes(np.zeros(w.num_rows, np.int8))) if sparse_depths else None
    block_density = pipe.support_density(w.depth_modes[sparse_depths[0]]) if sparse_depths else None

    # The step and the dense baseline step, each captured once as a CUDA graph.
    graph = pipe.graph(pipe.wise_step)
    graph_dense = pipe.graph(pipe.dense_step)
    for _ in range(3):
        graph.replay()
        graph_dense.replay()
    torch.cuda.synchronize()

    clock = ClockSampler(local)
    wall0 = time.time()
    # Headline: K steps replayed from the graph, CUDA events around them.
    ms = graph_region(pipe, graph, args.steps, dist)
    ms_dense_graph = graph_region(pipe, graph_dense, args.steps, dist)
    # Per-launch view: the same K steps launched eagerly with CUDA events
    # around every launch (per-mode times and the roofline of the partial pass).
    ms_eager, events = timed_region(pipe, pipe.wise_step, args.steps, dist)
    ms_dense, events_dense = timed_region(pipe, pipe.dense_step, args.steps, dist)
    # One partial of the first discover depth and of the first sparse depth,
    # timed inside the captured step (marginal cost).
    in_step = {}
    for t, mode, calls in pipe.wise_step:
        if mode in ("discover", "sparse") and mode not in {m for _, m in in_step} and \
                any(c[0] == "partial" for c in calls):
            in_step[(t, mode)] = partial_in_step_ms(pipe, ms, t, args.steps, dist)
    clocks = clock.stop()
    wall = time.time() - wall0

    # Max over ranks.
    ms, ms_dense_graph, ms_eager, ms_dense = max_over_ranks(
        [ms, ms_dense_graph, ms_eager, ms_dense], dist, "cuda")

    per = summarize_events(events)
    per_dense = summarize_events(events_dense)
    peak, peak_kind = peaks()

    # Dominant kernel: the split partial pass (all depths of the WISE step).
    part_bytes = sum(kv[(tt, m)] for (tt, m, k) in per if k == "partial")
    part_ms = sum(v for (tt, m, k), v in per.items() if k == "partial")
    achieved = part_bytes / (part_ms * 1e-3) / 1e9
    # Kernels launched in the timed regions: the graph replays and the eager
    # passes, each over K WISE steps and K dense steps, the three end-to-end
    # regions' K WISE steps each, and the in-step partial timings' K steps
    # with one extra partial each.
    launches = (2 * (pipe.launches_per_step(pipe.wise_step) +
                     pipe.launches_per_step(pipe.dense_step)) +
                3 * pipe.launches_per_step(pipe.wise_step) +
                len(in_step) * (pipe.launches_per_step(pipe.wise_step) + 1)) * args.steps

    R = w.num_rows
    modes = mode_table(per, per_dense, kv, R, w.num_depths, peak)
    for (tt, m) in in_step:
        t_in = max_over_ranks([in_step[(tt, m)]], dist, "cuda")[0]
        modes[f"depth{tt}_{m}"].update({
            "partial_in_step_us": round(t_in * 1e3, 2),
            "partial_in_step_frac_of_measured_hbm": round(kv[(tt, m)] / (t_in * 1e-3) / 1e9 / peak, 3),
            "in_step_note": "marginal time of one more such partial launch (over a private "
                            "copy of the K/V pool, so no L2 reuse) inside the captured "
                            "step, whose launches overlap the previous kernel; partial_us "
                            "above is the eager launch bracketed by events"})
    modes["dense"].update({"step_ms_eager": round(ms_dense / args.steps, 4),
                           "step_ms_graph": round(ms_dense_graph / args.steps, 4)})

    # End to end: the pipelined region (two buffer sets, copies overlapping
    # the compute), then the same steps with each step's copies in line.
    pipe_b = Pipeline(w, tiles_per_item=args.tiles_per_item, fold=args.fold,
                      head_union=args.head_union, lse_discover=args.lse_discover,
                      overlap=args.overlap, share=pipe, sparse_list=not args.no_sparse_list,
                      dense_list=not args.no_dense_list,
                    early_lists=args.early, mixed_list=not args.no_mixed_list)
    graph_b = pipe_b.graph(pipe_b.wise_step)
    e2e_ms, h2d, d2h = e2e_pipelined([pipe, pipe_b], [graph, graph_b], args.steps)
    e2e_serial_ms, _, _ = e2e_region(pipe, args.steps, graph)
    e2e_eager_ms, _, _ = e2e_region(pipe, args.steps)
    rows_per_step = R * w.num_depths
    e2e_ms, e2e_serial_ms, e2e_eager_ms = max_over_ranks([e2e_ms, e2e_serial_ms, e2e_eager_ms],
                                                         dist, "cuda")
    value = whole_job_rate(world, rows_per_step, args.steps, ms)
    e2e_value = whole_job_rate(world, rows_per_step, args.steps, e2e_ms)

    # The default run also measures the metric's other contexts (4K, the
    # ragged 8K mixed batch) and the 32K grouped-query workload, each with
    # fewer steps, on one GPU.
    sweep = None
    variant = args.fold or args.head_union or args.lse_discover or args.overlap
    if (not args.no_sweep and world == 1 and args.workload == WORKLOAD and args.rows is None
            and not variant):
        del pipe_b, graph_b
        torch.cuda.empty_cache()
        sweep_steps = max(5, min(args.steps, 50))
        sclock = ClockSampler(local)
        sweep = {name: sweep_workload(name, args, sweep_steps, peak) for name in SWEEP}
        # The GQA workload over the selection threshold: the step against
        # the reused-union density it leaves the sparse depths.
        if "gqa_32k" in sweep and args.eta is None:
            pts = [eta_point("gqa_32k", e, args, sweep_steps) for e in ETA_SWEEP]
            for pt in pts:
                launches += pt.pop("launches")
            sweep["gqa_32k"]["eta_sweep"] = pts
        sweep_clocks = sclock.stop()
        for name, res in sweep.items():
            launches += 2 * sweep_steps * res.pop("launches_per_step")
            launches += 2 * sweep_steps * res.pop("dense_launches_per_step")

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; Ouro-1.4B decode shapes, planted support)",
        "config": {"workload": f"{args.workload}: {R} rows x {int(w.seq_lens.max())} tokens, "
                               f"{w.num_q_heads} q / {w.num_kv_heads} kv heads, D={w.head_dim}, "
                               f"page {w.page_size}, B=32, eta={w.eta}, 4 depths"
                               + (", sparse depths on the head union of the mask" if args.head_union else "")
                               + (", discovery from the LSE (second read of K)" if args.lse_discover else "")
                               + (", finish folded into the partial pass" if pipe.folded else "")
                               + (", consecutive depths overlap (two slot sets, early start)" if pipe.overlap else "")
                               + (", sparse depths on the work list the union depth's finish "
                                  "builds (no compaction launch)" if pipe.sparse_list else "")
                               + (", dense and discover depths on work lists derived from the "
                                  "row lengths (no compaction launch)" if pipe.dense_list else "")
                               + (", consecutive depths on alternate slot sets, a depth on the "
                                  "dense list or a ready list starting beside the previous finish"
                                  if pipe.early_lists else "")
                               + (", mixed depths on a work list built from their modes and masks "
                                  "(no compaction launch)" if pipe.mixed_list else ""),
                   "rows_per_step": rows_per_step, "parallelism": f"replicas x{world} (rows independent)",
                   "l2": f"inputs larger than L2: "
                         f"{w.num_depths * pipe.kv_bytes(np.zeros(w.num_rows, np.int8)) / 1e9:.2f} GB "
                         f"of K/V per step (129 MB L2)",
                   "timing": "value: CUDA-graph replay of the step, CUDA events around the K "
                             "replays; modes and roofline: eager launches with CUDA events "
                             "around every launch on the launching stream, each step queued "
                             "behind a spin kernel so that no event bracket holds host "
                             "submission time",
                   "union_density": round(density, 4) if density else None,
                   "support_density_blocks": round(block_density, 4) if block_density else None},
        "modes": modes,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "frac_of_nominal_8000_gbs": round(achieved / 8000.0, 4),
                     "traffic": (round(traffic) if (traffic := recorded_traffic(R, args.workload)) else None),
                     "algorithmic_bytes_per_launch": round(
                         part_bytes / sum(1 for k in per if k[2] == "partial")),
                     "kernel": ("partial_kernel (split-KV partial pass with the finish folded in, all four depths)"
                                if pipe.folded else "partial_kernel (split-KV partial pass, all four depths)"),
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)" if peak_kind == "measured" else peak_kind},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "per step: one packed host->device copy of the inputs, the step's C-ABI "
                        "calls replayed from their CUDA graph, one packed device->host copy of "
                        "the results; two buffer sets, so step i+1's input copy and step i-1's "
                        "result copy (own copy streams) overlap step i's compute",
                "serial_value": round(whole_job_rate(world, rows_per_step, args.steps,
                                                     e2e_serial_ms), 1),
                "eager_calls_value": round(whole_job_rate(world, rows_per_step, args.steps,
                                                          e2e_eager_ms), 1),
                "variants": "serial_value: each step's copies in line with it, one buffer set; "
                            "eager_calls_value: the same with the C-ABI calls made one by one"},
        "eager": {"ms_per_step": round(ms_eager / args.steps, 4),
                  "rows_per_s": round(whole_job_rate(world, rows_per_step, args.steps, ms_eager), 1),
                  "note": "every launch bracketed by CUDA events"},
        "speedup_vs_dense": round(ms_dense_graph / ms, 3),
        "speedup_vs_dense_pages": PAGES_SPEEDUP.get(args.workload),
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed": round(wall, 2),
    }
    if sweep is not None:
        result["modes_by_workload"] = sweep
        result["modes_by_workload_clocks"] = sweep_clocks
        result["config"]["sweep"] = (f"after the headline: {', '.join(SWEEP)}, each with its WISE "
                                     f"and dense steps replayed from CUDA graphs "
                                     f"({sweep_steps} steps) and launched eagerly for the "
                                     f"per-mode table; K/V drawn on the device; gqa_32k also "
                                     f"at eta {', '.join(str(e) for e in ETA_SWEEP)} "
                                     f"(graph replays only)")
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = run_oracle_sample(args.workload, rows=16, eta=args.eta)
    if rank == 0:
        print(json.dumps(result))
    if dist:
        dist.destroy_process_group()


def sparse_scaling_main(args):
    """Sparse-mode time against the selected tiles and against the context.

    Each point is one sparse call over 64 rows (--rows) x 16 heads (MHA, D=128, bf16):
    the work list built from the mask (wise_build_sparse_list), partial pass
    and finish on it, and for contrast the same call on a compaction
    (compaction, partial pass, finish); each launch timed with CUDA events on
    the launching stream (mean of 30 calls, the L2 flushed by a 512 MiB write
    before each).  Sweep 1 holds 8 selected tiles per (row, head) and grows the
    context 1K -> 128K (the K/V pool then holds 69 GB); sweep 2 holds the
    context at 8K and grows the selected tiles 1 -> 256 (every block).  The
    dense call at each context is timed the same way for contrast."""
    import numpy as np
    import torch
    import block_sparse_paged_split_gb300 as W
    from block_sparse_paged_split_gb300 import wise
    from block_sparse_paged_split_gb300.build import build_library
    from block_sparse_paged_split_gb300.workload import sparse_scaling_inputs

    build_library()
    lib = wise.library()
    torch.cuda.set_device(0)
    if args.gqa:
        # Grouped-query heads (the tensor-core consumer): 32 query / 8 KV heads.
        R, H, Hq, D, reps = args.rows or 16, 8, 32, 128, 30
        points = ([(L, 16, True) for L in (4096, 8192, 16384, 32768, 65536, 131072)] +
                  [(32768, k, False) for k in (1, 4, 64, 256, 1024)])
    else:
        R, H, Hq, D, reps = args.rows or 64, 16, 16, 128, 30
        points = ([(L, 8, True) for L in (1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072)] +
                  [(8192, k, False) for k in (1, 2, 4, 16, 32, 64, 128, 256)])
    peak, peak_kind = peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    if args.point:
        L, k = (int(x) for x in args.point.split(":"))
        points = [(L, k, False)]
    rows = []
    for L, k, with_dense in points:
        d = sparse_scaling_inputs(R, H, D, L, k, seed=4242 + L + k,
                                  shared_blocks=args.shared_blocks, num_q_heads=Hq)
        shape = W.make_shape(num_rows=R, num_q_heads=Hq, num_kv_heads=H, head_dim=D, page_size=16,
                             max_pages_per_row=d["page_table"].shape[1], num_pages=d["num_pages"],
                             max_blocks=d["max_blocks"], dtype=W.DTYPE_BF16, eta=0.95)
        ws = W.alloc_workspace(shape)
        out = torch.empty_like(d["q"])
        lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        S = ctypes.byref(shape)
        st = stream.cuda_stream
        args_common = (d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                       d["page_table"].data_ptr(), d["seq_lens"].data_ptr())

        def call(modes_t, sup, on_list):
            m = modes_t.data_ptr()
            t = []
            if on_list:  # every row sparse: list 1 from the mask, both passes on it
                L1 = ctypes.c_uint32(W.FLAG_SPARSE_LIST)
                launches = ((lib.wise_build_sparse_list, (S, args_common[4], sup.data_ptr(),
                                                          ws.data_ptr(), ws.numel(), st)),
                            (lib.wise_decode_partial_ex, (S,) + args_common + (None, ws.data_ptr(),
                                                                               ws.numel(), L1, st)),
                            (lib.wise_decode_finish_ex, (S, None, args_common[4], ws.data_ptr(),
                                                         ws.numel(), L1, None, out.data_ptr(),
                                                         lse.data_ptr(), st)))
            else:
                launches = ((lib.wise_compact_tiles, (S, m, args_common[4], sup.data_ptr(),
                                                      ws.data_ptr(), ws.numel(), st)),
                            (lib.wise_decode_partial, (S,) + args_common + (m, ws.data_ptr(),
                                                                            ws.numel(), st)),
                            (lib.wise_decode_finish, (S, m, args_common[4], ws.data_ptr(),
                                                      ws.numel(), sup.data_ptr(), out.data_ptr(),
                                                      lse.data_ptr(), st)))
            for fn, a in launches:
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                t.append(e)
                rc = fn(*a)
                if rc != 0:
                    raise RuntimeError(lib.wise_last_error().decode())
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            t.append(e)
            return t

        def timed(modes_t, sup, on_list=False):
            calls, comp, parts, fin = [], [], [], []
            for i in range(reps + 3):
                flush.fill_(i & 0xFF)
                t = call(modes_t, sup, on_list)
                torch.cuda.synchronize()
                if i >= 3:
                    calls.append(t[0].elapsed_time(t[3]) * 1e3)
                    comp.append(t[0].elapsed_time(t[1]) * 1e3)
                    parts.append(t[1].elapsed_time(t[2]) * 1e3)
                    fin.append(t[2].elapsed_time(t[3]) * 1e3)
            # Means: event timestamps step in about 2 us on GB300, and the mean of
            # many calls averages that quantisation out where a median keeps it.
            return (statistics.fmean(calls), statistics.fmean(parts), statistics.fmean(comp),
                    statistics.fmean(fin))

        sparse = torch.full((R,), W.MODE_SPARSE, dtype=torch.int8, device="cuda")
        call_us, part_us, build_us, fin_us = timed(sparse, d["support"], on_list=True)
        c_call_us, c_part_us, c_comp_us, c_fin_us = timed(sparse, d["support"])
        tiles = R * H * min(k, d["max_blocks"])
        sel_bytes = tiles * 32 * D * 2 * 2
        row = {"context": L, "selected_tiles_per_head": min(k, d["max_blocks"]),
               "sparse_call_us": round(call_us, 2), "sparse_build_us": round(build_us, 2),
               "sparse_partial_us": round(part_us, 2), "sparse_finish_us": round(fin_us, 2),
               "selected_kv_bytes": sel_bytes,
               "partial_gbs": round(sel_bytes / (part_us * 1e-6) / 1e9, 1),
               "partial_frac": round(sel_bytes / (part_us * 1e-6) / 1e9 / peak, 3),
               "call_frac": round(sel_bytes / (call_us * 1e-6) / 1e9 / peak, 3),
               "compaction_call_us": round(c_call_us, 2), "compaction_us": round(c_comp_us, 2),
               "compaction_partial_us": round(c_part_us, 2),
               "compaction_finish_us": round(c_fin_us, 2)}
        if with_dense:
            dense = torch.zeros((R,), dtype=torch.int8, device="cuda")
            dense_call, dense_part, _, _ = timed(dense, torch.zeros_like(d["support"]))
            dense_bytes = R * H * L * D * 2 * 2
            row.update({"dense_call_us": round(dense_call, 2),
                        "dense_partial_frac": round(dense_bytes / (dense_part * 1e-6) / 1e9 / peak, 3)})
        rows.append(row)
        del d, ws, out, lse
        torch.cuda.empty_cache()
    print(json.dumps({"sparse_scaling": rows, "rows": R, "heads": H, "q_heads": Hq, "head_dim": D,
                      "blocks": "shared by a row's heads" if args.shared_blocks else "per head",
                      "peak_gbs": peak, "peak_kind": peak_kind, "reps": reps,
                      "l2": "flushed by a 512 MiB write before every call"}))


def main_reference(args):
    world, rank = rank_env()[0], rank_env()[1]
    if rank != 0:
        return
    K, Wm = args.steps, args.warmup
    # Each step: the C++ fp32 oracle on a 16-row sample of the workload through
    # the 4 depths on every host thread (tens of milliseconds); the warm-up
    # passes run untimed inside the child before the K timed ones.
    rows = 16
    from block_sparse_paged_split_gb300.workload import make_workload
    w_ref = make_workload(args.workload, **eta_kw(args.eta))  # its shape only (no inputs drawn)
    t0 = time.perf_counter()
    res = run_oracle_sample(args.workload, rows=rows, seconds_1t=0.0, reps=K, warmup=Wm,
                            eta=args.eta)
    value = res["value"]
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
           "n_gpus": world, "steps": K, "warmup": Wm,
           "ms_per_step": round(1e3 * rows * 4 / value, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": f"{args.workload}: {w_ref.num_rows} rows x "
                                  f"{int(w_ref.seq_lens.max())} tokens, {w_ref.num_q_heads} q / "
                                  f"{w_ref.num_kv_heads} kv heads, D={w_ref.head_dim}, page "
                                  f"{w_ref.page_size}, B=32, eta={w_ref.eta}, 4 depths",
                      "sample": f"{rows} of its rows per step through the oracle"},
           "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": res["cores"],
                            "kind": "oracle", "sample": res["sample"],
                            "per_mode_rows_per_s": res["per_mode_rows_per_s"]},
           "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "wall_s": round(time.perf_counter() - t0, 1)}
    print(json.dumps(out))


if __name__ == "__main__":
    a = parse()
    if a.oracle_sample is not None:
        oracle_sample_main(a.oracle_sample)
    elif a.record_traffic is not None:
        record_traffic(a.record_traffic, a.rows or 64, a.workload)
    elif a.sparse_scaling:
        sparse_scaling_main(a)
    elif a.impl == "reference":
        main_reference(a)
    else:
        main_ours(a)
