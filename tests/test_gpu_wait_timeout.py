"""The failure path on the GPU without a fault: the library's mbarrier waits
are bounded by %globaltimer (500 ms), and a wait that runs out sets
WISE_DEVERR_WAIT_TIMEOUT in a status word instead of hanging.  The self-test
entry point waits on a barrier nothing arrives on; the host reads the status
bit, and the next decode call on the same context is correct."""
import time

import numpy as np
import pytest
import torch

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300.workload import custom_workload
from tests.gpu_harness import Batch, compare_outputs, gpu_call, oracle_call, words

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_the_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    W.wise.wise_selftest_wait_timeout(status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) & W.wise.DEVERR_WAIT_TIMEOUT
    assert 0.4 < waited < 30, waited  # the 500 ms limit, not a hang
    lens = np.array([64, 100, 40, 33], np.int32)
    w = custom_workload("timeout", R=4, Hq=4, Hkv=4, D=128, dtype="bf16", depths=1, n_planted=1,
                        seq_lens=lens, pool_factor=2, seed=5, depth_modes=[np.zeros(4, np.int8)])
    b = Batch(w)
    zero = np.zeros((4, 4, words(w)), np.uint32)
    g = gpu_call(b, 0, np.zeros(4, np.int8), zero)
    o = oracle_call(b, 0, np.zeros(4, np.int8), zero)
    assert not compare_outputs(w, g, o)
    assert int(g["ws"]["status"][0]) == 0
