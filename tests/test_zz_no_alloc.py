"""wise_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (for example code running inside someone else's CUDA-graph
capture, or a host framework that forbids allocations outside its own pool).
It uses the library's static 16 MiB device scratch instead of a workspace.

The GPU test calls it through the C ABI twice in a row (the second call finds
the first call's leftovers in the shared scratch), then once more with a
shape whose workspace layout differs, and checks each result against the
ordinary wise_decode with a caller-owned workspace bit for bit (both run the
same kernels on the same inputs), and that the scratch's status word, read
with wise_noalloc_status, is 0.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300 import wise
from block_sparse_paged_split_gb300.build import build_library
from block_sparse_paged_split_gb300.workload import custom_workload
from tests.gpu_harness import dev_support, np_support, shape_for, words


@pytest.fixture(scope="module")
def lib():
    build_library()
    return wise.library()


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    """Host-side: a shape whose workspace exceeds the 16 MiB scratch is refused
    with WISE_ERR_WORKSPACE before anything is enqueued."""
    big = W.make_shape(num_rows=64, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                       max_pages_per_row=2048, num_pages=65536, max_blocks=1024)
    assert W.wise_workspace_bytes(big) > (16 << 20)
    P = ctypes.c_void_p
    st = lib.wise_decode_noalloc(ctypes.byref(big), P(16), P(16), P(16), P(16), P(16), P(16),
                                 P(16), P(16), P(16), None)
    assert st == 3
    assert b"16777216" in lib.wise_last_error()


def _call(shape, d, pt, sl, modes, sup, ws=None):
    """wise_decode with `ws`, or wise_decode_noalloc when ws is None."""
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
    sup = sup.clone()
    if ws is None:
        W.wise.wise_decode_noalloc(shape, d["q"], d["k_cache"], d["v_cache"], pt, sl, modes, sup,
                                   out, lse)
    else:
        W.wise_decode(shape, d["q"], d["k_cache"], d["v_cache"], pt, sl, modes, sup, out, lse, ws)
    torch.cuda.synchronize()
    return out, lse, sup


@pytest.mark.gpu
def test_noalloc_matches_wise_decode_twice(lib):
    """Two calls in a row (a discover depth, then sparse / union rows on its
    mask), then a third with another shape and split size, whose workspace
    layout puts every region at other offsets in the shared scratch: each
    equals wise_decode with a caller-owned workspace bit for bit (the same
    kernels on the same inputs), and the scratch's status word reads 0."""
    lens = np.array([1, 33, 200, 517, 0, 1024], np.int32)
    R = len(lens)
    w = custom_workload("noalloc", R=R, Hq=8, Hkv=4, D=128, dtype="bf16", depths=2, n_planted=3,
                        seq_lens=lens, pool_factor=2, seed=17,
                        depth_modes=[np.zeros(R, np.int8)] * 2)
    shape = shape_for(w)
    assert W.wise_workspace_bytes(shape) <= (16 << 20)
    pt = torch.from_numpy(w.page_table).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    ws = W.alloc_workspace(shape)
    sup0 = dev_support(np.zeros((R, 4, words(w)), np.uint32))
    schedule = [(0, np.array([1, 1, 1, 1, 1, 0], np.int8)),   # discover (+ one dense row)
                (1, np.array([3, 3, 2, 3, 3, 3], np.int8))]   # sparse / union on the new mask
    sup = sup0
    for depth, modes_np in schedule:
        d = {k: v.cuda() for k, v in w.depth_inputs(depth).items()}
        modes = torch.from_numpy(modes_np).cuda()
        ref_out, ref_lse, ref_sup = _call(shape, d, pt, sl, modes, sup, ws)
        out, lse, new_sup = _call(shape, d, pt, sl, modes, sup)
        assert torch.equal(out, ref_out)
        assert np.array_equal(lse.cpu().numpy(), ref_lse.cpu().numpy())
        assert np.array_equal(np_support(new_sup), np_support(ref_sup))
        assert wise.wise_noalloc_status() == 0
        sup = ref_sup
    # A different layout: GQA 32/8 heads, longer rows, 2-block ranges.
    lens2 = np.array([3000, 40, 0, 1500], np.int32)
    w2 = custom_workload("noalloc2", R=4, Hq=32, Hkv=8, D=128, dtype="bf16", depths=1,
                         n_planted=4, seq_lens=lens2, pool_factor=1, seed=23,
                         depth_modes=[np.zeros(4, np.int8)])
    shape2 = shape_for(w2, tiles_per_item=2)
    assert W.wise_workspace_layout(shape2)["partial_ml"] != W.wise_workspace_layout(shape)["partial_ml"]
    assert W.wise_workspace_bytes(shape2) <= (16 << 20)
    d2 = {k: v.cuda() for k, v in w2.depth_inputs(0).items()}
    pt2 = torch.from_numpy(w2.page_table).cuda()
    sl2 = torch.from_numpy(w2.seq_lens).cuda()
    modes2 = torch.from_numpy(np.array([1, 3, 1, 2], np.int8)).cuda()
    rng = np.random.default_rng(3)
    bits = rng.random((4, 8, words(w2) * 32)) < 0.3
    s2 = dev_support(np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(4, 8, -1))
    ref_out, ref_lse, ref_sup = _call(shape2, d2, pt2, sl2, modes2, s2, W.alloc_workspace(shape2))
    out, lse, new_sup = _call(shape2, d2, pt2, sl2, modes2, s2)
    assert torch.equal(out, ref_out)
    assert np.array_equal(lse.cpu().numpy(), ref_lse.cpu().numpy())
    assert np.array_equal(np_support(new_sup), np_support(ref_sup))
    assert wise.wise_noalloc_status() == 0
