"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and its host-side checks reject bad arguments before
anything is enqueued (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300 import wise
from block_sparse_paged_split_gb300.build import INCLUDE, build_library

HEADER = os.path.join(INCLUDE, "wise.h")


@pytest.fixture(scope="module")
def lib():
    build_library()
    return wise.library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:wise_status|const char \*)\s*(wise_\w+)\(", text, re.M)))


def test_header_declares_the_path(lib):
    names = declared_functions()
    for required in ("wise_compact_tiles", "wise_decode_partial", "wise_decode_finish",
                     "wise_support_union", "wise_workspace_bytes", "wise_validate", "wise_decode"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _shape(**kw):
    base = dict(num_rows=4, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                max_pages_per_row=64, num_pages=256)
    base.update(kw)
    return W.make_shape(**base)


def test_workspace_layout_is_aligned_and_sized(lib):
    s = _shape()
    lay = W.wise_workspace_layout(s)
    assert lay["total_bytes"] == W.wise_workspace_bytes(s)
    offs = [lay[k] for k in ("head_info", "items", "partial_ml", "partial_acc", "tile_stats")]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    # max items: every (row, KV head) split into ceil(max_blocks / 8) block
    # ranges (the default range is 8 blocks)
    assert lay["max_items"] == 4 * 2 * -(-s.max_blocks // 8)
    assert lay["partial_acc"] - lay["partial_ml"] >= lay["max_items"] * 4 * 8
    # zero rows: header only
    assert W.wise_workspace_bytes(_shape(num_rows=0)) == 256


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, 2), ("num_kv_heads", 3, 1), ("num_q_heads", 24, 2), ("page_size", 12, 2),
    ("page_size", 8, 2),
    ("tile_tokens", 64, 2), ("max_blocks", 4097, 2), ("max_blocks", 0, 2), ("dtype", 7, 1),
    ("eta", 0.0, 1), ("eta", float("nan"), 1), ("scale", -1.0, 1), ("num_rows", -1, 1),
    ("num_pages", 0, 1), ("tiles_per_item", 17, 1), ("tiles_per_item", 3, 1)])
def test_shape_checks(lib, field, value, status):
    s = _shape()
    setattr(s, field, value)
    with pytest.raises(W.WiseError) as e:
        W.wise_workspace_bytes(s)
    assert e.value.status == status
    assert lib.wise_last_error().decode()


def test_host_checks_before_any_launch(lib):
    s = _shape()
    n = W.wise_workspace_bytes(s)
    P = ctypes.c_void_p
    # NULL workspace
    st = lib.wise_compact_tiles(ctypes.byref(s), P(16), P(16), None, None, n, None)
    assert st == 3
    # misaligned workspace
    st = lib.wise_compact_tiles(ctypes.byref(s), P(16), P(16), None, P(4096 + 8), n, None)
    assert st == 3
    # NULL lengths
    st = lib.wise_compact_tiles(ctypes.byref(s), P(16), None, None, P(4096), n, None)
    assert st == 1
    # workspace too small
    st = lib.wise_decode_partial(ctypes.byref(s), P(16), P(16), P(16), P(16), P(16), P(16),
                                 P(4096), n - 1, None)
    assert st == 3 and b"too small" in lib.wise_last_error()
    # NULL required pointers
    st = lib.wise_decode_partial(ctypes.byref(s), None, P(16), P(16), P(16), P(16), P(16),
                                 P(4096), n, None)
    assert st == 1
    # misaligned q
    st = lib.wise_decode_partial(ctypes.byref(s), P(18), P(16), P(16), P(16), P(16), P(16),
                                 P(4096), n, None)
    assert st == 1
    st = lib.wise_decode_finish(ctypes.byref(s), P(16), P(16), P(4096), n, None, P(24), P(16), None)
    assert st == 1  # out must be 16-byte aligned
    st = lib.wise_support_union(None, P(16), 5, None)
    assert st == 1
    assert lib.wise_support_union(None, None, 0, None) == 0   # nothing to do
    assert lib.wise_support_union(P(16), P(16), -1, None) == 1
    st = lib.wise_validate(ctypes.byref(s), P(16), P(16), P(16), None, None, None)
    assert st == 1
    assert lib.wise_status_string(4) == b"WISE_ERR_CUDA"


def test_zero_rows_is_a_no_op(lib):
    s = _shape(num_rows=0)
    n = W.wise_workspace_bytes(s)
    P = ctypes.c_void_p
    assert lib.wise_decode_partial(ctypes.byref(s), None, None, None, None, None, None,
                                   P(4096), n, None) == 0
    assert lib.wise_decode_finish(ctypes.byref(s), None, None, P(4096), n, None, None, None, None) == 0


def test_flag_checks(lib):
    s = _shape()
    n = W.wise_workspace_bytes(s)
    P = ctypes.c_void_p
    # unknown partial flags, and a partial-only flag given to the finish
    st = lib.wise_decode_partial_ex(ctypes.byref(s), P(16), P(16), P(16), P(16), P(16), P(16),
                                    P(4096), n, ctypes.c_uint32(1 << 10), None)
    assert st == 1 and b"flags" in lib.wise_last_error()
    st = lib.wise_decode_finish_ex(ctypes.byref(s), P(16), P(16), P(4096), n,
                                   ctypes.c_uint32(1 << 10), P(16), P(16), P(16), None)
    assert st == 1 and b"flags" in lib.wise_last_error()
    st = lib.wise_decode_partial_ex(ctypes.byref(s), P(16), P(16), P(16), P(16), P(16), P(16),
                                    P(4096), n, ctypes.c_uint32(W.FLAG_BUILD_SPARSE_LIST), None)
    assert st == 1  # a finish-only flag
    st = lib.wise_decode_finish_ex(ctypes.byref(s), P(16), P(16), P(4096), n,
                                   ctypes.c_uint32(W.FLAG_EARLY_START), P(16), P(16), P(16), None)
    assert st == 1
    # building the next sparse list needs the mask
    st = lib.wise_decode_finish_ex(ctypes.byref(s), P(16), P(16), P(4096), n,
                                   ctypes.c_uint32(W.FLAG_BUILD_SPARSE_LIST), None, P(16), P(16), None)
    assert st == 1 and b"support" in lib.wise_last_error()
    # a call on list 1 cannot rebuild it
    st = lib.wise_decode_finish_ex(ctypes.byref(s), P(16), P(16), P(4096), n,
                                   ctypes.c_uint32(W.FLAG_BUILD_SPARSE_LIST | W.FLAG_SPARSE_LIST),
                                   P(16), P(16), P(16), None)
    assert st == 1
    # a call on list 1 needs no modes; without the flag it does
    st = lib.wise_decode_partial_ex(ctypes.byref(s), P(16), P(16), P(16), P(16), P(16), None,
                                    P(4096), n, ctypes.c_uint32(0), None)
    assert st == 1
    lay = W.wise_workspace_layout(s)
    # the second slot set: three more aligned regions after the first set
    second = [lay[k] for k in ("partial_ml_1", "partial_acc_1", "tile_stats_1")]
    assert all(o % 256 == 0 for o in second) and min(second) > lay["tile_stats"]
    assert lay["total_bytes"] > max(second)
    # list 1: header inside the first 256 bytes, head info and T buckets of
    # max_items records after the second slot set
    assert 0 < lay["list1"] and lay["list1"] + 64 <= 256
    assert lay["head_info_1"] % 256 == 0 and lay["items_1"] % 256 == 0
    assert lay["head_info_1"] > max(second) and lay["items_1"] >= lay["head_info_1"] + 4 * 2 * 16
    assert lay["total_bytes"] >= lay["items_1"] + 8 * lay["max_items"] * 16


def test_dense_list_checks(lib):
    """WISE_FLAG_DENSE_LIST: at most DENSE_LIST_MAX_ROWS rows, not with list 1
    nor the folded finish, an early start only with WISE_FLAG_INPUTS_READY;
    checked on the host before anything is enqueued."""
    P = ctypes.c_void_p
    D = ctypes.c_uint32(W.FLAG_DENSE_LIST)
    big = _shape(num_rows=W.DENSE_LIST_MAX_ROWS + 1)
    nb = W.wise_workspace_bytes(big)
    assert lib.wise_decode_partial_ex(ctypes.byref(big), P(16), P(16), P(16), P(16), P(16), P(16),
                                      P(4096), nb, D, None) == 2  # WISE_ERR_UNSUPPORTED
    assert b"rows" in lib.wise_last_error()
    assert lib.wise_decode_finish_ex(ctypes.byref(big), P(16), P(16), P(4096), nb, D, None,
                                     P(16), P(16), None) == 2
    s = _shape()
    n = W.wise_workspace_bytes(s)
    # an early start on the dense list or list 1 needs WISE_FLAG_INPUTS_READY
    for flags in (W.FLAG_DENSE_LIST | W.FLAG_SPARSE_LIST, W.FLAG_DENSE_LIST | W.FLAG_EARLY_START,
                  W.FLAG_SPARSE_LIST | W.FLAG_EARLY_START):
        st = lib.wise_decode_partial_ex(ctypes.byref(s), P(16), P(16), P(16), P(16), P(16), P(16),
                                        P(4096), n, ctypes.c_uint32(flags), None)
        assert st == 1, flags
    st = lib.wise_decode_finish_ex(ctypes.byref(s), P(16), P(16), P(4096), n,
                                   ctypes.c_uint32(W.FLAG_DENSE_LIST | W.FLAG_SPARSE_LIST),
                                   None, P(16), P(16), None)
    assert st == 1
    assert W.DENSE_LIST_MAX_ROWS == 256


def test_workspace_reset_checks(lib):
    """wise_workspace_reset checks the shape and the workspace (NULL, too
    small, misaligned) before it enqueues anything."""
    s = _shape()
    n = W.wise_workspace_bytes(s)
    P = ctypes.c_void_p
    assert lib.wise_workspace_reset(ctypes.byref(s), None, n, None) == 3  # WISE_ERR_WORKSPACE
    assert lib.wise_workspace_reset(ctypes.byref(s), P(4096), n - 1, None) == 3
    assert b"too small" in lib.wise_last_error()
    assert lib.wise_workspace_reset(ctypes.byref(s), P(4096 + 16), n, None) == 3
    bad = _shape(head_dim=96)
    assert lib.wise_workspace_reset(ctypes.byref(bad), P(4096), n, None) == 2


def test_noalloc_status_rejects_a_null_pointer(lib):
    assert lib.wise_noalloc_status(None, None) == 1
    assert b"host_status" in lib.wise_last_error()


def test_build_sparse_list_checks(lib):
    """wise_build_sparse_list: the mask and the lengths are required, the
    workspace is checked; all before anything is enqueued."""
    P = ctypes.c_void_p
    s = _shape()
    n = W.wise_workspace_bytes(s)
    assert lib.wise_build_sparse_list(ctypes.byref(s), P(16), None, P(4096), n, None) == 1
    assert b"support" in lib.wise_last_error()
    assert lib.wise_build_sparse_list(ctypes.byref(s), None, P(16), P(4096), n, None) == 1
    assert lib.wise_build_sparse_list(ctypes.byref(s), P(16), P(16), P(4096), n - 1, None) == 3
    assert lib.wise_build_sparse_list(ctypes.byref(s), P(16), P(16), P(4100), n, None) == 3
    assert lib.wise_build_sparse_list(ctypes.byref(s), P(16), P(18), P(4096), n, None) == 1
    m = W.wise.wise_mask(None, None, 0, 0)
    assert lib.wise_build_sparse_list_m(ctypes.byref(s), P(16), ctypes.byref(m), P(4096), n,
                                        None) == 1
    assert lib.wise_build_sparse_list_m(ctypes.byref(s), P(16), None, P(4096), n, None) == 1


def test_build_list_and_list_modes_checks(lib):
    """wise_build_list needs the modes (the mask may be NULL: sparse rows then
    get no item); WISE_FLAG_LIST_MODES goes with WISE_FLAG_SPARSE_LIST, and
    its finish needs the modes."""
    P = ctypes.c_void_p
    s = _shape()
    n = W.wise_workspace_bytes(s)
    assert lib.wise_build_list(ctypes.byref(s), None, P(16), P(16), P(4096), n, None) == 1
    assert b"modes" in lib.wise_last_error()
    assert lib.wise_build_list(ctypes.byref(s), P(16), None, P(16), P(4096), n, None) == 1
    assert lib.wise_build_list(ctypes.byref(s), P(16), P(16), P(16), P(4096), n - 1, None) == 3
    LM = ctypes.c_uint32(W.FLAG_LIST_MODES)
    assert lib.wise_decode_partial_ex(ctypes.byref(s), P(16), P(16), P(16), P(16), P(16), P(16),
                                      P(4096), n, LM, None) == 1
    assert b"WISE_FLAG_SPARSE_LIST" in lib.wise_last_error()
    assert lib.wise_decode_finish_ex(ctypes.byref(s), P(16), P(16), P(4096), n, LM, None, P(16),
                                     P(16), None) == 1
    both = ctypes.c_uint32(W.FLAG_LIST_MODES | W.FLAG_SPARSE_LIST)
    assert lib.wise_decode_finish_ex(ctypes.byref(s), None, P(16), P(4096), n, both, None, P(16),
                                     P(16), None) == 1
    assert W.FLAG_LIST_MODES == 64


def test_max_blocks_limit(lib):
    """WISE_MAX_BLOCKS (rows of up to 128K tokens): the header, the binding and
    the shape check agree."""
    text = open(HEADER).read()
    assert re.search(r"#define WISE_MAX_BLOCKS (\d+)", text).group(1) == str(W.MAX_BLOCKS)
    ok = _shape(num_rows=2, num_q_heads=8, num_kv_heads=2, max_blocks=W.MAX_BLOCKS,
                max_pages_per_row=2 * W.MAX_BLOCKS)
    assert W.wise_workspace_bytes(ok) > 0
    bad = _shape(num_rows=2, num_q_heads=8, num_kv_heads=2, max_blocks=W.MAX_BLOCKS + 1,
                 max_pages_per_row=2 * W.MAX_BLOCKS + 2)
    n = ctypes.c_size_t(0)
    assert lib.wise_workspace_bytes(ctypes.byref(bad), ctypes.byref(n)) == 2  # WISE_ERR_UNSUPPORTED
    assert b"max_blocks" in lib.wise_last_error()


def test_default_split_size(lib):
    # short rows: 8 blocks a range
    s = _shape(num_rows=64, num_q_heads=16, num_kv_heads=16, max_blocks=32, max_pages_per_row=64)
    assert W.wise_workspace_layout(s)["max_items"] == 64 * 16 * 4
    # rows past 64 blocks with >= 4096 ranges of 16 blocks: 16 blocks a range
    s = _shape(num_rows=64, num_q_heads=16, num_kv_heads=16, max_blocks=128, max_pages_per_row=256)
    assert W.wise_workspace_layout(s)["max_items"] == 64 * 16 * 8
    # a small batch of long rows keeps 8 (enough items for every consumer)
    s = _shape(num_rows=2, num_q_heads=32, num_kv_heads=8, max_blocks=1024, max_pages_per_row=2048)
    assert W.wise_workspace_layout(s)["max_items"] == 2 * 8 * 128
    # the longest rows (4096 blocks, 128K tokens)
    s = _shape(num_rows=2, num_q_heads=8, num_kv_heads=2, max_blocks=4096, max_pages_per_row=8192)
    assert W.wise_workspace_layout(s)["max_items"] == 2 * 2 * 512
    # an explicit split size wins
    s = _shape(num_rows=2, num_q_heads=32, num_kv_heads=8, max_blocks=1024, max_pages_per_row=2048,
               tiles_per_item=16)
    assert W.wise_workspace_layout(s)["max_items"] == 2 * 8 * 64


def test_selftest_rejects_a_bad_status_pointer(lib):
    P = ctypes.c_void_p
    assert lib.wise_selftest_wait_timeout(None, None) == 1
    assert lib.wise_selftest_wait_timeout(P(4098), None) == 1
    assert b"status_word" in lib.wise_last_error()


def test_mask_descriptor_checks(lib):
    s = _shape()
    n = W.wise_workspace_bytes(s)
    P = ctypes.c_void_p
    mk = lambda words, slots, stride, num: W.wise.wise_mask(words, slots, stride, num)  # noqa: E731
    W_ = -(-s.max_blocks // 32)
    # no descriptor
    assert lib.wise_compact_tiles_m(ctypes.byref(s), P(16), P(16), None, P(4096), n, None) == 1
    # misaligned words or slots
    m = mk(18, None, 0, 0)
    assert lib.wise_compact_tiles_m(ctypes.byref(s), P(16), P(16), ctypes.byref(m), P(4096), n, None) == 1
    m = mk(16, 18, 0, 0)
    assert lib.wise_compact_tiles_m(ctypes.byref(s), P(16), P(16), ctypes.byref(m), P(4096), n, None) == 1
    # a slot stride shorter than one slot's masks
    m = mk(16, 16, s.num_kv_heads * W_ - 1, 4)
    assert lib.wise_decode_finish_m(ctypes.byref(s), P(16), P(16), P(4096), n, 0, ctypes.byref(m),
                                    P(16), P(16), None) == 1
    assert b"slot_stride" in lib.wise_last_error()
    m = mk(16, 16, 0, -1)
    assert lib.wise_validate_m(ctypes.byref(s), P(16), P(16), P(16), ctypes.byref(m), P(16), None) == 1
    # building list 1 needs mask words
    m = mk(None, None, 0, 0)
    assert lib.wise_decode_finish_m(ctypes.byref(s), P(16), P(16), P(4096), n,
                                    W.FLAG_BUILD_SPARSE_LIST, ctypes.byref(m), P(16), P(16), None) == 1


def test_make_mask_addresses_a_layer_of_the_pool():
    import torch
    pool = torch.zeros((5, 3, 2, 4), dtype=torch.int32)
    with pytest.raises(ValueError):
        W.make_mask(pool, torch.zeros(2, dtype=torch.int32), 1)  # a CPU tensor is refused
