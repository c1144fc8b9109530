"""Python binding of libwise.so: argument marshalling only.

Every function here has the name of the C entry point it calls (see
include/wise.h for the operation, layouts and error behaviour), takes torch
CUDA tensors, passes their device pointers and the current torch stream, and
raises WiseError on a non-OK status.  There is no fallback: if the library is
not built, the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Dict, Optional

import torch

from .build import LIBRARY

MODE_DENSE = 0
MODE_DISCOVER = 1
MODE_DISCOVER_UNION = 2
MODE_SPARSE = 3

DTYPE_BF16 = 0
DTYPE_F32 = 1

DEVERR_SEQ_LEN_CLAMPED = 1
DEVERR_WAIT_TIMEOUT = 2
DEVERR_BAD_WORK_LIST = 4

BAD_MODE = 1
BAD_SEQ_LEN = 2
BAD_PAGE = 4
EMPTY_SPARSE_SUPPORT = 8
BAD_SLOT = 16

_STATUS = {0: "WISE_OK", 1: "WISE_ERR_INVALID_ARG", 2: "WISE_ERR_UNSUPPORTED",
           3: "WISE_ERR_WORKSPACE", 4: "WISE_ERR_CUDA"}


class WiseError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


class wise_shape(ctypes.Structure):
    _fields_ = [("num_rows", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
                ("max_pages_per_row", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("tiles_per_item", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float), ("eta", ctypes.c_float)]


class wise_mask(ctypes.Structure):
    """Where the rows' masks live (see include/wise.h): the words of (row r,
    KV head g) are at words + slot(r) * slot_stride + g * W."""
    _fields_ = [("words", ctypes.c_void_p), ("row_slot", ctypes.c_void_p),
                ("slot_stride", ctypes.c_int64), ("num_slots", ctypes.c_int32)]


def make_mask(pool: Optional[torch.Tensor], row_slot: Optional[torch.Tensor] = None,
              layer: int = 0) -> wise_mask:
    """A mask descriptor over `pool`: an int32 CUDA tensor [num_rows,
    num_kv_heads, W] (row_slot None: row r's mask is pool[r]) or
    [slots, layers, num_kv_heads, W] with row_slot an int32 CUDA tensor
    [num_rows] (row r's mask is pool[row_slot[r], layer]; -1: none).  The
    descriptor holds raw pointers: keep the tensors alive while it is used."""
    if pool is None:
        return wise_mask(None, None, 0, 0)
    words = _ptr(pool, torch.int32, "pool")
    if row_slot is None:
        return wise_mask(words, None, 0, 0)
    if pool.dim() != 4:
        raise ValueError("a slot pool is [slots, layers, num_kv_heads, W]")
    S, Lyr, Hkv, Wd = pool.shape
    if not 0 <= layer < Lyr:
        raise ValueError(f"layer {layer} outside [0, {Lyr})")
    return wise_mask(words + layer * Hkv * Wd * 4, _ptr(row_slot, torch.int32, "row_slot"),
                     Lyr * Hkv * Wd, S)


class wise_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status_word", "num_items", "queue", "head_info", "items",
        "partial_ml", "partial_acc", "tile_stats", "tickets", "partial_ml_1", "partial_acc_1",
        "tile_stats_1", "max_items", "total_bytes", "list1", "head_info_1", "items_1")]


_lib: Optional[ctypes.CDLL] = None


def library() -> ctypes.CDLL:
    """The loaded libwise.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(f"{LIBRARY} is not built; run "
                               "`python -m block_sparse_paged_split_gb300.build`")
        lib = ctypes.CDLL(LIBRARY)
        P, S, I64, SZ = ctypes.c_void_p, ctypes.POINTER(wise_shape), ctypes.c_int64, ctypes.c_size_t
        U32 = ctypes.c_uint32
        sigs = {
            "wise_workspace_bytes": [S, ctypes.POINTER(ctypes.c_size_t)],
            "wise_workspace_layout": [S, ctypes.POINTER(wise_layout)],
            "wise_workspace_reset": [S, P, SZ, P],
            "wise_compact_tiles": [S, P, P, P, P, SZ, P],
            "wise_decode_partial": [S, P, P, P, P, P, P, P, SZ, P],
            "wise_decode_finish": [S, P, P, P, SZ, P, P, P, P],
            "wise_decode_partial_ex": [S, P, P, P, P, P, P, P, SZ, U32, P],
            "wise_decode_finish_ex": [S, P, P, P, SZ, U32, P, P, P, P],
            "wise_decode_partial_finish": [S, P, P, P, P, P, P, P, SZ, P, P, P, P],
            "wise_decode": [S, P, P, P, P, P, P, P, P, P, P, SZ, P],
            "wise_decode_noalloc": [S, P, P, P, P, P, P, P, P, P, P],
            "wise_support_union": [P, P, I64, P],
            "wise_support_head_union": [S, P, P],
            "wise_block_mass": [S, P, P, P, P, P, P, P, SZ, P],
            "wise_validate": [S, P, P, P, P, P, P],
            "wise_selftest_wait_timeout": [P, P],
            "wise_noalloc_status": [ctypes.POINTER(ctypes.c_int32), P],
            "wise_compact_tiles_m": [S, P, P, ctypes.POINTER(wise_mask), P, SZ, P],
            "wise_build_sparse_list": [S, P, P, P, SZ, P],
            "wise_build_sparse_list_m": [S, P, ctypes.POINTER(wise_mask), P, SZ, P],
            "wise_build_list": [S, P, P, P, P, SZ, P],
            "wise_build_list_m": [S, P, P, ctypes.POINTER(wise_mask), P, SZ, P],
            "wise_decode_finish_m": [S, P, P, P, SZ, U32, ctypes.POINTER(wise_mask), P, P, P],
            "wise_decode_m": [S, P, P, P, P, P, P, ctypes.POINTER(wise_mask), P, P, P, SZ, P],
            "wise_validate_m": [S, P, P, P, ctypes.POINTER(wise_mask), P, P],
        }
        for name, args in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.wise_status_string.argtypes = [ctypes.c_int]
        lib.wise_status_string.restype = ctypes.c_char_p
        lib.wise_last_error.argtypes = []
        lib.wise_last_error.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise WiseError(status, library().wise_last_error().decode())


def make_shape(*, num_rows: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
               page_size: int, max_pages_per_row: int, num_pages: int,
               max_blocks: Optional[int] = None, dtype: int = DTYPE_BF16, eta: float = 0.95,
               scale: float = 0.0, tiles_per_item: int = 0, tile_tokens: int = 32) -> wise_shape:
    if max_blocks is None:
        max_blocks = -(-max_pages_per_row * page_size // tile_tokens)
    return wise_shape(num_rows, num_q_heads, num_kv_heads, head_dim, page_size, tile_tokens,
                      max_pages_per_row, num_pages, max_blocks, tiles_per_item, dtype, scale, eta)


def mask_words(shape: wise_shape) -> int:
    return -(-shape.max_blocks // 32)


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _elem(shape: wise_shape) -> torch.dtype:
    return torch.bfloat16 if shape.dtype == DTYPE_BF16 else torch.float32


def wise_workspace_bytes(shape: wise_shape) -> int:
    n = ctypes.c_size_t()
    _check(library().wise_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)))
    return n.value


def wise_workspace_layout(shape: wise_shape) -> Dict[str, int]:
    lay = wise_layout()
    _check(library().wise_workspace_layout(ctypes.byref(shape), ctypes.byref(lay)))
    return {name: getattr(lay, name) for name, _ in wise_layout._fields_}


def wise_workspace_reset(shape: wise_shape, workspace: torch.Tensor, stream=None) -> None:
    _check(library().wise_workspace_reset(ctypes.byref(shape), _ptr(workspace, torch.uint8, "workspace"),
                                          workspace.numel(), _stream(stream)))


def alloc_workspace(shape: wise_shape, device=None) -> torch.Tensor:
    """A workspace of the right size (torch allocations are 256-byte aligned)."""
    return torch.empty(wise_workspace_bytes(shape), dtype=torch.uint8,
                       device=device or torch.device("cuda"))


def wise_compact_tiles(shape, modes, seq_lens, support, workspace, stream=None) -> None:
    _check(library().wise_compact_tiles(
        ctypes.byref(shape), _ptr(modes, torch.int8, "modes"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(support, torch.int32, "support"), _ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)))


def wise_build_sparse_list(shape, seq_lens, support, workspace, stream=None) -> None:
    """List 1 for a call in which every row is sparse, from the mask alone
    (then wise_decode_partial_ex / wise_decode_finish_ex with FLAG_SPARSE_LIST)."""
    _check(library().wise_build_sparse_list(
        ctypes.byref(shape), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(support, torch.int32, "support"), _ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)))


def wise_build_list(shape, modes, seq_lens, support, workspace, stream=None) -> None:
    """List 1 for a call of any modes (then wise_decode_partial_ex /
    wise_decode_finish_ex with FLAG_SPARSE_LIST | FLAG_LIST_MODES and the same
    modes); support may be None."""
    _check(library().wise_build_list(
        ctypes.byref(shape), _ptr(modes, torch.int8, "modes"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(support, torch.int32, "support"), _ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)))


def wise_decode_partial(shape, q, k_cache, v_cache, page_table, seq_lens, modes, workspace,
                        stream=None) -> None:
    e = _elem(shape)
    _check(library().wise_decode_partial(
        ctypes.byref(shape), _ptr(q, e, "q"), _ptr(k_cache, e, "k_cache"), _ptr(v_cache, e, "v_cache"),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(modes, torch.int8, "modes"), _ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)))


def wise_decode_finish(shape, modes, seq_lens, workspace, support, out, lse, stream=None) -> None:
    e = _elem(shape)
    _check(library().wise_decode_finish(
        ctypes.byref(shape), _ptr(modes, torch.int8, "modes"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _ptr(support, torch.int32, "support"), _ptr(out, e, "out"), _ptr(lse, torch.float32, "lse"),
        _stream(stream)))


FLAG_SLOT_SET_1 = 1
FLAG_EARLY_START = 2
FLAG_BUILD_SPARSE_LIST = 4
FLAG_SPARSE_LIST = 8
FLAG_DENSE_LIST = 16
FLAG_INPUTS_READY = 32
FLAG_LIST_MODES = 64
DENSE_LIST_MAX_ROWS = 256
MAX_BLOCKS = 4096  # WISE_MAX_BLOCKS: largest max_blocks (rows of up to 128K tokens)


def wise_decode_partial_ex(shape, q, k_cache, v_cache, page_table, seq_lens, modes, workspace,
                           flags=0, stream=None) -> None:
    """flags: FLAG_SLOT_SET_1, FLAG_EARLY_START, FLAG_SPARSE_LIST (modes may
    then be None), FLAG_DENSE_LIST, FLAG_INPUTS_READY, FLAG_LIST_MODES."""
    e = _elem(shape)
    _check(library().wise_decode_partial_ex(
        ctypes.byref(shape), _ptr(q, e, "q"), _ptr(k_cache, e, "k_cache"), _ptr(v_cache, e, "v_cache"),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(modes, torch.int8, "modes"), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        flags, _stream(stream)))


def wise_decode_finish_ex(shape, modes, seq_lens, workspace, support, out, lse, flags=0,
                          stream=None) -> None:
    """flags: FLAG_SLOT_SET_1, FLAG_BUILD_SPARSE_LIST, FLAG_SPARSE_LIST (modes
    may then be None), FLAG_DENSE_LIST, FLAG_LIST_MODES (with FLAG_SPARSE_LIST:
    the list came from wise_build_list for these modes)."""
    e = _elem(shape)
    _check(library().wise_decode_finish_ex(
        ctypes.byref(shape), _ptr(modes, torch.int8, "modes"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), flags,
        _ptr(support, torch.int32, "support"), _ptr(out, e, "out"), _ptr(lse, torch.float32, "lse"),
        _stream(stream)))


def wise_decode_partial_finish(shape, q, k_cache, v_cache, page_table, seq_lens, modes, workspace,
                               support, out, lse, stream=None) -> None:
    e = _elem(shape)
    _check(library().wise_decode_partial_finish(
        ctypes.byref(shape), _ptr(q, e, "q"), _ptr(k_cache, e, "k_cache"), _ptr(v_cache, e, "v_cache"),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(modes, torch.int8, "modes"), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _ptr(support, torch.int32, "support"), _ptr(out, e, "out"), _ptr(lse, torch.float32, "lse"),
        _stream(stream)))


def wise_decode(shape, q, k_cache, v_cache, page_table, seq_lens, modes, support, out, lse,
                workspace, stream=None) -> None:
    e = _elem(shape)
    _check(library().wise_decode(
        ctypes.byref(shape), _ptr(q, e, "q"), _ptr(k_cache, e, "k_cache"), _ptr(v_cache, e, "v_cache"),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(modes, torch.int8, "modes"), _ptr(support, torch.int32, "support"),
        _ptr(out, e, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def wise_decode_noalloc(shape, q, k_cache, v_cache, page_table, seq_lens, modes, support, out,
                        lse, stream=None) -> None:
    """wise_decode without a workspace argument, for callers that cannot
    allocate device memory: the library's static 16 MiB device scratch is
    used instead (see include/wise.h for its limits and sharing rules)."""
    e = _elem(shape)
    _check(library().wise_decode_noalloc(
        ctypes.byref(shape), _ptr(q, e, "q"), _ptr(k_cache, e, "k_cache"), _ptr(v_cache, e, "v_cache"),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(modes, torch.int8, "modes"), _ptr(support, torch.int32, "support"),
        _ptr(out, e, "out"), _ptr(lse, torch.float32, "lse"), _stream(stream)))


def wise_noalloc_status(stream=None) -> int:
    """The WISE_DEVERR_* word of the last wise_decode_noalloc call in the
    current context (copied to the host; synchronises the stream)."""
    word = ctypes.c_int32(-1)
    _check(library().wise_noalloc_status(ctypes.byref(word), _stream(stream)))
    torch.cuda.synchronize()
    return word.value


def wise_compact_tiles_m(shape, modes, seq_lens, mask: wise_mask, workspace, stream=None) -> None:
    _check(library().wise_compact_tiles_m(
        ctypes.byref(shape), _ptr(modes, torch.int8, "modes"), _ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.byref(mask), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)))


def wise_build_sparse_list_m(shape, seq_lens, mask: wise_mask, workspace, stream=None) -> None:
    _check(library().wise_build_sparse_list_m(
        ctypes.byref(shape), _ptr(seq_lens, torch.int32, "seq_lens"), ctypes.byref(mask),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def wise_build_list_m(shape, modes, seq_lens, mask: wise_mask, workspace, stream=None) -> None:
    _check(library().wise_build_list_m(
        ctypes.byref(shape), _ptr(modes, torch.int8, "modes"), _ptr(seq_lens, torch.int32, "seq_lens"),
        ctypes.byref(mask), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)))


def wise_decode_finish_m(shape, modes, seq_lens, workspace, mask: wise_mask, out, lse, flags=0,
                         stream=None) -> None:
    e = _elem(shape)
    _check(library().wise_decode_finish_m(
        ctypes.byref(shape), _ptr(modes, torch.int8, "modes"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), flags, ctypes.byref(mask),
        _ptr(out, e, "out"), _ptr(lse, torch.float32, "lse"), _stream(stream)))


def wise_decode_m(shape, q, k_cache, v_cache, page_table, seq_lens, modes, mask: wise_mask, out,
                  lse, workspace, stream=None) -> None:
    e = _elem(shape)
    _check(library().wise_decode_m(
        ctypes.byref(shape), _ptr(q, e, "q"), _ptr(k_cache, e, "k_cache"), _ptr(v_cache, e, "v_cache"),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(modes, torch.int8, "modes"), ctypes.byref(mask), _ptr(out, e, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)))


def wise_validate_m(shape, page_table, seq_lens, modes, mask: wise_mask, err_word,
                    stream=None) -> None:
    _check(library().wise_validate_m(
        ctypes.byref(shape), _ptr(page_table, torch.int32, "page_table"),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(modes, torch.int8, "modes"),
        ctypes.byref(mask), _ptr(err_word, torch.int32, "err_word"), _stream(stream)))


def wise_support_union(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    if dst.numel() != src.numel():
        raise ValueError("dst and src must have the same number of words")
    _check(library().wise_support_union(_ptr(dst, torch.int32, "dst"), _ptr(src, torch.int32, "src"),
                                        dst.numel(), _stream(stream)))


def wise_block_mass(shape, q, k_cache, page_table, seq_lens, modes, lse, workspace,
                    stream=None) -> None:
    e = _elem(shape)
    _check(library().wise_block_mass(
        ctypes.byref(shape), _ptr(q, e, "q"), _ptr(k_cache, e, "k_cache"),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(modes, torch.int8, "modes"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def wise_support_head_union(shape, support, stream=None) -> None:
    _check(library().wise_support_head_union(ctypes.byref(shape), _ptr(support, torch.int32, "support"),
                                             _stream(stream)))


def wise_validate(shape, page_table, seq_lens, modes, support, err_word, stream=None) -> None:
    _check(library().wise_validate(
        ctypes.byref(shape), _ptr(page_table, torch.int32, "page_table"),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(modes, torch.int8, "modes"),
        _ptr(support, torch.int32, "support"), _ptr(err_word, torch.int32, "err_word"),
        _stream(stream)))


def wise_selftest_wait_timeout(status_word: torch.Tensor, stream=None) -> None:
    """Run the bounded-wait self-test (see include/wise.h): about 500 ms later
    the device int32 `status_word` has DEVERR_WAIT_TIMEOUT set."""
    _check(library().wise_selftest_wait_timeout(_ptr(status_word, torch.int32, "status_word"),
                                                 _stream(stream)))


def workspace_views(shape: wise_shape, workspace: torch.Tensor) -> Dict[str, torch.Tensor]:
    """Typed views of the workspace regions (for inspecting intermediates)."""
    lay = wise_workspace_layout(shape)
    R, Hq, Hkv, D = shape.num_rows, shape.num_q_heads, shape.num_kv_heads, shape.head_dim
    G = Hq // Hkv
    mi = lay["max_items"]

    def region(off, count, dt):
        nbytes = count * torch.tensor([], dtype=dt).element_size()
        return workspace[off:off + nbytes].view(dt)

    return {
        "status": region(lay["status_word"], 1, torch.int32),
        "num_items": region(lay["num_items"], 1, torch.int32),
        "head_info": region(lay["head_info"], R * Hkv * 4, torch.int32).view(R, Hkv, 4),
        "items": region(lay["items"], mi * 4, torch.int32).view(mi, 4),
        "queue": region(lay["queue"], 1, torch.int32),
        "partial_ml": region(lay["partial_ml"], mi * G * 2, torch.float32).view(mi, G, 2),
        "partial_acc": region(lay["partial_acc"], mi * G * D, torch.float32).view(mi, G, D),
        "tile_stats": region(lay["tile_stats"], R * Hq * shape.max_blocks * 2, torch.float32).view(R, Hq, shape.max_blocks, 2),
        "tickets": region(lay["tickets"], R * Hkv, torch.int32).view(R, Hkv),
        "partial_ml_1": region(lay["partial_ml_1"], mi * G * 2, torch.float32).view(mi, G, 2),
        "partial_acc_1": region(lay["partial_acc_1"], mi * G * D, torch.float32).view(mi, G, D),
        "tile_stats_1": region(lay["tile_stats_1"], R * Hq * shape.max_blocks * 2, torch.float32).view(R, Hq, shape.max_blocks, 2),
        "list1_counter": region(lay["list1"], 16, torch.int32),
        "head_info_1": region(lay["head_info_1"], R * Hkv * 4, torch.int32).view(R, Hkv, 4),
        "items_1": region(lay["items_1"], _tiles_per_item(shape) * mi * 4,
                          torch.int32).view(_tiles_per_item(shape), mi, 4),
    }


def _tiles_per_item(shape: wise_shape) -> int:
    """Blocks per split range T as the library resolves tiles_per_item = 0."""
    if shape.tiles_per_item:
        return shape.tiles_per_item
    items16 = shape.num_rows * shape.num_kv_heads * (-(-shape.max_blocks // 16))
    return 16 if shape.max_blocks > 64 and items16 >= 4096 else 8


LOG2E = 1.0 / math.log(2.0)
