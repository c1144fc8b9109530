"""WISE working-set paged decode attention for GB300 (sm_103a).

The compute lives in libwise.so (hand-written CUDA; C ABI in include/wise.h);
`block_sparse_paged_split_gb300.wise` is its Python binding.  Importing the
package does not load the library; the first call does, and raises if the
library has not been built.
"""
from .wise import (MODE_DENSE, MODE_DISCOVER, MODE_DISCOVER_UNION, MODE_SPARSE, DTYPE_BF16,
                   DTYPE_F32, WiseError, alloc_workspace, make_shape, mask_words,
                   wise_block_mass, wise_compact_tiles, wise_build_sparse_list, wise_build_sparse_list_m, wise_build_list, wise_build_list_m, wise_decode, wise_decode_finish, wise_decode_partial,
                   wise_decode_partial_finish, wise_decode_partial_ex, wise_decode_finish_ex,
                   FLAG_SLOT_SET_1, FLAG_EARLY_START, FLAG_BUILD_SPARSE_LIST, FLAG_SPARSE_LIST,
                   FLAG_DENSE_LIST, FLAG_INPUTS_READY, FLAG_LIST_MODES, DENSE_LIST_MAX_ROWS, MAX_BLOCKS, wise_workspace_reset,
                   wise_support_head_union, wise_support_union, wise_validate, wise_workspace_bytes,
                   wise_workspace_layout, workspace_views, wise_mask, make_mask,
                   wise_compact_tiles_m, wise_decode_finish_m, wise_decode_m, wise_validate_m)

__all__ = ["MODE_DENSE", "MODE_DISCOVER", "MODE_DISCOVER_UNION", "MODE_SPARSE", "DTYPE_BF16",
           "DTYPE_F32", "WiseError", "alloc_workspace", "make_shape", "mask_words",
           "wise_block_mass", "wise_compact_tiles", "wise_build_sparse_list", "wise_build_sparse_list_m", "wise_build_list", "wise_build_list_m", "wise_decode", "wise_decode_finish", "wise_decode_partial",
           "wise_decode_partial_finish", "wise_decode_partial_ex", "wise_decode_finish_ex",
           "FLAG_SLOT_SET_1", "FLAG_EARLY_START", "FLAG_BUILD_SPARSE_LIST", "FLAG_SPARSE_LIST",
           "FLAG_DENSE_LIST", "FLAG_INPUTS_READY", "FLAG_LIST_MODES", "DENSE_LIST_MAX_ROWS", "MAX_BLOCKS", "wise_workspace_reset",
           "wise_support_head_union", "wise_support_union", "wise_validate", "wise_workspace_bytes",
           "wise_workspace_layout", "workspace_views", "wise_mask", "make_mask",
           "wise_compact_tiles_m", "wise_decode_finish_m", "wise_decode_m", "wise_validate_m"]
