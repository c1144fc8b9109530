"""Masks addressed per request slot and layer (the [slot, layer, head, block]
bitmask of the WISE PR, "What changes", wise.py bullet), through the _m calls
of the C ABI: every call on a slot pool equals, bit for bit, the same call on
the masks gathered into a [row, head, word] array and scattered back, and
agrees with the oracle's slot-addressed decode."""
import numpy as np
import pytest
import torch

import block_sparse_paged_split_gb300 as W
from block_sparse_paged_split_gb300.workload import custom_workload
from tests.gpu_harness import (Batch, compare_outputs, dev_support, item_invariant_fails,
                               list1_schedule, np_support, oracle_module, shape_for, words)
from tests.oracle_pins import as_oracle_array
from oracle import wise_oracle as O

pytestmark = pytest.mark.gpu

LENS = np.array([1, 31, 300, 517, 0, 1024, 640, 64], np.int32)
SLOTS, LAYERS, LAYER = 11, 3, 1


def _setup(Hq, Hkv, lens=LENS, seed=71):
    R = len(lens)
    w = custom_workload("slots", R=R, Hq=Hq, Hkv=Hkv, D=128, dtype="bf16", depths=3, n_planted=3,
                        seq_lens=lens, pool_factor=2, seed=seed,
                        depth_modes=[np.zeros(R, np.int8)] * 3)
    rng = np.random.default_rng(seed)
    bits = rng.random((SLOTS, LAYERS, Hkv, words(w) * 32)) < 0.3
    pool = np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(
        SLOTS, LAYERS, Hkv, -1).copy()
    row_slot = rng.permutation(SLOTS)[:R].astype(np.int32)
    row_slot[2] = -1  # a row without a mask
    return w, pool, row_slot


def _gathered(pool, row_slot):
    return O.gather_slot_masks(pool, row_slot, LAYER)


def _scatter(pool, row_slot, sup):
    out = pool.copy()
    for r, s in enumerate(row_slot):
        if s >= 0:
            out[s, LAYER] = sup[r]
    return out


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_slot_pool_equals_gathered_masks(Hq, Hkv):
    w, pool_np, row_slot = _setup(Hq, Hkv)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    modes_np = np.array([1, 2, 1, 3, 3, 2, 0, 3], np.int8)
    modes = torch.from_numpy(modes_np).cuda()
    slots_t = torch.from_numpy(row_slot).cuda()
    d = b.dev(0)
    # on the pool, in place
    pool = dev_support(pool_np)
    out_a = torch.empty_like(d["q"])
    lse_a = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    W.wise_decode_m(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens, modes,
                    W.make_mask(pool, slots_t, LAYER), out_a, lse_a, W.alloc_workspace(shape))
    # on gathered masks, scattered back
    sup = dev_support(_gathered(pool_np, row_slot))
    out_b = torch.empty_like(d["q"])
    lse_b = torch.empty_like(lse_a)
    W.wise_decode(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table, b.seq_lens, modes, sup,
                  out_b, lse_b, W.alloc_workspace(shape))
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)
    assert np.array_equal(np_support(pool), _scatter(pool_np, row_slot, np_support(sup)))
    # the oracle's slot-addressed decode: outputs; the pool outside the
    # discovering rows' own slots is untouched
    c = b.cpu(0)
    o = oracle_module("f32").decode_layer_slots(
        as_oracle_array(c["q"]), as_oracle_array(c["k_cache"]), as_oracle_array(c["v_cache"]),
        w.page_table, w.seq_lens, modes_np, pool_np, row_slot, LAYER, eta=w.eta)
    g = {"out": out_a.double().cpu().numpy(), "lse": lse_a.cpu().numpy()}
    assert not compare_outputs(w, g, o)
    after = np_support(pool)
    written = {(int(s), LAYER) for r, s in enumerate(row_slot)
               if s >= 0 and modes_np[r] in (1, 2) and w.seq_lens[r] > 0}
    for sl in range(SLOTS):
        for ly in range(LAYERS):
            if (sl, ly) not in written:
                assert np.array_equal(after[sl, ly], pool_np[sl, ly]), (sl, ly)


@pytest.mark.parametrize("dense", [False, True])
def test_slot_pool_through_list1(dense):
    """Discover, union-discover building list 1, then a sparse call on list 1,
    all on the slot pool: equal to the gathered-mask calls (after their own
    compaction), bit for bit; list 1's items partition the oracle's lists of
    the slot masks.  dense: the two discovery depths on the dense list (no
    compaction at all on the pool side)."""
    w, pool_np, row_slot = _setup(4, 4, seed=73)
    b = Batch(w)
    R = w.num_rows
    shape = shape_for(w)
    slots_t = torch.from_numpy(row_slot).cuda()
    disc = torch.full((R,), W.MODE_DISCOVER, dtype=torch.int8, device="cuda")
    union = torch.full((R,), W.MODE_DISCOVER_UNION, dtype=torch.int8, device="cuda")

    def run(mask_of_call, flat: bool, dense_list: bool = False):
        ws = W.alloc_workspace(shape)
        W.wise_workspace_reset(shape, ws)
        outs = []
        for depth, m, flags in ((0, disc, 0), (1, union, W.FLAG_BUILD_SPARSE_LIST),
                                (2, None, W.FLAG_SPARSE_LIST)):
            d = b.dev(depth)
            out = torch.empty_like(d["q"])
            lse = torch.empty((R, 4), dtype=torch.float32, device="cuda")
            on_dense = dense_list and depth < 2
            if depth == 0 and not on_dense:
                if flat:
                    W.wise_compact_tiles(shape, m, b.seq_lens, mask_of_call, ws)
                else:
                    W.wise_compact_tiles_m(shape, m, b.seq_lens, mask_of_call, ws)
            if on_dense:
                flags |= W.FLAG_DENSE_LIST
            pflags = flags & (W.FLAG_SPARSE_LIST | W.FLAG_DENSE_LIST)
            W.wise_decode_partial_ex(shape, d["q"], d["k_cache"], d["v_cache"], b.page_table,
                                     b.seq_lens, m, ws, pflags)
            if flat:
                W.wise_decode_finish_ex(shape, m, b.seq_lens, ws, mask_of_call, out, lse, flags)
            else:
                W.wise_decode_finish_m(shape, m, b.seq_lens, ws, mask_of_call, out, lse, flags)
            torch.cuda.synchronize()
            outs.append((out.cpu(), lse.cpu()))
        return outs, {k: v.cpu() for k, v in W.workspace_views(shape, ws).items()}

    pool = dev_support(pool_np)
    a, va = run(W.make_mask(pool, slots_t, LAYER), flat=False, dense_list=dense)
    sup = dev_support(_gathered(pool_np, row_slot))
    bb, vb = run(sup, flat=True)
    # Depths 0 and 1 discover (their outputs do not depend on the mask); at
    # depth 2 the slot-less row differs by design: on the pool it has no mask,
    # while the gathered copy kept what the row discovered.
    keep = row_slot >= 0
    for depth, ((oa, la), (ob, lb)) in enumerate(zip(a, bb)):
        if depth < 2:
            assert torch.equal(oa, ob) and torch.equal(la, lb)
        else:
            assert torch.equal(oa[keep], ob[keep]) and torch.equal(la[keep], lb[keep])
    assert np.array_equal(np_support(pool), _scatter(pool_np, row_slot, np_support(sup)))
    # the slot-less row has no mask: no item in list 1, output 0 / -inf
    assert torch.all(a[2][0][2] == 0) and torch.all(torch.isneginf(a[2][1][2]))
    T = W.wise._tiles_per_item(shape)
    gathered_after = np_support(sup)
    gathered_after[row_slot < 0] = 0
    ref = O.compact_tiles(gathered_after, np.full(R, 3, np.int8), w.seq_lens, 32)
    fails = item_invariant_fails(list1_schedule(va, T), va["head_info_1"].numpy(), ref["lists"], T,
                                 -(-shape.max_blocks // T), w.seq_lens, None, 4,
                                 compact_slots=True)
    assert not fails, fails[:5]


def test_validate_flags_bad_slots():
    w, pool_np, row_slot = _setup(4, 4)
    shape = shape_for(w)
    pool = dev_support(pool_np)
    bad = row_slot.copy()
    bad[0], bad[1] = -2, SLOTS  # below -1, past the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    modes = torch.zeros(w.num_rows, dtype=torch.int8, device="cuda")
    W.wise_validate_m(shape, torch.from_numpy(w.page_table).cuda(), torch.from_numpy(w.seq_lens).cuda(),
                      modes, W.make_mask(pool, torch.from_numpy(bad).cuda(), LAYER), err)
    torch.cuda.synchronize()
    assert int(err.item()) & W.wise.BAD_SLOT
    err.zero_()
    W.wise_validate_m(shape, torch.from_numpy(w.page_table).cuda(), torch.from_numpy(w.seq_lens).cuda(),
                      modes, W.make_mask(pool, torch.from_numpy(row_slot).cuda(), LAYER), err)
    torch.cuda.synchronize()
    assert not (int(err.item()) & W.wise.BAD_SLOT)
