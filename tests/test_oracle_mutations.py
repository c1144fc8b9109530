"""Plant plausible mistakes in a private copy of the oracle (on the CPU) and
check that at least one pin catches each.  This is what makes the pins a real
check on the oracle rather than a restatement of it."""
import importlib.util
import math
import os

import numpy as np
import pytest

from tests import oracle_pins

ORACLE_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "wise_oracle.py")


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("wise_oracle_mutant", ORACLE_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def m_scale_squared(O):
    O.scores = lambda q, K, scale: (scale * scale) * (K @ q)


def m_slot_off_by_one(O):
    def row_kv(cache, page_row, L, g):
        P = cache.shape[1]
        j = np.arange(L)
        return O.to_f64(cache[np.asarray(page_row)[j // P], (j + 1) % P, g])
    O.row_kv = row_kv


def m_page_order_reversed(O):
    def row_kv(cache, page_row, L, g):
        P = cache.shape[1]
        j = np.arange(L)
        npg = -(-L // P)
        return O.to_f64(cache[np.asarray(page_row)[npg - 1 - j // P], j % P, g])
    O.row_kv = row_kv


def m_wrong_kv_head(O):
    orig = O.row_kv
    O.row_kv = lambda cache, page_row, L, g: orig(cache, page_row, L, (g + 1) % cache.shape[2])


def m_unnormalised_output(O):
    orig = O.attend

    def attend(q, K, V, active, scale):
        o, lse, s = orig(q, K, V, active, scale)
        return o * math.exp(0.0 if not np.isfinite(lse) else min(lse, 5.0) * 0.1), lse, s
    O.attend = attend


def m_tile_sum_without_max(O):
    def tile_stats(s, B):
        L = s.shape[0]
        nb = -(-L // B)
        m = np.array([s[b * B:min((b + 1) * B, L)].max() for b in range(nb)])
        l = np.array([np.exp(s[b * B:min((b + 1) * B, L)]).sum() for b in range(nb)])
        return m, l
    O.tile_stats = tile_stats


def m_masses_drop_partial_block(O):
    orig = O.block_masses

    def block_masses(s, lse, B):
        p = orig(s, lse, B)
        if s.shape[0] % B:
            p[-1] = 0.0
        return p
    O.block_masses = block_masses


def m_ties_to_higher_index(O):
    orig = O.select_blocks

    def select_blocks(p, eta):
        n = p.shape[0]
        rev = orig(p[::-1].copy(), eta)
        sel = rev["sel"][::-1].copy()
        return {**rev, "sel": sel, "order": n - 1 - rev["order"]}
    O.select_blocks = select_blocks


def m_strict_cutoff(O):
    def select_blocks(p, eta):
        n = p.shape[0]
        p32 = p.astype(np.float32).astype(np.float64)
        order = np.lexsort((np.arange(n), -p32))
        C = np.cumsum(p32[order])
        reach = np.nonzero(C > eta)[0]
        k = n if eta >= 1.0 else (int(reach[0]) + 1 if reach.size else n)
        sel = np.zeros(n, bool)
        sel[order[:k]] = True
        return {"sel": sel, "k": k, "order": order, "margin": 1.0, "gap": 1.0}
    O.select_blocks = select_blocks


def m_one_extra_block(O):
    orig = O.select_blocks

    def select_blocks(p, eta):
        res = orig(p, eta)
        k = min(res["k"] + 1, p.shape[0])
        sel = np.zeros(p.shape[0], bool)
        sel[res["order"][:k]] = True
        return {**res, "sel": sel, "k": k}
    O.select_blocks = select_blocks


def m_union_overwrites(O):
    O.support_union = lambda dst, src: np.asarray(src, np.uint32).copy()


def m_mask_ignored(O):
    O.mask_bits = lambda words, nb: np.ones(nb, dtype=bool)


def m_mask_bit_order_reversed(O):
    def mask_bits(words, nb):
        b = np.arange(nb)
        w = np.asarray(words, dtype=np.uint32)[b // 32]
        return ((w >> (31 - b % 32).astype(np.uint32)) & np.uint32(1)) == 1
    O.mask_bits = mask_bits


def m_compaction_drops_last_block(O):
    orig = O.compact_tiles

    def compact_tiles(support, modes, seq_lens, B):
        res = orig(support, modes, seq_lens, B)
        lists = [[lst[:-1] for lst in per] for per in res["lists"]]
        return {"lists": lists, "counts": np.maximum(res["counts"] - 1, 0)}
    O.compact_tiles = compact_tiles


def m_compaction_ignores_mode(O):
    orig = O.compact_tiles

    def compact_tiles(support, modes, seq_lens, B):
        return orig(support, np.full_like(np.asarray(modes), oracle_pins.MODE_SPARSE), seq_lens, B)
    O.compact_tiles = compact_tiles


def m_slot_ignored(O):
    """Rows index the pool by their row number instead of their slot."""
    orig = O.decode_layer_slots

    def decode_layer_slots(q, k, v, pt, sl, modes, pool, row_slot, layer, **kw):
        return orig(q, k, v, pt, sl, modes, pool, np.where(np.asarray(row_slot) >= 0,
                                                           np.arange(len(row_slot)), -1), layer, **kw)
    O.decode_layer_slots = decode_layer_slots


def m_slot_wrong_layer(O):
    orig = O.decode_layer_slots

    def decode_layer_slots(q, k, v, pt, sl, modes, pool, row_slot, layer, **kw):
        return orig(q, k, v, pt, sl, modes, pool, row_slot, (layer + 1) % pool.shape[1], **kw)
    O.decode_layer_slots = decode_layer_slots


def m_no_slot_reads_slot_zero(O):
    orig = O.decode_layer_slots

    def decode_layer_slots(q, k, v, pt, sl, modes, pool, row_slot, layer, **kw):
        return orig(q, k, v, pt, sl, modes, pool, np.maximum(np.asarray(row_slot), 0), layer, **kw)
    O.decode_layer_slots = decode_layer_slots


def m_head_union_skips_last_head(O):
    def support_head_union(support):
        sup = np.asarray(support, dtype=np.uint32)
        out = np.zeros_like(sup)
        acc = np.bitwise_or.reduce(sup[:, :-1], axis=1)
        out[:] = acc[:, None, :]
        return out
    O.support_head_union = support_head_union


MUTANTS = [m_scale_squared, m_slot_off_by_one, m_page_order_reversed, m_wrong_kv_head, m_unnormalised_output,
           m_tile_sum_without_max, m_masses_drop_partial_block, m_ties_to_higher_index,
           m_strict_cutoff, m_one_extra_block, m_union_overwrites, m_mask_ignored,
           m_mask_bit_order_reversed, m_compaction_drops_last_block,
           m_compaction_ignores_mode, m_head_union_skips_last_head, m_slot_ignored,
           m_slot_wrong_layer, m_no_slot_reads_slot_zero]


@pytest.mark.parametrize("mutate", MUTANTS, ids=lambda f: f.__name__)
def test_some_pin_catches_mutant(mutate):
    O = fresh_oracle()
    mutate(O)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            fails = pin(O)
        except Exception as e:  # a crash is also a catch
            fails = [repr(e)]
        if fails:
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutate.__name__}"
