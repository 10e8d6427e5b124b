"""Pins of the oracle's paged scatter, dequant and slot translation.

Paged addressing: "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats",
section 1 (PagedKV page / row / scale-row addressing), section 2
(kv_page_bytes), section 4 (dequant_k_cache.py: pages -> bf16 workspace).
Translation: "[sglang] Hoist DSv4 draft-extend SWA write locs", sections 1-2
(out[:n] = table[loc] as int32, out[n:] zeroed, n > capacity -> no buffer).
"""
import itertools

import numpy as np
import pytest

import oracle as O


def _address_model(layout, page_bits, slot):
    """Byte ranges of a slot's code row and scale row: a page is P code rows
    followed by P scale rows."""
    P = 1 << page_bits
    cb, sb = (512, 16) if layout == O.V41 else (256, 32)
    base = (slot // P) * P * (cb + sb)
    row = slot % P
    return (base + row * cb, cb), (base + P * cb + row * sb, sb)


@pytest.mark.parametrize("layout", [O.V41, O.FP4])
def test_store_bruteforce_tiny_pool(layout):
    page_bits, pages = 2, 2
    slots = pages << page_bits
    rng = np.random.default_rng(60)
    x = rng.standard_normal((3, 512)).astype(np.float32) * 4
    rows = [O.token_bytes(layout, 0, x[t]) for t in range(3)]
    nb = slots * O.bytes_per_token(layout)
    checked = 0
    for n in range(0, 4):
        for loc in itertools.permutations(range(slots), n):
            pool = np.zeros(nb, np.uint8)
            assert O.store(layout, page_bits, 0, x[:n], np.array(loc), pool) == O.OK
            model = np.zeros(nb, np.uint8)
            for t, slot in enumerate(loc):
                (co, cl), (so, sl) = _address_model(layout, page_bits, slot)
                model[co:co + cl] = rows[t][0]
                model[so:so + sl] = rows[t][1]
            assert (pool == model).all(), loc
            checked += 1
    assert checked == 1 + 8 + 56 + 336


@pytest.mark.parametrize("layout", [O.V41, O.FP4])
def test_compress_bruteforce_tiny_pool(layout):
    page_bits, slots, r = 2, 8, 2
    rng = np.random.default_rng(61)
    v = rng.standard_normal((3 * r, 512)).astype(np.float32)
    s = rng.standard_normal((3 * r, 512)).astype(np.float32)
    rows = [O.group_bytes(layout, r, 0, v[g * r:(g + 1) * r], s[g * r:(g + 1) * r]) for g in range(3)]
    nb = slots * O.bytes_per_token(layout)
    for loc in itertools.permutations(range(slots), 3):
        pool = np.zeros(nb, np.uint8)
        assert O.compress(layout, page_bits, r, 0, v, s, np.array(loc), pool) == O.OK
        model = np.zeros(nb, np.uint8)
        for g, slot in enumerate(loc):
            (co, cl), (so, sl) = _address_model(layout, page_bits, slot)
            model[co:co + cl] = rows[g][0]
            model[so:so + sl] = rows[g][1]
        assert (pool == model).all()


def test_store_out_of_range_slot_is_skipped():
    x = np.ones((2, 512), np.float32)
    pool = np.zeros(8 * 528, np.uint8)
    assert O.store(O.V41, 2, 0, x, np.array([8, 3]), pool) == O.ERANGE
    ref = np.zeros(8 * 528, np.uint8)
    O.store(O.V41, 2, 0, x[1:], np.array([3]), ref)
    assert (pool == ref).all()
    assert O.store(O.V41, 2, 0, x, np.array([-1, 3]), np.zeros(8 * 528, np.uint8)) == O.ERANGE


def _bf16_of(v):
    return O.bf16_bits(np.asarray(v, np.float32))


@pytest.mark.parametrize("layout", [O.V41, O.FP4])
def test_dequant_page_table_bruteforce(layout):
    page_bits, pages = 2, 4
    P = 1 << page_bits
    rng = np.random.default_rng(62)
    n = 10
    x = (rng.standard_t(3, (n, 512)) * 0.5).astype(np.float32)
    loc = rng.permutation(pages * P)[:n]
    pool = np.zeros(pages * P * O.bytes_per_token(layout), np.uint8)
    assert O.store(layout, page_bits, 0, x, loc, pool) == O.OK
    for pt in itertools.permutations(range(pages)):
        pt = np.array(pt, np.int32)
        rc, ws = O.dequant(layout, page_bits, pool, pt, pages * P)
        assert rc == O.OK
        for t in range(pages * P):
            slot = pt[t // P] * P + t % P
            hit = np.flatnonzero(loc == slot)
            if len(hit) == 0:
                assert (ws[t] == 0).all()
                continue
            codes, scales = O.token_bytes(layout, 0, x[hit[0]])
            if layout == O.V41:
                vals = O.e4m3_decode(codes) * np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32)
            else:
                nib = np.stack([codes & 0xF, codes >> 4], 1).reshape(-1)
                vals = O.e2m1_decode(nib) * np.repeat(O.e4m3_decode(scales[:16]), 32)
            assert (ws[t] == _bf16_of(vals)).all()


def test_dequant_rejects_ragged_and_bad_pages():
    pool = np.zeros(2 * 4 * 528, np.uint8)
    assert O.dequant(O.V41, 2, pool, np.array([0, 1], np.int32), 6)[0] == O.EINVAL
    assert O.dequant(O.V41, 2, pool, np.array([0, 2], np.int32), 8)[0] == O.ERANGE


def test_dequant_is_exact_inverse_on_code_grid():
    """Values already on a block's grid survive quant -> dequant exactly (V41)."""
    rng = np.random.default_rng(63)
    codes = rng.integers(0, 256, 512).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E
    vals = O.e4m3_decode(codes)
    for b in range(16):          # make each block's amax land in [256, 448]
        blk = vals[b * 32:(b + 1) * 32]
        blk[0] = 448.0 if b % 2 else 256.0
    y = (vals * 2.0 ** -20).astype(np.float32)
    pool = np.zeros(4 * 528, np.uint8)
    O.store(O.V41, 2, 0, y[None], np.array([1]), pool)
    rc, ws = O.dequant(O.V41, 2, pool, np.array([0], np.int32), 4)
    assert rc == O.OK
    assert (ws[1] == _bf16_of(y)).all()


def test_translate_bruteforce():
    rng = np.random.default_rng(64)
    table = rng.integers(0, 1 << 10, 1 << 12).astype(np.int32)
    for n, cap in [(0, 0), (0, 5), (7, 7), (100, 300), (1000, 1000)]:
        loc = rng.integers(0, 1 << 12, n)
        rc, out = O.translate(loc, table, cap)
        assert rc == O.OK
        for i in range(n):
            assert out[i] == table[loc[i]]
        assert (out[n:] == 0).all() and out.dtype == np.int32


def test_translate_capacity_and_range():
    table = np.arange(16, dtype=np.int32) * 3
    rc, out = O.translate(np.arange(5), table, 4)
    assert rc == O.ECAP and (out == 0x7EEEEEEE).all()       # nothing written
    rc, out = O.translate(np.array([1, 16, -1, 2]), table, 6)
    assert rc == O.ERANGE
    assert list(out) == [3, -1, -1, 6, 0, 0]


@pytest.mark.parametrize("layout", [O.V41, O.FP4])
def test_dequant_slots_equals_paged_rows(layout):
    """Selected-slot dequant returns exactly the rows the paged dequant gives
    for those slots (identity page table); -1 is a zero row."""
    page_bits, pages = 2, 8
    P = 1 << page_bits
    rng = np.random.default_rng(65)
    x = (rng.standard_t(3, (20, 512)) * 0.5).astype(np.float32)
    loc = rng.permutation(pages * P)[:20]
    pool = np.zeros(pages * P * O.bytes_per_token(layout), np.uint8)
    assert O.store(layout, page_bits, 0, x, loc, pool) == O.OK
    rc, full = O.dequant(layout, page_bits, pool, np.arange(pages, dtype=np.int32), pages * P)
    assert rc == O.OK
    for slots in (np.arange(pages * P), rng.permutation(pages * P)[:11], np.array([5, -1, 5, 0])):
        rc, got = O.dequant_slots(layout, pool, slots, page_bits)
        assert rc == O.OK
        for i, s in enumerate(slots):
            assert (got[i] == (0 if s == -1 else full[s])).all()


def test_dequant_slots_range_rule():
    pool = np.zeros(8 * 528, np.uint8)
    rc, got = O.dequant_slots(O.V41, pool, np.array([1, 8, -2]), 2)
    assert rc == O.ERANGE
    assert (got[0] == 0).all() and (got[1:] == 0xBEEF).all()
