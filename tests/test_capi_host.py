"""The C ABI without a GPU: the library loads, exports every entry point that
include/kvq.h declares, reports the layout sizes, and rejects bad arguments
on the host before anything is launched (no call here reaches a launch)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from compress_kv_write_gb300 import build
    build.build()
    from compress_kv_write_gb300 import kvq
    return kvq.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert {"kvq_store", "kvq_compress", "kvq_dequant", "kvq_translate_loc"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_sizes(L):
    assert L.kvq_bytes_per_token(1) == 528
    assert L.kvq_bytes_per_token(2) == 288
    assert L.kvq_bytes_per_token(3) == 0
    assert L.kvq_page_bytes(1, 6) == 33792
    assert L.kvq_page_bytes(2, 6) == 18432
    assert L.kvq_page_bytes(1, 0) == 0
    assert L.kvq_page_bits_supported(6) == 1 and L.kvq_page_bits_supported(5) == 0
    assert L.kvq_status_string(3) == b"n exceeds the output capacity"


A = 0x10000          # a 16-byte aligned fake device address (never dereferenced)


def _store(L, layout=1, page_bits=6, flags=0, x=A, x_dtype=1, n=4, stride=512, loc=A, loc_dtype=0,
           w=None, cs=None, rows=0, pos=None, pool=A, slots=64):
    return L.kvq_store(layout, page_bits, flags, x, x_dtype, n, stride, loc, loc_dtype, w, 1e-6,
                       cs, rows, pos, pool, slots, None, None)


def test_store_rejects_on_host(L):
    assert _store(L, layout=0) == 1
    assert _store(L, layout=3) == 1
    assert _store(L, page_bits=0) == 1
    assert _store(L, page_bits=17) == 1
    assert _store(L, page_bits=5) == 2          # valid, not compiled
    assert _store(L, flags=4) == 1
    assert _store(L, x=None) == 1
    assert _store(L, x=A + 4) == 1               # misaligned rows
    assert _store(L, stride=511) == 1
    assert _store(L, stride=516, x_dtype=1) == 1  # 1032 B rows: not 16-B aligned
    assert _store(L, x_dtype=2) == 1
    assert _store(L, loc=None) == 1
    assert _store(L, loc_dtype=2) == 1
    assert _store(L, pool=None) == 1
    assert _store(L, slots=65) == 1              # not whole pages
    assert _store(L, n=-1) == 1
    assert _store(L, flags=2) == 1               # norm without weight
    assert _store(L, flags=1, cs=A, rows=0, pos=A) == 1
    assert _store(L, flags=1, cs=A, rows=8, pos=None) == 1
    assert _store(L, n=0) == 0                   # nothing to do: no launch
    assert _store(L, n=0, x=None, loc=None) == 0  # empty inputs may be null


def test_compress_rejects_on_host(L):
    def c(ratio=4, flags=0, v=A, s=A, n=8, loc=A, pool=A, slots=64, layout=1):
        return L.kvq_compress(layout, 6, ratio, flags, v, s, n, None, 0, None, loc, pool, slots,
                              None, None)
    assert c(ratio=3) == 2
    assert c(ratio=0) == 1
    assert c(flags=2) == 2
    assert c(flags=1) == 1                       # RoPE without a table
    assert c(v=None) == 1
    assert c(s=A + 8) == 1
    assert c(loc=A + 2) == 1
    assert c(layout=9) == 1
    assert c(n=0) == 0


def test_dequant_rejects_on_host(L):
    def d(n=128, pages=2, pt=A, out=A, stride=512, page_bits=6):
        return L.kvq_dequant(1, page_bits, A, pages, pt, n, out, stride, None, None)
    assert d(n=100) == 1                          # not whole pages
    assert d(pages=0) == 1
    assert d(pt=None) == 1
    assert d(out=A + 2) == 1
    assert d(stride=500) == 1
    assert d(page_bits=5) == 2
    assert d(n=0) == 0


def test_translate_rejects_on_host(L):
    assert L.kvq_translate_loc(A, 1, 10, A, 100, A, 9, None, None) == 3    # capacity
    assert L.kvq_translate_loc(A, 2, 1, A, 100, A, 9, None, None) == 1
    assert L.kvq_translate_loc(None, 1, 4, A, 100, A, 9, None, None) == 1
    assert L.kvq_translate_loc(A + 4, 1, 4, A, 100, A, 9, None, None) == 1  # int64 misaligned
    assert L.kvq_translate_loc(A, 0, 0, A, 100, A, 0, None, None) == 0


def test_dequant_slots_rejects_on_host(L):
    def d(layout=1, page_bits=6, pool=A, slots_n=64, idx=A, dt=0, n=4, out=A, stride=512):
        return L.kvq_dequant_slots(layout, page_bits, pool, slots_n, idx, dt, n, out, stride, None, None)
    assert d(layout=5) == 1
    assert d(page_bits=3) == 2
    assert d(pool=A + 8) == 1
    assert d(slots_n=65) == 1
    assert d(dt=3) == 1
    assert d(idx=None) == 1
    assert d(idx=A + 4, dt=1) == 1
    assert d(out=A + 8) == 1
    assert d(stride=256) == 1
    assert d(n=-1) == 1
    assert d(n=0, idx=None, out=None) == 0


def test_compress_decode_rejects_on_host(L):
    def c(ratio=4, flags=0, v=A, s=A, n=8, state=A, count=A, req=None, n_state=8, loc=A, layout=1):
        return L.kvq_compress_decode(layout, 6, ratio, flags, v, s, n, state, count, req, n_state,
                                     None, 0, None, loc, A, 64, None, None)
    assert c(ratio=3) == 2
    assert c(ratio=0) == 1
    assert c(flags=2) == 2
    assert c(flags=1) == 1                 # RoPE without a table
    assert c(state=None) == 1
    assert c(state=A + 4) == 1
    assert c(count=None) == 1
    assert c(n=9, req=None, n_state=8) == 1  # more requests than state rows, no index
    assert c(loc=None) == 1
    assert c(n_state=0) == 1
    assert c(n=0) == 0
