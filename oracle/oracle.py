"""ctypes + numpy wrapper of the C oracle (test infrastructure only).

Every array argument is a numpy array; bf16 data travels as its uint16 bit
pattern.  The functions mirror ``kvq_oracle.h``; each C function cites the
page passage it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import tempfile

import numpy as np

__all__ = [
    "V41", "FP4", "F32", "BF16", "ROPE", "NORM", "OK", "EINVAL", "ECAP", "ERANGE",
    "e4m3_encode", "e4m3_decode", "e2m1_encode", "e2m1_decode", "bf16_bits",
    "bf16_round", "bf16_to_f32", "code_bytes", "scale_bytes", "bytes_per_token",
    "page_bytes", "encode_v41", "encode_fp4", "rmsnorm", "rope", "pool",
    "token_prequant", "group_prequant", "token_bytes", "group_bytes", "store",
    "compress", "dequant", "dequant_slots", "translate",
]

V41, FP4 = 1, 2
F32, BF16 = 0, 1
ROPE, NORM = 1, 2
OK, EINVAL, ECAP, ERANGE = 0, 1, 3, 5
D = 512

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_SO = os.path.join(_HERE, "_build", "libkvq_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction) into oracle/_build/."""
    srcs = [_SRC, os.path.join(_HERE, "kvq_oracle.h")]
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= max(os.path.getmtime(s) for s in srcs)):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(_SO))
    os.close(fd)
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _p(t):
    return C.POINTER(t)


_SIGS = {
    "or_e4m3_encode_n": (None, [_p(C.c_float), _p(C.c_uint8), C.c_int64]),
    "or_e4m3_decode_n": (None, [_p(C.c_uint8), _p(C.c_double), C.c_int64]),
    "or_e2m1_encode_n": (None, [_p(C.c_float), _p(C.c_uint8), C.c_int64]),
    "or_e2m1_decode_n": (None, [_p(C.c_uint8), _p(C.c_double), C.c_int64]),
    "or_bf16_bits_n": (None, [_p(C.c_float), _p(C.c_uint16), C.c_int64]),
    "or_code_bytes": (C.c_size_t, [C.c_int]),
    "or_scale_bytes": (C.c_size_t, [C.c_int]),
    "or_bytes_per_token": (C.c_size_t, [C.c_int]),
    "or_page_bytes": (C.c_size_t, [C.c_int, C.c_int]),
    "or_encode_v41": (None, [_p(C.c_float), _p(C.c_uint8), _p(C.c_uint8)]),
    "or_encode_fp4": (None, [_p(C.c_float), _p(C.c_uint8), _p(C.c_uint8)]),
    "or_rmsnorm": (None, [_p(C.c_float), _p(C.c_float), C.c_float]),
    "or_rope": (None, [_p(C.c_float), _p(C.c_float)]),
    "or_pool": (None, [_p(C.c_float), _p(C.c_float), C.c_int, _p(C.c_float)]),
    "or_token_prequant": (C.c_int, [C.c_uint, C.c_void_p, C.c_int, _p(C.c_float),
                                    C.c_float, _p(C.c_float), _p(C.c_float)]),
    "or_group_prequant": (C.c_int, [C.c_int, C.c_uint, _p(C.c_float), _p(C.c_float),
                                    _p(C.c_float), _p(C.c_float)]),
    "or_token_bytes": (C.c_int, [C.c_int, C.c_uint, C.c_void_p, C.c_int, _p(C.c_float),
                                 C.c_float, _p(C.c_float), _p(C.c_uint8), _p(C.c_uint8)]),
    "or_group_bytes": (C.c_int, [C.c_int, C.c_int, C.c_uint, _p(C.c_float), _p(C.c_float),
                                 _p(C.c_float), _p(C.c_uint8), _p(C.c_uint8)]),
    "or_store": (C.c_int, [C.c_int, C.c_int, C.c_uint, C.c_void_p, C.c_int, C.c_int64,
                           C.c_int64, _p(C.c_int64), _p(C.c_float), C.c_float,
                           _p(C.c_float), C.c_int64, _p(C.c_int32), _p(C.c_uint8),
                           C.c_int64]),
    "or_compress": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_uint, _p(C.c_float),
                              _p(C.c_float), C.c_int64, _p(C.c_float), C.c_int64,
                              _p(C.c_int32), _p(C.c_int64), _p(C.c_uint8), C.c_int64]),
    "or_dequant": (C.c_int, [C.c_int, C.c_int, _p(C.c_uint8), C.c_int64, _p(C.c_int32),
                             C.c_int64, _p(C.c_uint16), C.c_int64]),
    "or_dequant_slots": (C.c_int, [C.c_int, C.c_int, _p(C.c_uint8), C.c_int64, _p(C.c_int64),
                                   C.c_int64, _p(C.c_uint16), C.c_int64]),
    "or_translate": (C.c_int, [_p(C.c_int64), C.c_int64, _p(C.c_int32), C.c_int64,
                               _p(C.c_int32), C.c_int64]),
}


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    if _lib is None:
        so = build()
        L = C.CDLL(so)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ---------------------------------------------------------------- helpers

def _arr(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(C.POINTER(ctype))


def _x_dtype(x):
    if x.dtype == np.float32:
        return F32
    if x.dtype in (np.uint16, np.int16):
        return BF16
    raise TypeError("x must be float32 or bf16 bits (uint16)")


# ---------------------------------------------------------------- formats

def e4m3_encode(x):
    x = _arr(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().or_e4m3_encode_n(_ptr(x, C.c_float), _ptr(out, C.c_uint8), x.size)
    return out


def e4m3_decode(c):
    c = _arr(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().or_e4m3_decode_n(_ptr(c, C.c_uint8), _ptr(out, C.c_double), c.size)
    return out


def e2m1_encode(x):
    x = _arr(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().or_e2m1_encode_n(_ptr(x, C.c_float), _ptr(out, C.c_uint8), x.size)
    return out


def e2m1_decode(c):
    c = _arr(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().or_e2m1_decode_n(_ptr(c, C.c_uint8), _ptr(out, C.c_double), c.size)
    return out


def bf16_bits(x):
    x = _arr(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().or_bf16_bits_n(_ptr(x, C.c_float), _ptr(out, C.c_uint16), x.size)
    return out


def bf16_to_f32(b):
    b = _arr(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_round(x):
    return bf16_to_f32(bf16_bits(x))


# ---------------------------------------------------------------- sizes

def code_bytes(layout):
    return int(lib().or_code_bytes(layout))


def scale_bytes(layout):
    return int(lib().or_scale_bytes(layout))


def bytes_per_token(layout):
    return int(lib().or_bytes_per_token(layout))


def page_bytes(layout, page_bits):
    return int(lib().or_page_bytes(layout, page_bits))


# ---------------------------------------------------------------- rows

def encode_v41(y):
    y = _arr(y, np.float32)
    assert y.shape == (D,)
    codes = np.empty(512, np.uint8)
    scales = np.empty(16, np.uint8)
    lib().or_encode_v41(_ptr(y, C.c_float), _ptr(codes, C.c_uint8), _ptr(scales, C.c_uint8))
    return codes, scales


def encode_fp4(y):
    y = _arr(y, np.float32)
    assert y.shape == (D,)
    codes = np.empty(256, np.uint8)
    scales = np.empty(32, np.uint8)
    lib().or_encode_fp4(_ptr(y, C.c_float), _ptr(codes, C.c_uint8), _ptr(scales, C.c_uint8))
    return codes, scales


def rmsnorm(y, w, eps):
    y = np.array(y, dtype=np.float32, copy=True)
    w = _arr(w, np.float32)
    lib().or_rmsnorm(_ptr(y, C.c_float), _ptr(w, C.c_float), eps)
    return y


def rope(y, cs_row):
    y = np.array(y, dtype=np.float32, copy=True)
    cs = _arr(cs_row, np.float32)
    assert cs.shape == (64,)
    lib().or_rope(_ptr(y, C.c_float), _ptr(cs, C.c_float))
    return y


def pool(v, s):
    v = _arr(v, np.float32)
    s = _arr(s, np.float32)
    r = v.shape[0]
    assert v.shape == (r, D) and s.shape == (r, D)
    out = np.empty(D, np.float32)
    lib().or_pool(_ptr(v, C.c_float), _ptr(s, C.c_float), r, _ptr(out, C.c_float))
    return out


def token_prequant(flags, x_row, norm_weight=None, eps=1e-6, cs_row=None):
    x_row = np.ascontiguousarray(x_row)
    y = np.empty(D, np.float32)
    w = None if norm_weight is None else _arr(norm_weight, np.float32)
    cs = None if cs_row is None else _arr(cs_row, np.float32)
    rc = lib().or_token_prequant(flags, x_row.ctypes.data, _x_dtype(x_row), _ptr(w, C.c_float),
                                 eps, _ptr(cs, C.c_float), _ptr(y, C.c_float))
    assert rc == OK, rc
    return y


def group_prequant(ratio, flags, values, scores, cs_row=None):
    v = _arr(values, np.float32)
    s = _arr(scores, np.float32)
    cs = None if cs_row is None else _arr(cs_row, np.float32)
    y = np.empty(D, np.float32)
    rc = lib().or_group_prequant(ratio, flags, _ptr(v, C.c_float), _ptr(s, C.c_float),
                                 _ptr(cs, C.c_float), _ptr(y, C.c_float))
    assert rc == OK, rc
    return y


def token_bytes(layout, flags, x_row, norm_weight=None, eps=1e-6, cs_row=None):
    """(codes, scale row) one token occupies."""
    x_row = np.ascontiguousarray(x_row)
    codes = np.zeros(512, np.uint8)
    scales = np.zeros(32, np.uint8)
    w = None if norm_weight is None else _arr(norm_weight, np.float32)
    cs = None if cs_row is None else _arr(cs_row, np.float32)
    rc = lib().or_token_bytes(layout, flags, x_row.ctypes.data, _x_dtype(x_row),
                              _ptr(w, C.c_float), eps, _ptr(cs, C.c_float),
                              _ptr(codes, C.c_uint8), _ptr(scales, C.c_uint8))
    assert rc == OK, rc
    return codes[:code_bytes(layout)], scales[:scale_bytes(layout)]


def group_bytes(layout, ratio, flags, values, scores, cs_row=None):
    v = _arr(values, np.float32)
    s = _arr(scores, np.float32)
    cs = None if cs_row is None else _arr(cs_row, np.float32)
    codes = np.zeros(512, np.uint8)
    scales = np.zeros(32, np.uint8)
    rc = lib().or_group_bytes(layout, ratio, flags, _ptr(v, C.c_float), _ptr(s, C.c_float),
                              _ptr(cs, C.c_float), _ptr(codes, C.c_uint8),
                              _ptr(scales, C.c_uint8))
    assert rc == OK, rc
    return codes[:code_bytes(layout)], scales[:scale_bytes(layout)]


# ---------------------------------------------------------------- whole calls

def store(layout, page_bits, flags, x, loc, pool_bytes, norm_weight=None, eps=1e-6,
          cos_sin=None, pos=None):
    """Quantise rows of x [n, 512] and scatter them into pool_bytes (uint8, in place).
    Returns the oracle status."""
    x = np.ascontiguousarray(x)
    assert x.ndim == 2 and x.shape[1] == D
    loc = _arr(loc, np.int64)
    assert pool_bytes.dtype == np.uint8 and pool_bytes.flags.c_contiguous
    slots = pool_bytes.size // bytes_per_token(layout)
    w = None if norm_weight is None else _arr(norm_weight, np.float32)
    cs = None if cos_sin is None else _arr(cos_sin, np.float32)
    ps = None if pos is None else _arr(pos, np.int32)
    rows = 0 if cs is None else cs.shape[0]
    return lib().or_store(layout, page_bits, flags, x.ctypes.data, _x_dtype(x), x.shape[0],
                          x.shape[1], _ptr(loc, C.c_int64), _ptr(w, C.c_float), eps,
                          _ptr(cs, C.c_float), rows, _ptr(ps, C.c_int32),
                          _ptr(pool_bytes, C.c_uint8), slots)


def compress(layout, page_bits, ratio, flags, values, scores, loc, pool_bytes,
             cos_sin=None, group_pos=None):
    v = _arr(values, np.float32)
    s = _arr(scores, np.float32)
    assert v.shape == s.shape and v.shape[1] == D and v.shape[0] % ratio == 0
    n_groups = v.shape[0] // ratio
    loc = _arr(loc, np.int64)
    slots = pool_bytes.size // bytes_per_token(layout)
    cs = None if cos_sin is None else _arr(cos_sin, np.float32)
    gp = None if group_pos is None else _arr(group_pos, np.int32)
    rows = 0 if cs is None else cs.shape[0]
    return lib().or_compress(layout, page_bits, ratio, flags, _ptr(v, C.c_float),
                             _ptr(s, C.c_float), n_groups, _ptr(cs, C.c_float), rows,
                             _ptr(gp, C.c_int32), _ptr(loc, C.c_int64),
                             _ptr(pool_bytes, C.c_uint8), slots)


def dequant(layout, page_bits, pool_bytes, page_table, n_tokens):
    """Returns (status, bf16 bits uint16 [n_tokens, 512])."""
    pb = page_bytes(layout, page_bits)
    pool_pages = pool_bytes.size // pb
    pt = _arr(page_table, np.int32)
    out = np.zeros((n_tokens, D), np.uint16)
    rc = lib().or_dequant(layout, page_bits, _ptr(pool_bytes, C.c_uint8), pool_pages,
                          _ptr(pt, C.c_int32), n_tokens, _ptr(out, C.c_uint16), D)
    return rc, out


def dequant_slots(layout, pool_bytes, slots, page_bits=6, out=None):
    """Returns (status, bf16 bits uint16 [n, 512]) of the tokens in `slots`."""
    slots = _arr(slots, np.int64)
    pool_slots = pool_bytes.size // bytes_per_token(layout)
    if out is None:
        out = np.full((slots.size, D), 0xBEEF, np.uint16)
    rc = lib().or_dequant_slots(layout, page_bits, _ptr(pool_bytes, C.c_uint8), pool_slots,
                                _ptr(slots, C.c_int64), slots.size, _ptr(out, C.c_uint16), D)
    return rc, out


def translate(loc, full_to_swa, capacity):
    """Returns (status, int32 [capacity])."""
    loc = _arr(loc, np.int64)
    tab = _arr(full_to_swa, np.int32)
    out = np.full(capacity, 0x7EEEEEEE, np.int32)
    rc = lib().or_translate(_ptr(loc, C.c_int64), loc.size, _ptr(tab, C.c_int32), tab.size,
                            _ptr(out, C.c_int32), capacity)
    return rc, out
