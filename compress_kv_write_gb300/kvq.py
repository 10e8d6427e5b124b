"""Thin Python binding of libkvq.so (include/kvq.h): argument marshalling only.

Every function takes torch CUDA tensors, checks dtype / shape / device, and
passes raw device pointers and the current CUDA stream to the C entry point
of the same name.  All compute runs in the library's kernels; there is no
CPU path.  A missing library raises ImportError.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

V41, V41_FP4 = 1, 2
F32, BF16 = 0, 1
I32, I64 = 0, 1
FLAG_ROPE, FLAG_NORM = 1, 2
DEVERR_SLOT, DEVERR_POS, DEVERR_PAGE, DEVERR_LOC, DEVERR_STATE = 1, 2, 4, 8, 32
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CAPACITY, ERR_LAUNCH = 0, 1, 2, 3, 4
HEAD_DIM = 512

_lib = None


class KVQError(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


_SIGS = {
    "kvq_bytes_per_token": (C.c_size_t, [C.c_int]),
    "kvq_page_bytes": (C.c_size_t, [C.c_int, C.c_int]),
    "kvq_page_bits_supported": (C.c_int, [C.c_int]),
    "kvq_status_string": (C.c_char_p, [C.c_int]),
    "kvq_translate_loc": (C.c_int, [C.c_void_p, C.c_int, C.c_int64, C.c_void_p, C.c_int64,
                                    C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p]),
    "kvq_store": (C.c_int, [C.c_int, C.c_int, C.c_uint, C.c_void_p, C.c_int, C.c_int64,
                            C.c_int64, C.c_void_p, C.c_int, C.c_void_p, C.c_float, C.c_void_p,
                            C.c_int64, C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p,
                            C.c_void_p]),
    "kvq_compress": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_uint, C.c_void_p, C.c_void_p,
                               C.c_int64, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                               C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p]),
    "kvq_compress_decode": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_uint, C.c_void_p, C.c_void_p,
                                      C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64,
                                      C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_int64, C.c_void_p, C.c_void_p]),
    "kvq_dequant_slots": (C.c_int, [C.c_int, C.c_int, C.c_void_p, C.c_int64, C.c_void_p, C.c_int,
                                    C.c_int64, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p]),
    "kvq_dequant": (C.c_int, [C.c_int, C.c_int, C.c_void_p, C.c_int64, C.c_void_p, C.c_int64,
                              C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p]),
}


def library_path() -> str:
    return _build.SO


def lib():
    """The loaded libkvq.so.  Raises ImportError when it has not been built."""
    global _lib
    if _lib is None:
        path = _build.SO
        if not os.path.exists(path):
            raise ImportError(f"libkvq.so is not built ({path}); run compress_kv_write_gb300.build.build()")
        L = C.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kvq_status_string(status).decode()


def bytes_per_token(layout: int) -> int:
    return int(lib().kvq_bytes_per_token(layout))


def page_bytes(layout: int, page_bits: int) -> int:
    return int(lib().kvq_page_bytes(layout, page_bits))


def page_bits_supported(page_bits: int) -> bool:
    return bool(lib().kvq_page_bits_supported(page_bits))


# ------------------------------------------------------------------ helpers

def _check(status: int, fn: str):
    if status != OK:
        raise KVQError(status, fn)


def _cuda(t, name, dtypes=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    return t


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _idx_dtype(t, name):
    if t.dtype == torch.int32:
        return I32
    if t.dtype == torch.int64:
        return I64
    raise TypeError(f"{name} must be int32 or int64")


def _contig1d(t, name):
    if t.dim() != 1 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 1-D tensor")


# ------------------------------------------------------------------ entry points

def kvq_translate_loc(full_loc, full_to_swa, out, n=None, err=None, stream=None):
    """out[:n] = full_to_swa[full_loc] (int32), out[n:] = 0; once per step.
    Raises KVQError(ERR_CAPACITY) when n > out.numel()."""
    _cuda(full_loc, "full_loc")
    _cuda(full_to_swa, "full_to_swa", (torch.int32,))
    _cuda(out, "out", (torch.int32,))
    for t, nm in ((full_loc, "full_loc"), (full_to_swa, "full_to_swa"), (out, "out")):
        _contig1d(t, nm)
    n = full_loc.numel() if n is None else int(n)
    st = lib().kvq_translate_loc(_ptr(full_loc), _idx_dtype(full_loc, "full_loc"), n,
                                 _ptr(full_to_swa), full_to_swa.numel(), _ptr(out), out.numel(),
                                 _ptr(err), _stream(stream))
    _check(st, "kvq_translate_loc")
    return out


def kvq_store(layout, page_bits, flags, x, loc, pool, pool_slots, *, norm_weight=None,
              eps=1e-6, cos_sin=None, pos=None, err=None, stream=None):
    """Quantise rows x [n, >=512] (fp32 / bf16) into slots loc of the paged pool."""
    _cuda(x, "x", (torch.float32, torch.bfloat16))
    _cuda(loc, "loc")
    _cuda(pool, "pool", (torch.uint8,))
    if x.dim() != 2 or x.shape[1] < HEAD_DIM or x.stride(1) != 1:
        raise ValueError("x must be [n, >=512] with unit inner stride")
    _contig1d(loc, "loc")
    if loc.numel() != x.shape[0]:
        raise ValueError("loc must hold one slot per row")
    if pool.numel() < pool_slots * bytes_per_token(layout):
        raise ValueError("pool is smaller than pool_slots tokens")
    if norm_weight is not None:
        _cuda(norm_weight, "norm_weight", (torch.float32,))
        if norm_weight.numel() != HEAD_DIM or not norm_weight.is_contiguous():
            raise ValueError("norm_weight must be contiguous [512]")
    rows = 0
    if cos_sin is not None:
        _cuda(cos_sin, "cos_sin", (torch.float32,))
        if cos_sin.dim() != 2 or cos_sin.shape[1] != 64 or not cos_sin.is_contiguous():
            raise ValueError("cos_sin must be contiguous [rows, 64]")
        rows = cos_sin.shape[0]
    if pos is not None:
        _cuda(pos, "pos", (torch.int32,))
        _contig1d(pos, "pos")
        if pos.numel() != x.shape[0]:
            raise ValueError("pos must hold one position per row")
    st = lib().kvq_store(layout, page_bits, flags, _ptr(x), BF16 if x.dtype == torch.bfloat16 else F32,
                         x.shape[0], x.stride(0), _ptr(loc), _idx_dtype(loc, "loc"),
                         _ptr(norm_weight), float(eps), _ptr(cos_sin), rows, _ptr(pos), _ptr(pool),
                         int(pool_slots), _ptr(err), _stream(stream))
    _check(st, "kvq_store")


def kvq_compress(layout, page_bits, ratio, flags, values, scores, loc, pool, pool_slots, *,
                 cos_sin=None, group_pos=None, err=None, stream=None):
    """Softmax-pool groups of `ratio` rows of values/scores [n*ratio, 512] fp32
    and store the result of group g into slot loc[g]."""
    _cuda(values, "values", (torch.float32,))
    _cuda(scores, "scores", (torch.float32,))
    _cuda(loc, "loc", (torch.int32,))
    _cuda(pool, "pool", (torch.uint8,))
    if values.shape != scores.shape or values.dim() != 2 or values.shape[1] != HEAD_DIM:
        raise ValueError("values and scores must both be [n*ratio, 512]")
    if not values.is_contiguous() or not scores.is_contiguous():
        raise ValueError("values and scores must be contiguous")
    if values.shape[0] % ratio:
        raise ValueError("rows must be a multiple of ratio")
    n_groups = values.shape[0] // ratio
    _contig1d(loc, "loc")
    if loc.numel() != n_groups:
        raise ValueError("loc must hold one slot per group")
    if pool.numel() < pool_slots * bytes_per_token(layout):
        raise ValueError("pool is smaller than pool_slots tokens")
    rows = 0
    if cos_sin is not None:
        _cuda(cos_sin, "cos_sin", (torch.float32,))
        if cos_sin.dim() != 2 or cos_sin.shape[1] != 64 or not cos_sin.is_contiguous():
            raise ValueError("cos_sin must be contiguous [rows, 64]")
        rows = cos_sin.shape[0]
    if group_pos is not None:
        _cuda(group_pos, "group_pos", (torch.int32,))
        _contig1d(group_pos, "group_pos")
        if group_pos.numel() != n_groups:
            raise ValueError("group_pos must hold one position per group")
    st = lib().kvq_compress(layout, page_bits, ratio, flags, _ptr(values), _ptr(scores), n_groups,
                            _ptr(cos_sin), rows, _ptr(group_pos), _ptr(loc), _ptr(pool),
                            int(pool_slots), _ptr(err), _stream(stream))
    _check(st, "kvq_compress")


def kvq_dequant(layout, page_bits, pool, pool_pages, page_table, out, err=None, stream=None):
    """out [n_tokens, >=512] bf16 <- pages page_table[t >> page_bits] of pool."""
    _cuda(pool, "pool", (torch.uint8,))
    _cuda(page_table, "page_table", (torch.int32,))
    _cuda(out, "out", (torch.bfloat16,))
    _contig1d(page_table, "page_table")
    if out.dim() != 2 or out.shape[1] < HEAD_DIM or out.stride(1) != 1:
        raise ValueError("out must be [n_tokens, >=512] bf16 with unit inner stride")
    n_tokens = out.shape[0]
    if page_table.numel() * (1 << page_bits) != n_tokens:
        raise ValueError("out must have page_table.numel() * 2^page_bits rows")
    if pool.numel() < pool_pages * page_bytes(layout, page_bits):
        raise ValueError("pool is smaller than pool_pages pages")
    st = lib().kvq_dequant(layout, page_bits, _ptr(pool), int(pool_pages), _ptr(page_table),
                           n_tokens, _ptr(out), out.stride(0), _ptr(err), _stream(stream))
    _check(st, "kvq_dequant")


def kvq_dequant_slots(layout, page_bits, pool, pool_slots, slots, out, err=None, stream=None):
    """out [n, >=512] bf16 <- the tokens in slots [n] (int32/int64); slot -1 gives a zero row."""
    _cuda(pool, "pool", (torch.uint8,))
    _cuda(slots, "slots")
    _cuda(out, "out", (torch.bfloat16,))
    _contig1d(slots, "slots")
    if out.dim() != 2 or out.shape[1] < HEAD_DIM or out.stride(1) != 1 or out.shape[0] != slots.numel():
        raise ValueError("out must be [slots.numel(), >=512] bf16 with unit inner stride")
    if pool.numel() < pool_slots * bytes_per_token(layout):
        raise ValueError("pool is smaller than pool_slots tokens")
    st = lib().kvq_dequant_slots(layout, page_bits, _ptr(pool), int(pool_slots), _ptr(slots),
                                 _idx_dtype(slots, "slots"), slots.numel(), _ptr(out), out.stride(0),
                                 _ptr(err), _stream(stream))
    _check(st, "kvq_dequant_slots")


def kvq_compress_decode(layout, page_bits, ratio, flags, values, scores, state, count, loc, pool,
                        pool_slots, *, req=None, cos_sin=None, group_pos=None, err=None, stream=None):
    """One decode step of the ratio-r compressor: request i appends row
    (values[i], scores[i]) to the open group held in state[req[i]] /
    count[req[i]]; a group's ratio-th row pools, quantises and stores it into
    slot loc[i]."""
    _cuda(values, "values", (torch.float32,))
    _cuda(scores, "scores", (torch.float32,))
    _cuda(state, "state", (torch.float32,))
    _cuda(count, "count", (torch.int32,))
    _cuda(loc, "loc", (torch.int32,))
    _cuda(pool, "pool", (torch.uint8,))
    if values.shape != scores.shape or values.dim() != 2 or values.shape[1] != HEAD_DIM:
        raise ValueError("values and scores must both be [n, 512]")
    if not values.is_contiguous() or not scores.is_contiguous():
        raise ValueError("values and scores must be contiguous")
    n = values.shape[0]
    if state.dim() != 3 or state.shape[1:] != (3, HEAD_DIM) or not state.is_contiguous():
        raise ValueError("state must be contiguous [n_state, 3, 512]")
    _contig1d(count, "count")
    if count.numel() != state.shape[0]:
        raise ValueError("count must hold one entry per state row")
    _contig1d(loc, "loc")
    if loc.numel() != n:
        raise ValueError("loc must hold one slot per request")
    if req is not None:
        _cuda(req, "req", (torch.int32,))
        _contig1d(req, "req")
        if req.numel() != n:
            raise ValueError("req must hold one state index per request")
    if pool.numel() < pool_slots * bytes_per_token(layout):
        raise ValueError("pool is smaller than pool_slots tokens")
    rows = 0
    if cos_sin is not None:
        _cuda(cos_sin, "cos_sin", (torch.float32,))
        if cos_sin.dim() != 2 or cos_sin.shape[1] != 64 or not cos_sin.is_contiguous():
            raise ValueError("cos_sin must be contiguous [rows, 64]")
        rows = cos_sin.shape[0]
    if group_pos is not None:
        _cuda(group_pos, "group_pos", (torch.int32,))
        _contig1d(group_pos, "group_pos")
        if group_pos.numel() != n:
            raise ValueError("group_pos must hold one position per request")
    st = lib().kvq_compress_decode(layout, page_bits, ratio, flags, _ptr(values), _ptr(scores), n,
                                   _ptr(state), _ptr(count), _ptr(req), state.shape[0], _ptr(cos_sin),
                                   rows, _ptr(group_pos), _ptr(loc), _ptr(pool), int(pool_slots),
                                   _ptr(err), _stream(stream))
    _check(st, "kvq_compress_decode")
