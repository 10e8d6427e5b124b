"""Comparison rules between the CUDA path and the oracle (test helpers).

Bit-exact paths (plain store, scatter, translation, dequant): bytes equal.
Paths with fp32 math before the quantiser (RMSNorm, softmax pooling): codes
may differ by at most one quantisation step on at most 0.1% of the elements,
and each dequantised GPU value may be off the oracle's pre-quantisation fp32
value by at most the oracle's own quantisation error plus one grid step at
that magnitude times the block scale.
"""
import concurrent.futures as cf
import os

import numpy as np

import oracle as O

CODE_BUDGET = 1e-3
THREADS = max(1, min(32, os.cpu_count() or 1))


def oracle_map(fn, items, threads=THREADS):
    """fn over items on host threads (the C oracle releases the GIL while it
    runs), results in order."""
    items = list(items)
    if threads <= 1 or len(items) <= 1:
        return [fn(it) for it in items]
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))


def group_prequant_many(ratio, flags, v, s, cs_rows):
    """The oracle's pre-quantisation rows of G groups: v, s [G*ratio, 512],
    cs_rows [G, 64] (or None); returns float32 [G, 512]."""
    G = v.shape[0] // ratio
    chunks = [(a, min(G, a + 64)) for a in range(0, G, 64)]

    def run(ab):
        a, b = ab
        return np.stack([O.group_prequant(ratio, flags, v[i * ratio:(i + 1) * ratio], s[i * ratio:(i + 1) * ratio],
                                          None if cs_rows is None else cs_rows[i]) for i in range(a, b)])
    out = oracle_map(run, chunks)
    return np.concatenate(out) if out else np.zeros((0, 512), np.float32)


def token_prequant_many(flags, x, norm_weight, eps, cs_rows):
    """The oracle's pre-quantisation rows of n tokens x [n, 512]; cs_rows [n, 64]."""
    n = x.shape[0]
    chunks = [(a, min(n, a + 256)) for a in range(0, n, 256)]

    def run(ab):
        a, b = ab
        return np.stack([O.token_prequant(flags, x[t], norm_weight, eps, None if cs_rows is None else cs_rows[t])
                         for t in range(a, b)])
    out = oracle_map(run, chunks)
    return np.concatenate(out) if out else np.zeros((0, 512), np.float32)


def encode_many(layout, y):
    """Oracle code and scale rows of pre-quantisation rows y [n, 512]."""
    enc = O.encode_v41 if layout == O.V41 else O.encode_fp4
    rows = [enc(y[i]) for i in range(y.shape[0])]
    return np.stack([r[0] for r in rows]), np.stack([r[1] for r in rows])


def _log(ndiff, total):
    """Append the observed difference count to $KVQ_PARITY_LOG (if set)."""
    path = os.environ.get("KVQ_PARITY_LOG")
    if path:
        name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
        with open(path, "a") as f:
            f.write(f"{name} {ndiff} {total} {ndiff / max(1, total):.3e}\n")


def np_u8(t):
    return t.detach().cpu().numpy().view(np.uint8)


def gather_rows(pool_u8, layout, page_bits, slots):
    """(codes [n, CB], scale rows [n, SB]) of the given slots of a flat pool."""
    P = 1 << page_bits
    cb, sb = (512, 16) if layout == O.V41 else (256, 32)
    pb = P * (cb + sb)
    slots = np.asarray(slots, np.int64)
    page, row = slots // P, slots % P
    cidx = (page * pb + row * cb)[:, None] + np.arange(cb)[None, :]
    sidx = (page * pb + P * cb + row * sb)[:, None] + np.arange(sb)[None, :]
    return pool_u8[cidx], pool_u8[sidx]


def gather_rows_torch(pool, layout, page_bits, slots):
    """Same as gather_rows, done on the device, returned as numpy."""
    import torch
    P = 1 << page_bits
    cb, sb = (512, 16) if layout == O.V41 else (256, 32)
    pb = P * (cb + sb)
    s = torch.as_tensor(np.asarray(slots, np.int64), device=pool.device)
    page, row = s // P, s % P
    cidx = (page * pb + row * cb)[:, None] + torch.arange(cb, device=pool.device)[None, :]
    sidx = (page * pb + P * cb + row * sb)[:, None] + torch.arange(sb, device=pool.device)[None, :]
    return pool[cidx].cpu().numpy(), pool[sidx].cpu().numpy()


def decode_rows(layout, codes, scales):
    """float64 [n, 512] values of code / scale rows."""
    n = codes.shape[0]
    if layout == O.V41:
        v = O.e4m3_decode(codes).reshape(n, 16, 32)
        s = 2.0 ** (scales[:, :16].astype(np.float64) - 127)
        return (v * s[:, :, None]).reshape(n, 512)
    nib = np.stack([codes & 0xF, codes >> 4], axis=2).reshape(n, 512)
    v = O.e2m1_decode(nib).reshape(n, 16, 32)
    s = O.e4m3_decode(scales[:, :16])
    return (v * s[:, :, None]).reshape(n, 512)


def _grid_step(layout, mag):
    """Spacing of the element grid at magnitude `mag` (scale 1)."""
    mag = np.abs(mag)
    if layout == O.V41:
        e = np.floor(np.log2(np.maximum(mag, 2.0**-6)))
        return 2.0 ** (e - 3)
    return np.where(mag < 2, 0.5, np.where(mag < 4, 1.0, 2.0))


def block_scale(layout, scales):
    n = scales.shape[0]
    if layout == O.V41:
        s = 2.0 ** (scales[:, :16].astype(np.float64) - 127)
    else:
        s = O.e4m3_decode(scales[:, :16])
    return np.repeat(s.reshape(n, 16), 32, axis=1)


def check_tolerance(layout, g_codes, g_scales, o_codes, o_scales, y_oracle, budget=CODE_BUDGET):
    """Assert the tolerance rule; returns (n differing elements, n elements)."""
    n = g_codes.shape[0]
    if layout == O.FP4:
        assert (g_scales[:, 16:] == 0).all(), "FP4 padding must be zero"
    gd = decode_rows(layout, g_codes, g_scales)
    od = decode_rows(layout, o_codes, o_scales)
    gS = block_scale(layout, g_scales)
    oS = block_scale(layout, o_scales)
    S = np.maximum(gS, oS)
    # element-wise code difference (a scale mismatch makes the block differ)
    diff = gd != od
    ndiff = int(diff.sum())
    total = n * 512
    _log(ndiff, total)
    assert ndiff <= budget * total, f"{ndiff} of {total} elements differ"
    # one grid step at the larger of the two magnitudes, in units of the scale
    mag = np.maximum(np.abs(gd), np.abs(od)) / S
    step = _grid_step(layout, mag) * S
    assert (np.abs(gd - od) <= step + 0.0)[diff].all(), "a code differs by more than one step"
    y = y_oracle.astype(np.float64)
    own = np.abs(od - y)
    assert (np.abs(gd - y) <= own + step).all(), "dequantised value outside one step of the oracle"
    return ndiff, total
