"""Block quantisation pins: hand-worked blocks (tests/golden), the
dequant-of-quant error bound, and the footprint closed forms.

Layouts: "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats",
section 1 (V41 = 512 e4m3 codes + 16 ue8m0 scales = 528 B/token; V41_FP4 =
512 e2m1 codes + one e4m3 scale per 32 values, 288 B/token) and "Why is this
good" 1 (-9.6% and -50.7% against V4's 584 B/token).
"""
import numpy as np
import pytest

import oracle as O
from golden_io import load_blocks


def _deq_v41(codes, scales):
    v = O.e4m3_decode(codes).reshape(16, 32)
    return (v * (2.0 ** (scales.astype(np.float64) - 127))[:, None]).reshape(-1)


def _deq_fp4(codes, scales):
    nib = np.empty(512, np.uint8)
    nib[0::2] = codes & 0xF
    nib[1::2] = codes >> 4
    v = O.e2m1_decode(nib).reshape(16, 32)
    return (v * O.e4m3_decode(scales[:16])[:, None]).reshape(-1)


@pytest.mark.parametrize("blk", [0, 7, 15])
@pytest.mark.parametrize("case", load_blocks("v41_blocks.txt"), ids=lambda c: c[0])
def test_v41_handworked(case, blk):
    name, x, scale, codes, deq = case
    y = np.zeros(512, np.float32)
    y[blk * 32:(blk + 1) * 32] = x
    c, s = O.encode_v41(y)
    assert s[blk] == scale
    assert (np.delete(s, blk) == 0).all()
    cb = c[blk * 32:(blk + 1) * 32]
    for i in range(32):
        assert cb[i] == codes.get(i, 0x00), (name, i)
    d = _deq_v41(c, s)[blk * 32:(blk + 1) * 32]
    for i, v in deq.items():
        assert d[i] == np.float64(np.float32(v)) or d[i] == v, (name, i, d[i], v)


@pytest.mark.parametrize("blk", [0, 9, 15])
@pytest.mark.parametrize("case", load_blocks("fp4_blocks.txt"), ids=lambda c: c[0])
def test_fp4_handworked(case, blk):
    name, x, scale, codes, deq = case
    y = np.zeros(512, np.float32)
    y[blk * 32:(blk + 1) * 32] = x
    c, s = O.encode_fp4(y)
    assert s[blk] == scale
    assert (np.delete(s[:16], blk) == 0).all()
    assert (s[16:] == 0).all()           # the 16 B of stated padding
    cb = c[blk * 16:(blk + 1) * 16]
    for j in range(16):
        assert cb[j] == codes.get(j, 0x00), (name, j, hex(cb[j]))
    d = _deq_fp4(c, s)[blk * 32:(blk + 1) * 32]
    for i, v in deq.items():
        assert d[i] == v, (name, i, d[i], v)


def test_footprint_closed_forms():
    assert O.bytes_per_token(O.V41) == 528
    assert O.bytes_per_token(O.FP4) == 288
    assert O.page_bytes(O.V41, 6) == 64 * 528 == 33792
    assert O.page_bytes(O.FP4, 6) == 64 * 288 == 18432
    # 512 codes + 16 scales; 256 packed codes + 16 scales + 16 pad
    assert O.code_bytes(O.V41) + O.scale_bytes(O.V41) == 512 + 16
    assert O.code_bytes(O.FP4) == 256 and O.scale_bytes(O.FP4) == 32
    assert round((1 - 528 / 584) * 100, 1) == 9.6
    assert round((1 - 288 / 584) * 100, 1) == 50.7


def _rand_rows(rng, n):
    x = rng.standard_normal((n, 512)).astype(np.float32)
    x *= (10.0 ** rng.uniform(-6, 6, (n, 16)).astype(np.float32)).repeat(32, axis=1)
    x[rng.random((n, 512)) < 0.01] *= 50
    return x


def test_v41_error_bound():
    """|x - deq| <= max(2^-4 |x|, 2^-10 S) when |x|/S <= 448, else |x| - 448 S."""
    rng = np.random.default_rng(5)
    for y in _rand_rows(rng, 200):
        c, s = O.encode_v41(y)
        d = _deq_v41(c, s)
        S = np.repeat(2.0 ** (s.astype(np.float64) - 127), 32)
        a = np.abs(y.astype(np.float64))
        err = np.abs(y - d)
        inrange = a / S <= 448
        assert (err[inrange] <= np.maximum(2.0**-4 * a, 2.0**-10 * S)[inrange]).all()
        assert np.allclose(err[~inrange], (a - 448 * S)[~inrange], rtol=0, atol=0)
        assert (err <= a / 8 + 2.0**-10 * S).all()


def test_fp4_error_bound():
    """|x - deq| <= S for blocks whose scale is a normal e4m3 (6*2^-6 <= amax <= 2688)."""
    rng = np.random.default_rng(6)
    x = rng.standard_t(3, (200, 512)).astype(np.float32) * 0.5
    for y in x:
        c, s = O.encode_fp4(y)
        d = _deq_fp4(c, s)
        S = np.repeat(O.e4m3_decode(s[:16]), 32)
        amax = np.repeat(np.abs(y.reshape(16, 32)).max(1), 32)
        ok = (amax >= 6 * 2.0**-6) & (amax <= 2688)
        assert (np.abs(y - d)[ok] <= S[ok]).all()


def test_v41_scale_from_exponent_bits():
    """Scale byte = exponent field of amax - 8: doubling the block adds one."""
    rng = np.random.default_rng(7)
    y = rng.standard_normal(512).astype(np.float32)
    _, s1 = O.encode_v41(y)
    c2, s2 = O.encode_v41(y * 2)
    c1, _ = O.encode_v41(y)
    assert (s2.astype(int) - s1 == 1).all()
    assert (c1 == c2).all()
