"""Pins of the oracle's number formats against things other than itself.

* E4M3: torch's float8_e4m3fn cast (a library routine) inside the finite range,
  and a brute-force nearest-value search over every finite code.
* E2M1: brute-force nearest-value search over the eight OCP MX E2M1 values.
* bf16: torch's bfloat16 cast, including ties and subnormals.
Format definitions: OCP FP8 (E4M3) and OCP Microscaling v1.0 (E2M1), the
formats named in "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4 formats",
section 1.
"""
import numpy as np
import pytest
import torch

import oracle as O

pytestmark = []


def _all_e4m3_finite():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    return codes, O.e4m3_decode(codes)


def test_e4m3_decode_table_points():
    # OCP FP8: 0x01 = 2^-9, 0x08 = 2^-6, 0x38 = 1, 0x7E = 448, 0xFE = -448, 0x7F NaN
    v = O.e4m3_decode(np.array([0x01, 0x07, 0x08, 0x38, 0x40, 0x7E, 0xFE, 0x80], np.uint8))
    assert list(v) == [2.0**-9, 7 * 2.0**-9, 2.0**-6, 1.0, 2.0, 448.0, -448.0, 0.0]
    assert np.signbit(v[-1])
    assert np.isnan(O.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_roundtrip_every_code():
    codes, vals = _all_e4m3_finite()
    back = O.e4m3_encode(vals.astype(np.float32))
    assert (back == codes).all()


def test_e4m3_matches_torch_cast():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 50,
        rng.standard_normal(50000).astype(np.float32) * 1e-3,
        (rng.uniform(-463.9, 463.9, 50000)).astype(np.float32),
    ])
    # every rounding midpoint between neighbouring finite codes, and +-1 ulp around it
    _, vals = _all_e4m3_finite()
    pos = np.unique(vals[vals >= 0])
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    mids = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    x = np.concatenate([x, mids, -mids]).astype(np.float32)
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(x)
    assert (got == ref).all(), x[got != ref][:10]


def test_e4m3_saturates():
    x = np.array([448, 449, 463.9, 464, 480, 1e6, 3e38, -500, -1e30], np.float32)
    got = O.e4m3_encode(x)
    assert list(got) == [0x7E] * 6 + [0x7E, 0xFE, 0xFE]


def test_e4m3_bruteforce_nearest_ties_even():
    codes, vals = _all_e4m3_finite()
    pos_codes = codes[(codes & 0x80) == 0]
    pos_vals = vals[(codes & 0x80) == 0]
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.uniform(0, 448, 20000), 2.0 ** rng.uniform(-14, 8.8, 20000)]).astype(np.float32)
    x = np.concatenate([x, ((pos_vals[1:] + pos_vals[:-1]) / 2).astype(np.float32)])
    x = x[x <= 448]
    got = O.e4m3_encode(x)
    for xi, gi in zip(x, got):
        d = np.abs(pos_vals - float(xi))
        best = np.flatnonzero(d == d.min())
        if len(best) == 1:
            exp = pos_codes[best[0]]
        else:  # a tie: the code whose mantissa LSB is 0
            exp = [pos_codes[b] for b in best if pos_codes[b] % 2 == 0][0]
        assert gi == exp, (xi, gi, exp)


def test_e4m3_negative_and_signed_zero():
    x = np.array([-1.0, -0.0, -1e-30, 0.0, 1e-30], np.float32)
    assert list(O.e4m3_encode(x)) == [0xB8, 0x80, 0x80, 0x00, 0x00]


E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_table():
    v = O.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert list(v[:8]) == E2M1_VALUES
    assert list(v[8:]) == [-a for a in E2M1_VALUES]


def test_e2m1_bruteforce_nearest_ties_even():
    rng = np.random.default_rng(3)
    grid = np.array(E2M1_VALUES)
    mids = (grid[1:] + grid[:-1]) / 2
    x = np.concatenate([rng.uniform(0, 7, 50000), mids, np.nextafter(mids, 0), np.nextafter(mids, 9),
                        [6.0, 6.5, 100.0, 0.0]]).astype(np.float32)
    got = O.e2m1_encode(x)
    for xi, gi in zip(x, got):
        if xi >= 6:
            assert gi == 7
            continue
        d = np.abs(grid - float(xi))
        best = np.flatnonzero(d == d.min())
        exp = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert gi == exp, (xi, gi, exp)
    neg = O.e2m1_encode(-x)
    assert ((neg & 7) == got).all() and (neg >= 8).all()


def test_bf16_matches_torch_cast():
    rng = np.random.default_rng(4)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 100000),
        # exact ties: lower 16 bits == 0x8000, both parities of the kept LSB
        (rng.integers(0, 2**31, 20000, dtype=np.uint64).astype(np.uint32) & 0x7F7F0000 | 0x8000).view(np.float32),
        # subnormal binary32
        (rng.integers(1, 2**23, 20000).astype(np.uint32)).view(np.float32),
    ]).astype(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.bf16_bits(x)
    assert (got == ref).all()
