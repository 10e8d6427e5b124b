"""Pins of the oracle's pre-quantisation math: RoPE, K RMSNorm, softmax pooling.

RoPE and the fused norm: "[sglang] DeepSeek V4.1 Paged KV Cache: V41 and FP4
formats", store-latency table rows "store + RoPE" / "fused K norm + RoPE".
Pooling: the c1/c2 ratio compressors (same page, section 2) and the C4A/C128A
compressor of "[vLLM] DeepSeek V4 Sparse FP8 Compressor kernel", section 2
(online max/sum softmax).  Checks use closed forms and invariants, not the
oracle's own formulas.
"""
import numpy as np
import pytest

import oracle as O


def _table(angles):
    return np.concatenate([np.cos(angles), np.sin(angles)]).astype(np.float32)


def test_rope_is_complex_multiplication():
    rng = np.random.default_rng(10)
    for _ in range(20):
        y = rng.standard_normal(512).astype(np.float32)
        ang = rng.uniform(-np.pi, np.pi, 32)
        cs = _table(ang)
        out = O.rope(y, cs)
        assert (out[:448] == y[:448]).all()
        z = (y[448::2].astype(np.float64) + 1j * y[449::2]) * (cs[:32].astype(np.float64) + 1j * cs[32:])
        assert np.allclose(out[448::2], z.real, rtol=0, atol=4e-7 * (1 + np.abs(z)))
        assert np.allclose(out[449::2], z.imag, rtol=0, atol=4e-7 * (1 + np.abs(z)))


def test_rope_special_angles():
    rng = np.random.default_rng(11)
    y = rng.standard_normal(512).astype(np.float32)
    ident = np.concatenate([np.ones(32), np.zeros(32)]).astype(np.float32)
    assert (O.rope(y, ident) == y).all()
    quarter = np.concatenate([np.zeros(32), np.ones(32)]).astype(np.float32)
    out = O.rope(y, quarter)           # (a, b) -> (-b, a)
    assert (out[448::2] == -y[449::2]).all() and (out[449::2] == y[448::2]).all()


def test_rope_preserves_pair_norm_and_adds_angles():
    rng = np.random.default_rng(12)
    y = rng.standard_normal(512).astype(np.float32)
    a1, a2 = rng.uniform(-3, 3, 32), rng.uniform(-3, 3, 32)
    two = O.rope(O.rope(y, _table(a1)), _table(a2))
    one = O.rope(y, _table(a1 + a2))
    assert np.allclose(two, one, atol=2e-6)
    n0 = y[448::2].astype(np.float64) ** 2 + y[449::2].astype(np.float64) ** 2
    n1 = two[448::2].astype(np.float64) ** 2 + two[449::2].astype(np.float64) ** 2
    assert np.allclose(n0, n1, rtol=1e-5)


def test_rmsnorm_constant_vector():
    w = np.random.default_rng(13).normal(1, 0.1, 512).astype(np.float32)
    for c in [1.0, -3.0, 0.25, 1e3]:
        y = O.rmsnorm(np.full(512, c, np.float32), w, 1e-6)
        exp = np.sign(c) * w / np.sqrt(1 + 1e-6 / c**2)
        assert np.allclose(y, exp, rtol=3e-7, atol=0)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(14)
    x = rng.standard_normal(512).astype(np.float32) * 3
    ones = np.ones(512, np.float32)
    y = O.rmsnorm(x, ones, 0.0)
    assert abs(np.mean(y.astype(np.float64) ** 2) - 1) < 1e-6
    y2 = O.rmsnorm(x * 8, ones, 0.0)          # power-of-two scale: exact
    assert (y2 == y).all()
    w = rng.normal(1, 0.1, 512).astype(np.float32)
    yw = O.rmsnorm(x, w, 0.0)
    assert np.allclose(yw, y * w, rtol=1e-6)


def test_pool_r1_is_identity():
    rng = np.random.default_rng(15)
    v = rng.standard_normal((1, 512)).astype(np.float32)
    s = rng.standard_normal((1, 512)).astype(np.float32) * 30
    assert (O.pool(v, s) == v[0]).all()


@pytest.mark.parametrize("r", [2, 4, 128])
def test_pool_equal_scores_is_mean(r):
    rng = np.random.default_rng(16 + r)
    v = rng.standard_normal((r, 512)).astype(np.float32)
    s = np.tile(rng.standard_normal(512).astype(np.float32), (r, 1))
    mean = v.astype(np.float64).mean(0)
    assert np.allclose(O.pool(v, s), mean, rtol=0, atol=1e-6)


@pytest.mark.parametrize("r", [2, 4, 128])
def test_pool_dominant_score_selects_row(r):
    rng = np.random.default_rng(20 + r)
    v = rng.standard_normal((r, 512)).astype(np.float32)
    s = rng.standard_normal((r, 512)).astype(np.float32)
    pick = rng.integers(0, r, 512)
    s[pick, np.arange(512)] += 200.0       # e^-190 is far below half an fp32 ulp
    assert (O.pool(v, s) == v[pick, np.arange(512)]).all()


def test_pool_two_rows_sigmoid_closed_form():
    rng = np.random.default_rng(30)
    v = rng.standard_normal((2, 512)).astype(np.float32)
    s = rng.standard_normal((2, 512)).astype(np.float32) * 3
    sig = 1 / (1 + np.exp(-(s[1].astype(np.float64) - s[0])))
    exp = v[0] + (v[1].astype(np.float64) - v[0]) * sig
    assert np.allclose(O.pool(v, s), exp, rtol=0, atol=1e-6)


@pytest.mark.parametrize("r", [4, 128])
def test_pool_convex_and_invariant(r):
    rng = np.random.default_rng(40 + r)
    v = rng.standard_normal((r, 512)).astype(np.float32)
    s = (rng.standard_normal((r, 512)) * 2).astype(np.float32)
    out = O.pool(v, s)
    assert (out >= v.min(0)).all() and (out <= v.max(0)).all()
    perm = rng.permutation(r)
    assert np.allclose(O.pool(v[perm], s[perm]), out, rtol=0, atol=2e-7)
    assert np.allclose(O.pool(v, s + 5.0), out, rtol=0, atol=1e-5)


def test_token_prequant_bf16_rounding_rule():
    """fp32 math (norm/RoPE) is rounded to bf16; an untouched fp32 row is not."""
    rng = np.random.default_rng(50)
    x = rng.standard_normal(512).astype(np.float32)
    assert (O.token_prequant(0, x) == x).all()
    ident = np.concatenate([np.ones(32), np.zeros(32)]).astype(np.float32)
    y = O.token_prequant(O.ROPE, x, cs_row=ident)
    assert (y == O.bf16_round(x)).all()
