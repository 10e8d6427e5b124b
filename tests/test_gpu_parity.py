"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Workloads follow the write path's configurations (see compress_kv_write_gb300.synth):
the small fp32 V41 store + dequant; the bf16 store / store + RoPE / fused
norm + RoPE batch sweep; the FP4 store + full-pool paged dequant; the
translated C4A compressor; the mixed-length C128A compressor (both layouts);
plus codec sweeps, every compiled instance on ragged sizes, and the error
paths.  Plain store, RoPE store, scatter, translation and dequant must be
bit-exact; the norm and pooling paths follow the tolerance rule in
tests/parity.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from parity import (check_tolerance, decode_rows, encode_many, gather_rows, gather_rows_torch,
                    group_prequant_many, np_u8, oracle_map, token_prequant_many)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def K():
    from compress_kv_write_gb300 import build
    build.build()
    import compress_kv_write_gb300 as K
    K.lib()
    return K


def _bf16_np(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _err(K):
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _oracle_store_rows(layout, flags, x_np, norm_weight=None, eps=1e-6, cos_sin=None, pos=None):
    """Oracle rows of x stored into a compact pool at slots 0..n-1."""
    n = x_np.shape[0]
    slots = max(64, -(-n // 64) * 64)
    pool = np.zeros(slots * O.bytes_per_token(layout), np.uint8)
    rc = O.store(layout, 6, flags, x_np, np.arange(n), pool, norm_weight=norm_weight, eps=eps,
                 cos_sin=cos_sin, pos=pos)
    assert rc == O.OK
    return gather_rows(pool, layout, 6, np.arange(n))


# --------------------------------------------------------------------------- small fp32 config

def test_fp32_store_and_dequant_64_tokens(K):
    """64 fp32 N(0,1) rows (seed 0) into a 4-page V41 pool at a random
    injective map of the 256 slots, then the dequant: whole pool and whole
    workspace bit-exact."""
    from compress_kv_write_gb300 import synth
    x = synth.normal((64, 512), "cpu", 0, "x")
    loc = synth.injective_slots(64, 256, "cpu", 0)
    pool_o = np.zeros(256 * 528, np.uint8)
    assert O.store(O.V41, 6, 0, x.numpy(), loc.numpy(), pool_o) == O.OK
    pool = torch.zeros(256 * 528, dtype=torch.uint8, device=DEV)
    err = _err(K)
    K.kvq_store(K.V41, 6, 0, x.to(DEV), loc.to(DEV), pool, 256, err=err)
    pt = torch.arange(4, dtype=torch.int32)
    out = torch.full((256, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    K.kvq_dequant(K.V41, 6, pool, 4, pt.to(DEV), out, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert (np_u8(pool) == pool_o).all()
    rc, ws = O.dequant(O.V41, 6, pool_o, pt.numpy(), 256)
    assert rc == O.OK
    assert (_bf16_np(out) == ws).all()


# --------------------------------------------------------------------------- every instance, ragged

@pytest.mark.parametrize("page_bits", [2, 6])
@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("loc64", [False, True])
@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_store_instances_ragged(K, page_bits, layout, dtype, loc64, flags):
    """Every store instance on ragged batches of 1, 37, 301, 1537 and 3100
    rows, which cover every store mapping: one CTA per token, two tokens per
    CTA (301 rows plain and FP4, 1537 with RoPE only) and the persistent
    kernels.  The plain and RoPE paths bit-exact over the whole pool; the
    norm paths under the tolerance rule, the batches pooled into one
    comparison."""
    from compress_kv_write_gb300 import synth
    slots = 4096
    rng_seed = page_bits * 1000 + layout * 100 + flags * 10 + int(loc64)
    acc = [[], [], [], [], []]
    for n in (1, 37, 301, 1537, 3100):
        x = synth.store_rows_bf16(n, "cpu", rng_seed + n)
        if dtype == "f32":
            x = x.float() * 1.25          # not bf16-representable in general
        loc = synth.injective_slots(n, slots, "cpu", rng_seed + n,
                                    dtype=torch.int64 if loc64 else torch.int32)
        w = synth.norm_weight("cpu", rng_seed)
        cs = synth.rope_table(4096, "cpu")
        pos = synth.positions(n, "cpu", rng_seed + n, max_pos=4096)
        x_np = x.numpy() if dtype == "f32" else _bf16_np(x)
        pool_o = np.zeros(slots * O.bytes_per_token(layout), np.uint8)
        assert O.store(layout, page_bits, flags, x_np, loc.numpy(), pool_o,
                       norm_weight=w.numpy(), eps=1e-6, cos_sin=cs.numpy(), pos=pos.numpy()) == O.OK
        pool = torch.zeros(slots * O.bytes_per_token(layout), dtype=torch.uint8, device=DEV)
        err = _err(K)
        K.kvq_store(layout, page_bits, flags, x.to(DEV), loc.to(DEV), pool, slots,
                    norm_weight=w.to(DEV) if flags & 2 else None, eps=1e-6,
                    cos_sin=cs.to(DEV) if flags & 1 else None,
                    pos=pos.to(DEV) if flags & 1 else None, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        got = np_u8(pool)
        if flags & 2 == 0:            # plain and RoPE paths: bit-exact
            assert (got == pool_o).all(), (n, np.flatnonzero(got != pool_o)[:8])
        else:
            g = gather_rows(got, layout, page_bits, loc.numpy())
            o = gather_rows(pool_o, layout, page_bits, loc.numpy())
            y = token_prequant_many(flags, x_np, w.numpy(), 1e-6, cs.numpy()[pos.numpy()])
            for a, b in zip(acc, (g[0], g[1], o[0], o[1], y)):
                a.append(b)
            written = int(g[0].astype(np.int64).sum() + g[1].astype(np.int64).sum())
            assert int(got.astype(np.int64).sum()) == written   # nothing else touched
    if flags & 2:
        check_tolerance(layout, *[np.concatenate(a) for a in acc])


# --------------------------------------------------------------------------- codecs

def _all_mappings(x):
    """x itself (a small batch: one CTA per token), x tiled to 600 rows or
    more (two tokens per CTA for the plain and FP4 stores) and x tiled past
    3072 rows (the persistent kernels), so that a codec pin covers every store
    mapping."""
    return [x, np.tile(x, (-(-600 // x.shape[0]), 1)), np.tile(x, (-(-3073 // x.shape[0]), 1))]


def test_codec_every_bf16_pattern(K):
    """All finite bf16 bit patterns through the plain store, both layouts,
    both store mappings."""
    bits = np.arange(65536, dtype=np.uint32)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    pat = bits[finite].astype(np.uint16)
    rng = np.random.default_rng(0)
    pat = pat[rng.permutation(pat.size)]
    pad = (-pat.size) % 512
    pat1 = np.concatenate([pat, np.zeros(pad, np.uint16)]).reshape(-1, 512)
    for pat in _all_mappings(pat1):
        n = pat.shape[0]
        slots = -(-n // 64) * 64
        x = torch.from_numpy(pat.view(np.int16)).view(torch.bfloat16).to(DEV)
        for layout in (1, 2):
            rows_o = _oracle_store_rows(layout, 0, pat)
            pool = torch.zeros(slots * O.bytes_per_token(layout), dtype=torch.uint8, device=DEV)
            loc = torch.arange(n, dtype=torch.int32, device=DEV)
            K.kvq_store(layout, 6, 0, x, loc, pool, slots)
            torch.cuda.synchronize()
            g = gather_rows(np_u8(pool), layout, 6, np.arange(n))
            assert (g[0] == rows_o[0]).all() and (g[1] == rows_o[1]).all(), (n, layout)


def _midpoint_rows(anchor, grid):
    """fp32 rows whose blocks start with `anchor` (pinning the block scale) and
    hold the grid's midpoints and their neighbours, both signs."""
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    vals = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1e30)), grid.astype(np.float32)])
    vals = np.concatenate([vals, -vals])
    per = 31
    nblk = -(-vals.size // per)
    vals = np.concatenate([vals, np.zeros(nblk * per - vals.size, np.float32)]).reshape(nblk, per)
    blocks = np.concatenate([np.full((nblk, 1), anchor, np.float32), vals], axis=1)
    nb = -(-nblk // 16) * 16
    blocks = np.concatenate([blocks, np.zeros((nb - nblk, 32), np.float32)])
    return blocks.reshape(-1, 512)


def test_codec_e4m3_midpoints(K):
    codes = np.array([c for c in range(128) if c != 0x7F], np.uint8)
    grid = np.unique(O.e4m3_decode(codes))
    x = _midpoint_rows(448.0, grid)          # byte 127: multiplier 1
    x = np.concatenate([x, _midpoint_rows(511.0, np.array([448.0, 460.0, 464.0, 480.0, 500.0]))])
    for x in _all_mappings(x):
        rows_o = _oracle_store_rows(O.V41, 0, x)
        n = x.shape[0]
        pool = torch.zeros(-(-n // 64) * 64 * 528, dtype=torch.uint8, device=DEV)
        K.kvq_store(K.V41, 6, 0, torch.from_numpy(x).to(DEV), torch.arange(n, device=DEV), pool,
                    -(-n // 64) * 64)
        torch.cuda.synchronize()
        g = gather_rows(np_u8(pool), O.V41, 6, np.arange(n))
        assert (g[1] == rows_o[1]).all(), n
        assert (g[0] == rows_o[0]).all(), (n, np.argwhere(g[0] != rows_o[0])[:5])


def test_codec_e2m1_midpoints(K):
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    x = _midpoint_rows(6.0, grid)            # scale 1.0
    x = np.concatenate([x, _midpoint_rows(6.0, np.array([5.9, 6.0, 6.2, 7.0, 100.0]))])
    x = np.clip(x, -6, 6)                    # keep the block amax at 6
    for x in _all_mappings(x):
        rows_o = _oracle_store_rows(O.FP4, 0, x)
        n = x.shape[0]
        slots = -(-n // 64) * 64
        pool = torch.zeros(slots * 288, dtype=torch.uint8, device=DEV)
        K.kvq_store(K.V41_FP4, 6, 0, torch.from_numpy(x).to(DEV), torch.arange(n, device=DEV), pool, slots)
        torch.cuda.synchronize()
        g = gather_rows(np_u8(pool), O.FP4, 6, np.arange(n))
        assert (g[1] == rows_o[1]).all(), n
        assert (g[0] == rows_o[0]).all(), n


def test_fp4_every_scale_byte(K):
    """Every non-zero e4m3 block scale (bytes 1..126) through the FP4 store: a
    block whose amax is 6 x the scale's value sets that scale, and its other
    31 values sweep the e2m1 grid, its midpoints and their neighbours at that
    scale (both signs).  The stored code and scale bytes, and the dequant,
    must equal the oracle's, so every entry of the kernel's reciprocal table
    and every scale its quotient can produce is exercised.  The 8 rows run
    alone (one CTA per token), tiled to 520 rows (two tokens per CTA) and to
    3080 rows (the persistent kernel with its reciprocal table)."""
    codes = np.arange(1, 127, dtype=np.uint8)
    S = O.e4m3_decode(codes)
    amax = (S * 6).astype(np.float32)
    assert (O.e4m3_encode((amax / np.float32(6)).astype(np.float32)) == codes).all()
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    mids = (grid[1:] + grid[:-1]) / 2
    unit = np.concatenate([grid[:-1], mids, mids * (1 - 2.0**-20), mids * (1 + 2.0**-20)])  # 28 values
    unit = np.concatenate([unit, [-0.25, -1.5, -3.0]])                                   # 31 values
    rows = []
    for i, s_ in enumerate(S):
        blk = np.concatenate([[amax[i]], unit * s_]).astype(np.float32)
        blk[1::2] *= -1 if i % 2 else 1
        rows.append(blk)
    nb = -(-len(rows) // 16) * 16
    rows += [np.zeros(32, np.float32)] * (nb - len(rows))
    x1 = np.stack(rows).reshape(-1, 512)
    for dtype, reps in (("f32", 1), ("bf16", 1), ("f32", 65), ("bf16", 65), ("f32", 385), ("bf16", 385)):
        x = np.tile(x1, (reps, 1))
        xx = x if dtype == "f32" else O.bf16_bits(x).reshape(x.shape)
        rows_o = _oracle_store_rows(O.FP4, 0, xx)
        n = x.shape[0]
        slots = -(-n // 64) * 64
        pool = torch.zeros(slots * 288, dtype=torch.uint8, device=DEV)
        xt = torch.from_numpy(x).to(DEV) if dtype == "f32" else \
            torch.from_numpy(xx.view(np.int16)).view(torch.bfloat16).to(DEV)
        err = _err(K)
        K.kvq_store(K.V41_FP4, 6, 0, xt, torch.arange(n, device=DEV), pool, slots, err=err)
        out = torch.empty((slots, 512), dtype=torch.bfloat16, device=DEV)
        K.kvq_dequant(K.V41_FP4, 6, pool, slots // 64, torch.arange(slots // 64, dtype=torch.int32, device=DEV),
                      out, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        g = gather_rows(np_u8(pool), O.FP4, 6, np.arange(n))
        assert (g[1] == rows_o[1]).all(), dtype
        assert (g[0] == rows_o[0]).all(), dtype
        pool_o = np.zeros(slots * 288, np.uint8)
        assert O.store(O.FP4, 6, 0, xx, np.arange(n), pool_o) == O.OK
        rc, ws = O.dequant(O.FP4, 6, pool_o, np.arange(slots // 64, dtype=np.int32), slots)
        assert rc == O.OK and (_bf16_np(out) == ws).all()
        if dtype == "f32":  # every scale byte 1..126 appears
            assert set(np.unique(g[1][:, :16])) >= set(range(1, 127))


@pytest.mark.parametrize("layout", [1, 2])
def test_codec_dequant_every_code_and_scale(K, layout):
    """Every (code, scale byte) pair through the paged dequant."""
    P = 64
    bpt = O.bytes_per_token(layout)
    pool = np.zeros(P * bpt, np.uint8)
    cb, sb = (512, 16) if layout == 1 else (256, 32)
    for t in range(P):
        pool[t * cb:(t + 1) * cb] = (np.arange(cb) + 7 * t) % 256
        s = (np.arange(16) + 16 * t) % 256
        pool[P * cb + t * sb:P * cb + t * sb + 16] = s
    out = torch.empty((P, 512), dtype=torch.bfloat16, device=DEV)
    K.kvq_dequant(layout, 6, torch.from_numpy(pool).to(DEV), 1,
                  torch.zeros(1, dtype=torch.int32, device=DEV), out)
    torch.cuda.synchronize()
    rc, ws = O.dequant(layout, 6, pool, np.zeros(1, np.int32), P)
    got = _bf16_np(out)
    gf = O.bf16_to_f32(got)
    of = O.bf16_to_f32(ws)
    nan = np.isnan(of)
    assert (np.isnan(gf) == nan).all()
    assert (got[~nan] == ws[~nan]).all()


# --------------------------------------------------------------------------- store batch sweep

POOL_SLOTS_1 = 1 << 20


@pytest.fixture(scope="module")
def sweep_inputs():
    from compress_kv_write_gb300 import synth
    n = 16384
    x = synth.store_rows_bf16(n, DEV, 0)
    loc = synth.injective_slots(n, POOL_SLOTS_1, DEV, 0)
    pos = synth.positions(n, DEV, 0)
    cs = synth.rope_table(65536, DEV)
    w = synth.norm_weight(DEV, 0)
    return x, loc, pos, cs, w


@pytest.mark.parametrize("flags", [0, 1, 3])
def test_store_batch_sweep(K, sweep_inputs, flags):
    """bf16 rows with outliers, pool of 2^20 slots: store, store + RoPE and
    fused K RMSNorm + RoPE at every batch size of the sweep (1, 8, 64, 512,
    16384) and at 1024 and 1025 tokens (the small-batch kernel's limit with
    the norm), each into a fresh pool.  Plain and RoPE stores are bit-exact; the fused
    norm path follows the tolerance rule with the batches pooled into one
    comparison."""
    x_all, loc_all, pos_all, cs, w = sweep_inputs
    cs_np, w_np = cs.cpu().numpy(), w.cpu().numpy()
    acc = [[], [], [], [], []]
    for bs in (1, 8, 64, 512, 1024, 1025, 16384):
        x, loc, pos = x_all[:bs], loc_all[:bs], pos_all[:bs]
        pool = torch.zeros(POOL_SLOTS_1 * 528, dtype=torch.uint8, device=DEV)
        err = _err(K)
        K.kvq_store(K.V41, 6, flags, x, loc, pool, POOL_SLOTS_1, norm_weight=w, eps=1e-6,
                    cos_sin=cs, pos=pos, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        g = gather_rows_torch(pool, O.V41, 6, loc.cpu().numpy())
        x_np, pos_np = _bf16_np(x), pos.cpu().numpy()
        o = _oracle_store_rows(O.V41, flags, x_np, w_np, 1e-6, cs_np, pos_np)
        if flags & 2:
            y = token_prequant_many(flags, x_np, w_np, 1e-6, cs_np[pos_np])
            for a, b in zip(acc, (g[0], g[1], o[0], o[1], y)):
                a.append(b)
        else:
            assert (g[0] == o[0]).all() and (g[1] == o[1]).all(), bs
        written = int(g[0].astype(np.int64).sum() + g[1].astype(np.int64).sum())
        assert int(pool.sum(dtype=torch.int64).item()) == written
    if flags & 2:
        check_tolerance(O.V41, *[np.concatenate(a) for a in acc])


@pytest.mark.parametrize("flags,switch", [(1, 12288), (0, 16384), (2, 65536), (3, 65536)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("loc64", [False, True])
def test_v41_store_both_persistent_mappings(K, flags, switch, dtype, loc64):
    """Large V41 batches take the half-warp kernel, smaller ones one warp per
    token; the switch sits at 12288 tokens with RoPE only, 16384 for the plain
    store and 65536 with the norm.  One batch on each side of it (page_bits 2
    for the first, 6 for the second): the plain and RoPE stores bit-exact over
    the whole pool, the norm paths under the tolerance rule with both batches
    pooled."""
    from compress_kv_write_gb300 import synth
    slots = 1 << (2 * switch).bit_length()
    cs = synth.rope_table(8192, "cpu")
    acc = [[], [], [], [], []]
    for n, page_bits in ((switch - 1, 2), (switch + 1, 6)):
        seed = 70 + flags * 8 + int(loc64) * 2 + (dtype == "f32") + n % 3
        x = synth.store_rows_bf16(n, "cpu", seed)
        if dtype == "f32":
            x = x.float() * 1.25
        loc = synth.injective_slots(n, slots, "cpu", seed, dtype=torch.int64 if loc64 else torch.int32)
        pos = synth.positions(n, "cpu", seed, max_pos=8192)
        w = synth.norm_weight("cpu", seed)
        x_np = x.numpy() if dtype == "f32" else _bf16_np(x)
        pool_o = np.zeros(slots * 528, np.uint8)
        assert O.store(O.V41, page_bits, flags, x_np, loc.numpy(), pool_o, norm_weight=w.numpy(), eps=1e-6,
                       cos_sin=cs.numpy(), pos=pos.numpy()) == O.OK
        pool = torch.zeros(slots * 528, dtype=torch.uint8, device=DEV)
        err = _err(K)
        K.kvq_store(K.V41, page_bits, flags, x.to(DEV), loc.to(DEV), pool, slots,
                    norm_weight=w.to(DEV) if flags & 2 else None, eps=1e-6,
                    cos_sin=cs.to(DEV) if flags & 1 else None, pos=pos.to(DEV) if flags & 1 else None, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        got = np_u8(pool)
        if flags & 2 == 0:
            assert (got == pool_o).all(), (n, np.flatnonzero(got != pool_o)[:8])
        else:
            g = gather_rows(got, O.V41, page_bits, loc.numpy())
            o = gather_rows(pool_o, O.V41, page_bits, loc.numpy())
            y = token_prequant_many(flags, x_np, w.numpy(), 1e-6, cs.numpy()[pos.numpy()])
            for a, b in zip(acc, (g[0], g[1], o[0], o[1], y)):
                a.append(b)
            written = int(g[0].astype(np.int64).sum() + g[1].astype(np.int64).sum())
            assert int(got.astype(np.int64).sum()) == written   # nothing else touched
    if flags & 2:
        check_tolerance(O.V41, *[np.concatenate(a) for a in acc])


@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("flags", [0, 1, 3])
def test_store_random_batch_sizes(K, layout, flags):
    """Seeded log-uniform batch sizes from 1 to 40000 tokens (and the sizes
    on each side of every switch between the store mappings), bf16 rows,
    int32 or int64 slots: the plain and RoPE paths bit-exact over the whole
    pool, the norm path under the tolerance rule with all batches pooled."""
    from compress_kv_write_gb300 import synth
    rng = np.random.default_rng(300 + 10 * layout + flags)
    sizes = sorted(set(int(v) for v in np.exp(rng.uniform(0, np.log(40000), 6))) |
                   {256, 257, 512, 513, 1536, 1537, 3072, 3073, 12287, 12288, 16383, 16384})
    slots = 1 << 17
    cs = synth.rope_table(8192, "cpu")
    acc = [[], [], [], [], []]
    for n in sizes:
        seed = 500 + n
        x = synth.store_rows_bf16(n, "cpu", seed)
        loc = synth.injective_slots(n, slots, "cpu", seed, dtype=torch.int64 if n % 2 else torch.int32)
        pos = synth.positions(n, "cpu", seed, max_pos=8192)
        w = synth.norm_weight("cpu", seed)
        x_np = _bf16_np(x)
        rows_o = _oracle_store_rows(layout, flags, x_np, w.numpy(), 1e-6, cs.numpy(), pos.numpy())
        pool = torch.zeros(slots * O.bytes_per_token(layout), dtype=torch.uint8, device=DEV)
        err = _err(K)
        K.kvq_store(layout, 6, flags, x.to(DEV), loc.to(DEV), pool, slots,
                    norm_weight=w.to(DEV) if flags & 2 else None, eps=1e-6,
                    cos_sin=cs.to(DEV) if flags & 1 else None, pos=pos.to(DEV) if flags & 1 else None, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0, n
        g = gather_rows_torch(pool, layout, 6, loc.numpy())
        if flags & 2:
            y = token_prequant_many(flags, x_np, w.numpy(), 1e-6, cs.numpy()[pos.numpy()])
            for a, b in zip(acc, (g[0], g[1], rows_o[0], rows_o[1], y)):
                a.append(b)
        else:
            assert (g[0] == rows_o[0]).all() and (g[1] == rows_o[1]).all(), n
        written = int(g[0].astype(np.int64).sum() + g[1].astype(np.int64).sum())
        assert int(pool.sum(dtype=torch.int64).item()) == written, n   # nothing else touched
    if flags & 2:
        check_tolerance(layout, *[np.concatenate(a) for a in acc])


# --------------------------------------------------------------------------- FP4 store + dequant

POOL_SLOTS_2 = 1 << 21


@pytest.mark.parametrize("bs", [16384, 262144])
def test_fp4_store_and_full_pool_dequant(K, bs):
    """Student-t(3) x 0.5 bf16 rows into a 2^21-slot FP4 pool, then the paged
    dequant of the whole pool through a permuted page table."""
    from compress_kv_write_gb300 import synth
    x = synth.student_t_rows_bf16(bs, DEV, 0)
    loc = synth.injective_slots(bs, POOL_SLOTS_2, DEV, 0)
    pool = torch.zeros(POOL_SLOTS_2 * 288, dtype=torch.uint8, device=DEV)
    err = _err(K)
    K.kvq_store(K.V41_FP4, 6, 0, x, loc, pool, POOL_SLOTS_2, err=err)
    n_pages = POOL_SLOTS_2 >> 6
    pt = synth.page_table_perm(n_pages, DEV, 0)
    out = torch.empty((POOL_SLOTS_2, 512), dtype=torch.bfloat16, device=DEV)
    K.kvq_dequant(K.V41_FP4, 6, pool, n_pages, pt, out, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    # every stored row, bit-exact
    loc_np = loc.cpu().numpy()
    g = gather_rows_torch(pool, O.FP4, 6, loc_np)
    o = _oracle_store_rows(O.FP4, 0, _bf16_np(x))
    assert (g[0] == o[0]).all() and (g[1] == o[1]).all()
    written = int(g[0].astype(np.int64).sum() + g[1].astype(np.int64).sum())
    assert int(pool.sum(dtype=torch.int64).item()) == written
    # dequant: every logical page, the oracle on host threads in chunks of pages
    pool_np = np_u8(pool)
    pt_np = pt.cpu().numpy()
    chunk = 1024
    spans = [(a, min(n_pages, a + chunk)) for a in range(0, n_pages, chunk)]

    def ref(ab):
        a, b = ab
        rc, ws = O.dequant(O.FP4, 6, pool_np, pt_np[a:b], (b - a) * 64)
        assert rc == O.OK
        return ws
    nonzero = 0
    for i in range(0, len(spans), 16):
        part = spans[i:i + 16]
        for (a, b), ws in zip(part, oracle_map(ref, part)):
            got = out[a * 64:b * 64].view(torch.int16)
            want = torch.from_numpy(ws.view(np.int16)).to(DEV)
            assert torch.equal(got, want), (a, b)
            nonzero += int(np.count_nonzero(ws))
    assert nonzero > 0


# --------------------------------------------------------------------------- C4A + translation

def test_translate_and_c4a(K):
    """65536 fp32 rows (values N(0,1), scores N(0,2)) in 16384 groups of 4;
    out_cache_loc injective into a 2^20-slot full pool, translated once to
    a 2^17-slot SWA pool; RoPE at positions 4g; V41 store."""
    from compress_kv_write_gb300 import synth
    G, r = 16384, 4
    full_slots, swa_slots = 1 << 20, 1 << 17
    v, s = synth.compressor_rows(G * r, DEV, 0, score_std=math.sqrt(2.0))
    full_loc = synth.injective_slots(G, full_slots, DEV, 0)
    table = synth.swa_table(full_slots, swa_slots, full_loc, DEV, 0)
    cap = G + 1000
    swa_loc = torch.full((cap,), 12345, dtype=torch.int32, device=DEV)
    err = _err(K)
    K.kvq_translate_loc(full_loc, table, swa_loc, err=err)
    gpos = (torch.arange(G, dtype=torch.int32, device=DEV) * r)
    cs = synth.rope_table(65536, DEV)
    pool = torch.zeros(swa_slots * 528, dtype=torch.uint8, device=DEV)
    K.kvq_compress(K.V41, 6, r, K.FLAG_ROPE, v, s, swa_loc[:G], pool, swa_slots, cos_sin=cs,
                   group_pos=gpos, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rc, tr = O.translate(full_loc.cpu().numpy(), table.cpu().numpy(), cap)
    assert rc == O.OK
    assert (swa_loc.cpu().numpy() == tr).all()
    slots = tr[:G]
    assert np.unique(slots).size == G
    v_np, s_np, cs_np = v.cpu().numpy(), s.cpu().numpy(), cs.cpu().numpy()
    pool_o = np.zeros(swa_slots * 528, np.uint8)
    rc = O.compress(O.V41, 6, r, O.ROPE, v_np, s_np, slots, pool_o, cos_sin=cs_np,
                    group_pos=gpos.cpu().numpy())
    assert rc == O.OK
    got = np_u8(pool)
    g = gather_rows(got, O.V41, 6, slots)
    o = gather_rows(pool_o, O.V41, 6, slots)
    y = group_prequant_many(r, O.ROPE, v_np, s_np, cs_np[np.arange(G) * r])
    check_tolerance(O.V41, g[0], g[1], o[0], o[1], y)
    written = int(g[0].astype(np.int64).sum() + g[1].astype(np.int64).sum())
    assert int(got.astype(np.int64).sum()) == written


@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("r", [1, 2, 4, 128])
def test_compress_small_exhaustive(K, layout, r):
    """Every compiled ratio on ragged group counts (1, 3, 45 and 97 groups),
    each launch compared with the oracle over the whole pool.  r = 1 is the
    identity (bit-exact); for r > 1 the groups of all four launches are
    pooled into one comparison under the 0.1% code budget."""
    from compress_kv_write_gb300 import synth
    slots = 512
    gc, gs_, oc, os_, ys = [], [], [], [], []
    for G in (1, 3, 45, 97):
        v, s = synth.compressor_rows(G * r, "cpu", G + r, score_std=2.0)
        loc = synth.injective_slots(G, slots, "cpu", G, dtype=torch.int32)
        gpos = synth.positions(G, "cpu", G, max_pos=1024)
        cs = synth.rope_table(1024, "cpu")
        pool_o = np.zeros(slots * O.bytes_per_token(layout), np.uint8)
        assert O.compress(layout, 6, r, O.ROPE, v.numpy(), s.numpy(), loc.numpy(), pool_o,
                          cos_sin=cs.numpy(), group_pos=gpos.numpy()) == O.OK
        pool = torch.zeros_like(torch.from_numpy(pool_o), device=DEV)
        err = _err(K)
        K.kvq_compress(layout, 6, r, K.FLAG_ROPE, v.to(DEV), s.to(DEV), loc.to(DEV), pool, slots,
                       cos_sin=cs.to(DEV), group_pos=gpos.to(DEV), err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        got = np_u8(pool)
        g = gather_rows(got, layout, 6, loc.numpy())
        o = gather_rows(pool_o, layout, 6, loc.numpy())
        if r == 1:   # r = 1 pooling is the identity: bit-exact
            assert (g[0] == o[0]).all() and (g[1] == o[1]).all()
        gc.append(g[0])
        gs_.append(g[1])
        oc.append(o[0])
        os_.append(o[1])
        ys.append(group_prequant_many(r, O.ROPE, v.numpy(), s.numpy(), cs.numpy()[gpos.numpy()]))
        written = int(g[0].astype(np.int64).sum() + g[1].astype(np.int64).sum())
        assert int(got.astype(np.int64).sum()) == written
    if r > 1:
        check_tolerance(layout, np.concatenate(gc), np.concatenate(gs_), np.concatenate(oc),
                        np.concatenate(os_), np.concatenate(ys))


# --------------------------------------------------------------------------- C128A mixed batch

@pytest.mark.parametrize("layout", [1, 2])
def test_c128a_mixed_batch(K, layout):
    """256 requests, log-uniform lengths in [128, 32768] (multiples of 128),
    values N(0,1), scores N(0,4); 128-row groups at positions 128 * local
    group index.  Every group is compared with the oracle (pooled on host
    threads, in chunks of groups copied back from the device)."""
    from compress_kv_write_gb300 import synth
    r = 128
    lens = synth.request_lengths(256, seed=0)
    gpos = synth.group_positions(lens, r).to(DEV)
    G = gpos.numel()
    pool_slots = 1 << 20
    v, s = synth.compressor_rows(G * r, DEV, 0, score_std=2.0)
    loc = synth.injective_slots(G, pool_slots, DEV, 0, dtype=torch.int32)
    cs = synth.rope_table(32768, DEV)
    pool = torch.zeros(pool_slots * O.bytes_per_token(layout), dtype=torch.uint8, device=DEV)
    err = _err(K)
    K.kvq_compress(layout, 6, r, K.FLAG_ROPE, v, s, loc, pool, pool_slots, cos_sin=cs,
                   group_pos=gpos, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    loc_np, gpos_np, cs_np = loc.cpu().numpy(), gpos.cpu().numpy(), cs.cpu().numpy()
    g = gather_rows_torch(pool, layout, 6, loc_np)
    ys = []
    step = 1024
    for a in range(0, G, step):
        b = min(G, a + step)
        vi = v[a * r:b * r].cpu().numpy()
        si = s[a * r:b * r].cpu().numpy()
        ys.append(group_prequant_many(r, O.ROPE, vi, si, cs_np[gpos_np[a:b]]))
    y = np.concatenate(ys)
    oc, osc = encode_many(layout, y)
    check_tolerance(layout, g[0], g[1], oc, osc, y)
    # nothing but the groups' rows was written
    written = int(g[0].astype(np.int64).sum() + g[1].astype(np.int64).sum())
    assert int(pool.sum(dtype=torch.int64).item()) == written


# --------------------------------------------------------------------------- error paths

def test_error_paths(K):
    from compress_kv_write_gb300 import synth
    x = synth.store_rows_bf16(4, DEV, 1)
    pool = torch.zeros(64 * 528, dtype=torch.uint8, device=DEV)
    # n = 0 enqueues nothing
    K.kvq_store(K.V41, 6, 0, x[:0], torch.zeros(0, dtype=torch.int64, device=DEV), pool, 64)
    # out-of-range slots: flagged and skipped, the other rows written
    err = _err(K)
    loc = torch.tensor([3, 64, -5, 7], device=DEV)
    K.kvq_store(K.V41, 6, 0, x, loc, pool, 64, err=err)
    torch.cuda.synchronize()
    assert err.item() == K.kvq.DEVERR_SLOT
    ref = np.zeros(64 * 528, np.uint8)
    O.store(O.V41, 6, 0, _bf16_np(x), np.array([3, 64, -5, 7]), ref)
    assert (np_u8(pool) == ref).all()
    # out-of-range RoPE position
    err.zero_()
    pool.zero_()
    cs = synth.rope_table(16, DEV)
    K.kvq_store(K.V41, 6, K.FLAG_ROPE, x, torch.tensor([0, 1, 2, 3], device=DEV), pool, 64,
                cos_sin=cs, pos=torch.tensor([0, 16, 3, -1], dtype=torch.int32, device=DEV), err=err)
    torch.cuda.synchronize()
    assert err.item() == K.kvq.DEVERR_POS
    g = gather_rows(np_u8(pool), O.V41, 6, np.arange(4))
    assert (g[1][[1, 3]] == 0).all() and (g[1][[0, 2]] != 0).any()
    # the same two checks on the FP4 layout, with the norm: bad rows flagged and skipped
    for flags, loc_, pos_, bit in ((K.FLAG_NORM, [3, 64, -5, 7], None, K.kvq.DEVERR_SLOT),
                                   (K.FLAG_NORM | K.FLAG_ROPE, [0, 1, 2, 3], [0, 16, 3, -1], K.kvq.DEVERR_POS)):
        err.zero_()
        fpool = torch.zeros(64 * 288, dtype=torch.uint8, device=DEV)
        w = synth.norm_weight(DEV, 1)
        K.kvq_store(K.V41_FP4, 6, flags, x, torch.tensor(loc_, device=DEV), fpool, 64, norm_weight=w, eps=1e-6,
                    cos_sin=cs if pos_ else None,
                    pos=torch.tensor(pos_, dtype=torch.int32, device=DEV) if pos_ else None, err=err)
        torch.cuda.synchronize()
        assert err.item() == bit
        ref = np.zeros(64 * 288, np.uint8)
        O.store(O.FP4, 6, flags, _bf16_np(x), np.array(loc_), ref, norm_weight=w.cpu().numpy(), eps=1e-6,
                cos_sin=cs.cpu().numpy() if pos_ else None, pos=np.array(pos_, np.int32) if pos_ else None)
        got = np_u8(fpool)
        assert ((got != 0) == (ref != 0)).mean() > 0.99   # the same rows written (norm: within tolerance)
        if pos_:
            gf = gather_rows(got, O.FP4, 6, np.arange(4))
            assert (gf[1][[1, 3]] == 0).all() and (gf[0][[1, 3]] == 0).all()
        else:
            gf = gather_rows(got, O.FP4, 6, np.array([3, 7]))
            assert (gf[1][:, :16] != 0).any()
    # bad page-table entry: flagged, that page untouched
    err.zero_()
    out = torch.full((128, 512), 7.0, dtype=torch.bfloat16, device=DEV)
    K.kvq_dequant(K.V41, 6, pool, 1, torch.tensor([0, 1], dtype=torch.int32, device=DEV), out, err=err)
    torch.cuda.synchronize()
    assert err.item() == K.kvq.DEVERR_PAGE
    assert (out[64:] == 7.0).all()
    # translation: capacity error enqueues nothing; bad locs -> -1
    outb = torch.full((4,), 99, dtype=torch.int32, device=DEV)
    with pytest.raises(K.KVQError) as e:
        K.kvq_translate_loc(torch.arange(5, device=DEV), torch.arange(8, dtype=torch.int32, device=DEV), outb)
    assert e.value.status == K.kvq.ERR_CAPACITY
    torch.cuda.synchronize()
    assert (outb == 99).all()
    err.zero_()
    K.kvq_translate_loc(torch.tensor([1, 9, -1], dtype=torch.int32, device=DEV),
                        torch.arange(8, dtype=torch.int32, device=DEV) * 2, outb, err=err)
    torch.cuda.synchronize()
    assert outb.cpu().tolist() == [2, -1, -1, 0]
    assert err.item() == K.kvq.DEVERR_LOC


# --------------------------------------------------------------------------- one step across layers

def test_step_translates_once_for_all_layers(K):
    """One decode step of a 3-layer model: the step's full-pool slots are
    translated to SWA slots once and every layer's store uses them.  The pools
    equal those written with the translation repeated inside every layer, and
    each layer equals the oracle (RoPE store: bit-exact)."""
    from compress_kv_write_gb300 import synth
    L, n, full_slots, swa_slots = 3, 200, 1 << 14, 1 << 10
    full_loc = synth.injective_slots(n, full_slots, DEV, 5)
    table = synth.swa_table(full_slots, swa_slots, full_loc, DEV, 5)
    xs = [synth.store_rows_bf16(n, DEV, 50 + l) for l in range(L)]
    pos = synth.positions(n, DEV, 5, max_pos=4096)
    cs = synth.rope_table(4096, DEV)
    swa = torch.zeros(n, dtype=torch.int32, device=DEV)
    hoisted = [torch.zeros(swa_slots * 528, dtype=torch.uint8, device=DEV) for _ in range(L)]
    per_layer = [torch.zeros(swa_slots * 528, dtype=torch.uint8, device=DEV) for _ in range(L)]
    err = _err(K)
    K.kvq_translate_loc(full_loc, table, swa, err=err)
    for l in range(L):
        K.kvq_store(K.V41, 6, K.FLAG_ROPE, xs[l], swa, hoisted[l], swa_slots, cos_sin=cs, pos=pos, err=err)
    for l in range(L):
        swa_l = torch.full((n,), -7, dtype=torch.int32, device=DEV)
        K.kvq_translate_loc(full_loc, table, swa_l, err=err)
        K.kvq_store(K.V41, 6, K.FLAG_ROPE, xs[l], swa_l, per_layer[l], swa_slots, cos_sin=cs, pos=pos, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rc, tr = O.translate(full_loc.cpu().numpy(), table.cpu().numpy(), n)
    assert rc == O.OK
    for l in range(L):
        assert torch.equal(hoisted[l], per_layer[l])
        ref = np.zeros(swa_slots * 528, np.uint8)
        assert O.store(O.V41, 6, O.ROPE, _bf16_np(xs[l]), tr, ref, cos_sin=cs.cpu().numpy(),
                       pos=pos.cpu().numpy()) == O.OK
        assert (np_u8(hoisted[l]) == ref).all()


# --------------------------------------------------------------------------- selected-slot dequant

@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("page_bits", [2, 6])
def test_dequant_slots_small(K, layout, page_bits):
    """Random, repeated, padding (-1) and out-of-range slots: bit-exact rows,
    untouched rows for bad slots, the slot error bit set."""
    from compress_kv_write_gb300 import synth
    slots_n = 512
    x = synth.student_t_rows_bf16(300, "cpu", 9)
    loc = synth.injective_slots(300, slots_n, "cpu", 9)
    pool_o = np.zeros(slots_n * O.bytes_per_token(layout), np.uint8)
    assert O.store(layout, page_bits, 0, _bf16_np(x), loc.numpy(), pool_o) == O.OK
    pool = torch.from_numpy(pool_o).to(DEV)
    rng = np.random.default_rng(layout * 10 + page_bits)
    for idx_dtype in (torch.int32, torch.int64):
        sel = rng.integers(0, slots_n, 203)
        sel[[3, 50, 51]] = -1
        sel[[7, 100]] = [slots_n, -5]
        slots = torch.as_tensor(sel, dtype=idx_dtype, device=DEV)
        out = torch.full((sel.size, 512), 3.0, dtype=torch.bfloat16, device=DEV)
        err = _err(K)
        K.kvq_dequant_slots(layout, page_bits, pool, slots_n, slots, out, err=err)
        torch.cuda.synchronize()
        assert err.item() == K.kvq.DEVERR_SLOT
        ref_out = np.full((sel.size, 512), O.bf16_bits(np.float32(3.0)), np.uint16)
        rc, ref = O.dequant_slots(layout, pool_o, sel, page_bits, out=ref_out)
        assert rc == O.ERANGE
        assert (_bf16_np(out) == ref).all()


def test_dequant_slots_fp4_pool_2m(K):
    """262144 selected slots of a full 2^21-slot FP4 pool (every slot written)."""
    from compress_kv_write_gb300 import synth
    pool_slots, n = 1 << 21, 1 << 18
    pool = torch.zeros(pool_slots * 288, dtype=torch.uint8, device=DEV)
    chunk = 1 << 18
    x = synth.student_t_rows_bf16(chunk, DEV, 3)
    for c in range(pool_slots // chunk):
        K.kvq_store(K.V41_FP4, 6, 0, x, torch.arange(c * chunk, (c + 1) * chunk, device=DEV), pool, pool_slots)
    sel = synth.injective_slots(n, pool_slots, DEV, 4)
    out = torch.empty((n, 512), dtype=torch.bfloat16, device=DEV)
    err = _err(K)
    K.kvq_dequant_slots(K.V41_FP4, 6, pool, pool_slots, sel, out, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    sel_np = sel.cpu().numpy()
    pool_np = np_u8(pool)
    spans = [(a, min(n, a + 8192)) for a in range(0, n, 8192)]

    def ref(ab):
        rc, r_ = O.dequant_slots(O.FP4, pool_np, sel_np[ab[0]:ab[1]], 6)
        assert rc == O.OK
        return r_
    want = np.concatenate(oracle_map(ref, spans))
    assert (_bf16_np(out) == want).all()


# --------------------------------------------------------------------------- more page sizes

@pytest.mark.parametrize("page_bits", [4, 8])
@pytest.mark.parametrize("layout", [1, 2])
def test_page_sizes_16_and_256(K, page_bits, layout):
    """Pages of 16 and 256 tokens: store + RoPE (batches of 300, 1100 and 3200
    rows: one CTA per token, two tokens per CTA, the persistent kernels),
    ratio-1 compressor (identity, bit-exact), paged dequant through a
    permuted page table and the selected-slot dequant, all against the
    oracle."""
    from compress_kv_write_gb300 import synth
    P = 1 << page_bits
    pages = max(8, 9216 // P)
    slots = pages * P
    n = 4600
    x = synth.store_rows_bf16(n, "cpu", page_bits)
    loc = synth.injective_slots(n, slots, "cpu", page_bits)
    cs = synth.rope_table(1024, "cpu")
    pos = synth.positions(n, "cpu", page_bits, max_pos=1024)
    pool_o = np.zeros(slots * O.bytes_per_token(layout), np.uint8)
    assert O.store(layout, page_bits, O.ROPE, _bf16_np(x), loc.numpy(), pool_o, cos_sin=cs.numpy(),
                   pos=pos.numpy()) == O.OK
    g = 20
    v, s = synth.compressor_rows(g, "cpu", page_bits)
    cloc = torch.as_tensor(np.setdiff1d(np.arange(slots), loc.numpy())[:g], dtype=torch.int32)
    assert O.compress(layout, page_bits, 1, 0, v.numpy(), s.numpy(), cloc.numpy(), pool_o) == O.OK
    pool = torch.zeros(slots * O.bytes_per_token(layout), dtype=torch.uint8, device=DEV)
    err = _err(K)
    for b0, b1 in ((0, 300), (300, 1400), (1400, n)):
        K.kvq_store(layout, page_bits, K.FLAG_ROPE, x[b0:b1].to(DEV), loc[b0:b1].to(DEV), pool, slots,
                    cos_sin=cs.to(DEV), pos=pos[b0:b1].to(DEV), err=err)
    K.kvq_compress(layout, page_bits, 1, 0, v.to(DEV), s.to(DEV), cloc.to(DEV), pool, slots, err=err)
    pt = synth.page_table_perm(pages, "cpu", page_bits)
    ws = torch.empty((slots, 512), dtype=torch.bfloat16, device=DEV)
    K.kvq_dequant(layout, page_bits, pool, pages, pt.to(DEV), ws, err=err)
    sel = torch.as_tensor(np.random.default_rng(page_bits).integers(-1, slots, 97), dtype=torch.int64)
    gs = torch.empty((97, 512), dtype=torch.bfloat16, device=DEV)
    K.kvq_dequant_slots(layout, page_bits, pool, slots, sel.to(DEV), gs, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert (np_u8(pool) == pool_o).all()
    rc, ref = O.dequant(layout, page_bits, pool_o, pt.numpy(), slots)
    assert rc == O.OK and (_bf16_np(ws) == ref).all()
    rc, ref = O.dequant_slots(layout, pool_o, sel.numpy(), page_bits)
    assert rc == O.OK and (_bf16_np(gs) == ref).all()


# --------------------------------------------------------------------------- decode-time compressor

@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("r,wide", [(1, False), (2, False), (4, False), (128, False), (1, True), (2, True),
                                    (4, True)])
def test_compress_decode_streams(K, layout, r, wide):
    """Rows arrive one per call to a random subset of request slots, in random
    order (state indexed through req); every group a slot completes is
    compared with the oracle's pooling of that group's r rows.  r = 1 is the
    identity (bit-exact); the others follow the pooling tolerance (0.1% code
    budget over all completed groups: 16 to 48 request slots, so that every
    ratio completes dozens of groups).  The wide cases send all 1100 request
    slots a row in every call (1100 CTAs, some SMs holding several)."""
    rng = np.random.default_rng(100 * layout + r + (7 if wide else 0))
    n_state = 1100 if wide else (48 if r < 128 else 16)
    calls = 3 * r + 2 if r < 128 else 2 * r + 3
    pool_slots = max(1024, -(-calls * n_state // 64) * 64)  # a fresh destination per row
    from compress_kv_write_gb300 import synth
    cs = synth.rope_table(2048, DEV)
    cs_np = cs.cpu().numpy()
    state = torch.zeros((n_state, 3, 512), dtype=torch.float32, device=DEV)
    count = torch.zeros(n_state, dtype=torch.int32, device=DEV)
    pool = torch.zeros(pool_slots * O.bytes_per_token(layout), dtype=torch.uint8, device=DEV)
    err = _err(K)
    seen = [[] for _ in range(n_state)]  # rows each slot has received: (v, s)
    groups = []                           # (slot, first row index, dest slot, pos)
    free_slots = list(rng.permutation(pool_slots))
    for call in range(calls):
        active = np.flatnonzero(rng.random(n_state) < (0.8 if r < 128 and not wide else 1.0))
        if active.size == 0:
            continue
        req = rng.permutation(active).astype(np.int32)
        v = rng.standard_normal((req.size, 512)).astype(np.float32)
        s = (rng.standard_normal((req.size, 512)) * 2).astype(np.float32)
        loc = np.empty(req.size, np.int32)
        gpos = np.empty(req.size, np.int32)
        for j, rs in enumerate(req):
            k = len(seen[rs])
            seen[rs].append((v[j], s[j]))
            loc[j] = free_slots.pop()
            gpos[j] = (k // r) * r % 2048
            if k % r == r - 1:
                groups.append((rs, k - r + 1, loc[j], gpos[j]))
        K.kvq_compress_decode(layout, 6, r, K.FLAG_ROPE, torch.from_numpy(v).to(DEV), torch.from_numpy(s).to(DEV),
                              state, count, torch.from_numpy(loc).to(DEV), pool, pool_slots,
                              req=torch.from_numpy(req).to(DEV), cos_sin=cs, group_pos=torch.from_numpy(gpos).to(DEV),
                              err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert groups, "some groups completed"
    assert (count.cpu().numpy() == np.array([len(x) % r for x in seen])).all()
    got = np_u8(pool)
    g = gather_rows(got, layout, 6, [x[2] for x in groups])
    oc, osc, ys = [], [], []
    for rs, k0, dst, pos in groups:
        vv = np.stack([seen[rs][k][0] for k in range(k0, k0 + r)])
        ss = np.stack([seen[rs][k][1] for k in range(k0, k0 + r)])
        c_, s_ = O.group_bytes(layout, r, O.ROPE, vv, ss, cs_np[pos])
        oc.append(c_)
        osc.append(s_)
        ys.append(O.group_prequant(r, O.ROPE, vv, ss, cs_np[pos]))
    oc, osc = np.stack(oc), np.stack(osc)
    if r == 1:
        assert (g[0] == oc).all() and (g[1] == osc).all()
    else:
        check_tolerance(layout, g[0], g[1], oc, osc, np.stack(ys))
    written = int(g[0].astype(np.int64).sum() + g[1].astype(np.int64).sum())
    assert int(got.astype(np.int64).sum()) == written  # open groups wrote nothing


def test_compress_decode_bad_state_index(K):
    state = torch.zeros((2, 3, 512), dtype=torch.float32, device=DEV)
    count = torch.tensor([0, 7], dtype=torch.int32, device=DEV)  # slot 1: count >= ratio
    pool = torch.zeros(64 * 528, dtype=torch.uint8, device=DEV)
    v = torch.ones((3, 512), device=DEV)
    err = _err(K)
    K.kvq_compress_decode(K.V41, 6, 4, 0, v, v, state, count, torch.tensor([1, 2, 3], dtype=torch.int32, device=DEV),
                          pool, 64, req=torch.tensor([0, 1, 5], dtype=torch.int32, device=DEV), err=err)
    torch.cuda.synchronize()
    assert err.item() == K.kvq.DEVERR_STATE
    assert count.cpu().tolist() == [1, 7]
    assert int(pool.sum().item()) == 0


# --------------------------------------------------------------------------- strided rows

@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("flags", [0, 1, 3])
def test_store_strided_rows(K, layout, dtype, flags):
    """x is the K slice of a wider projection: 512 columns at a 128-byte offset
    inside wider rows (x_row_stride > 512).  The pool must hold the bytes the
    oracle writes from the contiguous copy of the same rows.  3500 rows in
    three calls of 100, 300 and 3100 rows: every store mapping."""
    from compress_kv_write_gb300 import synth
    n, slots = 3500, 4096
    seed = 900 + layout * 10 + flags
    xc = synth.store_rows_bf16(n, "cpu", seed)
    if dtype == "f32":
        xc = xc.float() * 1.25
    pad = 128 // xc.element_size()
    wide = torch.zeros((n, 512 + 3 * pad), dtype=xc.dtype)
    wide[:, pad:pad + 512] = xc
    x = wide.to(DEV)[:, pad:pad + 512]
    assert x.stride(0) == 512 + 3 * pad and not x.is_contiguous()
    loc = synth.injective_slots(n, slots, "cpu", seed)
    w = synth.norm_weight("cpu", seed)
    cs = synth.rope_table(4096, "cpu")
    pos = synth.positions(n, "cpu", seed, max_pos=4096)
    x_np = xc.numpy() if dtype == "f32" else _bf16_np(xc)
    pool_o = np.zeros(slots * O.bytes_per_token(layout), np.uint8)
    assert O.store(layout, 6, flags, x_np, loc.numpy(), pool_o, norm_weight=w.numpy(), eps=1e-6,
                   cos_sin=cs.numpy(), pos=pos.numpy()) == O.OK
    pool = torch.zeros(slots * O.bytes_per_token(layout), dtype=torch.uint8, device=DEV)
    err = _err(K)
    for b0, b1 in ((0, 100), (100, 400), (400, n)):
        xb = x[b0:b1]
        assert xb.stride(0) == 512 + 3 * pad
        K.kvq_store(layout, 6, flags, xb, loc[b0:b1].to(DEV), pool, slots,
                    norm_weight=w.to(DEV) if flags & 2 else None, eps=1e-6,
                    cos_sin=cs.to(DEV) if flags & 1 else None, pos=pos[b0:b1].to(DEV) if flags & 1 else None,
                    err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = np_u8(pool)
    if flags & 2 == 0:
        assert (got == pool_o).all()
    else:
        g = gather_rows(got, layout, 6, loc.numpy())
        o = gather_rows(pool_o, layout, 6, loc.numpy())
        y = np.stack([O.token_prequant(flags, x_np[t], w.numpy(), 1e-6, cs.numpy()[pos[t]]) for t in range(n)])
        check_tolerance(layout, g[0], g[1], o[0], o[1], y)


@pytest.mark.parametrize("layout", [1, 2])
def test_dequant_into_strided_workspace(K, layout):
    """Both dequants write into 512 columns of a wider bf16 workspace; the
    columns around them stay untouched."""
    from compress_kv_write_gb300 import synth
    slots, n = 256, 256
    x = synth.store_rows_bf16(n, "cpu", 31)
    loc = synth.injective_slots(n, slots, "cpu", 31)
    pool_o = np.zeros(slots * O.bytes_per_token(layout), np.uint8)
    assert O.store(layout, 6, 0, _bf16_np(x), loc.numpy(), pool_o) == O.OK
    pool = torch.from_numpy(pool_o).to(DEV)
    pt = synth.page_table_perm(4, "cpu", 31)
    rc, ws_o = O.dequant(layout, 6, pool_o, pt.numpy(), slots)
    assert rc == O.OK
    sel = torch.tensor([3, -1, 200, 77, 0, 255], dtype=torch.int64)
    rc, sel_o = O.dequant_slots(layout, pool_o, sel.numpy())
    assert rc == O.OK
    sentinel = torch.tensor([0x7E11], dtype=torch.int16).view(torch.bfloat16)
    for out_rows, run, ref in ((slots, lambda o, e: K.kvq_dequant(layout, 6, pool, 4, pt.to(DEV), o, err=e), ws_o),
                               (6, lambda o, e: K.kvq_dequant_slots(layout, 6, pool, slots, sel.to(DEV), o, err=e),
                                sel_o)):
        wide = sentinel.expand(out_rows, 512 + 3 * 64).contiguous().to(DEV)
        err = _err(K)
        run(wide[:, 64:576], err)
        torch.cuda.synchronize()
        assert err.item() == 0
        w16 = wide.cpu().view(torch.int16).numpy().view(np.uint16)
        assert (w16[:, 64:576] == ref).all()
        assert (w16[:, :64] == 0x7E11).all() and (w16[:, 576:] == 0x7E11).all()


@pytest.mark.parametrize("flags", [0, 1, 3])
def test_store_many_tokens_per_warp(K, flags):
    """262144 V41 tokens: every warp of the persistent grid holds more than 32
    tokens, so the per-lane slot / position batches are reloaded inside the
    loop; the whole pool must match the oracle."""
    from compress_kv_write_gb300 import synth
    n, slots = 1 << 18, 1 << 20
    x = synth.store_rows_bf16(n, DEV, 7)
    loc = synth.injective_slots(n, slots, DEV, 7)
    pos = synth.positions(n, DEV, 7)
    cs = synth.rope_table(65536, DEV)
    w = synth.norm_weight(DEV, 7)
    pool = torch.zeros(slots * 528, dtype=torch.uint8, device=DEV)
    err = _err(K)
    K.kvq_store(K.V41, 6, flags, x, loc, pool, slots, norm_weight=w, eps=1e-6, cos_sin=cs, pos=pos, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    x_np, loc_np, pos_np = _bf16_np(x), loc.cpu().numpy(), pos.cpu().numpy()
    cs_np, w_np = cs.cpu().numpy(), w.cpu().numpy()
    pool_o = np.zeros(slots * 528, np.uint8)
    assert O.store(O.V41, 6, flags, x_np, loc_np, pool_o, norm_weight=w_np, eps=1e-6, cos_sin=cs_np,
                   pos=pos_np) == O.OK
    got = np_u8(pool)
    if flags & 2 == 0:
        assert (got == pool_o).all()
    else:
        g = gather_rows(got, O.V41, 6, loc_np)
        o = gather_rows(pool_o, O.V41, 6, loc_np)
        y = token_prequant_many(flags, x_np, w_np, 1e-6, cs_np[pos_np])
        check_tolerance(O.V41, g[0], g[1], o[0], o[1], y)


# --------------------------------------------------------------------------- hand-worked blocks

def test_kernels_reproduce_handworked_blocks(K):
    """Every hand-worked block of tests/golden, stored by the CUDA store kernels
    (fp32 input, no fused math) in quant blocks 0, 9 and 15 of its own token:
    the code and scale bytes must be the hand-derived ones, and the paged
    dequant must give the hand-derived values.  The batch runs alone (one
    CTA per token) and tiled into every other store mapping (two tokens per
    CTA, the persistent kernels; the first copy is checked)."""
    from golden_io import load_blocks
    for layout, fname, tiled in ((O.V41, "v41_blocks.txt", 0), (O.FP4, "fp4_blocks.txt", 0),
                                 (O.V41, "v41_blocks.txt", 1), (O.FP4, "fp4_blocks.txt", 1),
                                 (O.V41, "v41_blocks.txt", 2), (O.FP4, "fp4_blocks.txt", 2)):
        cases = load_blocks(fname)
        blocks = (0, 9, 15)
        n1 = len(cases) * len(blocks)
        x = np.zeros((n1, 512), np.float32)
        for ci, (_, vals, _, _, _) in enumerate(cases):
            for bi, blk in enumerate(blocks):
                x[ci * len(blocks) + bi, blk * 32:(blk + 1) * 32] = vals
        x = _all_mappings(x)[tiled]
        n = x.shape[0]
        slots = max(64, -(-n // 64) * 64)
        pool = torch.zeros(slots * O.bytes_per_token(layout), dtype=torch.uint8, device=DEV)
        loc = torch.arange(n, dtype=torch.int64, device=DEV)
        err = _err(K)
        K.kvq_store(layout, 6, 0, torch.from_numpy(x).to(DEV), loc, pool, slots, err=err)
        out = torch.empty((slots, 512), dtype=torch.bfloat16, device=DEV)
        K.kvq_dequant(layout, 6, pool, slots // 64, torch.arange(slots // 64, dtype=torch.int32, device=DEV),
                      out, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        codes, scales = gather_rows(np_u8(pool), layout, 6, np.arange(n))
        deq = out.float().cpu().numpy()
        if tiled:  # every copy of the batch stored alike
            assert (codes == np.tile(codes[:n1], (n // n1, 1))).all()
            assert (scales == np.tile(scales[:n1], (n // n1, 1))).all()
        cpb = 32 if layout == O.V41 else 16          # code bytes per quant block
        for ci, (name, _, scale, cbytes, dvals) in enumerate(cases):
            for bi, blk in enumerate(blocks):
                t = ci * len(blocks) + bi
                assert scales[t, blk] == scale, (name, blk)
                assert (np.delete(scales[t, :16], blk) == 0).all(), name
                if layout == O.FP4:
                    assert (scales[t, 16:] == 0).all(), name
                cb = codes[t, blk * cpb:(blk + 1) * cpb]
                for j in range(cpb):
                    assert cb[j] == cbytes.get(j, 0x00), (name, blk, j, hex(cb[j]))
                for i, v in dvals.items():
                    assert deq[t, blk * 32 + i] == np.float32(v), (name, blk, i, deq[t, blk * 32 + i], v)


@pytest.mark.parametrize("flags", [0, 1, 3])
def test_bad_rows_in_a_large_batch(K, flags):
    """20000 V41 tokens (several per warp, so the staggered first copy and, for
    norm + RoPE, the one-warp CTAs are in play) with out-of-range slots and
    positions scattered through the batch: the error word carries the flags,
    the bad rows write nothing and every other row matches the oracle."""
    from compress_kv_write_gb300 import synth
    n, slots = 20000, 1 << 16
    x = synth.store_rows_bf16(n, "cpu", 11)
    loc = synth.injective_slots(n, slots, "cpu", 11)
    pos = synth.positions(n, "cpu", 11, max_pos=4096)
    bad_slot = np.arange(17, n, 997)
    loc[bad_slot[0::2]] = slots          # one past the end
    loc[bad_slot[1::2]] = -3
    bad_pos = np.arange(500, n, 1511) if flags & 1 else np.array([], np.int64)
    pos[bad_pos] = 4096                  # one past the table
    cs = synth.rope_table(4096, "cpu")
    w = synth.norm_weight("cpu", 11)
    pool = torch.zeros(slots * 528, dtype=torch.uint8, device=DEV)
    err = _err(K)
    K.kvq_store(K.V41, 6, flags, x.to(DEV), loc.to(DEV), pool, slots, norm_weight=w.to(DEV), eps=1e-6,
                cos_sin=cs.to(DEV), pos=pos.to(DEV), err=err)
    torch.cuda.synchronize()
    want = K.kvq.DEVERR_SLOT | (K.kvq.DEVERR_POS if flags & 1 else 0)
    assert err.item() == want
    good = np.setdiff1d(np.arange(n), np.union1d(bad_slot, bad_pos))
    x_np = _bf16_np(x)
    pool_o = np.zeros(slots * 528, np.uint8)
    assert O.store(O.V41, 6, flags, x_np[good], loc.numpy()[good], pool_o, norm_weight=w.numpy(), eps=1e-6,
                   cos_sin=cs.numpy(), pos=pos.numpy()[good]) == O.OK
    got = np_u8(pool)
    if flags & 2 == 0:
        assert (got == pool_o).all()
    else:
        g = gather_rows(got, O.V41, 6, loc.numpy()[good])
        o = gather_rows(pool_o, O.V41, 6, loc.numpy()[good])
        y = token_prequant_many(flags, x_np[good], w.numpy(), 1e-6, cs.numpy()[pos.numpy()[good]])
        check_tolerance(O.V41, g[0], g[1], o[0], o[1], y)
        # nothing outside the good rows' slots was written
        mask = np.zeros(slots, bool)
        mask[loc.numpy()[good]] = True
        cz, sz = gather_rows(got, O.V41, 6, np.flatnonzero(~mask))
        assert (cz == 0).all() and (sz == 0).all()


@pytest.mark.parametrize("flags", [0, 1])
def test_fp4_bad_rows_in_a_large_batch(K, flags):
    """The FP4 half-warp kernel on 20000 tokens (several pairs per warp, so the
    staggered first copy is in play) with out-of-range slots and positions:
    flagged, skipped, and every other row bit-exact to the oracle."""
    from compress_kv_write_gb300 import synth
    n, slots = 20000, 1 << 16
    bpt = O.bytes_per_token(O.FP4)
    x = synth.student_t_rows_bf16(n, "cpu", 13)
    loc = synth.injective_slots(n, slots, "cpu", 13)
    pos = synth.positions(n, "cpu", 13, max_pos=4096)
    bad_slot = np.arange(29, n, 1009)
    loc[bad_slot] = slots + 5
    bad_pos = np.arange(300, n, 1213) if flags & 1 else np.array([], np.int64)
    pos[bad_pos] = -1
    cs = synth.rope_table(4096, "cpu")
    pool = torch.zeros(slots * bpt, dtype=torch.uint8, device=DEV)
    err = _err(K)
    K.kvq_store(K.V41_FP4, 6, flags, x.to(DEV), loc.to(DEV), pool, slots, cos_sin=cs.to(DEV), pos=pos.to(DEV),
                err=err)
    torch.cuda.synchronize()
    assert err.item() == K.kvq.DEVERR_SLOT | (K.kvq.DEVERR_POS if flags & 1 else 0)
    good = np.setdiff1d(np.arange(n), np.union1d(bad_slot, bad_pos))
    pool_o = np.zeros(slots * bpt, np.uint8)
    assert O.store(O.FP4, 6, flags, _bf16_np(x)[good], loc.numpy()[good], pool_o, cos_sin=cs.numpy(),
                   pos=pos.numpy()[good]) == O.OK
    assert (np_u8(pool) == pool_o).all()
