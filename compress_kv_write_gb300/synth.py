"""Seeded synthetic inputs for the KV write path (tests and benchmark).

This module only draws inputs; it holds none of the write path's arithmetic.
Every tensor comes from its own torch.Generator stream, seeded from
(seed, stream id), on the device the caller names, so a workload is the same
wherever it is drawn on the same device type.  Shapes and distributions
follow the workloads of the write path:

* store rows: bf16 [n, 512] ~ N(0, 1) with 1% of elements x50 (outliers);
  fp32 [n, 512] ~ N(0, 1) for the small fp32 store.
* K RMSNorm weight ~ N(1, 0.1), eps 1e-6.
* RoPE: positions uniform in [0, 65536); fp32 cos/sin table [rows, 64]
  (32 cosines then 32 sines of pos * 10000^(-2i/64)), built in float64.
* FP4 rows: bf16 0.5 * Student-t(nu = 3).
* compressor rows: fp32 values ~ N(0, 1), scores ~ N(0, sigma^2).
* slots: a random injective map into the pool (a prefix of a permutation).
* full -> SWA table: random int32 entries, made injective on the slots a
  step uses.
* mixed C128A batch: request lengths log-uniform in [128, 32768], rounded to
  multiples of 128.
"""
from __future__ import annotations

import math

import torch

STREAM = {
    "x": 1, "values": 2, "scores": 3, "pos": 4, "loc": 5, "table": 6, "weight": 7,
    "outlier": 8, "lens": 9, "page_table": 10, "swa_perm": 11, "chi2": 12,
}


def generator(device, seed: int, stream: str) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed((int(seed) * 1_000_003 + STREAM[stream]) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal(shape, device, seed, stream, std=1.0, mean=0.0, dtype=torch.float32):
    g = generator(device, seed, stream)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def store_rows_bf16(n, device, seed=0, outlier_p=0.01, outlier_scale=50.0):
    """bf16 [n, 512] ~ N(0, 1); each element independently x50 with p = 0.01."""
    x = normal((n, 512), device, seed, "x")
    g = generator(device, seed, "outlier")
    mask = torch.rand((n, 512), generator=g, device=device) < outlier_p
    x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def student_t_rows_bf16(n, device, seed=0, nu=3, scale=0.5):
    """bf16 [n, 512] = scale * Z / sqrt(chi2_nu / nu)."""
    z = normal((n, 512), device, seed, "x")
    g = generator(device, seed, "chi2")
    chi2 = torch.zeros((n, 512), device=device)
    for _ in range(nu):
        w = torch.randn((n, 512), generator=g, device=device)
        chi2.add_(w * w)
    return (scale * z / torch.sqrt(chi2 / nu)).to(torch.bfloat16)


def norm_weight(device, seed=0):
    return normal((512,), device, seed, "weight", std=0.1, mean=1.0)


def positions(n, device, seed=0, max_pos=65536):
    g = generator(device, seed, "pos")
    return torch.randint(0, max_pos, (n,), generator=g, device=device, dtype=torch.int32)


def rope_table(rows, device, theta=10000.0, rope_dim=64):
    """fp32 [rows, rope_dim]: cos then sin of pos * theta^(-2i/rope_dim), i < rope_dim/2."""
    half = rope_dim // 2
    inv_freq = theta ** (-torch.arange(half, dtype=torch.float64) * 2.0 / rope_dim)
    ang = torch.arange(rows, dtype=torch.float64)[:, None] * inv_freq[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32).to(device)


def injective_slots(n, pool_slots, device, seed=0, stream="loc", dtype=torch.int64):
    """n distinct slots in [0, pool_slots), in random order."""
    if n > pool_slots:
        raise ValueError("more rows than pool slots")
    g = generator(device, seed, stream)
    return torch.randperm(pool_slots, generator=g, device=device)[:n].to(dtype)


def page_table_perm(n_pages, device, seed=0):
    g = generator(device, seed, "page_table")
    return torch.randperm(n_pages, generator=g, device=device).to(torch.int32)


def swa_table(full_slots, swa_slots, used_full, device, seed=0):
    """int32 [full_slots] of SWA slots, distinct on the entries in used_full."""
    g = generator(device, seed, "table")
    tab = torch.randint(0, swa_slots, (full_slots,), generator=g, device=device, dtype=torch.int32)
    g2 = generator(device, seed, "swa_perm")
    perm = torch.randperm(swa_slots, generator=g2, device=device)[: used_full.numel()]
    tab[used_full.long()] = perm.to(torch.int32)
    return tab


def compressor_rows(n_rows, device, seed=0, score_std=math.sqrt(2.0)):
    """fp32 values ~ N(0, 1) and scores ~ N(0, score_std^2), [n_rows, 512] each."""
    v = normal((n_rows, 512), device, seed, "values")
    s = normal((n_rows, 512), device, seed, "scores", std=score_std)
    return v, s


def request_lengths(n_requests=256, lo=128, hi=32768, multiple=128, seed=0):
    """Log-uniform lengths in [lo, hi], rounded to a multiple, drawn on the CPU."""
    g = generator("cpu", seed, "lens")
    u = torch.rand(n_requests, generator=g, dtype=torch.float64)
    raw = lo * (hi / lo) ** u
    lens = (torch.round(raw / multiple) * multiple).clamp(lo, hi).to(torch.int64)
    return lens


def group_positions(lengths, ratio):
    """Position of each ratio-group: ratio * (its index inside its request)."""
    parts = [torch.arange(int(L) // ratio, dtype=torch.int32) * ratio for L in lengths]
    return torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int32)
