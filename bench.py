"""Benchmark of the GB300 KV-cache write path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the write path over one batch of synthetic input.  With
no --workload the headline is the mixed C128A compressor (256 requests of
log-uniform length, about 1.5 M fp32 value + score rows pooled 128 to one
into a V41 pool: the largest configuration of the path), and every other
configured workload is timed in the same run and reported under
"workloads": the small fp32 store + dequant, the store / store + RoPE /
fused K norm + RoPE V41 stores at 16384 tokens, the FP4 store at 16384 and
262144 tokens, the FP4 full-pool and selected-slot dequants, the translated
C4A compressor, C128A into FP4, the decode-time C4A compressor, a 61-layer
step behind one translation, and the hot-L2 latency table at bs 1/8/64/512.
--workload NAME times that workload alone (--suite adds the others).

Timing, per workload: W eager warm-up steps; CUDA graphs holding exactly K
steps (captured launches of the C ABI) are replayed between two CUDA events
on the launching stream, behind a bounded device-side sleep so that the host
has queued every replay before the first event (the region holds GPU
execution only, not submission); then the dominant kernel alone is replayed
in graphs for at least about 25 ms (the per-launch time behind
roofline.achieved).  Inputs rotate over enough distinct sets that every step
reads from HBM (each rotation set exceeds the 129 MB L2).  Rank 0 prints one
JSON line.  --impl reference times the CPU oracle (one thread and one thread
per host core) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0
METRIC = "KV tokens/s and achieved HBM GB/s (% of GB300 roofline) per layout/ratio"

# algorithmic bytes per unit (rows read + loc + pos + cos/sin row + payload written)
B_STORE = 1024 + 8 + 528
B_STORE_ROPE = B_STORE + 4 + 256
B_FP4_STORE = 1024 + 8 + 272
B_FP4_DEQ = 272 + 1024
B_TRANSLATE = 8 + 4 + 4


def b_compress(r, payload=528):
    return r * 4096 + 4 + 4 + 256 + payload


DEFAULT_STEPS = {
    "store_norm_rope": 20, "store_rope": 20, "store": 20, "small": 20,
    "fp4_store": 20, "fp4_store_16k": 20, "fp4_dequant": 20, "c4a": 20, "c128a": 20, "c128a_fp4": 20,
    "layers": 20, "dequant_select": 20, "c4a_decode": 20,
}
HEADLINE = "c128a"
# the rest of the configured workloads, timed in the same run as the headline
SUITE = ["small", "store", "store_rope", "store_norm_rope", "fp4_store_16k", "fp4_store", "fp4_dequant",
         "dequant_select", "c4a", "c4a_decode", "c128a_fp4", "layers"]

# the workloads: one per configuration of the write path
SPECS = {
    # 64 fp32 rows into a 4-page V41 pool, followed by the dequant of the 4 pages
    "small": dict(kind="store", flags=0, bs=64, pool_slots=256, layout=1, fp32=True, dequant=True),
    "store": dict(kind="store", flags=0, bs=16384, pool_slots=1 << 20, layout=1),
    "store_rope": dict(kind="store", flags=1, bs=16384, pool_slots=1 << 20, layout=1),
    "store_norm_rope": dict(kind="store", flags=3, bs=16384, pool_slots=1 << 20, layout=1),
    "fp4_store": dict(kind="store", flags=0, bs=262144, pool_slots=1 << 21, layout=2, student_t=True),
    "fp4_store_16k": dict(kind="store", flags=0, bs=16384, pool_slots=1 << 21, layout=2, student_t=True),
    "fp4_dequant": dict(kind="dequant", pool_slots=1 << 21, layout=2),
    # decode-time C4A: one new row per request per step, the open group's softmax carried as state
    "c4a_decode": dict(kind="decode", ratio=4, layout=1, requests=16384, pool_slots=1 << 17,
                       score_std=math.sqrt(2.0)),
    # the consumer side: the rows a sparse attention selects, gathered by slot
    "dequant_select": dict(kind="select", pool_slots=1 << 21, layout=2, n=1 << 18),
    "c4a": dict(kind="compress", ratio=4, layout=1, score_std=math.sqrt(2.0), groups=16384,
                full_slots=1 << 20, swa_slots=1 << 17),
    "c128a": dict(kind="compress", ratio=128, layout=1, score_std=2.0, requests=256,
                  pool_slots=1 << 20),
    # one decode step of a 61-layer model: the step's slots translated full -> SWA once, then
    # every layer stores its K rows (norm + RoPE, V41) into its own SWA pool
    "layers": dict(kind="layers", layers=61, bs=512, flags=3, layout=1, full_slots=1 << 20,
                   swa_slots=1 << 17),
    "c128a_fp4": dict(kind="compress", ratio=128, layout=2, score_std=2.0, requests=256,
                      pool_slots=1 << 20),
}


def describe(name):
    """(config dict, unit name) of a workload, without touching a GPU."""
    sp = SPECS[name]
    lay = "V41" if sp["layout"] == 1 else "V41_FP4"
    if sp["kind"] == "store":
        cfg = {"workload": name, "layout": lay, "flags": {0: "none", 1: "rope", 3: "norm+rope"}[sp["flags"]],
               "bs": sp["bs"], "x_dtype": "f32" if sp.get("fp32") else "bf16", "loc_dtype": "int64",
               "page_size": 64, "pool_slots": sp["pool_slots"],
               "rows": "0.5*Student-t(3)" if sp.get("student_t") else
                       ("N(0,1)" if sp.get("fp32") else "N(0,1), 1% x50 outliers")}
        if sp["flags"] & 1:
            cfg["rope"] = "last 64 dims, theta 1e4, positions U[0,65536), fp32 table"
        if sp["flags"] & 2:
            cfg["norm"] = "RMSNorm over 512 dims, w~N(1,0.1), eps 1e-6"
        if sp.get("dequant"):
            cfg["dequant"] = "the pool's pages back to bf16 after the store (identity page table)"
        return cfg, "tokens"
    if sp["kind"] == "dequant":
        return {"workload": name, "layout": lay, "tokens": sp["pool_slots"], "page_size": 64,
                "page_table": "random permutation of the pool's pages",
                "rows": "0.5*Student-t(3) stored by the FP4 store"}, "tokens"
    if sp["kind"] == "decode":
        return {"workload": name, "layout": lay, "ratio": sp["ratio"], "requests": sp["requests"],
                "state": "3 x 512 fp32 per request (running max, sum, weighted sum)",
                "phases": "request i starts at count i % ratio: a quarter complete a group each step",
                "pool_slots": sp["pool_slots"], "page_size": 64, "rope": "last 64 dims"}, "input tokens"
    if sp["kind"] == "select":
        return {"workload": name, "layout": lay, "pool_slots": sp["pool_slots"], "selected": sp["n"],
                "slots": "random distinct int64 slots of the whole pool", "page_size": 64,
                "rows": "0.5*Student-t(3) stored by the FP4 store"}, "tokens"
    if sp["kind"] == "layers":
        return {"workload": name, "layout": lay, "layers": sp["layers"], "bs": sp["bs"],
                "flags": "norm+rope", "x_dtype": "bf16", "loc_dtype": "int64 full slots -> int32 SWA slots",
                "full_slots": sp["full_slots"], "swa_slots_per_layer": sp["swa_slots"], "page_size": 64,
                "translate": "once per step, shared by every layer"}, "KV tokens (tokens x layers)"
    cfg = {"workload": name, "layout": lay, "ratio": sp["ratio"], "page_size": 64,
           "values": "N(0,1) fp32", "scores": f"N(0,{sp['score_std'] ** 2:g}) fp32",
           "rope": "last 64 dims at the group's position"}
    if sp["ratio"] == 4:
        cfg.update(groups=sp["groups"], input_tokens=sp["groups"] * 4, full_slots=sp["full_slots"],
                   swa_slots=sp["swa_slots"], translate="once per step, int64 full loc -> int32 SWA slot")
    else:
        cfg.update(requests=sp["requests"], lengths="log-uniform [128, 32768], multiples of 128",
                   pool_slots=sp["pool_slots"])
    return cfg, "input tokens"


# ----------------------------------------------------------------------------- workloads

class Workload:
    """Inputs on the GPU, one step, and the numbers that describe it."""

    R = 1                     # rotating input sets
    units = 0                 # KV tokens per step (the metric's unit)
    bytes_total = 0           # algorithmic bytes per step, all kernels
    bytes_dominant = 0        # algorithmic bytes of the dominant kernel per launch
    launches = 1              # our kernel launches per step
    dominant = ""

    def __init__(self, name, dev):
        import compress_kv_write_gb300 as K
        import torch
        self.K, self.name, self.dev = K, name, dev
        self.spec = SPECS[name]
        self.config, self.unit_name = describe(name)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(self, i):
        raise NotImplementedError

    def dominant_step(self, i):
        self.step(i)


def _rotation(per_set_bytes, cap=64):
    return max(1, min(cap, math.ceil(2.5 * L2_BYTES / max(1, per_set_bytes))))


def store_kernel_name(layout, flags, bs):
    """The store kernel a batch of bs tokens runs on (layout 1 = V41, flags
    1 = RoPE, 2 = norm): the library's small-batch kernel (one or two tokens
    per CTA) up to 1024 tokens with the norm, 3072 for the V41 store + RoPE
    and 1536 otherwise, its persistent kernels beyond."""
    if bs <= (1024 if flags & 2 else 3072 if (layout == 1 and flags == 1) else 1536):
        return "store_token_kernel"
    if layout != 1:
        return "store_half_kernel"
    # V41: the half-warp kernel from 12288 tokens with RoPE only, 16384 plain,
    # 65536 with the norm; one warp per token below
    return "store_half_kernel" if bs >= {1: 12288, 0: 16384}.get(flags, 65536) else "store_warp_kernel"


class StoreWorkload(Workload):
    """bs rows -> paged pool: store, store + RoPE, fused K RMSNorm + RoPE."""

    def __init__(self, name, dev):
        super().__init__(name, dev)
        import torch
        from compress_kv_write_gb300 import synth
        sp = self.spec
        self.flags, self.bs, self.layout = sp["flags"], sp["bs"], sp["layout"]
        self.pool_slots = sp["pool_slots"]
        bs = self.bs
        self.pool = torch.zeros(self.pool_slots * self.K.bytes_per_token(self.layout),
                                dtype=torch.uint8, device=dev)
        row_bytes = 2048 if sp.get("fp32") else 1024
        self.R = _rotation(bs * (row_bytes + 12))
        self.x, self.loc, self.pos = [], [], []
        for r in range(self.R):
            if sp.get("fp32"):
                x = synth.normal((bs, 512), dev, r, "x")
            elif sp.get("student_t"):
                x = synth.student_t_rows_bf16(bs, dev, r)
            else:
                x = synth.store_rows_bf16(bs, dev, r)
            self.x.append(x)
            self.loc.append(synth.injective_slots(bs, self.pool_slots, dev, r))
            self.pos.append(synth.positions(bs, dev, r))
        self.cs = synth.rope_table(65536, dev)
        self.w = synth.norm_weight(dev, 0)
        self.units = bs
        payload = 528 if self.layout == 1 else 272
        per = row_bytes + 8 + payload + ((4 + 256) if self.flags & 1 else 0)
        self.bytes_total = self.bytes_dominant = bs * per
        self.dominant = store_kernel_name(self.layout, self.flags, bs)
        if sp.get("dequant"):   # the pool's pages back to bf16 after each store
            self.n_pages = self.pool_slots >> 6
            self.pt = torch.arange(self.n_pages, dtype=torch.int32, device=dev)
            self.ws = torch.empty((self.pool_slots, 512), dtype=torch.bfloat16, device=dev)
            self.launches = 2
            self.bytes_total += self.pool_slots * (payload + 1024) + self.n_pages * 4
        total = self.R * bs * (row_bytes + 12)
        self.config["l2"] = (f"rotating {self.R} input sets ({total / 2**20:.0f} MB > 129 MB L2)"
                             if total > L2_BYTES else
                             f"latency config: {self.R} input sets ({total / 2**20:.1f} MB) stay in L2")

    def _store(self, x, loc, pos):
        rope = self.flags & 1
        self.K.kvq_store(self.layout, 6, self.flags, x, loc, self.pool, self.pool_slots,
                         norm_weight=self.w if self.flags & 2 else None, eps=1e-6,
                         cos_sin=self.cs if rope else None, pos=pos if rope else None, err=self.err)

    def step(self, i):
        r = i % self.R
        self._store(self.x[r], self.loc[r], self.pos[r])
        if self.spec.get("dequant"):
            self.K.kvq_dequant(self.layout, 6, self.pool, self.n_pages, self.pt, self.ws, err=self.err)

    def dominant_step(self, i):
        r = i % self.R
        self._store(self.x[r], self.loc[r], self.pos[r])

    # End to end: each step's rows, slots and positions arrive as ONE pinned host
    # buffer [rows | slots | positions]; it is copied into one of two device
    # buffers on a copy stream while the previous step's store runs, and the
    # step's error word is read back.
    def e2e_setup(self):
        import torch
        x0, l0, p0 = self.x[0], self.loc[0], self.pos[0]
        self.e2e_parts = [(x0.numel() * x0.element_size(), x0.dtype, x0.shape),
                          (l0.numel() * 8, torch.int64, l0.shape), (p0.numel() * 4, torch.int32, p0.shape)]
        total = sum(b for b, _, _ in self.e2e_parts)
        host = torch.empty(total, dtype=torch.uint8).pin_memory()
        off = 0
        for (b, dt, shp), t in zip(self.e2e_parts, (x0, l0, p0)):
            host[off:off + b].copy_(t.cpu().contiguous().view(torch.uint8).reshape(-1))
            off += b
        self.hbuf = host
        self.dbufs = [torch.empty(total, dtype=torch.uint8, device=self.dev) for _ in range(2)]
        self.dviews = []
        for d in self.dbufs:
            views, off = [], 0
            for b, dt, shp in self.e2e_parts:
                views.append(d[off:off + b].view(dt).view(shp))
                off += b
            self.dviews.append(views)
        self.copy_stream = torch.cuda.Stream(device=self.dev)
        self.copied = [torch.cuda.Event() for _ in range(2)]
        self.done = [torch.cuda.Event() for _ in range(2)]
        for e in self.done:
            e.record()
        self.herr = torch.zeros(1, dtype=torch.int32).pin_memory()
        self.e2e_i = 0
        return total, 4

    def e2e_step(self):
        import torch
        b = self.e2e_i & 1
        self.e2e_i += 1
        compute = torch.cuda.current_stream()
        self.copy_stream.wait_event(self.done[b])       # the store that last read this buffer
        with torch.cuda.stream(self.copy_stream):
            self.dbufs[b].copy_(self.hbuf, non_blocking=True)
            self.copied[b].record(self.copy_stream)
        compute.wait_event(self.copied[b])
        dx, dloc, dpos = self.dviews[b]
        self._store(dx, dloc, dpos)
        if self.spec.get("dequant"):
            self.K.kvq_dequant(self.layout, 6, self.pool, self.n_pages, self.pt, self.ws, err=self.err)
        self.done[b].record(compute)
        self.herr.copy_(self.err, non_blocking=True)

class DequantWorkload(Workload):
    """Full-pool paged dequant of a 2^21-slot FP4 pool into a bf16 workspace."""

    def __init__(self, name, dev):
        super().__init__(name, dev)
        import torch
        from compress_kv_write_gb300 import synth
        self.layout, self.pool_slots = self.spec["layout"], self.spec["pool_slots"]
        self.pool = torch.zeros(self.pool_slots * self.K.bytes_per_token(self.layout),
                                dtype=torch.uint8, device=dev)
        chunk = 1 << 18
        x = synth.student_t_rows_bf16(chunk, dev, 0)
        for c in range(self.pool_slots // chunk):     # fill the pool with the FP4 store
            loc = torch.arange(c * chunk, (c + 1) * chunk, device=dev)
            self.K.kvq_store(self.layout, 6, 0, x, loc, self.pool, self.pool_slots)
        del x
        self.n_pages = self.pool_slots >> 6
        self.pt = synth.page_table_perm(self.n_pages, dev, 0)
        self.out = torch.empty((self.pool_slots, 512), dtype=torch.bfloat16, device=dev)
        self.units = self.pool_slots
        self.bytes_total = self.bytes_dominant = self.pool_slots * B_FP4_DEQ + self.n_pages * 4
        self.dominant = "dequant_kernel"
        self.config["l2"] = (f"pool {self.pool_slots * 288 / 2**20:.0f} MB read + workspace "
                             f"{self.pool_slots * 1024 / 2**20:.0f} MB written per step > 129 MB L2")

    def step(self, i):
        self.K.kvq_dequant(self.layout, 6, self.pool, self.n_pages, self.pt, self.out, err=self.err)

    def e2e_setup(self):
        import torch
        self.hpt = self.pt.cpu().pin_memory()
        self.dpt = torch.empty_like(self.pt)
        self.hout = torch.empty((self.pool_slots, 512), dtype=torch.bfloat16).pin_memory()
        return self.hpt.numel() * 4, self.hout.numel() * 2

    def e2e_step(self):
        self.dpt.copy_(self.hpt, non_blocking=True)
        self.K.kvq_dequant(self.layout, 6, self.pool, self.n_pages, self.dpt, self.out, err=self.err)
        self.hout.copy_(self.out, non_blocking=True)


class CompressWorkload(Workload):
    """Ratio-r softmax compressor; C4A also translates its slots once per step."""

    def __init__(self, name, dev):
        super().__init__(name, dev)
        import torch
        from compress_kv_write_gb300 import synth
        sp = self.spec
        self.r, self.layout = sp["ratio"], sp["layout"]
        payload = 528 if self.layout == 1 else 272
        r = self.r
        if r == 4:
            G = sp["groups"]
            self.full_slots, self.pool_slots = sp["full_slots"], sp["swa_slots"]
            per_set = G * r * 4096
            self.R = _rotation(per_set, cap=8)
            self.v, self.s, self.full_loc, self.table = [], [], [], []
            for k in range(self.R):
                v, s = synth.compressor_rows(G * r, dev, k, score_std=sp["score_std"])
                fl = synth.injective_slots(G, self.full_slots, dev, k)
                self.v.append(v)
                self.s.append(s)
                self.full_loc.append(fl)
                self.table.append(synth.swa_table(self.full_slots, self.pool_slots, fl, dev, k))
            self.gpos = torch.arange(G, dtype=torch.int32, device=dev) * r
            self.cs = synth.rope_table(65536, dev)
            self.swa_loc = torch.zeros(G, dtype=torch.int32, device=dev)
            self.launches = 2
            self.bytes_total = G * (B_TRANSLATE + b_compress(r, payload))
            self.config["l2"] = f"rotating {self.R} input sets ({self.R * per_set / 2**20:.0f} MB > 129 MB L2)"
        else:
            lens = synth.request_lengths(sp["requests"], seed=0)
            self.gpos = synth.group_positions(lens, r).to(dev)
            G = self.gpos.numel()
            self.pool_slots = sp["pool_slots"]
            v, s = synth.compressor_rows(G * r, dev, 0, score_std=sp["score_std"])
            self.v, self.s = [v], [s]
            self.loc = synth.injective_slots(G, self.pool_slots, dev, 0, dtype=torch.int32)
            self.cs = synth.rope_table(32768, dev)
            self.bytes_total = G * b_compress(r, payload)
            self.config.update(groups=G, input_tokens=G * r)
            self.config["l2"] = f"inputs {G * r * 4096 / 2**30:.2f} GB per step > 129 MB L2"
        self.G = G
        self.pool = torch.zeros(self.pool_slots * self.K.bytes_per_token(self.layout),
                                dtype=torch.uint8, device=dev)
        self.units = G * r
        self.bytes_dominant = G * b_compress(r, payload)
        self.dominant = "compress_kernel"

    def _compress(self, v, s, loc):
        self.K.kvq_compress(self.layout, 6, self.r, self.K.FLAG_ROPE, v, s, loc, self.pool,
                            self.pool_slots, cos_sin=self.cs, group_pos=self.gpos, err=self.err)

    def step(self, i):
        k = i % self.R
        if self.r == 4:
            self.K.kvq_translate_loc(self.full_loc[k], self.table[k], self.swa_loc, err=self.err)
            self._compress(self.v[k], self.s[k], self.swa_loc)
        else:
            self._compress(self.v[k], self.s[k], self.loc)

    def dominant_step(self, i):
        k = i % self.R
        self._compress(self.v[k], self.s[k], self.swa_loc if self.r == 4 else self.loc)

    # End to end: the step's values and scores arrive from pinned host memory.  The mixed C128A
    # batch is cut into chunks of groups: each chunk is copied on a copy stream and compressed as
    # soon as it has landed, so the kernel runs under the next chunk's copy (the host link, about
    # 210 GB/s on these machines, bounds the step).  The step's error word is read back.
    def e2e_setup(self):
        import torch
        self.hv = self.v[0].cpu().pin_memory()
        self.hs = self.s[0].cpu().pin_memory()
        self.dv = torch.empty_like(self.v[0])
        self.ds = torch.empty_like(self.s[0])
        self.herr = torch.zeros(1, dtype=torch.int32).pin_memory()
        h2d = 2 * self.hv.numel() * 4
        if self.r == 4:
            self.hloc = self.full_loc[0].cpu().pin_memory()
            self.dloc = torch.empty_like(self.full_loc[0])
            h2d += self.hloc.numel() * 8
            self.chunks = [(0, self.G)]
        else:
            n = 8
            self.chunks = [(self.G * i // n, self.G * (i + 1) // n) for i in range(n)]
        self.copy_stream = torch.cuda.Stream(device=self.dev)
        self.copied = [torch.cuda.Event() for _ in self.chunks]
        self.done = torch.cuda.Event()
        self.done.record()
        return h2d, 4

    def e2e_step(self):
        import torch
        compute = torch.cuda.current_stream()
        r = self.r
        self.copy_stream.wait_event(self.done)  # the previous step has read the device buffers
        with torch.cuda.stream(self.copy_stream):
            if r == 4:
                self.dloc.copy_(self.hloc, non_blocking=True)
            for (a, b), ev in zip(self.chunks, self.copied):
                self.dv[a * r:b * r].copy_(self.hv[a * r:b * r], non_blocking=True)
                self.ds[a * r:b * r].copy_(self.hs[a * r:b * r], non_blocking=True)
                ev.record(self.copy_stream)
        for (a, b), ev in zip(self.chunks, self.copied):
            compute.wait_event(ev)
            if r == 4:
                self.K.kvq_translate_loc(self.dloc, self.table[0], self.swa_loc, err=self.err)
                loc = self.swa_loc
            else:
                loc = self.loc[a:b]
            self.K.kvq_compress(self.layout, 6, r, self.K.FLAG_ROPE, self.dv[a * r:b * r], self.ds[a * r:b * r],
                                loc, self.pool, self.pool_slots, cos_sin=self.cs, group_pos=self.gpos[a:b],
                                err=self.err)
        self.done.record(compute)
        self.herr.copy_(self.err, non_blocking=True)


class DecodeWorkload(Workload):
    """Decode-time ratio-r compressor over many requests, one row each per step."""

    def __init__(self, name, dev):
        super().__init__(name, dev)
        import torch
        from compress_kv_write_gb300 import synth
        sp = self.spec
        self.r, self.layout, self.n, self.pool_slots = sp["ratio"], sp["layout"], sp["requests"], sp["pool_slots"]
        self.R = 4
        self.v, self.s = [], []
        for k in range(self.R):
            v, s = synth.compressor_rows(self.n, dev, k, score_std=sp["score_std"])
            self.v.append(v)
            self.s.append(s)
        self.state = torch.zeros((self.n, 3, 512), dtype=torch.float32, device=dev)
        self.count = (torch.arange(self.n, dtype=torch.int32, device=dev) % self.r).contiguous()
        self.loc = synth.injective_slots(self.n, self.pool_slots, dev, 0, dtype=torch.int32)
        self.gpos = synth.positions(self.n, dev, 0)
        self.cs = synth.rope_table(65536, dev)
        self.pool = torch.zeros(self.pool_slots * self.K.bytes_per_token(self.layout), dtype=torch.uint8,
                                device=dev)
        payload = 528 if self.layout == 1 else 272
        r = self.r
        self.units = self.n
        self.bytes_total = self.bytes_dominant = int(
            self.n * (4096 + 8) + self.n * (r - 1) / r * 6144 * 2 + self.n / r * (4 + 4 + 256 + payload))
        self.dominant = "compress_decode_kernel"
        self.config["l2"] = (f"rotating {self.R} row sets of {self.n * 4096 / 2**20:.0f} MB; state "
                             f"{self.n * 6144 / 2**20:.0f} MB read and written every step")

    def _call(self, v, s):
        self.K.kvq_compress_decode(self.layout, 6, self.r, self.K.FLAG_ROPE, v, s, self.state, self.count,
                                   self.loc, self.pool, self.pool_slots, cos_sin=self.cs,
                                   group_pos=self.gpos, err=self.err)

    def step(self, i):
        self._call(self.v[i % self.R], self.s[i % self.R])

    def e2e_setup(self):
        import torch
        self.hv = self.v[0].cpu().pin_memory()
        self.hs = self.s[0].cpu().pin_memory()
        self.dv = torch.empty_like(self.v[0])
        self.ds = torch.empty_like(self.s[0])
        self.herr = torch.zeros(1, dtype=torch.int32).pin_memory()
        return 2 * self.hv.numel() * 4, 4

    def e2e_step(self):
        self.dv.copy_(self.hv, non_blocking=True)
        self.ds.copy_(self.hs, non_blocking=True)
        self._call(self.dv, self.ds)
        self.herr.copy_(self.err, non_blocking=True)


class SelectWorkload(Workload):
    """Dequant of the rows a sparse attention selects from a full FP4 pool."""

    def __init__(self, name, dev):
        super().__init__(name, dev)
        import torch
        from compress_kv_write_gb300 import synth
        sp = self.spec
        self.layout, self.pool_slots, self.n = sp["layout"], sp["pool_slots"], sp["n"]
        self.pool = torch.zeros(self.pool_slots * self.K.bytes_per_token(self.layout),
                                dtype=torch.uint8, device=dev)
        chunk = 1 << 18
        x = synth.student_t_rows_bf16(chunk, dev, 0)
        for c in range(self.pool_slots // chunk):
            loc = torch.arange(c * chunk, (c + 1) * chunk, device=dev)
            self.K.kvq_store(self.layout, 6, 0, x, loc, self.pool, self.pool_slots)
        del x
        self.R = 4
        self.sel = [synth.injective_slots(self.n, self.pool_slots, dev, r) for r in range(self.R)]
        self.out = torch.empty((self.n, 512), dtype=torch.bfloat16, device=dev)
        self.units = self.n
        payload = 528 if self.layout == 1 else 272
        self.bytes_total = self.bytes_dominant = self.n * (payload + 1024 + 8)
        self.dominant = "dequant_slots_kernel"
        self.config["l2"] = (f"pool {self.pool_slots * 288 / 2**20:.0f} MB, random rows; output "
                             f"{self.n * 1024 / 2**20:.0f} MB per step > 129 MB L2")

    def step(self, i):
        self.K.kvq_dequant_slots(self.layout, 6, self.pool, self.pool_slots, self.sel[i % self.R],
                                 self.out, err=self.err)

    def e2e_setup(self):
        import torch
        self.hsel = self.sel[0].cpu().pin_memory()
        self.dsel = torch.empty_like(self.sel[0])
        self.hout = torch.empty((self.n, 512), dtype=torch.bfloat16).pin_memory()
        return self.hsel.numel() * 8, self.hout.numel() * 2

    def e2e_step(self):
        self.dsel.copy_(self.hsel, non_blocking=True)
        self.K.kvq_dequant_slots(self.layout, 6, self.pool, self.pool_slots, self.dsel, self.out,
                                 err=self.err)
        self.hout.copy_(self.out, non_blocking=True)


class LayersWorkload(Workload):
    """One step of an L-layer model: translate the step's full-pool slots to SWA
    slots once, then store each layer's K rows (norm + RoPE, V41) into that
    layer's SWA pool with the shared translated slots."""

    def __init__(self, name, dev):
        super().__init__(name, dev)
        import torch
        from compress_kv_write_gb300 import synth
        sp = self.spec
        self.L, self.bs, self.flags = sp["layers"], sp["bs"], sp["flags"]
        self.full_slots, self.swa_slots = sp["full_slots"], sp["swa_slots"]
        per_set = self.L * self.bs * (1024 + 12)
        self.R = _rotation(per_set, cap=8)
        self.x, self.full_loc, self.table, self.pos = [], [], [], []
        for r in range(self.R):
            self.x.append([synth.store_rows_bf16(self.bs, dev, 1000 * r + l) for l in range(self.L)])
            fl = synth.injective_slots(self.bs, self.full_slots, dev, r)
            self.full_loc.append(fl)
            self.table.append(synth.swa_table(self.full_slots, self.swa_slots, fl, dev, r))
            self.pos.append(synth.positions(self.bs, dev, r))
        self.cs = synth.rope_table(65536, dev)
        self.w = [synth.norm_weight(dev, l) for l in range(self.L)]
        self.pools = [torch.zeros(self.swa_slots * 528, dtype=torch.uint8, device=dev) for _ in range(self.L)]
        self.swa_loc = torch.zeros(self.bs, dtype=torch.int32, device=dev)
        self.launches = 1 + self.L
        self.units = self.bs * self.L
        per_store = self.bs * B_STORE_ROPE
        self.bytes_dominant = per_store
        self.bytes_total = self.L * per_store + self.bs * B_TRANSLATE
        self.dominant = store_kernel_name(1, self.flags, self.bs)
        self.config["l2"] = (f"rotating {self.R} step input sets ({self.R * per_set / 2**20:.0f} MB) "
                             f"over {self.L} pools of {self.swa_slots * 528 / 2**20:.0f} MB")

    def _layer(self, r, l):
        self.K.kvq_store(1, 6, self.flags, self.x[r][l], self.swa_loc, self.pools[l], self.swa_slots,
                         norm_weight=self.w[l], eps=1e-6, cos_sin=self.cs, pos=self.pos[r], err=self.err)

    def step(self, i):
        r = i % self.R
        self.K.kvq_translate_loc(self.full_loc[r], self.table[r], self.swa_loc, err=self.err)
        for l in range(self.L):
            self._layer(r, l)

    def step_unhoisted(self, i):
        """The same step with the translation repeated inside every layer."""
        r = i % self.R
        for l in range(self.L):
            self.K.kvq_translate_loc(self.full_loc[r], self.table[r], self.swa_loc, err=self.err)
            self._layer(r, l)

    def dominant_step(self, i):
        self._layer(i % self.R, i % self.L)

    def e2e_setup(self):
        import torch
        self.hx = [x.cpu().pin_memory() for x in self.x[0]]
        self.hloc = self.full_loc[0].cpu().pin_memory()
        self.dx = [torch.empty_like(x) for x in self.x[0]]
        self.dloc = torch.empty_like(self.full_loc[0])
        self.herr = torch.zeros(1, dtype=torch.int32).pin_memory()
        return sum(x.numel() * 2 for x in self.hx) + self.hloc.numel() * 8, 4

    def e2e_step(self):
        self.dloc.copy_(self.hloc, non_blocking=True)
        self.K.kvq_translate_loc(self.dloc, self.table[0], self.swa_loc, err=self.err)
        for l in range(self.L):
            self.dx[l].copy_(self.hx[l], non_blocking=True)
            self.K.kvq_store(1, 6, self.flags, self.dx[l], self.swa_loc, self.pools[l], self.swa_slots,
                             norm_weight=self.w[l], eps=1e-6, cos_sin=self.cs, pos=self.pos[0], err=self.err)
        self.herr.copy_(self.err, non_blocking=True)


def make_workload(name, dev, tokens=None):
    """tokens (profiling only): shrink the workload to about this many KV tokens."""
    if tokens:
        sp = dict(SPECS[name])
        if sp["kind"] == "store":
            sp["bs"] = int(tokens)
        elif sp["kind"] == "dequant":
            sp["pool_slots"] = max(1 << 18, (int(tokens) >> 18) << 18)
        elif sp["kind"] == "layers":
            sp["bs"] = max(1, int(tokens) // sp["layers"])
        elif sp["kind"] == "select":
            sp["n"] = int(tokens)
        elif sp["kind"] == "decode":
            sp["requests"] = int(tokens)
        elif sp["ratio"] == 4:
            sp["groups"] = max(1, int(tokens) // 4)
        else:
            sp["requests"] = max(1, int(tokens) * 256 // 1_500_000)
        SPECS[name] = sp
    kind = SPECS[name]["kind"]
    cls = {"store": StoreWorkload, "dequant": DequantWorkload, "compress": CompressWorkload,
           "layers": LayersWorkload, "select": SelectWorkload, "decode": DecodeWorkload}[kind]
    return cls(name, dev)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock, utilisation and throttle reasons while
    running; samples with the GPU busy count as under load."""

    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        return self.summarise(self.lines)

    @classmethod
    def summarise(cls, lines):
        busy, idle, mx, reasons = [], [], [], set()
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 7:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
                util = float(parts[2])
            except ValueError:
                continue
            mx.append(smax)
            if util >= 50:
                busy.append(sm)
                for nm, p in zip(cls.REASONS, parts[3:]):
                    if p.lower() == "active":
                        reasons.add(nm)
            else:
                idle.append(sm)
        if not busy and not idle:
            return None
        use = busy or idle
        return {"sm_mhz": statistics.median(use), "sm_max_mhz": max(mx), "samples": len(use),
                "samples_total": len(busy) + len(idle), "under_load": bool(busy), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- helpers

def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


_STORE_SOURCES = ("kvq_store.cu", "kvq_store_small.cu", "kvq_store.cuh")
KERNEL_SOURCES = {"store": _STORE_SOURCES, "dequant": ("kvq_dequant.cu",), "compress": ("kvq_compress.cu",),
                  "layers": _STORE_SOURCES, "select": ("kvq_dequant.cu",), "decode": ("kvq_decode.cu",)}


def traffic_from_profiles(workload):
    """DRAM bytes per launch of the dominant kernel, from the committed ncu
    summary (profiles/traffic.txt), if that kernel's sources are unchanged
    since the counters were taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    sha = kernel_source_sha(workload)
    for ln in lines:
        p = ln.split()
        if len(p) >= 4 and not ln.startswith("#") and p[0] == workload and p[3] == sha:
            return float(p[2])
    return None


def _code_only(text):
    """C++ source without comments and with whitespace runs collapsed, so that
    editing a comment does not count as changing a kernel."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha(workload):
    """Hash of the code (comments dropped) of the dominant kernel's translation
    unit and the shared headers."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "compress_kv_write_gb300", "csrc")
    files = [*KERNEL_SOURCES[SPECS[workload]["kind"]], "kvq_device.cuh", "kvq_launch.cuh"]
    for fn in files:
        with open(os.path.join(d, fn), encoding="utf-8") as f:
            h.update(fn.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def max_over_ranks(value, device=None):
    """The largest of every rank's value (the slowest rank's time); the value
    itself when there is no process group of more than one rank."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def host_cpu():
    """(model name, usable cores) of this host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith(("model name", "cpu part")):
                    model = ln.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    import platform
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    return f"{model or 'unknown'} ({platform.machine()})", cores


def capture_graphs(wl, steps, chunk, stream, fn=None):
    """CUDA graphs holding exactly `steps` calls of fn (default: wl.step):
    (graph, replays) pairs."""
    import torch
    fn = fn or wl.step
    plan = []
    full, rem = divmod(steps, chunk)
    offset = 0
    for n, reps in ((chunk, full), (rem, 1)):
        if n == 0 or reps == 0:
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(offset + i)
        plan.append((g, reps))
        offset += n
    return plan


# A device-side sleep ahead of each timed region, long enough for the host to
# queue every graph replay of the region before the GPU reaches the first
# event: the region then holds GPU execution only.
SLEEP_CYCLES = 20_000_000  # about 10 ms at the 2.07 GHz SM clock


def time_plan(plan, stream):
    """Milliseconds between two events around the replays of `plan`, queued
    behind a bounded device-side sleep."""
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(SLEEP_CYCLES)
        e0.record(stream)
        for g, reps in plan:
            for _ in range(reps):
                g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def replay_once(plan, stream):
    import torch
    with torch.cuda.stream(stream):
        for g, _ in plan:
            g.replay()
    torch.cuda.synchronize()


def dominant_launch_ms(wl, stream, est_ms, target_ms=25.0, min_launches=50, chunk_max=512):
    """Per-launch time of the dominant kernel alone, replayed in graphs for at
    least about target_ms (inputs rotating as in the step)."""
    n = int(max(min_launches, min(200_000, math.ceil(target_ms / max(est_ms, 1e-4)))))
    chunk = min(n, chunk_max)
    n = max(chunk, (n // chunk) * chunk)
    plan = capture_graphs(wl, n, chunk, stream, fn=wl.dominant_step)
    replay_once(plan, stream)
    ms = time_plan(plan, stream)
    del plan
    return ms / n, n


def run_workload(wl, K, W, stream, dev, world):
    """The timed K-step region and the dominant kernel's per-launch time."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(W):
            wl.step(i)
    stream.synchronize()
    assert wl.err.item() == 0, f"device error during warm-up of {wl.name}"
    chunk = max(1, min(K, max(wl.R, 1) * max(1, 512 // max(wl.R, 1))))
    plan = capture_graphs(wl, K, chunk, stream)
    replay_once(plan, stream)  # uploads the graphs
    import torch.distributed as dist
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ms = time_plan(plan, stream)
    if world > 1:
        dist.barrier()
    del plan
    assert wl.err.item() == 0, f"device error in the timed region of {wl.name}"
    ms = max_over_ranks(ms, dev)
    ms_per_step = ms / K
    dom_ms, dom_n = dominant_launch_ms(wl, stream, ms_per_step / max(1, wl.launches))
    dom_ms = max_over_ranks(dom_ms, dev)
    assert wl.err.item() == 0, f"device error in the dominant-kernel replay of {wl.name}"
    return ms, ms_per_step, dom_ms, dom_n


def workload_record(wl, K, ms, ms_per_step, dom_ms, dom_n, world, peak):
    achieved = wl.bytes_dominant / (dom_ms / 1e3) / 1e9
    rec = {
        "value": wl.units * K * world / (ms / 1e3), "unit": f"{wl.unit_name}/s", "ms_per_step": ms_per_step,
        "step_gbs": wl.bytes_total / (ms_per_step / 1e3) / 1e9,
        "kernel": wl.dominant, "kernel_us_per_launch": dom_ms * 1e3, "kernel_launches_timed": dom_n,
        "algorithmic_bytes_per_launch": wl.bytes_dominant, "achieved_gbs": achieved, "frac": achieved / peak,
        "traffic": traffic_from_profiles(wl.name), "launches_per_step": wl.launches,
    }
    if wl.launches == 1:
        # the K-step region and the long replay time the same launches
        rec["k_steps_vs_long_replay"] = ms_per_step / dom_ms
    return rec


def add_l2_flush(wl, dev, nbytes=512 << 20):
    """Profiling only: read a buffer four times the L2 after every step, so
    that the lines a step left dirty in L2 are written back to DRAM inside
    the next kernel (a capture of both kernels then counts the write-back
    that a capture of the step's kernels alone cannot see)."""
    import torch
    buf = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)
    step, dominant = wl.step, wl.dominant_step

    def flushed(fn):
        def run(i):
            fn(i)
            buf.sum()
        return run
    wl.step, wl.dominant_step = flushed(step), flushed(dominant)
    wl.config["l2_flush"] = f"profiling: a {nbytes >> 20} MB read after every step (not a bench number)"


def hoist_record(wl, K, ms_per_step, stream):
    """The layers step with the slot translation repeated inside every layer
    (the un-hoisted form), timed the same way."""
    n = max(K, 50)
    plan = capture_graphs(wl, n, min(n, 64), stream, fn=wl.step_unhoisted)
    replay_once(plan, stream)
    un_ms = time_plan(plan, stream) / n
    return {"hoisted_ms_per_step": ms_per_step, "translate_per_layer_ms_per_step": un_ms,
            "speedup": un_ms / ms_per_step, "layers": wl.L}


# ----------------------------------------------------------------------------- arms

def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()

    K, W = args.steps, args.warmup
    stream = torch.cuda.Stream(device=dev)
    peak, peak_src = measured_hbm_peak()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[local] if vis else local)
    if rank == 0 and not args.no_clocks:
        sampler.start()
        time.sleep(0.3)

    wl = make_workload(args.workload, dev, args.tokens)
    if args.flush_l2:
        add_l2_flush(wl, dev)
    ms, ms_per_step, dom_ms, dom_n = run_workload(wl, K, W, stream, dev, world)
    head = workload_record(wl, K, ms, ms_per_step, dom_ms, dom_n, world, peak)
    hoist = hoist_record(wl, K, ms_per_step, stream) if hasattr(wl, "step_unhoisted") else None

    # end to end through the API: pinned host inputs -> device, result back, every step
    h2d, d2h = wl.e2e_setup()
    e2e_steps = max(3, min(K, args.e2e_steps))
    with torch.cuda.stream(stream):
        wl.e2e_step()
    stream.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            wl.e2e_step()
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    e2e_value = wl.units * e2e_steps * world / e2e_s
    config = dict(wl.config, units=wl.unit_name, parallelism=f"replicas{world}",
                  timing="CUDA graphs of exactly K steps behind a device-side sleep (GPU execution only), "
                         "CUDA events; per-launch kernel time from a >= 25 ms replay of the dominant kernel")
    launches = wl.launches * K
    name = wl.name
    del wl
    torch.cuda.empty_cache()

    # every other configured workload, timed in the same run
    suite = {}
    names = [n for n in SUITE if n != name] if args.suite else []
    for n in names:
        w2 = make_workload(n, dev)
        r = run_workload(w2, K, W, stream, dev, world)
        suite[n] = workload_record(w2, K, *r, world, peak)
        if hasattr(w2, "step_unhoisted"):
            suite[n]["hoist"] = hoist_record(w2, K, r[1], stream)
        suite[n]["config"] = w2.config
        del w2
        torch.cuda.empty_cache()
    latency = run_latency_table(dev, stream) if (args.suite and rank == 0) else None
    clocks = sampler.stop() if (rank == 0 and not args.no_clocks) else None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(name, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config,
            "gbs": head["step_gbs"],
            "roofline": {"bound": "hbm", "achieved": head["achieved_gbs"], "peak": peak, "unit": "GB/s",
                         "frac": head["frac"], "peak_source": f"{peak_src} hbm_gbs (of {peak_src})",
                         "kernel": head["kernel"], "algorithmic_bytes": head["algorithmic_bytes_per_launch"],
                         "kernel_us_per_launch": head["kernel_us_per_launch"],
                         "kernel_launches_timed": head["kernel_launches_timed"],
                         "traffic": head["traffic"]},
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": launches,
            **({"hoist": hoist} if hoist else {}),
            **({"workloads": suite} if suite else {}),
            **({"latency_us": latency} if latency else {}),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def oracle_sample(name, n_rows):
    """CPU inputs for the oracle, drawn by the same generators (on the CPU)."""
    import numpy as np
    import torch
    from compress_kv_write_gb300 import synth
    import oracle as O
    spec = SPECS[name]
    kind = spec["kind"]
    if kind == "select":
        n_pages = max(1, n_rows // 64)
        x_np = synth.student_t_rows_bf16(n_pages * 64, "cpu", 0).view(torch.int16).numpy().view(np.uint16)
        pool = np.zeros(n_pages * 64 * 288, np.uint8)
        assert O.store(O.FP4, 6, 0, x_np, np.arange(n_pages * 64), pool) == O.OK
        return dict(pool=pool, slots=np.random.default_rng(0).permutation(n_pages * 64))
    if kind in ("store", "layers"):
        n = n_rows
        if spec.get("fp32"):
            x_np = synth.normal((n, 512), "cpu", 0, "x").numpy()
        elif spec.get("student_t"):
            x_np = synth.student_t_rows_bf16(n, "cpu", 0).view(torch.int16).numpy().view(np.uint16)
        else:
            x_np = synth.store_rows_bf16(n, "cpu", 0).view(torch.int16).numpy().view(np.uint16)
        return dict(x=x_np, pos=synth.positions(n, "cpu", 0).numpy(),
                    cs=synth.rope_table(65536, "cpu").numpy(), w=synth.norm_weight("cpu", 0).numpy())
    if kind == "dequant":
        n_pages = max(1, n_rows // 64)
        x_np = synth.student_t_rows_bf16(n_pages * 64, "cpu", 0).view(torch.int16).numpy().view(np.uint16)
        pool = np.zeros(n_pages * 64 * 288, np.uint8)
        assert O.store(O.FP4, 6, 0, x_np, np.arange(n_pages * 64), pool) == O.OK
        return dict(pages=pool)
    r = spec["ratio"]  # compress and decode: the oracle pools whole groups of r rows
    g = max(1, n_rows // r)
    v, s = synth.compressor_rows(g * r, "cpu", 0, score_std=spec["score_std"])
    return dict(v=v.numpy(), s=s.numpy(), gpos=(np.arange(g, dtype=np.int32) * r),
                cs=synth.rope_table(65536, "cpu").numpy())


def oracle_run(name, smp, n_units, first=0):
    """Run the oracle over about n_units tokens of the sample, starting at unit
    `first` (wrapping); returns the tokens done."""
    import numpy as np
    import oracle as O
    spec = SPECS[name]
    kind = spec["kind"]
    layout = spec.get("layout", 1)
    if kind == "select":
        size = smp["slots"].size
        n = max(1, min(n_units, size))
        a = first % max(1, size - n + 1)
        rc, _ = O.dequant_slots(O.FP4, smp["pool"], smp["slots"][a:a + n], 6)
        assert rc == O.OK
        return n
    if kind in ("store", "layers"):
        size = smp["x"].shape[0]
        n = min(n_units, size)
        a = first % max(1, size - n + 1)
        slots = max(64, -(-n // 64) * 64)
        pool = np.zeros(slots * O.bytes_per_token(layout), np.uint8)
        rc = O.store(layout, 6, spec["flags"], smp["x"][a:a + n], np.arange(n), pool, norm_weight=smp["w"],
                     eps=1e-6, cos_sin=smp["cs"], pos=smp["pos"][a:a + n])
        assert rc == O.OK
        return n
    if kind == "dequant":
        pages = smp["pages"].size // (64 * 288)
        n_pages = max(1, min(n_units // 64, pages))
        a = (first // 64) % max(1, pages - n_pages + 1)
        rc, _ = O.dequant(O.FP4, 6, smp["pages"], np.arange(a, a + n_pages, dtype=np.int32), n_pages * 64)
        assert rc == O.OK
        return n_pages * 64
    r = spec["ratio"]
    size = smp["gpos"].size
    g = max(1, min(n_units // r, size))
    a = (first // r) % max(1, size - g + 1)
    slots = max(64, -(-g // 64) * 64)
    pool = np.zeros(slots * O.bytes_per_token(layout), np.uint8)
    rc = O.compress(layout, 6, r, O.ROPE, smp["v"][a * r:(a + g) * r], smp["s"][a * r:(a + g) * r], np.arange(g),
                    pool, cos_sin=smp["cs"], group_pos=smp["gpos"][a:a + g])
    assert rc == O.OK
    return g * r


def _sample_rows(name):
    spec = SPECS[name]
    if spec["kind"] in ("compress", "decode"):
        return spec["ratio"] * (64 if spec["ratio"] >= 128 else 1024)
    return min(4096, spec.get("bs", 4096))


def _chunk_units(name):
    spec = SPECS[name]
    if spec["kind"] in ("compress", "decode"):
        return spec["ratio"] * (1 if spec["ratio"] >= 128 else 64)
    return min(256, spec.get("bs", 256))


def oracle_timed(name, smp, seconds, threads):
    """The oracle over disjoint chunks of the sample for about `seconds`, on
    `threads` host threads (the C oracle releases the GIL while it runs).
    Returns (units done, seconds)."""
    import concurrent.futures as cf
    chunk = _chunk_units(name)
    stop = time.perf_counter() + seconds

    def worker(k):
        done, i = 0, 0
        while time.perf_counter() < stop:
            done += oracle_run(name, smp, chunk, first=(k + i * threads) * chunk)
            i += 1
        return done

    t0 = time.perf_counter()
    if threads == 1:
        done = worker(0)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            done = sum(ex.map(worker, range(threads)))
    return done, time.perf_counter() - t0


def cpu_baseline(name, seconds):
    """The oracle (plain C, built -O2 without FMA contraction) on a bounded
    sample of the workload: one host thread, then one thread per host core
    over disjoint chunks; value = the all-core figure."""
    import oracle as O
    O.build()
    smp = oracle_sample(name, _sample_rows(name))
    model, cores = host_cpu()
    units = describe(name)[1]
    d1, t1 = oracle_timed(name, smp, seconds / 2, 1)
    dn, tn = oracle_timed(name, smp, seconds / 2, cores)
    return {"value": dn / tn, "unit": "tokens/s", "cores": cores, "kind": "oracle", "cpu": model,
            "single_thread": {"value": d1 / t1, "unit": "tokens/s", "cores": 1},
            "sample": f"{dn} {units} of the {name} workload in {tn:.1f} s on {cores} threads (disjoint chunks "
                      f"of {_chunk_units(name)}); one thread: {d1} in {t1:.1f} s; C oracle, gcc -O2"}


def run_reference(args):
    """The CPU oracle as the reference arm, on the same workload and metric,
    one thread per host core over disjoint chunks.  Runs no GPU code; under
    torchrun only rank 0 works."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle as O
    O.build()
    name = args.workload
    smp = oracle_sample(name, _sample_rows(name))
    model, cores = host_cpu()
    K, W = args.steps, args.warmup
    per_step_s = args.ref_seconds / max(1, K + W)
    for _ in range(W):
        oracle_timed(name, smp, per_step_s, cores)
    done, dt = 0, 0.0
    for _ in range(K):
        d, t = oracle_timed(name, smp, per_step_s, cores)
        done += d
        dt += t
    value = done / dt
    config, unit_name = describe(name)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": dt * 1e3 / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(config, units=unit_name, parallelism="cpu oracle, rank 0 only"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "cpu": model,
                         "sample": f"{done // K} {unit_name} per step of the {name} workload on {cores} "
                                   f"threads (disjoint chunks of {_chunk_units(name)})"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_latency_table(dev, stream, reps=1000):
    """Per-launch latency of the store family and the c1 / c2 decode compressors
    at the small batches of the store-latency table ([P1], bs 1/8/64/512):
    CUDA graphs of back-to-back launches on one set of inputs (hot L2, as a
    latency microbenchmark), per-launch time = graph time / launches, the best
    of five replays."""
    import torch
    import compress_kv_write_gb300 as K
    from compress_kv_write_gb300 import synth
    pool_slots = 1 << 20
    pool = torch.zeros(pool_slots * 528, dtype=torch.uint8, device=dev)
    cs = synth.rope_table(65536, dev)
    w = synth.norm_weight(dev, 0)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
        replay_once([(g, 1)], stream)
        best = min(time_plan([(g, 1)], stream) for _ in range(5))  # short regions: best of five
        return best * 1e3 / reps

    table = {}
    for bs in (1, 8, 64, 512):
        x = synth.store_rows_bf16(bs, dev, bs)
        loc = synth.injective_slots(bs, pool_slots, dev, bs)
        pos = synth.positions(bs, dev, bs)
        for name, flags in (("store", 0), ("store + RoPE", 1), ("fused K norm + RoPE", 3)):
            us = timed(lambda: K.kvq_store(1, 6, flags, x, loc, pool, pool_slots, norm_weight=w, eps=1e-6,
                                           cos_sin=cs, pos=pos))
            table.setdefault(name, {})[bs] = round(us, 3)
        v, sc = synth.compressor_rows(bs, dev, bs)
        loc32 = loc.to(torch.int32)
        for name, r in (("c1", 1), ("c2", 2)):
            state = torch.zeros((bs, 3, 512), dtype=torch.float32, device=dev)
            count = torch.zeros(bs, dtype=torch.int32, device=dev)
            us = timed(lambda: K.kvq_compress_decode(1, 6, r, K.FLAG_ROPE, v, sc, state, count, loc32, pool,
                                                     pool_slots, cos_sin=cs, group_pos=pos))
            table.setdefault(name, {})[bs] = round(us, 3)
    del pool
    torch.cuda.empty_cache()
    return table


def run_sweep(args):
    """The latency table alone, as its own JSON line."""
    import torch
    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    stream = torch.cuda.Stream(device=dev)
    reps = max(1000, args.steps)
    table = run_latency_table(dev, stream, reps)
    us512 = table["fused K norm + RoPE"][512]
    line = {
        "metric": METRIC, "value": 512 / (us512 * 1e-6), "unit": "tokens/s", "n_gpus": 1, "steps": reps,
        "warmup": 3, "ms_per_step": us512 / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "latency sweep (value: fused K norm + RoPE, V41, bs 512)",
                   "layout": "V41", "x_dtype": "bf16", "pool_slots": 1 << 20,
                   "l2": "hot: one input set per batch size (latency microbenchmark)",
                   "c1_c2": "kvq_compress_decode, ratio 1 / 2, one row per request, RoPE"},
        "latency_us": table,
        "gpu_launches": reps,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None, choices=sorted(DEFAULT_STEPS) + ["sweep"],
                    help=f"time one workload (default: {HEADLINE} as the headline, with every other "
                         "configured workload timed in the same run)")
    ap.add_argument("--suite", action="store_true", help="with --workload: time the other workloads too")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=None,
                    help="profiling only: shrink the workload to about this many tokens")
    ap.add_argument("--flush-l2", action="store_true",
                    help="profiling only: evict L2 after every step (counts the write-back in ncu)")
    args = ap.parse_args(argv)
    if args.workload is None:
        args.workload = HEADLINE
        args.suite = args.tokens is None and not args.flush_l2
    if args.steps is None:
        args.steps = DEFAULT_STEPS.get(args.workload, 20)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.workload == "sweep":
        if args.impl == "reference":
            raise SystemExit("the latency sweep has no reference arm")
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
