"""The benchmark's multi-rank path on CPU (gloo, world size 2).

The write path shards with no exchange: each rank runs an independent
replica, and the only collective is the max over ranks of the timed region.
These tests run that logic with two gloo ranks, and check that the reference
arm (the CPU oracle) works on rank 0 alone.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_SCRIPT = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank, world, local = bench.dist_env()
assert world == 2 and rank in (0, 1)
slowest = bench.max_over_ranks(1.5 + rank)
print("RESULT", rank, slowest, flush=True)
dist.barrier()
dist.destroy_process_group()
"""


def _launch(script, port, extra_env=None):
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   LOCAL_RANK=str(rank), WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", script], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=240)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_max_over_ranks_gloo():
    outs = _launch(RANK_SCRIPT.format(root=ROOT), _free_port())
    for rank, out in enumerate(outs):
        line = [ln for ln in out.splitlines() if ln.startswith("RESULT")][0].split()
        assert int(line[1]) == rank and float(line[2]) == 2.5


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def test_reference_arm_rank0_only():
    """Under a 2-rank launch the reference arm prints one JSON line on rank 0
    and nothing on rank 1, and runs no GPU code."""
    script = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
              "bench.main(['--impl', 'reference', '--workload', 'store_norm_rope', '--steps', '3', "
              "'--warmup', '3', '--ref-seconds', '0.5'])")
    outs = _launch(script, _free_port())
    lines0 = [ln for ln in outs[0].splitlines() if ln.startswith("{")]
    assert len(lines0) == 1
    d = json.loads(lines0[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert not [ln for ln in outs[1].splitlines() if ln.startswith("{")]
