"""bench.py's host-side logic without a GPU: every workload describes itself,
its oracle sample runs, the committed traffic table is found, and the
reference arm (the CPU oracle) prints one JSON line with the contract's keys."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}


@pytest.mark.parametrize("name", sorted(bench.SPECS))
def test_workload_description_and_oracle_sample(name):
    cfg, unit = bench.describe(name)
    assert cfg["workload"] == name and unit
    smp = bench.oracle_sample(name, bench._sample_rows(name) if bench.SPECS[name]["kind"] != "compress"
                              or bench.SPECS[name]["ratio"] < 128 else 256)
    done = bench.oracle_run(name, smp, bench._chunk_units(name))
    assert done >= 1
    assert len(bench.kernel_source_sha(name)) == 16


def test_traffic_table_follows_the_sources():
    """A committed capture resolves to its traffic figure only while the
    dominant kernel's sources are unchanged since it was taken; a stale
    capture gives None (the JSON line then carries null)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    rows = [ln.split() for ln in open(path).read().splitlines() if ln.strip() and not ln.startswith("#")]
    assert rows
    for p in rows:
        name, sha = p[0], p[3]
        assert name in bench.SPECS
        got = bench.traffic_from_profiles(name)
        if sha == bench.kernel_source_sha(name):
            assert got is not None and got > 0, name
        elif not any(q[0] == name and q[3] == bench.kernel_source_sha(name) for q in rows):
            assert got is None, name


@pytest.mark.parametrize("name", ["store_norm_rope", "fp4_dequant", "c4a"])
def test_reference_arm_json(name, monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", name, "--steps", "3", "--warmup", "3",
                    "--ref-seconds", "0.3"])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["config"]["workload"] == name
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["cpu"]


def test_cpu_baseline_threads_and_model():
    """The CPU baseline reports one thread and one thread per host core, with
    the host CPU named."""
    cb = bench.cpu_baseline("store_norm_rope", 0.4)
    model, cores = bench.host_cpu()
    assert cb["cores"] == cores >= 1 and cb["cpu"] == model and model
    assert cb["value"] > 0 and cb["single_thread"]["value"] > 0 and cb["single_thread"]["cores"] == 1


def test_default_is_the_largest_config_with_the_suite():
    """No --workload: the mixed C128A batch is the headline and the suite holds
    every other configured workload."""
    assert bench.HEADLINE == "c128a"
    assert set(bench.SUITE) | {bench.HEADLINE} == set(bench.SPECS)


def test_clock_summary_uses_busy_samples():
    busy = "2070, 2070, 100, Not Active, Not Active, Not Active, Active"
    idle = "345, 2070, 0, Not Active, Not Active, Not Active, Not Active"
    c = bench.ClockSampler.summarise([idle, busy, busy, idle])
    assert c["sm_mhz"] == 2070 and c["samples"] == 2 and c["under_load"]
    assert c["reasons"] == ["sw_power_cap"]
    c = bench.ClockSampler.summarise([idle])
    assert not c["under_load"] and c["sm_mhz"] == 345


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--impl", "reference", "--warmup", "2"])


def test_source_hash_ignores_comments_only():
    a = "int f(int x) {  // doubles\n  return 2 * x; /* no overflow\n check */ }\n"
    b = "int f(int x) {\n  // a different comment\n  return 2 * x;\n}\n"
    c = "int f(int x) { return 3 * x; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def _csrc_constant(fname, name):
    import re
    text = open(os.path.join(ROOT, "compress_kv_write_gb300", "csrc", fname)).read()
    return int(re.search(r"constexpr int64_t " + name + r" = (\d+);", text).group(1))


def test_store_kernel_names_follow_the_library_dispatch():
    """bench.py names the store kernel a batch runs on (the dominant kernel of
    a store record): its size limits are the library's dispatch constants."""
    small_norm = _csrc_constant("kvq_store.cuh", "kSmallNormMax")
    small_rope = _csrc_constant("kvq_store.cuh", "kSmallRopeTwoMax")
    small = _csrc_constant("kvq_store.cuh", "kSmallTwoMax")
    rope_half = _csrc_constant("kvq_store.cu", "kRopeHalfMin")
    plain_half = _csrc_constant("kvq_store.cu", "kPlainHalfMin")
    norm_half = _csrc_constant("kvq_store.cu", "kNormHalfMin")
    name = bench.store_kernel_name
    for layout, flags, limit in ((1, 0, small), (1, 1, small_rope), (1, 2, small_norm), (1, 3, small_norm),
                                 (2, 0, small), (2, 1, small), (2, 3, small_norm)):
        assert name(layout, flags, limit) == "store_token_kernel"
        assert name(layout, flags, limit + 1) != "store_token_kernel"
    assert name(1, 1, rope_half - 1) == "store_warp_kernel"
    assert name(1, 1, rope_half) == "store_half_kernel"
    assert name(1, 0, plain_half - 1) == "store_warp_kernel" and name(1, 0, plain_half) == "store_half_kernel"
    for flags in (2, 3):
        assert name(1, flags, norm_half - 1) == "store_warp_kernel"
        assert name(1, flags, norm_half) == "store_half_kernel"
    assert name(2, 0, 16384) == "store_half_kernel"


def test_kernel_sources_exist():
    for files in bench.KERNEL_SOURCES.values():
        for fn in files:
            assert os.path.exists(os.path.join(ROOT, "compress_kv_write_gb300", "csrc", fn)), fn
