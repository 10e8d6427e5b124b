"""Build libkvq.so (the C ABI of include/kvq.h) for sm_103a with nvcc.

Each translation unit under csrc/ is compiled in parallel to an object file,
then the objects are linked into ``compress_kv_write_gb300/_build/libkvq.so``
against the shared CUDA runtime (the one PyTorch already loaded).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
SO = os.path.join(BUILD, "libkvq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + [os.path.join(ROOT, "include", "kvq.h"), os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(SO):
        return False
    t = os.path.getmtime(SO)
    return all(os.path.getmtime(d) <= t for d in _deps())


def cflags(extra=()):
    return (["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
             "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
            + ARCH + list(extra))


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile and link libkvq.so; returns its path."""
    if not force and up_to_date():
        return SO
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    objdir = tempfile.mkdtemp(prefix="obj_", dir=BUILD)
    try:
        def compile_one(src):
            obj = os.path.join(objdir, os.path.basename(src) + ".o")
            cmd = [exe, "-c", src, "-o", obj] + cflags(extra)
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout, r.stderr)
            return obj

        srcs = _sources()
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
            objs = list(ex.map(compile_one, srcs))
        fd, tmp = tempfile.mkstemp(suffix=".so", dir=BUILD)
        os.close(fd)
        cmd = [exe, "-shared", "-o", tmp] + objs + ["-cudart", "shared"] + ARCH
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, SO)
    finally:
        shutil.rmtree(objdir, ignore_errors=True)
    return SO


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
