"""Builds the CUDA library in-tree for sm_103a (nvcc, no cmake).

Each translation unit compiles in parallel; the objects link into
``libdsa.so`` beside this file.  Host code carries no machine-specific flags
so the same sources build on x86_64 and aarch64.
"""

from __future__ import annotations

import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libdsa.so")
BUILD_DIR = os.path.join(ROOT, "_build", platform.machine())
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "indexer.cu", "indexer_nvfp4.cu", "topk.cu", "mla.cu", "cache_write.cu", "dcp.cu", "block_topk.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                   "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")] + list(extra)


_ELF_MACHINE = {"x86_64": 0x3E, "AMD64": 0x3E, "aarch64": 0xB7, "arm64": 0xB7}


def foreign_binary(path: str) -> bool:
    """True when an ELF file was built for another CPU than this one."""
    want = _ELF_MACHINE.get(platform.machine())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return True
    if len(head) < 20 or head[:4] != b"\x7fELF" or want is None:
        return True
    return int.from_bytes(head[18:20], "little") != want


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out) or foreign_binary(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "dsa.h"))
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or ptxas_info or _stale(o, [s] + headers):
            extra = ["-Xptxas", "-v"] if ptxas_info else []
            jobs.append([nvcc()] + _flags(extra) + ["-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        logs = list(ex.map(run, jobs))
    if verbose or ptxas_info:
        for l in logs:
            print(l)
    if jobs or not os.path.exists(LIB) or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        run([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, ptxas_info="--ptxas" in sys.argv))
