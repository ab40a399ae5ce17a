"""Build the two fillers of the synthetic input generator in-tree.

``libsynth_host.so`` is built by gcc (no GPU needed) and ``libsynth_dev.so``
by nvcc for sm_103a.  Both are rebuilt when a source is newer than the
library.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SO = os.path.join(HERE, "libsynth_host.so")
DEV_SO = os.path.join(HERE, "libsynth_dev.so")
_CORE = os.path.join(HERE, "synth_core.h")


def _stale(target: str, *sources: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _run(cmd: list[str]) -> None:
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("build failed: %s\n%s\n%s" % (" ".join(cmd), res.stdout, res.stderr))


def build_host(force: bool = False) -> str:
    src = os.path.join(HERE, "synth_host.c")
    if force or _stale(HOST_SO, src, _CORE):
        tmp = HOST_SO + ".tmp%d" % os.getpid()
        _run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
              "-Wall", "-o", tmp, src])
        os.replace(tmp, HOST_SO)
    return HOST_SO


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    p = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(p):
        return p
    raise RuntimeError("nvcc not found")


def build_device(force: bool = False) -> str:
    src = os.path.join(HERE, "synth_dev.cu")
    if force or _stale(DEV_SO, src, _CORE):
        tmp = DEV_SO + ".tmp%d" % os.getpid()
        _run([nvcc_path(), "-O3", "-std=c++17", "-fmad=false",
              "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-Xcompiler", "-fPIC", "-shared", "-o", tmp, src])
        os.replace(tmp, DEV_SO)
    return DEV_SO


if __name__ == "__main__":
    print(build_host(force=True))
    print(build_device(force=True))
