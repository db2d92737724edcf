"""Build libpfkv.so (and the synthetic-input helper libsynth.so) with nvcc for
sm_103a, in-tree, compiling translation units in parallel."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libpfkv.so")

SYNTH_SRC = os.path.join(ROOT, "synth", "csrc", "synth_fill.cu")
SYNTH_OUT = os.path.join(ROOT, "synth", "_build")
SYNTH_LIB = os.path.join(SYNTH_OUT, "libsynth.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
                     "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pfkv.h")]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("build step failed: " + " ".join(cmd))
    return r.stdout + r.stderr


def build_pfkv(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    if not force and not _stale(LIB, _deps()):
        return LIB
    nvcc = _nvcc()
    srcs = _sources()
    objs = [os.path.join(OUT, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = ["-Xptxas", "-v"] if verbose else []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        logs = list(ex.map(lambda so: _run([nvcc, *NVCC_FLAGS, *extra, "-c", so[0], "-o", so[1]]),
                           zip(srcs, objs)))
    if verbose:
        for lg in logs:
            sys.stderr.write(lg)
    tmp = LIB + f".tmp{os.getpid()}"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


def build_synth(force: bool = False) -> str:
    os.makedirs(SYNTH_OUT, exist_ok=True)
    if not force and not _stale(SYNTH_LIB, [SYNTH_SRC]):
        return SYNTH_LIB
    tmp = SYNTH_LIB + f".tmp{os.getpid()}"
    _run([_nvcc(), *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", SYNTH_SRC, "-o", tmp])
    os.replace(tmp, SYNTH_LIB)
    return SYNTH_LIB


def build_all(force: bool = False, verbose: bool = False):
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        f1 = ex.submit(build_pfkv, force, verbose)
        f2 = ex.submit(build_synth, force)
        return f1.result(), f2.result()


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv, verbose="-v" in sys.argv))
