"""Build libssmscan.so in-tree with nvcc for sm_103a (B300).

    python selective_state_space_121_b300/build.py [--force] [-v] [--ptxas]

Each translation unit under csrc/ compiles in parallel to an object file, then
they link (with the CUDA runtime linked statically) into
selective_state_space_121_b300/libssmscan.so. The pipe-throughput probes under
probe/ build separately into libssmprobe.so (measurement only; the scan library
does not use them). No GPU is needed to build (nvcc cross-compiles).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libssmscan.so")
PROBE_SRC = os.path.join(PKG, "probe", "pipe_rates.cu")
PROBE_LIB = os.path.join(PKG, "libssmprobe.so")
OBJDIR = os.path.join(PKG, "_build")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(INCLUDE, "ssm_scan.h"), os.path.abspath(__file__)]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


def _obj(src):
    return os.path.join(OBJDIR, os.path.basename(src)[:-3] + ".o")


def build_probe(force: bool = False, verbose: bool = False) -> str:
    """libssmprobe.so from probe/pipe_rates.cu (one translation unit)."""
    deps = [PROBE_SRC, os.path.join(INCLUDE, "ssm_probe.h"), os.path.abspath(__file__)]
    if not force and os.path.exists(PROBE_LIB) and os.path.getmtime(PROBE_LIB) > max(map(os.path.getmtime, deps)):
        return PROBE_LIB
    tmp = PROBE_LIB + ".tmp"
    cmd = [NVCC, *ARCH, *FLAGS, "-shared", "-cudart", "static", "-o", tmp, PROBE_SRC]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    build_probe(force, verbose)
    if not force and not stale():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(INCLUDE, "ssm_scan.h"), os.path.abspath(__file__)]
    newest_header = max(os.path.getmtime(h) for h in headers)
    procs = []
    objs = []
    for src in _sources():
        obj = _obj(src)
        objs.append(obj)
        if not force and os.path.exists(obj) and os.path.getmtime(obj) > max(os.path.getmtime(src), newest_header) \
                and not extra:
            continue
        cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stdout.write(out.decode())
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = LIB + ".tmp"
    cmd = [NVCC, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", "-o", tmp, *objs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv or "--ptxas" in sys.argv,
          extra=("-Xptxas", "-v") if "--ptxas" in sys.argv else ())
    print(LIB)
