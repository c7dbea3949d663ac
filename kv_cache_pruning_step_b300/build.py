"""Build libsprint.so (the SPRINT C-ABI library) for sm_103a with nvcc.

    python -m kv_cache_pruning_step_b300.build [--debug]

Objects go to _build/ at the repository root; the shared library is written
next to this file so that it ships with the package directory.  --debug
builds libsprint_debug.so instead (SPRINT_DEBUG_CHECKS=1: device-side
invariant checks that report SPRINT_STATUS_DEBUG_CHECK); the binding loads
it when SPRINT_LIBRARY names it.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "libsprint.so")
OUT_DEBUG = os.path.join(PKG, "libsprint_debug.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
         "-I" + os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _needs(obj, src, deps):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src] + deps)


def build(debug: bool = False, verbose: bool = False, force: bool = False) -> str:
    bdir = os.path.join(ROOT, "_build", "debug" if debug else "release")
    os.makedirs(bdir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "sprint.h"))
    extra = ["-DSPRINT_DEBUG_CHECKS=1"] if debug else []
    objs, jobs = [], []
    for src in sources():
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _needs(obj, src, headers):
            cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    out = OUT_DEBUG if debug else OUT
    if jobs or not os.path.exists(out) or force:
        link = [NVCC, *ARCH, "-shared", "-o", out, *objs]
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--debug", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/smem usage")
    ap.add_argument("--force", action="store_true")
    a = ap.parse_args()
    print(build(debug=a.debug, verbose=a.verbose, force=a.force))
