"""Build the native libraries in-tree: the sm_103a CUDA library (libpagedattn.so), the
device-side input generator used by tests and the benchmark (libpasynth.so) and the CPU
oracle (liboracle.so, test infrastructure).

    python -m paged_kv_cache_223_gb300._build
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
from typing import List

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_223_gb300")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "_lib", "libpagedattn.so")
SYNTH_LIB = os.path.join(ROOT, "synth", "_lib", "libpasynth.so")
SYNTH_HOST_LIB = os.path.join(ROOT, "synth", "_lib", "libsynthhost.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest(paths: List[str]) -> float:
    return max(os.path.getmtime(p) for p in paths)


def _build_so(name: str, srcs: List[str], deps: List[str], out: str, includes: List[str], force: bool) -> str:
    if not force and os.path.exists(out) and os.path.getmtime(out) >= _newest(srcs + deps):
        return out
    objdir = os.path.join(BUILD_DIR, name)
    os.makedirs(objdir, exist_ok=True)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    inc = [f"-I{d}" for d in includes]

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc()] + ARCH + NVCC_FLAGS + inc + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = out + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {out} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


def build_cuda(force: bool = False) -> str:
    csrc = os.path.join(PKG, "csrc")
    srcs = sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cpp")))
    deps = sorted(glob.glob(os.path.join(csrc, "*.h")) + glob.glob(os.path.join(csrc, "*.cuh")) +
                  [os.path.join(INCLUDE, "pagedattn.h")])
    return _build_so("pagedattn", srcs, deps, LIB, [INCLUDE, csrc], force)


def build_synth(force: bool = False) -> str:
    src = os.path.join(ROOT, "synth", "csrc", "synth.cu")
    return _build_so("synth", [src], [], SYNTH_LIB, [], force)


def build_synth_host(force: bool = False) -> str:
    src = os.path.join(ROOT, "synth", "csrc", "synth_host.c")
    out = SYNTH_HOST_LIB
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(out), exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               src, "-o", tmp])
        os.replace(tmp, out)
    return out


def build_oracle(force: bool = False) -> str:
    import importlib
    import sys
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    return importlib.import_module("oracle").build(force=force)


def build_all(force: bool = False) -> List[str]:
    with cf.ThreadPoolExecutor(max_workers=4) as ex:
        futs = [ex.submit(build_cuda, force), ex.submit(build_synth, force), ex.submit(build_synth_host, force),
                ex.submit(build_oracle, force)]
        return [f.result() for f in futs]


if __name__ == "__main__":
    import sys
    for p in build_all(force="--force" in sys.argv):
        print(p)
