"""Build ``libpaged_attn.so`` in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel into ``_build/``; the shared
library links the CUDA runtime statically so it loads without a driver (the
symbol-export tests run on machines with no GPU).  Re-running only rebuilds
what changed.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libpaged_attn.so")

SOURCES = ["pa_api.cpp", "pa_misc.cu", "attn_d64.cu", "attn_d128.cu", "group_d64.cu",
           "group_d128.cu", "attn8_d64.cu", "attn8_d128.cu", "group8_d64.cu", "group8_d128.cu",
           "pa_spec.cu", "pa_no_alloc.cu",
           "pa_runner.cpp", "pa_block_manager.cpp"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE,
         "-I" + CSRC]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    p = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(p):
        return p
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _headers():
    hs = [os.path.join(INCLUDE, "paged_attn.h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def _mtime(p):
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def _compile(src: str, obj: str, extra):
    cmd = [nvcc_path(), *GENCODE, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile every translation unit that changed and link the library; return its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = list(extra_flags or [])
    newest_header = max(_mtime(h) for h in _headers())
    jobs = []
    objs = []
    for name in SOURCES:
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD_DIR, name + ".o")
        objs.append(obj)
        if force or _mtime(obj) < max(_mtime(src), newest_header):
            jobs.append((src, obj))
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            futs = {ex.submit(_compile, s, o, extra): s for s, o in jobs}
            for f in concurrent.futures.as_completed(futs):
                log = f.result()
                if verbose and log:
                    print(f"[{os.path.basename(futs[f])}]\n{log}", file=sys.stderr)
    if force or jobs or _mtime(LIB_PATH) < max(_mtime(o) for o in objs):
        tmp = LIB_PATH + ".tmp"
        cmd = [nvcc_path(), *GENCODE, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(force="--force" in sys.argv, verbose=v or bool(extra), extra_flags=extra))
