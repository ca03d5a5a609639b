"""Build ``libpaged_attn.so`` in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel into ``_build/``; the shared
library links the CUDA runtime statically so it loads without a driver (the
symbol-export tests run on machines with no GPU).  Re-running only rebuilds
what changed: each object, and the library, is keyed on a hash of what it is
built from (source and header contents, compiler flags, nvcc version and host
architecture), stored beside it, so a binary built elsewhere or from other
sources is never reused.
"""
from __future__ import annotations

import concurrent.futures
import functools
import hashlib
import os
import platform
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
           "pa_spec.cu", "pa_no_alloc.cu", "attn_tc_d128.cu", "stream_d64.cu", "stream_d128.cu",
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


@functools.lru_cache(maxsize=1)
def _toolchain_id() -> str:
    r = subprocess.run([nvcc_path(), "--version"], capture_output=True, text=True)
    return r.stdout.strip().splitlines()[-1] if r.returncode == 0 else "unknown nvcc"


def _digest(parts) -> str:
    h = hashlib.sha256()
    for x in parts:
        h.update(x if isinstance(x, bytes) else str(x).encode())
        h.update(b"\0")
    return h.hexdigest()


def _read(p) -> bytes:
    with open(p, "rb") as f:
        return f.read()


def _stamp_ok(path: str, stamp: str) -> bool:
    s = path + ".sha256"
    return os.path.exists(path) and os.path.exists(s) and _read(s).decode().strip() == stamp


def _write_stamp(path: str, stamp: str) -> None:
    with open(path + ".sha256", "w") as f:
        f.write(stamp + "\n")


def _compile(src: str, obj: str, extra):
    cmd = [nvcc_path(), *GENCODE, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile every translation unit whose inputs changed and link the library; return
    its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = list(extra_flags or [])
    common = [platform.machine(), _toolchain_id(), *GENCODE, *FLAGS, *extra]
    headers = sorted(_headers())
    header_bytes = [x for h in headers for x in (os.path.basename(h), _read(h))]
    jobs = []
    objs = []
    stamps = []
    for name in SOURCES:
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD_DIR, name + ".o")
        stamp = _digest([*common, name, _read(src), *header_bytes])
        objs.append(obj)
        stamps.append(stamp)
        if force or not _stamp_ok(obj, stamp):
            jobs.append((src, obj, stamp))
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            futs = {ex.submit(_compile, s, o, extra): (s, o, st) for s, o, st in jobs}
            for f in concurrent.futures.as_completed(futs):
                log = f.result()
                src, obj, stamp = futs[f]
                _write_stamp(obj, stamp)
                if verbose and log:
                    print(f"[{os.path.basename(src)}]\n{log}", file=sys.stderr)
    link = [nvcc_path(), *GENCODE, "-shared", "-cudart", "static"]
    lib_stamp = _digest([platform.machine(), _toolchain_id(), *link, *stamps])
    if force or jobs or not _stamp_ok(LIB_PATH, lib_stamp):
        tmp = LIB_PATH + ".tmp"
        r = subprocess.run([*link, "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
        _write_stamp(LIB_PATH, lib_stamp)
    return LIB_PATH


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(force="--force" in sys.argv, verbose=v or bool(extra), extra_flags=extra))
