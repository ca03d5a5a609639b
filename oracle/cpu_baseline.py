"""Time the fp64 oracle, as it stands, on a bounded sample of a named workload.

TEST INFRASTRUCTURE ONLY: used by the benchmark's CPU-baseline leg and its
``--impl reference`` arm.  Run as a module in a child process so that the
BLAS thread count can be pinned before NumPy loads:

    OPENBLAS_NUM_THREADS=1 OMP_NUM_THREADS=1 python -m oracle.cpu_baseline decode_8b 10

prints one JSON object: KV bytes read by the oracle (unique pages of the
sequences it processed), seconds, GB/s, the worker count and the sample
description.  A name ending in ``_fp8`` times the FP8-page oracle on that
workload's FP8 variant (variant seed 0).  The workload's new tokens are
scattered into the caches before timing; the timed work is the oracle's paged
attention over whole sequences.  It runs on every host core this process may
use (one worker process per core, each with single-threaded BLAS): worker i
takes sequences i, i + P, i + 2P, ... of the batch, wrapping, until ``seconds``
have elapsed.  The workers are forked from this process, which never touches
a GPU.
"""
from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402
from oracle import fp8 as F  # noqa: E402
from oracle import oracle as O  # noqa: E402


def threads_used() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "") != "1":
            return len(os.sched_getaffinity(0))
    return 1


def prepare(name: str):
    if name.endswith("_fp8"):
        w = W.fp8_variant(W.FULL[name[:-4]](), seed=0)
        k, v = F.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                                   w.k_scale, w.v_scale, w.block_size)
        return w, k, v
    w = W.FULL[name]()
    k, v = O.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping,
                               w.block_size)
    return w, k, v


def seq_bytes(w, seqs) -> int:
    used = set()
    for b in seqs:
        nblk = -(-int(w.context_lens[b]) // w.block_size)
        used.update(int(x) for x in w.block_tables[b, :nblk])
    return len(used) * w.num_kv_heads * w.page_bytes()


def run_seqs(w, k, v, seqs):
    """Oracle attention over exactly ``seqs``, one sequence at a time; returns seconds."""
    t0 = time.perf_counter()
    for b in seqs:
        if w.kv_dtype == "fp8":
            F.paged_attention(w.q, k, v, w.k_scale, w.v_scale, w.block_tables, w.context_lens,
                              w.scale, w.num_kv_heads, w.block_size, seqs=[b])
        else:
            O.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                              w.num_kv_heads, w.block_size, seqs=[b])
    return time.perf_counter() - t0


def time_passes(w, k, v, seconds: float):
    """Oracle passes over the batch on one core, one sequence at a time, until ``seconds``
    elapsed."""
    return _worker_passes(w, k, v, seconds, 0, 1)


def _worker_passes(w, k, v, seconds, first, stride):
    done = []
    t0 = time.perf_counter()
    b = first % w.num_seqs
    while not done or time.perf_counter() - t0 < seconds:
        run_seqs(w, k, v, [b])
        done.append(b)
        b = (b + stride) % w.num_seqs
    dt = time.perf_counter() - t0
    nbytes = sum(seq_bytes(w, [x]) for x in done)
    return {"bytes": nbytes, "seconds": dt, "gbps": nbytes / dt / 1e9, "seqs": len(done),
            "seq_steps_per_s": len(done) / dt}


_STATE = {}


def _pool_task(args):
    first, stride, seconds = args
    w, k, v = _STATE["wkv"]
    return _worker_passes(w, k, v, seconds, first, stride)


def _pool_seqs(seqs):
    w, k, v = _STATE["wkv"]
    return run_seqs(w, k, v, seqs)


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


def make_pool(w, k, v, workers: int):
    """A pool of ``workers`` processes forked from this (GPU-free) process, sharing the
    prepared workload."""
    import multiprocessing as mp
    _STATE["wkv"] = (w, k, v)
    return mp.get_context("fork").Pool(workers)


def time_passes_parallel(w, k, v, seconds: float, workers: int):
    """``workers`` processes run oracle passes for ``seconds`` each; GB/s over the slowest
    worker's time."""
    t0 = time.perf_counter()
    with make_pool(w, k, v, workers) as pool:
        parts = pool.map(_pool_task, [(i, workers, seconds) for i in range(workers)])
    wall = time.perf_counter() - t0
    nbytes = sum(p["bytes"] for p in parts)
    nseq = sum(p["seqs"] for p in parts)
    # Each worker stops after its own `seconds`; the slowest sets the wall time.
    slowest = max(p["seconds"] for p in parts)
    return {"bytes": nbytes, "seconds": slowest, "wall_seconds": wall,
            "gbps": nbytes / slowest / 1e9, "seqs": nseq, "seq_steps_per_s": nseq / slowest}


def main(argv):
    name = argv[1] if len(argv) > 1 else "decode_8b"
    seconds = float(argv[2]) if len(argv) > 2 else 10.0
    workers = int(argv[3]) if len(argv) > 3 else host_cores()
    w, k, v = prepare(name)
    r = time_passes_parallel(w, k, v, seconds, workers)
    r.update({"workload": name, "cores": workers,
              "sample": f"{r['seqs']} whole sequences of the {name} batch, fp64 paged "
                        f"attention on {workers} worker processes (one per host core, "
                        f"single-threaded BLAS; worker i takes sequences i, i+{workers}, ..., "
                        f"wrapping) for {seconds:g} s; reshape_and_cache untimed"})
    print(json.dumps(r))


if __name__ == "__main__":
    main(sys.argv)
