"""Run the fp64 oracle over every sequence of a full-size workload on all host cores.

The oracle's per-sequence work is NumPy arithmetic (BLAS products, ufuncs) that
releases the GIL, so disjoint sequence subsets run on a thread pool in this
process: no process pool, so nothing is forked from a process that holds a CUDA
context, and the pools are shared rather than copied.
"""
import concurrent.futures
import os

import numpy as np


def all_rows(fn, num_seqs, *args, workers=None, **kwargs):
    """``fn(*args, seqs=subset, **kwargs)`` over interleaved subsets of 0..num_seqs-1;
    the rows of each subset are taken from its own call.  ``fn`` returns an array whose
    first axis is the sequence (rows outside ``seqs`` unspecified)."""
    workers = workers or max(1, min(num_seqs, len(os.sched_getaffinity(0))))
    subsets = [list(range(i, num_seqs, workers)) for i in range(workers)]
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        parts = list(ex.map(lambda s: (s, fn(*args, seqs=s, **kwargs)), subsets))
    out = np.array(parts[0][1], copy=True)
    for s, r in parts[1:]:
        out[s] = r[s]
    return out
