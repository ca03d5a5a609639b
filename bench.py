#!/usr/bin/env python
"""Benchmark of the paged decode-attention hot path on GB300.

One step = one pass of the whole path over one batch: reshape_and_cache of
the batch's new tokens, then paged attention over every sequence's cache
(split-KV partitions + merge, and the read-once shared-prefix kernel for the
shared-prefix workload).  Default workload: the 8B-shape decode batch (64
sequences, 32 query / 8 kv heads, head_dim 128, block_size 16, contexts
uniform in [512, 4096], blocks shuffled through a pool 1.25x the need).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the fp64 CPU oracle, same metric
    python bench.py --aux-kernels            # reshape_and_cache and block copy alone
    python bench.py --spec-accept            # the speculative acceptance kernel
    python bench.py --runner-sweep           # small-batch step latency, graph runner

Prints one JSON line (rank 0).  ``value`` is KV-read GB/s of the whole step
(algorithmic bytes: every (block, kv head) page a step must read, once, x the
K and V page bytes) over the device time of K steps, summed over ranks; each
rank runs its own replica (the path shards by sequence with no exchange).
After the headline workload, every other workload and the FP8-page variants
are timed briefly in the same run and reported under ``configs``.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "paged decode-attention KV-read GB/s vs GB300 HBM peak; seq-steps/sec"
L2_BYTES = 129 * 1000 * 1000     # GB300 L2
KERNEL_SOURCES = ["pa_attn.cuh", "pa_attn_stream.cuh", "pa_ptx.cuh"]   # attention kernels, PTX
KERNEL_PARAMS = "pa_internal.h"                  # its constants and AttnParams (up to the struct end)
WORKLOAD_DESC = {
    "tiny": "2 seqs (ctx 37, 100), 4 q = 4 kv heads, head_dim 64, 16-block pool",
    "decode_8b": "64 seqs, ctx uniform [512, 4096], 32 q / 8 kv heads, head_dim 128",
    "decode_70b": "256 seqs, ctx log-uniform [128, 8192], 64 q / 8 kv heads, head_dim 128",
    "spec_verify": "32 seqs x 5 drafts, ctx uniform [2048, 16384], 32 q / 8 kv heads",
    "shared_prefix": "2 groups x 8 seqs sharing a 2048-token prefix, ctx 32768, 32 q / 8 kv "
                     "heads, 512-token partitions",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0 = about 1.5 s worth)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="decode_8b")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window (positions each query token sees); 0 = none")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="KV page format (fp8 = E4M3 pages with per-kv-head scales)")
    ap.add_argument("--partition-size", type=int, default=-1,
                    help="split-KV partition tokens (-1 = the workload's, 0 = library default)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--runner-sweep", action="store_true",
                    help="per-step latency of small batches: direct calls vs the graph runner")
    ap.add_argument("--spec-accept", action="store_true",
                    help="time the speculative acceptance kernel (greedy and sampling)")
    ap.add_argument("--aux-kernels", action="store_true",
                    help="time reshape_and_cache (bf16, FP8) and the block copy on their own")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (and FP8 variants) timed after the headline")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ----------------------------------------------------------------------------- helpers

def max_over_ranks(value: float, world: int, device=None) -> float:
    """The maximum of ``value`` over all ranks (the slowest replica sets the time)."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(bytes_per_rank_step: int, world: int, steps: int, ms_max: float) -> float:
    """KV bytes read by every rank over ``steps`` steps, divided by the slowest rank's time."""
    return bytes_per_rank_step * world * steps / (ms_max * 1e-3) / 1e9


def replica_workload(name: str, rank: int):
    """Rank ``rank``'s replica: the named workload drawn with its own seed (same shapes)."""
    import workloads as W
    make = W.FULL[name]
    default_seed = make.__defaults__[0] if make.__defaults__ else 0
    return make(default_seed + 1000 * rank)

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def strip_comments(src: bytes) -> bytes:
    """C/C++ source without its comments (string and character literals kept), and
    without blank lines and trailing spaces: what the compiler sees of the code."""
    out, i, n = bytearray(), 0, len(src)
    while i < n:
        c = src[i:i + 1]
        if src.startswith(b"//", i):
            j = src.find(b"\n", i)
            i = n if j < 0 else j
        elif src.startswith(b"/*", i):
            j = src.find(b"*/", i + 2)
            i = n if j < 0 else j + 2
        elif c in (b'"', b"'"):
            j = i + 1
            while j < n and src[j:j + 1] != c:
                j += 2 if src[j:j + 1] == b"\\" else 1
            out += src[i:j + 1]
            i = j + 1
        else:
            out += c
            i += 1
    lines = [ln.rstrip() for ln in bytes(out).split(b"\n")]
    return b"\n".join(ln for ln in lines if ln)


def kernel_source_hash():
    """Hash of what the attention kernels are compiled from (comments aside): their
    templates, their PTX helpers, and the constants and parameter struct they read
    (launcher declarations excluded)."""
    csrc = os.path.join(ROOT, "paged_kv_cache_221_gb300", "csrc")
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(strip_comments(f.read()))
    with open(os.path.join(csrc, KERNEL_PARAMS), "rb") as f:
        text = f.read()
    end = text.find(b"};", text.find(b"struct AttnParams"))
    h.update(strip_comments(text[:end + 2]))
    return h.hexdigest()[:16]


def recorded_capture(workload):
    """The committed ncu record of the attention call on this workload (its kernels and
    their DRAM bytes per launch), if the kernel sources have not changed since it was
    captured; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_src_sha") != kernel_source_hash():
        return None
    return e


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        """Median SM clock, maximum SM clock and active throttle reasons of the samples
        taken between t0 and t1 (wall clock)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in list(self.lines):
            if not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(workload, seconds):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "oracle.cpu_baseline", workload, str(seconds)],
                       cwd=ROOT, env=env, capture_output=True, text=True)
    if r.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"failed: {r.stderr.strip().splitlines()[-1:]}"}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": round(d["gbps"], 4), "unit": "GB/s", "cores": d["cores"], "kind": "oracle",
            "sample": d["sample"], "seconds": round(d["seconds"], 2),
            "seq_steps_per_s": round(d["seq_steps_per_s"], 3)}


def workload_config(w, ps, world, window=0):
    base = w.name[:-4] if w.name.endswith("_fp8") else w.name
    desc = WORKLOAD_DESC.get(base, base)
    if w.kv_dtype == "fp8":
        desc += "; FP8 (E4M3) K/V pages, per-kv-head scales"
    if window > 0:
        desc += f"; sliding window of {window} positions (only the pages under the windows " \
                f"are read and counted)"
    pool = (w.k_codes.nbytes + w.v_codes.nbytes) if w.kv_dtype == "fp8" else 2 * w.k_cache.nbytes
    return {"workload": w.name, "desc": desc, "kv_dtype": w.kv_dtype,
            "num_seqs": w.num_seqs, "query_tokens": w.num_query_tokens,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size, "pool_blocks": w.num_blocks,
            "partition_size": ps, "global_batch": w.num_seqs * world, "window": window,
            "l2": (("inputs larger than L2: each step reads %.2f GB of a %.2f GB pool "
                    "(L2 129 MB)") % (w.kv_bytes() / 1e9, pool / 1e9)) if pool > L2_BYTES else
                  (("inputs smaller than L2 (%.2f MB pool): L2-resident and launch-bound, "
                    "not a bandwidth figure") % (pool / 1e6)),
            "parallelism": "replicas" if world == 1 else f"replicas x{world}"}


def window_kv_bytes(w, window):
    """Algorithmic bytes with a sliding window: every (block, kv head) page from the
    block of the first query's first visible position to the context end, once."""
    used = set()
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        first = max(0, L - w.num_query_tokens - window + 1) // w.block_size
        nblk = -(-L // w.block_size)
        used.update(int(x) for x in w.block_tables[b, first:nblk])
    return len(used) * w.num_kv_heads * w.page_bytes()


def data_desc(w):
    if w.kv_dtype == "fp8":
        return ("synthetic (seeded N(0,1) bf16 q and new K/V, random E4M3 codes in the pool, "
                "random block placement)")
    return "synthetic (seeded N(0,1) bf16 q/K/V, random block placement)"


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    # Pin BLAS to one thread per process before NumPy loads; the oracle runs on every
    # host core as that many worker processes.
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    sys.path.insert(0, ROOT)
    from oracle import cpu_baseline as C

    w, k, v = C.prepare(args.workload + ("_fp8" if args.kv_dtype == "fp8" else ""))
    cores = C.host_cores()
    steps = args.steps if args.steps > 0 else 10
    # per-step sample: whole sequences for about 0.5 s of every core (less when many
    # steps are asked), spread over the workers one sequence per task
    per_seq = max(C.run_seqs(w, k, v, [0]), 1e-4)
    budget = 150.0 / max(1, steps + args.warmup)
    n = max(1, min(w.num_seqs, int(min(0.5, budget) * cores / per_seq)))
    ring = list(range(w.num_seqs)) * 2

    def sample(i):
        s0 = (i * n) % w.num_seqs
        return ring[s0:s0 + n]

    with C.make_pool(w, k, v, cores) as pool:
        def run(sm):
            t0 = time.perf_counter()
            pool.map(C._pool_seqs, [[b] for b in sm], chunksize=1)
            return time.perf_counter() - t0

        for i in range(args.warmup):
            run(sample(i))
        nbytes = 0
        nseq = 0
        dt = 0.0
        for i in range(steps):
            sm = sample(i)
            dt += run(sm)
            nbytes += sum(C.seq_bytes(w, [b]) for b in sm)
            nseq += len(sm)
    gbps = nbytes / dt / 1e9
    ps = w.partition_size
    line = {"impl": "reference", "metric": METRIC, "value": round(gbps, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(dt / steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": data_desc(w),
            "config": workload_config(w, ps, 1),
            "seq_steps_per_s": round(nseq / dt, 3),
            "cpu_baseline": {"value": round(gbps, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"{n} whole sequence(s) of the {w.name} batch per step "
                                       f"on {cores} worker processes (fp64 paged attention, "
                                       f"reshape untimed)"},
            "e2e": {"value": round(gbps, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GB300 arm

EXTRA_CONFIGS = ["tiny", "decode_70b", "spec_verify", "shared_prefix", "decode_8b:fp8",
                 "decode_70b:fp8", "spec_verify:fp8", "shared_prefix:fp8"]
L2_FLUSH_BYTES = 256 << 20      # written between the distribution pass's timed steps


def percentile(xs, q):
    s = sorted(xs)
    if not s:
        return None
    i = min(len(s) - 1, max(0, int(round(q / 100.0 * (len(s) - 1)))))
    return s[i]


class Case:
    """One workload on the device, its step (one pass of the whole hot path) captured as
    CUDA graphs, and the measurements of that step."""

    def __init__(self, pa, w, args, dev, window=0, partition_size=-1):
        import numpy as np
        import torch
        self.pa, self.torch, self.np = pa, torch, np
        self.w, self.dev, self.window = w, dev, window
        self.fp8 = w.kv_dtype == "fp8"
        if window > 0:
            w.seq_group = None               # the window runs the per-sequence path
            w.group_prefix_blocks = None
        self.ps = w.partition_size if partition_size < 0 else partition_size

        def td(a):
            t = torch.from_numpy(np.ascontiguousarray(a))
            if a.dtype == np.uint16:
                t = t.view(torch.int16).view(torch.bfloat16)
            return t.to(dev)

        self.q = td(w.q)
        self.k, self.v = (td(w.k_codes), td(w.v_codes)) if self.fp8 else \
            (td(w.k_cache), td(w.v_cache))
        self.ks, self.vs = (td(w.k_scale), td(w.v_scale)) if self.fp8 else (None, None)
        self.tables, self.lens = td(w.block_tables), td(w.context_lens)
        self.nk, self.nv, self.slots = td(w.new_key), td(w.new_value), td(w.slot_mapping)
        self.grouped = w.seq_group is not None
        self.sg = td(w.seq_group) if self.grouped else None
        self.gp = td(w.group_prefix_blocks) if self.grouped else None
        T = w.num_query_tokens
        need = pa.workspace_size(w.num_seqs, w.num_q_heads, T, w.max_context_len, w.head_dim,
                                 16, self.ps, w.max_prefix_blocks if self.grouped else 0)
        self.need = need
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(self.q)
        self.kv_bytes = w.kv_bytes() if window <= 0 else window_kv_bytes(w, window)
        # our kernels per step: attention (+ split-KV merge) (+ reshape + shared-prefix kernel)
        self.launches_per_step = 1 + (1 if need > 0 else 0) + (2 if self.grouped else 0)
        self.stream = torch.cuda.current_stream(dev)

    # Per-sequence workloads: one fused call (reshape_and_cache inside the attention
    # launch).  Shared-prefix workload: reshape_and_cache, then the shared-prefix call.
    def reshape(self):
        pa = self.pa
        if self.grouped and self.fp8:
            pa.reshape_and_cache_fp8(self.nk, self.nv, self.k, self.v, self.slots, self.ks,
                                     self.vs)
        elif self.grouped:
            pa.reshape_and_cache(self.nk, self.nv, self.k, self.v, self.slots)

    def attend(self):
        pa, w = self.pa, self.w
        if self.window > 0:
            pa.attention(self.q, self.k, self.v, self.tables, self.lens, w.max_context_len,
                         w.scale, self.ps, self.ws, self.out, self.nk, self.nv,
                         window_size=self.window, k_scale=self.ks, v_scale=self.vs)
        elif self.grouped:
            pa.decode_shared_prefix(self.q, self.k, self.v, self.tables, self.lens, self.sg,
                                    self.gp, w.max_group_size, w.max_prefix_blocks,
                                    w.max_context_len, w.scale, self.ps, self.ws, self.out,
                                    k_scale=self.ks, v_scale=self.vs)
        elif self.fp8:
            pa.verify_fp8(self.q, self.k, self.v, self.ks, self.vs, self.tables, self.lens,
                          w.max_context_len, w.scale, self.ps, self.ws, self.out, self.nk,
                          self.nv)
        else:
            pa.verify(self.q, self.k, self.v, self.tables, self.lens, w.max_context_len,
                      w.scale, self.ps, self.ws, self.out, self.nk, self.nv)

    def capture(self, warmup):
        torch, pa = self.torch, self.pa
        # warm-up outside capture (sets kernel attributes), then one graph per phase
        for _ in range(max(3, warmup)):
            self.reshape()
            self.attend()
        torch.cuda.synchronize(self.dev)
        assert pa.get_device_error(self.dev) == 0
        self.g_reshape = torch.cuda.CUDAGraph() if self.grouped else None
        self.g_attend = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(self.stream)
        with torch.cuda.stream(side):
            if self.grouped:
                with torch.cuda.graph(self.g_reshape, stream=side):
                    self.reshape()
            with torch.cuda.graph(self.g_attend, stream=side):
                self.attend()
        self.stream.wait_stream(side)
        for _ in range(max(3, warmup)):
            self.step()
        torch.cuda.synchronize(self.dev)

    def step(self):
        if self.g_reshape is not None:
            self.g_reshape.replay()
        self.g_attend.replay()

    def default_steps(self, seconds):
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for _ in range(20):
            self.step()
        e1.record(self.stream)
        e1.synchronize()
        per = e0.elapsed_time(e1) / 20
        return int(max(50, min(20000, seconds * 1000.0 / max(per, 1e-3))))

    def time_steps(self, steps, world):
        """K steps back to back, as a serving loop submits them (no event between steps);
        for the shared-prefix workload also the attention graph alone, K times."""
        torch = self.torch
        ev = lambda: torch.cuda.Event(enable_timing=True)      # noqa: E731
        start, stop, a_start, a_stop = ev(), ev(), ev(), ev()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(self.dev)
        t0 = time.time()
        start.record(self.stream)
        for _ in range(steps):
            self.step()
        stop.record(self.stream)
        if self.grouped:
            a_start.record(self.stream)
            for _ in range(steps):
                self.g_attend.replay()
            a_stop.record(self.stream)
        torch.cuda.synchronize(self.dev)
        t1 = time.time()
        if world > 1:
            dist.barrier()
        ms_total = max_over_ranks(start.elapsed_time(stop), world, self.dev)
        attn_avg = (a_start.elapsed_time(a_stop) / steps) if self.grouped else \
            start.elapsed_time(stop) / steps
        return ms_total, attn_avg, (t0, t1)

    def distribution(self, n):
        """Per-step device times of n steps, each bracketed by its own CUDA events on the
        launching stream, with a write of L2_FLUSH_BYTES (larger than L2) before each."""
        torch = self.torch
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=self.dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for e0, e1 in evs:
            flush.fill_(1.0)
            e0.record(self.stream)
            self.step()
            e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        ts = [e0.elapsed_time(e1) for e0, e1 in evs]
        del flush
        return {"p50_ms": round(percentile(ts, 50), 5), "p90_ms": round(percentile(ts, 90), 5),
                "min_ms": round(min(ts), 5), "n": n,
                "how": f"each step between its own CUDA events, a {L2_FLUSH_BYTES >> 20} MiB "
                       f"buffer written before each (L2 flush)"}

    def e2e(self, steps, world, args):
        """The same metric end to end through the public API: pinned host inputs in, the
        step, the output back to the host, every step."""
        torch, np, pa, w = self.torch, self.np, self.pa, self.w
        T = w.num_query_tokens
        total_bytes = self.kv_bytes * world
        h = {n: torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for n, a in
             (("q", w.q.view(np.int16)), ("nk", w.new_key.view(np.int16)),
              ("nv", w.new_value.view(np.int16)), ("slots", w.slot_mapping),
              ("tables", w.block_tables), ("lens", w.context_lens))}
        d_in = {"q": self.q.view(torch.int16), "nk": self.nk.view(torch.int16),
                "nv": self.nv.view(torch.int16), "slots": self.slots, "tables": self.tables,
                "lens": self.lens}
        h_out = torch.empty(self.out.shape, dtype=torch.int16).pin_memory()
        bi = sum(t.numel() * t.element_size() for t in h.values())
        bo = h_out.numel() * h_out.element_size()
        e2e_steps = max(10, min(steps, 1000))

        def binding_step():
            for n_ in h:
                d_in[n_].copy_(h[n_], non_blocking=True)
            self.reshape()
            self.attend()
            h_out.copy_(self.out.view(torch.int16), non_blocking=True)

        def timed(f):
            for _ in range(3):
                f()
            torch.cuda.synchronize(self.dev)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(self.stream)
            for _ in range(e2e_steps):
                f()
            s1.record(self.stream)
            torch.cuda.synchronize(self.dev)
            return max_over_ranks(s0.elapsed_time(s1) / e2e_steps, world, self.dev)

        e2e_ms = timed(binding_step)
        binding = {"value": round(total_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                   "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                   "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                   "path": "pinned host inputs -> H2D -> the step's library calls (Python "
                           "binding, no graph) -> D2H of the bf16 output"}
        if self.grouped:
            return binding
        # The serving path: the graph runner (one captured graph per batch class) with the
        # same pools; per step the inputs go into its static buffers, one replay, the
        # output comes back.
        used = set(int(x) for x in w.block_tables.ravel() if x >= 0)
        pad = next(bb for bb in range(w.num_blocks) if bb not in used)
        # partition size 0: the class is captured with the library default, as the
        # device-timed call uses it
        runner = pa.GraphRunner(self.k, self.v, w.num_q_heads, w.max_context_len,
                                w.max_blocks_per_seq, pad, max(self.ps, 0),
                                classes=(w.num_seqs,),
                                num_query_tokens=T, scale=w.scale, window_size=self.window,
                                k_scale=self.ks, v_scale=self.vs, host_staging=True)
        # the step's inputs sit in the runner's page-locked host buffers; every replay
        # copies them in, runs the step and copies the output back
        runner.h_q.view(torch.int16).copy_(h["q"].view(runner.h_q.shape))
        runner.h_new_key.view(torch.int16).copy_(h["nk"].view(runner.h_new_key.shape))
        runner.h_new_value.view(torch.int16).copy_(h["nv"].view(runner.h_new_value.shape))
        runner.h_block_tables.copy_(h["tables"])
        runner.h_context_lens.copy_(h["lens"])
        # one copy of the runner's input range (inputs laid out back to back)
        bir = (runner.h_context_lens.data_ptr() + runner.h_context_lens.numel() * 4 -
               runner.h_q.data_ptr())
        bor = runner.h_out.numel() * runner.h_out.element_size()
        r_ms = timed(lambda: runner.step(w.num_seqs))
        runner.close()
        return {"value": round(total_bytes / (r_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": bir, "d2h_bytes_per_step": bor,
                "ms_per_step": round(r_ms, 4), "steps": e2e_steps,
                "path": "pa_runner_step: one graph replay that copies the step's inputs "
                        "from page-locked host buffers, runs the attention step and copies "
                        "the bf16 output back to the host",
                "binding_path": binding}

    def roofline(self, attn_avg, peak, peak_kind):
        achieved = self.kv_bytes / (attn_avg * 1e-3) / 1e9
        # the recorded captures are of full-context launches
        rec = recorded_capture(self.w.name) if self.window <= 0 else None
        kern = rec["kernel"] if rec else "attention kernel"
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": rec["dram_bytes_per_launch"] if rec else None,
                "kernel": f"attention call ({kern} + splitkv_reduce_kernel)",
                "peak_source": f"{peak_kind} hbm_gbs",
                "launch_ms_avg": round(attn_avg, 5)}


def make_workload(spec, rank):
    """'name' or 'name:fp8' -> the replica workload of this rank."""
    import workloads as W
    name, _, fmt = spec.partition(":")
    w = replica_workload(name, rank)
    if fmt == "fp8":
        w = W.fp8_variant(w, seed=rank)
    return w


def run_gb300(args):
    import torch

    rank, world, local = dist_env()
    sys.path.insert(0, ROOT)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import paged_kv_cache_221_gb300 as pa

    spec = args.workload + (":fp8" if args.kv_dtype == "fp8" else "")
    c = Case(pa, make_workload(spec, rank), args, dev, args.window, args.partition_size)
    w = c.w
    c.capture(args.warmup)
    steps = args.steps if args.steps > 0 else c.default_steps(1.5)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ms_total, attn_avg, win = c.time_steps(steps, world)
    # keep sampling under the same load until there are enough samples
    t_end = time.time() + 0.6
    while time.time() < t_end:
        for _ in range(50):
            c.step()
        torch.cuda.synchronize(dev)
    clocks = sampler.summary(win[0], time.time())
    assert pa.get_device_error(dev) == 0, "device error during the timed region"
    peak, peak_kind = measured_peaks()
    line = {
        "metric": METRIC, "value": round(whole_job_gbps(c.kv_bytes, world, steps, ms_total), 2),
        "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(ms_total / steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV / f16 MMA / fp32 softmax" if c.fp8 else "bf16",
        "data": data_desc(w),
        "config": workload_config(w, c.ps, world, args.window),
        "seq_steps_per_s": round(w.num_seqs * world * steps / (ms_total * 1e-3), 1),
        "kv_bytes_per_step": c.kv_bytes,
        "roofline": c.roofline(attn_avg, peak, peak_kind),
        "distribution": c.distribution(min(steps, 100)),
        "clocks": clocks,
        "gpu_launches": c.launches_per_step * steps,
        "timing": "CUDA graph of the step replayed K times back to back between two CUDA "
                  "events on the launching stream (shared-prefix: reshape graph + attention "
                  "graph per step, and the attention graph alone K times for the call); "
                  "distribution: per-step events with an L2 flush before each step",
    }
    if not args.no_e2e:
        line["e2e"] = c.e2e(steps, world, args)
    del c
    torch.cuda.empty_cache()

    # Every other workload (and the FP8 page variants), briefly, in the same run.
    configs = {}
    if not args.no_configs and args.window <= 0 and args.partition_size < 0:
        for sp in EXTRA_CONFIGS:
            if sp == spec:
                continue
            cc = Case(pa, make_workload(sp, rank), args, dev)
            cc.capture(3)
            k_steps = cc.default_steps(0.3)
            t0 = time.time()
            ms_t, a_avg, _ = cc.time_steps(k_steps, world)
            # the sampler keeps running: take this config's samples under its own load
            t_end = time.time() + 0.35
            while time.time() < t_end:
                for _ in range(20):
                    cc.step()
                torch.cuda.synchronize(dev)
            ent = {"value": round(whole_job_gbps(cc.kv_bytes, world, k_steps, ms_t), 2),
                   "unit": "GB/s", "steps": k_steps,
                   "ms_per_step": round(ms_t / k_steps, 5),
                   "seq_steps_per_s": round(cc.w.num_seqs * world * k_steps / (ms_t * 1e-3),
                                            1),
                   "kv_bytes_per_step": cc.kv_bytes,
                   "roofline": cc.roofline(a_avg, peak, peak_kind),
                   "distribution": cc.distribution(min(k_steps, 50)),
                   "clocks": sampler.summary(t0, time.time()),
                   "gpu_launches": cc.launches_per_step * k_steps,
                   "config": workload_config(cc.w, cc.ps, world)}
            assert pa.get_device_error(dev) == 0, f"device error in {sp}"
            if not args.no_e2e:
                ent["e2e"] = cc.e2e(min(k_steps, 200), world, args)
            configs[cc.w.name] = ent
            del cc
            torch.cuda.empty_cache()
    sampler.stop()
    if configs:
        line["configs"] = configs

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec.replace(":fp8", "_fp8"), args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_runner_sweep(args):
    """Batches of 1 .. 16 sequences of the 8B-shape decode workload, one token each:
    the step through the Python binding (host checks + launches) against the same step
    replayed from the graph runner's class graphs (pad + one graph launch).  Host time
    per step, measured over many steps with a device synchronisation at the end."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_221_gb300 as pa
    import workloads as W
    w = W.FULL["decode_8b"]()
    dev = torch.device("cuda", 0)

    def td(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.to(dev)

    k, v = td(w.k_cache), td(w.v_cache)
    used = set(int(x) for x in w.block_tables.ravel() if x >= 0)
    pad = next(b for b in range(w.num_blocks) if b not in used)
    mcl = int(w.context_lens.max())
    classes = (1, 2, 4, 8, 16)
    r = pa.GraphRunner(k, v, w.num_q_heads, mcl, w.max_blocks_per_seq, pad, 0,
                       classes=classes, scale=w.scale)
    ws = torch.empty(max(pa.workspace_size(16, w.num_q_heads, 1, mcl, 128, 16, 0), 256),
                     dtype=torch.uint8, device=dev)
    rows = []
    for B in range(1, 17):
        q, tb, ln = td(w.q[:B]), td(w.block_tables[:B]), td(w.context_lens[:B])
        nk, nv = td(w.new_key[:B]), td(w.new_value[:B])
        out = torch.empty_like(q)
        r.q[:B].copy_(q)
        r.new_key[:B].copy_(nk)
        r.new_value[:B].copy_(nv)
        r.block_tables[:B].copy_(tb)
        r.context_lens[:B].copy_(ln)

        def direct():
            pa.verify(q, k, v, tb, ln, mcl, w.scale, 0, ws, out, nk, nv)

        def graph():
            r.step(B)

        res = {"B": B, "class": r.class_of(B)}
        stream = torch.cuda.current_stream(dev)
        for name, f in (("direct", direct), ("graph", graph)):
            for _ in range(20):
                f()
            torch.cuda.synchronize(dev)
            n = 300
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            e0.record(stream)
            for _ in range(n):
                f()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            res[name + "_wall_us"] = round((time.perf_counter() - t0) / n * 1e6, 2)
            res[name + "_device_us"] = round(e0.elapsed_time(e1) / n * 1e3, 2)
            # host cost alone: issue with the device idle between calls
            host = 0.0
            for _ in range(50):
                torch.cuda.synchronize(dev)
                h0 = time.perf_counter()
                f()
                host += time.perf_counter() - h0
            res[name + "_host_us"] = round(host / 50 * 1e6, 2)
        rows.append(res)
    r.close()
    print(json.dumps({"metric": "decode step latency, batches of 1-16 (8B shape, one token "
                                "per sequence)", "unit": "us per step (wall clock with the device "
                                "kept busy; device time by CUDA events; host issue time with "
                                "the device idle)",
                      "classes": list(classes), "partition_size": "library default per batch",
                      "max_context_len": mcl, "rows": rows}), flush=True)


def run_spec_accept_timing(args):
    """The speculative acceptance kernel on random probabilities (uniform drafts)."""
    import torch
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_221_gb300 as pa
    g = torch.Generator(device="cuda").manual_seed(0)
    rows = []
    for B, K, V in ((32, 5, 128256), (64, 5, 32000), (8, 8, 151936)):
        p = torch.rand(B, K + 1, V, device="cuda", generator=g)
        p /= p.sum(-1, keepdim=True)
        q = torch.rand(B, K, V, device="cuda", generator=g)
        q /= q.sum(-1, keepdim=True)
        d = torch.randint(0, V, (B, K), device="cuda", dtype=torch.int32, generator=g)
        a = torch.randint(0, 1 << 24, (B, K), device="cuda", dtype=torch.int32, generator=g)
        s = torch.randint(-(1 << 31), (1 << 31) - 1, (B,), device="cuda", dtype=torch.int32,
                          generator=g)
        for greedy in (False, True):
            def f():
                pa.spec_accept(p, d, q, a, s, greedy=greedy)
            for _ in range(5):
                f()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(50):
                f()
            e1.record()
            e1.synchronize()
            rows.append({"B": B, "K": K, "V": V, "greedy": greedy,
                         "us": round(e0.elapsed_time(e1) / 50 * 1000, 1)})
    print(json.dumps({"metric": "speculative acceptance kernel time", "unit": "us per call",
                      "rows": rows}), flush=True)


def prefill_slots(n_tokens, n_blocks, block_size, seed):
    """Slot mapping of a prefill chunk of n_tokens: sequences of 128 .. 2048 tokens (the
    last one cut at the chunk's end), each filling consecutive slots of distinct, randomly
    chosen blocks from their first slot."""
    import numpy as np
    rng = np.random.default_rng(seed)
    blocks = iter(rng.permutation(n_blocks))
    out = []
    while len(out) < n_tokens:
        L = min(int(rng.integers(128, 2049)), n_tokens - len(out))
        for j in range(0, L, block_size):
            b = next(blocks)
            out.extend(range(b * block_size, b * block_size + min(block_size, L - j)))
    return np.array(out, dtype=np.int64)


def run_aux_kernels(args):
    """The hot path's small kernels on their own: reshape_and_cache (bf16 and FP8 pages)
    for one decode step's new tokens and for a prefill-sized chunk, and the copy-on-write
    block copy.  Each case is 20 launches captured in a CUDA graph, replayed 10 times
    between two CUDA events; bytes are the algorithmic reads + writes of one launch."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_221_gb300 as pa
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)
    peak, peak_kind = measured_peaks()
    Hkv, D, BS = 8, 128, 16
    rows = []

    def timed(f, n_inner=20, n_outer=10):
        f()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for _ in range(n_inner):
                    f()
        torch.cuda.current_stream(dev).wait_stream(side)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n_outer):
            graph.replay()
        e1.record()
        e1.synchronize()
        assert pa.get_device_error(dev) == 0
        return e0.elapsed_time(e1) / (n_inner * n_outer) * 1e3     # us per launch

    def row(kernel, case, nbytes, us):
        gbps = nbytes / (us * 1e-6) / 1e9
        rows.append({"kernel": kernel, "case": case, "bytes": nbytes, "us": round(us, 3),
                     "gbps": round(gbps, 1), "frac": round(gbps / peak, 4)})

    for N, case in ((256, "one 70B-shape decode step: 256 new tokens"),
                    (16384, "a 16384-token prefill chunk (sequences of 128-2048 tokens in "
                            "consecutive slots)")):
        nb = int(N / BS * 1.25) + 16
        k = torch.zeros(nb, Hkv, BS, D, dtype=torch.bfloat16, device=dev)
        v = torch.zeros_like(k)
        key = torch.randn(N, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
        val = torch.randn(N, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
        if N == 256:
            # a decode step: one new token per sequence, each at its own slot
            slots = torch.randperm(nb * BS, device=dev, generator=g)[:N].to(torch.int64)
        else:
            # a prefill chunk: sequences of 128 .. 2048 tokens one after another, each
            # filling consecutive slots of its own randomly placed blocks
            slots = torch.from_numpy(prefill_slots(N, nb, BS, seed=5)).to(dev)
        vec = N * Hkv * D * 2
        us = timed(lambda: pa.reshape_and_cache(key, val, k, v, slots))
        row("reshape_and_cache_kernel", case, 2 * vec + 2 * vec + N * 8, us)
        k8 = torch.zeros(nb, Hkv, BS, D, dtype=torch.uint8, device=dev)
        v8 = torch.zeros(nb, Hkv, D, BS, dtype=torch.uint8, device=dev)
        ks = torch.full((Hkv,), 1 / 64, device=dev)
        vs = torch.full((Hkv,), 1 / 32, device=dev)
        us = timed(lambda: pa.reshape_and_cache_fp8(key, val, k8, v8, slots, ks, vs))
        row("reshape_and_cache_fp8_kernel", case, 2 * vec + vec + N * 8, us)
        del k, v, k8, v8
    nb = 8192
    k = torch.randn(nb, Hkv, BS, D, device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn(nb, Hkv, BS, D, device=dev, generator=g).to(torch.bfloat16)
    for P in (64, 2048):
        perm = torch.randperm(nb, device=dev, generator=g)
        pairs = torch.stack([perm[:P], perm[P:2 * P]], 1).to(torch.int32).contiguous()
        us = timed(lambda: pa.copy_blocks(k, v, pairs))
        row("copy_blocks_kernel", f"{P} block pairs, 8 kv heads, head_dim 128",
            P * 2 * Hkv * BS * D * 2 * 2 + P * 8, us)
    print(json.dumps({"metric": "auxiliary kernels: algorithmic bytes (reads + writes) per "
                                "launch over the launch time",
                      "unit": "GB/s", "peak": peak, "peak_source": f"{peak_kind} hbm_gbs",
                      "timing": "20 launches in a CUDA graph, replayed 10 times between two "
                                "CUDA events",
                      "rows": rows}), flush=True)


def main():
    args = parse_args()
    if args.runner_sweep:
        run_runner_sweep(args)
        return
    if args.spec_accept:
        run_spec_accept_timing(args)
        return
    if args.aux_kernels:
        run_aux_kernels(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
