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

Prints one JSON line (rank 0).  ``value`` is KV-read GB/s of the whole step
(algorithmic bytes: every (block, kv head) page a step must read, once, x the
K and V page bytes) over the device time of K steps, summed over ranks; each
rank runs its own replica (the path shards by sequence with no exchange).
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
KERNEL_SOURCES = ["pa_attn.cuh", "pa_ptx.cuh"]   # the attention kernel template and its PTX
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
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
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


def kernel_source_hash():
    """Hash of what the attention kernel is compiled from: its template, its PTX helpers,
    and the constants and parameter struct it reads (launcher declarations excluded)."""
    csrc = os.path.join(ROOT, "paged_kv_cache_221_gb300", "csrc")
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(f.read())
    with open(os.path.join(csrc, KERNEL_PARAMS), "rb") as f:
        text = f.read()
    end = text.find(b"};", text.find(b"struct AttnParams"))
    h.update(text[:end + 2])
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch of the attention kernel from a committed ncu summary, if the
    kernel sources have not changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_src_sha") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


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
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
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
    # Pin BLAS to one thread before NumPy loads.
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    sys.path.insert(0, ROOT)
    from oracle import cpu_baseline as C

    w, k, v = C.prepare(args.workload + ("_fp8" if args.kv_dtype == "fp8" else ""))
    # per-step sample: enough whole sequences for ~0.5 s, fewer when many steps are asked
    steps = args.steps if args.steps > 0 else 10
    per_seq = max(C.run_seqs(w, k, v, [0]), 1e-4)
    budget = 150.0 / max(1, steps + args.warmup)
    n = max(1, min(w.num_seqs, int(min(0.5, budget) / per_seq)))
    ring = list(range(w.num_seqs)) * 2

    def sample(i):
        s0 = (i * n) % w.num_seqs
        return ring[s0:s0 + n]

    for i in range(args.warmup):
        C.run_seqs(w, k, v, sample(i))
    nbytes = 0
    nseq = 0
    dt = 0.0
    for i in range(steps):
        sm = sample(i)
        dt += C.run_seqs(w, k, v, sm)
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
            "cpu_baseline": {"value": round(gbps, 4), "unit": "GB/s", "cores": C.threads_used(),
                             "kind": "oracle",
                             "sample": f"{n} whole sequence(s) of the {w.name} batch per step "
                                       f"(fp64 paged attention, reshape untimed)"},
            "e2e": {"value": round(gbps, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GB300 arm

def run_gb300(args):
    import numpy as np
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

    w = replica_workload(args.workload, rank)
    fp8 = args.kv_dtype == "fp8"
    if fp8:
        import workloads as W
        w = W.fp8_variant(w, seed=rank)
    if args.window > 0:
        w.seq_group = None                  # the window runs the per-sequence path
        w.group_prefix_blocks = None
    ps = w.partition_size if args.partition_size < 0 else args.partition_size

    def td(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.to(dev)

    q = td(w.q)
    k, v = (td(w.k_codes), td(w.v_codes)) if fp8 else (td(w.k_cache), td(w.v_cache))
    ks, vs = (td(w.k_scale), td(w.v_scale)) if fp8 else (None, None)
    tables, lens = td(w.block_tables), td(w.context_lens)
    nk, nv, slots = td(w.new_key), td(w.new_value), td(w.slot_mapping)
    grouped = w.seq_group is not None
    sg = td(w.seq_group) if grouped else None
    gp = td(w.group_prefix_blocks) if grouped else None
    T = w.num_query_tokens
    need = pa.workspace_size(w.num_seqs, w.num_q_heads, T, w.max_context_len, w.head_dim, 16,
                             ps, w.max_prefix_blocks if grouped else 0)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    kv_bytes = w.kv_bytes() if args.window <= 0 else window_kv_bytes(w, args.window)

    # Per-sequence workloads: one fused call (reshape_and_cache inside the attention
    # launch).  Shared-prefix workload: reshape_and_cache, then the shared-prefix call.
    def reshape():
        if grouped and fp8:
            pa.reshape_and_cache_fp8(nk, nv, k, v, slots, ks, vs)
        elif grouped:
            pa.reshape_and_cache(nk, nv, k, v, slots)

    def attend():
        if args.window > 0:
            pa.attention(q, k, v, tables, lens, w.max_context_len, w.scale, ps, ws, out, nk, nv,
                         window_size=args.window, k_scale=ks, v_scale=vs)
        elif grouped:
            pa.decode_shared_prefix(q, k, v, tables, lens, sg, gp, w.max_group_size,
                                    w.max_prefix_blocks, w.max_context_len, w.scale, ps, ws, out,
                                    k_scale=ks, v_scale=vs)
        elif fp8:
            pa.verify_fp8(q, k, v, ks, vs, tables, lens, w.max_context_len, w.scale, ps, ws, out,
                          nk, nv)
        else:
            pa.verify(q, k, v, tables, lens, w.max_context_len, w.scale, ps, ws, out,
                      nk, nv)

    # our kernels per step: attention (+ split-KV merge) (+ reshape + shared-prefix kernel)
    launches_per_step = 1 + (1 if need > 0 else 0) + (2 if grouped else 0)
    two_graphs = grouped

    stream = torch.cuda.current_stream(dev)
    # warm-up outside capture (sets kernel attributes), then capture one graph per phase
    for _ in range(max(3, args.warmup)):
        reshape()
        attend()
    torch.cuda.synchronize(dev)
    assert pa.get_device_error(dev) == 0
    g_reshape = torch.cuda.CUDAGraph() if two_graphs else None
    g_attend = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        if two_graphs:
            with torch.cuda.graph(g_reshape, stream=side):
                reshape()
        with torch.cuda.graph(g_attend, stream=side):
            attend()
    stream.wait_stream(side)

    class _NoGraph:
        def replay(self):
            pass

    if g_reshape is None:
        g_reshape = _NoGraph()
    for _ in range(max(3, args.warmup)):
        g_reshape.replay()
        g_attend.replay()
    torch.cuda.synchronize(dev)

    # step count: about 1.5 s of timed work unless given
    steps = args.steps
    if steps <= 0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(20):
            g_reshape.replay()
            g_attend.replay()
        e1.record(stream)
        e1.synchronize()
        per = e0.elapsed_time(e1) / 20
        steps = int(max(50, min(20000, 1500.0 / max(per, 1e-3))))

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_start, a_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # K steps back to back, as a serving loop submits them (no event between steps)
    start.record(stream)
    for i in range(steps):
        g_reshape.replay()
        g_attend.replay()
    stop.record(stream)
    if two_graphs:
        # the attention phase alone (the reshape phase is idempotent), same step count
        a_start.record(stream)
        for i in range(steps):
            g_attend.replay()
        a_stop.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    # keep sampling under the same load until there are enough samples
    t_end = time.time() + 0.6
    while time.time() < t_end:
        for _ in range(50):
            g_reshape.replay()
            g_attend.replay()
        torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    assert pa.get_device_error(dev) == 0, "device error during the timed region"

    ms_total = max_over_ranks(start.elapsed_time(stop), world, dev)
    ms_step = ms_total / steps
    # average duration of the attention call: the whole step for per-sequence workloads
    attn_avg = (a_start.elapsed_time(a_stop) / steps) if two_graphs else \
        start.elapsed_time(stop) / steps
    total_bytes = kv_bytes * world
    value = whole_job_gbps(kv_bytes, world, steps, ms_total)

    # end to end through the public API: pinned host inputs in, output back, every step
    e2e = None
    if not args.no_e2e:
        h = {n: torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for n, a in
             (("q", w.q.view(np.int16)), ("nk", w.new_key.view(np.int16)),
              ("nv", w.new_value.view(np.int16)), ("slots", w.slot_mapping),
              ("tables", w.block_tables), ("lens", w.context_lens))}
        d_in = {"q": q.view(torch.int16), "nk": nk.view(torch.int16), "nv": nv.view(torch.int16),
                "slots": slots, "tables": tables, "lens": lens}
        h_out = torch.empty(out.shape, dtype=torch.int16).pin_memory()
        bi = sum(t.numel() * t.element_size() for t in h.values())
        bo = h_out.numel() * h_out.element_size()
        e2e_steps = max(10, min(steps, 1000))
        for _ in range(3):
            for n_ in h:
                d_in[n_].copy_(h[n_], non_blocking=True)
            reshape()
            attend()
            h_out.copy_(out.view(torch.int16), non_blocking=True)
        torch.cuda.synchronize(dev)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(e2e_steps):
            for n_ in h:
                d_in[n_].copy_(h[n_], non_blocking=True)
            reshape()
            attend()
            h_out.copy_(out.view(torch.int16), non_blocking=True)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(s0.elapsed_time(s1) / e2e_steps, world, dev)
        e2e_binding = {"value": round(total_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                       "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                       "path": "pinned host inputs -> H2D -> the step's library calls (Python "
                               "binding, no graph) -> D2H of the bf16 output"}
        e2e = e2e_binding
        if not grouped:
            # The serving path: the graph runner (one captured graph per batch class) with
            # the same pools; per step the inputs go into its static buffers, one replay,
            # the output comes back.
            used = set(int(x) for x in w.block_tables.ravel() if x >= 0)
            pad = next(bb for bb in range(w.num_blocks) if bb not in used)
            rps = ps if ps > 0 else pa.default_partition_size(w.num_seqs, w.num_kv_heads,
                                                              w.max_context_len)
            runner = pa.GraphRunner(k, v, w.num_q_heads, w.max_context_len,
                                    w.max_blocks_per_seq, pad, rps, classes=(w.num_seqs,),
                                    num_query_tokens=T, scale=w.scale, window_size=args.window,
                                    k_scale=ks, v_scale=vs, host_staging=True)
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

            def runner_step():
                runner.step(w.num_seqs)

            for _ in range(3):
                runner_step()
            torch.cuda.synchronize(dev)
            s0.record(stream)
            for _ in range(e2e_steps):
                runner_step()
            s1.record(stream)
            torch.cuda.synchronize(dev)
            r_ms = max_over_ranks(s0.elapsed_time(s1) / e2e_steps, world, dev)
            runner.close()
            e2e = {"value": round(total_bytes / (r_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                   "h2d_bytes_per_step": bir, "d2h_bytes_per_step": bor,
                   "ms_per_step": round(r_ms, 4), "steps": e2e_steps,
                   "path": "pa_runner_step: one graph replay that copies the step's inputs "
                           "from page-locked host buffers, runs the attention step and copies "
                           "the bf16 output back to the host",
                   "binding_path": e2e_binding}

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    achieved = kv_bytes / (attn_avg * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV / f16 MMA / fp32 softmax" if fp8 else "bf16",
        "data": data_desc(w),
        "config": workload_config(w, ps, world, args.window),
        "seq_steps_per_s": round(w.num_seqs * world * steps / (ms_total * 1e-3), 1),
        "kv_bytes_per_step": kv_bytes,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     # the recorded captures are of full-context launches
                     "traffic": recorded_traffic(w.name) if args.window <= 0 else None,
                     "kernel": "attention call (paged_attn_kernel + splitkv_reduce_kernel)",
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "launch_ms_avg": round(attn_avg, 5)},
        "clocks": clocks,
        "gpu_launches": launches_per_step * steps,
        "timing": "CUDA graph of the step replayed K times back to back between two CUDA "
                  "events on the launching stream (shared-prefix: reshape graph + attention "
                  "graph per step, and the attention graph alone K times for the call)",
    }
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload + ("_fp8" if fp8 else ""),
                                            args.cpu_seconds)
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


def main():
    args = parse_args()
    if args.runner_sweep:
        run_runner_sweep(args)
        return
    if args.spec_accept:
        run_spec_accept_timing(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
