"""Helpers shared by the GPU tests: move a workload to the device, run the
library's hot path on it, and compare against oracle values."""
import numpy as np
import torch

import paged_kv_cache_221_gb300 as pa

MAX_ABS = 1e-2      # bf16 output vs fp64 oracle: max abs error ...
BF16_ULP_REL = 2.0 ** -8   # ... or one bf16 ulp of the oracle value, whichever is larger
MAX_REL_L2 = 2e-3   # bf16 output vs fp64 oracle: relative L2 error


def abs_bound(ref):
    """Per-element bound on |output - oracle|: 1e-2, or one bf16 ulp (at most 2^-8 of
    the value) where the oracle value is above 2.56.  Rounding the exact result to bf16
    alone errs by up to half an ulp, which exceeds 1e-2 once |value| >= 4, so a plain
    1e-2 bound cannot hold there for any bf16 output."""
    return np.maximum(MAX_ABS, BF16_ULP_REL * np.abs(ref))


def to_dev(a, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(device)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Dev:
    """Device copies of a workload's arrays."""

    def __init__(self, w, device="cuda"):
        self.w = w
        self.q = to_dev(w.q, device)
        self.k = to_dev(w.k_cache, device)
        self.v = to_dev(w.v_cache, device)
        self.tables = to_dev(w.block_tables, device)
        self.lens = to_dev(w.context_lens, device)
        self.new_key = to_dev(w.new_key, device)
        self.new_value = to_dev(w.new_value, device)
        self.slots = to_dev(w.slot_mapping, device)
        self.seq_group = None if w.seq_group is None else to_dev(w.seq_group, device)
        self.group_prefix = None if w.group_prefix_blocks is None else \
            to_dev(w.group_prefix_blocks, device)

    def reshape(self):
        pa.reshape_and_cache(self.new_key, self.new_value, self.k, self.v, self.slots)

    def attend_append(self, partition_size=None, workspace=None, out=None):
        """reshape_and_cache fused into the attention launch (pa_decode_append)."""
        w = self.w
        ps = w.partition_size if partition_size is None else partition_size
        return pa.verify(self.q, self.k, self.v, self.tables, self.lens, w.max_context_len,
                         w.scale, ps, workspace, out, self.new_key, self.new_value)

    def attend(self, partition_size=None, shared=True, workspace=None, out=None):
        w = self.w
        ps = w.partition_size if partition_size is None else partition_size
        if shared and w.seq_group is not None:
            return pa.decode_shared_prefix(self.q, self.k, self.v, self.tables, self.lens,
                                           self.seq_group, self.group_prefix, w.max_group_size,
                                           w.max_prefix_blocks, w.max_context_len, w.scale, ps,
                                           workspace, out)
        return pa.verify(self.q, self.k, self.v, self.tables, self.lens, w.max_context_len,
                         w.scale, ps, workspace, out)


def errors(out: torch.Tensor, ref: np.ndarray, seqs=None):
    g = out.float().cpu().double().numpy()
    if seqs is not None:
        g, ref = g[seqs], ref[seqs]
    d = g - ref
    return float(np.abs(d).max()), float(np.linalg.norm(d) / np.linalg.norm(ref)), g


def assert_close(out, ref, seqs=None, what=""):
    mx, rel, g = errors(out, ref, seqs)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    r = ref if seqs is None else ref[seqs]
    over = np.abs(g - r) - abs_bound(r)
    assert over.max() <= 0 and rel <= MAX_REL_L2, \
        f"{what}: max abs {mx:.3e} (bound exceeded by {max(over.max(), 0):.3e}), rel L2 {rel:.3e}"
    return mx, rel

