"""fp64 oracle of sliding-window paged attention.

TEST INFRASTRUCTURE ONLY (same rules as ``oracle.py``).

Sliding-window attention changes which cached positions a query attends to:
each query looks only at the most recent positions ("ranksignal" post, the
attention kernels section: sliding-window attention looks only at the latest
tokens; the window size is lost in extraction, so it is a parameter here).
Reading: query token t of a sequence of length L sits at position
pos = L - T + t and attends to positions j with pos - W < j <= pos (the last W
positions, itself included), W >= 1.  Everything else (paging, GQA, scale,
softmax in full precision) is as in ``oracle.py``, whose helpers are used; for
FP8 pages the gathers of ``fp8.py`` are used.
"""
from __future__ import annotations

import numpy as np

from . import fp8 as F
from . import oracle as O


def visible_range(context_len: int, num_query_tokens: int, t: int, window: int):
    """[first, last] positions query token t sees with a window of `window` positions."""
    last = context_len - num_query_tokens + t
    first = max(0, last - window + 1)
    return first, last


def paged_attention(q_bits, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                    block_size, window, seqs=None, k_scale=None, v_scale=None):
    """fp64 output [B, T, Hq, D]; bf16 pools, or FP8 code pools when k_scale is given."""
    B, T, Hq, D = q_bits.shape
    out = np.full((B, T, Hq, D), np.nan)
    for b in (range(B) if seqs is None else seqs):
        L = int(context_lens[b])
        gathered = {}
        for h in range(Hq):
            g = O.kv_head_of(h, Hq, num_kv_heads)
            if g not in gathered:
                if k_scale is None:
                    gathered[g] = (O.gather_context(k_cache, block_tables[b], L, g, block_size),
                                   O.gather_context(v_cache, block_tables[b], L, g, block_size))
                else:
                    gathered[g] = (F.gather_k(k_cache, block_tables[b], L, g, k_scale, block_size),
                                   F.gather_v(v_cache, block_tables[b], L, g, v_scale, block_size))
            Kc, Vc = gathered[g]
            for t in range(T):
                first, last = visible_range(L, T, t, window)
                q = O.bf16_bits_to_f64(q_bits[b, t, h])
                p = O.softmax(O.scores(Kc[first:last + 1], q, scale))
                out[b, t, h] = p @ Vc[first:last + 1]
    return out


def run_workload(w, window, seqs=None):
    """reshape_and_cache of the new tokens, then sliding-window attention (fp64)."""
    if w.kv_dtype == "fp8":
        k, v = F.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                                   w.k_scale, w.v_scale, w.block_size)
        return paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                               w.num_kv_heads, w.block_size, window, seqs, w.k_scale,
                               w.v_scale), k, v
    k, v = O.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping,
                               w.block_size)
    return paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale, w.num_kv_heads,
                           w.block_size, window, seqs), k, v
