"""Scalar brute-force paged attention, for tiny inputs only.

TEST INFRASTRUCTURE ONLY (see ``oracle.py``).  It shares nothing with
``oracle.py`` either: pure Python loops over positions and dimensions, one
``math.exp`` per weight, the physical slot of every position looked up one at a
time, and no NumPy arithmetic.  It exists to pin ``oracle.paged_attention``
against an independent restatement of the same definition ("LLM inference
optimization: KV cache", §3.1 attention over cached K/V; §4.1 block table;
"PagedAttention, décodage spéculatif, MoE et Blackwell", §1 parallel
verification of K draft tokens).
"""
from __future__ import annotations

import math
import struct


def _bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def attend_one(q_bits, k_cache, v_cache, table_row, context_len, num_query_tokens, t, h,
               num_kv_heads, scale, block_size):
    """Output vector (list of floats) of one query row, by direct summation."""
    Hq = len(q_bits)
    group = Hq // num_kv_heads
    kvh = h // group
    D = len(q_bits[h])
    q = [_bf16(q_bits[h][d]) for d in range(D)]
    last = context_len - num_query_tokens + t          # last visible position
    scores = []
    for j in range(last + 1):
        blk = int(table_row[j // block_size])
        off = j % block_size
        acc = 0.0
        for d in range(D):
            acc += q[d] * _bf16(k_cache[blk][kvh][off][d])
        scores.append(scale * acc)
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    total = sum(w)
    out = [0.0] * D
    for j in range(last + 1):
        blk = int(table_row[j // block_size])
        off = j % block_size
        p = w[j] / total
        for d in range(D):
            out[d] += p * _bf16(v_cache[blk][kvh][off][d])
    return out


def paged_attention(q_bits, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                    block_size):
    """Nested lists [B][T][Hq][D] of floats."""
    qb = q_bits.tolist()
    kc = k_cache.tolist()
    vc = v_cache.tolist()
    tables = block_tables.tolist()
    B = len(qb)
    T = len(qb[0])
    Hq = len(qb[0][0])
    return [[[attend_one(qb[b][t], kc, vc, tables[b], int(context_lens[b]), T, t, h,
                         num_kv_heads, scale, block_size)
              for h in range(Hq)] for t in range(T)] for b in range(B)]
