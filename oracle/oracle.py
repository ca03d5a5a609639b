"""fp64 CPU oracle for the paged decode-attention hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA path
(no kernels, headers, helpers or tables); the one thing both sides share is the
seeded input generator ``workloads.py``, which holds no attention arithmetic.

What it computes is the plain definition of the result, written out slowly:

* ``reshape_and_cache``: each new token's key and value vectors are stored in
  the cache slot the slot mapping names ("LLM inference optimization: KV
  cache", §3.1 and its diagram: the K and V of the new token are saved into the
  KV cache; "PagedAttention, décodage spéculatif, MoE et Blackwell", §1: the
  cache is cut into fixed-size blocks placed anywhere in memory).
* ``gather_context``: the block table maps logical block ``j // block_size`` of
  a sequence to a physical block ("PagedAttention, ..." §1, pagination de type
  système d'exploitation; "LLM inference optimization: KV cache", §4.1), so the
  contiguous K (or V) of a sequence is obtained by reading, for each position
  ``j``, slot ``j % block_size`` of that physical block.
* ``paged_attention``: the query of the new token attends over the cached K and
  V ("LLM inference optimization: KV cache", §3.1), with a softmax over the
  visible positions kept in full precision ("ranksignal" post, the note that
  almost every scheme keeps the softmax in its original precision).  With
  ``num_query_tokens = T > 1`` the T draft tokens are verified in one parallel
  pass ("PagedAttention, ..." §1, vérification parallèle; "LLM inference
  optimization: KV cache", §5.2): draft ``t`` occupies position ``L - T + t``
  and sees positions ``j <= L - T + t`` (causal mask among the drafts).

Readings where the pages are silent (each listed in the design notes):
pool layout ``[num_blocks, num_kv_heads, block_size, head_dim]``; query head
``h`` reads kv head ``h // (Hq / Hkv)``; ``context_len`` counts the new token
(or the drafts); scale is a parameter (1/sqrt(head_dim) in every workload).

Inputs are bf16 bit patterns (uint16 arrays); every value is widened to fp64
before any arithmetic.  Results are fp64 and are not rounded.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the upper half of an IEEE binary32: shift into place, view, widen."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, block_size):
    """Write new K/V rows into their cache slots; returns new (k_cache, v_cache) copies.

    key, value: uint16 [N, Hkv, D]; caches: uint16 [NB, Hkv, BS, D];
    slot_mapping: int [N], slot = physical_block * block_size + offset.
    A negative slot marks a padding token and is skipped.  Two tokens naming
    the same slot have no defined result, so they are rejected.  Bits are copied
    unchanged.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    seen = set()
    num_blocks = k_out.shape[0]
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        if slot in seen:
            raise ValueError(f"slot {slot} written twice")
        seen.add(slot)
        block, offset = divmod(slot, block_size)
        if block >= num_blocks:
            raise IndexError(f"slot {slot} outside the pool")
        k_out[block, :, offset, :] = key[i]
        v_out[block, :, offset, :] = value[i]
    return k_out, v_out


def gather_context(cache, block_table_row, context_len, kv_head, block_size):
    """Contiguous fp64 [context_len, D] rows of one kv head of one sequence."""
    positions = np.arange(context_len)
    physical = np.asarray(block_table_row)[positions // block_size]
    if (physical < 0).any() or (physical >= cache.shape[0]).any():
        raise IndexError("block table entry outside the pool")
    return bf16_bits_to_f64(cache[physical, kv_head, positions % block_size, :])


def softmax(scores: np.ndarray) -> np.ndarray:
    """Softmax of a 1-D fp64 vector, with the maximum subtracted first."""
    z = scores - scores.max()
    e = np.exp(z)
    return e / e.sum()


def kv_head_of(q_head: int, num_q_heads: int, num_kv_heads: int) -> int:
    """Grouped-query mapping: consecutive groups of Hq/Hkv query heads share a kv head."""
    return q_head // (num_q_heads // num_kv_heads)


def visible_length(context_len: int, num_query_tokens: int, t: int) -> int:
    """Number of positions query token ``t`` sees: positions 0 .. L - T + t."""
    return context_len - num_query_tokens + t + 1


def scores(Kc: np.ndarray, q: np.ndarray, scale: float) -> np.ndarray:
    """Scaled dot products of one query vector with every cached key row."""
    return scale * (Kc @ q)


def attention_weights(q_bits, k_cache, block_tables, context_lens, scale, num_kv_heads,
                      block_size, b, t, h):
    """Softmax weights of (sequence b, query token t, query head h) over its visible positions."""
    B, T, Hq, D = q_bits.shape
    g = kv_head_of(h, Hq, num_kv_heads)
    L = int(context_lens[b])
    n = visible_length(L, T, t)
    Kc = gather_context(k_cache, block_tables[b], L, g, block_size)[:n]
    q = bf16_bits_to_f64(q_bits[b, t, h])
    return softmax(scores(Kc, q, scale))


def paged_attention(q_bits, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                    block_size, seqs=None):
    """fp64 output [B, T, Hq, D] (rows of sequences not in ``seqs`` are left as NaN).

    For each sequence the K and V of each kv head are first gathered into a
    contiguous array through the block table, then every query row attends
    over its visible prefix of that array.
    """
    B, T, Hq, D = q_bits.shape
    out = np.full((B, T, Hq, D), np.nan)
    for b in (range(B) if seqs is None else seqs):
        L = int(context_lens[b])
        gathered = {}
        for h in range(Hq):
            g = kv_head_of(h, Hq, num_kv_heads)
            if g not in gathered:
                gathered[g] = (gather_context(k_cache, block_tables[b], L, g, block_size),
                               gather_context(v_cache, block_tables[b], L, g, block_size))
            Kc, Vc = gathered[g]
            for t in range(T):
                n = visible_length(L, T, t)
                q = bf16_bits_to_f64(q_bits[b, t, h])
                p = softmax(scores(Kc[:n], q, scale))
                out[b, t, h] = p @ Vc[:n]
    return out


def run_workload(w, seqs=None):
    """reshape_and_cache of the workload's new tokens, then paged attention (fp64)."""
    k, v = reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping,
                             w.block_size)
    return paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale, w.num_kv_heads,
                           w.block_size, seqs=seqs), k, v
