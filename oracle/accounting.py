"""Memory accounting the pages state in words, written out as functions.

TEST INFRASTRUCTURE ONLY (see ``oracle.py``).  These pin the benchmark's byte
counting to the pages' own formula and worked figures.

* ``kv_cache_bytes``: the KV-cache size formula, 2 (K and V) x batch x sequence
  length x layers x heads x head dimension x bytes per value ("LLM inference
  optimization: KV cache", §3.2).
* ``reservation_unused_fraction``: share of a contiguous max-length reservation
  left empty ("PagedAttention, décodage spéculatif, MoE et Blackwell", §1, the
  fragmentation problem: 200 tokens used of a 32,768-token reservation leaves
  more than 99 % unused).
* ``paged_unused_fraction``: share of allocated block slots left empty when a
  sequence only gets the blocks it needs (at most one partly filled block;
  "LLM inference optimization: KV cache", §4.2: waste below a few percent).
* ``bandwidth_bound_seconds``: time to stream a number of bytes at a given
  bandwidth ("LLM inference optimization: KV cache", §2.3, 140 GB at 2 TB/s
  takes 0.07 s, about 14 tokens per second).
"""
from __future__ import annotations

import math


def kv_cache_bytes(batch, seq_len, layers, heads, head_dim, bytes_per_value):
    return 2 * batch * seq_len * layers * heads * head_dim * bytes_per_value


def reservation_unused_fraction(used_tokens, reserved_tokens):
    return (reserved_tokens - used_tokens) / reserved_tokens


def paged_unused_fraction(used_tokens, block_size):
    allocated = math.ceil(used_tokens / block_size) * block_size
    return (allocated - used_tokens) / allocated


def bandwidth_bound_seconds(num_bytes, bytes_per_second):
    return num_bytes / bytes_per_second
