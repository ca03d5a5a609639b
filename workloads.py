"""Seeded synthetic workloads for paged decode attention.

This module only *creates inputs*: random query/key/value values rounded to
bf16, random context lengths, a shuffled pool of physical KV blocks and the
per-sequence block tables that point into it.  It contains none of the
attention arithmetic, so both the CPU oracle (``oracle/``) and the CUDA path
(``paged_kv_cache_221_gb300``) can consume the same inputs without sharing any
code of the method itself.

Paging model (the KV cache is cut into fixed-size physical blocks of
``block_size`` tokens, placed anywhere in one shared pool; a block table maps a
sequence's logical blocks to physical ones): "PagedAttention, décodage
spéculatif, MoE et Blackwell", §1 (pagination de type système d'exploitation);
"LLM inference optimization: KV cache", §4.1.

Conventions used by every workload:

* ``k_cache`` / ``v_cache``: uint16 bf16 bit patterns, shape
  ``[num_blocks, num_kv_heads, block_size, head_dim]``.
* ``block_tables``: int32 ``[num_seqs, max_blocks_per_seq]``; unused entries
  are -1.
* ``context_lens``: int32 ``[num_seqs]``; the length *includes* the
  ``num_query_tokens`` newest tokens (the new decode token, or the speculative
  drafts).
* ``q``: uint16 bf16 ``[num_seqs, num_query_tokens, num_q_heads, head_dim]``.
* The K/V of the newest ``num_query_tokens`` positions of every sequence are
  *not* in the pool: they are ``new_key`` / ``new_value``
  (``[num_seqs * num_query_tokens, num_kv_heads, head_dim]``) with their
  destination ``slot_mapping`` (int64, ``slot = physical_block * block_size +
  offset``).  Their pool slots, every slot past the context end and every
  unused block hold the bf16 NaN pattern ``NAN_BITS``, so a kernel that reads
  a slot it should not (or attends before writing the new tokens) produces
  NaN.
* Shared-prefix workloads put the same physical prompt blocks at the front of
  every member's block table (copy-on-write sharing, "PagedAttention, ..."
  §1, "Partage de mémoire").
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os
from typing import Optional

import numpy as np

NAN_BITS = np.uint16(0x7FC0)   # a quiet-NaN bf16 pattern used as the "never read" sentinel
NAN_E4M3 = np.uint8(0x7F)       # the E4M3 NaN code, the same sentinel for FP8 pages
BLOCK_SIZE = 16                 # tokens per physical block (the pages' example value)

# Chunk size for random generation (elements): each chunk has its own seeded generator
# and temporaries of a few hundred MB; chunks run on a thread pool.
_CHUNK = 1 << 25


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return uint16 bits.

    Inputs are finite (normal draws), so no NaN/Inf special-casing is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _chunked(rng: np.random.Generator, n: int, dtype, fill) -> np.ndarray:
    """n values made chunk by chunk by ``fill(chunk_rng, count)``.  Each chunk has its
    own generator seeded from ``rng`` (so the result depends only on ``rng``'s state,
    not on scheduling), and chunks are filled on a thread pool (NumPy's generators
    and ufuncs release the GIL on large arrays)."""
    out = np.empty(n, dtype=dtype)
    starts = list(range(0, n, _CHUNK))
    seeds = rng.integers(0, 1 << 63, size=len(starts), dtype=np.int64)

    def one(i):
        s = starts[i]
        e = min(n, s + _CHUNK)
        out[s:e] = fill(np.random.default_rng(int(seeds[i])), e - s)

    if len(starts) <= 1:
        for i in range(len(starts)):
            one(i)
    else:
        with concurrent.futures.ThreadPoolExecutor(min(len(starts), os.cpu_count() or 4)) as ex:
            list(ex.map(one, range(len(starts))))
    return out


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) float32 draws rounded to bf16, generated in chunks; returns uint16 bits."""
    n = int(np.prod(shape))
    return _chunked(rng, n, np.uint16, lambda g, c: f32_to_bf16_bits(
        g.standard_normal(c, dtype=np.float32))).reshape(shape)


@dataclasses.dataclass
class Workload:
    name: str
    num_seqs: int
    num_query_tokens: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray        # int32 [B]
    block_tables: np.ndarray        # int32 [B, MBS]
    q: np.ndarray                   # uint16 [B, T, Hq, D]
    k_cache: np.ndarray             # uint16 [NB, Hkv, BS, D] (newest tokens not yet written)
    v_cache: np.ndarray             # uint16 [NB, Hkv, BS, D]
    new_key: np.ndarray             # uint16 [N, Hkv, D]
    new_value: np.ndarray           # uint16 [N, Hkv, D]
    slot_mapping: np.ndarray        # int64 [N]
    scale: float
    partition_size: int = 0         # tokens per split-KV partition (0 = library default)
    seq_group: Optional[np.ndarray] = None          # int32 [B], -1 = not in a group
    group_prefix_blocks: Optional[np.ndarray] = None  # int32 [num_groups]
    # FP8 (E4M3) pages (``fp8_variant``): codes instead of bf16 pools, plus per-kv-head scales
    kv_dtype: str = "bf16"
    k_codes: Optional[np.ndarray] = None            # uint8 [NB, Hkv, BS, D]
    v_codes: Optional[np.ndarray] = None            # uint8 [NB, Hkv, D, BS] (page transposed)
    k_scale: Optional[np.ndarray] = None            # float32 [Hkv]
    v_scale: Optional[np.ndarray] = None            # float32 [Hkv]

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max())

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_groups(self) -> int:
        return 0 if self.group_prefix_blocks is None else int(len(self.group_prefix_blocks))

    @property
    def max_group_size(self) -> int:
        if self.seq_group is None:
            return 0
        g = self.seq_group[self.seq_group >= 0]
        return int(np.bincount(g).max()) if g.size else 0

    @property
    def max_prefix_blocks(self) -> int:
        return 0 if self.group_prefix_blocks is None else int(self.group_prefix_blocks.max())

    def unique_pages(self) -> int:
        """Distinct (physical block, kv head) pages the attention must read once.

        Every block covering a token < context_len is counted whole (a page is
        read whole, tail slots included); a block shared by several tables is
        counted once.
        """
        used = set()
        for b in range(self.num_seqs):
            nblk = -(-int(self.context_lens[b]) // self.block_size)
            used.update(int(x) for x in self.block_tables[b, :nblk])
        return len(used) * self.num_kv_heads

    def logical_pages(self) -> int:
        """(block, kv head) pages summed over sequences (shared blocks counted per sequence)."""
        nblk = -(-self.context_lens.astype(np.int64) // self.block_size)
        return int(nblk.sum()) * self.num_kv_heads

    def page_bytes(self) -> int:
        """Bytes of one K page plus one V page (2 bytes per value for bf16, 1 for fp8)."""
        return 2 * self.block_size * self.head_dim * (1 if self.kv_dtype == "fp8" else 2)

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes of one attention pass: unique pages x (K + V) page bytes."""
        return self.unique_pages() * self.page_bytes()


def _assign_tables(rng, nblk_per_seq, num_blocks, shared=None):
    """Random physical placement.  ``shared`` = list of (member seq ids, n prefix blocks)."""
    perm = rng.permutation(num_blocks).astype(np.int32)
    B = len(nblk_per_seq)
    mbs = int(max(nblk_per_seq))
    tables = np.full((B, mbs), -1, dtype=np.int32)
    cursor = 0
    prefix_of = {}
    for members, npre in (shared or []):
        ids = perm[cursor:cursor + npre]
        cursor += npre
        for b in members:
            prefix_of[b] = ids
    for b in range(B):
        start = 0
        if b in prefix_of:
            ids = prefix_of[b]
            tables[b, :len(ids)] = ids
            start = len(ids)
        n = int(nblk_per_seq[b]) - start
        tables[b, start:start + n] = perm[cursor:cursor + n]
        cursor += n
    assert cursor <= num_blocks
    return tables, perm[:cursor]


def _fill_pool(rng, num_blocks, used_ids, Hkv, BS, D):
    """Pool filled with NaN sentinels; used blocks get N(0,1) bf16 values."""
    k = np.full((num_blocks, Hkv, BS, D), NAN_BITS, dtype=np.uint16)
    v = np.full((num_blocks, Hkv, BS, D), NAN_BITS, dtype=np.uint16)
    used_ids = np.sort(np.asarray(used_ids))
    k[used_ids] = normal_bf16(rng, (len(used_ids), Hkv, BS, D))
    v[used_ids] = normal_bf16(rng, (len(used_ids), Hkv, BS, D))
    return k, v


def build(name, context_lens, *, num_q_heads, num_kv_heads, head_dim, num_query_tokens=1,
          block_size=BLOCK_SIZE, seed=0, pool_factor=1.25, num_blocks=None, shared=None,
          tables=None, partition_size=0) -> Workload:
    """Assemble a workload.

    ``shared``: list of (member seq ids, number of prefix blocks) groups whose
    members point at the same physical prompt blocks.  ``tables``: explicit
    block tables (bypasses random placement; ``num_blocks`` must be given).
    """
    rng = np.random.default_rng(seed)
    L = np.asarray(context_lens, dtype=np.int32)
    B = len(L)
    T = num_query_tokens
    assert (L >= T).all(), "every context must hold its query tokens"
    nblk = -(-L.astype(np.int64) // block_size)
    if tables is None:
        if shared:
            shared_blocks = sum(n for _, n in shared)
            private = int(nblk.sum()) - sum(n * len(m) for m, n in shared)
            need = shared_blocks + private
        else:
            need = int(nblk.sum())
        if num_blocks is None:
            num_blocks = int(math.ceil(pool_factor * need))
        tables, used = _assign_tables(rng, nblk, num_blocks, shared)
    else:
        tables = np.asarray(tables, dtype=np.int32)
        assert num_blocks is not None
        used = np.unique(np.concatenate([tables[b, :nblk[b]] for b in range(B)]))
    k_cache, v_cache = _fill_pool(rng, num_blocks, used, num_kv_heads, block_size, head_dim)

    # Tail slots of each sequence's last block are never valid context.
    for b in range(B):
        last = int(tables[b, nblk[b] - 1])
        off = int(L[b]) - (int(nblk[b]) - 1) * block_size
        if off < block_size:
            k_cache[last, :, off:, :] = NAN_BITS
            v_cache[last, :, off:, :] = NAN_BITS

    # The newest T tokens of each sequence arrive as new K/V plus a slot each.
    slots = np.empty(B * T, dtype=np.int64)
    for b in range(B):
        for t in range(T):
            pos = int(L[b]) - T + t
            slots[b * T + t] = int(tables[b, pos // block_size]) * block_size + pos % block_size
    blk, off = slots // block_size, slots % block_size
    new_key = np.ascontiguousarray(k_cache[blk, :, off, :])
    new_value = np.ascontiguousarray(v_cache[blk, :, off, :])
    k_cache[blk, :, off, :] = NAN_BITS
    v_cache[blk, :, off, :] = NAN_BITS

    q = normal_bf16(rng, (B, T, num_q_heads, head_dim))
    seq_group = group_prefix = None
    if shared:
        seq_group = np.full(B, -1, dtype=np.int32)
        group_prefix = np.zeros(len(shared), dtype=np.int32)
        for gi, (members, npre) in enumerate(shared):
            seq_group[list(members)] = gi
            group_prefix[gi] = npre
    return Workload(name=name, num_seqs=B, num_query_tokens=T, num_q_heads=num_q_heads,
                    num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                    num_blocks=int(num_blocks), context_lens=L, block_tables=tables, q=q,
                    k_cache=k_cache, v_cache=v_cache, new_key=new_key, new_value=new_value,
                    slot_mapping=slots, scale=1.0 / math.sqrt(head_dim),
                    partition_size=partition_size, seq_group=seq_group,
                    group_prefix_blocks=group_prefix)


def random_e4m3_codes(rng: np.random.Generator, shape, exp_lo=9, exp_hi=13) -> np.ndarray:
    """Random E4M3 bit patterns: uniform sign bit, exponent field uniform in
    [exp_lo, exp_hi], uniform 3-bit mantissa (no NaN code for exp_hi <= 14)."""
    n = int(np.prod(shape))

    def fill(g, c):
        sign = g.integers(0, 2, c, dtype=np.uint8)
        ex = g.integers(exp_lo, exp_hi + 1, c, dtype=np.uint8)
        man = g.integers(0, 8, c, dtype=np.uint8)
        return (sign << np.uint8(7)) | (ex << np.uint8(3)) | man

    return _chunked(rng, n, np.uint8, fill).reshape(shape)


def fp8_variant(w: Workload, seed: int = 0, scale_lo=1.0 / 96, scale_hi=1.0 / 48) -> Workload:
    """The same workload with FP8 (E4M3) pages.

    Same lengths, tables, queries, new tokens (bf16, still to be quantised by
    reshape_and_cache) and slots.  Context slots hold random codes (exponent
    field 9..13: magnitudes 4 .. 120 before scaling); every slot that holds
    the bf16 sentinel in ``w`` (unused blocks, tails, the new tokens' slots)
    holds the E4M3 NaN code.  Scales are one float32 per kv head, uniform in
    [scale_lo, scale_hi].  V pages are stored transposed (``[D, BS]``).
    """
    rng = np.random.default_rng(seed + 5000)
    NB, Hkv, BS, D = w.k_cache.shape
    sentinel = w.k_cache[:, 0, :, 0] == NAN_BITS                   # [NB, BS]
    k_codes = random_e4m3_codes(rng, (NB, Hkv, BS, D))
    v_codes = random_e4m3_codes(rng, (NB, Hkv, D, BS))
    blk, tok = np.nonzero(sentinel)
    k_codes[blk, :, tok, :] = NAN_E4M3
    v_codes[blk, :, :, tok] = NAN_E4M3
    k_scale = rng.uniform(scale_lo, scale_hi, Hkv).astype(np.float32)
    v_scale = rng.uniform(scale_lo, scale_hi, Hkv).astype(np.float32)
    return dataclasses.replace(w, name=w.name + "_fp8", kv_dtype="fp8", k_cache=None,
                               v_cache=None, k_codes=k_codes, v_codes=v_codes,
                               k_scale=k_scale, v_scale=v_scale)


# --------------------------------------------------------------------------
# The five named workloads.  Seeds: tiny=0, 8B=1, 70B=2, verify=3, prefix=4.
# ``scale_down`` shrinks batch/lengths for fast oracle-sized variants with the
# same structure (used by the parity tests); 1 = full size.
# --------------------------------------------------------------------------

def tiny(seed=0) -> Workload:
    """2 seqs (ctx 37 and 100), 4 q = 4 kv heads, head_dim 64, 16 physical blocks.

    The block tables are the first 3 and the next 7 ids of a seeded
    permutation of the 16 block ids.
    """
    rng = np.random.default_rng(seed + 1000)
    perm = rng.permutation(16).astype(np.int32)
    tables = np.full((2, 7), -1, dtype=np.int32)
    tables[0, :3] = perm[:3]
    tables[1, :7] = perm[3:10]
    return build("tiny", [37, 100], num_q_heads=4, num_kv_heads=4, head_dim=64, seed=seed,
                 num_blocks=16, tables=tables)


def decode_8b(seed=1, batch=64, lo=512, hi=4096) -> Workload:
    """8B-shape decode: ctx ~ U[lo, hi], 32 q / 8 kv heads, head_dim 128, pool 1.25x."""
    rng = np.random.default_rng(seed + 1000)
    L = rng.integers(lo, hi + 1, size=batch)
    return build("decode_8b", L, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=seed)


def decode_70b(seed=2, batch=256, lo=128, hi=8192) -> Workload:
    """70B-shape decode: ctx log-uniform in [lo, hi], 64 q / 8 kv heads, head_dim 128."""
    rng = np.random.default_rng(seed + 1000)
    L = np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi), size=batch))).astype(np.int64)
    L = np.clip(L, lo, hi)
    return build("decode_70b", L, num_q_heads=64, num_kv_heads=8, head_dim=128, seed=seed)


def spec_verify(seed=3, batch=32, lo=2048, hi=16384, drafts=5) -> Workload:
    """Speculative verify: 5 draft query tokens per seq, ctx ~ U[lo, hi], 32 q / 8 kv heads."""
    rng = np.random.default_rng(seed + 1000)
    L = rng.integers(lo, hi + 1, size=batch)
    return build("spec_verify", L, num_q_heads=32, num_kv_heads=8, head_dim=128,
                 num_query_tokens=drafts, seed=seed)


def shared_prefix(seed=4, groups=2, members=8, prompt=2048, total=32768,
                  partition_size=512) -> Workload:
    """Long-context shared prefix: ``groups`` x ``members`` seqs share a ``prompt``-token
    copy-on-write prefix, private suffixes up to ``total`` tokens, split-KV over
    ``partition_size``-token partitions."""
    assert prompt % BLOCK_SIZE == 0
    B = groups * members
    L = np.full(B, total, dtype=np.int64)
    shared = [(list(range(g * members, (g + 1) * members)), prompt // BLOCK_SIZE)
              for g in range(groups)]
    return build("shared_prefix", L, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=seed,
                 shared=shared, partition_size=partition_size)


FULL = {
    "tiny": tiny,
    "decode_8b": decode_8b,
    "decode_70b": decode_70b,
    "spec_verify": spec_verify,
    "shared_prefix": shared_prefix,
}

# Oracle-sized variants with the same structure (a few seconds of fp64 CPU work).
SMALL = {
    "tiny": tiny,
    "decode_8b": lambda seed=1: decode_8b(seed, batch=6, lo=100, hi=1200),
    "decode_70b": lambda seed=2: decode_70b(seed, batch=8, lo=20, hi=1500),
    "spec_verify": lambda seed=3: spec_verify(seed, batch=5, lo=5, hi=1500),
    "shared_prefix": lambda seed=4: shared_prefix(seed, groups=2, members=3, prompt=320,
                                                  total=1400, partition_size=128),
}
