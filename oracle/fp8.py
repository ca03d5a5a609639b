"""fp64 CPU oracle for FP8 (E4M3) KV pages.

TEST INFRASTRUCTURE ONLY (same rules as ``oracle.py``: only the tests, the
smoke check and the benchmark's CPU legs may import it; it shares no code with
the CUDA path).

Halving the bytes of every cached value halves what decode has to load, and
8-bit floats are the usual compromise for the KV cache, with the softmax kept
in its original precision ("ranksignal" post, Quantifier : des nombres plus
petits; "PagedAttention, décodage spéculatif, MoE et Blackwell", §3 on FP8).
The scheme on that page is: find the bounds of the tensor, scale into the
format's range, round.  Here the scale is one float per kv head for K and one
for V, chosen by the caller; a value x of kv head h is stored as the E4M3 code
nearest to ``float32(x) / float32(scale[h])`` and read back as
``decode(code) * scale[h]``.

E4M3 (the "fn" variant: no infinities), from the format's definition: sign
bit, 4-bit exponent field ``e`` with bias 7, 3-bit mantissa ``m``;
``e = 0`` encodes the subnormals ``m * 2^-9``; ``e = 15, m = 7`` is NaN; every
other code is ``(1 + m/8) * 2^(e-7)``; the largest finite magnitude is 448.
Encoding rounds to the nearest representable value, ties to the even code
(mantissa LSB 0), saturates finite and infinite magnitudes above 448 to 448
(keeping the sign), maps NaN to 0x7F, and keeps the sign of values that round
to zero.

Storage (the library's documented layout; readings, since the pages give
none): K pages ``k_codes[block, kv_head, token_in_block, dim]`` (token-major,
as in bf16); V pages transposed, ``v_codes[block, kv_head, dim,
token_in_block]``.
"""
from __future__ import annotations

import numpy as np

from . import oracle as O

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code, from the format definition."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# All 256 code values (index = code), built once from e4m3_value.
DECODE_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
# Non-negative finite values in code order 0x00 .. 0x7E (strictly increasing).
_POS_VALUES = DECODE_TABLE[:0x7F]


def decode(codes: np.ndarray) -> np.ndarray:
    """fp64 values of an array of E4M3 codes."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of fp64/fp32 values: nearest, ties to even, saturating."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)            # saturate (inf included)
    hi = np.searchsorted(_POS_VALUES, a, side="left")   # first value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(NAN_CODE), code).astype(np.uint8)


def quantize(bits_bf16: np.ndarray, scale: float) -> np.ndarray:
    """Codes of bf16 values divided by ``scale`` (the division in IEEE float32)."""
    q = O.bf16_bits_to_f64(bits_bf16).astype(np.float32) / np.float32(scale)
    return encode(q.astype(np.float64))


def reshape_and_cache(key, value, k_codes, v_codes, slot_mapping, k_scale, v_scale,
                      block_size):
    """Quantise and store each new token's K/V in its slot; returns new code pools.

    key, value: uint16 bf16 [N, Hkv, D]; k_codes: uint8 [NB, Hkv, BS, D];
    v_codes: uint8 [NB, Hkv, D, BS]; k_scale, v_scale: float32 [Hkv].
    Negative slots are padding and are skipped; a slot written twice is rejected.
    """
    k_out = np.array(k_codes, copy=True)
    v_out = np.array(v_codes, copy=True)
    seen = set()
    num_blocks, hkv = k_out.shape[0], k_out.shape[1]
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        if slot in seen:
            raise ValueError(f"slot {slot} written twice")
        seen.add(slot)
        block, offset = divmod(slot, block_size)
        if block >= num_blocks:
            raise IndexError(f"slot {slot} outside the pool")
        for h in range(hkv):
            k_out[block, h, offset, :] = quantize(key[i, h], k_scale[h])
            v_out[block, h, :, offset] = quantize(value[i, h], v_scale[h])
    return k_out, v_out


def gather_k(k_codes, block_table_row, context_len, kv_head, k_scale, block_size):
    """Dequantised contiguous K rows [context_len, D] of one kv head of one sequence."""
    positions = np.arange(context_len)
    physical = np.asarray(block_table_row)[positions // block_size]
    if (physical < 0).any() or (physical >= k_codes.shape[0]).any():
        raise IndexError("block table entry outside the pool")
    codes = k_codes[physical, kv_head, positions % block_size, :]
    return decode(codes) * float(np.float32(k_scale[kv_head]))


def gather_v(v_codes, block_table_row, context_len, kv_head, v_scale, block_size):
    """Dequantised contiguous V rows [context_len, D] (pages stored transposed)."""
    positions = np.arange(context_len)
    physical = np.asarray(block_table_row)[positions // block_size]
    if (physical < 0).any() or (physical >= v_codes.shape[0]).any():
        raise IndexError("block table entry outside the pool")
    codes = v_codes[physical, kv_head, :, positions % block_size]      # [L, D]
    return decode(codes) * float(np.float32(v_scale[kv_head]))


def paged_attention(q_bits, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens,
                    scale, num_kv_heads, block_size, seqs=None):
    """fp64 attention over the dequantised pages; same masking and output as the bf16 oracle."""
    B, T, Hq, D = q_bits.shape
    out = np.full((B, T, Hq, D), np.nan)
    for b in (range(B) if seqs is None else seqs):
        L = int(context_lens[b])
        gathered = {}
        for h in range(Hq):
            g = O.kv_head_of(h, Hq, num_kv_heads)
            if g not in gathered:
                gathered[g] = (gather_k(k_codes, block_tables[b], L, g, k_scale, block_size),
                               gather_v(v_codes, block_tables[b], L, g, v_scale, block_size))
            Kc, Vc = gathered[g]
            for t in range(T):
                n = O.visible_length(L, T, t)
                q = O.bf16_bits_to_f64(q_bits[b, t, h])
                p = O.softmax(O.scores(Kc[:n], q, scale))
                out[b, t, h] = p @ Vc[:n]
    return out


def run_workload(w, seqs=None):
    """Quantised reshape_and_cache of the new tokens, then attention (fp64)."""
    k, v = reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                             w.k_scale, w.v_scale, w.block_size)
    return paged_attention(w.q, k, v, w.k_scale, w.v_scale, w.block_tables, w.context_lens,
                           w.scale, w.num_kv_heads, w.block_size, seqs=seqs), k, v
