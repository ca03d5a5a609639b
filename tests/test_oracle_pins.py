"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each pin is a plain function so that the planted-mistake test at the bottom can
re-run every pin against deliberately broken copies of the oracle and check
that each broken copy fails at least one of them.

Sources of truth used here: an independent scalar brute force, library
attention (torch's scaled_dot_product_attention in fp64 on the CPU), closed
forms (L = 1, q = 0, a two-key example), invariants the paging definition
implies (physical placement and copy-on-write sharing cannot change the
result), and the worked figures the pages print.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import accounting, brute
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def full_caches(w):
    """Caches with the workload's new tokens scattered in (NumPy fancy indexing, not the oracle)."""
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    s = w.slot_mapping
    k[s // w.block_size, :, s % w.block_size, :] = w.new_key
    v[s // w.block_size, :, s % w.block_size, :] = w.new_value
    return k, v


def run(ora, w, k=None, v=None, q=None, tables=None):
    if k is None:
        k, v = full_caches(w)
    return ora.paged_attention(w.q if q is None else q, k, v,
                               w.block_tables if tables is None else tables,
                               w.context_lens, w.scale, w.num_kv_heads, w.block_size)


def bits(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def gqa_verify_case(seed=7):
    """3 seqs, 3 query tokens, 8 q heads over 2 kv heads, head_dim 16, random placement."""
    return W.build("gqa_verify", [3, 17, 40], num_q_heads=8, num_kv_heads=2, head_dim=16,
                   num_query_tokens=3, seed=seed)


# ----------------------------------------------------------------------------- pins

def pin_brute_tiny(ora):
    w = W.tiny()
    k, v = full_caches(w)
    ref = np.array(brute.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                                         w.num_kv_heads, w.block_size))
    np.testing.assert_allclose(run(ora, w, k, v), ref, rtol=0, atol=1e-12)


def pin_brute_gqa_verify(ora):
    w = gqa_verify_case()
    k, v = full_caches(w)
    ref = np.array(brute.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                                         w.num_kv_heads, w.block_size))
    np.testing.assert_allclose(run(ora, w, k, v), ref, rtol=0, atol=1e-12)


def pin_permutation_invariance(ora):
    """Moving blocks to other physical ids (and rewriting the tables) changes nothing."""
    w = gqa_verify_case(seed=11)
    k, v = full_caches(w)
    base = run(ora, w, k, v)
    perm = np.random.default_rng(5).permutation(w.num_blocks)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1)
    np.testing.assert_array_equal(run(ora, w, k2, v2, tables=tables), base)


def pin_shared_equals_duplicated(ora):
    """A table that shares prefix blocks equals one pointing at private copies of them."""
    w = W.build("shared", [70, 90, 33], num_q_heads=4, num_kv_heads=2, head_dim=16,
                shared=[([0, 1, 2], 2)], seed=3)
    k, v = full_caches(w)
    base = run(ora, w, k, v)
    nb = w.num_blocks
    extra = 2 * 2                       # two extra private copies of the 2 shared blocks
    k2 = np.concatenate([k, np.zeros((extra,) + k.shape[1:], k.dtype)])
    v2 = np.concatenate([v, np.zeros((extra,) + v.shape[1:], v.dtype)])
    tables = w.block_tables.copy()
    nxt = nb
    for b in (1, 2):
        for j in range(2):
            src = tables[b, j]
            k2[nxt] = k[src]
            v2[nxt] = v[src]
            tables[b, j] = nxt
            nxt += 1
    assert len(set(tables[:, :2].ravel().tolist())) == 6
    np.testing.assert_allclose(run(ora, w, k2, v2, tables=tables), base, rtol=0, atol=1e-12)


def pin_weights_sum_to_one(ora):
    w = gqa_verify_case(seed=13)
    k, v = full_caches(w)
    out = run(ora, w, k, v)
    for b in range(w.num_seqs):
        for t in range(w.num_query_tokens):
            for h in range(w.num_q_heads):
                p = ora.attention_weights(w.q, k, w.block_tables, w.context_lens, w.scale,
                                          w.num_kv_heads, w.block_size, b, t, h)
                assert abs(p.sum() - 1.0) < 1e-12
                assert (p >= 0).all()
                L = int(w.context_lens[b])
                assert len(p) == L - w.num_query_tokens + t + 1
                g = h // (w.num_q_heads // w.num_kv_heads)
                Vc = O.bf16_bits_to_f64(np.stack(
                    [v[w.block_tables[b, j // 16], g, j % 16] for j in range(len(p))]))
                np.testing.assert_allclose(p @ Vc, out[b, t, h], rtol=0, atol=1e-12)


def pin_single_block_equals_dense(ora):
    """A context inside one block equals textbook attention (torch SDPA, fp64, CPU)."""
    for T, L in [(1, 16), (3, 11), (2, 2)]:
        w = W.build("dense", [L, L], num_q_heads=6, num_kv_heads=2, head_dim=32,
                    num_query_tokens=T, seed=20 + L)
        k, v = full_caches(w)
        out = run(ora, w, k, v)
        G = w.num_q_heads // w.num_kv_heads
        for b in range(2):
            blk = w.block_tables[b, 0]
            K = torch.from_numpy(O.bf16_bits_to_f64(k[blk, :, :L, :]))      # [Hkv, L, D]
            V = torch.from_numpy(O.bf16_bits_to_f64(v[blk, :, :L, :]))
            Q = torch.from_numpy(O.bf16_bits_to_f64(w.q[b])).permute(1, 0, 2)  # [Hq, T, D]
            K = K.repeat_interleave(G, dim=0)
            V = V.repeat_interleave(G, dim=0)
            rows = torch.arange(T)[:, None]
            cols = torch.arange(L)[None, :]
            mask = cols <= (L - T + rows)
            ref = torch.nn.functional.scaled_dot_product_attention(
                Q, K, V, attn_mask=mask, scale=w.scale)                      # [Hq, T, D]
            np.testing.assert_allclose(out[b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def pin_length_one(ora):
    """One cached token: the output is that token's V row, exactly."""
    w = W.build("L1", [1, 1], num_q_heads=4, num_kv_heads=2, head_dim=16, seed=31)
    k, v = full_caches(w)
    out = run(ora, w, k, v)
    for b in range(2):
        blk = w.block_tables[b, 0]
        for h in range(4):
            np.testing.assert_array_equal(out[b, 0, h], O.bf16_bits_to_f64(v[blk, h // 2, 0]))


def pin_zero_query_mean(ora):
    """q = 0 makes every score equal: the output is the mean of the visible V rows."""
    w = W.build("q0", [45, 19], num_q_heads=4, num_kv_heads=4, head_dim=8,
                num_query_tokens=2, seed=41)
    k, v = full_caches(w)
    q = np.zeros_like(w.q)
    out = run(ora, w, k, v, q=q)
    for b in range(2):
        L = int(w.context_lens[b])
        for t in range(2):
            n = L - 2 + t + 1
            for h in range(4):
                rows = [O.bf16_bits_to_f64(v[w.block_tables[b, j // 16], h, j % 16])
                        for j in range(n)]
                np.testing.assert_allclose(out[b, t, h], np.mean(rows, axis=0), rtol=0,
                                           atol=1e-12)


def pin_two_key_closed_form(ora):
    """q = (1, 0), keys (2, 0) and (0, 0), values e1 and e2, scale 1: weights e^2/(e^2+1), 1/(e^2+1)."""
    q = bits([[[[1.0, 0.0]]]])                             # [B=1, T=1, Hq=1, D=2]
    k = np.full((1, 1, 16, 2), W.NAN_BITS, np.uint16)
    v = np.full((1, 1, 16, 2), W.NAN_BITS, np.uint16)
    k[0, 0, :2] = bits([[2.0, 0.0], [0.0, 0.0]])
    v[0, 0, :2] = bits([[1.0, 0.0], [0.0, 1.0]])
    out = ora.paged_attention(q, k, v, np.array([[0]], np.int32), np.array([2], np.int32), 1.0,
                              1, 16)
    e2 = math.exp(2.0)
    np.testing.assert_allclose(out[0, 0, 0], [e2 / (e2 + 1), 1 / (e2 + 1)], rtol=0, atol=1e-15)


def pin_verify_rows_are_stacked_decodes(ora):
    """Draft t of a verify pass equals a one-token decode whose context ends at that draft."""
    w = gqa_verify_case(seed=17)
    k, v = full_caches(w)
    out = run(ora, w, k, v)
    T = w.num_query_tokens
    for t in range(T):
        lens = w.context_lens - T + 1 + t
        dec = ora.paged_attention(w.q[:, t:t + 1], k, v, w.block_tables, lens, w.scale,
                                  w.num_kv_heads, w.block_size)
        np.testing.assert_allclose(out[:, t], dec[:, 0], rtol=0, atol=1e-13)


def pin_reshape_and_cache(ora):
    w = gqa_verify_case(seed=19)
    k, v = ora.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping,
                                 w.block_size)
    s = w.slot_mapping
    np.testing.assert_array_equal(k[s // 16, :, s % 16, :], w.new_key)
    np.testing.assert_array_equal(v[s // 16, :, s % 16, :], w.new_value)
    mask = np.ones(k.shape[0] * 16, bool)
    mask[s] = False
    kk = k.transpose(0, 2, 1, 3).reshape(-1, *k.shape[1:2], k.shape[3])
    k0 = w.k_cache.transpose(0, 2, 1, 3).reshape(-1, *k.shape[1:2], k.shape[3])
    np.testing.assert_array_equal(kk[mask], k0[mask])
    # padding tokens (slot < 0) are skipped
    s2 = s.copy()
    s2[0] = -1
    k3, _ = ora.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, s2, 16)
    np.testing.assert_array_equal(k3[s[0] // 16, :, s[0] % 16], w.k_cache[s[0] // 16, :, s[0] % 16])
    with pytest.raises(ValueError):
        ora.reshape_and_cache(w.new_key[:2], w.new_value[:2], w.k_cache, w.v_cache,
                              np.array([s[0], s[0]]), 16)


PINS = [pin_brute_tiny, pin_brute_gqa_verify, pin_permutation_invariance,
        pin_shared_equals_duplicated, pin_weights_sum_to_one, pin_single_block_equals_dense,
        pin_length_one, pin_zero_query_mean, pin_two_key_closed_form,
        pin_verify_rows_are_stacked_decodes, pin_reshape_and_cache]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(O)


# ----------------------------------------------------------------------------- planted mistakes

class Mutant:
    """The oracle module with one function replaced (the real module is never touched)."""

    def __init__(self, **overrides):
        self._o = overrides

    def __getattr__(self, name):
        if name in self._o:
            return self._o[name]
        f = getattr(O, name)
        if callable(f) and getattr(f, "__module__", "") == O.__name__:
            # rebind globals so oracle-internal calls see the overrides
            import types
            g = dict(f.__globals__)
            g.update(self._o)
            return types.FunctionType(f.__code__, g, f.__name__, f.__defaults__, f.__closure__)
        return f


def _bad_gather_transposed(cache, row, L, g, bs):
    pos = np.arange(L)
    return O.bf16_bits_to_f64(cache[np.asarray(row)[pos % bs], g, pos // bs, :])


def _bad_gather_logical(cache, row, L, g, bs):
    pos = np.arange(L)
    return O.bf16_bits_to_f64(cache[pos // bs, g, pos % bs, :])


def _bad_reshape(key, value, k_cache, v_cache, slots, bs):
    k, v = np.array(k_cache), np.array(v_cache)
    for i, s in enumerate(np.asarray(slots).tolist()):
        if s < 0:
            continue
        k[s % bs, :, s // bs] = key[i]       # block and offset swapped
        v[s % bs, :, s // bs] = value[i]
    return k, v


def _bad_bf16(bits):
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(15)
    return u.view(np.float32).astype(np.float64)


MUTANTS = {
    "gqa_mapping_modulo": dict(kv_head_of=lambda h, hq, hkv: h % hkv),
    "mask_off_by_one": dict(visible_length=lambda L, T, t: L - T + t),
    "no_causal_mask": dict(visible_length=lambda L, T, t: L),
    "mask_reversed": dict(visible_length=lambda L, T, t: L - t),
    "gather_transposed": dict(gather_context=_bad_gather_transposed),
    "gather_ignores_table": dict(gather_context=_bad_gather_logical),
    "scale_dropped": dict(scores=lambda K, q, s: K @ q),
    "scale_squared": dict(scores=lambda K, q, s: s * s * (K @ q)),
    "softmax_unnormalised": dict(softmax=lambda z: np.exp(z - z.max())),
    "softmax_sign": dict(softmax=lambda z: np.exp(-(z - z.min())) / np.exp(-(z - z.min())).sum()),
    "reshape_block_offset_swapped": dict(reshape_and_cache=_bad_reshape),
    "bf16_shift": dict(bf16_bits_to_f64=_bad_bf16),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    m = Mutant(**MUTANTS[name])
    failed = []
    for pin in PINS:
        try:
            pin(m)
        except Exception:            # AssertionError, IndexError, ... all count as caught
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"


# ----------------------------------------------------------------------------- page figures

def test_page_figures():
    g = json.load(open(os.path.join(GOLDEN, "page_figures.json")))
    assert W.BLOCK_SIZE == g["block_size"]["value"]
    r = g["reservation_example"]
    assert accounting.reservation_unused_fraction(r["used_tokens"], r["reserved_tokens"]) > \
        r["unused_fraction_above"]
    m = g["memory_wall"]
    sec = accounting.bandwidth_bound_seconds(m["bytes"], m["bytes_per_second"])
    assert sec == pytest.approx(m["seconds"])
    assert round(1 / sec) == m["tokens_per_second_about"]
    bound = g["paged_waste_below"]["fraction"]
    for L in range(20 * 16, 4096, 37):
        assert accounting.paged_unused_fraction(L, W.BLOCK_SIZE) < bound


def test_benchmark_byte_count_matches_kv_formula():
    """The workload's algorithmic KV bytes equal the pages' KV-size formula (one layer).

    With block-aligned lengths and no sharing, pages read = tokens / 16 per kv
    head, so unique-page bytes must equal 2 x tokens x heads x head_dim x 2 bytes.
    """
    w = W.build("acct", [160, 32, 512], num_q_heads=8, num_kv_heads=4, head_dim=64, seed=2)
    want = sum(accounting.kv_cache_bytes(1, int(L), 1, w.num_kv_heads, w.head_dim, 2)
               for L in w.context_lens)
    assert w.kv_bytes() == want
    # sharing: a group's prefix is counted once
    s = W.build("acct2", [64, 64], num_q_heads=4, num_kv_heads=2, head_dim=16,
                shared=[([0, 1], 2)], seed=2)
    assert s.unique_pages() == (2 + 2 + 2) * 2
    assert s.logical_pages() == 8 * 2


def test_workload_sentinels():
    """Slots past the context and the newest tokens hold NaN until reshape_and_cache runs."""
    w = W.tiny()
    s = w.slot_mapping
    assert (w.k_cache[s // 16, :, s % 16] == W.NAN_BITS).all()
    k, _ = full_caches(w)
    for b in range(2):
        L = int(w.context_lens[b])
        last = w.block_tables[b, (L - 1) // 16]
        assert (k[last, :, L % 16 or 16:] == W.NAN_BITS).all()
        assert not (k[last, :, :(L - 1) % 16 + 1] == W.NAN_BITS).any()


def test_f32_to_bf16_rounding():
    """Round-to-nearest-even against torch's own bf16 conversion."""
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0]      # ties to even, exact values
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(W.f32_to_bf16_bits(x), ref)


def test_oracle_on_small_workloads_is_finite():
    """Every small named workload runs through the oracle without touching a NaN sentinel."""
    for name, make in W.SMALL.items():
        w = make()
        out, _, _ = O.run_workload(w)
        assert np.isfinite(out).all(), name
