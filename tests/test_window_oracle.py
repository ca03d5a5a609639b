"""Pins of the sliding-window oracle against facts that do not come from it.

Sources of truth: a window at least as long as the context is plain attention
(the pinned oracle); a window of one position returns that position's V exactly;
for one query token, attending to the last W positions equals plain attention
over a sequence whose block table starts at the window (when the window starts
on a block boundary); verify rows equal stacked single-token decodes; and an
independent scalar brute force.  Planted mistakes each fail a pin.
"""
import math
import types

import numpy as np
import pytest

import workloads as W
from fp8_cases import exact_fp8_case
from oracle import fp8 as F
from oracle import oracle as O
from oracle import window as WIN


def full_pools(w):
    return O.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping,
                               w.block_size)


def case(seed=21, T=1, lens=(40, 64, 100)):
    return W.build("win", list(lens), num_q_heads=8, num_kv_heads=2, head_dim=16,
                   num_query_tokens=T, seed=seed)


def pin_long_window_is_plain_attention(win):
    w = case(T=3)
    k, v = full_pools(w)
    want = O.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                             w.num_kv_heads, 16)
    got = win.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                              w.num_kv_heads, 16, int(w.context_lens.max()))
    np.testing.assert_array_equal(got, want)


def pin_window_of_one_is_own_value(win):
    w = case(T=2)
    k, v = full_pools(w)
    got = win.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                              w.num_kv_heads, 16, 1)
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        for t in range(2):
            pos = L - 2 + t
            blk, off = w.block_tables[b, pos // 16], pos % 16
            for h in range(w.num_q_heads):
                g = h // (w.num_q_heads // w.num_kv_heads)
                np.testing.assert_array_equal(got[b, t, h], O.bf16_bits_to_f64(v[blk, g, off]))


def pin_window_equals_truncated_table(win):
    """T = 1, window W with L - W a multiple of 16: plain attention over the table
    that starts at block (L - W) / 16 with context W."""
    w = case(T=1, lens=(80, 96, 112))
    k, v = full_pools(w)
    Wn = 48
    got = win.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                              w.num_kv_heads, 16, Wn)
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        start = (L - Wn) // 16
        tab = np.full((1, w.block_tables.shape[1]), -1, dtype=np.int32)
        nb = -(-Wn // 16)
        tab[0, :nb] = w.block_tables[b, start:start + nb]
        want = O.paged_attention(w.q[b:b + 1], k, v, tab, np.array([Wn], dtype=np.int32),
                                 w.scale, w.num_kv_heads, 16)
        np.testing.assert_allclose(got[b:b + 1], want, rtol=1e-12, atol=1e-14)


def pin_verify_rows_are_stacked_windowed_decodes(win):
    w = case(T=4)
    k, v = full_pools(w)
    Wn = 7
    got = win.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                              w.num_kv_heads, 16, Wn)
    for t in range(4):
        lens = w.context_lens - 4 + t + 1
        one = win.paged_attention(w.q[:, t:t + 1], k, v, w.block_tables, lens, w.scale,
                                  w.num_kv_heads, 16, Wn)
        np.testing.assert_allclose(got[:, t:t + 1], one, rtol=1e-12, atol=1e-14)


def pin_brute_force(win):
    w = case(T=2, lens=(20, 35))
    k, v = full_pools(w)
    Wn = 9
    got = win.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                              w.num_kv_heads, 16, Wn)
    f = lambda bits: float(O.bf16_bits_to_f64(np.array([bits]))[0])
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        for t in range(2):
            pos = L - 2 + t
            js = [j for j in range(L) if pos - Wn < j <= pos]
            for h in range(w.num_q_heads):
                g = h // 4
                sc = []
                for j in js:
                    blk, off = w.block_tables[b, j // 16], j % 16
                    sc.append(w.scale * sum(f(w.q[b, t, h, d]) * f(k[blk, g, off, d])
                                            for d in range(16)))
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                for d in range(16):
                    o = sum(e[i] * f(v[w.block_tables[b, js[i] // 16], g, js[i] % 16, d])
                            for i in range(len(js))) / sum(e)
                    assert abs(o - got[b, t, h, d]) < 1e-12


def pin_run_workload_long_window_is_plain_step(win):
    """The whole windowed step (append, then attention) with a window covering every
    context equals the pinned plain step, bit for bit, for both page formats."""
    w = case(T=3)
    got, k, v = win.run_workload(w, int(w.context_lens.max()))
    want, kw, vw = O.run_workload(w)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(k, kw)
    np.testing.assert_array_equal(v, vw)
    w8, _ = exact_fp8_case(seed=23, lens=(9, 33, 48), T=3)
    got, k, v = win.run_workload(w8, int(w8.context_lens.max()))
    want, kw, vw = F.run_workload(w8)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(k, kw)
    np.testing.assert_array_equal(v, vw)


def pin_run_workload_window_of_one_is_new_value(win):
    """A window of one position: every query token returns the V it appended itself,
    for both page formats (the FP8 case's new values are exact E4M3 values)."""
    w = case(T=2)
    w8, _ = exact_fp8_case(seed=29, lens=(6, 31, 50), T=2)
    for wk in (w, w8):
        got = win.run_workload(wk, 1)[0]
        G = wk.num_q_heads // wk.num_kv_heads
        for b in range(wk.num_seqs):
            for t in range(2):
                for h in range(wk.num_q_heads):
                    want = O.bf16_bits_to_f64(wk.new_value[b * 2 + t, h // G])
                    np.testing.assert_array_equal(got[b, t, h], want)


PINS = [pin_long_window_is_plain_attention, pin_window_of_one_is_own_value,
        pin_window_equals_truncated_table, pin_verify_rows_are_stacked_windowed_decodes,
        pin_brute_force, pin_run_workload_long_window_is_plain_step,
        pin_run_workload_window_of_one_is_new_value]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(WIN)


class Mutant:
    def __init__(self, **overrides):
        self._o = overrides

    def __getattr__(self, name):
        if name in self._o:
            return self._o[name]
        f = getattr(WIN, name)
        if isinstance(f, types.FunctionType) and f.__module__ == WIN.__name__:
            g = dict(f.__globals__)
            g.update(self._o)
            return types.FunctionType(f.__code__, g, f.__name__, f.__defaults__, f.__closure__)
        return f


def _run_window_plus_one(w, window, seqs=None):
    return WIN.run_workload(w, window + 1, seqs)


def _run_fp8_as_bf16(w, window, seqs=None):
    k, v = O.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping,
                               w.block_size)
    return WIN.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                               w.num_kv_heads, w.block_size, window, seqs), k, v


def _run_fp8_scales_swapped(w, window, seqs=None):
    if w.kv_dtype != "fp8":
        return WIN.run_workload(w, window, seqs)
    k, v = F.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                               w.k_scale, w.v_scale, w.block_size)
    return WIN.paged_attention(w.q, k, v, w.block_tables, w.context_lens, w.scale,
                               w.num_kv_heads, w.block_size, window, seqs, w.v_scale,
                               w.k_scale), k, v


MUTANTS = {
    "run_workload_window_plus_one": dict(run_workload=_run_window_plus_one),
    "run_workload_fp8_as_bf16": dict(run_workload=_run_fp8_as_bf16),
    "run_workload_fp8_scales_swapped": dict(run_workload=_run_fp8_scales_swapped),
    "window_one_too_long": dict(visible_range=lambda L, T, t, w: (max(0, L - T + t - w), L - T + t)),
    "window_from_context_end": dict(visible_range=lambda L, T, t, w: (max(0, L - w), L - T + t)),
    "window_not_clamped": dict(visible_range=lambda L, T, t, w: (L - T + t - w + 1, L - T + t)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    m = Mutant(**MUTANTS[name])
    failed = []
    for pin in PINS:
        try:
            pin(m)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
