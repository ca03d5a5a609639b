"""Pins of the speculative-acceptance oracle against facts that do not come from it.

Sources of truth: closed forms of the greedy rule and of the integer inverse-CDF
draw, and the mathematical guarantee of rejection sampling: whatever the draft
distribution, the first emitted token follows the target distribution, the
first draft is kept with probability sum_x min(p(x), q(x)), and once it is kept
the next emitted token follows the target's next distribution.  These are
checked by sampling with independent random numbers (5-sigma bounds).  The
planted-mistake test re-runs every pin against broken copies of the oracle.
"""
import types

import numpy as np
import pytest

from oracle import spec_sampling as S


def normalised(rng, n, V, sharp=1.0):
    x = rng.gamma(sharp, size=(n, V))
    return (x / x.sum(axis=1, keepdims=True)).astype(np.float32)


# ----------------------------------------------------------------------------- pins

def pin_greedy_closed_forms(s):
    p = np.zeros((4, 6), dtype=np.float32)
    p[0, 2] = 0.9
    p[1, 4] = 0.6
    p[2, 1] = 0.5
    p[3, 5] = 0.7
    p += 0.01
    out, n = s.speculative_step(p, None, [2, 4, 3], None, 0, True)
    assert (out, n) == ([2, 4, 1, -1], 2)               # third draft wrong: target's token
    out, n = s.speculative_step(p, None, [2, 4, 1], None, 0, True)
    assert (out, n) == ([2, 4, 1, 5], 3)                # all kept: bonus token
    out, n = s.speculative_step(p, None, [0, 4, 1], None, 0, True)
    assert (out, n) == ([2, -1, -1, -1], 0)
    tie = np.full((2, 5), 0.2, dtype=np.float32)
    out, n = s.speculative_step(tie, None, [3], None, 0, True)
    assert (out, n) == ([0, -1], 0)                     # ties: the lowest index


def pin_inverse_cdf_closed_forms(s):
    w = [0, 3, 0, 5]
    assert s.inverse_cdf_draw(w, 0) == 1
    assert s.inverse_cdf_draw(w, (1 << 32) - 1) == 3
    assert s.inverse_cdf_draw(w, 1 << 31) == 3          # target floor(8/2) = 4 -> prefix 8
    assert s.inverse_cdf_draw(w, (3 << 29) - 1) == 1    # target floor(3 - 2^-29) = 2
    assert s.inverse_cdf_draw(w, 3 << 29) == 3          # target 3: the prefix must exceed it
    assert s.inverse_cdf_draw([0, 0], 5) is None
    r = np.array([0.5, 0.25, 0.0, 0.25], dtype=np.float32)
    assert s.quantised_weights(r) == [1 << 39, 1 << 38, 0, 1 << 38]


def pin_keep_rule_closed_forms(s):
    assert s.keep_draft(0.3, 0.3, (1 << 24) - 1)         # p == q: always kept
    assert not s.keep_draft(0.0, 0.3, 0)                 # p == 0: never kept
    assert s.keep_draft(0.2, 0.4, (1 << 23) - 1)         # ratio 1/2: kept below a = 2^23
    assert not s.keep_draft(0.2, 0.4, 1 << 23)


def _sample_runs(s, seed, n, K=3, V=5):
    rng = np.random.default_rng(seed)
    p = normalised(rng, K + 1, V)
    q = normalised(rng, K, V, sharp=0.5)
    first = np.zeros(V)
    kept1 = 0
    second = np.zeros(V)
    for _ in range(n):
        drafts = [int(rng.choice(V, p=q[i] / q[i].sum())) for i in range(K)]
        a24 = rng.integers(0, 1 << 24, size=K)
        s32 = int(rng.integers(0, 1 << 32))
        out, kept = s.speculative_step(p, q, drafts, a24, s32, False)
        assert 0 <= kept <= K and out[kept] >= 0 and all(t == -1 for t in out[kept + 1:])
        assert out[:kept] == drafts[:kept]
        first[out[0]] += 1
        if kept >= 1:
            kept1 += 1
            second[out[1]] += 1
    return p, q, first, kept1, second


def _within(counts, probs, n):
    sigma = np.sqrt(n * probs * (1 - probs)) + 1e-9
    return np.all(np.abs(counts - n * probs) <= 5 * sigma + 1)


def pin_rejection_sampling_keeps_target_distribution(s):
    n = 20000
    p, q, first, kept1, second = _sample_runs(s, 3, n)
    p64 = p.astype(np.float64)
    assert _within(first, p64[0] / p64[0].sum(), n)
    acc = np.minimum(p64[0], q[0].astype(np.float64)).sum()
    assert abs(kept1 - n * acc) <= 5 * np.sqrt(n * acc * (1 - acc)) + 1
    assert _within(second, p64[1] / p64[1].sum(), kept1)


def pin_bonus_follows_last_target_row(s):
    """When the drafts equal the target rows' certain tokens, every draft is kept and the
    bonus token follows the last target row."""
    rng = np.random.default_rng(8)
    V, K, n = 4, 2, 8000
    p = np.zeros((K + 1, V), dtype=np.float32)
    p[0, 1] = 1.0
    p[1, 3] = 1.0
    p[K] = np.array([0.1, 0.2, 0.3, 0.4], dtype=np.float32)
    q = p[:K].copy()
    counts = np.zeros(V)
    for _ in range(n):
        out, kept = s.speculative_step(p, q, [1, 3], rng.integers(0, 1 << 24, size=K),
                                       int(rng.integers(0, 1 << 32)), False)
        assert kept == K
        counts[out[K]] += 1
    assert _within(counts, p[K].astype(np.float64), n)


PINS = [pin_greedy_closed_forms, pin_inverse_cdf_closed_forms, pin_keep_rule_closed_forms,
        pin_rejection_sampling_keeps_target_distribution, pin_bonus_follows_last_target_row]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(S)


def test_batch_matches_single_sequences():
    rng = np.random.default_rng(4)
    B, K, V = 3, 4, 50
    p = np.stack([normalised(rng, K + 1, V) for _ in range(B)])
    q = np.stack([normalised(rng, K, V) for _ in range(B)])
    drafts = rng.integers(0, V, size=(B, K))
    a24 = rng.integers(0, 1 << 24, size=(B, K))
    s32 = rng.integers(0, 1 << 32, size=B)
    toks, kept = S.run_batch(p, q, drafts, a24, s32, False)
    for b in range(B):
        t, n = S.speculative_step(p[b], q[b], drafts[b], a24[b], int(s32[b]), False)
        assert toks[b].tolist() == t and kept[b] == n


# ----------------------------------------------------------------------------- planted mistakes

class Mutant:
    def __init__(self, **overrides):
        self._o = overrides

    def __getattr__(self, name):
        if name in self._o:
            return self._o[name]
        f = getattr(S, name)
        if isinstance(f, types.FunctionType) and f.__module__ == S.__name__:
            g = dict(f.__globals__)
            g.update(self._o)
            return types.FunctionType(f.__code__, g, f.__name__, f.__defaults__, f.__closure__)
        return f


def _ratio_inverted(p_x, q_x, a24):
    return float(np.float32(p_x)) * float(a24) < float(np.float32(q_x)) * S.TWO24


def _residual_reversed(p_row, q_row):
    return S.residual(q_row, p_row)


def _draw_ge(weights, s32):
    total = sum(weights)
    if total == 0:
        return None
    target = (int(s32) * total) >> 32
    run = 0
    for x, wx in enumerate(weights):
        run += wx
        if run >= target:
            return x
    return len(weights) - 1


def _argmax_highest(p):
    p = np.asarray(p)
    return int(np.flatnonzero(p == p.max())[-1])


def _keep_always(p_x, q_x, a24):
    return True


MUTANTS = {
    "ratio_inverted": dict(keep_draft=_ratio_inverted),
    "residual_reversed": dict(residual=_residual_reversed),
    "inverse_cdf_off_by_one": dict(inverse_cdf_draw=_draw_ge),
    "ties_highest_index": dict(argmax_lowest=_argmax_highest),
    "never_reject": dict(keep_draft=_keep_always),
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
