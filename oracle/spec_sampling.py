"""Speculative-decoding acceptance: the CPU oracle of the library's accept kernel.

TEST INFRASTRUCTURE ONLY (same rules as ``oracle.py``: only the tests, the
smoke check and the benchmark's CPU legs may import it; it shares no code with
the CUDA path).

A draft model proposes K tokens; the target model scores all of them in one
pass; the target keeps the drafts that agree with it, stops at the first one
that does not (every later draft is dropped with it), and then emits one token
of its own ("ranksignal" post, Spéculer : plusieurs tokens par passe;
"PagedAttention, décodage spéculatif, MoE et Blackwell", §1, vérification
parallèle; "LLM inference optimization: KV cache", §5.2).  With rejection
sampling the output tokens follow exactly the target's distribution ("LLM
inference optimization: KV cache", §5.3).  Two rules:

* greedy: draft i is kept while it equals the target's most probable token at
  position i (the lowest index among equal maxima); at the first position where
  it differs, or after all K drafts (the bonus position K), the target's most
  probable token is emitted;
* sampling (the textbook rejection-sampling rule): draft x_i is kept with
  probability min(1, p_i(x_i) / q_i(x_i)); at the first rejection the emitted
  token is drawn from the residual max(0, p_i - q_i), normalised; after all K
  drafts it is drawn from p_K.

The random numbers are inputs, and every decision is written in exact
arithmetic so that any correct implementation reaches the same tokens:

* acceptance uses a 24-bit uniform a_i (the low 24 bits of the given integer):
  keep iff q * a_i < p * 2^24, both sides exact in fp64 (p, q are float32);
* the final draw uses a 32-bit uniform s and weights quantised to multiples of
  2^-40: w(x) = floor(r(x) * 2^40) with r(x) = max(0, p(x) - q(x)) evaluated in
  float32 (or r = p at the bonus position); W = sum of w; the token is the
  smallest x whose prefix sum of w exceeds floor(s * W / 2^32).  If W is 0 (no
  residual mass left after rounding) the target's most probable token is
  emitted instead.

Probabilities are inputs (the softmax that produces them is outside this step).
"""
from __future__ import annotations

import numpy as np

TWO24 = float(1 << 24)
QUANT_SHIFT = 40


def argmax_lowest(p) -> int:
    """Index of the largest value, the lowest index among equal maxima."""
    p = np.asarray(p)
    return int(np.flatnonzero(p == p.max())[0])


def keep_draft(p_x, q_x, a24) -> bool:
    """Rejection test: keep iff a24 / 2^24 < p / q, written as q * a24 < p * 2^24 (exact)."""
    return float(np.float32(q_x)) * float(int(a24) & 0xFFFFFF) < float(np.float32(p_x)) * TWO24


def residual(p_row, q_row) -> np.ndarray:
    """max(0, p - q) in float32."""
    d = np.asarray(p_row, dtype=np.float32) - np.asarray(q_row, dtype=np.float32)
    return np.maximum(d, np.float32(0))


def quantised_weights(r_row) -> list:
    """floor(r * 2^40) as Python integers (r float32 in [0, 1], the product is exact)."""
    scaled = np.asarray(r_row, dtype=np.float32).astype(np.float64) * float(1 << QUANT_SHIFT)
    return [int(v) for v in np.floor(scaled)]


def inverse_cdf_draw(weights, s32):
    """Smallest x with sum(weights[:x+1]) > floor(s32 * W / 2^32); None if W == 0."""
    total = sum(weights)
    if total == 0:
        return None
    target = (int(s32) * total) >> 32
    run = 0
    for x, wx in enumerate(weights):
        run += wx
        if run > target:
            return x
    raise AssertionError("unreachable: target < total")


def speculative_step(p, q, drafts, a24, s32, greedy):
    """One sequence.  p: float32 [K+1, V] target probabilities, q: float32 [K, V] draft
    probabilities (unused when greedy), drafts: int [K], a24: [K] 24-bit uniforms,
    s32: 32-bit uniform.  Returns (tokens [K+1] with -1 after the emitted ones,
    number of drafts kept)."""
    K = len(drafts)
    out = [-1] * (K + 1)
    for i in range(K):
        x = int(drafts[i])
        if greedy:
            ok = x == argmax_lowest(p[i])
        else:
            ok = keep_draft(p[i][x], q[i][x], a24[i])
        if not ok:
            if greedy:
                final = argmax_lowest(p[i])
            else:
                final = inverse_cdf_draw(quantised_weights(residual(p[i], q[i])), s32)
                if final is None:
                    final = argmax_lowest(p[i])
            out[:i] = [int(d) for d in drafts[:i]]
            out[i] = final
            return out, i
    if greedy:
        final = argmax_lowest(p[K])
    else:
        final = inverse_cdf_draw(quantised_weights(np.asarray(p[K], dtype=np.float32)), s32)
        if final is None:
            final = argmax_lowest(p[K])
    out[:K] = [int(d) for d in drafts]
    out[K] = final
    return out, K


def run_batch(p, q, drafts, a24, s32, greedy):
    """Every sequence of a batch: p [B, K+1, V], q [B, K, V] (or None), drafts [B, K],
    a24 [B, K], s32 [B].  Returns (tokens [B, K+1] int32, kept [B] int32)."""
    B, K = np.asarray(drafts).shape
    toks = np.full((B, K + 1), -1, dtype=np.int32)
    kept = np.zeros(B, dtype=np.int32)
    for b in range(B):
        t, n = speculative_step(p[b], None if q is None else q[b], drafts[b],
                                None if a24 is None else a24[b],
                                0 if s32 is None else s32[b], greedy)
        toks[b] = t
        kept[b] = n
    return toks, kept
