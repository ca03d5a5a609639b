"""Speculative acceptance on the GPU (through the C ABI) against the oracle.

Every output (emitted tokens and the number of kept drafts) is an integer
decided in exact arithmetic on both sides, so the comparison is exact.
"""
import numpy as np
import pytest
import torch

from oracle import spec_sampling as S

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU-only hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert pa.get_device_error() == 0, "device error word was set"


def probs(rng, shape, sharp):
    x = rng.gamma(sharp, size=shape)
    return (x / x.sum(axis=-1, keepdims=True)).astype(np.float32)


def case(seed, B, K, V, sharp=0.3):
    rng = np.random.default_rng(seed)
    p = probs(rng, (B, K + 1, V), sharp)
    q = probs(rng, (B, K, V), sharp)
    drafts = np.zeros((B, K), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            # mostly drafts drawn from q, some forced to the target's best token
            if rng.random() < 0.3:
                drafts[b, i] = int(np.argmax(p[b, i]))
            else:
                qq = q[b, i].astype(np.float64)
                drafts[b, i] = int(rng.choice(V, p=qq / qq.sum()))
    a24 = rng.integers(0, 1 << 24, size=(B, K), dtype=np.uint32)
    s32 = rng.integers(0, 1 << 32, size=B, dtype=np.uint64).astype(np.uint32)
    return p, q, drafts, a24, s32


def run_gpu(p, q, drafts, a24, s32, greedy):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    toks, kept = pa.spec_accept(d(p), d(drafts), d(q), d(a24.view(np.int32)),
                                d(s32.view(np.int32)), greedy=greedy)
    return toks.cpu().numpy(), kept.cpu().numpy()


@pytest.mark.parametrize("greedy", [False, True])
@pytest.mark.parametrize("B,K,V", [(1, 1, 5), (8, 5, 1000), (32, 5, 32000), (4, 8, 128256),
                                   (3, 0, 777), (16, 3, 50257)])
def test_matches_oracle(greedy, B, K, V):
    p, q, drafts, a24, s32 = case(B * 1000 + K * 10 + V % 97, B, K, V)
    want_t, want_k = S.run_batch(p, None if greedy else q, drafts, a24, s32, greedy)
    got_t, got_k = run_gpu(p, q, drafts, a24, s32, greedy)
    np.testing.assert_array_equal(got_k, want_k)
    np.testing.assert_array_equal(got_t, want_t)


def test_many_seeds_sampling():
    for seed in range(6):
        p, q, drafts, a24, s32 = case(seed, 24, 4, 4099, sharp=1.0)
        want = S.run_batch(p, q, drafts, a24, s32, False)
        got = run_gpu(p, q, drafts, a24, s32, False)
        np.testing.assert_array_equal(got[1], want[1])
        np.testing.assert_array_equal(got[0], want[0])


def test_identical_distributions_keep_every_draft():
    p, q, drafts, a24, s32 = case(5, 8, 5, 3000)
    q = p[:, :5].copy()
    a24 = np.full_like(a24, (1 << 24) - 1)
    toks, kept = run_gpu(p, q, drafts, a24, s32, False)
    assert (kept == 5).all()
    want = S.run_batch(p, q, drafts, a24, s32, False)
    np.testing.assert_array_equal(toks, want[0])


def test_empty_residual_falls_back_to_argmax():
    """p equals q except p(draft) = 0: the draft is rejected and max(0, p - q) is all zero."""
    p, q, drafts, a24, s32 = case(6, 4, 2, 600)
    for b in range(4):
        p[b, 0] = q[b, 0]
        p[b, 0, drafts[b, 0]] = 0.0
    want = S.run_batch(p, q, drafts, a24, s32, False)
    toks, kept = run_gpu(p, q, drafts, a24, s32, False)
    assert (kept == 0).all()
    np.testing.assert_array_equal(toks, want[0])
    assert [int(t) for t in toks[:, 0]] == [int(np.argmax(p[b, 0])) for b in range(4)]


def test_extreme_uniforms():
    p, q, drafts, a24, s32 = case(7, 8, 3, 2048)
    for s in (0, (1 << 32) - 1):
        s32 = np.full(8, s, dtype=np.uint32)
        want = S.run_batch(p, q, drafts, a24, s32, False)
        got = run_gpu(p, q, drafts, a24, s32, False)
        np.testing.assert_array_equal(got[0], want[0])


def test_bad_draft_token_reports_bounds():
    p, q, drafts, a24, s32 = case(8, 2, 3, 100)
    drafts[1, 0] = 100                           # the first draft is always examined
    toks, kept = run_gpu(p, q, drafts, a24, s32, False)
    assert pa.get_device_error() == 5
    assert kept[1] == 0 and 0 <= toks[1, 0] < 100 and (toks[1, 1:] == -1).all()
    want = S.run_batch(p[:1], q[:1], drafts[:1], a24[:1], s32[:1], False)
    np.testing.assert_array_equal(toks[:1], want[0])     # other sequences unaffected
