"""Copy-on-write on the GPU: the block-copy kernel bit for bit against the
oracle, and forked sequences decoding through the native block manager's
tables, checked against attention over each sequence's own contiguous history.

Tolerance for attention outputs as in the other parity tests: max abs error
<= 1e-2 (or one bf16 ulp of the oracle value, where that is larger) and relative
L2 error <= 2e-3 against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import block_manager as OBM
from oracle import oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU-only hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402
from gpu_util import assert_close, bits, to_dev  # noqa: E402

BS = 16


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert pa.get_device_error() == 0, "device error word was set"


def random_pool(rng, nb, hkv, d):
    return (W.normal_bf16(rng, (nb, hkv, BS, d)), W.normal_bf16(rng, (nb, hkv, BS, d)))


@pytest.mark.parametrize("hkv,d,npairs", [(8, 128, 1), (8, 128, 37), (4, 64, 200), (1, 64, 5)])
def test_copy_blocks_bit_exact(hkv, d, npairs):
    rng = np.random.default_rng(hkv * 1000 + npairs)
    nb = 3 * npairs + 8
    k, v = random_pool(rng, nb, hkv, d)
    ids = rng.permutation(nb)
    pairs = list(zip(ids[:npairs].tolist(), ids[npairs:2 * npairs].tolist()))
    kref, vref = OBM.copy_blocks(k, v, pairs)
    dk, dv = to_dev(k), to_dev(v)
    pa.copy_blocks(dk, dv, pairs)
    np.testing.assert_array_equal(bits(dk), kref)
    np.testing.assert_array_equal(bits(dv), vref)


def test_copy_blocks_empty_and_self_pair():
    rng = np.random.default_rng(5)
    k, v = random_pool(rng, 6, 2, 64)
    dk, dv = to_dev(k), to_dev(v)
    pa.copy_blocks(dk, dv, [])
    pa.copy_blocks(dk, dv, [(3, 3)])
    np.testing.assert_array_equal(bits(dk), k)
    np.testing.assert_array_equal(bits(dv), v)


def test_copy_blocks_bad_pair_reports_bounds():
    rng = np.random.default_rng(6)
    k, v = random_pool(rng, 6, 2, 64)
    dk, dv = to_dev(k), to_dev(v)
    pa.copy_blocks(dk, dv, [(1, 2), (0, 6), (-1, 4)])
    assert pa.get_device_error() == 5
    kref, vref = OBM.copy_blocks(k, v, [(1, 2)])        # the valid pair still ran
    np.testing.assert_array_equal(bits(dk), kref)
    np.testing.assert_array_equal(bits(dv), vref)


def contiguous_attention(q, hist_k, hist_v, hkv, scale):
    """Attention of each sequence over its own token history laid out contiguously
    (block b*m + j holds tokens 16j..16j+15 of sequence b): the definition that
    copy-on-write must preserve."""
    B = len(hist_k)
    m = max(-(-len(h) // BS) for h in hist_k)
    d = q.shape[-1]
    kc = np.zeros((B * m, hkv, BS, d), dtype=np.uint16)
    vc = np.zeros_like(kc)
    tables = np.arange(B * m, dtype=np.int32).reshape(B, m)
    lens = np.array([len(h) for h in hist_k], dtype=np.int32)
    for b in range(B):
        for j, (kr, vr) in enumerate(zip(hist_k[b], hist_v[b])):
            kc[b * m + j // BS, :, j % BS] = kr
            vc[b * m + j // BS, :, j % BS] = vr
    return O.paged_attention(q, kc, vc, tables, lens, scale, hkv, BS)


@pytest.mark.parametrize("prompt,children,steps", [(37, 4, 20), (32, 3, 18), (5, 6, 40)])
def test_forked_sequences_decode_through_the_manager(prompt, children, steps):
    """Prompt prefill, fork, then decode steps where every sequence appends its own
    token: the manager's copies run on the device, new K/V go in with
    reshape_and_cache, attention reads the manager's tables.  The pool must
    equal the oracle's bit for bit and every output must match attention over the
    sequence's own history."""
    hq, hkv, d = 16, 4, 128
    scale = d ** -0.5
    rng = np.random.default_rng(prompt * 100 + children)
    nb = 64
    k_pool = np.zeros((nb, hkv, BS, d), dtype=np.uint16)
    v_pool = np.zeros_like(k_pool)
    dk, dv = to_dev(k_pool), to_dev(v_pool)
    mgr = pa.BlockManager(nb, BS)
    ref = OBM.BlockManager(nb, BS)

    seqs = [0] + list(range(1, children + 1))
    pk = W.normal_bf16(rng, (prompt, hkv, d))
    pv = W.normal_bf16(rng, (prompt, hkv, d))
    mgr.add_sequence(0, prompt)
    ref.add_sequence(0, prompt)
    table0, _ = mgr.block_table([0], -(-prompt // BS))
    slots = np.array([int(table0[0, j // BS]) * BS + j % BS for j in range(prompt)])
    k_pool, v_pool = O.reshape_and_cache(pk, pv, k_pool, v_pool, slots, BS)
    pa.reshape_and_cache(to_dev(pk), to_dev(pv), dk, dv, to_dev(slots.astype(np.int64)))
    hist_k = {0: list(pk)}
    hist_v = {0: list(pv)}
    for c in seqs[1:]:
        mgr.fork(0, c)
        ref.fork(0, c)
        hist_k[c] = list(pk)
        hist_v[c] = list(pv)

    copies_seen = 0
    for step in range(steps):
        slot_list, pairs = [], []
        for s in seqs:
            got = mgr.append_slot(s)
            assert got == ref.append_slot(s)
            slot_list.append(got[0])
            if got[1] is not None:
                pairs.append(got[1])
        copies_seen += len(pairs)
        nk = W.normal_bf16(rng, (len(seqs), hkv, d))
        nv = W.normal_bf16(rng, (len(seqs), hkv, d))
        k_pool, v_pool = OBM.copy_blocks(k_pool, v_pool, pairs)
        k_pool, v_pool = O.reshape_and_cache(nk, nv, k_pool, v_pool, np.array(slot_list), BS)
        pa.copy_blocks(dk, dv, pairs)
        pa.reshape_and_cache(to_dev(nk), to_dev(nv), dk, dv,
                             to_dev(np.array(slot_list, dtype=np.int64)))
        for i, s in enumerate(seqs):
            hist_k[s].append(nk[i])
            hist_v[s].append(nv[i])

        if step % 5 == 4 or step == steps - 1:
            np.testing.assert_array_equal(bits(dk), k_pool)
            np.testing.assert_array_equal(bits(dv), v_pool)
            L = prompt + step + 1
            mb = -(-L // BS) + 1
            tables, lens = mgr.block_table(seqs, mb)
            q = W.normal_bf16(rng, (len(seqs), 1, hq, d))
            want = contiguous_attention(q, [hist_k[s] for s in seqs],
                                        [hist_v[s] for s in seqs], hkv, scale)
            for psize in (0, 16):
                out = pa.decode(to_dev(q), dk, dv, tables.cuda(), lens.cuda(), L, scale, psize)
                assert_close(out, want, what=f"step {step} psize {psize}")
    # one copy per sequence that shared the partly filled last prompt block
    assert copies_seen == (children if prompt % BS else 0)
    mgr.close()
