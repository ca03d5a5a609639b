"""The tcgen05 (tensor-memory) attention kernel: multi-query tiles of 17-32 query
rows per kv head at head_dim 128 (speculative verify), against the fp64 oracle.

Shapes are chosen around the kernel's structure: groups of 8 pages (128 tokens)
per score MMA, so context lengths and partition sizes leave partial groups and
ragged last pages; row counts 17, 18, 20, 24 and 32 (the MMA's N is 32); the
fused append; sliding windows; a block id outside the pool.  Tolerance: bf16
output max abs error <= 1e-2 (or one bf16 ulp of the oracle value, where that is
larger), relative L2 error <= 2e-3.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from oracle import window as WIN

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU-only hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402
from gpu_util import Dev, assert_close, bits  # noqa: E402

LENS = [17, 100, 127, 128, 129, 255, 256, 257, 1000, 1023, 1024, 1025, 2047, 2049, 3000]


@pytest.fixture(autouse=True)
def tcgen05_kernel(monkeypatch):
    """Route 17-32-row tiles to the tcgen05 kernel for every test of this file."""
    monkeypatch.setenv("PA_VERIFY_KERNEL", "tcgen05")
    yield
    assert pa.get_device_error() == 0, "device error word was set"


@pytest.mark.parametrize("hq,hkv,T", [(32, 8, 5), (64, 8, 4), (16, 8, 9), (24, 8, 6), (8, 1, 3),
                                      (16, 1, 2), (32, 2, 2)])
def test_row_counts_and_lengths(hq, hkv, T):
    w = W.build("tc_rows", [max(L, T) for L in LENS], num_q_heads=hq, num_kv_heads=hkv,
                head_dim=128, num_query_tokens=T, seed=hq * 7 + T)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    for ps in (16, 48, 128, 272, 0):
        assert_close(d.attend(partition_size=ps), ref, what=f"{hq}/{hkv} T{T} ps{ps}")


@pytest.mark.parametrize("ps", [0, 128, 400])
def test_fused_append(ps):
    w = W.build("tc_append", LENS, num_q_heads=32, num_kv_heads=8, head_dim=128,
                num_query_tokens=5, seed=11)
    ref, kref, vref = O.run_workload(w)
    d = Dev(w)
    out = d.attend_append(partition_size=ps)
    assert_close(out, ref, what=f"append ps{ps}")
    np.testing.assert_array_equal(bits(d.k), kref)
    np.testing.assert_array_equal(bits(d.v), vref)


@pytest.mark.parametrize("window", [1, 16, 17, 130, 700])
def test_windows(window):
    w = W.build("tc_win", LENS, num_q_heads=32, num_kv_heads=8, head_dim=128,
                num_query_tokens=5, seed=13)
    ref, _, _ = WIN.run_workload(w, window)
    d = Dev(w)
    for ps in (0, 64):
        out = pa.attention(d.q, d.k, d.v, d.tables, d.lens, w.max_context_len, w.scale, ps,
                           None, None, d.new_key, d.new_value, window_size=window)
        assert_close(out, ref, what=f"window {window} ps{ps}")


def test_constant_v_is_exactly_one():
    """V = 1 everywhere: the softmax-weighted sum is exactly 1 (P's two bf16 parts
    sum to P, and the row sum divides it out)."""
    w = W.build("tc_ones", LENS, num_q_heads=32, num_kv_heads=8, head_dim=128,
                num_query_tokens=5, seed=17)
    one = np.uint16(0x3F80)
    w.v_cache = np.where(w.v_cache == W.NAN_BITS, w.v_cache, one).astype(np.uint16)
    w.new_value = np.full_like(w.new_value, one)
    d = Dev(w)
    d.reshape()
    for ps in (0, 64):
        out = d.attend(partition_size=ps).float().cpu().numpy()
        np.testing.assert_allclose(out, 1.0, rtol=0, atol=2e-3)


def test_peaked_scores_move_the_reference_max():
    """Queries scaled x40 and keys growing along the context: the reference max of
    each row moves many times, so O is rescaled in tensor memory repeatedly."""
    w = W.build("tc_peak", LENS, num_q_heads=32, num_kv_heads=8, head_dim=128,
                num_query_tokens=5, seed=19)
    q = (w.q.astype(np.uint32) << 16).view(np.float32) * 40.0
    w.q = W.f32_to_bf16_bits(q)
    k = (w.k_cache.astype(np.uint32) << 16).view(np.float32).copy()
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        for j in range(L - w.num_query_tokens):
            blk, off = w.block_tables[b, j // 16], j % 16
            k[blk, :, off, :] *= 1.0 + 3.0 * j / L
    finite = np.isfinite(k)
    w.k_cache = np.where(finite, W.f32_to_bf16_bits(np.where(finite, k, 0.0)),
                         w.k_cache).astype(np.uint16)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    for ps in (0, 256):
        assert_close(d.attend(partition_size=ps), ref, what=f"peaked ps{ps}")


def test_bad_block_id_reports_bounds_and_others_unaffected():
    w = W.build("tc_bad", [300, 500, 700], num_q_heads=32, num_kv_heads=8, head_dim=128,
                num_query_tokens=5, seed=23)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    d.tables[1, 3] = w.num_blocks + 5
    out = d.attend(partition_size=0)
    assert pa.get_device_error() == 5          # PA_ERR_BOUNDS
    assert_close(out[[0, 2]], ref[[0, 2]], what="unaffected sequences")


def test_deterministic():
    w = W.SMALL["spec_verify"]()
    d = Dev(w)
    d.reshape()
    a = d.attend(partition_size=0).clone()
    b = d.attend(partition_size=0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_the_tcgen05_kernel_is_the_one_that_runs():
    """With PA_VERIFY_KERNEL=tcgen05 the verify tiles run on the tcgen05 kernel (not on
    the persistent or the one-CTA-per-unit mma.sync kernel)."""
    w = W.build("tc_which", LENS, num_q_heads=32, num_kv_heads=8, head_dim=128,
                num_query_tokens=5, seed=17)
    d = Dev(w)
    d.reshape()
    d.attend(partition_size=0)
    assert pa.last_attention_kernel() == "tcgen05"
