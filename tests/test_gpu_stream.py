"""The persistent attention kernel (at most 8 query rows per kv head, or 17-24 for
speculative verify) against the one-CTA-per-unit kernel and the fp64 oracle.

The persistent kernel runs a different schedule (a dense largest-first unit
list, units claimed from a counter or taken in a fixed order, pages streamed across unit
boundaries) but each unit's arithmetic is that of the one-CTA-per-unit kernel:
page lane q takes the unit's pages q, q + PL, ... and the lanes merge in the same
order.  So its output must be bit-identical to the one-CTA-per-unit kernel's
(PA_DECODE_KERNEL=persistent and =per_unit select them; unset, the library
chooses), and within the bf16 tolerance of the
oracle (max abs error <= 1e-2 or one bf16 ulp of the oracle value, whichever is
larger; relative L2 error <= 2e-3).

Cases cover the schedule's edges: ragged lengths around partition boundaries,
many partitions per sequence and single-partition sequences in one batch, one
sequence, partition sizes whose split needs scratch (units claimed from the
counter) and ones that need none (a fixed order), GQA ratios 1, 4 and 8 and two
query tokens, verify tiles of 18, 20 and 24 rows (three row columns and a merge
buffer), head_dim 64 and 128, FP8 pages, the fused append, sliding windows,
the 256-sequence limit of the in-CTA unit list and one sequence more (the
one-CTA-per-unit kernel then runs), and the full 8B-, 70B-shape and verify
batches.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import fp8 as F
from oracle import oracle as O
from oracle import window as WIN

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU-only hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402
from gpu_util import Dev, assert_close, bits, to_dev  # noqa: E402

LENS = [1, 15, 16, 17, 100, 255, 256, 257, 700, 1023, 1024, 1025, 2047, 2048, 2049, 3000, 5000]


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert pa.get_device_error() == 0, "device error word was set"


def both(monkeypatch, run):
    """run() with the persistent kernel and with the one-CTA-per-unit kernel; the two
    outputs must be bit-identical.  Returns the persistent kernel's output."""
    monkeypatch.setenv("PA_DECODE_KERNEL", "persistent")
    a = run()
    torch.cuda.synchronize()
    monkeypatch.setenv("PA_DECODE_KERNEL", "per_unit")
    b = run()
    torch.cuda.synchronize()
    monkeypatch.delenv("PA_DECODE_KERNEL")
    np.testing.assert_array_equal(bits(a), bits(b))
    return a


@pytest.mark.parametrize("hq,hkv,T,D", [(32, 8, 1, 128), (64, 8, 1, 128), (8, 8, 1, 128),
                                        (16, 8, 2, 128), (32, 8, 1, 64), (16, 2, 1, 64),
                                        (32, 8, 5, 128), (16, 8, 9, 128), (64, 8, 3, 128),
                                        (24, 8, 6, 64)])
def test_lengths_and_partitions(monkeypatch, hq, hkv, T, D):
    w = W.build("stream_lens", [max(L, T) for L in LENS], num_q_heads=hq, num_kv_heads=hkv,
                head_dim=D, num_query_tokens=T, seed=hq + 3 * T + D)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    for ps in (16, 48, 128, 1536, 0, 8192):
        out = both(monkeypatch, lambda: d.attend(partition_size=ps))
        assert_close(out, ref, what=f"{hq}/{hkv} T{T} D{D} ps{ps}")


def test_one_sequence(monkeypatch):
    w = W.build("stream_one", [4097], num_q_heads=32, num_kv_heads=8, head_dim=128, seed=5)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    for ps in (16, 256, 0):
        assert_close(both(monkeypatch, lambda: d.attend(partition_size=ps)), ref,
                     what=f"one sequence ps{ps}")


@pytest.mark.parametrize("ps,T", [(0, 1), (64, 1), (272, 1), (0, 5), (96, 5)])
def test_fused_append(monkeypatch, ps, T):
    w = W.build("stream_append", [max(L, T) for L in LENS], num_q_heads=32, num_kv_heads=8,
                head_dim=128, num_query_tokens=T, seed=9 + T)
    ref, kref, vref = O.run_workload(w)
    outs = []
    for mode in ("persistent", "per_unit"):
        monkeypatch.setenv("PA_DECODE_KERNEL", mode)
        d = Dev(w)                           # fresh pools: the append writes them
        outs.append(bits(d.attend_append(partition_size=ps)))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits(d.k), kref)
        np.testing.assert_array_equal(bits(d.v), vref)
    monkeypatch.delenv("PA_DECODE_KERNEL")
    np.testing.assert_array_equal(outs[0], outs[1])
    out = torch.from_numpy(outs[0].view(np.int16)).view(torch.bfloat16)
    assert_close(out, ref, what=f"append ps{ps}")


@pytest.mark.parametrize("ps,T", [(0, 1), (96, 1), (0, 5), (160, 5)])
def test_fp8_pages(monkeypatch, ps, T):
    w = W.fp8_variant(W.build("stream_fp8", [max(L, T) for L in LENS], num_q_heads=32,
                              num_kv_heads=8, head_dim=128, num_query_tokens=T, seed=21 + T),
                      seed=2)
    k, v = F.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                               w.k_scale, w.v_scale, 16)
    ref = F.paged_attention(w.q, k, v, w.k_scale, w.v_scale, w.block_tables, w.context_lens,
                            w.scale, w.num_kv_heads, 16)
    q, kc, vc = to_dev(w.q), to_dev(k), to_dev(v)
    ks, vs = to_dev(w.k_scale), to_dev(w.v_scale)
    tables, lens = to_dev(w.block_tables), to_dev(w.context_lens)
    out = both(monkeypatch, lambda: pa.verify_fp8(q, kc, vc, ks, vs, tables, lens,
                                                  w.max_context_len, w.scale, ps))
    assert_close(out, ref, what=f"fp8 ps{ps}")


@pytest.mark.parametrize("window,T", [(1, 1), (16, 1), (17, 1), (600, 1), (3, 5), (700, 5)])
def test_windows(monkeypatch, window, T):
    w = W.build("stream_win", [max(L, T) for L in LENS], num_q_heads=32, num_kv_heads=8,
                head_dim=128, num_query_tokens=T, seed=31 + T)
    ref, _, _ = WIN.run_workload(w, window)
    d = Dev(w)
    for ps in (0, 64):
        def run():
            return pa.attention(d.q, d.k, d.v, d.tables, d.lens, w.max_context_len, w.scale, ps,
                                None, None, d.new_key, d.new_value, window_size=window)
        # the fused append rewrites the same values on every call
        assert_close(both(monkeypatch, run), ref, what=f"window {window} ps{ps}")


@pytest.mark.parametrize("B", [256, 257])
def test_unit_list_limit(monkeypatch, B):
    rng = np.random.default_rng(B)
    lens = rng.integers(1, 3000, size=B)
    w = W.build("stream_many", lens, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=B)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    for ps in (256, 0):
        assert_close(both(monkeypatch, lambda: d.attend(partition_size=ps)), ref,
                     what=f"{B} sequences ps{ps}")


@pytest.mark.parametrize("name", ["decode_8b", "decode_70b", "spec_verify"])
def test_full_size_bit_identical(monkeypatch, name):
    """The benchmark's batches in its launch configuration (fused append, default
    partitions), bf16 and FP8 pages; the oracle comparison of every row of these
    is in the full-size parity tests."""
    w = W.FULL[name]()
    outs = []
    for mode in ("persistent", "per_unit"):
        monkeypatch.setenv("PA_DECODE_KERNEL", mode)
        outs.append(bits(Dev(w).attend_append()))
    np.testing.assert_array_equal(outs[0], outs[1])
    w8 = W.fp8_variant(w, seed=0)
    outs = []
    for mode in ("persistent", "per_unit"):
        monkeypatch.setenv("PA_DECODE_KERNEL", mode)
        q, kc, vc = to_dev(w8.q), to_dev(w8.k_codes), to_dev(w8.v_codes)
        out = pa.verify_fp8(q, kc, vc, to_dev(w8.k_scale), to_dev(w8.v_scale),
                            to_dev(w8.block_tables), to_dev(w8.context_lens),
                            w8.max_context_len, w8.scale, w8.partition_size, None, None,
                            to_dev(w8.new_key), to_dev(w8.new_value))
        outs.append(bits(out))
    monkeypatch.delenv("PA_DECODE_KERNEL")
    np.testing.assert_array_equal(outs[0], outs[1])


@pytest.mark.parametrize("fill", [0x00, 0xFF])
def test_claim_modes_on_one_scratch(monkeypatch, fill):
    """The first launch on a scratch takes units in a fixed order and leaves the claim
    counter ready (the split-KV merge resets it); the launches after it claim units from
    the counter.  Every launch gives the same bits as the one-CTA-per-unit kernel."""
    rng = np.random.default_rng(fill + 3)
    w = W.build("stream_claim", rng.integers(1, 4000, size=96), num_q_heads=32,
                num_kv_heads=8, head_dim=128, seed=fill + 3)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    ps = 512
    need = pa.workspace_size(w.num_seqs, w.num_q_heads, 1, w.max_context_len, w.head_dim, 16,
                             ps, 0)
    monkeypatch.setenv("PA_DECODE_KERNEL", "per_unit")
    want = bits(d.attend(partition_size=ps))
    monkeypatch.setenv("PA_DECODE_KERNEL", "persistent")
    ws = torch.full((max(need, 256),), fill, dtype=torch.uint8, device="cuda")
    for i in range(4):
        out = d.attend(partition_size=ps, workspace=ws)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits(out), want, err_msg=f"launch {i}")
    monkeypatch.delenv("PA_DECODE_KERNEL")
    assert_close(out, ref, what="claim modes")


@pytest.mark.parametrize("bad", [0, 9])
def test_context_above_bound_reports_bounds(monkeypatch, bad):
    """A context above max_context_len: the persistent kernel sets the bounds bit, writes
    nothing for that sequence and gives every other sequence its result.  Sequence 0's
    first partitions open CTAs (their first record is then empty); sequence 9's come from
    the unit list."""
    monkeypatch.setenv("PA_DECODE_KERNEL", "persistent")
    w = W.build("stream_bad", LENS, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=41)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    lens = w.context_lens.copy()
    lens[bad] = w.max_context_len + 16
    d.lens = to_dev(lens)
    keep = [b for b in range(w.num_seqs) if b != bad]
    for ps in (64, 0):
        out = torch.full_like(d.q, float("nan"))
        pa.verify(d.q, d.k, d.v, d.tables, d.lens, w.max_context_len, w.scale, ps, None, out)
        torch.cuda.synchronize()
        assert pa.get_device_error() == 5
        assert torch.isnan(out[bad].float()).all()
        assert_close(out, ref, seqs=keep, what=f"bad length in sequence {bad}, ps{ps}")
    monkeypatch.delenv("PA_DECODE_KERNEL")


@pytest.mark.parametrize("T,kv,mode,ps,want", [(1, "bf16", None, 2048, "per_unit"),
                                                (1, "bf16", None, 256, "persistent"),
                                                (1, "fp8", None, 2048, "persistent"),
                                                (5, "bf16", None, 256, "persistent"),
                                                (5, "bf16", None, 2048, "per_unit"),
                                                (1, "bf16", "persistent", 2048, "persistent"),
                                                (5, "fp8", "per_unit", 256, "per_unit"),
                                                (2, "bf16", "persistent", 256, "per_unit")])
def test_kernel_choice(monkeypatch, T, kv, mode, ps, want):
    """Which kernel a call runs (pa_last_attention_kernel): the library's choice and
    PA_DECODE_KERNEL's override.  The library takes the persistent kernel for FP8 pages,
    and for bf16 pages when the launch has at least 4 units (bound) per resident CTA: with
    17 sequences up to 5000 tokens that is 2720 units at 256-token partitions, 408 at
    2048-token ones, against 456 resident CTAs for 4 rows (304 for 20).  Ten rows per kv
    head (T = 2, G = 5) are not served by the persistent kernel."""
    if mode is None:
        monkeypatch.delenv("PA_DECODE_KERNEL", raising=False)
    else:
        monkeypatch.setenv("PA_DECODE_KERNEL", mode)
    hq = 40 if T == 2 else 32
    w = W.build("stream_which", [max(L, T) for L in LENS], num_q_heads=hq, num_kv_heads=8,
                head_dim=128, num_query_tokens=T, seed=51)
    if kv == "fp8":
        w = W.fp8_variant(w, seed=1)
        q, kc, vc = to_dev(w.q), to_dev(w.k_codes), to_dev(w.v_codes)
        pa.verify_fp8(q, kc, vc, to_dev(w.k_scale), to_dev(w.v_scale), to_dev(w.block_tables),
                      to_dev(w.context_lens), w.max_context_len, w.scale, ps)
    else:
        d = Dev(w)
        d.reshape()
        d.attend(partition_size=ps)
    torch.cuda.synchronize()
    monkeypatch.delenv("PA_DECODE_KERNEL", raising=False)
    assert pa.last_attention_kernel() == want
