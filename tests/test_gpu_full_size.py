"""Full-size parity: every sequence of every workload, bf16 and FP8 pages.

Each workload runs at full size in the launch configuration the benchmark
times (the fused append call for per-sequence workloads; reshape_and_cache,
then the shared-prefix call, for the shared-prefix workload), and every output
row of every sequence is compared with the fp64 oracle (bf16 output: max abs
error <= 1e-2 or one bf16 ulp of the oracle value, whichever is larger; relative
L2 error <= 2e-3).  The appended slots are compared
bit for bit (bf16) or code for code (FP8).
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import fp8 as F
from oracle import oracle as O
from oracle_threads import all_rows

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU-only hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402
from gpu_util import MAX_REL_L2, Dev, abs_bound, bits, errors, to_dev  # noqa: E402

NAMES = ["tiny", "decode_8b", "decode_70b", "spec_verify", "shared_prefix"]


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert pa.get_device_error() == 0, "device error word was set"


def check_every_row(out, ref, what):
    """The per-element abs bound over every element of every row, relative L2 over the whole
    output."""
    mx, rel, g = errors(out, ref)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    over = (np.abs(g - ref) - abs_bound(ref)).reshape(g.shape[0], -1).max(axis=1)
    worst = int(np.argmax(over))
    assert over.max() <= 0, f"{what}: max abs {mx:.3e}, bound exceeded in sequence {worst}"
    assert rel <= MAX_REL_L2, f"{what}: rel L2 {rel:.3e}"


@pytest.mark.parametrize("name", NAMES)
def test_full_size_every_sequence_bf16(name):
    w = W.FULL[name]()
    d = Dev(w)
    if w.seq_group is None:
        out = d.attend_append()
    else:
        d.reshape()
        out = d.attend()
    torch.cuda.synchronize()
    k, v = O.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping, 16)
    ref = all_rows(O.paged_attention, w.num_seqs, w.q, k, v, w.block_tables, w.context_lens,
                   w.scale, w.num_kv_heads, 16)
    check_every_row(out, ref, f"{name} full")
    s = w.slot_mapping
    np.testing.assert_array_equal(bits(d.k)[s // 16, :, s % 16, :], w.new_key)
    np.testing.assert_array_equal(bits(d.v)[s // 16, :, s % 16, :], w.new_value)


@pytest.mark.parametrize("name", NAMES)
def test_full_size_every_sequence_fp8(name):
    w = W.fp8_variant(W.FULL[name](), seed=0)
    q, kc, vc = to_dev(w.q), to_dev(w.k_codes), to_dev(w.v_codes)
    ks, vs = to_dev(w.k_scale), to_dev(w.v_scale)
    tables, lens = to_dev(w.block_tables), to_dev(w.context_lens)
    nk, nv, slots = to_dev(w.new_key), to_dev(w.new_value), to_dev(w.slot_mapping)
    if w.seq_group is None:
        out = pa.verify_fp8(q, kc, vc, ks, vs, tables, lens, w.max_context_len, w.scale,
                            w.partition_size, None, None, nk, nv)
    else:
        pa.reshape_and_cache_fp8(nk, nv, kc, vc, slots, ks, vs)
        need = pa.workspace_size(w.num_seqs, w.num_q_heads, 1, w.max_context_len, w.head_dim,
                                 16, w.partition_size, w.max_prefix_blocks)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        out = pa.decode_shared_prefix(q, kc, vc, tables, lens, to_dev(w.seq_group),
                                      to_dev(w.group_prefix_blocks), w.max_group_size,
                                      w.max_prefix_blocks, w.max_context_len, w.scale,
                                      w.partition_size, ws, None, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    k, v = F.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                               w.k_scale, w.v_scale, 16)
    ref = all_rows(F.paged_attention, w.num_seqs, w.q, k, v, w.k_scale, w.v_scale,
                   w.block_tables, w.context_lens, w.scale, w.num_kv_heads, 16)
    check_every_row(out, ref, f"{name} fp8 full")
    s = w.slot_mapping
    kd, vd = kc.cpu().numpy(), vc.cpu().numpy()
    np.testing.assert_array_equal(kd[s // 16, :, s % 16, :], k[s // 16, :, s % 16, :])
    np.testing.assert_array_equal(vd[s // 16, :, :, s % 16], v[s // 16, :, :, s % 16])
