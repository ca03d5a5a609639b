"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerance for every attention output (bf16) against the fp64 oracle: max abs
error <= 1e-2 (or one bf16 ulp of the oracle value, where that is larger) and
relative L2 error <= 2e-3.  reshape_and_cache is compared
bit for bit over the whole pool.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU-only hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402
from gpu_util import Dev, assert_close, bits, errors, to_dev  # noqa: E402


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert pa.get_device_error() == 0, "device error word was set"


# ----------------------------------------------------------------------------- small configs

SMALL_NAMES = sorted(W.SMALL)


@pytest.mark.parametrize("name", SMALL_NAMES)
def test_small_config_matches_oracle(name):
    w = W.SMALL[name]()
    ref, kref, vref = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    np.testing.assert_array_equal(bits(d.k), kref)
    np.testing.assert_array_equal(bits(d.v), vref)
    out = d.attend()
    assert_close(out, ref, what=name)


@pytest.mark.parametrize("name", ["decode_8b", "spec_verify", "decode_70b", "shared_prefix"])
@pytest.mark.parametrize("psize", [16, 48, 128, 512, 0])
def test_partition_sizes(name, psize):
    """Split-KV with many partition sizes (ragged last partitions, empty ones) stays in tolerance."""
    w = W.SMALL[name]()
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    assert_close(d.attend(partition_size=psize), ref, what=f"{name} psize {psize}")


@pytest.mark.parametrize("lens", [[368, 384, 400, 411, 496], [767, 768, 784, 785, 960]])
def test_merge_partition_counts(lens):
    """Split-KV merge at the boundary of its two load schedules.  With one-block
    partitions, at most 31 partitions (first case) give 2 merging warps per row and
    more give 4 (second case); a warp holding up to 12 partitions issues all their
    loads at once, one holding 13 or more loops over them (23/24 partitions: 12 per
    warp; 25/26: 13; 48: 12 per warp of 4; 49/50: 13 on the first)."""
    w = W.build("merge_edge", lens, num_q_heads=32, num_kv_heads=8, head_dim=128,
                seed=sum(lens) % 997)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    assert_close(d.attend(partition_size=16), ref, what=f"merge {lens}")
    # the same rows through the fused append call
    d2 = Dev(w)
    assert_close(d2.attend_append(partition_size=16), ref, what=f"merge append {lens}")


def test_unsplit_without_workspace():
    """partition_size 0 and no workspace: every sequence in one CTA per kv head."""
    w = W.SMALL["decode_8b"]()
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    lib = pa.library()
    out = torch.empty_like(d.q)
    import ctypes
    vp = ctypes.c_void_p
    st = lib.pa_decode(vp(out.data_ptr()), vp(d.q.data_ptr()), vp(d.k.data_ptr()),
                       vp(d.v.data_ptr()), vp(d.tables.data_ptr()), w.max_blocks_per_seq,
                       vp(d.lens.data_ptr()), w.max_context_len, w.num_seqs, w.num_blocks,
                       w.num_q_heads, w.num_kv_heads, w.head_dim, 16, w.scale, 0, None, 0,
                       vp(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    assert_close(out, ref, what="unsplit")


# ----------------------------------------------------------------------------- edge cases

EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 511, 512, 513]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("hq,hkv,T", [(4, 4, 1), (32, 8, 1), (64, 8, 1), (32, 8, 5), (16, 1, 4),
                                      (8, 2, 3)])
def test_edge_lengths_and_head_layouts(D, hq, hkv, T):
    lens = [max(L, T) for L in EDGE_LENS]
    w = W.build("edge", lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=D, num_query_tokens=T,
                seed=D + hq + T)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    for ps in (16, 64, 0):
        assert_close(d.attend(partition_size=ps), ref, what=f"D{D} {hq}/{hkv} T{T} ps{ps}")


def test_all_positions_are_drafts():
    """Verify with context_len == T: draft t sees drafts 0..t only."""
    w = W.build("drafts_only", [4, 4, 9], num_q_heads=8, num_kv_heads=2, head_dim=128,
                num_query_tokens=4, seed=3)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    assert_close(d.attend(), ref, what="drafts only")


def test_empty_batch():
    w = W.tiny()
    d = Dev(w)
    q = d.q[:0]
    out = pa.verify(q, d.k, d.v, d.tables[:0], d.lens[:0], max_context_len=16, scale=0.125)
    assert out.shape[0] == 0


def test_length_one_is_v0_bit_exact():
    w = W.build("L1", [1, 1, 1], num_q_heads=8, num_kv_heads=2, head_dim=128, seed=9)
    d = Dev(w)
    d.reshape()
    out = d.attend()
    G = 4
    for b in range(3):
        blk = w.block_tables[b, 0]
        for h in range(8):
            v0 = w.new_value[b, h // G]
            np.testing.assert_array_equal(bits(out[b, 0, h]), v0)


def test_constant_v_gives_exactly_one():
    """Softmax weights sum to one: with V = 1 everywhere the bf16 output is exactly 1.0."""
    w = W.SMALL["spec_verify"]()
    d = Dev(w)
    d.reshape()
    one = torch.ones(1, dtype=torch.bfloat16, device="cuda")
    nblk = -(-w.context_lens // 16)
    for b in range(w.num_seqs):
        ids = torch.as_tensor(w.block_tables[b, :nblk[b]].astype(np.int64), device="cuda")
        d.v[ids] = one                         # tail slots too: all finite
    out = d.attend(partition_size=64)
    assert bool((out == 1.0).all())


def test_permutation_invariance_bit_identical():
    """Moving blocks to other physical ids changes no output bit."""
    w = W.SMALL["decode_70b"]()
    d = Dev(w)
    d.reshape()
    a = d.attend(partition_size=64).clone()
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(0)).cuda()
    k2 = torch.empty_like(d.k)
    v2 = torch.empty_like(d.v)
    k2[perm] = d.k
    v2[perm] = d.v
    t = d.tables.long()
    t2 = torch.where(t >= 0, perm[t.clamp(min=0)], t).int()
    b = pa.verify(d.q, k2, v2, t2, d.lens, w.max_context_len, w.scale, 64)
    assert torch.equal(bits_t(a), bits_t(b))


def bits_t(t):
    return t.view(torch.int16)


def test_shared_prefix_equals_plain_decode():
    """The read-once shared-prefix path agrees with plain decode on the same tables."""
    w = W.SMALL["shared_prefix"]()
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    shared = d.attend(shared=True)
    plain = d.attend(shared=False)
    assert_close(shared, ref, what="shared")
    assert_close(plain, ref, what="plain")
    mx, rel, _ = errors(shared, plain.float().cpu().double().numpy())
    assert mx <= 1e-2 and rel <= 2e-3


def test_shared_prefix_many_member_chunks():
    """Groups larger than one CTA's rows are split into member chunks."""
    B = 20
    shared = [(list(range(0, 11)), 5), (list(range(11, 20)), 3)]
    lens = [5 * 16 + 7 * i + 1 for i in range(11)] + [3 * 16 + 11 * i for i in range(9)]
    w = W.build("chunks", lens, num_q_heads=32, num_kv_heads=4, head_dim=128, seed=5,
                shared=shared, partition_size=32)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    assert_close(d.attend(shared=True), ref, what="chunks")


def test_repeated_calls_are_deterministic():
    w = W.SMALL["decode_8b"]()
    d = Dev(w)
    d.reshape()
    a = d.attend(partition_size=128).clone()
    b = d.attend(partition_size=128).clone()
    assert torch.equal(bits_t(a), bits_t(b))


def test_non_default_stream():
    w = W.SMALL["spec_verify"]()
    ref, _, _ = O.run_workload(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = Dev(w)
        d.reshape()
        out = d.attend()
    s.synchronize()
    assert_close(out, ref, what="side stream")


def test_reshape_padding_slots_skipped():
    w = W.SMALL["decode_70b"]()
    d = Dev(w)
    slots = w.slot_mapping.copy()
    slots[::2] = -1
    d.slots = to_dev(slots)
    d.reshape()
    kref, vref = O.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, slots, 16)
    np.testing.assert_array_equal(bits(d.k), kref)
    np.testing.assert_array_equal(bits(d.v), vref)


# ----------------------------------------------------------------------------- errors

def test_workspace_too_small():
    w = W.SMALL["decode_8b"]()
    d = Dev(w)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        d.attend(partition_size=16, workspace=ws)
    assert e.value.status == 3


def test_bad_block_id_reports_bounds():
    w = W.SMALL["decode_8b"]()
    d = Dev(w)
    d.reshape()
    d.tables[1, 2] = w.num_blocks + 7
    d.tables[2, 0] = -3
    d.attend(partition_size=64)
    assert pa.get_device_error() == 5


def test_bad_slot_reports_bounds():
    w = W.SMALL["decode_8b"]()
    d = Dev(w)
    slots = w.slot_mapping.copy()
    slots[0] = w.num_blocks * 16 + 3
    d.slots = to_dev(slots)
    d.reshape()
    assert pa.get_device_error() == 5


def test_context_above_bound_reports_bounds():
    w = W.SMALL["decode_8b"]()
    d = Dev(w)
    d.reshape()
    pa.verify(d.q, d.k, d.v, d.tables, d.lens, w.max_context_len - 1, w.scale, 64)
    assert pa.get_device_error() == 5


def test_wait_timeout_self_test():
    """A bounded wait on a barrier nothing signals gives up and reports a timeout."""
    pa.selftest_wait_timeout(2_000_000)      # 2 ms
    assert pa.get_device_error() == 6
    # the context is still healthy
    w = W.tiny()
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    assert_close(d.attend(), ref, what="after timeout")


# ----------------------------------------------------------------------------- softmax range

def _f32(bits_u16):
    return (bits_u16.astype(np.uint32) << np.uint32(16)).view(np.float32)


def test_peaked_scores_rescale_many_times():
    """Queries scaled x40: scores span ~100 (log2 units), the running max jumps often."""
    w = W.SMALL["spec_verify"]()
    w.q = W.f32_to_bf16_bits(_f32(w.q) * 40.0)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    for ps in (64, 0):
        assert_close(d.attend(partition_size=ps), ref, what=f"peaked ps{ps}")


def test_scores_growing_along_the_context():
    """K rows scaled up with their position: the max rises page after page."""
    w = W.SMALL["decode_70b"]()
    k = _f32(w.k_cache).copy()
    nk = _f32(w.new_key).copy()
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        for j in range(L):
            f = 1.0 + 6.0 * j / L
            blk, off = w.block_tables[b, j // 16], j % 16
            if j >= L - w.num_query_tokens:
                nk[b * w.num_query_tokens + (j - (L - w.num_query_tokens))] *= f
            else:
                k[blk, :, off, :] *= f
    finite = np.isfinite(k)
    kb = W.f32_to_bf16_bits(np.where(finite, k, 0.0))
    w.k_cache = np.where(finite, kb, w.k_cache)
    w.new_key = W.f32_to_bf16_bits(nk)
    ref, _, _ = O.run_workload(w)
    d = Dev(w)
    d.reshape()
    for ps in (32, 0):
        assert_close(d.attend(partition_size=ps), ref, what=f"growing ps{ps}")


# ----------------------------------------------------------------------------- fused append

@pytest.mark.parametrize("name", ["tiny", "decode_8b", "decode_70b", "spec_verify"])
@pytest.mark.parametrize("psize", [32, 0])
def test_append_equals_reshape_then_attend(name, psize):
    """pa_decode_append writes the same pool bits and the same output bits as
    pa_reshape_and_cache followed by the attention call, and matches the oracle."""
    w = W.SMALL[name]()
    ref, kref, vref = O.run_workload(w)
    a = Dev(w)
    out_a = a.attend_append(partition_size=psize).clone()
    np.testing.assert_array_equal(bits(a.k), kref)
    np.testing.assert_array_equal(bits(a.v), vref)
    b = Dev(w)
    b.reshape()
    out_b = b.attend(partition_size=psize)
    assert torch.equal(bits_t(out_a), bits_t(out_b))
    assert_close(out_a, ref, what=f"append {name}")


def test_append_edge_lengths():
    lens = [max(L, 3) for L in EDGE_LENS]
    w = W.build("edge_append", lens, num_q_heads=16, num_kv_heads=4, head_dim=128,
                num_query_tokens=3, seed=77)
    ref, kref, _ = O.run_workload(w)
    d = Dev(w)
    for ps in (16, 0):
        out = d.attend_append(partition_size=ps)
        assert_close(out, ref, what=f"append edge ps{ps}")
    np.testing.assert_array_equal(bits(d.k), kref)
