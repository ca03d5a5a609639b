"""CUDA-graph runner with batch-size classes: every padded replay must give, for the
real rows, exactly the output of a direct pa_attention call with the same
partition size (bit for bit), and the fp64 oracle's within tolerance; the pool
must change only at the appended slots and in the padding block."""
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
from gpu_util import assert_close, bits, to_dev  # noqa: E402


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert pa.get_device_error() == 0, "device error word was set"


def make(T=1, n=16, seed=31):
    rng = np.random.default_rng(seed)
    lens = rng.integers(max(T, 20), 900, size=n)
    return W.build("runner", lens, num_q_heads=32, num_kv_heads=8, head_dim=128,
                   num_query_tokens=T, seed=seed)


def pad_block_of(w):
    used = set(int(x) for x in w.block_tables.ravel() if x >= 0)
    return next(b for b in range(w.num_blocks) if b not in used)


def sub(w, B):
    """The first B sequences' inputs (and their new-token rows)."""
    T = w.num_query_tokens
    return (w.q[:B], w.new_key[:B * T], w.new_value[:B * T], w.block_tables[:B],
            w.context_lens[:B], w.slot_mapping[:B * T])


@pytest.mark.parametrize("T", [1, 5])
def test_padded_replays_match_direct_calls(T):
    w = make(T)
    mcl, psize = int(w.context_lens.max()), 256
    k, v = to_dev(w.k_cache), to_dev(w.v_cache)
    pad = pad_block_of(w)
    r = pa.GraphRunner(k, v, w.num_q_heads, mcl, w.max_blocks_per_seq, pad, psize,
                       classes=(1, 2, 4, 8, 16), num_query_tokens=T, scale=w.scale)
    assert r.class_of(13) == 16 and r.class_of(16) == 16 and r.class_of(17) == -1
    for B in (1, 3, 8, 13, 16):
        q, nk, nv, tb, ln, slots = sub(w, B)
        r.q[:B].copy_(to_dev(q))
        r.new_key[:B * T].copy_(to_dev(nk))
        r.new_value[:B * T].copy_(to_dev(nv))
        r.block_tables[:B].copy_(to_dev(tb))
        r.context_lens[:B].copy_(to_dev(ln))
        r.step(B)
        got = r.out[:B].clone()
        # direct call on a fresh pool copy, same partition size and context bound
        k2, v2 = to_dev(w.k_cache), to_dev(w.v_cache)
        want = pa.attention(to_dev(q), k2, v2, to_dev(tb), to_dev(ln), mcl, w.scale, psize,
                            new_key=to_dev(nk), new_value=to_dev(nv))
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"B={B}"
        kref, vref = O.reshape_and_cache(nk, nv, w.k_cache, w.v_cache, slots, 16)
        ref = O.paged_attention(q, kref, vref, tb, ln, w.scale, w.num_kv_heads, 16)
        assert_close(got, ref, what=f"runner B={B} T={T}")
    # the runner's pool: every appended slot holds its token; only the padding block and
    # those slots differ from the initial pool
    kb = bits(k)
    s = w.slot_mapping
    np.testing.assert_array_equal(kb[s // 16, :, s % 16, :], w.new_key)
    kb[s // 16, :, s % 16, :] = w.k_cache[s // 16, :, s % 16, :]
    kb[pad] = w.k_cache[pad]
    np.testing.assert_array_equal(kb, w.k_cache)
    with pytest.raises(pa.PagedAttnError) as e:
        r.step(17)
    assert e.value.status == 2
    r.close()


def test_default_partition_per_class():
    """partition_size 0: each class is captured with the library default for its size, and
    a padded replay equals a direct call made with that class's default."""
    w = make(T=1, n=16, seed=44)
    mcl = int(w.context_lens.max())
    k, v = to_dev(w.k_cache), to_dev(w.v_cache)
    r = pa.GraphRunner(k, v, w.num_q_heads, mcl, w.max_blocks_per_seq, pad_block_of(w), 0,
                       classes=(1, 4, 16), scale=w.scale)
    for B in (1, 3, 16):
        c = r.class_of(B)
        psize = pa.default_partition_size(c, w.num_kv_heads, mcl)
        q, nk, nv, tb, ln, slots = sub(w, B)
        r.q[:B].copy_(to_dev(q))
        r.new_key[:B].copy_(to_dev(nk))
        r.new_value[:B].copy_(to_dev(nv))
        r.block_tables[:B].copy_(to_dev(tb))
        r.context_lens[:B].copy_(to_dev(ln))
        r.step(B)
        k2, v2 = to_dev(w.k_cache), to_dev(w.v_cache)
        want = pa.attention(to_dev(q), k2, v2, to_dev(tb), to_dev(ln), mcl, w.scale, psize,
                            new_key=to_dev(nk), new_value=to_dev(nv))
        assert torch.equal(r.out[:B].view(torch.int16), want.view(torch.int16)), f"B={B}"
    r.close()


def test_host_staging_copies_inside_the_graph():
    """With host staging the class graph copies the host inputs in and the output back:
    the host output rows equal a direct call, and host padding rows are rewritten."""
    w = make(T=1, n=16, seed=52)
    mcl, psize = int(w.context_lens.max()), 256
    k, v = to_dev(w.k_cache), to_dev(w.v_cache)
    pad = pad_block_of(w)
    r = pa.GraphRunner(k, v, w.num_q_heads, mcl, w.max_blocks_per_seq, pad, psize,
                       classes=(2, 8, 16), scale=w.scale, host_staging=True)
    for B in (1, 5, 16):
        q, nk, nv, tb, ln, _ = sub(w, B)
        r.h_q[:B].copy_(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16))
        r.h_new_key[:B].copy_(torch.from_numpy(nk.view(np.int16)).view(torch.bfloat16))
        r.h_new_value[:B].copy_(torch.from_numpy(nv.view(np.int16)).view(torch.bfloat16))
        r.h_block_tables[:B].copy_(torch.from_numpy(tb))
        r.h_context_lens[:B].copy_(torch.from_numpy(ln))
        r.step(B)
        torch.cuda.synchronize()
        c = r.class_of(B)
        assert (r.h_block_tables[B:c] == pad).all() and (r.h_context_lens[B:c] == 1).all()
        k2, v2 = to_dev(w.k_cache), to_dev(w.v_cache)
        want = pa.attention(to_dev(q), k2, v2, to_dev(tb), to_dev(ln), mcl, w.scale, psize,
                            new_key=to_dev(nk), new_value=to_dev(nv))
        assert torch.equal(r.h_out[:B].view(torch.int16), want.cpu().view(torch.int16)), f"B={B}"
    r.close()


def test_runner_with_window_and_fp8_pages():
    base = make(T=2, n=8, seed=5)
    w = W.fp8_variant(base, seed=2)
    mcl, psize, window = int(w.context_lens.max()), 128, 200
    k, v = to_dev(w.k_codes), to_dev(w.v_codes)
    ks, vs = to_dev(w.k_scale), to_dev(w.v_scale)
    r = pa.GraphRunner(k, v, w.num_q_heads, mcl, w.max_blocks_per_seq, pad_block_of(w), psize,
                       classes=(2, 8), num_query_tokens=2, scale=w.scale, window_size=window,
                       k_scale=ks, v_scale=vs)
    from oracle import window as WIN
    ref_all, _, _ = WIN.run_workload(w, window)
    for B in (1, 5, 8):
        q, nk, nv, tb, ln, _ = sub(w, B)
        r.q[:B].copy_(to_dev(q))
        r.new_key[:B * 2].copy_(to_dev(nk))
        r.new_value[:B * 2].copy_(to_dev(nv))
        r.block_tables[:B].copy_(to_dev(tb))
        r.context_lens[:B].copy_(to_dev(ln))
        r.step(B)
        assert_close(r.out[:B], ref_all[:B], what=f"fp8 window runner B={B}")
    r.close()


def test_bad_configuration_rejected():
    w = make(n=2)
    k, v = to_dev(w.k_cache), to_dev(w.v_cache)
    with pytest.raises(pa.PagedAttnError):
        pa.GraphRunner(k, v, 32, 900, w.max_blocks_per_seq, 0, -16)      # partition_size < 0
    with pytest.raises(pa.PagedAttnError):
        pa.GraphRunner(k, v, 32, 900, w.max_blocks_per_seq, w.num_blocks, 256)  # pad block
