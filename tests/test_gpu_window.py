"""Sliding-window attention on the GPU (pa_attention through the C ABI) against the
fp64 window oracle: bf16 and FP8 pages, separate and fused append, split and
unsplit.  Tolerance as elsewhere: max abs error <= 1e-2, relative L2 <= 2e-3.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import window as WIN
from oracle_threads import all_rows

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU-only hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402
from gpu_util import Dev, assert_close, bits, to_dev  # noqa: E402


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert pa.get_device_error() == 0, "device error word was set"


def attend(d, window, psize, fused):
    w = d.w
    nk = d.new_key if fused else None
    nv = d.new_value if fused else None
    if not fused:
        d.reshape()
    return pa.attention(d.q, d.k, d.v, d.tables, d.lens, w.max_context_len, w.scale, psize,
                        new_key=nk, new_value=nv, window_size=window)


class Dev8(Dev):
    def __init__(self, w):
        self.w = w
        self.q = to_dev(w.q)
        self.k = to_dev(w.k_codes)
        self.v = to_dev(w.v_codes)
        self.ks, self.vs = to_dev(w.k_scale), to_dev(w.v_scale)
        self.tables, self.lens = to_dev(w.block_tables), to_dev(w.context_lens)
        self.new_key, self.new_value = to_dev(w.new_key), to_dev(w.new_value)
        self.slots = to_dev(w.slot_mapping)


def attend8(d, window, psize):
    w = d.w
    return pa.attention(d.q, d.k, d.v, d.tables, d.lens, w.max_context_len, w.scale, psize,
                        new_key=d.new_key, new_value=d.new_value, window_size=window,
                        k_scale=d.ks, v_scale=d.vs)


@pytest.mark.parametrize("name", ["decode_8b", "spec_verify", "decode_70b"])
@pytest.mark.parametrize("window", [1, 16, 17, 100, 1000])
def test_small_configs(name, window):
    w = W.SMALL[name]()
    ref, _, _ = WIN.run_workload(w, window)
    for psize, fused in ((16, False), (64, True), (0, True)):
        d = Dev(w)
        assert_close(attend(d, window, psize, fused), ref,
                     what=f"{name} window {window} ps {psize} fused {fused}")


EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 511, 512, 513]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("hq,hkv,T", [(32, 8, 1), (32, 8, 5), (16, 1, 4)])
@pytest.mark.parametrize("window", [3, 16, 40])
def test_edge_lengths(D, hq, hkv, T, window):
    lens = [max(L, T) for L in EDGE_LENS]
    w = W.build("edge_win", lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=D,
                num_query_tokens=T, seed=D + hq + T + window)
    ref, _, _ = WIN.run_workload(w, window)
    for ps in (16, 0):
        assert_close(attend(Dev(w), window, ps, True), ref,
                     what=f"D{D} {hq}/{hkv} T{T} window {window} ps{ps}")


@pytest.mark.parametrize("name", ["decode_8b", "spec_verify"])
@pytest.mark.parametrize("window", [5, 64, 300])
def test_fp8_pages(name, window):
    base = W.SMALL[name]()
    w = W.fp8_variant(base, seed=3)
    ref, _, _ = WIN.run_workload(w, window)
    for ps in (32, 0):
        assert_close(attend8(Dev8(w), window, ps), ref, what=f"fp8 {name} window {window}")


def test_window_covering_the_context_is_bit_identical_to_plain():
    w = W.SMALL["spec_verify"]()
    for ps in (64, 0):
        d1, d2 = Dev(w), Dev(w)
        plain = attend(d1, 0, ps, True)
        wide = attend(d2, int(w.context_lens.max()) + 7, ps, True)
        assert torch.equal(bits_t(plain), bits_t(wide))


def bits_t(t):
    return t.view(torch.int16)


def test_negative_window_rejected():
    w = W.SMALL["tiny"]()
    d = Dev(w)
    with pytest.raises(pa.PagedAttnError) as e:
        attend(d, -1, 0, False)
    assert e.value.status == 1


@pytest.mark.parametrize("name,window", [("spec_verify", 4096), ("decode_70b", 1024)])
def test_full_size_every_sequence(name, window):
    w = W.FULL[name]()
    d = Dev(w)
    out = attend(d, window, 0, True)
    torch.cuda.synchronize()
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    s = w.slot_mapping
    k[s // 16, :, s % 16, :] = w.new_key
    v[s // 16, :, s % 16, :] = w.new_value
    ref = all_rows(WIN.paged_attention, w.num_seqs, w.q, k, v, w.block_tables, w.context_lens,
                   w.scale, w.num_kv_heads, 16, window)
    assert_close(out, ref, what=f"{name} window {window} full")
