"""Host-side argument checks of the C ABI entry points beyond pa_decode: each bad
argument is rejected with the status the header documents, before any CUDA call.

The device pointers passed here are fake (aligned non-null integers); they are
never dereferenced because every call returns during validation.  The tests
therefore run only on hosts without a GPU, where a call that got past its checks
would fail on its first CUDA call instead of launching a kernel.
"""
import ctypes

import pytest
import torch

import __graft_entry__
from paged_kv_cache_221_gb300 import _lib

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="fake device pointers: host-only argument checks")

E = {v: k for k, v in _lib.STATUS_NAMES.items()}
OK, INVALID, UNSUPPORTED = E["PA_OK"], E["PA_ERR_INVALID_ARG"], E["PA_ERR_UNSUPPORTED"]
vp = ctypes.c_void_p
P = vp(256)                  # a fake 16-byte aligned device pointer
F = ctypes.cast(ctypes.c_void_p(512), ctypes.POINTER(ctypes.c_float))   # fake scale array


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return _lib.load()


def attention(lib, **kw):
    """pa_attention with a valid small bf16 decode configuration, overridden by kw."""
    a = dict(out=P, q=P, nk=None, nv=None, k=P, v=P, ks=None, vs=None, dtype=0, window=0,
             tables=P, mbs=4, lens=P, mcl=64, B=1, T=1, NB=4, hq=4, hkv=4, D=64, BS=16,
             scale=0.125, psize=0, ws=None, wsb=0)
    a.update(kw)
    return lib.pa_attention(a["out"], a["q"], a["nk"], a["nv"], a["k"], a["v"], a["ks"],
                            a["vs"], a["dtype"], a["window"], a["tables"], a["mbs"], a["lens"],
                            a["mcl"], a["B"], a["T"], a["NB"], a["hq"], a["hkv"], a["D"],
                            a["BS"], a["scale"], a["psize"], a["ws"], a["wsb"], None)


def test_attention_arguments(lib):
    assert attention(lib, B=0) == OK                                  # empty batch: no-op
    assert attention(lib, dtype=2) == INVALID                         # unknown page type
    assert attention(lib, nk=P) == INVALID                            # new_key without new_value
    assert attention(lib, window=-1) == INVALID
    assert attention(lib, dtype=1) == INVALID                         # FP8 without scales
    assert attention(lib, dtype=1, ks=F) == INVALID                   # ... or without v_scale
    assert attention(lib, T=0) == INVALID
    assert attention(lib, T=5, mcl=4) == INVALID                      # context below T
    assert attention(lib, hq=64, hkv=1, T=2) == UNSUPPORTED           # 128 rows per kv head
    assert attention(lib, k=vp(264)) == INVALID                       # misaligned pool
    assert attention(lib, psize=-16) == INVALID


def test_append_entry_points_need_new_tokens(lib):
    args = [P, P, None, None, P, P, P, 4, P, 64, 1, 1, 4, 4, 4, 64, 16, 0.125, 0, None, 0, None]
    assert lib.pa_decode_append(*args) == INVALID
    fp8 = args[:6] + [F, F] + args[6:]
    assert lib.pa_decode_append_fp8(*fp8) == INVALID
    args[10] = 0                                                      # empty batch
    assert lib.pa_decode_append(*args) == OK


def test_shared_prefix_arguments(lib):
    base = [P, P, P, P, P, 4, P, 64, 2, 4, 4, 4, 64, 16, 0.125, 0, P, P]
    assert lib.pa_decode_shared_prefix(*base, -1, 2, 2, None, 0, None) == INVALID
    # a group needs its tables: seq_group missing
    bad = base[:16] + [None, P]
    assert lib.pa_decode_shared_prefix(*bad, 1, 2, 2, None, 0, None) == INVALID
    # more prefix blocks than the context holds
    assert lib.pa_decode_shared_prefix(*base, 1, 2, 5, None, 0, None) == INVALID
    fp8 = base[:4] + [F, F] + base[4:]
    assert lib.pa_decode_shared_prefix_fp8(*fp8, -1, 2, 2, None, 0, None) == INVALID
    nos = base[:4] + [None, None] + base[4:]
    assert lib.pa_decode_shared_prefix_fp8(*nos, 1, 2, 2, None, 0, None) == INVALID


def test_windowed_fp8_call_needs_both_scales(lib):
    assert attention(lib, window=8, dtype=1, ks=F, vs=None) == INVALID
    assert attention(lib, window=8, dtype=1, ks=None, vs=F) == INVALID


def test_reshape_fp8_arguments(lib):
    def call(**kw):
        a = dict(k=P, v=P, kc=P, vc=P, slots=P, ks=F, vs=F, n=4, NB=4, hkv=2, D=64, BS=16)
        a.update(kw)
        return lib.pa_reshape_and_cache_fp8(a["k"], a["v"], a["kc"], a["vc"], a["slots"],
                                            a["ks"], a["vs"], a["n"], a["NB"], a["hkv"],
                                            a["D"], a["BS"], None)
    assert call(n=0) == OK
    assert call(D=60) == INVALID
    assert call(BS=8) == UNSUPPORTED
    assert call(ks=None) == INVALID
    assert call(vs=None) == INVALID
    assert call(slots=None) == INVALID
    assert call(kc=vp(264)) == INVALID                                # misaligned pool
    assert call(NB=0) == INVALID


def test_copy_blocks_arguments(lib):
    def call(n=2, pairs=P, NB=4, D=64, BS=16, k=P):
        return lib.pa_copy_blocks(k, P, pairs, n, NB, 2, D, BS, None)
    assert call(n=0) == OK
    assert call(n=-1) == INVALID
    assert call(BS=8) == UNSUPPORTED
    assert call(n=70000) == UNSUPPORTED
    assert call(pairs=None) == INVALID
    assert call(k=vp(264)) == INVALID
    assert call(D=12) == INVALID


def test_spec_accept_arguments(lib):
    def call(B=2, K=3, V=100, greedy=0, p=P, q=P, drafts=P, a=P, s=P, out=P, kept=P):
        return lib.pa_spec_accept(p, q, drafts, a, s, B, K, V, greedy, out, kept, None)
    assert call(B=0) == OK
    assert call(V=0) == INVALID
    assert call(B=-1) == INVALID
    assert call(V=(1 << 19) + 1) == UNSUPPORTED
    assert call(K=65) == UNSUPPORTED
    assert call(p=None) == INVALID
    assert call(drafts=None) == INVALID
    assert call(out=None) == INVALID
    assert call(s=None) == INVALID                                    # sampling needs uniforms
    assert call(q=None) == INVALID                                    # ... and draft probabilities
    assert call(a=None) == INVALID


def runner_create(lib, **kw):
    c = dict(hq=4, hkv=4, D=64, BS=16, T=1, mbs=4, mcl=64, NB=8, dtype=0, window=0, psize=0,
             scale=0.125, pad=7, classes=(1, 2, 4))
    c.update(kw)
    arr = (ctypes.c_int * max(1, len(c["classes"])))(*c["classes"])
    cfg = _lib.RunnerConfig(c["hq"], c["hkv"], c["D"], c["BS"], c["T"], c["mbs"], c["mcl"],
                            c["NB"], c["dtype"], c["window"], c["psize"], c["scale"], c["pad"],
                            len(c["classes"]), arr)
    buf = _lib.RunnerBuffers(out=256, q=256, block_tables=256, context_lens=256, k_cache=256,
                             v_cache=256)
    out = ctypes.c_void_p()
    return lib.pa_runner_create(ctypes.byref(cfg), ctypes.byref(buf), ctypes.byref(out))


def test_runner_configuration_errors(lib):
    assert runner_create(lib, classes=()) == INVALID                  # no class
    assert runner_create(lib, classes=(2, 2)) == INVALID              # not strictly increasing
    assert runner_create(lib, classes=(4, 2)) == INVALID
    assert runner_create(lib, classes=(0, 2)) == INVALID
    assert runner_create(lib, pad=8) == INVALID                       # padding block outside
    assert runner_create(lib, pad=-1) == INVALID
    assert runner_create(lib, psize=-16) == INVALID
    assert runner_create(lib, T=0) == INVALID
    assert runner_create(lib, T=5, mcl=4) == INVALID                  # context below T
    assert lib.pa_runner_class_of(None, 3) == -1
    assert lib.pa_runner_step(None, 1, None) == INVALID
