"""pa_decode_static_scratch: decode for callers that may not allocate device memory.

Such callers (a plugin that its host runtime gives only its input and output
buffers, or a server that reserves all device memory at start-up and must not
call cudaMalloc afterwards) cannot hand pa_decode the split-KV scratch it needs
for long contexts.  pa_decode_static_scratch takes that scratch from a fixed
32 MiB array inside the library instead.  These tests call it through the C
ABI.  Its output must be bit-identical to pa_decode given caller scratch (the
same kernels and the same partition plan) and within the bf16 tolerance of the
fp64 oracle, on two calls in a row with a call of another shape between them.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402
from gpu_util import Dev, assert_close, bits, to_dev  # noqa: E402

STATIC_SCRATCH_BYTES = 32 << 20
PA_ERR_INVALID_ARG, PA_ERR_WORKSPACE = 1, 3
vp = ctypes.c_void_p


def _ptr(t):
    return vp(0 if t is None else t.data_ptr())


def _stream():
    return vp(torch.cuda.current_stream().cuda_stream)


def _shape(d, max_context_len=None, tables=None):
    w = d.w
    tb = d.tables if tables is None else tables
    return dict(tables=tb, mbs=tb.shape[1],
                mcl=w.max_context_len if max_context_len is None else max_context_len)


def call_static(lib, d, out, psize, **kw):
    w, s = d.w, _shape(d, **kw)
    return lib.pa_decode_static_scratch(
        _ptr(out), _ptr(d.q), _ptr(d.k), _ptr(d.v), _ptr(s["tables"]), s["mbs"],
        _ptr(d.lens), s["mcl"], w.num_seqs, w.num_blocks, w.num_q_heads,
        w.num_kv_heads, w.head_dim, 16, w.scale, psize, _stream())


def call_pa_decode(lib, d, out, psize, ws, nbytes, **kw):
    w, s = d.w, _shape(d, **kw)
    return lib.pa_decode(_ptr(out), _ptr(d.q), _ptr(d.k), _ptr(d.v), _ptr(s["tables"]),
                         s["mbs"], _ptr(d.lens), s["mcl"], w.num_seqs, w.num_blocks,
                         w.num_q_heads, w.num_kv_heads, w.head_dim, 16, w.scale, psize,
                         _ptr(ws), nbytes, _stream())


def with_caller_scratch(lib, d, psize):
    """pa_decode with scratch the caller allocated; returns (output, scratch bytes needed)."""
    w = d.w
    need = lib.pa_workspace_size(w.num_seqs, w.num_q_heads, 1, w.max_context_len, w.head_dim,
                                 16, psize, 0)
    # the scratch pa_decode needs with this kv-head count (pa_workspace_size is the bound
    # over kv-head counts when psize is 0)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    out = torch.full_like(d.q, float("nan"))
    assert call_pa_decode(lib, d, out, psize, ws, need) == 0
    return out, need


def prepared(w):
    d = Dev(w)
    d.reshape()
    return d


@pytest.mark.parametrize("psize", [0, 256])
def test_static_scratch_equals_pa_decode(psize):
    """Two calls on the 8B-shape batch with a call of another shape and partition size
    between them: each output bit-identical to pa_decode with caller scratch, and within
    tolerance of the oracle."""
    lib = pa.library()
    w = W.FULL["decode_8b"]()
    d = prepared(w)
    ref_bits = bits(with_caller_scratch(lib, d, psize)[0])
    need = lib.pa_workspace_size(w.num_seqs, w.num_q_heads, 1, w.max_context_len, w.head_dim,
                                 16, psize, 0)
    assert 0 < need <= STATIC_SCRATCH_BYTES      # the split path really uses the scratch
    oracle_out, _, _ = O.run_workload(w)

    # another shape, whose partials land in the same array at other offsets
    w2 = W.SMALL["decode_70b"]()
    d2 = prepared(w2)
    ref2 = bits(with_caller_scratch(lib, d2, 48)[0])

    for i in range(2):
        out = torch.full_like(d.q, float("nan"))
        assert call_static(lib, d, out, psize) == 0
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits(out), ref_bits, err_msg=f"call {i}")
        assert_close(out, oracle_out, what=f"static scratch call {i}")
        if i == 0:
            out2 = torch.full_like(d2.q, float("nan"))
            assert call_static(lib, d2, out2, 48) == 0
            torch.cuda.synchronize()
            np.testing.assert_array_equal(bits(out2), ref2, err_msg="other shape")
    assert pa.get_device_error() == 0


def _padded_tables(w, mbs):
    t = np.zeros((w.num_seqs, mbs), dtype=np.int32)
    t[:, :w.block_tables.shape[1]] = w.block_tables
    return to_dev(t)


def test_static_scratch_oversized_default_runs_whole_sequences():
    """partition_size 0 with a declared max_context_len whose default split needs more
    than 32 MiB: the call attends over whole sequences, as pa_decode without scratch does."""
    lib = pa.library()
    rng = np.random.default_rng(7)
    lens = rng.integers(1, 300, size=256)
    w = W.build("static_oversize", lens, num_q_heads=64, num_kv_heads=8, head_dim=128, seed=7)
    d = prepared(w)
    mcl, mbs = 32768, 2048
    tables = _padded_tables(w, mbs)
    need = pa.workspace_size(w.num_seqs, w.num_q_heads, 1, mcl, 128, 16, 0)
    assert need > STATIC_SCRATCH_BYTES
    ref = torch.full_like(d.q, float("nan"))
    assert call_pa_decode(lib, d, ref, 0, None, 0, max_context_len=mcl, tables=tables) == 0
    out = torch.full_like(d.q, float("nan"))
    assert call_static(lib, d, out, 0, max_context_len=mcl, tables=tables) == 0
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(out), bits(ref))
    assert_close(out, O.run_workload(w)[0], what="oversized default")
    assert pa.get_device_error() == 0


def test_static_scratch_rejects_oversized_explicit_partition():
    """An explicit partition size whose partials exceed 32 MiB is refused before any
    launch; an argument error in the same call is reported first."""
    lib = pa.library()
    need = lib.pa_workspace_size(256, 64, 1, 8192, 128, 16, 16, 0)
    assert need > STATIC_SCRATCH_BYTES
    d16 = vp(256)                                  # never dereferenced: rejected on the host
    st = lib.pa_decode_static_scratch(d16, d16, d16, d16, d16, 512, d16, 8192, 256, 40000, 64, 8,
                                      128, 16, 0.088, 16, _stream())
    assert st == PA_ERR_WORKSPACE
    # 60 q heads over 8 kv heads is not a GQA layout: INVALID_ARG, not WORKSPACE
    st = lib.pa_decode_static_scratch(d16, d16, d16, d16, d16, 512, d16, 8192, 256, 40000, 60, 8,
                                      128, 16, 0.088, 16, _stream())
    assert st == PA_ERR_INVALID_ARG
