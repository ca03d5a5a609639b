"""pa_decode_static_scratch: decode for callers that may not allocate device memory.

Such callers (a plugin that its host runtime gives only its input and output
buffers, or a server that reserves all device memory at start-up and must not
call cudaMalloc afterwards) cannot hand pa_decode the split-KV scratch it needs
for long contexts.  pa_decode_static_scratch takes that scratch from a fixed
32 MiB array inside the library instead.  These tests call it through the C
ABI and check it against pa_decode with caller-provided scratch, on two calls
in a row.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402
from gpu_util import MAX_ABS, MAX_REL_L2, Dev, errors  # noqa: E402

STATIC_SCRATCH_BYTES = 32 << 20
vp = ctypes.c_void_p


def _ptr(t):
    return vp(0 if t is None else t.data_ptr())


def _stream():
    return vp(torch.cuda.current_stream().cuda_stream)


def call_static(lib, d, out, psize):
    w = d.w
    return lib.pa_decode_static_scratch(
        _ptr(out), _ptr(d.q), _ptr(d.k), _ptr(d.v), _ptr(d.tables), w.max_blocks_per_seq,
        _ptr(d.lens), w.max_context_len, w.num_seqs, w.num_blocks, w.num_q_heads,
        w.num_kv_heads, w.head_dim, 16, w.scale, psize, _stream())


def call_with_workspace(lib, d, out, psize):
    w = d.w
    need = lib.pa_workspace_size(w.num_seqs, w.num_q_heads, 1, w.max_context_len, w.head_dim,
                                 16, psize, 0)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    st = lib.pa_decode(_ptr(out), _ptr(d.q), _ptr(d.k), _ptr(d.v), _ptr(d.tables),
                       w.max_blocks_per_seq, _ptr(d.lens), w.max_context_len, w.num_seqs,
                       w.num_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim, 16, w.scale,
                       psize, _ptr(ws), need, _stream())
    return st, need


@pytest.mark.parametrize("name,psize", [("decode_8b", 0), ("decode_8b", 256)])
def test_static_scratch_matches_pa_decode(name, psize):
    lib = pa.library()
    w = W.FULL[name]()
    d = Dev(w)
    d.reshape()
    ref = torch.empty_like(d.q)
    st, need = call_with_workspace(lib, d, ref, psize)
    assert st == 0
    assert 0 < need <= STATIC_SCRATCH_BYTES      # the split path really uses the scratch
    ref_np = ref.float().cpu().double().numpy()
    for _ in range(2):                             # two calls in a row share the array
        out = torch.full_like(d.q, float("nan"))
        assert call_static(lib, d, out, psize) == 0
        torch.cuda.synchronize()
        mx, rel, g = errors(out, ref_np)
        assert np.isfinite(g).all()
        assert mx <= MAX_ABS and rel <= MAX_REL_L2, (mx, rel)
    assert pa.get_device_error() == 0


def test_static_scratch_rejects_oversized_request():
    """A shape whose split-KV partials exceed 32 MiB is refused before any launch."""
    lib = pa.library()
    need = lib.pa_workspace_size(256, 64, 1, 8192, 128, 16, 16, 0)
    assert need > STATIC_SCRATCH_BYTES
    d16 = vp(256)                                  # never dereferenced: rejected on the host
    st = lib.pa_decode_static_scratch(d16, d16, d16, d16, d16, 512, d16, 8192, 256, 40000, 64, 8,
                                      128, 16, 0.088, 16, _stream())
    assert st == 3                                 # PA_ERR_WORKSPACE
