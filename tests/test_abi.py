"""The C-ABI library builds, loads without a GPU, exports every declared symbol,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from paged_kv_cache_221_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_attn.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.pa_status_string(code).decode() == name
    assert lib.pa_version() == 102


def test_workspace_size_host_only(lib):
    # one partition per sequence: no scratch
    assert lib.pa_workspace_size(64, 32, 1, 512, 128, 16, 0, 0) == 0
    # 4096 tokens in 512-token partitions: 8 slots per row, (D + 2) floats per slot, 256-B rounded
    rows = 64 * 32

    def r256(x):
        return (x + 255) // 256 * 256

    def want(slots):        # [O partials][(m, l) pairs][256-B work-unit counter]
        return r256(rows * slots * 128 * 4) + r256(rows * slots * 8) + 256

    assert lib.pa_workspace_size(64, 32, 1, 4096, 128, 16, 512, 0) == want(8)
    # default: the largest need over kv-head counts; one kv head (64 pairs, a small
    # batch) splits 4096 tokens into 512-token partitions: 8 slots per row
    assert lib.pa_workspace_size(64, 32, 1, 4096, 128, 16, 0, 0) == want(8)
    assert lib.pa_default_partition_size(64, 8, 4096, 16) == 1536
    assert lib.pa_default_partition_size(64, 8, 100, 16) == 112
    assert lib.pa_default_partition_size(32, 8, 16384, 16) == 2048
    assert lib.pa_default_partition_size(256, 8, 8192, 16) == 3072
    # small batches (< 256 (sequence, kv head) pairs): about 512 CTAs (1024 above
    # 4096 tokens), partitions of at least 128 tokens
    assert lib.pa_default_partition_size(1, 8, 3750, 16) == 128        # 64 parts -> 59 -> 128
    assert lib.pa_default_partition_size(4, 8, 3750, 16) == 240        # 16 parts
    assert lib.pa_default_partition_size(8, 8, 3750, 16) == 480        # 8 parts
    assert lib.pa_default_partition_size(16, 8, 3750, 16) == 944       # 4 parts
    assert lib.pa_default_partition_size(16, 8, 7850, 16) == 992       # 8 parts (1024 CTAs)
    assert lib.pa_default_partition_size(1, 8, 900, 16) == 912         # short: whole
    # shared prefix always needs scratch
    assert lib.pa_workspace_size(2, 4, 1, 64, 64, 16, 64, 2) > 0


def _decode(lib, **kw):
    a = dict(out=16, q=16, k=16, v=16, tables=16, mbs=4, lens=16, mcl=64, B=1, NB=4, hq=4,
             hkv=4, D=64, BS=16, scale=0.125, psize=0, ws=None, wsb=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.pa_decode(vp(a["out"]), vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["tables"]),
                         a["mbs"], vp(a["lens"]), a["mcl"], a["B"], a["NB"], a["hq"], a["hkv"],
                         a["D"], a["BS"], a["scale"], a["psize"], vp(a["ws"]), a["wsb"], None)


def test_argument_errors_return_before_launch(lib):
    E = {v: k for k, v in _lib.STATUS_NAMES.items()}
    assert _decode(lib, B=0) == E["PA_OK"]                       # empty batch: no-op
    assert _decode(lib, q=None) == E["PA_ERR_INVALID_ARG"]
    assert _decode(lib, out=8) == E["PA_ERR_INVALID_ARG"]        # misaligned
    assert _decode(lib, hq=6, hkv=4) == E["PA_ERR_INVALID_ARG"]  # Hq % Hkv
    assert _decode(lib, D=96) == E["PA_ERR_UNSUPPORTED"]
    assert _decode(lib, BS=32) == E["PA_ERR_UNSUPPORTED"]
    assert _decode(lib, hq=128, hkv=1) == E["PA_ERR_UNSUPPORTED"]   # 128 rows per kv head
    assert _decode(lib, mcl=65) == E["PA_ERR_INVALID_ARG"]       # > mbs * 16
    assert _decode(lib, psize=24) == E["PA_ERR_INVALID_ARG"]     # not a block multiple
    assert _decode(lib, psize=16) == E["PA_ERR_WORKSPACE"]       # split needs scratch
    vp = ctypes.c_void_p
    assert lib.pa_reshape_and_cache(vp(16), vp(16), vp(16), vp(16), vp(16), 4, 4, 2, 60, 16,
                                    None) == E["PA_ERR_INVALID_ARG"]
    assert lib.pa_reshape_and_cache(vp(16), vp(16), vp(16), vp(16), vp(16), 4, 4, 2, 64, 8,
                                    None) == E["PA_ERR_UNSUPPORTED"]
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 4, 2, 64, 16,
                                    None) == E["PA_OK"]
    assert lib.pa_selftest_wait_timeout(10, None) == E["PA_ERR_INVALID_ARG"]


def test_library_has_no_driver_link_dependency(lib):
    """The library must load on hosts without the driver: no libcuda.so at link time."""
    import subprocess
    r = subprocess.run(["ldd", _lib.LIB_PATH], capture_output=True, text=True)
    assert "libcuda.so" not in r.stdout
    assert "libtorch" not in r.stdout
