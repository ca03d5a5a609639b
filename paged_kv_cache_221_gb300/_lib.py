"""ctypes declarations of the C ABI in ``include/paged_attn.h``.

Loading fails loudly if ``libpaged_attn.so`` has not been built: there is no
fallback implementation of any operation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpaged_attn.so")

PA_OK = 0
STATUS_NAMES = {
    0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_WORKSPACE",
    4: "PA_ERR_CUDA", 5: "PA_ERR_BOUNDS", 6: "PA_ERR_TIMEOUT", 7: "PA_ERR_OUT_OF_BLOCKS",
}

class RunnerConfig(ctypes.Structure):
    """pa_runner_config."""
    _fields_ = [("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_query_tokens", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
                ("max_context_len", ctypes.c_int), ("num_blocks", ctypes.c_int),
                ("kv_dtype", ctypes.c_int), ("window_size", ctypes.c_int),
                ("partition_size", ctypes.c_int), ("scale", ctypes.c_float),
                ("pad_block", ctypes.c_int), ("num_classes", ctypes.c_int),
                ("classes", ctypes.POINTER(ctypes.c_int))]


class RunnerBuffers(ctypes.Structure):
    """pa_runner_buffers."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("out", "q", "new_key", "new_value",
                                                 "block_tables", "context_lens", "k_cache",
                                                 "v_cache", "k_scale", "v_scale", "workspace")] + \
               [("workspace_bytes", ctypes.c_size_t)] + \
               [(n, ctypes.c_void_p) for n in ("h_q", "h_new_key", "h_new_value",
                                                 "h_block_tables", "h_context_lens", "h_out")]


# Every symbol the header declares, with (restype, argtypes).
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [_i]),
    "pa_version": (_i, []),
    "pa_last_attention_kernel": (_i, []),
    "pa_reshape_and_cache": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "pa_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "pa_default_partition_size": (_i, [_i, _i, _i, _i]),
    "pa_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i,
                       _vp, _sz, _vp]),
    "pa_verify": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f,
                       _i, _vp, _sz, _vp]),
    "pa_decode_append": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i,
                              _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "pa_decode_shared_prefix": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                                     _i, _f, _i, _vp, _vp, _i, _i, _i, _vp, _sz, _vp]),
    "pa_decode_shared_prefix_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i,
                                         _i, _i, _i, _i, _f, _i, _vp, _vp, _i, _i, _i, _vp, _sz,
                                         _vp]),
    "pa_decode_static_scratch": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i,
                                      _i, _i, _f, _i, _vp]),
    "pa_copy_blocks": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "pa_spec_accept": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp]),
    "pa_reshape_and_cache_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                      _vp]),
    "pa_decode_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                           _i, _f, _i, _vp, _sz, _vp]),
    "pa_verify_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                           _i, _i, _f, _i, _vp, _sz, _vp]),
    "pa_attention": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp, _i, _vp, _i, _i,
                          _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "pa_decode_append_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i,
                                  _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "pa_bm_create": (_i, [_i, _i, ctypes.POINTER(_vp)]),
    "pa_bm_destroy": (None, [_vp]),
    "pa_bm_add_sequence": (_i, [_vp, _i, _i]),
    "pa_bm_fork": (_i, [_vp, _i, _i]),
    "pa_bm_append_slot": (_i, [_vp, _i, ctypes.POINTER(ctypes.c_int64),
                               ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "pa_bm_free_sequence": (_i, [_vp, _i]),
    "pa_bm_block_table": (_i, [_vp, _vp, _i, _i, _vp, _vp]),
    "pa_bm_num_free_blocks": (_i, [_vp]),
    "pa_bm_ref_count": (_i, [_vp, _i]),
    "pa_bm_num_tokens": (_i, [_vp, _i]),
    "pa_runner_create": (_i, [ctypes.POINTER(RunnerConfig), ctypes.POINTER(RunnerBuffers),
                              ctypes.POINTER(_vp)]),
    "pa_runner_step": (_i, [_vp, _i, _vp]),
    "pa_runner_class_of": (_i, [_vp, _i]),
    "pa_runner_destroy": (None, [_vp]),
    "pa_get_device_error": (_i, [_vp]),
    "pa_selftest_wait_timeout": (_i, [ctypes.c_ulonglong, _vp]),
}

_lib = None


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library (once) and declare every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; "
            f"g.build()' or python paged_kv_cache_221_gb300/build.py)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PagedAttnError(fn, status)
