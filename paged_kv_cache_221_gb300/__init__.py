"""GB300-native paged decode attention.

A thin PyTorch binding over the C ABI of ``libpaged_attn.so`` (declared in
``include/paged_attn.h``).  This module only checks tensor shapes, dtypes and
devices and marshals pointers and the current CUDA stream; every step of the
computation runs in the library's sm_103a kernels.  PyTorch is used for device
memory and streams only.

Layouts (bf16 unless stated):
    q, out        [num_seqs, num_query_tokens, num_q_heads, head_dim]
    k_cache,
    v_cache       [num_blocks, num_kv_heads, block_size, head_dim]
    block_tables  [num_seqs, max_blocks_per_seq] int32
    context_lens  [num_seqs] int32 (counts the newest token / the drafts)
    key, value    [num_tokens, num_kv_heads, head_dim]
    slot_mapping  [num_tokens] int64

FP8 (E4M3) pages (``reshape_and_cache_fp8``, ``decode_fp8``, ``verify_fp8``):
    k_cache       [num_blocks, num_kv_heads, block_size, head_dim] uint8 codes
    v_cache       [num_blocks, num_kv_heads, head_dim, block_size] uint8 codes
    k_scale,
    v_scale       [num_kv_heads] float32 (value = code value * scale)
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import numpy as np
import torch

from . import _lib
from ._lib import PagedAttnError, STATUS_NAMES

__all__ = ["reshape_and_cache", "decode", "verify", "decode_shared_prefix", "workspace_size",
           "default_partition_size", "get_device_error", "selftest_wait_timeout", "library",
           "copy_blocks", "BlockManager", "reshape_and_cache_fp8", "decode_fp8", "verify_fp8",
           "attention", "spec_accept", "GraphRunner",
           "PagedAttnError", "STATUS_NAMES"]


def library() -> ctypes.CDLL:
    """The loaded ``libpaged_attn.so`` (raises ImportError if it was not built)."""
    return _lib.load()


def _vp(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(dev: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need(name, t, dtype, ndim, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor) -> None:
    """Scatter new K/V rows into their cache slots (in place, bit-exact)."""
    _need("k_cache", k_cache, torch.bfloat16, 4)
    dev = k_cache.device
    _need("v_cache", v_cache, torch.bfloat16, 4, dev)
    _need("key", key, torch.bfloat16, 3, dev)
    _need("value", value, torch.bfloat16, 3, dev)
    _need("slot_mapping", slot_mapping, torch.int64, 1, dev)
    NB, Hkv, BS, D = k_cache.shape
    N = key.shape[0]
    if v_cache.shape != k_cache.shape or key.shape != (N, Hkv, D) or value.shape != key.shape \
            or slot_mapping.shape[0] != N:
        raise ValueError("inconsistent shapes")
    st = library().pa_reshape_and_cache(_vp(key), _vp(value), _vp(k_cache), _vp(v_cache),
                                        _vp(slot_mapping), N, NB, Hkv, D, BS, _stream(dev))
    _lib.check("pa_reshape_and_cache", st)


def _fp8_pools(k_cache, v_cache, k_scale, v_scale):
    _need("k_cache", k_cache, torch.uint8, 4)
    dev = k_cache.device
    _need("v_cache", v_cache, torch.uint8, 4, dev)
    NB, Hkv, BS, D = k_cache.shape
    if tuple(v_cache.shape) != (NB, Hkv, D, BS):
        raise ValueError("v_cache must be [num_blocks, num_kv_heads, head_dim, block_size]")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _need(name, t, torch.float32, 1, dev)
        if t.shape[0] != Hkv:
            raise ValueError(f"{name} must have num_kv_heads entries")
    return dev, NB, Hkv, BS, D


def reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                          k_scale: torch.Tensor, v_scale: torch.Tensor) -> None:
    """Quantise new bf16 K/V rows to E4M3 (value / scale) and store them in FP8 pages."""
    dev, NB, Hkv, BS, D = _fp8_pools(k_cache, v_cache, k_scale, v_scale)
    _need("key", key, torch.bfloat16, 3, dev)
    _need("value", value, torch.bfloat16, 3, dev)
    _need("slot_mapping", slot_mapping, torch.int64, 1, dev)
    N = key.shape[0]
    if key.shape != (N, Hkv, D) or value.shape != key.shape or slot_mapping.shape[0] != N:
        raise ValueError("inconsistent shapes")
    st = library().pa_reshape_and_cache_fp8(_vp(key), _vp(value), _vp(k_cache), _vp(v_cache),
                                            _vp(slot_mapping), _vp(k_scale), _vp(v_scale), N,
                                            NB, Hkv, D, BS, _stream(dev))
    _lib.check("pa_reshape_and_cache_fp8", st)


def verify_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               k_scale: torch.Tensor, v_scale: torch.Tensor, block_tables: torch.Tensor,
               context_lens: torch.Tensor, max_context_len: Optional[int] = None,
               scale: Optional[float] = None, partition_size: int = 0,
               workspace: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, new_key: Optional[torch.Tensor] = None,
               new_value: Optional[torch.Tensor] = None) -> torch.Tensor:
    """``verify`` (T >= 1 query tokens per sequence) over FP8 pages.

    With ``new_key`` / ``new_value`` (bf16, [B*T, Hkv, D] or [B, T, Hkv, D]) the query
    tokens' K/V are quantised and stored at positions L-T .. L-1 inside the same launch.
    """
    dev, NB, Hkv, BS, D = _fp8_pools(k_cache, v_cache, k_scale, v_scale)
    _need("q", q, torch.bfloat16, 4, dev)
    _need("block_tables", block_tables, torch.int32, 2, dev)
    _need("context_lens", context_lens, torch.int32, 1, dev)
    B, T, Hq, Dq = q.shape
    if Dq != D or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else T   # host sync
    mcl = int(max_context_len)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need("out", out, torch.bfloat16, 4, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    need = workspace_size(B, Hq, T, mcl, D, BS, partition_size, 0) if B else 0
    ws, wsb = _workspace(dev, workspace, need)
    if new_key is not None or new_value is not None:
        for name, t in (("new_key", new_key), ("new_value", new_value)):
            if t is None or t.numel() != B * T * Hkv * D:
                raise ValueError(f"{name} must hold [B, T, Hkv, D] values")
            _need(name, t, torch.bfloat16, t.dim(), dev)
        st = library().pa_decode_append_fp8(
            _vp(out), _vp(q), _vp(new_key), _vp(new_value), _vp(k_cache), _vp(v_cache),
            _vp(k_scale), _vp(v_scale), _vp(block_tables), block_tables.shape[1],
            _vp(context_lens), mcl, B, T, NB, Hq, Hkv, D, BS, scale, partition_size, _vp(ws),
            wsb, _stream(dev))
        _lib.check("pa_decode_append_fp8", st)
        return out
    st = library().pa_verify_fp8(_vp(out), _vp(q), _vp(k_cache), _vp(v_cache), _vp(k_scale),
                                 _vp(v_scale), _vp(block_tables), block_tables.shape[1],
                                 _vp(context_lens), mcl, B, T, NB, Hq, Hkv, D, BS, scale,
                                 partition_size, _vp(ws), wsb, _stream(dev))
    _lib.check("pa_verify_fp8", st)
    return out


def attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor,
              max_context_len: Optional[int] = None, scale: Optional[float] = None,
              partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
              out: Optional[torch.Tensor] = None, new_key: Optional[torch.Tensor] = None,
              new_value: Optional[torch.Tensor] = None, window_size: int = 0,
              k_scale: Optional[torch.Tensor] = None,
              v_scale: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The general per-sequence call (``pa_attention``): q [B, T, Hq, D]; bf16 pools, or FP8
    pools when ``k_scale`` / ``v_scale`` are given; optional fused append of the query
    tokens' K/V; ``window_size`` > 0 for sliding-window attention (each query token sees
    its last ``window_size`` positions)."""
    fp8 = k_scale is not None
    if fp8:
        dev, NB, Hkv, BS, D = _fp8_pools(k_cache, v_cache, k_scale, v_scale)
        _need("q", q, torch.bfloat16, 4, dev)
        _need("block_tables", block_tables, torch.int32, 2, dev)
        _need("context_lens", context_lens, torch.int32, 1, dev)
        B, T, Hq, Dq = q.shape
        if Dq != D or block_tables.shape[0] != B or context_lens.shape[0] != B:
            raise ValueError("inconsistent shapes")
        if max_context_len is None:
            max_context_len = int(context_lens.max().item()) if B else T   # host sync
        mcl = int(max_context_len)
        if out is None:
            out = torch.empty_like(q)
        else:
            _need("out", out, torch.bfloat16, 4, dev)
    else:
        dev, B, T, Hq, D, NB, Hkv, BS, mcl, out = _attn_common(q, k_cache, v_cache, block_tables,
                                                              context_lens, max_context_len, out)
    if (new_key is None) != (new_value is None):
        raise ValueError("new_key and new_value go together")
    if new_key is not None:
        for name, t in (("new_key", new_key), ("new_value", new_value)):
            if t.numel() != B * T * Hkv * D:
                raise ValueError(f"{name} must hold [B, T, Hkv, D] values")
            _need(name, t, torch.bfloat16, t.dim(), dev)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    need = workspace_size(B, Hq, T, mcl, D, BS, partition_size, 0) if B else 0
    ws, wsb = _workspace(dev, workspace, need)
    st = library().pa_attention(_vp(out), _vp(q), _vp(new_key), _vp(new_value), _vp(k_cache),
                                _vp(v_cache), _vp(k_scale), _vp(v_scale), 1 if fp8 else 0,
                                int(window_size), _vp(block_tables), block_tables.shape[1],
                                _vp(context_lens), mcl, B, T, NB, Hq, Hkv, D, BS, scale,
                                partition_size, _vp(ws), wsb, _stream(dev))
    _lib.check("pa_attention", st)
    return out


def decode_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               k_scale: torch.Tensor, v_scale: torch.Tensor, block_tables: torch.Tensor,
               context_lens: torch.Tensor, max_context_len: Optional[int] = None,
               scale: Optional[float] = None, partition_size: int = 0,
               workspace: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, new_key: Optional[torch.Tensor] = None,
               new_value: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Single-token decode over FP8 pages; q is [B, Hq, D] or [B, 1, Hq, D].

    With ``new_key`` / ``new_value`` ([B, Hkv, D] bf16) the new token is quantised and
    stored at position L-1 of every sequence inside the same launch."""
    squeeze = q.dim() == 3
    q4 = q.unsqueeze(1) if squeeze else q
    if q4.shape[1] != 1:
        raise ValueError("decode_fp8 takes one query token per sequence (use verify_fp8)")
    o4 = None if out is None else (out.unsqueeze(1) if squeeze else out)
    r = verify_fp8(q4, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                   max_context_len, scale, partition_size, workspace, o4, new_key, new_value)
    return r.squeeze(1) if squeeze else r


def workspace_size(num_seqs: int, num_q_heads: int, num_query_tokens: int, max_context_len: int,
                   head_dim: int, block_size: int = 16, partition_size: int = 0,
                   max_prefix_blocks: int = 0) -> int:
    """Scratch bytes an attention call with these sizes needs (0 if none)."""
    return int(library().pa_workspace_size(num_seqs, num_q_heads, num_query_tokens,
                                           max_context_len, head_dim, block_size, partition_size,
                                           max_prefix_blocks))


def default_partition_size(num_seqs: int, num_kv_heads: int, max_context_len: int,
                           block_size: int = 16) -> int:
    return int(library().pa_default_partition_size(num_seqs, num_kv_heads, max_context_len,
                                                   block_size))


def _attn_common(q, k_cache, v_cache, block_tables, context_lens, max_context_len, out):
    _need("k_cache", k_cache, torch.bfloat16, 4)
    dev = k_cache.device
    _need("v_cache", v_cache, torch.bfloat16, 4, dev)
    _need("q", q, torch.bfloat16, 4, dev)
    _need("block_tables", block_tables, torch.int32, 2, dev)
    _need("context_lens", context_lens, torch.int32, 1, dev)
    B, T, Hq, D = q.shape
    NB, Hkv, BS, Dk = k_cache.shape
    if v_cache.shape != k_cache.shape or Dk != D or block_tables.shape[0] != B or \
            context_lens.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else T   # host sync
    if out is None:
        out = torch.empty_like(q)
    else:
        _need("out", out, torch.bfloat16, 4, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    return dev, B, T, Hq, D, NB, Hkv, BS, int(max_context_len), out


def _workspace(dev, workspace, need):
    if workspace is None:
        if need == 0:
            return None, 0
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    elif not (workspace.is_cuda and workspace.device == dev and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor on the cache's device")
    return workspace, workspace.numel() * workspace.element_size()


def verify(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables: torch.Tensor, context_lens: torch.Tensor,
           max_context_len: Optional[int] = None, scale: Optional[float] = None,
           partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
           out: Optional[torch.Tensor] = None, new_key: Optional[torch.Tensor] = None,
           new_value: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Attention of T draft tokens per sequence ([B, T, Hq, D]) with a causal mask among drafts.

    With ``new_key`` / ``new_value`` ([B*T, Hkv, D] or [B, T, Hkv, D]) the query tokens' K/V
    are first stored at positions L-T .. L-1 of every sequence, inside the same launch
    (reshape_and_cache fused).
    """
    dev, B, T, Hq, D, NB, Hkv, BS, mcl, out = _attn_common(q, k_cache, v_cache, block_tables,
                                                          context_lens, max_context_len, out)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    need = workspace_size(B, Hq, T, mcl, D, BS, partition_size, 0) if B else 0
    ws, wsb = _workspace(dev, workspace, need)
    lib = library()
    if new_key is not None or new_value is not None:
        for name, t in (("new_key", new_key), ("new_value", new_value)):
            if t is None or t.numel() != B * T * Hkv * D:
                raise ValueError(f"{name} must hold [B, T, Hkv, D] values")
            _need(name, t, torch.bfloat16, t.dim(), dev)
        st = lib.pa_decode_append(_vp(out), _vp(q), _vp(new_key), _vp(new_value), _vp(k_cache),
                                  _vp(v_cache), _vp(block_tables), block_tables.shape[1],
                                  _vp(context_lens), mcl, B, T, NB, Hq, Hkv, D, BS, scale,
                                  partition_size, _vp(ws), wsb, _stream(dev))
        _lib.check("pa_decode_append", st)
        return out
    if T == 1:
        st = lib.pa_decode(_vp(out), _vp(q), _vp(k_cache), _vp(v_cache), _vp(block_tables),
                           block_tables.shape[1], _vp(context_lens), mcl, B, NB, Hq, Hkv, D, BS,
                           scale, partition_size, _vp(ws), wsb, _stream(dev))
        _lib.check("pa_decode", st)
    else:
        st = lib.pa_verify(_vp(out), _vp(q), _vp(k_cache), _vp(v_cache), _vp(block_tables),
                           block_tables.shape[1], _vp(context_lens), mcl, B, T, NB, Hq, Hkv, D,
                           BS, scale, partition_size, _vp(ws), wsb, _stream(dev))
        _lib.check("pa_verify", st)
    return out


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables: torch.Tensor, context_lens: torch.Tensor,
           max_context_len: Optional[int] = None, scale: Optional[float] = None,
           partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
           out: Optional[torch.Tensor] = None, new_key: Optional[torch.Tensor] = None,
           new_value: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Single-token decode attention; q is [B, Hq, D] or [B, 1, Hq, D] (out has q's shape).

    With ``new_key`` / ``new_value`` ([B, Hkv, D]) the new token's K/V is stored at position
    L-1 of every sequence inside the same launch before attention reads it.
    """
    squeeze = q.dim() == 3
    q4 = q.unsqueeze(1) if squeeze else q
    if q4.shape[1] != 1:
        raise ValueError("decode takes one query token per sequence (use verify for drafts)")
    o4 = None if out is None else (out.unsqueeze(1) if squeeze else out)
    r = verify(q4, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
               partition_size, workspace, o4, new_key, new_value)
    return r.squeeze(1) if squeeze else r


def decode_shared_prefix(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         block_tables: torch.Tensor, context_lens: torch.Tensor,
                         seq_group: torch.Tensor, group_prefix_blocks: torch.Tensor,
                         max_group_size: int, max_prefix_blocks: int,
                         max_context_len: Optional[int] = None, scale: Optional[float] = None,
                         partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                         out: Optional[torch.Tensor] = None, k_scale: Optional[torch.Tensor] = None,
                         v_scale: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode where groups of sequences share copy-on-write prefix blocks, read once per group.

    With ``k_scale`` / ``v_scale`` the pools are FP8 (E4M3) pages as for ``decode_fp8``."""
    squeeze = q.dim() == 3
    q4 = q.unsqueeze(1) if squeeze else q
    o4 = None if out is None else (out.unsqueeze(1) if squeeze else out)
    fp8 = k_scale is not None
    if fp8:
        dev, NB, Hkv, BS, D = _fp8_pools(k_cache, v_cache, k_scale, v_scale)
        _need("q", q4, torch.bfloat16, 4, dev)
        _need("block_tables", block_tables, torch.int32, 2, dev)
        _need("context_lens", context_lens, torch.int32, 1, dev)
        B, T, Hq, Dq = q4.shape
        if Dq != D or block_tables.shape[0] != B or context_lens.shape[0] != B:
            raise ValueError("inconsistent shapes")
        if max_context_len is None:
            max_context_len = int(context_lens.max().item()) if B else T   # host sync
        mcl = int(max_context_len)
        if o4 is None:
            o4 = torch.empty_like(q4)
        else:
            _need("out", o4, torch.bfloat16, 4, dev)
    else:
        dev, B, T, Hq, D, NB, Hkv, BS, mcl, o4 = _attn_common(q4, k_cache, v_cache, block_tables,
                                                             context_lens, max_context_len, o4)
    if T != 1:
        raise ValueError("decode_shared_prefix takes one query token per sequence")
    _need("seq_group", seq_group, torch.int32, 1, dev)
    _need("group_prefix_blocks", group_prefix_blocks, torch.int32, 1, dev)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    need = workspace_size(B, Hq, 1, mcl, D, BS, partition_size, max_prefix_blocks) if B else 0
    ws, wsb = _workspace(dev, workspace, need)
    if fp8:
        st = library().pa_decode_shared_prefix_fp8(
            _vp(o4), _vp(q4), _vp(k_cache), _vp(v_cache), _vp(k_scale), _vp(v_scale),
            _vp(block_tables), block_tables.shape[1], _vp(context_lens), mcl, B, NB, Hq, Hkv, D,
            BS, scale, partition_size, _vp(seq_group), _vp(group_prefix_blocks),
            group_prefix_blocks.shape[0], max_group_size, max_prefix_blocks, _vp(ws), wsb,
            _stream(dev))
        _lib.check("pa_decode_shared_prefix_fp8", st)
        return o4.squeeze(1) if squeeze else o4
    st = library().pa_decode_shared_prefix(
        _vp(o4), _vp(q4), _vp(k_cache), _vp(v_cache), _vp(block_tables), block_tables.shape[1],
        _vp(context_lens), mcl, B, NB, Hq, Hkv, D, BS, scale, partition_size, _vp(seq_group),
        _vp(group_prefix_blocks), group_prefix_blocks.shape[0], max_group_size,
        max_prefix_blocks, _vp(ws), wsb, _stream(dev))
    _lib.check("pa_decode_shared_prefix", st)
    return o4.squeeze(1) if squeeze else o4


def get_device_error(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    return int(library().pa_get_device_error(_stream(dev)))


LAST_KERNEL_NAMES = {0: "none", 1: "per_unit", 2: "persistent", 3: "tcgen05"}


def last_attention_kernel() -> str:
    """The kernel of this thread's last per-sequence attention launch: "none",
    "per_unit", "persistent" or "tcgen05" (a diagnostic)."""
    return LAST_KERNEL_NAMES[int(library().pa_last_attention_kernel())]


def selftest_wait_timeout(timeout_ns: int, device=None) -> None:
    """Launch the bounded-wait self test (read the outcome with get_device_error)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    _lib.check("pa_selftest_wait_timeout",
               library().pa_selftest_wait_timeout(int(timeout_ns), _stream(dev)))


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, pairs) -> None:
    """Copy whole physical blocks src -> dst in both pools (copy-on-write), bit-exact.

    ``pairs``: sequence of (src, dst) ids or an int32 tensor [n, 2] (host or device).
    """
    _need("k_cache", k_cache, torch.bfloat16, 4)
    dev = k_cache.device
    _need("v_cache", v_cache, torch.bfloat16, 4, dev)
    if v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent shapes")
    t = pairs if isinstance(pairs, torch.Tensor) else torch.tensor(list(pairs), dtype=torch.int32)
    t = t.to(device=dev, dtype=torch.int32).reshape(-1, 2).contiguous()
    if t.shape[0] == 0:
        return
    NB, Hkv, BS, D = k_cache.shape
    st = library().pa_copy_blocks(_vp(k_cache), _vp(v_cache), _vp(t), t.shape[0], NB, Hkv, D, BS,
                                  _stream(dev))
    _lib.check("pa_copy_blocks", st)


def spec_accept(target_probs: torch.Tensor, draft_tokens: torch.Tensor,
                draft_probs: Optional[torch.Tensor] = None,
                accept_uniforms: Optional[torch.Tensor] = None,
                sample_uniforms: Optional[torch.Tensor] = None, greedy: bool = False):
    """Speculative acceptance after verify: (out_tokens [B, K+1] int32, num_accepted [B]).

    target_probs float32 [B, K+1, V]; draft_tokens int32 [B, K]; for sampling also
    draft_probs float32 [B, K, V], accept_uniforms uint32-valued int32/int64 [B, K] (low 24
    bits used) and sample_uniforms [B] (32-bit values).  Uniform tensors are passed as
    int32 views of the 32-bit patterns.
    """
    _need("target_probs", target_probs, torch.float32, 3)
    dev = target_probs.device
    B, K1, V = target_probs.shape
    K = K1 - 1
    _need("draft_tokens", draft_tokens, torch.int32, 2, dev)
    if tuple(draft_tokens.shape) != (B, K):
        raise ValueError("draft_tokens must be [B, K]")
    if not greedy:
        _need("draft_probs", draft_probs, torch.float32, 3, dev)
        _need("accept_uniforms", accept_uniforms, torch.int32, 2, dev)
        _need("sample_uniforms", sample_uniforms, torch.int32, 1, dev)
        if tuple(draft_probs.shape) != (B, K, V) or tuple(accept_uniforms.shape) != (B, K) \
                or sample_uniforms.shape[0] != B:
            raise ValueError("inconsistent shapes")
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    kept = torch.empty(B, dtype=torch.int32, device=dev)
    st = library().pa_spec_accept(_vp(target_probs), _vp(draft_probs if not greedy else None),
                                  _vp(draft_tokens), _vp(accept_uniforms if not greedy else None),
                                  _vp(sample_uniforms if not greedy else None), B, K, V,
                                  1 if greedy else 0, _vp(out), _vp(kept), _stream(dev))
    _lib.check("pa_spec_accept", st)
    return out, kept


class GraphRunner:
    """CUDA graphs of the attention step for fixed batch-size classes (``pa_runner_*``).

    The runner captures one ``pa_attention`` call per class over static buffers sized for
    the largest class, which this object allocates and exposes: write a step's inputs into
    rows 0 .. B-1 of ``q``, ``new_key``, ``new_value``, ``block_tables`` and
    ``context_lens``, call ``step(B)``, read rows 0 .. B-1 of ``out``.  Rows B .. c-1 of
    the class c are padded on the device with a one-block sequence in ``pad_block`` (a
    physical block no sequence uses).  ``partition_size`` 0 captures each class with the
    library default for its batch size.

    With ``host_staging`` the runner also allocates page-locked host mirrors ``h_q``,
    ``h_new_key``, ``h_new_value``, ``h_block_tables``, ``h_context_lens`` and ``h_out``,
    and every class graph copies the inputs in and the output back itself: write the
    step's inputs into the host rows, call ``step(B)``, synchronise, read ``h_out``.
    """

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, num_q_heads: int,
                 max_context_len: int, max_blocks_per_seq: int, pad_block: int,
                 partition_size: int, classes=(1, 2, 4, 8, 16), num_query_tokens: int = 1,
                 scale: Optional[float] = None, window_size: int = 0, fused_append: bool = True,
                 k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                 host_staging: bool = False):
        self._lib = library()
        fp8 = k_scale is not None
        if fp8:
            dev, NB, Hkv, BS, D = _fp8_pools(k_cache, v_cache, k_scale, v_scale)
        else:
            _need("k_cache", k_cache, torch.bfloat16, 4)
            dev = k_cache.device
            _need("v_cache", v_cache, torch.bfloat16, 4, dev)
            NB, Hkv, BS, D = k_cache.shape
        classes = sorted(int(c) for c in classes)
        Bmax, T = classes[-1], int(num_query_tokens)
        self.classes = classes
        # the inputs live in one block (q, new_key, new_value, block_tables, context_lens,
        # 256-byte aligned), mirrored on the host when staging, so one copy moves them all
        shapes = [("q", (Bmax, T, num_q_heads, D), torch.bfloat16),
                  ("new_key", (Bmax * T, Hkv, D), torch.bfloat16),
                  ("new_value", (Bmax * T, Hkv, D), torch.bfloat16),
                  ("block_tables", (Bmax, max_blocks_per_seq), torch.int32),
                  ("context_lens", (Bmax,), torch.int32)]
        offs, total = [], 0
        for _, shp, dt in shapes:
            offs.append(total)
            n = int(np.prod(shp)) * torch.tensor([], dtype=dt).element_size()
            total += (n + 255) // 256 * 256

        def carve(block):
            return {name: block[o:o + int(np.prod(shp)) * torch.tensor([], dtype=dt)
                                .element_size()].view(dt).view(shp)
                    for (name, shp, dt), o in zip(shapes, offs)}

        self._dblock = torch.zeros(total, dtype=torch.uint8, device=dev)
        d = carve(self._dblock)
        self.q, self.block_tables, self.context_lens = d["q"], d["block_tables"], d["context_lens"]
        self.new_key = d["new_key"] if fused_append else None
        self.new_value = d["new_value"] if fused_append else None
        self.block_tables.fill_(pad_block)
        self.context_lens.fill_(T)
        self.out = torch.zeros_like(self.q)
        need = max(workspace_size(c, num_q_heads, T, max_context_len, D, BS, partition_size, 0)
                   for c in classes)
        self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        self._keep = (k_cache, v_cache, k_scale, v_scale)
        host = None
        if host_staging:
            self._hblock = torch.zeros(total, dtype=torch.uint8).pin_memory()
            hb = carve(self._hblock)
            self.h_q, self.h_block_tables = hb["q"], hb["block_tables"]
            self.h_context_lens = hb["context_lens"]
            self.h_new_key = hb["new_key"] if fused_append else None
            self.h_new_value = hb["new_value"] if fused_append else None
            self.h_block_tables.fill_(pad_block)
            self.h_context_lens.fill_(T)
            self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
            host = (self.h_q.data_ptr(),
                    self.h_new_key.data_ptr() if fused_append else None,
                    self.h_new_value.data_ptr() if fused_append else None,
                    self.h_block_tables.data_ptr(), self.h_context_lens.data_ptr(),
                    self.h_out.data_ptr())
        self._classes_c = (ctypes.c_int * len(classes))(*classes)
        cfg = _lib.RunnerConfig(num_q_heads, Hkv, D, BS, T, max_blocks_per_seq, max_context_len,
                                NB, 1 if fp8 else 0, int(window_size), int(partition_size),
                                1.0 / math.sqrt(D) if scale is None else float(scale),
                                int(pad_block), len(classes), self._classes_c)
        bufs = _lib.RunnerBuffers(self.out.data_ptr(), self.q.data_ptr(),
                                  self.new_key.data_ptr() if fused_append else None,
                                  self.new_value.data_ptr() if fused_append else None,
                                  self.block_tables.data_ptr(), self.context_lens.data_ptr(),
                                  k_cache.data_ptr(), v_cache.data_ptr(),
                                  k_scale.data_ptr() if fp8 else None,
                                  v_scale.data_ptr() if fp8 else None,
                                  self.workspace.data_ptr(),
                                  self.workspace.numel(), *(host or (None,) * 6))
        h = ctypes.c_void_p()
        torch.cuda.synchronize(dev)
        _lib.check("pa_runner_create", self._lib.pa_runner_create(ctypes.byref(cfg),
                                                                  ctypes.byref(bufs),
                                                                  ctypes.byref(h)))
        self._h = h
        self.device = dev

    def class_of(self, num_seqs: int) -> int:
        return int(self._lib.pa_runner_class_of(self._h, num_seqs))

    def step(self, num_seqs: int) -> None:
        _lib.check("pa_runner_step", self._lib.pa_runner_step(self._h, num_seqs,
                                                              _stream(self.device)))

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pa_runner_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BlockManager:
    """Host-side block manager of the paged KV cache (the library's native C++ manager).

    Sequences own ordered lists of physical blocks; ``fork`` shares them; the
    first append into a shared, partly filled block returns a copy to perform
    (copy-on-write).  New blocks are the lowest-numbered free ones.
    """

    def __init__(self, num_blocks: int, block_size: int = 16):
        self._lib = library()
        h = ctypes.c_void_p()
        _lib.check("pa_bm_create", self._lib.pa_bm_create(num_blocks, block_size, ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_sequence(self, seq_id: int, num_tokens: int) -> None:
        _lib.check("pa_bm_add_sequence", self._lib.pa_bm_add_sequence(self._h, seq_id, num_tokens))

    def fork(self, parent_id: int, child_id: int) -> None:
        _lib.check("pa_bm_fork", self._lib.pa_bm_fork(self._h, parent_id, child_id))

    def append_slot(self, seq_id: int):
        """Reserve the next token's slot: returns (slot, copy) with copy = (src, dst) or None."""
        slot = ctypes.c_int64()
        src, dst = ctypes.c_int32(), ctypes.c_int32()
        _lib.check("pa_bm_append_slot", self._lib.pa_bm_append_slot(
            self._h, seq_id, ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst)))
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def free_sequence(self, seq_id: int) -> None:
        _lib.check("pa_bm_free_sequence", self._lib.pa_bm_free_sequence(self._h, seq_id))

    def block_table(self, seq_ids, max_blocks_per_seq: int):
        """(block_tables int32 [n, max_blocks], context_lens int32 [n]) as host tensors."""
        ids = torch.tensor(list(seq_ids), dtype=torch.int32)
        n = ids.numel()
        tables = torch.empty((n, max_blocks_per_seq), dtype=torch.int32)
        lens = torch.empty(n, dtype=torch.int32)
        _lib.check("pa_bm_block_table", self._lib.pa_bm_block_table(
            self._h, _vp(ids) if n else None, n, max_blocks_per_seq,
            _vp(tables) if n else None, _vp(lens) if n else None))
        return tables, lens

    def num_free_blocks(self) -> int:
        return int(self._lib.pa_bm_num_free_blocks(self._h))

    def ref_count(self, block: int) -> int:
        return int(self._lib.pa_bm_ref_count(self._h, block))

    def num_tokens(self, seq_id: int) -> int:
        return int(self._lib.pa_bm_num_tokens(self._h, seq_id))
