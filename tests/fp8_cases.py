"""FP8 workloads whose every value is known exactly, for pinning the FP8 oracle's glue.

With power-of-two scales every E4M3 value times the scale is a bf16 value.  If
the new tokens are also chosen as E4M3 values times the scale, quantising them
is exact, and the whole FP8 workload has a bf16 twin: the same workload with
each code replaced by its value.  The conversions here use torch's
float8_e4m3fn (a library routine), never the oracle's own codec.
"""
import dataclasses

import numpy as np
import torch

import workloads as W


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy()).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def _bf16(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def exact_fp8_case(seed=13, lens=(5, 16, 17, 40), T=2):
    """(FP8 workload, its bf16 twin).  K and V scales differ from each other and
    per head, so a K/V scale mix-up changes the result."""
    w = W.build("fp8_exact", list(lens), num_q_heads=8, num_kv_heads=2, head_dim=32,
                num_query_tokens=T, seed=seed)
    w = W.fp8_variant(w, seed=seed)
    w.k_scale = np.array([2.0 ** -6, 2.0 ** -4], dtype=np.float32)
    w.v_scale = np.array([2.0 ** -5, 2.0 ** -7], dtype=np.float32)
    rng = np.random.default_rng(seed + 1)
    N, Hkv, D = w.new_key.shape
    kc = W.random_e4m3_codes(rng, (N, Hkv, D))
    vc = W.random_e4m3_codes(rng, (N, Hkv, D))
    w.new_key = _bf16(torch_decode(kc) * w.k_scale[None, :, None])
    w.new_value = _bf16(torch_decode(vc) * w.v_scale[None, :, None])
    kval = torch_decode(w.k_codes) * w.k_scale[None, :, None, None]
    vval = torch_decode(w.v_codes).transpose(0, 1, 3, 2) * w.v_scale[None, :, None, None]
    kb = np.where(np.isnan(kval), W.NAN_BITS, _bf16(kval)).astype(np.uint16)
    vb = np.where(np.isnan(vval), W.NAN_BITS, _bf16(vval)).astype(np.uint16)
    twin = dataclasses.replace(w, name="fp8_exact_twin", kv_dtype="bf16", k_cache=kb,
                               v_cache=vb, k_codes=None, v_codes=None, k_scale=None,
                               v_scale=None)
    return w, twin
