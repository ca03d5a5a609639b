"""Pins of the FP8 (E4M3) oracle against facts that do not come from it.

Sources of truth: torch's float8_e4m3fn conversions (a library routine, in both
directions), the format's saturation and NaN rules, the documented storage
layout checked by scalar loops, and a reduction to the pinned bf16 oracle: with
power-of-two scales every dequantised value is exactly a bf16 value, so
attention over FP8 pages must equal bf16 attention over those values.  The
planted-mistake test re-runs every pin against broken copies of the oracle.
"""
import types

import numpy as np
import pytest
import torch

import workloads as W
from fp8_cases import exact_fp8_case
from oracle import fp8 as F
from oracle import oracle as O

ALL_CODES = np.arange(256, dtype=np.uint8)


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy()).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode(x32):
    return torch.from_numpy(np.asarray(x32, dtype=np.float32).copy()).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def small_fp8(seed=11, pow2=False):
    w = W.build("fp8_case", [5, 16, 17, 40], num_q_heads=8, num_kv_heads=2, head_dim=32,
                num_query_tokens=2, seed=seed)
    w = W.fp8_variant(w, seed=seed)
    if pow2:
        w.k_scale = np.array([2.0 ** -6, 2.0 ** -4], dtype=np.float32)
        w.v_scale = np.array([2.0 ** -5, 2.0 ** -7], dtype=np.float32)
    return w


# ----------------------------------------------------------------------------- pins

def pin_decode_matches_torch(f):
    got = f.decode(ALL_CODES)
    want = torch_decode(ALL_CODES)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def pin_encode_matches_torch(f):
    pos = torch_decode(ALL_CODES[:0x7F])                      # 0 .. 448, increasing
    mids = (pos[:-1] + pos[1:]) / 2                           # exact ties (float32-exact)
    rng = np.random.default_rng(3)
    rand = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 4000))
    x = np.concatenate([pos, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                        np.nextafter(mids.astype(np.float32), np.float32(1000)), rand,
                        [0.0, 2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -12]]).astype(np.float32)
    x = np.concatenate([x, -x])
    assert np.array_equal(f.encode(x.astype(np.float64)), torch_encode(x))


def pin_encode_saturates_and_nan(f):
    x = np.array([448.0, 449.0, 464.0, 480.0, 1e6, np.inf, -np.inf, -1e6, np.nan, -0.0])
    assert f.encode(x).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x80]


def pin_round_trip(f):
    finite = ALL_CODES[~np.isnan(torch_decode(ALL_CODES))]
    assert np.array_equal(f.encode(f.decode(finite)), finite)


def pin_quantize_divides_in_float32(f):
    rng = np.random.default_rng(4)
    bits = W.normal_bf16(rng, (2000,))
    for s in (np.float32(1 / 64.0), np.float32(0.0137), np.float32(3.0)):
        x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float() / float(s)
        x = x.clamp(-448, 448)                     # torch does not saturate; the format does
        assert np.array_equal(f.quantize(bits, s), torch_encode(x.numpy()))
    # Quotients that round (in float32) onto an exact tie of two codes while the
    # exact quotient is off the tie: only a float32 division gets these right.
    pos = torch_decode(ALL_CODES[:0x7F])
    mids = ((pos[:-1] + pos[1:]) / 2)[20:].astype(np.float32)
    xs = W.normal_bf16(rng, (4000,))
    xf = O.bf16_bits_to_f64(xs).astype(np.float32)
    hits = 0
    for i in range(len(xs)):
        m = mids[i % len(mids)]
        s = np.float32(abs(xf[i]) / m)
        if not np.isfinite(s) or s == 0:
            continue
        q32 = np.float32(xf[i]) / s
        if abs(q32) != m or abs(float(xf[i]) / float(s)) == float(m):
            continue
        hits += 1
        assert f.quantize(xs[i:i + 1], s)[0] == torch_encode(np.array([q32]))[0]
    assert hits > 50


def pin_reshape_layout(f):
    w = small_fp8()
    k, v = f.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                               w.k_scale, w.v_scale, w.block_size)
    written = set()
    for i, slot in enumerate(w.slot_mapping.tolist()):
        blk, off = divmod(slot, w.block_size)
        for h in range(w.num_kv_heads):
            kx = torch.from_numpy(w.new_key[i, h].view(np.int16).copy()).view(
                torch.bfloat16).float() / float(w.k_scale[h])
            vx = torch.from_numpy(w.new_value[i, h].view(np.int16).copy()).view(
                torch.bfloat16).float() / float(w.v_scale[h])
            kc, vc = torch_encode(kx.numpy()), torch_encode(vx.numpy())
            for d in range(w.head_dim):
                assert k[blk, h, off, d] == kc[d]          # K: [block, head, token, dim]
                assert v[blk, h, d, off] == vc[d]          # V: [block, head, dim, token]
        written.add((blk, off))
    for blk in range(w.num_blocks):                        # everything else untouched
        for off in range(w.block_size):
            if (blk, off) not in written:
                assert np.array_equal(k[blk, :, off, :], w.k_codes[blk, :, off, :])
                assert np.array_equal(v[blk, :, :, off], w.v_codes[blk, :, :, off])
    pad = w.slot_mapping.copy()
    pad[0] = -1
    k2, _ = f.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, pad,
                                w.k_scale, w.v_scale, w.block_size)
    b0, o0 = divmod(int(w.slot_mapping[0]), w.block_size)
    assert np.array_equal(k2[b0, :, o0, :], w.k_codes[b0, :, o0, :])
    with pytest.raises(ValueError):
        f.reshape_and_cache(w.new_key[:2], w.new_value[:2], w.k_codes, w.v_codes,
                            np.array([pad[1], pad[1]]), w.k_scale, w.v_scale, w.block_size)


def pin_attention_reduces_to_bf16(f):
    """Power-of-two scales (different for K and V, and per head): dequantised values
    are exact bf16 values; FP8 attention must equal bf16 attention over them."""
    w = small_fp8(pow2=True)
    k, v = f.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                               w.k_scale, w.v_scale, w.block_size)
    kval = torch_decode(k) * w.k_scale[None, :, None, None]
    vval = torch_decode(v).transpose(0, 1, 3, 2) * w.v_scale[None, :, None, None]
    kb = W.f32_to_bf16_bits(kval.astype(np.float32))
    vb = W.f32_to_bf16_bits(vval.astype(np.float32))
    ref = O.paged_attention(w.q, kb, vb, w.block_tables, w.context_lens, w.scale,
                            w.num_kv_heads, w.block_size)
    got = f.paged_attention(w.q, k, v, w.k_scale, w.v_scale, w.block_tables, w.context_lens,
                            w.scale, w.num_kv_heads, w.block_size)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def pin_run_workload_reduces_to_bf16(f):
    """The whole FP8 step (quantised append of the new tokens, then attention) on a
    workload whose every value is exact equals the pinned bf16 oracle's step on the
    bf16 twin: outputs to 1e-12, and the appended slots hold exactly the twin's values
    (K and V scales differ, so mixing them up fails)."""
    w, twin = exact_fp8_case()
    got, k, v = f.run_workload(w)
    want, kb, vb = O.run_workload(twin)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)
    blk, off = np.divmod(w.slot_mapping, w.block_size)
    kval = torch_decode(k[blk, :, off, :]) * w.k_scale[None, :, None]
    vval = torch_decode(v[blk, :, :, off]) * w.v_scale[None, :, None]
    np.testing.assert_array_equal(kval, O.bf16_bits_to_f64(kb[blk, :, off, :]))
    np.testing.assert_array_equal(vval, O.bf16_bits_to_f64(vb[blk, :, off, :]))
    # only the named sequences are computed; the others stay NaN
    sub = f.run_workload(w, seqs=[1, 3])[0]
    np.testing.assert_array_equal(sub[[1, 3]], got[[1, 3]])
    assert np.isnan(sub[[0, 2]]).all()


PINS = [pin_decode_matches_torch, pin_encode_matches_torch, pin_encode_saturates_and_nan,
        pin_round_trip, pin_quantize_divides_in_float32, pin_reshape_layout,
        pin_attention_reduces_to_bf16, pin_run_workload_reduces_to_bf16]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(F)


def test_values_exact_in_bf16_when_scale_is_power_of_two():
    """Every E4M3 value times 2^k (k in -8..0) is a bf16 value: the reduction above is exact."""
    vals = torch_decode(ALL_CODES[:0x7F])
    for k in range(-8, 1):
        x = (vals * 2.0 ** k).astype(np.float32)
        back = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
        assert np.array_equal(back, x)


# ----------------------------------------------------------------------------- planted mistakes

class Mutant:
    """The fp8 oracle module with some globals replaced (the real module is untouched)."""

    def __init__(self, **overrides):
        self._o = overrides

    def __getattr__(self, name):
        if name in self._o:
            return self._o[name]
        f = getattr(F, name)
        if isinstance(f, types.FunctionType) and f.__module__ == F.__name__:
            g = dict(f.__globals__)
            g.update(self._o)
            return types.FunctionType(f.__code__, g, f.__name__, f.__defaults__, f.__closure__)
        return f


def _table(fn):
    return np.array([fn(c) for c in range(256)])


def _bias8(c):
    return F.e4m3_value(c) / 2.0


def _subnormal_as_normal(c):
    e, m = (c >> 3) & 15, c & 7
    if e == 0:
        return (-1.0 if c & 0x80 else 1.0) * (1 + m / 8) * 2.0 ** -7
    return F.e4m3_value(c)


def _encode_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    vals = F.DECODE_TABLE[:0x7F]
    hi = np.minimum(np.searchsorted(vals, a), 0x7E)
    lo = np.maximum(hi - 1, 0)
    code = np.where(vals[hi] - a <= a - vals[lo], hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def _encode_no_saturation(x):
    x = np.asarray(x, dtype=np.float64)
    c = F.encode(x)
    return np.where(np.abs(x) > 448.0, np.uint8(0x7F), c).astype(np.uint8)


def _encode_drops_sign(x):
    return F.encode(np.abs(np.asarray(x, dtype=np.float64)))


def _quantize_multiplies(bits, scale):
    return F.encode((O.bf16_bits_to_f64(bits).astype(np.float32) * np.float32(scale)))


def _quantize_in_f64(bits, scale):
    return F.encode(O.bf16_bits_to_f64(bits) / float(scale))


def _gather_v_with_k_layout(v_codes, row, L, g, v_scale, bs):
    pos = np.arange(L)
    phys = np.asarray(row)[pos // bs]
    return F.decode(v_codes[phys, g, :, :].reshape(L, -1)[:, : v_codes.shape[2]]) * float(
        v_scale[g])


def _gather_v_twice_scaled(v_codes, row, L, g, v_scale, bs):
    return 2.0 * F.gather_v(v_codes, row, L, g, v_scale, bs)


def _run_scales_swapped(w, seqs=None):
    k, v = F.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                               w.v_scale, w.k_scale, w.block_size)
    return F.paged_attention(w.q, k, v, w.v_scale, w.k_scale, w.block_tables, w.context_lens,
                             w.scale, w.num_kv_heads, w.block_size, seqs=seqs), k, v


def _run_no_append(w, seqs=None):
    k, v = w.k_codes, w.v_codes
    return F.paged_attention(w.q, k, v, w.k_scale, w.v_scale, w.block_tables, w.context_lens,
                             w.scale, w.num_kv_heads, w.block_size, seqs=seqs), k, v


def _run_append_scales_swapped(w, seqs=None):
    k, v = F.reshape_and_cache(w.new_key, w.new_value, w.k_codes, w.v_codes, w.slot_mapping,
                               w.v_scale, w.k_scale, w.block_size)
    return F.paged_attention(w.q, k, v, w.k_scale, w.v_scale, w.block_tables, w.context_lens,
                             w.scale, w.num_kv_heads, w.block_size, seqs=seqs), k, v


MUTANTS = {
    "run_workload_scales_swapped": dict(run_workload=_run_scales_swapped),
    "run_workload_no_append": dict(run_workload=_run_no_append),
    "run_workload_append_scales_swapped": dict(run_workload=_run_append_scales_swapped),
    "exponent_bias_8": dict(DECODE_TABLE=_table(_bias8)),
    "subnormal_as_normal": dict(DECODE_TABLE=_table(_subnormal_as_normal)),
    "ties_away_from_zero": dict(encode=_encode_ties_away),
    "no_saturation": dict(encode=_encode_no_saturation),
    "sign_dropped": dict(encode=_encode_drops_sign),
    "quantize_multiplies": dict(quantize=_quantize_multiplies),
    "quantize_in_fp64": dict(quantize=_quantize_in_f64),
    "v_pages_not_transposed": dict(gather_v=_gather_v_with_k_layout),
    "v_scale_wrong": dict(gather_v=_gather_v_twice_scaled),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    m = Mutant(**MUTANTS[name])
    failed = []
    for pin in PINS:
        try:
            pin(m)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
