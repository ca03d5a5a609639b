"""Parity of the FP8 (E4M3) page path (through the C ABI) with the fp64 FP8 oracle.

reshape_and_cache_fp8 is compared code for code over the whole pool.  Attention
outputs (bf16) must be within max abs error 1e-2 (or one bf16 ulp of the oracle
value, where that is larger) and relative L2 error 2e-3 of
attention over the dequantised pages in fp64.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import fp8 as F

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU-only hosts, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import __graft_entry__  # noqa: E402

__graft_entry__.build()

import paged_kv_cache_221_gb300 as pa  # noqa: E402
from gpu_util import assert_close, to_dev  # noqa: E402


@pytest.fixture(autouse=True)
def no_device_error():
    yield
    assert pa.get_device_error() == 0, "device error word was set"


class Dev8:
    """Device copies of an FP8 workload."""

    def __init__(self, w):
        self.w = w
        self.q = to_dev(w.q)
        self.k = to_dev(w.k_codes)
        self.v = to_dev(w.v_codes)
        self.ks = to_dev(w.k_scale)
        self.vs = to_dev(w.v_scale)
        self.tables = to_dev(w.block_tables)
        self.lens = to_dev(w.context_lens)
        self.new_key = to_dev(w.new_key)
        self.new_value = to_dev(w.new_value)
        self.slots = to_dev(w.slot_mapping)

    def reshape(self):
        pa.reshape_and_cache_fp8(self.new_key, self.new_value, self.k, self.v, self.slots,
                                 self.ks, self.vs)

    def attend(self, partition_size=None, workspace=None, out=None):
        w = self.w
        ps = w.partition_size if partition_size is None else partition_size
        return pa.verify_fp8(self.q, self.k, self.v, self.ks, self.vs, self.tables, self.lens,
                             w.max_context_len, w.scale, ps, workspace, out)

    def attend_append(self, partition_size=None):
        """reshape_and_cache_fp8 fused into the attention launch (pa_decode_append_fp8)."""
        w = self.w
        ps = w.partition_size if partition_size is None else partition_size
        return pa.verify_fp8(self.q, self.k, self.v, self.ks, self.vs, self.tables, self.lens,
                             w.max_context_len, w.scale, ps, None, None, self.new_key,
                             self.new_value)


def codes(t):
    return t.detach().cpu().numpy()


def fp8(name, size="small"):
    base = (W.SMALL if size == "small" else W.FULL)[name]()
    base.seq_group = None                    # FP8 pages: the per-sequence path
    base.group_prefix_blocks = None
    return W.fp8_variant(base, seed=len(name))


NAMES = ["tiny", "decode_8b", "decode_70b", "spec_verify", "shared_prefix"]


@pytest.mark.parametrize("name", NAMES)
def test_small_config_matches_oracle(name):
    w = fp8(name)
    ref, kref, vref = F.run_workload(w)
    d = Dev8(w)
    d.reshape()
    np.testing.assert_array_equal(codes(d.k), kref)
    np.testing.assert_array_equal(codes(d.v), vref)
    assert_close(d.attend(), ref, what=f"{name} fp8")


@pytest.mark.parametrize("name", ["decode_8b", "spec_verify", "decode_70b"])
@pytest.mark.parametrize("psize", [16, 48, 512, 0])
def test_partition_sizes(name, psize):
    w = fp8(name)
    ref, _, _ = F.run_workload(w)
    d = Dev8(w)
    d.reshape()
    assert_close(d.attend(partition_size=psize), ref, what=f"{name} fp8 psize {psize}")


EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 511, 512, 513]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("hq,hkv,T", [(4, 4, 1), (32, 8, 1), (64, 8, 1), (32, 8, 5), (16, 1, 4),
                                      (8, 2, 3)])
def test_edge_lengths_and_head_layouts(D, hq, hkv, T):
    lens = [max(L, T) for L in EDGE_LENS]
    base = W.build("edge8", lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=D,
                   num_query_tokens=T, seed=D + hq + T)
    w = W.fp8_variant(base, seed=D + T)
    ref, kref, vref = F.run_workload(w)
    d = Dev8(w)
    d.reshape()
    np.testing.assert_array_equal(codes(d.k), kref)
    np.testing.assert_array_equal(codes(d.v), vref)
    for ps in (16, 64, 0):
        assert_close(d.attend(partition_size=ps), ref, what=f"fp8 D{D} {hq}/{hkv} T{T} ps{ps}")


def test_every_code_in_the_pages():
    """Pages cycling through all 254 finite codes (subnormals, zeros, +-448) with
    power-of-two scales; K and V use different orders of the codes."""
    base = W.build("allcodes", [300, 64, 17], num_q_heads=8, num_kv_heads=2, head_dim=128,
                   seed=9)
    w = W.fp8_variant(base, seed=9)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    live = w.k_codes != W.NAN_E4M3
    w.k_codes[live] = np.resize(finite, int(live.sum()))
    live = w.v_codes != W.NAN_E4M3
    w.v_codes[live] = np.resize(finite[::-1], int(live.sum()))
    w.k_scale = np.array([2.0 ** -7, 2.0 ** -8], dtype=np.float32)
    w.v_scale = np.array([2.0 ** -6, 2.0 ** -9], dtype=np.float32)
    ref, _, _ = F.run_workload(w)
    d = Dev8(w)
    d.reshape()
    for ps in (32, 0):
        assert_close(d.attend(partition_size=ps), ref, what=f"all codes ps{ps}")


def test_quantisation_edge_values_bit_exact():
    """New values at ties, subnormals, saturation and signed zeros, quantised on the GPU
    exactly as the oracle's float32-divide-then-round rule."""
    rng = np.random.default_rng(12)
    N, Hkv, D = 64, 2, 128
    pos = F.decode(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    vals = np.concatenate([pos, -pos, mids, -mids, [500.0, -600.0, 1e30, -1e30, 0.0, -0.0,
                                                    1e-30, -1e-30, 2.0 ** -10, -(2.0 ** -10)]])
    vals = np.resize(vals, N * Hkv * D).astype(np.float32)
    rng.shuffle(vals)
    key = W.f32_to_bf16_bits(vals).reshape(N, Hkv, D)
    value = W.f32_to_bf16_bits(vals[::-1].copy()).reshape(N, Hkv, D)
    k_scale = np.array([1.0, 0.5], dtype=np.float32)           # exact ties survive the divide
    v_scale = np.array([0.25, 0.0137], dtype=np.float32)
    NB = 8
    kc = np.full((NB, Hkv, 16, D), 0x7F, dtype=np.uint8)
    vc = np.full((NB, Hkv, D, 16), 0x7F, dtype=np.uint8)
    slots = rng.permutation(NB * 16)[:N].astype(np.int64)
    kref, vref = F.reshape_and_cache(key, value, kc, vc, slots, k_scale, v_scale, 16)
    dk, dv = to_dev(kc), to_dev(vc)
    pa.reshape_and_cache_fp8(to_dev(key), to_dev(value), dk, dv, to_dev(slots),
                             to_dev(k_scale), to_dev(v_scale))
    np.testing.assert_array_equal(codes(dk), kref)
    np.testing.assert_array_equal(codes(dv), vref)


def _prefill_slots(rng, seq_lens, first_offsets, NB, pad_every=0):
    """Slot mapping of a prefill chunk: each sequence's tokens fill consecutive slots of
    distinct random blocks, starting at first_offsets[i] inside its first block; a
    padding token (-1) after every pad_every tokens when pad_every > 0."""
    blocks = list(rng.permutation(NB))
    slots = []
    for L, o in zip(seq_lens, first_offsets):
        pos = o
        blk = blocks.pop()
        for _ in range(L):
            if pos == 16:
                blk, pos = blocks.pop(), 0
            slots.append(blk * 16 + pos)
            pos += 1
            if pad_every and len(slots) % pad_every == 0:
                slots.append(-1)
    return np.array(slots, dtype=np.int64)


@pytest.mark.parametrize("D,hkv", [(128, 8), (128, 1), (64, 2), (96, 2)])
@pytest.mark.parametrize("layout", ["aligned", "offset", "padded"])
def test_prefill_chunk_code_for_code(D, hkv, layout):
    """A prefill chunk: runs of whole blocks written in order (16-byte transposed V rows)
    next to partial blocks, sequences that start at any token of a 32-token tile, and
    padding tokens, code for code against the oracle over the whole pool.  head_dim 96
    takes the byte-wise kernel."""
    rng = np.random.default_rng(D + hkv)
    lens = [48, 5, 16, 33, 70, 1, 17, 64, 31]
    offs = {"aligned": [0] * len(lens), "offset": [3, 0, 9, 15, 0, 7, 0, 1, 12],
            "padded": [0, 4, 0, 0, 2, 0, 0, 0, 5]}[layout]
    NB = 64
    slots = _prefill_slots(rng, lens, offs, NB, pad_every=37 if layout == "padded" else 0)
    N = len(slots)
    key = W.normal_bf16(rng, (N, hkv, D))
    value = W.normal_bf16(rng, (N, hkv, D))
    k_scale = rng.uniform(0.004, 0.03, size=hkv).astype(np.float32)
    v_scale = rng.uniform(0.004, 0.03, size=hkv).astype(np.float32)
    kc = np.full((NB, hkv, 16, D), 0x5A, dtype=np.uint8)
    vc = np.full((NB, hkv, D, 16), 0xA5, dtype=np.uint8)
    kref, vref = F.reshape_and_cache(key, value, kc, vc, slots, k_scale, v_scale, 16)
    dk, dv = to_dev(kc), to_dev(vc)
    pa.reshape_and_cache_fp8(to_dev(key), to_dev(value), dk, dv, to_dev(slots),
                             to_dev(k_scale), to_dev(v_scale))
    np.testing.assert_array_equal(codes(dk), kref)
    np.testing.assert_array_equal(codes(dv), vref)
    assert pa.get_device_error() == 0


def test_nan_input_stays_nan():
    key = np.full((1, 1, 64), 0x7FC0, dtype=np.uint16)           # bf16 NaN
    value = np.full((1, 1, 64), 0xFFC0, dtype=np.uint16)         # negative NaN
    kc = np.zeros((2, 1, 16, 64), dtype=np.uint8)
    vc = np.zeros((2, 1, 64, 16), dtype=np.uint8)
    dk, dv = to_dev(kc), to_dev(vc)
    one = to_dev(np.ones(1, dtype=np.float32))
    pa.reshape_and_cache_fp8(to_dev(key), to_dev(value), dk, dv,
                             to_dev(np.array([19], dtype=np.int64)), one, one)
    k, v = codes(dk), codes(dv)
    assert set(np.unique(k[1, 0, 3, :]).tolist()) <= {0x7F, 0xFF}
    assert set(np.unique(v[1, 0, :, 3]).tolist()) <= {0x7F, 0xFF}
    assert not k[0].any() and not v[0].any()


def test_constant_v_gives_one():
    """V codes all 1.0 with scale 1: the output is 1 up to the f16 rounding of P."""
    w = fp8("decode_8b")
    w.v_codes[w.v_codes != W.NAN_E4M3] = 0x38                   # 1.0
    w.v_scale = np.ones_like(w.v_scale)
    w.new_value = np.full_like(w.new_value, 0x3F80)              # bf16 1.0
    d = Dev8(w)
    d.reshape()
    for ps in (32, 0):
        out = d.attend(partition_size=ps).float()
        assert torch.isfinite(out).all()
        assert float((out - 1).abs().max()) <= 2e-3


def test_bad_block_id_reports_bounds():
    w = fp8("decode_8b")
    d = Dev8(w)
    d.reshape()
    d.tables[1, 2] = w.num_blocks + 7
    d.attend(partition_size=64)
    assert pa.get_device_error() == 5


def test_argument_errors():
    w = fp8("tiny")
    d = Dev8(w)
    with pytest.raises(ValueError):                         # V pages must be transposed
        pa.verify_fp8(d.q, d.k, d.k, d.ks, d.vs, d.tables, d.lens)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.verify_fp8(d.q, d.k, d.v, d.ks, d.vs, d.tables, d.lens, w.max_context_len, w.scale,
                      24)                                       # not a block multiple
    assert e.value.status == 1


@pytest.mark.parametrize("name", ["tiny", "decode_8b", "decode_70b", "spec_verify"])
@pytest.mark.parametrize("psize", [32, 0])
def test_append_matches_oracle(name, psize):
    """The fused append writes the same codes as reshape_and_cache_fp8 and attends correctly."""
    w = fp8(name)
    ref, kref, vref = F.run_workload(w)
    d = Dev8(w)
    out = d.attend_append(partition_size=psize)
    np.testing.assert_array_equal(codes(d.k), kref)
    np.testing.assert_array_equal(codes(d.v), vref)
    assert_close(out, ref, what=f"{name} fp8 append ps{psize}")


@pytest.mark.parametrize("D", [64, 128])
def test_append_edge_lengths(D):
    lens = [max(L, 3) for L in EDGE_LENS]
    base = W.build("edge8_append", lens, num_q_heads=16, num_kv_heads=4, head_dim=D,
                   num_query_tokens=3, seed=78 + D)
    w = W.fp8_variant(base, seed=5)
    ref, kref, vref = F.run_workload(w)
    d = Dev8(w)
    for ps in (16, 0):
        d = Dev8(w)
        out = d.attend_append(partition_size=ps)
        assert_close(out, ref, what=f"fp8 append edge D{D} ps{ps}")
    np.testing.assert_array_equal(codes(d.k), kref)
    np.testing.assert_array_equal(codes(d.v), vref)


def shared_fp8(size="small"):
    base = (W.SMALL if size == "small" else W.FULL)["shared_prefix"]()
    return W.fp8_variant(base, seed=13)


@pytest.mark.parametrize("psize", [128, 256, 0])
def test_shared_prefix_read_once(psize):
    """FP8 pages through the shared-prefix call: matches the oracle, and matches the
    per-sequence FP8 call within tolerance."""
    w = shared_fp8()
    ref, _, _ = F.run_workload(w)
    d = Dev8(w)
    d.reshape()
    sg, gp = to_dev(w.seq_group), to_dev(w.group_prefix_blocks)
    out = pa.decode_shared_prefix(d.q, d.k, d.v, d.tables, d.lens, sg, gp, w.max_group_size,
                                  w.max_prefix_blocks, w.max_context_len, w.scale, psize,
                                  k_scale=d.ks, v_scale=d.vs)
    assert_close(out, ref, what=f"fp8 shared prefix ps{psize}")
    plain = d.attend(partition_size=psize)
    assert_close(out, plain.float().cpu().double().numpy(), what="fp8 shared vs plain")


def _spread_queries(w, seed):
    """Query rows of very different magnitudes: each (sequence, token, head) row times
    2^e, e uniform in [-8, 3]; one row of zeros per sequence; and one row per sequence
    whose dims fall from 1 to 2^-20 of its largest.  Every row must keep its own
    scores through the query's conversion for the tensor cores (a per-row factor
    applied to the wrong row, or lost low-order parts, show here)."""
    rng = np.random.default_rng(seed)
    qf = (w.q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qf *= np.exp2(rng.integers(-8, 4, size=qf.shape[:3]))[..., None]
    qf[:, 0, 1, :] = 0.0
    qf[:, -1, 2, :] *= np.exp2(-np.arange(qf.shape[-1]) * 20.0 / qf.shape[-1])
    w.q = W.f32_to_bf16_bits(qf.astype(np.float32))
    return w


@pytest.mark.parametrize("D,T", [(128, 1), (128, 5), (64, 1), (64, 4), (128, 2)])
def test_query_rows_of_different_magnitudes(monkeypatch, D, T):
    """Both attention kernels on spread query rows: within tolerance of the oracle and
    bit-identical to each other."""
    lens = [max(L, T) for L in (300, 1000, 17, 2048, 513, 64, 5, 1500)]
    base = W.build("qmag", lens, num_q_heads=32, num_kv_heads=8, head_dim=D,
                   num_query_tokens=T, seed=D + 7 * T)
    w = _spread_queries(W.fp8_variant(base, seed=D + T), seed=D * T)
    ref, _, _ = F.run_workload(w)
    d = Dev8(w)
    d.reshape()
    for ps in (48, 0):
        outs = []
        for mode in ("per_unit", "persistent"):
            monkeypatch.setenv("PA_DECODE_KERNEL", mode)
            outs.append(d.attend(partition_size=ps))
            torch.cuda.synchronize()
        monkeypatch.delenv("PA_DECODE_KERNEL")
        for out in outs:
            assert_close(out, ref, what=f"fp8 query magnitudes D{D} T{T} ps{ps}")
        np.testing.assert_array_equal(outs[0].cpu().view(torch.int16).numpy(),
                                      outs[1].cpu().view(torch.int16).numpy())


def test_shared_prefix_query_rows_of_different_magnitudes():
    """The shared-prefix kernel (one CTA carries every member's rows) on spread rows."""
    w = _spread_queries(shared_fp8(), seed=5)
    ref, _, _ = F.run_workload(w)
    d = Dev8(w)
    d.reshape()
    sg, gp = to_dev(w.seq_group), to_dev(w.group_prefix_blocks)
    for psize in (128, 0):
        out = pa.decode_shared_prefix(d.q, d.k, d.v, d.tables, d.lens, sg, gp,
                                      w.max_group_size, w.max_prefix_blocks,
                                      w.max_context_len, w.scale, psize, k_scale=d.ks,
                                      v_scale=d.vs)
        assert_close(out, ref, what=f"fp8 shared prefix query magnitudes ps{psize}")


def test_default_partition_for_long_contexts():
    """FP8 pages past 4096-token contexts default to 4096-token partitions: a scratch
    sized for them is enough with partition_size 0 (the bf16 default, 2048 tokens,
    would need more and be refused), and the result is that of an explicit 4096."""
    w = fp8("spec_verify", "full")
    d = Dev8(w)
    d.reshape()
    need4096 = pa.workspace_size(w.num_seqs, w.num_q_heads, w.num_query_tokens,
                                 w.max_context_len, w.head_dim, 16, 4096, 0)
    need2048 = pa.workspace_size(w.num_seqs, w.num_q_heads, w.num_query_tokens,
                                 w.max_context_len, w.head_dim, 16, 2048, 0)
    assert need4096 < need2048
    ws = torch.empty(need4096, dtype=torch.uint8, device="cuda")
    out0 = d.attend(partition_size=0, workspace=ws)
    out4096 = d.attend(partition_size=4096, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out0.view(torch.int16), out4096.view(torch.int16))
