"""Block manager and copy-on-write: the oracle against the definition, the native
manager against the oracle, and the waste of paged versus contiguous allocation."""
import json
import os
import random

import numpy as np
import pytest

import __graft_entry__
from oracle import accounting
from oracle import block_manager as OBM
from paged_kv_cache_221_gb300 import _lib

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BS = 16


def random_ops(seed, n_ops=400, num_blocks=64):
    """A reproducible random mix of add / fork / append / free operations."""
    rng = random.Random(seed)
    ops, live, next_id = [], [], 0
    for _ in range(n_ops):
        r = rng.random()
        if not live or r < 0.12:
            ops.append(("add", next_id, rng.randint(0, 70)))
            live.append(next_id)
            next_id += 1
        elif r < 0.25:
            ops.append(("fork", rng.choice(live), next_id))
            live.append(next_id)
            next_id += 1
        elif r < 0.32 and len(live) > 1:
            s = rng.choice(live)
            ops.append(("free", s))
            live.remove(s)
        else:
            ops.append(("append", rng.choice(live)))
    return ops, num_blocks


class ContentModel:
    """What each sequence must read back: its own token history (values are unique)."""

    def __init__(self):
        self.hist = {}
        self.counter = 0

    def new_token(self):
        self.counter += 1
        return self.counter


def run_oracle_with_content(ops, num_blocks):
    """Apply ops to the oracle manager and to a pool of token values; check every
    sequence reads exactly its own history through its table after every op."""
    bm = OBM.BlockManager(num_blocks, BS)
    pool = np.zeros(num_blocks * BS, dtype=np.int64)
    cm = ContentModel()
    trace = []
    for op in ops:
        try:
            if op[0] == "add":
                bm.add_sequence(op[1], op[2])
                vals = [cm.new_token() for _ in range(op[2])]
                for j, val in enumerate(vals):
                    pool[bm.tables[op[1]][j // BS] * BS + j % BS] = val
                cm.hist[op[1]] = vals
                trace.append(("add", "ok"))
            elif op[0] == "fork":
                bm.fork(op[1], op[2])
                cm.hist[op[2]] = list(cm.hist[op[1]])
                trace.append(("fork", "ok"))
            elif op[0] == "append":
                slot, copy = bm.append_slot(op[1])
                if copy is not None:
                    src, dst = copy
                    pool[dst * BS:(dst + 1) * BS] = pool[src * BS:(src + 1) * BS]
                val = cm.new_token()
                pool[slot] = val
                cm.hist[op[1]].append(val)
                trace.append(("append", slot, copy))
            else:
                bm.free_sequence(op[1])
                del cm.hist[op[1]]
                trace.append(("free", "ok"))
        except OBM.OutOfBlocks:
            trace.append((op[0], "out_of_blocks"))
            continue
        except ValueError:          # an op on a sequence whose add ran out of blocks
            trace.append((op[0], "invalid"))
            continue
        # the definition: every live sequence sees exactly its own tokens
        for seq, hist in cm.hist.items():
            table = bm.tables[seq]
            assert len(table) == -(-len(hist) // BS)
            got = [pool[table[j // BS] * BS + j % BS] for j in range(len(hist))]
            assert got == hist, (op, seq)
        # bookkeeping invariants
        listed = [b for t in bm.tables.values() for b in t]
        assert sum(bm.refs) == len(listed)
        for b, r in enumerate(bm.refs):
            assert r == listed.count(b)
    return bm, trace


@pytest.mark.parametrize("seed", range(6))
def test_oracle_block_manager_meets_the_definition(seed):
    ops, nb = random_ops(seed)
    bm, trace = run_oracle_with_content(ops, nb)
    assert any(t[0] == "append" and len(t) == 3 and t[2] is not None for t in trace), \
        "the op mix must exercise copy-on-write"
    for seq in list(bm.tables):
        bm.free_sequence(seq)
    assert len(bm.free_blocks()) == nb


def test_planted_mistake_no_copy_on_write_is_caught():
    """A manager that writes into shared blocks without copying breaks the definition."""
    class NoCow(OBM.BlockManager):
        def append_slot(self, seq):
            table = self.tables[seq]
            pos = self.tokens[seq]
            if pos % self.block_size == 0:
                table.append(self._new_block())
            self.tokens[seq] = pos + 1
            return table[-1] * self.block_size + pos % self.block_size, None

    ops, nb = random_ops(1)
    orig = OBM.BlockManager
    OBM.BlockManager = NoCow
    try:
        with pytest.raises(AssertionError):
            run_oracle_with_content(ops, nb)
    finally:
        OBM.BlockManager = orig


# ----------------------------------------------------------------------------- block copy

def _copy_case(seed=5, nb=12, hkv=3, d=8):
    """Pools whose every element is distinct, and copy pairs (no destination is a source)."""
    rng = np.random.default_rng(seed)
    vals = rng.permutation(2 * nb * hkv * BS * d).astype(np.uint16)
    k = vals[:nb * hkv * BS * d].reshape(nb, hkv, BS, d)
    v = vals[nb * hkv * BS * d:].reshape(nb, hkv, BS, d)
    pairs = [(0, 7), (3, 4), (3, 9), (11, 2)]
    return k, v, pairs


def pin_copy_blocks_scalar(cb):
    """Every element of each destination block, both pools, equals the source's, read by
    scalar loops; every other block is unchanged, and the inputs are not modified."""
    k, v, pairs = _copy_case()
    k0, v0 = k.copy(), v.copy()
    kk, vv = cb(k, v, pairs)
    np.testing.assert_array_equal(k, k0)
    np.testing.assert_array_equal(v, v0)
    nb, hkv, bs, d = k.shape
    dst = {b for _, b in pairs}
    for src, b in pairs:
        for h in range(hkv):
            for o in range(bs):
                for x in range(d):
                    assert kk[b, h, o, x] == k0[src, h, o, x]
                    assert vv[b, h, o, x] == v0[src, h, o, x]
    for b in range(nb):
        if b not in dst:
            assert (kk[b] == k0[b]).all() and (vv[b] == v0[b]).all()


def pin_copy_blocks_empty(cb):
    k, v, _ = _copy_case(seed=6)
    kk, vv = cb(k, v, [])
    np.testing.assert_array_equal(kk, k)
    np.testing.assert_array_equal(vv, v)


COPY_PINS = [pin_copy_blocks_scalar, pin_copy_blocks_empty]


@pytest.mark.parametrize("pin", COPY_PINS, ids=[p.__name__ for p in COPY_PINS])
def test_copy_pin(pin):
    pin(OBM.copy_blocks)


def _copy_swapped(k_cache, v_cache, pairs):
    return OBM.copy_blocks(k_cache, v_cache, [(d, s) for s, d in pairs])


def _copy_k_only(k_cache, v_cache, pairs):
    k, _ = OBM.copy_blocks(k_cache, v_cache, pairs)
    return k, np.array(v_cache, copy=True)


def _copy_in_place(k_cache, v_cache, pairs):
    for s, d in pairs:
        k_cache[d] = k_cache[s]
        v_cache[d] = v_cache[s]
    return k_cache, v_cache


def _copy_first_head(k_cache, v_cache, pairs):
    k, v = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    for s, d in pairs:
        k[d, 0] = k_cache[s, 0]
        v[d, 0] = v_cache[s, 0]
    return k, v


COPY_MUTANTS = {"src_dst_swapped": _copy_swapped, "k_pool_only": _copy_k_only,
                "inputs_modified": _copy_in_place, "first_head_only": _copy_first_head}


@pytest.mark.parametrize("name", sorted(COPY_MUTANTS))
def test_copy_planted_mistake_is_caught(name):
    failed = []
    for pin in COPY_PINS:
        try:
            pin(COPY_MUTANTS[name])
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return _lib.load()


@pytest.mark.parametrize("seed", range(6))
def test_native_manager_matches_oracle(lib, seed):
    import paged_kv_cache_221_gb300 as pa
    ops, nb = random_ops(seed)
    o = OBM.BlockManager(nb, BS)
    n = pa.BlockManager(nb, BS)
    for op in ops:
        kind = op[0]
        try:
            if kind == "add":
                o.add_sequence(op[1], op[2])
            elif kind == "fork":
                o.fork(op[1], op[2])
            elif kind == "append":
                want = o.append_slot(op[1])
            else:
                o.free_sequence(op[1])
            o_err = None
        except OBM.OutOfBlocks:
            o_err = 7
        except ValueError:
            o_err = 1
        try:
            if kind == "add":
                n.add_sequence(op[1], op[2])
            elif kind == "fork":
                n.fork(op[1], op[2])
            elif kind == "append":
                got = n.append_slot(op[1])
            else:
                n.free_sequence(op[1])
            n_err = None
        except pa.PagedAttnError as e:
            n_err = e.status
        assert o_err == n_err, op
        if kind == "append" and o_err is None:
            assert got == want, op
        assert n.num_free_blocks() == len(o.free_blocks())
        for b in range(nb):
            assert n.ref_count(b) == o.refs[b]
        seqs = sorted(o.tables)
        if seqs:
            mb = max(len(t) for t in o.tables.values()) or 1
            tables, lens = n.block_table(seqs, mb)
            for i, s in enumerate(seqs):
                row = o.tables[s] + [-1] * (mb - len(o.tables[s]))
                assert tables[i].tolist() == row
                assert int(lens[i]) == o.tokens[s]
    n.close()


def test_native_manager_errors(lib):
    import paged_kv_cache_221_gb300 as pa
    m = pa.BlockManager(4, BS)
    m.add_sequence(1, 40)                   # 3 blocks
    with pytest.raises(pa.PagedAttnError) as e:
        m.add_sequence(2, 40)               # needs 3, 1 free
    assert e.value.status == 7
    assert m.num_free_blocks() == 1         # unchanged
    with pytest.raises(pa.PagedAttnError) as e:
        m.add_sequence(1, 1)                # duplicate id
    assert e.value.status == 1
    m.fork(1, 2)
    slot, copy = m.append_slot(2)           # 41st token into the shared third block
    assert copy is not None and copy[0] != copy[1]
    assert m.ref_count(copy[0]) == 1 and m.ref_count(copy[1]) == 1
    with pytest.raises(pa.PagedAttnError) as e:
        m.append_slot(1)                    # parent's block is private again; fits
        m.append_slot(3)                    # unknown sequence
    assert e.value.status == 1
    m.close()


def test_paged_waste_against_contiguous_reservation():
    """The fragmentation argument measured: contiguous max-length reservations
    waste most of the memory for short outputs; paged allocation wastes less
    than one block per sequence."""
    g = json.load(open(os.path.join(GOLDEN, "page_figures.json")))
    reserve = g["reservation_example"]["reserved_tokens"]
    rng = np.random.default_rng(0)
    lens = rng.integers(320, 4000, size=40)
    bm = OBM.BlockManager(int(sum(-(-lens // BS))), BS)
    for i, L in enumerate(lens):
        bm.add_sequence(i, int(L))
    allocated = sum(len(t) for t in bm.tables.values()) * BS
    paged_waste = 1 - lens.sum() / allocated
    contiguous_waste = 1 - lens.sum() / (reserve * len(lens))
    assert contiguous_waste > 0.9
    assert paged_waste < g["paged_waste_below"]["fraction"]
    assert accounting.reservation_unused_fraction(200, reserve) > 0.99
