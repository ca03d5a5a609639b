"""The sliding-window byte count the benchmark reports equals a brute-force count of
the (block, kv head) pages that hold at least one position some query row sees,
taken from the window oracle's visible ranges; a window covering every context
gives the plain count."""
import numpy as np
import pytest

import bench
import workloads as W
from oracle import window as WIN


def brute_pages(w, window):
    used = set()
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        for t in range(w.num_query_tokens):
            first, last = WIN.visible_range(L, w.num_query_tokens, t, window)
            for pos in range(first, last + 1):
                used.add(int(w.block_tables[b, pos // w.block_size]))
    return len(used) * w.num_kv_heads * w.page_bytes()


@pytest.mark.parametrize("name", ["decode_8b", "spec_verify", "decode_70b", "tiny"])
@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 1000])
def test_window_bytes_match_brute_force(name, window):
    w = W.SMALL[name]()
    assert bench.window_kv_bytes(w, window) == brute_pages(w, window)


@pytest.mark.parametrize("name", ["decode_8b", "spec_verify", "decode_70b"])
def test_covering_window_is_the_plain_count(name):
    w = W.SMALL[name]()
    assert bench.window_kv_bytes(w, int(w.context_lens.max())) == w.kv_bytes()


def test_fp8_pages_halve_the_window_bytes():
    w = W.SMALL["spec_verify"]()
    w8 = W.fp8_variant(w, seed=1)
    assert 2 * bench.window_kv_bytes(w8, 64) == bench.window_kv_bytes(w, 64)
    assert np.array_equal(w8.block_tables, w.block_tables)
