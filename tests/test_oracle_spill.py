"""Pins for the oracle's page spill and restore (CPU only).

Source: prismix.dev/news/833001997676, section "Multi-level prefix reuse with host-KV safety net"
(cache pages copied out to host memory and back). The pins tie the oracle to things other than
its own code: the page size follows from the 144 bytes per token per KV head of the golden layout
file, a spill of pages 0..n-1 is the first n blocks of the pool (the pool is an array of page
blocks), and pages moved through an arena to other page ids, with the block table renamed to
match, read back through the independent paged-layout gather as the same rows.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "layout_bytes.json")


def _page_bytes(kv_heads):
    per_token_head = json.load(open(GOLDEN))["nvfp4"]  # 144 B: K and V codes + scales
    return per_token_head * 64 * kv_heads


def _pool(rng, num_pages, kv_heads):
    return rng.integers(0, 256, size=num_pages * _page_bytes(kv_heads), dtype=np.uint8)


@pytest.mark.parametrize("kv_heads", [1, 3, 4])
def test_spill_of_the_first_pages_is_the_start_of_the_pool(kv_heads):
    rng = np.random.default_rng(1)
    pool = _pool(rng, 7, kv_heads)
    n = 5
    arena = np.zeros(n * _page_bytes(kv_heads), np.uint8)
    assert oracle.spill_pages(pool, 7, kv_heads, np.arange(n), arena) == 0
    assert np.array_equal(arena, pool[:n * _page_bytes(kv_heads)])


def test_spill_follows_the_page_ids_and_repeats():
    rng = np.random.default_rng(2)
    H, P = 4, 9
    pb = _page_bytes(H)
    pool = _pool(rng, P, H)
    ids = np.array([8, 0, 3, 3, 5], np.int32)
    arena = np.zeros(len(ids) * pb, np.uint8)
    oracle.spill_pages(pool, P, H, ids, arena)
    for i, p in enumerate(ids):
        assert np.array_equal(arena[i * pb:(i + 1) * pb], pool[p * pb:(p + 1) * pb])


def test_round_trip_restores_exactly_the_spilled_pages():
    rng = np.random.default_rng(3)
    H, P = 2, 12
    pb = _page_bytes(H)
    pool = _pool(rng, P, H)
    ids = rng.permutation(P)[:7].astype(np.int32)
    arena = np.zeros(len(ids) * pb, np.uint8)
    oracle.spill_pages(pool, P, H, ids, arena)
    fresh = np.zeros_like(pool)
    assert oracle.restore_pages(fresh, P, H, ids, arena) == 0
    for p in range(P):
        want = pool[p * pb:(p + 1) * pb] if p in ids else np.zeros(pb, np.uint8)
        assert np.array_equal(fresh[p * pb:(p + 1) * pb], want)


def test_relocated_pages_read_back_as_the_same_rows_through_the_gather():
    # two sequences on scattered pages; every page they use goes out to the arena and comes back
    # at a new page id; with the block table renamed the same way, the gather (an independent
    # oracle function that knows the in-page layout) returns identical K/V codes and scales
    rng = np.random.default_rng(4)
    H, P = 4, 16
    pool = _pool(rng, P, H)
    bt = np.array([[11, 2, 7], [5, 14, 0]], np.int32)
    used = bt.reshape(-1)
    arena = np.zeros(len(used) * _page_bytes(H), np.uint8)
    oracle.spill_pages(pool, P, H, used, arena)
    new_ids = rng.permutation(P)[:len(used)].astype(np.int32)
    moved = np.zeros_like(pool)
    oracle.restore_pages(moved, P, H, new_ids, arena)
    rename = dict(zip(used.tolist(), new_ids.tolist()))
    bt2 = np.vectorize(rename.get)(bt).astype(np.int32)
    for seq in range(2):
        a = oracle.paged_gather(pool, P, H, bt, seq, 0, 3 * 64)
        b = oracle.paged_gather(moved, P, H, bt2, seq, 0, 3 * 64)
        for x, y in zip(a[:4], b[:4]):
            assert np.array_equal(x, y)
        assert a[4] == b[4] == 0


def test_ids_outside_the_pool_are_counted_and_skipped():
    rng = np.random.default_rng(5)
    H, P = 1, 4
    pb = _page_bytes(H)
    pool = _pool(rng, P, H)
    ids = np.array([1, -1, P, 2], np.int32)
    arena = np.full(len(ids) * pb, 0xAB, np.uint8)
    assert oracle.spill_pages(pool, P, H, ids, arena) == 2
    assert np.all(arena[pb:3 * pb] == 0xAB)  # slots of the bad ids left as they were
    assert np.array_equal(arena[:pb], pool[pb:2 * pb])
    assert np.array_equal(arena[3 * pb:], pool[2 * pb:3 * pb])
    before = pool.copy()
    src = rng.integers(0, 256, size=len(ids) * pb, dtype=np.uint8)
    assert oracle.restore_pages(pool, P, H, ids, src) == 2
    assert np.array_equal(pool[pb:2 * pb], src[:pb])
    assert np.array_equal(pool[2 * pb:3 * pb], src[3 * pb:])
    assert np.array_equal(pool[:pb], before[:pb]) and np.array_equal(pool[3 * pb:], before[3 * pb:])


def test_no_pages_is_a_no_op():
    pool = np.arange(_page_bytes(2) * 3, dtype=np.uint64).astype(np.uint8)
    before = pool.copy()
    arena = np.zeros(16, np.uint8)
    assert oracle.spill_pages(pool, 3, 2, np.zeros(0, np.int32), arena) == 0
    assert oracle.restore_pages(pool, 3, 2, np.zeros(0, np.int32), arena) == 0
    assert np.array_equal(pool, before) and not arena.any()
