"""Page spill and restore on the GPU against the oracle (bit-exact), through the C ABI.

Source: prismix.dev/news/833001997676, section "Multi-level prefix reuse with host-KV safety
net" (cache pages moved out to host memory and back). The arena is page-locked host memory (the
kernel's own stores and loads cross the host link) or device memory; pageable memory is refused.
"""
import numpy as np
import pytest

import oracle
import synth
from kvrun import GpuRun

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _kv():
    import bit_kv_cache_03_gb300 as kv
    return kv


def _setup(kv_heads, num_pages, seed):
    kv = _kv()
    L = kv.make_layout(6 * kv_heads, kv_heads)
    pb = kv.kv_nvfp4_page_bytes(L)
    g = torch.Generator().manual_seed(seed)
    pool = torch.randint(0, 256, (num_pages * pb,), dtype=torch.uint8, generator=g).cuda()
    return kv, L, pb, pool


@pytest.mark.parametrize("kv_heads,num_pages,n", [(4, 50, 37), (1, 9, 9), (8, 20, 13), (4, 3000, 2500)])
def test_spill_matches_the_oracle(kv_heads, num_pages, n):
    kv, L, pb, pool = _setup(kv_heads, num_pages, 1 + n)
    rng = np.random.default_rng(n)
    ids = rng.integers(0, num_pages, size=n).astype(np.int32)  # repeats allowed
    arena = torch.full((n * pb,), 0x5A, dtype=torch.uint8).pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.kv_nvfp4_spill_pages(L, pool, num_pages, torch.from_numpy(ids).cuda(), n, arena, status)
    torch.cuda.synchronize()
    want = np.full(n * pb, 0x5A, np.uint8)
    assert oracle.spill_pages(pool.cpu().numpy(), num_pages, kv_heads, ids, want) == 0
    assert np.array_equal(arena.numpy(), want)
    assert int(status.item()) == 0


@pytest.mark.parametrize("kv_heads,num_pages,n", [(4, 40, 31), (2, 7, 7), (8, 16, 5)])
def test_restore_matches_the_oracle(kv_heads, num_pages, n):
    kv, L, pb, pool = _setup(kv_heads, num_pages, 100 + n)
    rng = np.random.default_rng(n + 7)
    ids = rng.permutation(num_pages)[:n].astype(np.int32)
    src = rng.integers(0, 256, size=n * pb, dtype=np.uint8)
    arena = torch.from_numpy(src).pin_memory()
    want = pool.cpu().numpy().copy()
    kv.kv_nvfp4_restore_pages(L, arena, torch.from_numpy(ids).cuda(), n, pool, num_pages)
    torch.cuda.synchronize()
    assert oracle.restore_pages(want, num_pages, kv_heads, ids, src) == 0
    assert np.array_equal(pool.cpu().numpy(), want)


def test_ids_outside_the_pool_are_flagged_and_skipped():
    kv, L, pb, pool = _setup(4, 6, 3)
    ids = np.array([2, -1, 6, 5], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    arena = torch.full((len(ids) * pb,), 0xC3, dtype=torch.uint8).pin_memory()
    d_ids = torch.from_numpy(ids).cuda()
    kv.kv_nvfp4_spill_pages(L, pool, 6, d_ids, len(ids), arena, status)
    torch.cuda.synchronize()
    want = np.full(len(ids) * pb, 0xC3, np.uint8)
    assert oracle.spill_pages(pool.cpu().numpy(), 6, 4, ids, want) == 2
    assert np.array_equal(arena.numpy(), want)
    assert int(status.item()) & kv.DEV_BAD_PAGE
    status.zero_()
    before = pool.cpu().numpy().copy()
    kv.kv_nvfp4_restore_pages(L, arena, d_ids, len(ids), pool, 6, status)
    torch.cuda.synchronize()
    assert oracle.restore_pages(before, 6, 4, ids, arena.numpy()) == 2
    assert np.array_equal(pool.cpu().numpy(), before)
    assert int(status.item()) & kv.DEV_BAD_PAGE


def test_device_arena_and_pageable_arena():
    kv, L, pb, pool = _setup(4, 10, 4)
    ids = torch.tensor([3, 1, 4], dtype=torch.int32, device="cuda")
    dev_arena = torch.zeros(3 * pb, dtype=torch.uint8, device="cuda")
    kv.kv_nvfp4_spill_pages(L, pool, 10, ids, 3, dev_arena)
    torch.cuda.synchronize()
    p = pool.view(10, pb)
    assert torch.equal(dev_arena.view(3, pb), p[[3, 1, 4]])
    pageable = np.zeros(3 * pb, np.uint8)  # not page-locked: refused before any launch
    with pytest.raises(kv.KVNVFP4Error, match=r"\(-1\)"):
        kv.kv_nvfp4_spill_pages(L, pool, 10, ids, 3, pageable)
    assert not pageable.any()


def test_attention_is_unchanged_after_pages_move_through_the_arena():
    # every page of the cache goes out to host memory and comes back at another page id; with the
    # block table renamed the same way, the decode output is bit-identical
    kv = _kv()
    w = synth.Workload("spill_move", [3000, 700, 65], q_len=1, seed=21, pool_pages=150)
    g = GpuRun(w)
    g.step(chunk_tokens=256)
    torch.cuda.synchronize()
    ref = g.output().copy()
    c = g.cache
    bt = c.block_table.cpu().numpy()
    used = np.concatenate([bt[s, :(int(w.seq_lens[s]) + 63) // 64] for s in range(w.num_seqs)])
    used = used.astype(np.int32)
    pb = kv.kv_nvfp4_page_bytes(c.layout)
    arena = torch.empty(len(used) * pb, dtype=torch.uint8).pin_memory()
    kv.kv_nvfp4_spill_pages(c.layout, c.pool, c.num_pages, torch.from_numpy(used).cuda(),
                            len(used), arena, c.status)
    free = np.setdiff1d(np.arange(c.num_pages), used)
    rng = np.random.default_rng(5)
    new_ids = rng.permutation(np.concatenate([free, used]))[:len(used)].astype(np.int32)
    c.pool.zero_()
    kv.kv_nvfp4_restore_pages(c.layout, arena, torch.from_numpy(new_ids).cuda(), len(used),
                              c.pool, c.num_pages, c.status)
    rename = dict(zip(used.tolist(), new_ids.tolist()))
    bt2 = bt.copy()
    for s in range(w.num_seqs):
        n = (int(w.seq_lens[s]) + 63) // 64
        bt2[s, :n] = [rename[int(x)] for x in bt[s, :n]]
    c.block_table.copy_(torch.from_numpy(bt2))
    c.plan(w.seq_lens, w.q_len, w.causal, 256)
    c.attend(g.q_codes, g.q_scales, g.out, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert np.array_equal(g.output(), ref)
    assert g.status() == 0


def test_full_cache_round_trip_at_the_bench_size():
    # the 8196 pages of the 4 x 131072-token cache, in the launch configuration the benchmark
    # times: out to a page-locked arena and back to a permutation of the page ids
    kv = _kv()
    w = synth.steady_decode()
    g = GpuRun(w)
    c = g.cache
    bt = c.block_table.cpu().numpy()
    used = np.concatenate([bt[s, :(int(w.seq_lens[s]) + 63) // 64] for s in range(w.num_seqs)])
    used = used.astype(np.int32)
    pb = kv.kv_nvfp4_page_bytes(c.layout)
    arena = torch.empty(len(used) * pb, dtype=torch.uint8).pin_memory()
    kv.kv_nvfp4_spill_pages(c.layout, c.pool, c.num_pages, torch.from_numpy(used).cuda(),
                            len(used), arena, c.status)
    torch.cuda.synchronize()
    pool = c.pool.view(c.num_pages, pb)
    a = arena.view(len(used), pb)
    rng = np.random.default_rng(0)
    for i in rng.choice(len(used), size=64, replace=False):  # sampled slots, byte for byte
        assert torch.equal(a[i], pool[int(used[i])].cpu())
    perm = rng.permutation(used).astype(np.int32)
    back = torch.zeros_like(c.pool)
    kv.kv_nvfp4_restore_pages(c.layout, arena, torch.from_numpy(perm).cuda(), len(used), back,
                              c.num_pages, c.status)
    torch.cuda.synchronize()
    got = back.view(c.num_pages, pb)
    assert torch.equal(got[torch.from_numpy(perm).long().cuda()], a.cuda())
    assert g.status() == 0
