"""The C-ABI library builds, loads on a machine without a GPU, exports every symbol declared in
include/kv_nvfp4.h, and rejects bad host arguments before touching CUDA (CPU only)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kv():
    from bit_kv_cache_03_gb300 import build
    build.build()
    import bit_kv_cache_03_gb300 as kv
    kv.lib()
    return kv


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kv_nvfp4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(kv):
    names = declared_functions()
    assert len(names) >= 12
    raw = ctypes.CDLL(kv.library_path())
    for n in names:
        assert hasattr(raw, n), f"{n} declared in the header but not exported"


def test_page_and_pool_bytes(kv):
    L = kv.make_layout()
    assert kv.kv_nvfp4_page_bytes(L) == 64 * 144 * 4 == 36864
    n = kv.kv_nvfp4_pool_bytes(L, 10)
    assert n == 10 * 36864 and n // (10 * 4 * 64) == 144


@pytest.mark.parametrize("bad", [dict(head_dim=64), dict(page_size=32), dict(num_q_heads=10),
                                 dict(num_q_heads=8192, num_kv_heads=4), dict(rot_dim=30),
                                 dict(rot_dim=136), dict(num_kv_heads=0)])
def test_layout_rejected(kv, bad):
    args = dict(num_q_heads=24, num_kv_heads=4, head_dim=128, page_size=64, rot_dim=32)
    args.update(bad)
    L = kv.Layout(**args)
    assert kv.lib().kv_nvfp4_layout_check(ctypes.byref(L)) == kv.KV_NVFP4_EINVAL


def test_rope_host_table_bit_identical_to_oracle(kv):
    for scale in (1.0, 600000.0 / 262144.0):
        t = np.empty((5000, 32), np.float32)
        kv.kv_nvfp4_rope_table_fill_host(t, 5000, 32, 1e7, scale)
        ref = oracle.rope_table(5000, 32, 1e7, scale)
        assert np.array_equal(t.view(np.uint32), ref.view(np.uint32))


def test_plan_sizes_and_validation(kv):
    L = kv.make_layout()
    n = kv.kv_nvfp4_plan_workspace_bytes(L, [4097], 1, True, 1024)
    assert n > 0
    # 4 x 131073 tokens, 4 groups spread over many CTAs: every group is split, one partial of
    # 4 heads x 4160 B per segment
    n2 = kv.kv_nvfp4_plan_workspace_bytes(L, [131073] * 4, 1, True, 1024)
    assert n2 >= 4 * 2 * 4 * 4160
    lib = kv.lib()
    sl = np.array([5, 3], np.int32)
    size = ctypes.c_size_t()
    # seq_len < q_len, chunk not a multiple of 64, null workspace: all rejected without CUDA
    assert lib.kv_nvfp4_plan_workspace_bytes(ctypes.byref(L), sl.ctypes.data, 2, 4, 1, 1024,
                                             ctypes.byref(size)) == kv.KV_NVFP4_EINVAL
    assert lib.kv_nvfp4_plan_workspace_bytes(ctypes.byref(L), sl.ctypes.data, 2, 1, 1, 100,
                                             ctypes.byref(size)) == kv.KV_NVFP4_EINVAL
    info = kv.PlanInfo()
    assert lib.kv_nvfp4_plan(ctypes.byref(L), sl.ctypes.data, 2, 1, 1, 1024, None, 0,
                             ctypes.byref(info), None) == kv.KV_NVFP4_EINVAL


def test_entry_points_reject_bad_arguments_before_cuda(kv):
    lib = kv.lib()
    L = kv.make_layout()
    bad = kv.Layout(24, 4, 64, 64, 32)
    assert lib.kv_nvfp4_append(ctypes.byref(bad), *([None] * 5), 1, None, 1, None, 1, 1, 1,
                               *([None] * 5)) == kv.KV_NVFP4_EINVAL
    # null K pointer
    assert lib.kv_nvfp4_append(ctypes.byref(L), *([None] * 5), 1, None, 1, None, 1, 1, 1,
                               *([None] * 5)) == kv.KV_NVFP4_EINVAL
    # T = 0 is a no-op that needs no buffers
    assert lib.kv_nvfp4_append(ctypes.byref(L), *([None] * 5), 0, None, 1, None, 1, 1, 1,
                               *([None] * 5)) == kv.KV_NVFP4_OK
    info = kv.PlanInfo()
    assert lib.kv_nvfp4_decode_attn(ctypes.byref(L), ctypes.byref(info), None, None, None,
                                    0.0, None, 1, None, 1, None, None, None) == kv.KV_NVFP4_EINVAL
    # more than four KV heads per page is rejected by the attention entry point
    L8 = kv.make_layout(8, 8)
    assert lib.kv_nvfp4_decode_attn(ctypes.byref(L8), ctypes.byref(info), None, None, None,
                                    0.0, None, 1, None, 1, None, None, None) == kv.KV_NVFP4_EINVAL
    assert kv.lib().kv_nvfp4_status_string(-1) == b"invalid argument"


@pytest.mark.parametrize("lens,q_len,causal,chunk,ctas,Hq,Hkv", [
    ([131073] * 4, 1, True, 64, 152, 24, 4), ([131073] * 4, 1, True, 1024, 152, 24, 4),
    ([5, 70, 1000, 200000], 1, True, 1024, 152, 24, 4), ([100008] * 4, 8, True, 1024, 152, 24, 4),
    ([3], 1, True, 64, 152, 24, 4), ([600064], 8192, True, 64, 152, 24, 4),
    ([2000, 37], 8, False, 256, 7, 24, 4), ([900, 3000], 5, True, 128, 11, 9, 3),
    ([70, 4000], 3, True, 64, 20, 8, 1), ([500], 1, True, 64, 9, 9, 3),
    ([3000, 70], 1, True, 128, 30, 24, 8), ([3000, 70], 1, True, 128, 30, 64, 4),
    ([900], 2, True, 64, 13, 40, 5),
])
def test_plan_covers_every_visible_page_once_and_balances(kv, lens, q_len, causal, chunk, ctas,
                                                          Hq, Hkv):
    L = kv.make_layout(Hq, Hkv)
    info, groups, segs, cta, split = kv.kv_nvfp4_plan_host(L, lens, q_len, causal, chunk, ctas)
    G = Hq // Hkv
    # at most 8 rows per KV head and at most 4 KV heads: 8-row tiles over every head; otherwise
    # 128-row tiles per KV head
    tile_rows, n_pairs = (8, 1) if G * q_len <= 8 and Hkv <= 4 else (128, Hkv)
    n_rg = (G * q_len + tile_rows - 1) // tile_rows
    assert info.num_row_groups == n_rg
    assert info.num_groups == len(lens) * n_pairs * n_rg == len(groups)
    # expected visited pages per group: up to the last key any row of the tile can see
    gi = np.arange(len(groups))
    s_, pr_, rg_ = groups[:, 0], groups[:, 1], groups[:, 2]
    assert np.all((pr_ >= 0) & (pr_ < n_pairs))
    assert np.array_equal(gi, (s_ * n_pairs + pr_) * n_rg + rg_)
    assert np.array_equal(groups[:, 3], np.asarray(lens)[s_])
    last_row = np.minimum(G * q_len - 1, tile_rows * rg_ + tile_rows - 1)
    vis = (groups[:, 3] - q_len + last_row // G + 1) if causal else groups[:, 3]
    assert np.array_equal(groups[:, 6], (vis + 63) // 64)
    # segments tile each group's [0, pages) exactly, in order, cut only at chunk boundaries
    cp = chunk // 64
    covered = {}
    for g, lo, hi, part in segs:
        assert lo < hi
        assert lo % cp == 0 and (hi % cp == 0 or hi == groups[g][6])
        covered.setdefault(g, []).append((lo, hi))
    for gi, rngs in covered.items():
        assert rngs[0][0] == 0 and rngs[-1][1] == groups[gi][6]
        assert all(a[1] == b[0] for a, b in zip(rngs, rngs[1:]))
        assert len(rngs) == groups[gi][4]
    assert set(covered) == set(range(info.num_groups))
    # CTA ranges are contiguous; per-CTA load within one chunk of the mean (the tile plan charges
    # each segment ten pages for its fixed costs and balances pages plus charges)
    assert cta[0] == 0 and cta[-1] == info.num_segments and np.all(np.diff(cta) >= 0)
    seg_pages = (segs[:, 2] - segs[:, 1]).astype(np.int64)
    csum = np.concatenate([[0], np.cumsum(seg_pages)])
    load = csum[cta[1:]] - csum[cta[:-1]]
    assert load.sum() == info.total_pages
    if tile_rows == 128:
        cost = load + 10 * np.diff(cta)
        assert cost.max() <= cost.sum() / info.grid + cp + 10 + 1
    else:
        mean = info.total_pages / info.grid
        assert load.max() <= mean + cp + 1
    # partial slots: split groups get contiguous slots, unsplit groups none
    by_group = {}
    for seg in segs:
        by_group.setdefault(int(seg[0]), []).append(int(seg[3]))
    for gi, (s, h, rg, ln, nseg, fp, pages, _) in enumerate(groups):
        parts = by_group[gi]
        if nseg > 1:
            assert parts == list(range(fp, fp + nseg))
        else:
            assert parts == [-1]
    # the merge launch's work list: exactly the split groups, in group order
    assert np.array_equal(split, np.flatnonzero(groups[:, 4] > 1))
    assert info.num_split_groups == len(split)
    assert info.off_split % 16 == 0 and info.off_partials % 16 == 0
    # one (m, l, O) partial per slot: rows x (128 + 2) floats for every KV head the group covers
    heads = 1 if tile_rows == 128 else Hkv
    part_bytes = heads * tile_rows * 130 * 4
    assert info.workspace_bytes >= info.off_partials + info.num_partials * part_bytes
    assert info.workspace_bytes < info.off_partials + info.num_partials * part_bytes + 256


def test_spill_restore_reject_bad_arguments_before_cuda(kv):
    lib = kv.lib()
    L = kv.make_layout()
    OK, EINVAL = kv.KV_NVFP4_OK, kv.KV_NVFP4_EINVAL
    # no pages: nothing to do, no buffer needed
    assert lib.kv_nvfp4_spill_pages(ctypes.byref(L), None, 1, None, 0, None, None, None) == OK
    assert lib.kv_nvfp4_restore_pages(ctypes.byref(L), None, None, 0, None, 1, None, None) == OK
    # negative count, null buffers, misaligned arena or pool, empty pool, bad layout
    assert lib.kv_nvfp4_spill_pages(ctypes.byref(L), 256, 4, 512, -1, 768, None, None) == EINVAL
    assert lib.kv_nvfp4_spill_pages(ctypes.byref(L), None, 4, 512, 2, 768, None, None) == EINVAL
    assert lib.kv_nvfp4_spill_pages(ctypes.byref(L), 256, 4, None, 2, 768, None, None) == EINVAL
    assert lib.kv_nvfp4_spill_pages(ctypes.byref(L), 256, 4, 512, 2, None, None, None) == EINVAL
    assert lib.kv_nvfp4_spill_pages(ctypes.byref(L), 256, 4, 512, 2, 777, None, None) == EINVAL
    assert lib.kv_nvfp4_spill_pages(ctypes.byref(L), 260, 4, 512, 2, 768, None, None) == EINVAL
    assert lib.kv_nvfp4_spill_pages(ctypes.byref(L), 256, 0, 512, 2, 768, None, None) == EINVAL
    assert lib.kv_nvfp4_restore_pages(ctypes.byref(L), 776, 512, 2, 256, 4, None, None) == EINVAL
    bad = kv.Layout(24, 4, 64, 64, 32)
    assert lib.kv_nvfp4_restore_pages(ctypes.byref(bad), 768, 512, 2, 256, 4, None, None) == EINVAL


def test_comparator_sizes_and_rejections_before_cuda(kv):
    lib = kv.lib()
    L = kv.make_layout()
    # per token per KV head: 512 (bf16), 264 (int8), 328 (NVFP4 K + fp16 V); 64 tokens x 4 heads
    assert [kv.kv_cmp_page_bytes(L, f) for f in (0, 1, 2)] == [64 * 4 * b for b in (512, 264, 328)]
    assert kv.kv_cmp_page_bytes(L, 3) == 0
    info = kv.PlanInfo()
    EINVAL = kv.KV_NVFP4_EINVAL
    assert lib.kv_cmp_append(ctypes.byref(L), 5, *([None] * 5), 1, None, 1, None, 1, 1, 1,
                             *([None] * 4)) == EINVAL
    assert lib.kv_cmp_append(ctypes.byref(L), 0, *([None] * 5), 0, None, 1, None, 1, 1, 1,
                             *([None] * 4)) == kv.KV_NVFP4_OK  # nothing to append
    assert lib.kv_cmp_decode_attn(ctypes.byref(L), 0, ctypes.byref(info), None, None, 0.0, None,
                                  1, None, 1, None, None, None) == EINVAL
    assert lib.kv_cmp_decode_attn(ctypes.byref(L), 7, ctypes.byref(info), 256, 256, 0.0, 256,
                                  1, 256, 1, 256, None, None) == EINVAL
    n = kv.kv_cmp_plan_workspace_bytes(L, [131073] * 4, 1, True, 64)
    assert n > 0


def test_noalloc_buffer_size_matches_the_header(kv):
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                            "kv_nvfp4.h")).read()
    m = re.search(r"#define KV_NVFP4_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", hdr)
    assert m is not None
    assert int(m.group(1)) << int(m.group(2)) == kv.NOALLOC_SCRATCH_BYTES
    # on a 152-SM GPU the tile-kernel plans of the verify shape (4 x 100,008 tokens, 8 new each)
    # and of the 600k prefill chunk fit the buffer
    L = kv.make_layout()
    for lens, q_len in (([100008] * 4, 8), ([600064], 8192)):
        info = kv.kv_nvfp4_plan_host(L, lens, q_len, True, 1024, 152)[0]
        assert info.workspace_bytes <= kv.NOALLOC_SCRATCH_BYTES


def test_decode_step_host_rejects_bad_arguments_before_cuda(kv):
    lib = kv.lib()
    L = kv.make_layout()
    sl = np.array([100, 200], np.int32)
    info = kv.PlanInfo()
    args = lambda q_len, hq: (ctypes.byref(L), sl.ctypes.data, 2, q_len, 1, 64, 256, 1 << 20, hq,
                              512, 768, 1024, 1280, 1536, 1792, 1000, 2048, 4, 8, 2304, 0.0, 2560,
                              2816, None, ctypes.byref(info), None)
    EINVAL = kv.KV_NVFP4_EINVAL
    assert lib.kv_nvfp4_decode_step_host(*args(1, None)) == EINVAL      # no host Q
    assert lib.kv_nvfp4_decode_step_host(*args(2, 256)) == EINVAL       # 12 rows per KV head
    bad = kv.Layout(24, 4, 64, 64, 32)
    a = list(args(1, 256))
    a[0] = ctypes.byref(bad)
    assert lib.kv_nvfp4_decode_step_host(*a) == EINVAL                  # head_dim 64
    a = list(args(1, 256))
    a[6] = 264                                                         # misaligned workspace
    assert lib.kv_nvfp4_decode_step_host(*a) == EINVAL


@pytest.mark.parametrize("lens,q_len,causal,chunk,ctas,Hq,Hkv", [
    ([2000, 37], 8, False, 256, 7, 24, 4), ([900, 3000], 5, True, 128, 11, 9, 3),
    ([5000, 300, 2100], 8, True, 128, 16, 24, 4), ([700], 16, True, 64, 5, 24, 4),
    ([4100, 4100], 8, True, 512, 9, 24, 4), ([1500, 20, 640], 12, False, 128, 13, 16, 2),
])
def test_tile_plan_minimises_the_largest_cta_cost(kv, lens, q_len, causal, chunk, ctas, Hq, Hkv):
    # The tile plan's CTAs cover the chunk stream (groups in order, each cut into chunks) in
    # contiguous ranges; a CTA costs its pages plus ten per segment (one segment per group it
    # touches). An exact dynamic program over all contiguous splits into at most `grid` ranges
    # gives the smallest possible largest cost, which the plan must reach.
    L = kv.make_layout(Hq, Hkv)
    info, groups, segs, cta, split = kv.kv_nvfp4_plan_host(L, lens, q_len, causal, chunk, ctas)
    assert (Hq // Hkv) * q_len > 8  # the tile kernel's plan
    cp = chunk // 64
    chunks = [(g, min(cp, int(groups[g][6]) - lo))
              for g in range(len(groups)) for lo in range(0, int(groups[g][6]), cp)]
    n, grid, inf = len(chunks), int(info.grid), float("inf")
    # cost[i][j]: one CTA taking chunks i .. j - 1
    cost = [[0] * (n + 1) for _ in range(n + 1)]
    for i in range(n):
        pages, segs_in = 0, 0
        for j in range(i + 1, n + 1):
            g, pg = chunks[j - 1]
            pages += pg
            segs_in += 1 if (j - 1 == i or chunks[j - 2][0] != g) else 0
            cost[i][j] = pages + 10 * segs_in
    best = [0.0] + [inf] * n  # best[j]: chunks[:j] over the CTAs so far
    for _ in range(grid):
        nxt = best[:]  # a CTA may stay empty
        for j in range(1, n + 1):
            nxt[j] = min(nxt[j], min(max(best[i], cost[i][j]) for i in range(j)))
        best = nxt
    seg_cost = (segs[:, 2] - segs[:, 1]).astype(np.int64) + 10
    csum = np.concatenate([[0], np.cumsum(seg_cost)])
    plan_max = int((csum[cta[1:]] - csum[cta[:-1]]).max())
    assert plan_max == best[n], (plan_max, best[n])
