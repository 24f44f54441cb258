"""Attention parity of the CUDA path against the oracle on small workloads (GPU)."""
import numpy as np
import pytest

import synth
from kvrun import MAX_ABS_TOL, REL_L2_TOL, GpuRun, OracleRun, attention_errors

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _check(w, chunk=None, steps=1):
    g = GpuRun(w)
    outs = []
    for _ in range(steps):
        g.step(chunk_tokens=chunk)
        torch.cuda.synchronize()
        outs.append(g.output())
    assert g.status() == 0
    ref = OracleRun(w).attention().reshape(outs[0].shape)
    for out in outs:
        max_abs, rel = attention_errors(out, ref)
        assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, (max_abs, rel)
    for out in outs[1:]:
        assert np.array_equal(out, outs[0])  # repeat calls on one workspace give the same result
    return outs[0], ref


@pytest.mark.parametrize("lens,q_len,causal,chunk", [
    ([0, 5, 63, 64, 65, 200, 1000], 1, True, 1024),
    ([0, 5, 63, 64, 65, 200, 1000], 1, True, 128),       # split-K with the ticket merge
    ([10, 700, 1500], 3, True, 192),
    ([10, 700, 1500], 3, False, 192),
    ([2000, 37], 8, True, 256),                          # verify-shaped: 48 rows, 6 row tiles
    ([5000], 1, True, 64),                               # one page per chunk, 79 chunks
])
def test_attention_small(lens, q_len, causal, chunk):
    w = synth.Workload("small", lens, q_len=q_len, causal=causal, seed=len(lens) + q_len,
                       chunk_tokens=chunk, pool_pages=sum((c + q_len + 63) // 64 for c in lens) + 5)
    _check(w, chunk=chunk, steps=2)


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (4, 4), (16, 2), (9, 3), (3, 3)])
def test_attention_other_group_sizes(Hq, Hkv):
    w = synth.Workload("groups", [300, 1200], q_len=2, seed=Hq * 10 + Hkv, q_heads=Hq,
                       kv_heads=Hkv, chunk_tokens=256)
    _check(w, chunk=256)


@pytest.mark.parametrize("Hq,Hkv,q_len", [
    (24, 8, 1), (48, 8, 1),     # 8 KV heads, GQA 3 and 6: the tile kernel (per KV-head pair)
    (48, 4, 1), (64, 4, 1),     # GQA 12 and 16: 12 and 16 rows per KV head
    (24, 8, 3), (40, 5, 2),     # more than one new token; an odd number of KV heads above 4
])
def test_attention_more_kv_heads_and_larger_groups(Hq, Hkv, q_len):
    w = synth.Workload("wide", [0, 700, 2100], q_len=q_len, seed=Hq + Hkv + q_len, q_heads=Hq,
                       kv_heads=Hkv, chunk_tokens=256)
    _check(w, chunk=256)


def test_fused_step_refuses_more_than_four_kv_heads():
    import bit_kv_cache_03_gb300 as kv
    w = synth.Workload("wide_fused", [300], q_len=1, seed=2, q_heads=24, kv_heads=8)
    g = GpuRun(w)
    g.cache.plan(w.seq_lens, w.q_len, w.causal, 256)
    with pytest.raises(kv.KVNVFP4Error, match=r"\(-1\)"):
        g.step_fused(plan=False)


def test_attention_position_scaling_and_full_rotation():
    w = synth.Workload("scaled", [3000], q_len=4, seed=5, rot_dim=128,
                       pos_scale=600000.0 / 262144.0, chunk_tokens=512)
    _check(w, chunk=512)


def test_attention_skips_bad_pages_and_flags_them():
    import bit_kv_cache_03_gb300 as kv
    w = synth.Workload("badpage", [500], q_len=1, seed=3, pool_pages=12)
    g = GpuRun(w)
    g.step()
    torch.cuda.synchronize()
    assert g.status() == 0
    # corrupt one entry of the block table, re-run attention only
    bt = g.cache.block_table
    bt[0, 2] = 10 ** 6
    g.cache.attend(g.q_codes, g.q_scales, g.out, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert g.status() & kv.DEV_BAD_PAGE
    assert np.all(np.isfinite(g.output()))


# More than 8 rows per KV head run on the tile kernel (tiles of 128 query rows of one KV head, both
# products on the tcgen05 tensor cores; tiles of at most 64 rows run in split-page mode).
@pytest.mark.parametrize("lens,q_len,causal,chunk", [
    ([300, 2000], 16, True, 256),        # 96 rows: a full 64-row tile and a ragged one
    ([257, 1000], 12, False, 128),       # 72 rows, every key visible
    ([3000], 256, True, 64),             # 1536 rows, 24 tiles per pair: many segments per CTA
    ([64, 65, 129], 2, True, 64),        # 12 rows; sequences ending on and just past a page
    ([4100], 11, True, 4160),            # one chunk per group: groups not split
    ([4000] * 4, 8, True, 128),          # split-page mode (48 rows), many blocks and segments per CTA
    ([3000, 1500], 8, False, 128),       # split-page mode, every key visible
    ([0, 1, 55, 56], 8, True, 128),      # split-page mode, one ragged page per sequence (no second page)
    ([0, 57, 120], 8, False, 64),        # the same without the causal mask, one-page chunks
])
def test_tile_kernel_shapes(lens, q_len, causal, chunk):
    w = synth.Workload("tile", lens, q_len=q_len, causal=causal, seed=q_len * 7 + len(lens),
                       chunk_tokens=chunk, pool_pages=sum((c + q_len + 63) // 64 for c in lens) + 3)
    _check(w, chunk=chunk, steps=2)


@pytest.mark.parametrize("Hq,Hkv,q_len", [(8, 1, 5), (9, 3, 5), (16, 2, 3), (6, 3, 9), (12, 4, 4),
                                          (32, 4, 8),    # 64 rows: the largest split-page tile
                                          (13, 1, 5)])   # 65 rows: the smallest full tile
def test_tile_kernel_group_sizes(Hq, Hkv, q_len):
    # odd head counts leave the last pair with one head
    w = synth.Workload("tile_groups", [200, 1300], q_len=q_len, seed=Hq * 10 + Hkv, q_heads=Hq,
                       kv_heads=Hkv, chunk_tokens=128)
    _check(w, chunk=128)


def test_tile_kernel_skips_bad_pages_and_flags_them():
    import bit_kv_cache_03_gb300 as kv
    w = synth.Workload("tile_badpage", [700], q_len=8, seed=11, pool_pages=20)
    g = GpuRun(w)
    g.step()
    torch.cuda.synchronize()
    assert g.status() == 0
    bt = g.cache.block_table
    bt[0, 3] = 10 ** 6
    g.cache.attend(g.q_codes, g.q_scales, g.out, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert g.status() & kv.DEV_BAD_PAGE
    assert np.all(np.isfinite(g.output()))
