"""Bit-exact parity of the fused quantize-append kernel against the oracle (GPU)."""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from kvrun import GpuRun, OracleRun, compare_pool

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _f32_to_bf16_bits(x):
    """Round fp32 to bf16 (nearest even) as test input construction."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _crafted_rows(n_rows, seed):
    """Rows that hit the encoders' corner cases: exact midpoints, zero and -0 blocks, subnormal
    and saturating scales, grid values times powers of two."""
    rng = np.random.default_rng(seed)
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_row_example.json")))
    rows = [np.array(g["row"], np.float32)]
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5], np.float32)
    while len(rows) < n_rows:
        kind = len(rows) % 5
        if kind == 0:
            x = rng.choice(grid, 128) * rng.choice([-1, 1], 128) * 2.0 ** rng.integers(-12, 9, (8, 1)).repeat(16, 1).ravel()
            x[::16] = 6 * 2.0 ** rng.integers(-12, 9)
        elif kind == 1:
            x = rng.normal(0, 1, 128) * np.exp(rng.uniform(-14, -6))   # subnormal scales
        elif kind == 2:
            x = rng.normal(0, 1, 128) * np.exp(rng.uniform(6, 12))     # large, saturating scales
        elif kind == 3:
            x = np.zeros(128); x[rng.integers(0, 128, 5)] = -0.0
            x[64:80] = rng.normal(0, 1e-3, 16)
        else:
            x = rng.normal(0, 1, 128)
            x[[3, 77, 101, 120]] *= 12
        rows.append(np.asarray(x, np.float32))
    return _f32_to_bf16_bits(np.stack(rows))


def _append_crafted(Hq, Hkv, T, seed, rot_dim=32):
    rows_q = _crafted_rows(T * Hq, seed) if Hq else None
    rows_k = _crafted_rows(T * Hkv, seed + 1)
    rows_v = _crafted_rows(T * Hkv, seed + 2)
    pages = (T + 63) // 64
    bt = synth.permutation(seed, 7, pages + 3)[:pages].reshape(1, pages)
    import bit_kv_cache_03_gb300 as kv
    cache = kv.PagedNVFP4Cache(pages + 3, bt, T, Hq or 4, Hkv, rot_dim)
    dev = cache.device
    def to_dev(a, heads):
        t = torch.from_numpy(a.reshape(T, heads, 128).view(np.int16))
        return t.to(dev).view(torch.bfloat16)
    pos = np.arange(T, dtype=np.int32)
    qc, qs = cache.quantized_q_buffers(T)
    cache.append(to_dev(rows_k, Hkv), to_dev(rows_v, Hkv),
                 torch.zeros(T, dtype=torch.int32, device=dev),
                 torch.from_numpy(pos).to(dev), q=to_dev(rows_q, Hq) if Hq else None,
                 q_codes=qc, q_scales=qs)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    table = oracle.rope_table(T, rot_dim, 1e7, 1.0)
    ek, eks = oracle.quantize_rows(rows_k, np.repeat(pos, Hkv), True, table, rot_dim)
    ev, evs = oracle.quantize_rows(rows_v, None, False, None, 0)
    kc, ks, vc, vs, _ = oracle.paged_gather(cache.pool.cpu().numpy(), pages + 3, Hkv, bt, 0, 0, T)
    assert np.array_equal(kc.reshape(-1, 64), ek) and np.array_equal(ks.reshape(-1, 8), eks)
    assert np.array_equal(vc.reshape(-1, 64), ev) and np.array_equal(vs.reshape(-1, 8), evs)
    if Hq:
        eq, eqs = oracle.quantize_rows(rows_q, np.repeat(pos, Hq), True, table, rot_dim)
        assert np.array_equal(qc.cpu().numpy().reshape(-1, 64), eq)
        assert np.array_equal(qs.cpu().numpy().reshape(-1, 8), eqs)


@pytest.mark.parametrize("Hq,Hkv,T,rot", [(24, 4, 77, 32), (8, 8, 130, 32), (6, 1, 64, 128),
                                          (0, 4, 1, 32), (24, 4, 200, 0), (24, 4, 65, 64),
                                          (24, 4, 33, 48), (4, 2, 70, 8), (3, 3, 1000, 120),
                                          (24, 4, 300, 32), (8, 2, 700, 64), (0, 4, 1100, 32)])
def test_append_crafted_rows_bitexact(Hq, Hkv, T, rot):
    _append_crafted(Hq, Hkv, T, seed=T + Hq, rot_dim=rot)


def test_append_small_workload_bitexact():
    w = synth.Workload("small_ragged", [0, 5, 63, 64, 65, 200, 1000], q_len=3, seed=11,
                       pool_pages=60)
    g = GpuRun(w)
    g.step()
    torch.cuda.synchronize()
    assert g.status() == 0
    o = OracleRun(w)
    bad = compare_pool(g, o)
    assert all(v == 0 for v in bad.values()), bad
    qc, qs = g.q_quant()
    assert np.array_equal(qc, o.qc) and np.array_equal(qs, o.qs)


def test_append_reports_bad_rows_and_skips_them():
    import bit_kv_cache_03_gb300 as kv
    bt = np.array([[0, 1], [2, 99]], np.int32)           # page 99 is outside a 3-page pool
    cache = kv.PagedNVFP4Cache(3, bt, 128, 24, 4, 32)
    dev = cache.device
    T = 4
    k = torch.randn(T, 4, 128, device=dev).to(torch.bfloat16)
    v = torch.randn(T, 4, 128, device=dev).to(torch.bfloat16)
    cache.pool.fill_(0xAB)
    sid = torch.tensor([0, 1, 5, 0], dtype=torch.int32, device=dev)      # seq 5 does not exist
    pos = torch.tensor([3, 70, 1, 200], dtype=torch.int32, device=dev)   # 70 -> page 99; 200 beyond
    cache.append(k, v, sid, pos)
    torch.cuda.synchronize()
    st = int(cache.status.item())
    assert st & kv.DEV_BAD_PAGE and st & kv.DEV_BAD_SEQ and st & kv.DEV_BAD_POS
    pool = cache.pool.cpu().numpy()
    changed = np.nonzero(pool != 0xAB)[0]
    # only page 0, slot 3 of every head was written (codes, scales of K and V)
    kc, ks, vc, vs, _ = oracle.paged_gather(pool, 3, 4, np.array([[0]], np.int32), 0, 3, 1)
    assert changed.size > 0 and changed.max() < 4 * 9216
    expected = set()
    for h in range(4):
        for j in range(64):
            expected.add(h * 4096 + (3 // 8) * 512 + (j // 16) * 128 + (3 % 8) * 16 + j % 16)
            expected.add(4 * 4608 + h * 4096 + 3 * 64 + j)
        for j in range(8):
            # K scales in the scale-copy order (4 heads: two full pairs): slot 3, half j // 4
            expected.add(4 * 4096 + (h // 2) * 1024 + (j // 4) * 512 + 3 * 16 + (h % 2) * 8 + j % 4)
            expected.add(4 * 8704 + h * 512 + 3 * 8 + j)
    assert set(changed.tolist()) <= expected
