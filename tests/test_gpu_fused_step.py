"""kv_nvfp4_decode_step (append inside the attention launch) against the two-call path and the
oracle (GPU): bit-identical pool bytes and Q codes, identical output, oracle parity."""
import numpy as np
import pytest

import oracle
import synth
from kvrun import MAX_ABS_TOL, REL_L2_TOL, GpuRun, OracleRun, attention_errors, compare_pool

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _pair(w, chunk):
    a, b = GpuRun(w), GpuRun(w)
    a.step(chunk_tokens=chunk)        # kv_nvfp4_append, then kv_nvfp4_decode_attn
    b.step_fused(chunk_tokens=chunk)  # kv_nvfp4_decode_step
    torch.cuda.synchronize()
    return a, b


@pytest.mark.parametrize("lens,q_len,Hq,Hkv,chunk", [
    ([0, 5, 63, 64, 65, 200, 1000], 1, 24, 4, 1024),
    ([0, 5, 63, 64, 65, 200, 1000], 1, 24, 4, 64),     # split groups: the merge launch too
    ([130, 700, 1500], 2, 8, 2, 128),                  # 2 new tokens x GQA 4 = 8 rows
    ([300, 1200], 1, 8, 1, 256),                       # GQA 8: all 8 rows computed
    ([100, 2000], 1, 9, 3, 256),                       # odd number of KV heads
    ([4000], 4, 4, 4, 512),                            # 4 new tokens, no GQA, page boundary
])
def test_fused_step_matches_two_calls_and_oracle(lens, q_len, Hq, Hkv, chunk):
    w = synth.Workload("fused", lens, q_len=q_len, seed=7 + q_len + Hkv, q_heads=Hq, kv_heads=Hkv,
                       chunk_tokens=chunk, pool_pages=sum((c + q_len + 63) // 64 for c in lens) + 3)
    a, b = _pair(w, chunk)
    assert a.status() == 0 and b.status() == 0
    o = OracleRun(w)
    bad = compare_pool(b, o)               # every cached and new code byte, bit-exact
    assert all(v == 0 for v in bad.values()), bad
    qa, qb = a.q_quant(), b.q_quant()
    assert np.array_equal(qa[0], qb[0]) and np.array_equal(qa[1], qb[1])
    assert np.array_equal(a.output(), b.output())
    max_abs, rel = attention_errors(b.output(), o.attention().reshape(b.output().shape))
    assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, (max_abs, rel)
    # a second step on the same cache rewrites the same rows: same result
    b.step_fused(chunk_tokens=chunk, q_out=False)
    torch.cuda.synchronize()
    assert np.array_equal(a.output(), b.output()) and b.status() == 0


@pytest.mark.parametrize("lens,q_len,Hq,Hkv,rot", [
    ([300, 1200], 1, 24, 4, 64),    # rotary dims spread over four 16-value blocks of a row
    ([500], 2, 8, 2, 128),          # every dim rotary
    ([700, 90], 1, 24, 4, 0),       # no RoPE
    ([900], 1, 12, 4, 48),          # a rotary width that ends inside a 16-value block
])
def test_fused_step_rotary_widths(lens, q_len, Hq, Hkv, rot):
    w = synth.Workload("fused_rot", lens, q_len=q_len, seed=19 + rot, q_heads=Hq, kv_heads=Hkv,
                       rot_dim=rot, chunk_tokens=128,
                       pool_pages=sum((c + q_len + 63) // 64 for c in lens) + 2)
    a, b = _pair(w, 128)
    assert a.status() == 0 and b.status() == 0
    o = OracleRun(w)
    bad = compare_pool(b, o)
    assert all(v == 0 for v in bad.values()), bad
    qa, qb = a.q_quant(), b.q_quant()
    assert np.array_equal(qa[0], qb[0]) and np.array_equal(qa[1], qb[1])
    assert np.array_equal(qb[0], o.qc) and np.array_equal(qb[1], o.qs)
    assert np.array_equal(a.output(), b.output())
    max_abs, rel = attention_errors(b.output(), o.attention().reshape(b.output().shape))
    assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, (max_abs, rel)


def test_fused_step_rejects_more_than_one_row_tile():
    import bit_kv_cache_03_gb300 as kv
    w = synth.Workload("fused_bad", [500], q_len=2, seed=3, chunk_tokens=256)  # 2 x GQA 6 = 12 rows
    g = GpuRun(w)
    g.cache.plan(w.seq_lens, w.q_len, w.causal, 256)
    with pytest.raises(kv.KVNVFP4Error, match=r"\(-1\)"):
        g.step_fused(plan=False)


def test_fused_step_flags_a_page_outside_the_pool():
    import bit_kv_cache_03_gb300 as kv
    w = synth.Workload("fused_badpage", [500], q_len=1, seed=4, pool_pages=12)
    g = GpuRun(w)
    bt = g.cache.block_table.clone()
    g.cache.block_table[0, 500 // 64] = 10 ** 6  # the page of the new token
    g.step_fused()
    torch.cuda.synchronize()
    assert g.status() & kv.DEV_BAD_PAGE
    g.cache.block_table.copy_(bt)


@pytest.mark.parametrize("pinned", [True, False])
def test_decode_step_from_host_buffers_matches_device_step(pinned):
    # kv_nvfp4_decode_step_host (new rows in, output out, plan, fused step in one call) against the
    # device-buffer step on the same inputs, three steps in a row with different new rows each
    # step: every pool byte and every output value identical. Page-locked host buffers take the
    # path where the GPU reads the rows and writes the output over the host link itself;
    # pageable ones take the copy path.
    w = synth.Workload("host_step", [700, 64, 3000], q_len=1, seed=21, chunk_tokens=128)
    ref = GpuRun(w)
    g = GpuRun(w)
    g.cache.plan(w.seq_lens, w.q_len, w.causal, 128)  # sizes the workspace
    q0, k0, v0, *_ = w.new_tokens()
    host = (lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()) \
        if pinned else (lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()))
    h_q, h_k, h_v = host(q0), host(k0), host(v0)
    d_q, d_k, d_v = (torch.empty_like(t, device="cuda") for t in (h_q, h_k, h_v))
    h_out = torch.full((g.out.numel(),), float("nan"), dtype=torch.float32)
    if pinned:
        h_out = h_out.pin_memory()
    for step in range(3):
        # this step's new rows: the workload's own rows for step 0, other seeded rows after
        ws = synth.Workload("host_step", [700, 64, 3000], q_len=1, seed=21 + 100 * step)
        q, k, v, *_ = ws.new_tokens()
        for t, a in ((h_q, q), (h_k, k), (h_v, v)):
            t.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)))
        for t, a in ((ref.q, q), (ref.k, k), (ref.v, v)):
            t.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16))
        ref.step_fused(chunk_tokens=128)
        g.cache.decode_step_host(np.asarray(w.seq_lens, np.int32), w.q_len, h_q, h_k, h_v, d_q,
                                 d_k, d_v, g.out, h_out, causal=w.causal, chunk_tokens=128,
                                 sm_scale=w.sm_scale)
        torch.cuda.synchronize()
        assert g.status() == 0 and ref.status() == 0
        assert np.array_equal(h_out.numpy(), ref.out.cpu().numpy()), step
        pg, pr = g.pool(), ref.pool()  # every stored slot (unused slots hold no data)
        for s_ in range(w.num_seqs):
            a = oracle.paged_gather(pg, w.pool_pages, w.kv_heads, w.block_table, s_, 0,
                                    int(w.seq_lens[s_]))
            b = oracle.paged_gather(pr, w.pool_pages, w.kv_heads, w.block_table, s_, 0,
                                    int(w.seq_lens[s_]))
            assert all(np.array_equal(x, y) for x, y in zip(a[:4], b[:4])), (step, s_)
        if step == 0:  # the workload's own new rows: every code byte as the oracle's
            bad = compare_pool(g, OracleRun(w))
            assert all(v == 0 for v in bad.values()), bad
