"""Parity on the five full-size workloads, in the launch configuration the benchmark times (GPU).

Every K/V row of every cached and appended token is compared bit-exactly with the oracle's
quantisation; attention is compared on every output row (decode and verify workloads) or on a
seeded row sample (the 600k prefill chunk, 196,608 rows)."""
import numpy as np
import pytest

import synth
from kvrun import (MAX_ABS_TOL, REL_L2_TOL, GpuRun, OracleRun, attention_errors, compare_pool,
                   cosine, sample_rows)

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _run(w, rows=None, chunk=None):
    g = GpuRun(w)
    g.step(chunk_tokens=chunk)
    torch.cuda.synchronize()
    assert g.status() == 0
    o = OracleRun(w)
    bad = compare_pool(g, o)
    assert all(v == 0 for v in bad.values()), bad
    qc, qs = g.q_quant()
    assert np.array_equal(qc, o.qc) and np.array_equal(qs, o.qs)
    out = g.output()
    if rows is None:
        ref = o.attention().reshape(out.shape)
        got = out
    else:
        ref = o.attention(rows)
        rs, rt, rh = rows
        got = out.reshape(w.num_seqs, w.q_len, w.q_heads, 128)[rs, rt, rh]
    max_abs, rel = attention_errors(got, ref)
    print(f"{w.name}: max_abs={max_abs:.3e} rel_l2={rel:.3e}")
    assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, (max_abs, rel)
    assert np.all(np.isfinite(out))
    return g, o, got, ref


def test_tiny_decode_4k():
    w = synth.tiny_decode()
    g, o, got, ref = _run(w)
    rows = o.all_rows()
    unq = o.attention_unquantized(rows)
    c = cosine(got, unq)
    print(f"cosine vs unquantised attention: {c:.4f}")
    assert c > 0.5


def test_steady_decode_4x128k():
    _run(synth.steady_decode())


def test_ragged_decode_8seq():
    _run(synth.ragged_decode())


def test_spec_verify_4x100k_q8():
    _run(synth.spec_verify())


def test_prefill_chunk_600k_sampled():
    w = synth.prefill_chunk()
    rows = sample_rows(w, 256, seed=0)
    # one chunk per sequence: every (kv head, 8-row tile) item streams the whole cache
    _run(w, rows=rows, chunk=((w.max_pos + 63) // 64) * 64)
