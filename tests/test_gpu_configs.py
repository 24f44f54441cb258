"""Parity on the five full-size workloads, in the launch configurations the benchmark times (GPU).

Every K/V row of every cached and appended token is compared bit-exactly with the oracle's
quantisation; attention is compared on every output row (decode and verify workloads) or on a
seeded row sample (the 600k prefill chunk, 196,608 rows). Each workload runs through the call and
the split-K chunk size that bench.py times for it:
  tiny / steady / ragged decode: kv_nvfp4_decode_step (the append inside the attention launch),
      chunks of 64 tokens, so the split-K merge runs;
  speculative verify and the 600k prefill chunk: kv_nvfp4_append + kv_nvfp4_decode_attn on the
      tile kernel, chunks of 128 tokens (verify) and 1024 tokens (prefill), so the tile kernel's
      merge runs as well.
The decode workloads are also run through the two-call path with the workload's own chunk size
(1024 tokens for the ragged workload).
"""
import numpy as np
import pytest

import synth
from kvrun import (MAX_ABS_TOL, REL_L2_TOL, GpuRun, OracleRun, attention_errors, compare_pool,
                   cosine, sample_rows)

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# the split-K chunk each workload is timed with in bench.py
BENCH_CHUNK = {"tiny_decode_4k": 64, "steady_decode_4x128k": 64, "ragged_decode_8seq": 64,
               "spec_verify_4x100k_q8": 128, "prefill_chunk_600k": 1024}


def _check(g, o, w, rows, label):
    torch.cuda.synchronize()
    assert g.status() == 0, (label, g.status())
    bad = compare_pool(g, o)
    assert all(v == 0 for v in bad.values()), (label, bad)
    qc, qs = g.q_quant()
    assert np.array_equal(qc, o.qc) and np.array_equal(qs, o.qs), label
    out = g.output()
    assert np.all(np.isfinite(out)), label
    if rows is None:
        ref = o.attention().reshape(out.shape)
        got = out
    else:
        ref = o.attention(rows)
        rs, rt, rh = rows
        got = out.reshape(w.num_seqs, w.q_len, w.q_heads, 128)[rs, rt, rh]
    max_abs, rel = attention_errors(got, ref)
    print(f"{w.name} [{label}]: max_abs={max_abs:.3e} rel_l2={rel:.3e}")
    assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, (label, max_abs, rel)
    return got


def _decode(w):
    """The benchmarked fused step (bench chunk), then the two-call path (workload chunk)."""
    g = GpuRun(w)
    o = OracleRun(w)
    chunk = BENCH_CHUNK[w.name]
    g.step_fused(chunk_tokens=chunk)
    assert g.cache.plan_info.num_split_groups > 0  # the merge launch ran
    got = _check(g, o, w, None, f"decode_step chunk {chunk}")
    g.out.zero_()
    g.step(chunk_tokens=w.chunk_tokens)
    _check(g, o, w, None, f"append + decode_attn chunk {w.chunk_tokens}")
    return g, o, got


def test_tiny_decode_4k():
    w = synth.tiny_decode()
    g, o, got = _decode(w)
    unq = o.attention_unquantized(o.all_rows())
    c = cosine(got, unq)
    print(f"cosine vs unquantised attention: {c:.4f}")
    assert c > 0.5


def test_steady_decode_4x128k():
    _decode(synth.steady_decode())


def test_ragged_decode_8seq():
    _decode(synth.ragged_decode())


def test_spec_verify_4x100k_q8():
    w = synth.spec_verify()
    g = GpuRun(w)
    o = OracleRun(w)
    g.step(chunk_tokens=BENCH_CHUNK[w.name])
    assert g.cache.plan_info.num_split_groups > 0  # the tile kernel's merge ran
    _check(g, o, w, None, f"append + decode_attn (tile kernel) chunk {BENCH_CHUNK[w.name]}")


def test_prefill_chunk_600k_sampled():
    w = synth.prefill_chunk()
    rows = sample_rows(w, 256, seed=0)
    g = GpuRun(w)
    o = OracleRun(w)
    g.step(chunk_tokens=BENCH_CHUNK[w.name])
    assert g.cache.plan_info.num_split_groups > 0
    _check(g, o, w, rows,
           f"append + decode_attn (tile kernel) chunk {BENCH_CHUNK[w.name]}, sampled rows")
    # one chunk per sequence (no split-K merge): the same sampled rows
    g.out.zero_()
    g.step(chunk_tokens=((w.max_pos + 63) // 64) * 64)
    _check(g, o, w, rows, "one chunk per sequence, sampled rows")
