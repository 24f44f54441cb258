"""Checks of the seeded input generator (CPU only): determinism, row addressing, distribution."""
import numpy as np

import synth


def test_rows_are_addressable_and_deterministic():
    a = synth.normal_bf16(0, synth.STREAM_K, 2, 100, 50, 4)
    b = synth.normal_bf16(0, synth.STREAM_K, 2, 130, 20, 4)
    assert np.array_equal(a[30:], b)
    assert np.array_equal(a, synth.normal_bf16(0, synth.STREAM_K, 2, 100, 50, 4, nthreads=1))
    assert not np.array_equal(a, synth.normal_bf16(1, synth.STREAM_K, 2, 100, 50, 4))
    assert not np.array_equal(a, synth.normal_bf16(0, synth.STREAM_V, 2, 100, 50, 4))


def test_distribution_and_outlier_channels():
    x = synth.bf16_bits_to_float(
        synth.normal_bf16(3, 1, 0, 0, 4096, 4, outliers=(3, 77, 101, 120), mult=12.0))
    base = np.delete(x, [3, 77, 101, 120], axis=2)
    assert abs(base.mean()) < 0.01 and abs(base.std() - 1) < 0.01
    out = x[:, :, [3, 77, 101, 120]]
    assert abs(out.std() / 12 - 1) < 0.03
    # bf16 values: low 16 bits of the fp32 pattern are zero by construction
    assert np.all(x.view(np.uint32) & 0xFFFF == 0)


def test_permutation_and_lengths():
    p = synth.permutation(0, synth.STREAM_PAGES, 40000)
    assert np.array_equal(np.sort(p), np.arange(40000))
    lens = synth.loguniform_int(0, synth.STREAM_LENS, 1000, 8192.0, 262144.0)
    assert lens.min() >= 8192 and lens.max() < 262144


def test_workload_block_tables():
    w = synth.steady_decode()
    assert w.block_table.shape == (4, 2049)
    used = w.block_table[w.block_table >= 0]
    assert len(used) == 8196 and len(np.unique(used)) == 8196 and used.max() < 40000
    r = synth.ragged_decode()
    assert r.num_seqs == 8 and r.pool_pages == sum(r.pages_per_seq)
    t = synth.tiny_decode()
    assert np.array_equal(t.block_table[0], np.arange(65))
    c5 = synth.prefill_chunk()
    assert c5.max_pos == 600064 and c5.pool_pages == 9376
