"""Pins for the oracle's scalar formats and row quantiser (CPU only).

The oracle is checked against things other than itself: the E2M1 grid the method states, the
E4M3 decoder and encoder of PyTorch's float8_e4m3fn type, a hand-worked row in tests/golden,
and the page's bytes-per-token figures.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_grid_exact():
    # The method's value set: {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6}, sign-magnitude codes.
    for c in range(16):
        v = oracle.e2m1_decode(c)
        mag = GRID[c & 7]
        assert abs(v) == mag
        assert np.signbit(v) == bool(c & 8)


def test_e2m1_encode_decode_identity_all_codes():
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_decode(c)) == c  # -0 keeps its sign (0x8)


@pytest.mark.parametrize("x,code", [
    (0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5.0, 0x6),
    (-0.25, 0x8), (-0.75, 0xA), (-1.25, 0xA), (-1.75, 0xC), (-2.5, 0xC), (-3.5, 0xE), (-5.0, 0xE),
    (0.2500001, 0x1), (0.7499999, 0x1), (5.0000005, 0x7), (6.0, 0x7), (7.0, 0x7), (1e9, 0x7),
    (-1e9, 0xF), (0.0, 0x0), (-0.0, 0x8), (1e-30, 0x0), (-1e-30, 0x8),
])
def test_e2m1_ties_and_saturation(x, code):
    # hand tie table: a value halfway between two grid points goes to the even code
    assert oracle.e2m1_encode(np.float32(x)) == code


def test_e2m1_encode_is_nearest_and_monotone():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.uniform(-8, 8, 4000), rng.normal(0, 2, 4000)]).astype(np.float32)
    grid = np.array(GRID + [-g for g in GRID])
    prev = None
    for x in np.sort(xs):
        v = oracle.e2m1_decode(oracle.e2m1_encode(float(x)))
        if abs(x) <= 6.0:
            assert abs(x - v) <= np.min(np.abs(x - grid)) + 1e-12
        else:
            assert v == np.copysign(6.0, x)
        if prev is not None:
            assert v >= prev
        prev = v


def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_decode(c) for c in range(256)], np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne_below_saturation():
    # torch rounds float -> float8_e4m3fn to nearest-even; it does not saturate, so compare only
    # below the first value that would round past 448 (464 is the midpoint 448 | 480).
    rng = np.random.default_rng(2)
    vals = [np.float32(x) for x in np.concatenate([
        rng.uniform(0, 463.9, 20000), np.exp(rng.uniform(np.log(1e-5), np.log(463.9), 20000)),
        rng.uniform(0, 2 ** -6, 4000)])]
    # every exact midpoint between neighbouring finite values (ties)
    pos = [oracle.e4m3_decode(c) for c in range(0x7F)]
    vals += [np.float32((a + b) / 2) for a, b in zip(pos[:-1], pos[1:])]
    vals += [np.float32(p) for p in pos]
    t = torch.tensor(np.array(vals, np.float32))
    ref = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(v)) for v in vals], np.uint8)
    assert np.array_equal(ref, ours)


@pytest.mark.parametrize("t,code", [(448.0, 0x7E), (463.9, 0x7E), (464.0, 0x7E), (500.0, 0x7E),
                                    (1e30, 0x7E), (0.0, 0x00), (2.0 ** -10, 0x00),
                                    (2.0 ** -10 * 1.0001, 0x01), (2.0 ** -9, 0x01)])
def test_e4m3_saturation_and_underflow(t, code):
    # reading: satfinite (never NaN), round-to-nearest-even at the bottom of the subnormals
    assert oracle.e4m3_encode(np.float32(t)) == code


def test_quantize_row_hand_worked_golden():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_row_example.json")))
    x = np.array(g["row"], np.float32)
    codes, scales = oracle.quantize_row(x)
    assert list(scales) == g["scales"]
    assert list(codes) == g["codes"]


def test_layout_bytes_match_page():
    g = json.load(open(os.path.join(GOLDEN, "layout_bytes.json")))
    d = g["head_dim"]
    assert oracle.bytes_per_token_head("nvfp4", d) == g["nvfp4"] == 144
    assert oracle.bytes_per_token_head("int8", d) == g["int8"] == 264
    assert oracle.bytes_per_token_head("bf16", d) == g["bf16"] == 512


def test_quantize_row_exact_on_representable_blocks():
    # values that are grid points times a power of two, amax = 6 * 2^k: quantisation is lossless
    rng = np.random.default_rng(3)
    for k in range(-8, 7):
        mags = rng.choice(GRID, size=(8, 16))
        signs = rng.choice([-1.0, 1.0], size=(8, 16))
        x = (mags * signs * 2.0 ** k).astype(np.float32)
        x[:, 0] = 6.0 * 2.0 ** k
        codes, scales = oracle.quantize_row(x.reshape(-1))
        back = oracle.dequant_rows(codes, scales)[0]
        assert np.array_equal(back, x.reshape(-1).astype(np.float64))


def test_quantize_row_error_bound():
    # per element: unsaturated codes are off by at most half the widest grid gap (1.0) times s;
    # saturated ones by at most amax - 6 s. Normal scales are within 2^-4 of amax / 6.
    rng = np.random.default_rng(4)
    for _ in range(200):
        x = (rng.normal(0, 1, 128) * np.exp(rng.uniform(-6, 6))).astype(np.float32)
        codes, scales = oracle.quantize_row(x)
        back = oracle.dequant_rows(codes, scales)[0]
        for b in range(8):
            blk = x[16 * b:16 * b + 16].astype(np.float64)
            amax = np.abs(blk).max()
            s = oracle.e4m3_decode(scales[b])
            if amax / 6 >= 2 ** -6:
                assert abs(s - amax / 6) <= amax / 6 * 2 ** -4
            else:
                assert abs(s - amax / 6) <= 2 ** -10
            if s > 0:
                err = np.abs(blk - back[16 * b:16 * b + 16])
                assert np.all(err <= max(s * 1.0, amax - 6 * s) + 1e-12)
