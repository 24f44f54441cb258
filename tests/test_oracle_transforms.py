"""Pins for the oracle's Hadamard rotation and RoPE (CPU only).

Checked against scipy's Sylvester Hadamard matrix, integer identities, an mpmath evaluation of
the RoPE angles, and rotation invariants; plus a hand example that fixes the (i, i+16) pairing.
"""
import math

import mpmath
import numpy as np
import scipy.linalg

import oracle


def test_fwht_scale_constant_bits():
    # rn(2^-3.5) = rn(1/sqrt(128))
    assert np.float32(oracle.fwht_scale()).view(np.uint32) == 0x3DB504F3


def test_fwht_columns_equal_sylvester_hadamard():
    H = scipy.linalg.hadamard(128)  # Sylvester construction, entries (-1)^popcount(i & j)
    c = np.float32(oracle.fwht_scale())
    for k in range(128):
        e = np.zeros(128, np.float32)
        e[k] = 1.0
        y = oracle.fwht128(e)
        assert np.array_equal(y, (H[:, k] * c).astype(np.float32))


def test_fwht_matrix_orthogonality_integer():
    c = float(np.float32(oracle.fwht_scale()))
    cols = []
    for k in range(128):
        e = np.zeros(128, np.float32)
        e[k] = 1.0
        cols.append(np.rint(oracle.fwht128(e) / c).astype(np.int64))
    M = np.stack(cols, axis=1)
    assert np.array_equal(M @ M.T, 128 * np.eye(128, dtype=np.int64))


def test_fwht_is_an_involution_and_preserves_dot_products():
    rng = np.random.default_rng(5)
    for _ in range(50):
        q = rng.normal(0, 1, 128).astype(np.float32)
        k = rng.normal(0, 1, 128).astype(np.float32)
        q[[3, 77, 101, 120]] *= 12
        k[[3, 77, 101, 120]] *= 12
        hq, hk = oracle.fwht128(q), oracle.fwht128(k)
        back = oracle.fwht128(hq)
        assert np.allclose(back, q, rtol=0, atol=2e-6 * np.abs(q).max() * math.sqrt(128))
        exact = float(np.dot(q.astype(np.float64), k.astype(np.float64)))
        got = float(np.dot(hq.astype(np.float64), hk.astype(np.float64)))
        bound = 1e-5 * float(np.linalg.norm(q) * np.linalg.norm(k))
        assert abs(got - exact) <= bound


def test_rope_table_within_half_ulp_of_exact():
    mpmath.mp.prec = 120
    theta, rot, f = 1e7, 32, 600000.0 / 262144.0
    positions = [0, 1, 2, 63, 64, 4095, 131072, 262143, 591871, 600063]
    for scale in (1.0, f):
        t = oracle.rope_table(600064, rot, theta, scale)
        for p in positions:
            for i in range(16):
                ang = (mpmath.mpf(p) / mpmath.mpf(scale)) * mpmath.power(
                    mpmath.mpf(theta), -mpmath.mpf(2 * i) / rot)
                for val, exact in ((t[p, i], mpmath.cos(ang)), (t[p, 16 + i], mpmath.sin(ang))):
                    ulp = float(np.spacing(np.float32(abs(float(exact))))) if exact != 0 else 1e-45
                    # half an fp32 ulp, plus a hair for the double evaluation of the angle
                    assert abs(float(val) - float(exact)) <= 0.5 * ulp * (1 + 1e-6) + 1e-15


def test_rope_pairing_hand_example():
    # position 1, frequency 0 has angle 1 rad: x = e_0 rotates into dims 0 and 16 (half-split)
    t = oracle.rope_table(2, 32, 1e7, 1.0)
    x = np.zeros(128, np.float32)
    x[0] = 1.0
    y = oracle.rope_apply(x, t, 1, 32)
    assert y[0] == np.float32(math.cos(1.0)) and y[16] == np.float32(math.sin(1.0))
    assert np.count_nonzero(y) == 2
    x = np.zeros(128, np.float32)
    x[16] = 1.0
    y = oracle.rope_apply(x, t, 1, 32)
    assert y[16] == np.float32(math.cos(1.0)) and y[0] == -np.float32(math.sin(1.0))
    # dims 32..127 pass through untouched
    x = np.arange(128, dtype=np.float32)
    y = oracle.rope_apply(x, t, 1, 32)
    assert np.array_equal(y[32:], x[32:])


def test_rope_position_zero_is_identity_and_relative_invariance():
    t = oracle.rope_table(5000, 32, 1e7, 1.0)
    rng = np.random.default_rng(6)
    q = rng.normal(0, 1, 128).astype(np.float32)
    k = rng.normal(0, 1, 128).astype(np.float32)
    assert np.array_equal(oracle.rope_apply(q, t, 0, 32), q)
    # <R(p) q, R(p') k> depends only on p - p'
    ref = None
    for p in (10, 500, 1234, 4000):
        a = oracle.rope_apply(q, t, p + 7, 32).astype(np.float64)
        b = oracle.rope_apply(k, t, p, 32).astype(np.float64)
        d = float(a @ b)
        if ref is None:
            ref = d
        assert abs(d - ref) <= 1e-4
    # norms preserved
    for p in (1, 77, 4999):
        assert abs(np.linalg.norm(oracle.rope_apply(q, t, p, 32)) - np.linalg.norm(q)) < 1e-5


def test_linear_position_scaling():
    # [YaRN] linear scaling by f: position p takes the angles of position p / f. With
    # f = 600000/262144 = 9375/4096 (exact in binary), p = 9375 m maps exactly onto 4096 m.
    f = 600000.0 / 262144.0
    ts = oracle.rope_table(600064, 32, 1e7, f)
    t1 = oracle.rope_table(262144, 32, 1e7, 1.0)
    for m in range(0, 64):
        assert np.array_equal(ts[9375 * m], t1[4096 * m])
    assert not np.array_equal(ts[9375], t1[9375])
