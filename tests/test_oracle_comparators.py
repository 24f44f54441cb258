"""Pins for the oracle's comparator formats (CPU only).

Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)": the NVFP4 row
(144 B per token per KV head) against int8 (264 B) and bf16 (512 B), and the upstream variant with
NVFP4 K and fp16 V. The pins tie each oracle function to something outside it: numpy's and torch's
float16 / bfloat16 conversions, closed-form properties of the int8 row code, the already pinned
RoPE and NVFP4 row functions, a pool whose every byte names its place, and torch's float64
scaled-dot-product attention.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "layout_bytes.json")


def _sweep_floats(rng, n=20000):
    mags = 2.0 ** rng.uniform(-30, 18, size=n)
    x = (mags * rng.choice([-1.0, 1.0], size=n)).astype(np.float32)
    edge = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 70000.0, 6.1035156e-05, 6.0e-8,
                     5.9604645e-08, 2.9802322e-08, 2.9802326e-08, 1.0 + 2.0 ** -11,
                     1.0 + 3 * 2.0 ** -11, -(1.0 + 2.0 ** -11), 3.0517578e-05], np.float32)
    return np.concatenate([x, edge])


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    x = _sweep_floats(rng)
    with np.errstate(over="ignore"):  # values past 65504 become inf on purpose
        want = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_f16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, want)


def test_f16_decode_of_every_pattern():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = h.view(np.float16).astype(np.float64)
    finite = np.isfinite(want)
    got = np.array([oracle.f16_to_double(int(v)) for v in h[finite]])
    assert np.array_equal(got, want[finite])


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = _sweep_floats(rng)
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32)  # exact halves
    x = np.concatenate([x, ties, -ties])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.float_to_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, want)


def test_int8_row_code_properties():
    rng = np.random.default_rng(2)
    for _ in range(50):
        x = (rng.standard_normal(128) * 10 ** rng.uniform(-3, 3)).astype(np.float32)
        codes, s = oracle.int8_quantize_row(x)
        amax = np.abs(x).max()
        assert s == np.float32(amax) / np.float32(127.0)
        i = int(np.abs(x).argmax())
        assert abs(int(codes[i])) == 127 and np.sign(codes[i]) == np.sign(x[i])
        assert np.all(np.abs(codes.astype(np.int32)) <= 127)
        err = np.abs(codes.astype(np.float64) * s - x.astype(np.float64))
        assert np.all(err <= 0.5 * s * (1 + 1e-6) + 1e-30)
    z, s = oracle.int8_quantize_row(np.zeros(128, np.float32))
    assert s == 0.0 and not z.any()
    # a power-of-two scale makes x / s exact: halves round to the even integer
    x = np.zeros(128, np.float32)
    x[0] = 127.0 * 0.25
    x[1:7] = np.array([0.5, 1.5, 2.5, -0.5, -1.5, 126.5], np.float32) * 0.25
    codes, s = oracle.int8_quantize_row(x)
    assert s == 0.25
    assert list(codes[:7]) == [127, 0, 2, 2, 0, -2, 126]


def test_row_bytes_follow_the_golden_budgets():
    g = json.load(open(GOLDEN))
    # per token per KV head: K row + V row
    assert oracle.cmp_row_bytes(0, 1) + oracle.cmp_row_bytes(0, 2) == g["bf16"]
    assert oracle.cmp_row_bytes(1, 1) + oracle.cmp_row_bytes(1, 2) == g["int8"]
    assert oracle.cmp_row_bytes(2, 1) == g["nvfp4"] // 2  # NVFP4 K row
    assert oracle.cmp_row_bytes(2, 2) == 256            # fp16 V row


def _rows(rng, n):
    x = rng.standard_normal((n, 128)).astype(np.float32)
    x[:, [3, 77]] *= 12
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_encodings_follow_the_pinned_pieces():
    rng = np.random.default_rng(3)
    rows = _rows(rng, 6)
    pos = np.array([0, 5, 77, 1000, 4095, 12], np.int32)
    table = oracle.rope_table(4096, 32, 1e7, 1.0)
    xf = rows.view(np.uint16).astype(np.uint32) << 16
    xf = xf.view(np.float32)
    rot = np.stack([oracle.rope_apply(xf[i].copy(), table, int(pos[i]), 32) for i in range(6)])
    # Q (every format) and bf16 K: bf16 of the rotated row
    qb = oracle.cmp_encode_rows(1, 0, rows, pos, table, 32).view(np.uint16)
    want = torch.from_numpy(rot).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(qb, want)
    assert np.array_equal(oracle.cmp_encode_rows(0, 1, rows, pos, table, 32).view(np.uint16), want)
    # bf16 V: the row as given; fp16 V of the upstream variant: numpy's rounding
    assert np.array_equal(oracle.cmp_encode_rows(0, 2, rows, pos, table, 32).view(np.uint16), rows)
    v16 = oracle.cmp_encode_rows(2, 2, rows, pos, table, 32).view(np.uint16)
    assert np.array_equal(v16, xf.astype(np.float16).view(np.uint16))
    # NVFP4 K of the upstream variant: the pinned row quantiser on the rotated row (no Hadamard)
    k4 = oracle.cmp_encode_rows(2, 1, rows, pos, table, 32)
    for i in range(6):
        c, s = oracle.quantize_row(rot[i])
        assert np.array_equal(k4[i, :64], c) and np.array_equal(k4[i, 64:], s)
    # int8 K: the row code of the rotated row, fp32 scale after the codes
    k8 = oracle.cmp_encode_rows(1, 1, rows, pos, table, 32)
    for i in range(6):
        c, s = oracle.int8_quantize_row(rot[i])
        assert np.array_equal(k8[i, :128].view(np.int8), c)
        assert k8[i, 128:].view(np.float32)[0] == np.float32(s)
    # decoding: exact values of every format
    d = oracle.cmp_decode_rows(1, 1, k8)
    assert np.array_equal(d[2], k8[2, :128].view(np.int8).astype(np.float64) *
                          np.float64(k8[2, 128:].view(np.float32)[0]))
    assert np.array_equal(oracle.cmp_decode_rows(2, 1, k4), oracle.dequant_rows(k4[:, :64], k4[:, 64:]))
    assert np.array_equal(oracle.cmp_decode_rows(2, 2, v16.view(np.uint8)),
                          v16.view(np.float16).astype(np.float64))


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_comparator_gather_layout(fmt):
    # every byte of the pool names (page, head, region, slot, byte), rows stored with their
    # 16-byte units permuted as the layout states; the gather must return each slot's own bytes
    # in row order
    P, H = 5, 3
    kb, vb = oracle.cmp_row_bytes(fmt, 1), oracle.cmp_row_bytes(fmt, 2)
    chunk = 64 * (kb + vb)
    pool = np.zeros(P * H * chunk, np.uint8)
    name = lambda p, h, reg, k, j: (p * 31 + h * 17 + reg * 7 + k * 3 + j) % 251
    def put(c, base, k, sw, vals):  # a row stored with 16-byte unit u at u ^ sw
        for j, x in enumerate(vals):
            c[base + (((j // 16) ^ sw) * 16) + j % 16] = x

    for p in range(P):
        for h in range(H):
            c = pool[(p * H + h) * chunk:(p * H + h + 1) * chunk]
            for k in range(64):
                if fmt == 0:
                    put(c, k * 256, k, k & 7, [name(p, h, 0, k, j) for j in range(256)])
                    put(c, 64 * 256 + k * 256, k, k & 7, [name(p, h, 1, k, j) for j in range(256)])
                elif fmt == 1:
                    put(c, k * 128, k, (k & 1) * 4, [name(p, h, 0, k, j) for j in range(128)])
                    c[8192 + k * 4:8192 + k * 4 + 4] = [name(p, h, 0, k, 128 + j) for j in range(4)]
                    put(c, 8448 + k * 128, k, ((k // 2) & 3) * 2, [name(p, h, 1, k, j) for j in range(128)])
                    c[16640 + k * 4:16640 + k * 4 + 4] = [name(p, h, 1, k, 128 + j) for j in range(4)]
                else:
                    c[k * 64:(k + 1) * 64] = [name(p, h, 0, k, j) for j in range(64)]
                    c[4096 + k * 8:4096 + k * 8 + 8] = [name(p, h, 0, k, 64 + j) for j in range(8)]
                    put(c, 4608 + k * 256, k, k & 7, [name(p, h, 1, k, j) for j in range(256)])
    bt = np.array([[3, 0, 4], [1, 2, 9]], np.int32)
    k, v, bad = oracle.cmp_paged_gather(fmt, pool, P, H, bt, 0, 40, 100)
    assert bad == 0
    for i in range(100):
        pos = 40 + i
        p, s = bt[0, pos // 64], pos % 64
        for h in range(H):
            assert list(k[i, h]) == [name(p, h, 0, s, j) for j in range(kb)]
            assert list(v[i, h]) == [name(p, h, 1, s, j) for j in range(vb)]
    *_, bad = oracle.cmp_paged_gather(fmt, pool, P, H, bt, 1, 100, 50)
    assert bad == 22 * H  # positions 128..149 sit on page id 9, outside the 5-page pool


def test_f64_attention_matches_torch_sdpa():
    rng = np.random.default_rng(4)
    Hq, Hkv, q_len = 6, 2, 2
    lens = np.array([9, 33], np.int32)
    tok_off = np.array([0, 9], np.int64)
    q = rng.standard_normal((2 * q_len * Hq, 128))
    k = rng.standard_normal((42 * Hkv, 128))
    v = rng.standard_normal((42 * Hkv, 128))
    rows = [(s, i, h) for s in range(2) for i in range(q_len) for h in range(Hq)]
    rs, rt, rh = (np.array(x, np.int32) for x in zip(*rows))
    scale = 1.0 / math.sqrt(128)
    got = oracle.attention_f64_rows(Hq, Hkv, q_len, True, scale, lens, tok_off, q, k, v, rs, rt, rh)
    for n, (s, i, h) in enumerate(rows):
        L = int(lens[s])
        kk = torch.from_numpy(k.reshape(-1, Hkv, 128)[tok_off[s]:tok_off[s] + L, h // 3])
        vv = torch.from_numpy(v.reshape(-1, Hkv, 128)[tok_off[s]:tok_off[s] + L, h // 3])
        qq = torch.from_numpy(q[(s * q_len + i) * Hq + h])[None]
        vis = L - q_len + i + 1
        mask = torch.arange(L) < vis
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq[None, None], kk[None, None], vv[None, None], attn_mask=mask[None, None, None],
            scale=scale)[0, 0, 0].numpy()
        assert np.allclose(got[n], ref, rtol=1e-6, atol=1e-6)
