"""Pins for the oracle's attention and paged-layout gather (CPU only).

Attention is checked against closed forms (one key, equal scores, two keys), against
torch's scaled_dot_product_attention in float64 on the oracle's own dequantised arrays (GQA head
mapping, causal offsets, scale), and the joint-rotation invariance of Q.K^T.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth


def _rand_quant(rng, n, scale=1.0):
    """Random codes/scales rows (valid finite E4M3 scales, not NaN)."""
    codes = rng.integers(0, 256, size=(n, 64), dtype=np.uint8)
    scales = rng.integers(0x20, 0x48, size=(n, 8), dtype=np.uint8)
    return codes, scales


def _attn(q_heads, kv_heads, q_len, causal, seq_lens, qc, qs, kc, ks, vc, vs, sm_scale=None):
    seq_lens = np.asarray(seq_lens, np.int32)
    tok_off = np.concatenate([[0], np.cumsum(seq_lens)[:-1]]).astype(np.int64)
    rows = [(s, i, h) for s in range(len(seq_lens)) for i in range(q_len) for h in range(q_heads)]
    rs, rt, rh = (np.array(x, np.int32) for x in zip(*rows))
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(128)
    return oracle.attention_rows(q_heads, kv_heads, q_len, causal, sm_scale, seq_lens, tok_off,
                                 qc, qs, kc, ks, vc, vs, rs, rt, rh)


def test_single_key_returns_that_value():
    rng = np.random.default_rng(7)
    qc, qs = _rand_quant(rng, 6)
    kc, ks = _rand_quant(rng, 1)
    vc, vs = _rand_quant(rng, 1)
    out = _attn(6, 1, 1, 1, [1], qc, qs, kc, ks, vc, vs)
    v = oracle.dequant_rows(vc, vs)[0].astype(np.float32)
    assert np.array_equal(out, np.tile(v, (6, 1)))


def test_equal_scores_give_the_mean():
    rng = np.random.default_rng(8)
    qc = np.zeros((6, 64), np.uint8)  # q = 0 -> every score 0
    qs = np.full((6, 8), 0x38, np.uint8)
    L = 37
    kc, ks = _rand_quant(rng, L)
    vc, vs = _rand_quant(rng, L)
    out = _attn(6, 1, 1, 1, [L], qc, qs, kc, ks, vc, vs)
    v = oracle.dequant_rows(vc, vs)
    assert np.allclose(out, np.tile(v.mean(0), (6, 1)), rtol=0, atol=1e-6 * np.abs(v).max())


def test_two_keys_closed_form():
    # q = e_0 * 1, k0 = e_0 * a, k1 = e_0 * b: weight of key 0 is 1 / (1 + exp(-(a - b) * scale))
    qc = np.zeros((1, 64), np.uint8); qc[0, 0] = 0x02          # q[0] = 1.0
    qs = np.full((1, 8), 0x38, np.uint8)                          # scales 1.0
    kc = np.zeros((2, 64), np.uint8); kc[0, 0] = 0x07; kc[1, 0] = 0x0D   # k0[0] = 6, k1[0] = -3
    ks = np.full((2, 8), 0x38, np.uint8)
    vc = np.zeros((2, 64), np.uint8); vc[0, 0] = 0x02; vc[1, 0] = 0x04   # v0[0] = 1, v1[0] = 2
    vs = np.full((2, 8), 0x38, np.uint8)
    sc = 0.5
    out = _attn(1, 1, 1, 1, [2], qc, qs, kc, ks, vc, vs, sm_scale=sc)
    w0 = 1.0 / (1.0 + math.exp(-(6.0 - (-3.0)) * sc))
    assert abs(out[0, 0] - (w0 * 1.0 + (1 - w0) * 2.0)) < 1e-6
    assert np.all(out[0, 1:] == 0)


def test_matches_torch_sdpa_gqa_causal():
    rng = np.random.default_rng(9)
    Hq, Hkv, q_len = 12, 4, 3
    seq_lens = [5, 40, 17]
    T = sum(seq_lens)
    kc, ks = _rand_quant(rng, T * Hkv)
    vc, vs = _rand_quant(rng, T * Hkv)
    qc, qs = _rand_quant(rng, len(seq_lens) * q_len * Hq)
    for causal in (1, 0):
        out = _attn(Hq, Hkv, q_len, causal, seq_lens, qc, qs, kc, ks, vc, vs)
        K = oracle.dequant_rows(kc, ks).reshape(T, Hkv, 128)
        V = oracle.dequant_rows(vc, vs).reshape(T, Hkv, 128)
        Q = oracle.dequant_rows(qc, qs).reshape(len(seq_lens), q_len, Hq, 128)
        ref_rows = []
        off = 0
        for s, L in enumerate(seq_lens):
            q = torch.from_numpy(Q[s]).permute(1, 0, 2)[None]                # [1, Hq, q_len, D]
            k = torch.from_numpy(K[off:off + L]).permute(1, 0, 2)[None]    # [1, Hkv, L, D]
            v = torch.from_numpy(V[off:off + L]).permute(1, 0, 2)[None]
            qpos = torch.arange(L - q_len, L)[:, None]
            kpos = torch.arange(L)[None, :]
            mask = (kpos <= qpos) if causal else torch.ones(q_len, L, dtype=torch.bool)
            o = torch.nn.functional.scaled_dot_product_attention(
                q, k, v, attn_mask=mask, scale=1.0 / math.sqrt(128), enable_gqa=True)
            ref_rows.append(o[0].permute(1, 0, 2).reshape(-1, 128).numpy())
            off += L
        ref = np.concatenate(ref_rows)
        assert np.allclose(out, ref, rtol=1e-6, atol=1e-6)


def test_joint_rotation_preserves_scores():
    # before quantisation, <H rope(q), H rope(k)> = <rope(q), rope(k)>: the rotation may be
    # applied to both sides without changing the attention scores
    w = synth.tiny_decode()
    t = oracle.rope_table(64, 32, 1e7, 1.0)
    q = synth.bf16_bits_to_float(w.q_rows(0, 50, 1)[0, 0])
    k = synth.bf16_bits_to_float(w.k_rows(0, 40, 1)[0, 0])
    rq, rk = oracle.rope_apply(q, t, 50, 32), oracle.rope_apply(k, t, 40, 32)
    hq, hk = oracle.fwht128(rq), oracle.fwht128(rk)
    a = float(rq.astype(np.float64) @ rk.astype(np.float64))
    b = float(hq.astype(np.float64) @ hk.astype(np.float64))
    assert abs(a - b) <= 1e-5 * np.linalg.norm(rq) * np.linalg.norm(rk)
    # and after quantisation the scores stay close (FP4 noise, outliers spread by the rotation)
    cq, sq = oracle.quantize_row(hq)
    ck, sk = oracle.quantize_row(hk)
    c = float(oracle.dequant_rows(cq, sq)[0] @ oracle.dequant_rows(ck, sk)[0])
    assert abs(c - a) <= 0.15 * np.linalg.norm(rq) * np.linalg.norm(rk)


def test_quantize_rows_composes_rope_fwht_quant():
    w = synth.tiny_decode()
    t = oracle.rope_table(300, 32, 1e7, 1.0)
    k = w.k_rows(0, 100, 5)              # [5, 4, 128]
    pos = np.repeat(np.arange(100, 105, dtype=np.int32), 4)
    codes, scales = oracle.quantize_rows(k.reshape(-1, 128), pos, True, t, 32)
    for r in range(20):
        x = synth.bf16_bits_to_float(k.reshape(-1, 128)[r])
        c, s = oracle.quantize_row(oracle.fwht128(oracle.rope_apply(x, t, int(pos[r]), 32)))
        assert np.array_equal(c, codes[r]) and np.array_equal(s, scales[r])
    v = w.v_rows(0, 100, 5)
    vc, vs = oracle.quantize_rows(v.reshape(-1, 128), None, False, None, 0)
    c, s = oracle.quantize_row(synth.bf16_bits_to_float(v.reshape(-1, 128)[3]))
    assert np.array_equal(c, vc[3]) and np.array_equal(s, vs[3])


@pytest.mark.parametrize("H", [3, 4])
def test_paged_gather_layout(H):
    # fill every byte of a pool with a value naming (page, region, head, slot, byte) per the
    # documented block layout, then check the gather returns each slot's own bytes
    P = 6
    blk = H * 9216
    pool = np.zeros(P * blk, np.uint8)
    for p in range(P):
        b = pool[p * blk:(p + 1) * blk]
        for h in range(H):
            for k in range(64):
                for j in range(64):
                    b[h * 4096 + (k // 8) * 512 + (j // 16) * 128 + (k % 8) * 16 + j % 16] = (p * 7 + h * 3 + k + j) % 251
                    b[H * 4608 + h * 4096 + k * 64 + j] = (p * 5 + h + 2 * k + j) % 253
                for j in range(8):
                    # K scale j of slot k: head pair h // 2, half c = j // 4; rows of 16 bytes
                    # (keys k % 32, both heads) for a full pair, 8 bytes for a last lone head
                    c, pair = j // 4, H * 4096 + (h // 2) * 1024
                    if h % 2 == 1 or h + 1 < H:
                        off = pair + c * 512 + (k % 32) * 16 + (h % 2) * 8 + (k // 32) * 4 + j % 4
                    else:
                        off = pair + c * 256 + (k % 32) * 8 + (k // 32) * 4 + j % 4
                    b[off] = (p + h * 11 + k + 3 * j) % 241
                    b[H * 8704 + h * 512 + k * 8 + j] = (p * 13 + h + k + j) % 239
    bt = np.array([[4, 1, 5], [0, 2, 3]], np.int32)
    kc, ks, vc, vs, bad = oracle.paged_gather(pool, P, H, bt, 1, 60, 70)
    assert bad == 0
    for i in range(70):
        pos = 60 + i
        p, k = bt[1, pos // 64], pos % 64
        for h in range(H):
            assert list(kc[i, h]) == [(p * 7 + h * 3 + k + j) % 251 for j in range(64)]
            assert list(vc[i, h]) == [(p * 5 + h + 2 * k + j) % 253 for j in range(64)]
            assert list(ks[i, h]) == [(p + h * 11 + k + 3 * j) % 241 for j in range(8)]
            assert list(vs[i, h]) == [(p * 13 + h + k + j) % 239 for j in range(8)]
    bt2 = np.array([[4, 9]], np.int32)
    *_, bad = oracle.paged_gather(pool, P, H, bt2, 0, 0, 100)
    assert bad == (100 - 64) * H
