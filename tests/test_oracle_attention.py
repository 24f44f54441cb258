"""Pins for the oracle's attention and paged-layout gather (CPU only).

Attention is checked against closed forms (one key, equal scores, two keys), against
torch's scaled_dot_product_attention in float64 on the oracle's own dequantised arrays (GQA head
mapping, causal offsets, scale), and the joint-rotation invariance of Q.K^T. The unquantised
reference (the baseline of the cosine report) is checked against torch float64 SDPA on rows rotated
by an independent float64 RoPE, and for the relative-position property of the key rotation.
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


def _rope64(x, pos, rot_dim, theta, pos_scale):
    """RoPE written independently in float64 with torch: pairs (i, i + rot_dim/2) rotated by
    (pos / pos_scale) * theta^(-2i/rot_dim). x [n, 128], pos [n]."""
    half = rot_dim // 2
    i = torch.arange(half, dtype=torch.float64)
    inv = theta ** (-2.0 * i / rot_dim)
    ang = (pos.to(torch.float64)[:, None] / pos_scale) * inv[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    a, b = x[:, :half], x[:, half:rot_dim]
    return torch.cat([a * c - b * s, b * c + a * s, x[:, rot_dim:]], dim=1)


@pytest.mark.parametrize("rot_dim,pos_scale,causal", [(32, 1.0, 1), (32, 600000 / 262144, 1),
                                                       (32, 1.0, 0), (128, 1.0, 1), (0, 1.0, 1)])
def test_unquantized_reference_matches_torch_sdpa(rot_dim, pos_scale, causal):
    # The unquantised attention behind the cosine report: bf16 q/k/v widened exactly, RoPE on q at
    # its own position (len - q_len + i) and on key t at position t, GQA head h -> kv head
    # h // group, causal offsets; against torch float64 SDPA on rows rotated by an independent
    # float64 RoPE. The oracle's fp32 table and products differ by rounding only (~1e-7).
    Hq, Hkv, q_len, theta = 12, 4, 3, 1e7
    seq_lens = [5, 70, 23]
    T = sum(seq_lens)
    q = synth.normal_bf16(5, 1, 0, 0, len(seq_lens) * q_len, Hq)
    k = synth.normal_bf16(5, 2, 0, 0, T, Hkv)
    v = synth.normal_bf16(5, 3, 0, 0, T, Hkv)
    max_pos = max(seq_lens)
    table = oracle.rope_table(max_pos, rot_dim, theta, pos_scale) if rot_dim else \
        np.zeros(1, np.float32)
    sl = np.asarray(seq_lens, np.int32)
    tok_off = np.concatenate([[0], np.cumsum(sl)[:-1]]).astype(np.int64)
    rows = [(s, i, h) for s in range(len(seq_lens)) for i in range(q_len) for h in range(Hq)]
    rs, rt, rh = (np.array(x, np.int32) for x in zip(*rows))
    sm = 1.0 / math.sqrt(128)
    out = oracle.attention_ref_rows(Hq, Hkv, q_len, causal, sm, sl, tok_off,
                                    q.reshape(-1, 128), k.reshape(-1, 128), v.reshape(-1, 128),
                                    table, rot_dim, rs, rt, rh)
    f64 = lambda a: torch.from_numpy(synth.bf16_bits_to_float(a).astype(np.float64))
    Q, K, V = f64(q), f64(k), f64(v)          # [S*q_len, Hq, D], [T, Hkv, D]
    ref = []
    off = 0
    for s, L in enumerate(seq_lens):
        qpos = torch.arange(L - q_len, L)
        kpos = torch.arange(L)
        qs = Q[s * q_len:(s + 1) * q_len]   # [q_len, Hq, D]
        ks, vs = K[off:off + L], V[off:off + L]
        if rot_dim:
            qs = _rope64(qs.reshape(-1, 128), qpos.repeat_interleave(Hq), rot_dim, theta,
                         pos_scale).reshape(q_len, Hq, 128)
            ks = _rope64(ks.reshape(-1, 128), kpos.repeat_interleave(Hkv), rot_dim, theta,
                         pos_scale).reshape(L, Hkv, 128)
        mask = (kpos[None, :] <= qpos[:, None]) if causal else torch.ones(q_len, L, dtype=torch.bool)
        o = torch.nn.functional.scaled_dot_product_attention(
            qs.permute(1, 0, 2)[None], ks.permute(1, 0, 2)[None], vs.permute(1, 0, 2)[None],
            attn_mask=mask, scale=sm, enable_gqa=True)
        ref.append(o[0].permute(1, 0, 2).reshape(-1, 128).numpy())
        off += L
    ref = np.concatenate(ref)
    assert np.allclose(out, ref, rtol=0, atol=2e-5), np.abs(out - ref).max()


def test_unquantized_reference_key_positions_are_relative():
    # RoPE makes a score depend on the query and key positions only through their difference.
    # Sequence B repeats sequence A's keys and values D positions later, after D keys of zeros
    # (score 0) whose values are zero; the query rows are the same bf16 rows, so B's query sits D
    # positions after A's. With the real keys' scores far above 0 the filler keys get weight
    # below e^-40, so the outputs agree to fp32 rounding if and only if every key is rotated at
    # its own position t and the query at len - q_len + i.
    Hq, Hkv, q_len, D, L = 4, 1, 2, 37, 9
    q = np.zeros((2 * q_len, Hq, 128), np.uint16)
    k = np.zeros((L + L + D, Hkv, 128), np.uint16)
    v = np.zeros_like(k)
    rng = np.random.default_rng(3)
    bf = lambda x: (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    # q and k both large along the rotary dims' partner pairs and a non-rotary dim, so that
    # every score is large and positive and depends on the relative position
    qa = np.zeros((q_len, Hq, 128), np.float32)
    qa[..., 0] = 8.0; qa[..., 16] = 8.0; qa[..., 100] = 24.0
    ka = np.zeros((L, Hkv, 128), np.float32)
    ka[..., 0] = rng.uniform(2, 4, (L, Hkv)); ka[..., 16] = rng.uniform(2, 4, (L, Hkv))
    ka[..., 100] = rng.uniform(3, 5, (L, Hkv))
    va = rng.standard_normal((L, Hkv, 128)).astype(np.float32)
    q[:q_len] = bf(qa); q[q_len:] = bf(qa)
    k[:L] = bf(ka); k[L + D:] = bf(ka)
    v[:L] = bf(va); v[L + D:] = bf(va)
    sl = np.array([L, L + D], np.int32)
    tok_off = np.array([0, L], np.int64)
    table = oracle.rope_table(L + D, 32, 1e7, 1.0)
    rows = [(s, i, h) for s in range(2) for i in range(q_len) for h in range(Hq)]
    rs, rt, rh = (np.array(x, np.int32) for x in zip(*rows))
    out = oracle.attention_ref_rows(Hq, Hkv, q_len, 1, 1.0, sl, tok_off, q.reshape(-1, 128),
                                    k.reshape(-1, 128), v.reshape(-1, 128), table, 32, rs, rt, rh)
    a, b = out[:q_len * Hq], out[q_len * Hq:]
    assert np.allclose(a, b, rtol=0, atol=1e-5), np.abs(a - b).max()
    # the positions matter: with both sequences' keys at the same absolute positions (no shift)
    # the two would differ, so the agreement above is not a trivial one
    t2 = oracle.rope_table(L + D, 32, 1e7, 1.0 / 64)
    out2 = oracle.attention_ref_rows(Hq, Hkv, q_len, 1, 1.0, sl, tok_off, q.reshape(-1, 128),
                                     k.reshape(-1, 128), v.reshape(-1, 128), t2, 32, rs, rt, rh)
    assert np.allclose(out2[:q_len * Hq], out2[q_len * Hq:], rtol=0, atol=1e-5)
    c = oracle.attention_ref_rows(Hq, Hkv, q_len, 1, 1.0, sl[:1], tok_off[:1], q[:q_len].reshape(-1, 128),
                                  k[:L].reshape(-1, 128), v[:L].reshape(-1, 128), t2, 32,
                                  rs[:q_len * Hq], rt[:q_len * Hq], rh[:q_len * Hq])
    assert not np.allclose(c, out[:q_len * Hq], rtol=0, atol=1e-3)
