"""Comparator KV formats (bf16, int8, NVFP4 K + fp16 V) on the GPU against the oracle.

Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)" (144 B per token
per KV head against 264 for int8 and 512 for bf16; upstream NVFP4 K with fp16 V). The appended
rows (and the bf16 Q rows) must be byte-identical to the oracle's encoding of the same bf16
inputs; the decode output must be within the attention tolerance of the oracle's fp64 attention
over the decoded rows.
"""
import numpy as np
import pytest

import oracle
import synth
from kvrun import MAX_ABS_TOL, REL_L2_TOL, attention_errors

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FORMATS = [0, 1, 2]


class CmpRun:
    def __init__(self, w: synth.Workload, fmt: int):
        import bit_kv_cache_03_gb300 as kv
        self.kv, self.w, self.fmt = kv, w, fmt
        self.dev = torch.device("cuda")
        self.L = kv.make_layout(w.q_heads, w.kv_heads, 128, 64, w.rot_dim)
        self.pb = kv.kv_cmp_page_bytes(self.L, fmt)
        self.pool = torch.zeros(w.pool_pages * self.pb, dtype=torch.uint8, device=self.dev)
        self.bt = torch.from_numpy(np.ascontiguousarray(w.block_table, np.int32)).to(self.dev)
        self.rope = torch.empty(max(1, w.max_pos * w.rot_dim), dtype=torch.float32, device=self.dev)
        kv.kv_nvfp4_rope_table_init(self.rope, w.max_pos, w.rot_dim, w.theta, w.pos_scale)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)
        for s, c in enumerate(w.cached_lens):
            if c == 0:
                continue
            k, v, pos = w.cached_tokens(s, 0, c)
            self._append(None, k, v, np.full(c, s, np.int32), pos, None)
        q, k, v, sid, pos = w.new_tokens()
        self.T = q.shape[0]
        self.q_out = torch.empty(self.T * w.q_heads * 128, dtype=torch.bfloat16, device=self.dev)
        self._append(q, k, v, sid, pos, self.q_out)
        self.out = torch.full((self.T * w.q_heads * 128,), float("nan"), dtype=torch.float32,
                              device=self.dev)

    def _bf16(self, a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(self.dev).view(torch.bfloat16)

    def _append(self, q, k, v, sid, pos, q_out):
        w = self.w
        self.kv.kv_cmp_append(self.L, self.fmt, None if q is None else self._bf16(q), self._bf16(k),
                              self._bf16(v), torch.from_numpy(sid).to(self.dev),
                              torch.from_numpy(pos).to(self.dev), len(pos), self.rope, w.max_pos,
                              self.bt, w.num_seqs, w.max_pages, w.pool_pages, self.pool, q_out,
                              self.status)

    def attend(self, chunk):
        w, kv = self.w, self.kv
        n = kv.kv_cmp_plan_workspace_bytes(self.L, w.seq_lens, w.q_len, w.causal, chunk)
        self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.dev)
        plan = kv.kv_cmp_plan(self.L, w.seq_lens, w.q_len, w.causal, chunk, self.ws, n)
        kv.kv_cmp_decode_attn(self.L, self.fmt, plan, self.ws, self.q_out, w.sm_scale, self.pool,
                              w.pool_pages, self.bt, w.max_pages, self.out, self.status)
        torch.cuda.synchronize()
        return self.out.view(self.T, w.q_heads, 128).cpu().numpy()


def _table(w):
    return oracle.rope_table(w.max_pos, w.rot_dim, w.theta, w.pos_scale)


def _encoded_seq(w, fmt, s, table, n=None):
    """The oracle's K and V rows of sequence s ([n, H, row bytes] each)."""
    L = int(w.seq_lens[s]) if n is None else n
    H = w.kv_heads
    pos = np.repeat(np.arange(L, dtype=np.int32), H)
    k = oracle.cmp_encode_rows(fmt, 1, w.k_rows(s, 0, L).reshape(-1, 128), pos, table, w.rot_dim)
    v = oracle.cmp_encode_rows(fmt, 2, w.v_rows(s, 0, L).reshape(-1, 128), pos, table, w.rot_dim)
    return k.reshape(L, H, -1), v.reshape(L, H, -1)


def _check_rows_and_q(r: CmpRun, table):
    w, fmt = r.w, r.fmt
    pool = r.pool.cpu().numpy()
    for s in range(w.num_seqs):
        k, v = _encoded_seq(w, fmt, s, table)
        gk, gv, bad = oracle.cmp_paged_gather(fmt, pool, w.pool_pages, w.kv_heads,
                                              w.block_table, s, 0, int(w.seq_lens[s]))
        assert bad == 0
        assert np.array_equal(gk, k), f"K rows of sequence {s}"
        assert np.array_equal(gv, v), f"V rows of sequence {s}"
    q, *_ = w.new_tokens()
    pos = np.repeat(np.concatenate([np.arange(int(L) - w.q_len, int(L)) for L in w.seq_lens]),
                    w.q_heads).astype(np.int32)
    want = oracle.cmp_encode_rows(fmt, 0, q.reshape(-1, 128), pos, table, w.rot_dim)
    got = r.q_out.view(torch.int16).cpu().numpy().view(np.uint8).reshape(want.shape)
    assert np.array_equal(got, want)


def _oracle_attention(w, fmt, table):
    ks, vs = [], []
    for s in range(w.num_seqs):
        k, v = _encoded_seq(w, fmt, s, table)
        ks.append(oracle.cmp_decode_rows(fmt, 1, k.reshape(-1, k.shape[-1])))
        vs.append(oracle.cmp_decode_rows(fmt, 2, v.reshape(-1, v.shape[-1])))
    q, *_ = w.new_tokens()
    pos = np.repeat(np.concatenate([np.arange(int(L) - w.q_len, int(L)) for L in w.seq_lens]),
                    w.q_heads).astype(np.int32)
    qd = oracle.cmp_decode_rows(fmt, 0, oracle.cmp_encode_rows(fmt, 0, q.reshape(-1, 128), pos,
                                                               table, w.rot_dim))
    rows = [(s, i, h) for s in range(w.num_seqs) for i in range(w.q_len) for h in range(w.q_heads)]
    rs, rt, rh = (np.array(x, np.int32) for x in zip(*rows))
    ref = oracle.attention_f64_rows(w.q_heads, w.kv_heads, w.q_len, w.causal, w.sm_scale,
                                    w.seq_lens, w.tok_off(), qd, np.concatenate(ks),
                                    np.concatenate(vs), rs, rt, rh)
    return ref.reshape(-1, w.q_heads, 128)


CASES = [
    # name, cached lengths, q_len, causal, chunk
    ("cmp_decode", [700, 64, 3], 1, True, 64),        # split groups, a one-page and a tiny seq
    ("cmp_verify", [300, 129], 2, True, 128),         # 12 rows per head: two row groups
    ("cmp_nocausal", [257, 1000], 3, False, 256),     # 18 rows, every key visible
]


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_comparator_append_and_decode_match_the_oracle(fmt, case):
    name, lens, q_len, causal, chunk = case
    w = synth.Workload(name, lens, q_len=q_len, causal=causal, seed=40 + fmt, chunk_tokens=chunk)
    r = CmpRun(w, fmt)
    table = _table(w)
    _check_rows_and_q(r, table)
    got = r.attend(chunk)
    assert np.isfinite(got).all()
    max_abs, rel = attention_errors(got, _oracle_attention(w, fmt, table))
    assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, (max_abs, rel)
    assert int(r.status.item()) == 0


@pytest.mark.parametrize("fmt", FORMATS)
def test_comparator_flags_a_page_outside_the_pool(fmt):
    kv = pytest.importorskip("bit_kv_cache_03_gb300")
    w = synth.Workload("cmp_bad", [200], q_len=1, seed=7)
    r = CmpRun(w, fmt)
    assert int(r.status.item()) == 0
    bt = r.bt.clone()
    r.bt[0, 1] = 10 ** 6  # the page of keys 64..127
    r.attend(64)
    assert int(r.status.item()) & kv.DEV_BAD_PAGE
    r.bt.copy_(bt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_comparator_bench_size_sampled(fmt):
    # the 4 x 131072-token cache in the launch configuration the benchmark times; the oracle
    # checks the new token's rows of sequence 0 (all 24 heads over 131073 keys) and every K/V row
    # of sequence 0
    w = synth.steady_decode()
    r = CmpRun(w, fmt)
    got = r.attend(64)
    table = _table(w)
    k, v = _encoded_seq(w, fmt, 0, table)
    pool = r.pool.cpu().numpy()
    gk, gv, bad = oracle.cmp_paged_gather(fmt, pool, w.pool_pages, w.kv_heads, w.block_table, 0,
                                          0, int(w.seq_lens[0]))
    assert bad == 0 and np.array_equal(gk, k) and np.array_equal(gv, v)
    kd = oracle.cmp_decode_rows(fmt, 1, k.reshape(-1, k.shape[-1]))
    vd = oracle.cmp_decode_rows(fmt, 2, v.reshape(-1, v.shape[-1]))
    q, *_ = w.new_tokens()
    L = int(w.seq_lens[0])
    qd = oracle.cmp_decode_rows(fmt, 0, oracle.cmp_encode_rows(
        fmt, 0, q[0].reshape(-1, 128), np.full(w.q_heads, L - 1, np.int32), table, w.rot_dim))
    rows = np.arange(w.q_heads, dtype=np.int32)
    ref = oracle.attention_f64_rows(w.q_heads, w.kv_heads, 1, True, w.sm_scale,
                                    np.array([L], np.int32), np.array([0], np.int64), qd, kd, vd,
                                    np.zeros(w.q_heads, np.int32), np.zeros(w.q_heads, np.int32),
                                    rows)
    max_abs, rel = attention_errors(got[0], ref)
    assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, (max_abs, rel)
    assert np.isfinite(got).all()
    assert int(r.status.item()) == 0
