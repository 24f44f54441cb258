"""Test/bench plumbing: run a synthetic workload through the CUDA path and through the oracle.

The two sides share only the seeded inputs from `synth`. The CUDA side goes through the C ABI
(via the Python binding); the oracle side re-quantises the same bf16 rows on the CPU.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
import synth


# ------------------------------------------------------------------------------------------------
# CUDA path
# ------------------------------------------------------------------------------------------------
class GpuRun:
    def __init__(self, w: synth.Workload, device="cuda", populate_batch=1 << 17, nthreads=0):
        import torch

        import bit_kv_cache_03_gb300 as kv
        self.w = w
        self.torch = torch
        self.kv = kv
        self.dev = torch.device(device)
        self.cache = kv.PagedNVFP4Cache(w.pool_pages, w.block_table, w.max_pos, w.q_heads,
                                        w.kv_heads, w.rot_dim, w.theta, w.pos_scale, device)
        self._populate(populate_batch, nthreads)
        q, k, v, sid, pos = w.new_tokens()
        self.T = q.shape[0]
        self.q = self._bf16(q)
        self.k = self._bf16(k)
        self.v = self._bf16(v)
        self.sid = torch.from_numpy(sid).to(self.dev)
        self.pos = torch.from_numpy(pos).to(self.dev)
        self.q_codes, self.q_scales = self.cache.quantized_q_buffers(self.T)
        self.out = torch.zeros(self.T * w.q_heads * 128, dtype=torch.float32, device=self.dev)

    def _bf16(self, a):
        t = self.torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
        return t.to(self.dev).view(self.torch.bfloat16)

    def _populate(self, batch, nthreads):
        """Quantize-append every cached token through the same append entry point."""
        w = self.w
        for s, c in enumerate(w.cached_lens):
            for p0 in range(0, c, batch):
                n = min(batch, c - p0)
                k, v, pos = w.cached_tokens(s, p0, n, nthreads)
                sid = np.full(n, s, np.int32)
                self.cache.append(self._bf16(k), self._bf16(v),
                                  self.torch.from_numpy(sid).to(self.dev),
                                  self.torch.from_numpy(pos).to(self.dev))

    def step(self, chunk_tokens=None, plan=True):
        """One pass of the hot path: append the new tokens (with Q), plan, attend."""
        w = self.w
        self.cache.append(self.k, self.v, self.sid, self.pos, q=self.q, q_codes=self.q_codes,
                          q_scales=self.q_scales)
        if plan:
            self.cache.plan(w.seq_lens, w.q_len, w.causal, chunk_tokens or w.chunk_tokens)
        self.cache.attend(self.q_codes, self.q_scales, self.out, sm_scale=w.sm_scale)

    def step_fused(self, chunk_tokens=None, plan=True, q_out=True):
        """The same step through kv_nvfp4_decode_step: the append of the new tokens inside the
        attention launch (requires group * q_len <= 8)."""
        w, c = self.w, self.cache
        if plan:
            c.plan(w.seq_lens, w.q_len, w.causal, chunk_tokens or w.chunk_tokens)
        c.decode_step(self.q, self.k, self.v, self.out, self.q_codes if q_out else None,
                      self.q_scales if q_out else None, sm_scale=w.sm_scale)

    def status(self) -> int:
        return int(self.cache.status.item())

    def output(self) -> np.ndarray:
        return self.out.view(self.T, self.w.q_heads, 128).cpu().numpy()

    def q_quant(self):
        H = self.w.q_heads
        return (self.q_codes.view(self.T, H, 64).cpu().numpy(),
                self.q_scales.view(self.T, H, 8).cpu().numpy())

    def pool(self):
        return self.cache.pool.cpu().numpy()


# ------------------------------------------------------------------------------------------------
# Oracle path
# ------------------------------------------------------------------------------------------------
class OracleRun:
    """Quantise every K/V row of the workload (cached + new) and the new Q rows on the CPU."""

    def __init__(self, w: synth.Workload, nthreads=0):
        self.w = w
        self.nthreads = nthreads
        self.table = oracle.rope_table(w.max_pos, w.rot_dim, w.theta, w.pos_scale)
        H = w.kv_heads
        n = w.kv_tokens
        self.kc = np.empty((n, H, 64), np.uint8)
        self.ks = np.empty((n, H, 8), np.uint8)
        self.vc = np.empty((n, H, 64), np.uint8)
        self.vs = np.empty((n, H, 8), np.uint8)
        self.tok_off = w.tok_off()
        for s in range(w.num_seqs):
            L = int(w.seq_lens[s])
            k = w.k_rows(s, 0, L, nthreads)
            v = w.v_rows(s, 0, L, nthreads)
            pos = np.repeat(np.arange(L, dtype=np.int32), H)
            kc, ks = oracle.quantize_rows(k.reshape(-1, 128), pos, True, self.table, w.rot_dim,
                                          nthreads)
            vc, vs = oracle.quantize_rows(v.reshape(-1, 128), None, False, None, 0, nthreads)
            o = self.tok_off[s]
            self.kc[o:o + L] = kc.reshape(L, H, 64)
            self.ks[o:o + L] = ks.reshape(L, H, 8)
            self.vc[o:o + L] = vc.reshape(L, H, 64)
            self.vs[o:o + L] = vs.reshape(L, H, 8)
        q, _, _, _, pos = w.new_tokens()
        self.q_bf16 = q
        qpos = np.repeat(pos, w.q_heads)
        qc, qs = oracle.quantize_rows(q.reshape(-1, 128), qpos, True, self.table, w.rot_dim,
                                      nthreads)
        self.qc = qc.reshape(-1, w.q_heads, 64)
        self.qs = qs.reshape(-1, w.q_heads, 8)

    def all_rows(self):
        w = self.w
        rs, rt, rh = np.meshgrid(np.arange(w.num_seqs), np.arange(w.q_len), np.arange(w.q_heads),
                                 indexing="ij")
        return rs.ravel().astype(np.int32), rt.ravel().astype(np.int32), rh.ravel().astype(np.int32)

    def attention(self, rows=None) -> np.ndarray:
        w = self.w
        rs, rt, rh = rows if rows is not None else self.all_rows()
        return oracle.attention_rows(w.q_heads, w.kv_heads, w.q_len, w.causal, w.sm_scale,
                                     w.seq_lens, self.tok_off, self.qc, self.qs, self.kc, self.ks,
                                     self.vc, self.vs, rs, rt, rh, self.nthreads)

    def attention_unquantized(self, rows):
        """Reference without rotation or quantisation (bf16 inputs, same RoPE, fp64 math)."""
        w = self.w
        rs, rt, rh = rows
        H = w.kv_heads
        k = np.concatenate([w.k_rows(s, 0, int(w.seq_lens[s])) for s in range(w.num_seqs)])
        v = np.concatenate([w.v_rows(s, 0, int(w.seq_lens[s])) for s in range(w.num_seqs)])
        return oracle.attention_ref_rows(w.q_heads, H, w.q_len, w.causal, w.sm_scale, w.seq_lens,
                                         self.tok_off, self.q_bf16.reshape(-1, 128),
                                         k.reshape(-1, 128), v.reshape(-1, 128), self.table,
                                         w.rot_dim, rs, rt, rh, self.nthreads)


# ------------------------------------------------------------------------------------------------
# comparisons
# ------------------------------------------------------------------------------------------------
MAX_ABS_TOL = 2e-3
REL_L2_TOL = 1e-3


def attention_errors(got: np.ndarray, ref: np.ndarray):
    got = got.astype(np.float64).reshape(-1, 128)
    ref = ref.astype(np.float64).reshape(-1, 128)
    max_abs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    rel_l2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    return max_abs, rel_l2


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a = a.astype(np.float64).ravel()
    b = b.astype(np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def compare_pool(g: GpuRun, o: OracleRun):
    """Bit-exact comparison of every K/V row of the workload as stored in the GPU pool.
    Returns the number of mismatching rows per kind."""
    w = g.w
    pool = g.pool()
    bad = {"k_codes": 0, "k_scales": 0, "v_codes": 0, "v_scales": 0}
    for s in range(w.num_seqs):
        L = int(w.seq_lens[s])
        o0 = o.tok_off[s]
        kc, ks, vc, vs, nbad = oracle.paged_gather(pool, w.pool_pages, w.kv_heads, w.block_table,
                                                   s, 0, L)
        assert nbad == 0
        bad["k_codes"] += int(np.any(kc != o.kc[o0:o0 + L], axis=-1).sum())
        bad["k_scales"] += int(np.any(ks != o.ks[o0:o0 + L], axis=-1).sum())
        bad["v_codes"] += int(np.any(vc != o.vc[o0:o0 + L], axis=-1).sum())
        bad["v_scales"] += int(np.any(vs != o.vs[o0:o0 + L], axis=-1).sum())
    return bad


def sample_rows(w: synth.Workload, n: int, seed: int = 0):
    """Seeded sample of query rows that always includes the first and last chunk token of every
    head (used where the full oracle pass is too long)."""
    rs, rt, rh = [], [], []
    for s in range(w.num_seqs):
        for h in range(w.q_heads):
            for i in (0, w.q_len - 1):
                rs.append(s); rt.append(i); rh.append(h)
    extra = max(0, n - len(rs))
    if extra:
        r_s = synth.uniform_int(seed, 200, extra, w.num_seqs)
        r_t = synth.uniform_int(seed, 201, extra, w.q_len)
        r_h = synth.uniform_int(seed, 202, extra, w.q_heads)
        rs += list(r_s); rt += list(r_t); rh += list(r_h)
    return (np.array(rs, np.int32), np.array(rt, np.int32), np.array(rh, np.int32))


def sm_scale(w):
    return 1.0 / math.sqrt(w.head_dim)
