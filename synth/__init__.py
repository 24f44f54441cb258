"""Seeded synthetic workloads for the NVFP4 KV cache (shared by the tests, the oracle and the bench).

Holds random-number generation and workload shapes only; none of the method's arithmetic.
The generator itself is C (``synth.c``, a counter-based splitmix64 stream with Box-Muller
normals rounded once to bf16), compiled on first use.

Workloads mirror the shapes the source pages describe for a Qwen-family 27B model with an NVFP4
KV cache (prismix.dev/news/833001997676, sections "NVFP4 KV cache (from scratch)" and "YaRN
context extension"): 24 query heads over 4 KV heads (GQA 6), head_dim 128, 64-token pages,
RoPE on the first 32 dims with theta = 1e7, bf16 Q/K/V ~ N(0, 1) with K and Q channels
3, 77, 101 and 120 scaled by 12 as outliers.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_SRC = os.path.join(_HERE, "synth.c")

STREAM_Q, STREAM_K, STREAM_V = 1, 2, 3
STREAM_PAGES, STREAM_LENS = 100, 101
OUTLIER_CHANNELS = (3, 77, 101, 120)
OUTLIER_MULT = 12.0


def build(force: bool = False) -> str:
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
                    _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u64, i32, f64, p = ctypes.c_uint64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
        L.synth_stream_key.argtypes = [u64, u64]
        L.synth_stream_key.restype = u64
        L.synth_draw.argtypes = [u64, u64]
        L.synth_draw.restype = u64
        L.synth_normal_bf16.argtypes = [u64, u64, i32, i32, i32, i32, i32, p, i32, f64, p, i32]
        L.synth_normal_bf16.restype = None
        L.synth_permutation.argtypes = [u64, u64, i32, p]
        L.synth_permutation.restype = None
        L.synth_loguniform_int.argtypes = [u64, u64, i32, f64, f64, p]
        L.synth_loguniform_int.restype = None
        L.synth_uniform_int.argtypes = [u64, u64, i32, i32, p]
        L.synth_uniform_int.restype = None
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def normal_bf16(seed, stream, seq, pos0, n_tok, heads, dim=128, outliers=(), mult=1.0,
                nthreads=0) -> np.ndarray:
    """bf16 bit patterns [n_tok, heads, dim] ~ N(0,1) for positions pos0.. of sequence `seq`."""
    out = np.empty((n_tok, heads, dim), np.uint16)
    o = np.asarray(outliers, np.int32)
    lib().synth_normal_bf16(seed, stream, seq, pos0, n_tok, heads, dim, _p(o), len(o), mult,
                            _p(out), nthreads)
    return out


def permutation(seed, stream, n) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().synth_permutation(seed, stream, n, _p(out))
    return out


def loguniform_int(seed, stream, n, lo, hi) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().synth_loguniform_int(seed, stream, n, lo, hi, _p(out))
    return out


def uniform_int(seed, stream, n, m) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().synth_uniform_int(seed, stream, n, m, _p(out))
    return out


def bf16_bits_to_float(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (a bit shift, no rounding)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


@dataclass
class Workload:
    """One attention layer's worth of paged NVFP4 cache plus one batch of new tokens.

    cached_lens[s] tokens of sequence s are already in the cache; the step appends q_len new
    tokens per sequence (positions cached_lens[s] .. cached_lens[s]+q_len-1) and attends with
    them. seq_lens = cached_lens + q_len.
    """
    name: str
    cached_lens: list
    q_len: int = 1
    causal: bool = True
    seed: int = 0
    q_heads: int = 24
    kv_heads: int = 4
    head_dim: int = 128
    page_size: int = 64
    rot_dim: int = 32
    theta: float = 1e7
    pos_scale: float = 1.0
    chunk_tokens: int = 1024
    pool_pages: int | None = None      # default: exactly the pages needed
    placement: str = "permuted"        # "identity" or "permuted"
    outliers: tuple = OUTLIER_CHANNELS
    outlier_mult: float = OUTLIER_MULT
    block_table: np.ndarray = field(init=False, repr=False)

    def __post_init__(self):
        self.cached_lens = [int(x) for x in self.cached_lens]
        P = self.page_size
        self.pages_per_seq = [(c + self.q_len + P - 1) // P for c in self.cached_lens]
        need = sum(self.pages_per_seq)
        if self.pool_pages is None:
            self.pool_pages = need
        assert self.pool_pages >= need, "pool too small for the workload"
        self.max_pages = max(self.pages_per_seq) if self.pages_per_seq else 1
        if self.placement == "identity":
            order = np.arange(self.pool_pages, dtype=np.int32)
        else:
            order = permutation(self.seed, STREAM_PAGES, self.pool_pages)
        bt = np.full((self.num_seqs, self.max_pages), -1, np.int32)
        at = 0
        for s, n in enumerate(self.pages_per_seq):
            bt[s, :n] = order[at:at + n]
            at += n
        self.block_table = bt

    # ---- shapes -----------------------------------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return len(self.cached_lens)

    @property
    def seq_lens(self) -> np.ndarray:
        return np.asarray(self.cached_lens, np.int32) + self.q_len

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def max_pos(self) -> int:
        return int(self.seq_lens.max())

    @property
    def kv_tokens(self) -> int:
        return int(self.seq_lens.sum())

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def tok_off(self) -> np.ndarray:
        """Start of each sequence in a flat [token] layout of all seq_lens tokens."""
        return np.concatenate([[0], np.cumsum(self.seq_lens)[:-1]]).astype(np.int64)

    # ---- values -----------------------------------------------------------------------------
    def k_rows(self, seq, pos0, n, nthreads=0):
        return normal_bf16(self.seed, STREAM_K, seq, pos0, n, self.kv_heads, self.head_dim,
                           self.outliers, self.outlier_mult, nthreads)

    def v_rows(self, seq, pos0, n, nthreads=0):
        return normal_bf16(self.seed, STREAM_V, seq, pos0, n, self.kv_heads, self.head_dim,
                           (), 1.0, nthreads)

    def q_rows(self, seq, pos0, n, nthreads=0):
        return normal_bf16(self.seed, STREAM_Q, seq, pos0, n, self.q_heads, self.head_dim,
                           self.outliers, self.outlier_mult, nthreads)

    def new_tokens(self):
        """The step's appended tokens, sequence-major: q [S*q_len, Hq, D], k/v [S*q_len, Hkv, D]
        (bf16 bits), seq ids and positions [S*q_len]."""
        qs, ks, vs, sid, pos = [], [], [], [], []
        for s, c in enumerate(self.cached_lens):
            qs.append(self.q_rows(s, c, self.q_len))
            ks.append(self.k_rows(s, c, self.q_len))
            vs.append(self.v_rows(s, c, self.q_len))
            sid.append(np.full(self.q_len, s, np.int32))
            pos.append(np.arange(c, c + self.q_len, dtype=np.int32))
        return (np.concatenate(qs), np.concatenate(ks), np.concatenate(vs),
                np.concatenate(sid), np.concatenate(pos))

    def cached_tokens(self, seq, pos0=0, n=None, nthreads=0):
        """Cached K/V rows of one sequence: k, v [n, Hkv, D] bf16 bits, positions [n]."""
        if n is None:
            n = self.cached_lens[seq] - pos0
        return (self.k_rows(seq, pos0, n, nthreads), self.v_rows(seq, pos0, n, nthreads),
                np.arange(pos0, pos0 + n, dtype=np.int32))


def tiny_decode(seed=0) -> Workload:
    """1 sequence, 4096 cached + 1 appended token, identity page table."""
    return Workload("tiny_decode_4k", [4096], q_len=1, seed=seed, placement="identity")


def steady_decode(seed=0) -> Workload:
    """4 sequences x 131072 cached + 1 new token; pages from a seeded permutation of a
    40,000-page pool."""
    return Workload("steady_decode_4x128k", [131072] * 4, q_len=1, seed=seed, pool_pages=40000)


def ragged_decode(seed=0) -> Workload:
    """8 sequences, cached lengths log-uniform in [8192, 262144], 1 new token each, seeded page
    placement, split-K over 1024-token chunks."""
    lens = loguniform_int(seed, STREAM_LENS, 8, 8192.0, 262144.0)
    return Workload("ragged_decode_8seq", list(lens), q_len=1, seed=seed, chunk_tokens=1024)


def spec_verify(seed=0) -> Workload:
    """4 sequences x 100000 cached + 8 query tokens (1 accepted + 7 draft), causal among the 8."""
    return Workload("spec_verify_4x100k_q8", [100000] * 4, q_len=8, causal=True, seed=seed)


def prefill_chunk(seed=0) -> Workload:
    """1 sequence, 591872 cached + an 8192-token causal chunk, positions scaled by 600000/262144."""
    return Workload("prefill_chunk_600k", [591872], q_len=8192, causal=True, seed=seed,
                    pos_scale=600000.0 / 262144.0)


CONFIGS = {
    "tiny": tiny_decode,
    "steady": steady_decode,
    "ragged": ragged_decode,
    "verify": spec_verify,
    "prefill": prefill_chunk,
}
