"""CPU oracle for the NVFP4 KV-cache method (ctypes wrapper over ``kv_oracle.cpp``).

TEST INFRASTRUCTURE ONLY. The product path (the CUDA library and its Python binding) never
imports this package; only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` do. The oracle shares no code with the CUDA path.

Every function states the page passage it restates:
  [NVFP4] prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)".
  [YaRN]  prismix.dev/news/833001997676, section "YaRN context extension".
  [Spill] prismix.dev/news/833001997676, section "Multi-level prefix reuse with host-KV safety
          net".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libkvoracle.so")
_SRC = os.path.join(_HERE, "kv_oracle.cpp")


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (strict IEEE: no contraction, no fast-math)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F64 = ctypes.c_double


def _declare(L):
    L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
    L.orc_e2m1_decode.restype = ctypes.c_float
    L.orc_e2m1_encode.argtypes = [ctypes.c_float]
    L.orc_e2m1_encode.restype = ctypes.c_uint8
    L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_decode.restype = ctypes.c_float
    L.orc_e4m3_encode.argtypes = [ctypes.c_float]
    L.orc_e4m3_encode.restype = ctypes.c_uint8
    L.orc_fwht_scale.argtypes = []
    L.orc_fwht_scale.restype = ctypes.c_float
    L.orc_rope_table.argtypes = [_I32, _I32, _F64, _F64, _P]
    L.orc_rope_table.restype = None
    L.orc_rope_apply.argtypes = [_P, _P, _I32, _I32]
    L.orc_rope_apply.restype = None
    L.orc_fwht128.argtypes = [_P]
    L.orc_fwht128.restype = None
    L.orc_quantize_row.argtypes = [_P, _P, _P]
    L.orc_quantize_row.restype = None
    L.orc_quantize_rows.argtypes = [_P, _I64, _P, _I32, _P, _I32, _P, _P, _I32]
    L.orc_quantize_rows.restype = None
    L.orc_dequant_rows.argtypes = [_P, _P, _I64, _P]
    L.orc_dequant_rows.restype = None
    L.orc_paged_gather.argtypes = [_P, _I32, _I32, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P]
    L.orc_paged_gather.restype = _I64
    L.orc_attention_rows.argtypes = [_I32, _I32, _I32, _I32, _F64, _P, _P, _P, _P, _P, _P, _P,
                                     _P, _I64, _P, _P, _P, _P, _I32]
    L.orc_attention_rows.restype = None
    L.orc_attention_ref_rows.argtypes = [_I32, _I32, _I32, _I32, _F64, _P, _P, _P, _P, _P, _P,
                                         _I32, _I64, _P, _P, _P, _P, _I32]
    L.orc_attention_ref_rows.restype = None
    for n in ("orc_bytes_per_token_head_nvfp4", "orc_bytes_per_token_head_int8",
              "orc_bytes_per_token_head_bf16"):
        getattr(L, n).argtypes = [_I32]
        getattr(L, n).restype = _I32
    L.orc_float_to_bf16.argtypes = [ctypes.c_float]
    L.orc_float_to_bf16.restype = ctypes.c_uint16
    L.orc_float_to_f16.argtypes = [ctypes.c_float]
    L.orc_float_to_f16.restype = ctypes.c_uint16
    L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
    L.orc_f16_to_double.restype = ctypes.c_double
    L.orc_int8_quantize_row.argtypes = [_P, _P, _P]
    L.orc_cmp_row_bytes.argtypes = [_I32, _I32]
    L.orc_cmp_row_bytes.restype = _I32
    L.orc_cmp_encode_rows.argtypes = [_I32, _I32, _P, _I64, _P, _P, _I32, _P]
    L.orc_cmp_decode_rows.argtypes = [_I32, _I32, _P, _I64, _P]
    L.orc_cmp_paged_gather.argtypes = [_I32, _P, _I32, _I32, _P, _I32, _I32, _I32, _I32, _P, _P]
    L.orc_cmp_paged_gather.restype = _I64
    L.orc_attention_f64_rows.argtypes = [_I32, _I32, _I32, _I32, _F64, _P, _P, _P, _P, _P, _I64,
                                         _P, _P, _P, _P, _I32]
    L.orc_spill_pages.argtypes = [_P, _I32, _I32, _P, _I32, _P]
    L.orc_spill_pages.restype = _I64
    L.orc_restore_pages.argtypes = [_P, _I32, _I32, _P, _I32, _P]
    L.orc_restore_pages.restype = _I64
    L.orc_num_threads.argtypes = []
    L.orc_num_threads.restype = _I32


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# --- scalar formats [NVFP4] -------------------------------------------------------------------

def e2m1_decode(code: int) -> float:
    return float(lib().orc_e2m1_decode(code))


def e2m1_encode(x: float) -> int:
    return int(lib().orc_e2m1_encode(x))


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(code))


def e4m3_encode(t: float) -> int:
    return int(lib().orc_e4m3_encode(t))


def fwht_scale() -> float:
    return float(lib().orc_fwht_scale())


# --- row transforms ------------------------------------------------------------------------------

def rope_table(max_pos: int, rot_dim: int, theta: float, pos_scale: float) -> np.ndarray:
    """[YaRN] cos/sin table, shape [max_pos, rot_dim] (cos in the first half, sin in the second)."""
    t = np.empty((max_pos, rot_dim), dtype=np.float32)
    lib().orc_rope_table(max_pos, rot_dim, theta, pos_scale, _ptr(t))
    return t


def rope_apply(x: np.ndarray, table: np.ndarray, pos: int, rot_dim: int) -> np.ndarray:
    y = np.ascontiguousarray(x, dtype=np.float32).copy()
    lib().orc_rope_apply(_ptr(y), _ptr(table), pos, rot_dim)
    return y


def fwht128(x: np.ndarray) -> np.ndarray:
    """[NVFP4] normalised Walsh-Hadamard rotation of one 128-vector (fp32)."""
    y = np.ascontiguousarray(x, dtype=np.float32).copy()
    lib().orc_fwht128(_ptr(y))
    return y


def quantize_row(x: np.ndarray):
    """[NVFP4] one fp32 row of 128 -> (64 code bytes, 8 scale bytes)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.empty(64, np.uint8)
    scales = np.empty(8, np.uint8)
    lib().orc_quantize_row(_ptr(x), _ptr(codes), _ptr(scales))
    return codes, scales


def quantize_rows(rows_bf16: np.ndarray, pos, rotate: bool, table, rot_dim: int,
                  nthreads: int = 0):
    """Quantise bf16 rows [n, 128] (uint16 bit patterns); Q/K rows get RoPE + Hadamard first."""
    rows = np.ascontiguousarray(rows_bf16.reshape(-1, 128), dtype=np.uint16)
    n = rows.shape[0]
    codes = np.empty((n, 64), np.uint8)
    scales = np.empty((n, 8), np.uint8)
    if rotate:
        pos_a = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, np.int32), (n,)))
        tbl = np.ascontiguousarray(table, dtype=np.float32)
        lib().orc_quantize_rows(_ptr(rows), n, _ptr(pos_a), 1, _ptr(tbl), rot_dim, _ptr(codes),
                                _ptr(scales), nthreads)
    else:
        lib().orc_quantize_rows(_ptr(rows), n, None, 0, None, 0, _ptr(codes), _ptr(scales),
                                nthreads)
    return codes, scales


def dequant_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes.reshape(-1, 64), dtype=np.uint8)
    s = np.ascontiguousarray(scales.reshape(-1, 8), dtype=np.uint8)
    out = np.empty((c.shape[0], 128), np.float64)
    lib().orc_dequant_rows(_ptr(c), _ptr(s), c.shape[0], _ptr(out))
    return out


def paged_gather(pool, num_pages, kv_heads, block_table, seq, pos0, n_tok):
    """Read tokens [pos0, pos0+n_tok) of one sequence out of a pool of page blocks (layout in
    kv_oracle.cpp). Returns (k_codes [n,H,64], k_scales [n,H,8], v_codes, v_scales, bad)."""
    pl = np.ascontiguousarray(pool, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    kc = np.empty((n_tok, kv_heads, 64), np.uint8)
    ks = np.empty((n_tok, kv_heads, 8), np.uint8)
    vc = np.empty((n_tok, kv_heads, 64), np.uint8)
    vs = np.empty((n_tok, kv_heads, 8), np.uint8)
    bad = lib().orc_paged_gather(_ptr(pl), num_pages, kv_heads, _ptr(bt), bt.shape[1], seq, pos0,
                                 n_tok, _ptr(kc), _ptr(ks), _ptr(vc), _ptr(vs))
    return kc, ks, vc, vs, int(bad)


# ---- comparator formats [NVFP4 "Result": 144 B vs int8 264 B vs bf16 512 B; upstream NVFP4 K with
# fp16 V]; fmt 0 = bf16, 1 = int8, 2 = NVFP4 K + fp16 V; kind 0 = Q, 1 = K, 2 = V ----
CMP_FORMATS = {"bf16": 0, "int8": 1, "k4v16": 2}


def float_to_bf16(x: float) -> int:
    return int(lib().orc_float_to_bf16(float(x)))


def float_to_f16(x: float) -> int:
    return int(lib().orc_float_to_f16(float(x)))


def f16_to_double(h: int) -> float:
    return float(lib().orc_f16_to_double(int(h)))


def int8_quantize_row(x: np.ndarray):
    """Per-row symmetric int8: returns (codes int8 [128], fp32 scale)."""
    xr = np.ascontiguousarray(x, np.float32)
    codes = np.empty(128, np.int8)
    sc = np.empty(1, np.float32)
    lib().orc_int8_quantize_row(_ptr(xr), _ptr(codes), _ptr(sc))
    return codes, float(sc[0])


def cmp_row_bytes(fmt: int, kind: int) -> int:
    return int(lib().orc_cmp_row_bytes(fmt, kind))


def cmp_encode_rows(fmt, kind, rows_bf16, pos, table, rot_dim) -> np.ndarray:
    """Comparator row encoding (see kv_oracle.cpp): [n][row bytes] uint8."""
    r = np.ascontiguousarray(rows_bf16, np.uint16).reshape(-1, 128)
    n = r.shape[0]
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos if pos is not None else 0, np.int32), (n,)))
    tbl = np.ascontiguousarray(table if table is not None else np.zeros(1), np.float32)
    out = np.empty((n, cmp_row_bytes(fmt, kind)), np.uint8)
    lib().orc_cmp_encode_rows(fmt, kind, _ptr(r), n, _ptr(p), _ptr(tbl), rot_dim, _ptr(out))
    return out


def cmp_decode_rows(fmt, kind, rows: np.ndarray) -> np.ndarray:
    r = np.ascontiguousarray(rows, np.uint8).reshape(-1, cmp_row_bytes(fmt, kind))
    out = np.empty((r.shape[0], 128), np.float64)
    lib().orc_cmp_decode_rows(fmt, kind, _ptr(r), r.shape[0], _ptr(out))
    return out


def cmp_paged_gather(fmt, pool, num_pages, kv_heads, block_table, seq, pos0, n_tok):
    """Rows of one sequence out of a comparator pool: (k_rows [n,H,kb], v_rows [n,H,vb], bad)."""
    pl = np.ascontiguousarray(pool, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    k = np.empty((n_tok, kv_heads, cmp_row_bytes(fmt, 1)), np.uint8)
    v = np.empty((n_tok, kv_heads, cmp_row_bytes(fmt, 2)), np.uint8)
    bad = lib().orc_cmp_paged_gather(fmt, _ptr(pl), num_pages, kv_heads, _ptr(bt), bt.shape[1],
                                     seq, pos0, n_tok, _ptr(k), _ptr(v))
    return k, v, int(bad)


def attention_f64_rows(q_heads, kv_heads, q_len, causal, sm_scale, seq_lens, tok_off, q, k, v,
                       row_seq, row_tok, row_head, nthreads: int = 0) -> np.ndarray:
    """fp64 attention over decoded rows (q [rows][128], k / v [tokens * kv_heads][128])."""
    sl = np.ascontiguousarray(seq_lens, np.int32)
    to = np.ascontiguousarray(tok_off, np.int64)
    rs = np.ascontiguousarray(row_seq, np.int32)
    rt = np.ascontiguousarray(row_tok, np.int32)
    rh = np.ascontiguousarray(row_head, np.int32)
    qq = np.ascontiguousarray(q, np.float64)
    kk = np.ascontiguousarray(k, np.float64)
    vv = np.ascontiguousarray(v, np.float64)
    out = np.empty((rs.shape[0], 128), np.float32)
    lib().orc_attention_f64_rows(q_heads, kv_heads, q_len, int(causal), sm_scale, _ptr(sl),
                                 _ptr(to), _ptr(qq), _ptr(kk), _ptr(vv), rs.shape[0], _ptr(rs),
                                 _ptr(rt), _ptr(rh), _ptr(out), nthreads)
    return out


def spill_pages(pool, num_pages, kv_heads, page_ids, arena):
    """[Spill] arena slot i <- pool page page_ids[i] (whole page blocks); a page id outside the
    pool is skipped, its slot left as it was. Writes into `arena` in place; returns the number of
    skipped ids."""
    pl = np.ascontiguousarray(pool, dtype=np.uint8)
    ids = np.ascontiguousarray(page_ids, dtype=np.int32)
    assert arena.dtype == np.uint8 and arena.flags.c_contiguous
    return int(lib().orc_spill_pages(_ptr(pl), num_pages, kv_heads, _ptr(ids), len(ids),
                                     _ptr(arena)))


def restore_pages(pool, num_pages, kv_heads, page_ids, arena):
    """[Spill] pool page page_ids[i] <- arena slot i; a page id outside the pool is skipped.
    Writes into `pool` in place; returns the number of skipped ids."""
    ar = np.ascontiguousarray(arena, dtype=np.uint8)
    ids = np.ascontiguousarray(page_ids, dtype=np.int32)
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    return int(lib().orc_restore_pages(_ptr(pool), num_pages, kv_heads, _ptr(ids), len(ids),
                                       _ptr(ar)))


def attention_rows(q_heads, kv_heads, q_len, causal, sm_scale, seq_lens, tok_off,
                   q_codes, q_scales, k_codes, k_scales, v_codes, v_scales,
                   row_seq, row_tok, row_head, nthreads: int = 0) -> np.ndarray:
    """fp64 attention over the dequantised cache for the requested rows; fp32 result [n, 128]."""
    sl = np.ascontiguousarray(seq_lens, np.int32)
    to = np.ascontiguousarray(tok_off, np.int64)
    rs = np.ascontiguousarray(row_seq, np.int32)
    rt = np.ascontiguousarray(row_tok, np.int32)
    rh = np.ascontiguousarray(row_head, np.int32)
    arrs = [np.ascontiguousarray(a, np.uint8) for a in
            (q_codes, q_scales, k_codes, k_scales, v_codes, v_scales)]
    out = np.empty((rs.shape[0], 128), np.float32)
    lib().orc_attention_rows(q_heads, kv_heads, q_len, int(causal), sm_scale, _ptr(sl), _ptr(to),
                             *[_ptr(a) for a in arrs], rs.shape[0], _ptr(rs), _ptr(rt), _ptr(rh),
                             _ptr(out), nthreads)
    return out


def attention_ref_rows(q_heads, kv_heads, q_len, causal, sm_scale, seq_lens, tok_off,
                       q_bf16, k_bf16, v_bf16, table, rot_dim, row_seq, row_tok, row_head,
                       nthreads: int = 0) -> np.ndarray:
    """Unquantised attention (bf16 inputs, same RoPE, no rotation) for cosine-similarity reports."""
    sl = np.ascontiguousarray(seq_lens, np.int32)
    to = np.ascontiguousarray(tok_off, np.int64)
    rs = np.ascontiguousarray(row_seq, np.int32)
    rt = np.ascontiguousarray(row_tok, np.int32)
    rh = np.ascontiguousarray(row_head, np.int32)
    q = np.ascontiguousarray(q_bf16, np.uint16)
    k = np.ascontiguousarray(k_bf16, np.uint16)
    v = np.ascontiguousarray(v_bf16, np.uint16)
    tbl = np.ascontiguousarray(table, np.float32)
    out = np.empty((rs.shape[0], 128), np.float32)
    lib().orc_attention_ref_rows(q_heads, kv_heads, q_len, int(causal), sm_scale, _ptr(sl),
                                 _ptr(to), _ptr(q), _ptr(k), _ptr(v), _ptr(tbl), rot_dim,
                                 rs.shape[0], _ptr(rs), _ptr(rt), _ptr(rh), _ptr(out), nthreads)
    return out


def bytes_per_token_head(fmt: str, head_dim: int = 128) -> int:
    """[NVFP4 "Result"] storage per token per KV head, K and V together."""
    return int(getattr(lib(), f"orc_bytes_per_token_head_{fmt}")(head_dim))


def num_threads() -> int:
    return int(lib().orc_num_threads())
