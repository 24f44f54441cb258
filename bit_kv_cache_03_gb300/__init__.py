"""NVFP4 KV cache for GB300: Python binding of the C ABI in include/kv_nvfp4.h.

Argument marshalling only: every step of the path runs in the CUDA library
(``_build/libkvnvfp4.so``, built from ``csrc/`` for sm_103a). Importing this package loads that
library and fails loudly if it is missing; there is no CPU fallback.

Method: prismix.dev/news/833001997676, sections "NVFP4 KV cache (from scratch)" and "YaRN context
extension" (NVFP4 K/V with E4M3 block scales, Hadamard-rotated K and Q, fused append, NVFP4 Q.K^T,
V dequantised for P.V, 144 bytes per token per KV head, linear RoPE position scaling).
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build_mod

_LIB_PATH = _build_mod.LIB_PATH

KV_NVFP4_OK = 0
KV_NVFP4_EINVAL = -1
KV_NVFP4_ECUDA = -2
KV_NVFP4_ENOSPACE = -3
DEV_BAD_PAGE, DEV_BAD_POS, DEV_BAD_SEQ, DEV_BAD_ROPE, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10
NOALLOC_SCRATCH_BYTES = 32 << 20  # KV_NVFP4_NOALLOC_SCRATCH_BYTES


class Layout(ctypes.Structure):
    """kv_nvfp4_layout"""
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("rot_dim", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    """kv_nvfp4_plan_info"""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_seqs", "q_len", "causal", "chunk_pages", "num_kv_heads", "num_row_groups",
        "num_groups", "num_segments", "num_partials", "grid", "max_seq_len", "num_split_groups")] + [
        ("total_kv_tokens", ctypes.c_int64), ("total_pages", ctypes.c_int64)] + [
        (n, ctypes.c_uint64) for n in ("off_groups", "off_segments", "off_cta", "off_split",
                                       "off_partials", "workspace_bytes")]


class KVNVFP4Error(RuntimeError):
    pass


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_F64 = ctypes.c_double
_SIG = {
    "kv_nvfp4_status_string": ([_I32], ctypes.c_char_p),
    "kv_nvfp4_version": ([], _I32),
    "kv_nvfp4_last_cuda_error": ([], ctypes.c_char_p),
    "kv_nvfp4_layout_check": ([ctypes.POINTER(Layout)], _I32),
    "kv_nvfp4_page_bytes": ([ctypes.POINTER(Layout)], ctypes.c_size_t),
    "kv_nvfp4_pool_bytes": ([ctypes.POINTER(Layout), _I32, ctypes.POINTER(ctypes.c_size_t)],
                            _I32),
    "kv_nvfp4_rope_table_bytes": ([_I32, _I32], ctypes.c_size_t),
    "kv_nvfp4_rope_table_fill_host": ([_P, _I32, _I32, _F64, _F64], _I32),
    "kv_nvfp4_rope_table_init": ([_P, _I32, _I32, _F64, _F64, _P], _I32),
    "kv_nvfp4_append": ([ctypes.POINTER(Layout), _P, _P, _P, _P, _P, _I32, _P, _I32, _P, _I32,
                         _I32, _I32, _P, _P, _P, _P, _P], _I32),
    "kv_nvfp4_plan_workspace_bytes": ([ctypes.POINTER(Layout), _P, _I32, _I32, _I32, _I32,
                                       ctypes.POINTER(ctypes.c_size_t)], _I32),
    "kv_nvfp4_plan": ([ctypes.POINTER(Layout), _P, _I32, _I32, _I32, _I32, _P, ctypes.c_size_t,
                       ctypes.POINTER(PlanInfo), _P], _I32),
    "kv_nvfp4_plan_host": ([ctypes.POINTER(Layout), _P, _I32, _I32, _I32, _I32, _I32, _P,
                            ctypes.c_size_t, ctypes.POINTER(PlanInfo)], _I32),
    "kv_nvfp4_decode_attn": ([ctypes.POINTER(Layout), ctypes.POINTER(PlanInfo), _P, _P, _P,
                              ctypes.c_float, _P, _I32, _P, _I32, _P, _P, _P], _I32),
    "kv_nvfp4_decode_step": ([ctypes.POINTER(Layout), ctypes.POINTER(PlanInfo), _P, _P, _P, _P, _P,
                              _I32, _P, _I32, _I32, _P, _P, _P, ctypes.c_float, _P, _P, _P], _I32),
    "kv_nvfp4_decode_step_host": ([ctypes.POINTER(Layout), _P, _I32, _I32, _I32, _I32, _P,
                                   ctypes.c_size_t, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _I32,
                                   _I32, _P, ctypes.c_float, _P, _P, _P, ctypes.POINTER(PlanInfo),
                                   _P], _I32),
    "kv_nvfp4_decode_attn_noalloc": ([ctypes.POINTER(Layout), _P, _I32, _I32, _I32, _I32, _P, _P,
                                      ctypes.c_float, _P, _I32, _P, _I32, _P, _P, _P], _I32),
    "kv_cmp_page_bytes": ([ctypes.POINTER(Layout), _I32], ctypes.c_size_t),
    "kv_cmp_append": ([ctypes.POINTER(Layout), _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _P, _I32,
                       _I32, _I32, _P, _P, _P, _P], _I32),
    "kv_cmp_plan_workspace_bytes": ([ctypes.POINTER(Layout), _P, _I32, _I32, _I32, _I32,
                                     ctypes.POINTER(ctypes.c_size_t)], _I32),
    "kv_cmp_plan": ([ctypes.POINTER(Layout), _P, _I32, _I32, _I32, _I32, _P, ctypes.c_size_t,
                     ctypes.POINTER(PlanInfo), _P], _I32),
    "kv_cmp_decode_attn": ([ctypes.POINTER(Layout), _I32, ctypes.POINTER(PlanInfo), _P, _P,
                            ctypes.c_float, _P, _I32, _P, _I32, _P, _P, _P], _I32),
    "kv_nvfp4_spill_pages": ([ctypes.POINTER(Layout), _P, _I32, _P, _I32, _P, _P, _P], _I32),
    "kv_nvfp4_restore_pages": ([ctypes.POINTER(Layout), _P, _P, _I32, _P, _I32, _P, _P], _I32),
}

_lib = None


def lib():
    """The loaded CUDA library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise KVNVFP4Error(
                f"CUDA library {_LIB_PATH} is missing: run "
                "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a) first")
        L = ctypes.CDLL(_LIB_PATH)
        for name, (args, res) in _SIG.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def library_path() -> str:
    return _LIB_PATH


def _check(status: int, what: str):
    if status != KV_NVFP4_OK:
        msg = lib().kv_nvfp4_status_string(status).decode()
        if status == KV_NVFP4_ECUDA:
            msg += ": " + lib().kv_nvfp4_last_cuda_error().decode()
        raise KVNVFP4Error(f"{what}: {msg} ({status})")


def _ptr(x) -> int | None:
    """Device/host address of a tensor-like (torch tensor, numpy array) or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_layout(num_q_heads=24, num_kv_heads=4, head_dim=128, page_size=64, rot_dim=32) -> Layout:
    L = Layout(num_q_heads, num_kv_heads, head_dim, page_size, rot_dim)
    _check(lib().kv_nvfp4_layout_check(ctypes.byref(L)), "kv_nvfp4_layout_check")
    return L


# ---- the C ABI, name for name -----------------------------------------------------------------

def kv_nvfp4_version() -> int:
    return int(lib().kv_nvfp4_version())


def kv_nvfp4_page_bytes(layout: Layout) -> int:
    return int(lib().kv_nvfp4_page_bytes(ctypes.byref(layout)))


def kv_nvfp4_pool_bytes(layout: Layout, num_pages: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().kv_nvfp4_pool_bytes(ctypes.byref(layout), num_pages, ctypes.byref(n)),
           "kv_nvfp4_pool_bytes")
    return n.value


def kv_nvfp4_rope_table_bytes(max_pos: int, rot_dim: int) -> int:
    return int(lib().kv_nvfp4_rope_table_bytes(max_pos, rot_dim))


def kv_nvfp4_rope_table_fill_host(h_table, max_pos, rot_dim, theta, pos_scale):
    _check(lib().kv_nvfp4_rope_table_fill_host(_ptr(h_table), max_pos, rot_dim, theta, pos_scale),
           "kv_nvfp4_rope_table_fill_host")


def kv_nvfp4_rope_table_init(d_table, max_pos, rot_dim, theta, pos_scale, stream=None):
    _check(lib().kv_nvfp4_rope_table_init(_ptr(d_table), max_pos, rot_dim, theta, pos_scale,
                                          _stream(stream)), "kv_nvfp4_rope_table_init")


def kv_nvfp4_append(layout, q, k, v, seq_ids, positions, T, rope_table, rope_max_pos,
                    block_table, num_seqs, max_pages, num_pages, pool, q_codes=None,
                    q_scales=None, status=None, stream=None):
    _check(lib().kv_nvfp4_append(
        ctypes.byref(layout), _ptr(q), _ptr(k), _ptr(v), _ptr(seq_ids), _ptr(positions), T,
        _ptr(rope_table), rope_max_pos, _ptr(block_table), num_seqs, max_pages, num_pages,
        _ptr(pool), _ptr(q_codes), _ptr(q_scales), _ptr(status), _stream(stream)),
        "kv_nvfp4_append")


def kv_nvfp4_plan_workspace_bytes(layout, seq_lens, q_len, causal, chunk_tokens) -> int:
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, np.int32)
    n = ctypes.c_size_t()
    _check(lib().kv_nvfp4_plan_workspace_bytes(ctypes.byref(layout), sl.ctypes.data, len(sl),
                                               q_len, int(causal), chunk_tokens, ctypes.byref(n)),
           "kv_nvfp4_plan_workspace_bytes")
    return n.value


def kv_nvfp4_plan(layout, seq_lens, q_len, causal, chunk_tokens, workspace, ws_bytes,
                  stream=None) -> PlanInfo:
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, np.int32)
    info = PlanInfo()
    _check(lib().kv_nvfp4_plan(ctypes.byref(layout), sl.ctypes.data, len(sl), q_len, int(causal),
                               chunk_tokens, _ptr(workspace), ws_bytes, ctypes.byref(info),
                               _stream(stream)), "kv_nvfp4_plan")
    return info


def kv_nvfp4_plan_host(layout, seq_lens, q_len, causal, chunk_tokens, num_ctas):
    """Host image of the plan tables for `num_ctas` CTAs: (info, groups [n,8], segments [n,4],
    cta ranges [num_ctas+1], split-group list [num_split_groups]) as numpy arrays."""
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, np.int32)
    info = PlanInfo()
    size = 1 << 16
    while True:
        buf = np.zeros(size, np.uint8)
        st = lib().kv_nvfp4_plan_host(ctypes.byref(layout), sl.ctypes.data, len(sl), q_len,
                                      int(causal), chunk_tokens, num_ctas, buf.ctypes.data, size,
                                      ctypes.byref(info))
        if st == KV_NVFP4_ENOSPACE:
            size *= 4
            continue
        _check(st, "kv_nvfp4_plan_host")
        break
    i32 = buf.view(np.int32)
    groups = i32[info.off_groups // 4: info.off_groups // 4 + 8 * info.num_groups].reshape(-1, 8)
    segs = i32[info.off_segments // 4: info.off_segments // 4 + 4 * info.num_segments].reshape(-1, 4)
    cta = i32[info.off_cta // 4: info.off_cta // 4 + info.grid + 1]
    split = i32[info.off_split // 4: info.off_split // 4 + info.num_split_groups]
    return info, groups.copy(), segs.copy(), cta.copy(), split.copy()


def kv_nvfp4_decode_attn(layout, plan: PlanInfo, workspace, q_codes, q_scales, sm_scale, pool,
                         num_pages, block_table, max_pages, out, status=None, stream=None):
    _check(lib().kv_nvfp4_decode_attn(
        ctypes.byref(layout), ctypes.byref(plan), _ptr(workspace), _ptr(q_codes), _ptr(q_scales),
        float(sm_scale), _ptr(pool), num_pages, _ptr(block_table), max_pages, _ptr(out),
        _ptr(status), _stream(stream)), "kv_nvfp4_decode_attn")


def kv_nvfp4_decode_step(layout, plan: PlanInfo, workspace, q, k, v, rope, rope_max_pos,
                         block_table, max_pages, num_pages, pool, q_codes_out, q_scales_out,
                         sm_scale, out, status=None, stream=None):
    """Append of the step's new tokens and decode attention in one launch (see the header)."""
    _check(lib().kv_nvfp4_decode_step(
        ctypes.byref(layout), ctypes.byref(plan), _ptr(workspace), _ptr(q), _ptr(k), _ptr(v),
        _ptr(rope), rope_max_pos, _ptr(block_table), max_pages, num_pages, _ptr(pool),
        _ptr(q_codes_out), _ptr(q_scales_out), float(sm_scale), _ptr(out), _ptr(status),
        _stream(stream)), "kv_nvfp4_decode_step")


def kv_nvfp4_decode_step_host(layout, seq_lens, q_len, causal, chunk_tokens, workspace, ws_bytes,
                              h_q, h_k, h_v, d_q, d_k, d_v, rope, rope_max_pos, block_table,
                              max_pages, num_pages, pool, sm_scale, d_out, h_out, status=None,
                              stream=None, plan_out=None):
    """One decode step from host buffers (see the header). seq_lens: int32 host lengths; h_*:
    host tensors (page-locked for asynchronous copies); d_*: device tensors."""
    import numpy as np
    sl = seq_lens if (isinstance(seq_lens, np.ndarray) and seq_lens.dtype == np.int32 and
                      seq_lens.flags.c_contiguous) else np.ascontiguousarray(seq_lens, np.int32)
    _check(lib().kv_nvfp4_decode_step_host(
        ctypes.byref(layout), sl.ctypes.data, len(sl), q_len, int(causal), chunk_tokens,
        _ptr(workspace), ws_bytes, _ptr(h_q), _ptr(h_k), _ptr(h_v), _ptr(d_q), _ptr(d_k),
        _ptr(d_v), _ptr(rope), rope_max_pos, _ptr(block_table), max_pages, num_pages, _ptr(pool),
        float(sm_scale), _ptr(d_out), _ptr(h_out), _ptr(status),
        ctypes.byref(plan_out) if plan_out is not None else None, _stream(stream)),
        "kv_nvfp4_decode_step_host")


# ---- comparator formats (bf16, int8, NVFP4 K + fp16 V) ----
KV_CMP_BF16, KV_CMP_INT8, KV_CMP_K4V16 = 0, 1, 2


def kv_cmp_page_bytes(layout, fmt) -> int:
    return int(lib().kv_cmp_page_bytes(ctypes.byref(layout), fmt))


def kv_cmp_append(layout, fmt, q, k, v, seq_ids, positions, T, rope_table, rope_max_pos,
                  block_table, num_seqs, max_pages, num_pages, pool, q_out=None, status=None,
                  stream=None):
    _check(lib().kv_cmp_append(
        ctypes.byref(layout), fmt, _ptr(q), _ptr(k), _ptr(v), _ptr(seq_ids), _ptr(positions), T,
        _ptr(rope_table), rope_max_pos, _ptr(block_table), num_seqs, max_pages, num_pages,
        _ptr(pool), _ptr(q_out), _ptr(status), _stream(stream)), "kv_cmp_append")


def kv_cmp_plan_workspace_bytes(layout, seq_lens, q_len, causal, chunk_tokens) -> int:
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, np.int32)
    n = ctypes.c_size_t()
    _check(lib().kv_cmp_plan_workspace_bytes(ctypes.byref(layout), sl.ctypes.data, len(sl), q_len,
                                             int(causal), chunk_tokens, ctypes.byref(n)),
           "kv_cmp_plan_workspace_bytes")
    return n.value


def kv_cmp_plan(layout, seq_lens, q_len, causal, chunk_tokens, workspace, ws_bytes,
                stream=None) -> PlanInfo:
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, np.int32)
    info = PlanInfo()
    _check(lib().kv_cmp_plan(ctypes.byref(layout), sl.ctypes.data, len(sl), q_len, int(causal),
                             chunk_tokens, _ptr(workspace), ws_bytes, ctypes.byref(info),
                             _stream(stream)), "kv_cmp_plan")
    return info


def kv_cmp_decode_attn(layout, fmt, plan: PlanInfo, workspace, q_rot, sm_scale, pool, num_pages,
                       block_table, max_pages, out, status=None, stream=None):
    _check(lib().kv_cmp_decode_attn(
        ctypes.byref(layout), fmt, ctypes.byref(plan), _ptr(workspace), _ptr(q_rot),
        float(sm_scale), _ptr(pool), num_pages, _ptr(block_table), max_pages, _ptr(out),
        _ptr(status), _stream(stream)), "kv_cmp_decode_attn")


def kv_nvfp4_spill_pages(layout, pool, num_pages, page_ids, n, arena, status=None, stream=None):
    """Arena slot i <- pool page page_ids[i] (page_ids on the device; arena page-locked host
    memory or device memory, n page blocks)."""
    _check(lib().kv_nvfp4_spill_pages(ctypes.byref(layout), _ptr(pool), num_pages, _ptr(page_ids),
                                      n, _ptr(arena), _ptr(status), _stream(stream)),
           "kv_nvfp4_spill_pages")


def kv_nvfp4_restore_pages(layout, arena, page_ids, n, pool, num_pages, status=None,
                           stream=None):
    """Pool page page_ids[i] <- arena slot i."""
    _check(lib().kv_nvfp4_restore_pages(ctypes.byref(layout), _ptr(arena), _ptr(page_ids), n,
                                        _ptr(pool), num_pages, _ptr(status), _stream(stream)),
           "kv_nvfp4_restore_pages")


def kv_nvfp4_decode_attn_noalloc(layout, seq_lens, q_len, causal, chunk_tokens, q_codes, q_scales,
                                 sm_scale, pool, num_pages, block_table, max_pages, out,
                                 status=None, stream=None):
    """Plan + decode attention with the library's fixed device buffer as the workspace, for
    callers that cannot allocate device memory (KV_NVFP4_ENOSPACE when the plan does not fit)."""
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, np.int32)
    _check(lib().kv_nvfp4_decode_attn_noalloc(
        ctypes.byref(layout), sl.ctypes.data, len(sl), q_len, int(causal), chunk_tokens,
        _ptr(q_codes), _ptr(q_scales), float(sm_scale), _ptr(pool), num_pages, _ptr(block_table),
        max_pages, _ptr(out), _ptr(status), _stream(stream)), "kv_nvfp4_decode_attn_noalloc")


from .cache import PagedNVFP4Cache  # noqa: E402  (device buffers for one layer, allocated by torch)
