"""The C-ABI library builds, loads on a machine without a GPU, exports every symbol declared in
include/kv_nvfp4.h, and rejects bad host arguments before touching CUDA (CPU only)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kv():
    from bit_kv_cache_03_gb300 import build
    build.build()
    import bit_kv_cache_03_gb300 as kv
    kv.lib()
    return kv


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kv_nvfp4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(kv):
    names = declared_functions()
    assert len(names) >= 12
    raw = ctypes.CDLL(kv.library_path())
    for n in names:
        assert hasattr(raw, n), f"{n} declared in the header but not exported"


def test_page_and_plane_bytes(kv):
    L = kv.make_layout()
    assert kv.kv_nvfp4_page_bytes(L) == 64 * 144 * 4 == 36864
    c, s = kv.kv_nvfp4_pool_plane_bytes(L, 10)
    assert c == 10 * 4 * 64 * 64 and s == 10 * 4 * 64 * 8
    assert (c + s) * 2 // (10 * 4 * 64) == 144


@pytest.mark.parametrize("bad", [dict(head_dim=64), dict(page_size=32), dict(num_q_heads=10),
                                 dict(num_q_heads=72, num_kv_heads=4), dict(rot_dim=30),
                                 dict(rot_dim=136)])
def test_layout_rejected(kv, bad):
    args = dict(num_q_heads=24, num_kv_heads=4, head_dim=128, page_size=64, rot_dim=32)
    args.update(bad)
    L = kv.Layout(**args)
    assert kv.lib().kv_nvfp4_layout_check(ctypes.byref(L)) == kv.KV_NVFP4_EINVAL


def test_rope_host_table_bit_identical_to_oracle(kv):
    for scale in (1.0, 600000.0 / 262144.0):
        t = np.empty((5000, 32), np.float32)
        kv.kv_nvfp4_rope_table_fill_host(t, 5000, 32, 1e7, scale)
        ref = oracle.rope_table(5000, 32, 1e7, scale)
        assert np.array_equal(t.view(np.uint32), ref.view(np.uint32))


def test_plan_sizes_and_validation(kv):
    L = kv.make_layout()
    n = kv.kv_nvfp4_plan_workspace_bytes(L, [4097], 1, 1024)
    assert n > 0
    # 4 x 131073 tokens, 1024-token chunks: 129 chunks each, 4 heads, 1 row tile, 4160 B partials
    n2 = kv.kv_nvfp4_plan_workspace_bytes(L, [131073] * 4, 1, 1024)
    assert n2 >= 4 * 129 * 4 * 4160
    lib = kv.lib()
    sl = np.array([5, 3], np.int32)
    size = ctypes.c_size_t()
    # seq_len < q_len, chunk not a multiple of 64, null workspace: all rejected without CUDA
    assert lib.kv_nvfp4_plan_workspace_bytes(ctypes.byref(L), sl.ctypes.data, 2, 4, 1024,
                                             ctypes.byref(size)) == kv.KV_NVFP4_EINVAL
    assert lib.kv_nvfp4_plan_workspace_bytes(ctypes.byref(L), sl.ctypes.data, 2, 1, 100,
                                             ctypes.byref(size)) == kv.KV_NVFP4_EINVAL
    info = kv.PlanInfo()
    assert lib.kv_nvfp4_plan(ctypes.byref(L), sl.ctypes.data, 2, 1, 1024, None, 0,
                             ctypes.byref(info), None) == kv.KV_NVFP4_EINVAL


def test_entry_points_reject_bad_arguments_before_cuda(kv):
    lib = kv.lib()
    L = kv.make_layout()
    bad = kv.Layout(24, 4, 64, 64, 32)
    assert lib.kv_nvfp4_append(ctypes.byref(bad), *([None] * 5), 1, None, 1, None, 1, 1, 1,
                               *([None] * 8), None) == kv.KV_NVFP4_EINVAL
    # null K pointer
    assert lib.kv_nvfp4_append(ctypes.byref(L), *([None] * 5), 1, None, 1, None, 1, 1, 1,
                               *([None] * 8), None) == kv.KV_NVFP4_EINVAL
    # T = 0 is a no-op that needs no buffers
    assert lib.kv_nvfp4_append(ctypes.byref(L), *([None] * 5), 0, None, 1, None, 1, 1, 1,
                               *([None] * 8), None) == kv.KV_NVFP4_OK
    info = kv.PlanInfo()
    assert lib.kv_nvfp4_decode_attn(ctypes.byref(L), ctypes.byref(info), None, None, None, 1,
                                    0.0, None, None, None, None, 1, None, 1, None, None,
                                    None) == kv.KV_NVFP4_EINVAL
    assert kv.lib().kv_nvfp4_status_string(-1) == b"invalid argument"
