"""kv_nvfp4_decode_attn_noalloc against the workspace path (GPU).

Some callers cannot allocate device memory: an inference engine that gives all of the GPU's
memory to its own arena at start-up and hands a layer only its inputs and outputs, or a plug-in
under an allocator it does not control. For them the library keeps the decode workspace in a fixed
buffer of its own. These tests call that entry point through the C ABI, twice in a row on the same
inputs, and compare each result with kv_nvfp4_plan + kv_nvfp4_decode_attn on a workspace that
PyTorch allocated, within the attention tolerance of the other GPU tests. The file is named to be
collected last.
"""
import numpy as np
import pytest

import synth
from kvrun import MAX_ABS_TOL, REL_L2_TOL, GpuRun, attention_errors

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _noalloc(g, out):
    w, c = g.w, g.cache
    g.kv.kv_nvfp4_decode_attn_noalloc(c.layout, w.seq_lens, w.q_len, w.causal, w.chunk_tokens,
                                      g.q_codes, g.q_scales, w.sm_scale, c.pool, c.num_pages,
                                      c.block_table, c.max_pages, out, c.status)


@pytest.mark.parametrize("lens,q_len,chunk", [
    ([5000, 300, 64], 1, 64),      # split groups: partials and the merge launch use the buffer
    ([2000, 37], 8, 256),          # verify-shaped: 48 rows per KV head, the tile kernel
])
def test_noalloc_matches_workspace_path_on_two_calls(lens, q_len, chunk):
    w = synth.Workload("noalloc", lens, q_len=q_len, causal=True, seed=11 + q_len,
                       chunk_tokens=chunk, pool_pages=sum((c + q_len + 63) // 64 for c in lens) + 3)
    g = GpuRun(w)
    g.step(chunk_tokens=chunk)  # append the new tokens, then the workspace path
    torch.cuda.synchronize()
    ref = g.output().astype(np.float64)
    for call in range(2):
        out = torch.full_like(g.out, float("nan"))
        _noalloc(g, out)
        torch.cuda.synchronize()
        got = out.view(g.T, w.q_heads, 128).cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: rows left unwritten"
        max_abs, rel = attention_errors(got, ref)
        assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, (call, max_abs, rel)
    assert g.status() == 0


def test_noalloc_rejects_a_plan_larger_than_its_buffer():
    import bit_kv_cache_03_gb300 as kv
    w = synth.Workload("noalloc_small", [300], q_len=1, seed=3, pool_pages=8)
    g = GpuRun(w)
    c = g.cache
    # 1,000,000 one-token sequences: the group and segment tables alone (48 B a sequence) are
    # past the buffer. The block table and the output below cover one sequence only, so the call
    # is safe only because the library refuses it on the host, before any GPU work: check first
    # that the plan is larger than the buffer (the constant mirrors the header, which a CPU test
    # keeps in step).
    lens = np.ones(1_000_000, np.int32)
    need = kv.kv_nvfp4_plan_workspace_bytes(c.layout, lens, 1, True, 64)
    assert need > kv.NOALLOC_SCRATCH_BYTES
    out = torch.zeros_like(g.out)
    with pytest.raises(kv.KVNVFP4Error, match=r"\(-3\)"):
        kv.kv_nvfp4_decode_attn_noalloc(c.layout, lens, 1, True, 64, g.q_codes, g.q_scales,
                                        w.sm_scale, c.pool, c.num_pages, c.block_table,
                                        c.max_pages, out, c.status)
    torch.cuda.synchronize()
    assert not out.any()  # rejected before any GPU work
