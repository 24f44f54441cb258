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
    # past the buffer, so the call returns ENOSPACE on the host. The output and the block table
    # are passed as null: were the plan ever to fit, the decode call's pointer checks would refuse
    # it (EINVAL) before any launch, so no call here can reach a kernel.
    lens = np.ones(1_000_000, np.int32)
    need = kv.kv_nvfp4_plan_workspace_bytes(c.layout, lens, 1, True, 64)
    assert need > kv.NOALLOC_SCRATCH_BYTES
    with pytest.raises(kv.KVNVFP4Error, match=r"\(-3\)"):
        kv.kv_nvfp4_decode_attn_noalloc(c.layout, lens, 1, True, 64, g.q_codes, g.q_scales,
                                        w.sm_scale, c.pool, c.num_pages, None, c.max_pages, None,
                                        c.status)
    torch.cuda.synchronize()
    assert g.status() == 0


def test_noalloc_is_refused_while_the_stream_is_capturing():
    # the work list is uploaded from host memory that each call rebuilds, so a graph replay would
    # read stale memory: the entry point refuses a capturing stream before enqueuing anything
    import bit_kv_cache_03_gb300 as kv
    w = synth.Workload("noalloc_capture", [500, 90], q_len=1, seed=5, chunk_tokens=64)
    g = GpuRun(w)
    g.step(chunk_tokens=64)
    torch.cuda.synchronize()
    ref = g.output().copy()
    out = torch.full_like(g.out, float("nan"))
    side = torch.zeros(16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    refused = None
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            side.add_(1.0)
            try:
                _noalloc(g, out)
            except kv.KVNVFP4Error as e:
                refused = str(e)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    assert refused is not None and "(-1)" in refused, refused
    assert torch.isnan(out).all()  # nothing was enqueued, into the graph or otherwise
    # the same call outside the capture runs as usual
    _noalloc(g, out)
    torch.cuda.synchronize()
    max_abs, rel = attention_errors(out.view(g.T, w.q_heads, 128).cpu().numpy(), ref)
    assert max_abs <= MAX_ABS_TOL and rel <= REL_L2_TOL, (max_abs, rel)
    assert g.status() == 0
