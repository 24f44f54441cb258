"""Benchmark: NVFP4 decode-attention KV-tokens/s and HBM GB/s (% of peak); append tokens/s.

Workload (one attention layer): 4 sequences x 131,072 cached tokens + 1 new token each, 24 query /
4 KV heads, head_dim 128, 64-token pages placed by a seeded permutation of a 40,000-page pool,
RoPE on 32 dims (theta 1e7), bf16 inputs ~ N(0,1) with K/Q outlier channels x12.

A step is one pass of the whole hot path: one kv_nvfp4_decode_step call, which quantises the
step's new tokens (Q, K, V: RoPE, Hadamard rotation, NVFP4), stores their K/V rows into the pool
and runs the split-K decode attention over the whole cache (two kernel launches: the attention
kernel with the append inside it, and the split-K merge). The step re-appends the same positions,
so every step sees the same cache. The W warm-up steps run directly before the K timed steps. The
same step as two calls (kv_nvfp4_append, then kv_nvfp4_decode_attn: three launches) and the
attention call alone are timed beside it. The KV read per step (302 MB) is larger than L2
(129 MB), so no L2 flush is needed between steps.

`value` is device time with inputs resident in HBM; `e2e` is one kv_nvfp4_decode_step_host call
per step, which adds the host->device copy of the new tokens from pinned memory, the split-K plan
upload and the device->host copy of the attention output. `roofline` covers the step call
(attention kernel + merge kernel), timed with CUDA events around the back-to-back steps.

`configs` holds every workload of the parity tests in the launch configuration the tests check:
the tiny and ragged decode workloads (kv_nvfp4_decode_step, back to back), the speculative
verify step and the 600k prefill chunk (append of the new tokens, then the attention call on the
tile kernel), each with KV-tokens/s, its HBM fraction and the cosine similarity of its output
with unquantised attention (bf16 inputs, same RoPE, float64; computed with torch on the GPU for
the report). The comparator KV formats (`comparators`) and the page spill / restore path
(`spill`) are timed too. `cpu_baseline` is the oracle on the host's cores: the headline step in
full on all threads, with rows for quantize-append and every workload on all threads and on one
(samples extrapolated and marked). `--impl reference` times the CPU oracle on a bounded sample
of the same workload.

Multi-GPU: the path has no exchange step, so N GPUs run N independent replicas (weak scaling);
value = units of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

METRIC = "NVFP4 decode attn KV-tokens/s & HBM GB/s (% of peak); append tokens/s"
UNIT = "KV-tokens/s"
CHUNK = 64  # split-K granularity: one page, so the plan balances CTAs to the page
WORKLOAD = "steady_decode: 4 seqs x 131072 cached + 1 new token, Hq 24 / Hkv 4, d 128, page 64, 40k-page pool"


def max_over_ranks(values, device=None):
    """Each value's maximum over all ranks of the initialised process group (as is at N = 1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def replica_throughput(world, units_per_rank, steps, elapsed_max):
    """Whole-job throughput of N independent replicas: the units all ranks processed divided by
    the slowest rank's time."""
    return world * units_per_rank * steps / elapsed_max


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor throughput (burst: the tile kernel is timed on its own)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def decode_traffic_profile():
    """DRAM bytes per step launch from the committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_step_steady_decode.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    src = os.path.join(ROOT, "bit_kv_cache_03_gb300", "csrc", "decode.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if d.get("decode_cu_sha256_16") != h:
        return None
    return d.get("dram_bytes_per_launch")


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample of the workload.

    Each step: quantise sequence 0's new token (24 Q heads, 4 K and 4 V heads) and run the fp64
    attention of one query head (cycling over the 24) over the first 1024 keys of that sequence.
    One KV-token unit is one key seen by all 24 query heads, so a step covers 1024 / 24 units."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    import synth
    w = synth.steady_decode()
    L = 1024
    table = oracle.rope_table(w.max_pos, w.rot_dim, w.theta, w.pos_scale)
    k = w.k_rows(0, 0, L)
    v = w.v_rows(0, 0, L)
    pos = np.repeat(np.arange(L, dtype=np.int32), w.kv_heads)
    kc, ks = oracle.quantize_rows(k[:-1].reshape(-1, 128), pos[:-w.kv_heads], True, table,
                                  w.rot_dim)
    vc, vs = oracle.quantize_rows(v[:-1].reshape(-1, 128), None, False, None, 0)
    q = w.q_rows(0, L - 1, 1)

    def step(h):
        kn, ksn = oracle.quantize_rows(k[-1:].reshape(-1, 128), pos[-w.kv_heads:], True, table,
                                       w.rot_dim, 1)
        vn, vsn = oracle.quantize_rows(v[-1:].reshape(-1, 128), None, False, None, 0, 1)
        qc, qs = oracle.quantize_rows(q.reshape(-1, 128), np.full(w.q_heads, L - 1, np.int32),
                                      True, table, w.rot_dim, 1)
        rows = (np.zeros(1, np.int32), np.zeros(1, np.int32), np.array([h], np.int32))
        oracle.attention_rows(w.q_heads, w.kv_heads, 1, True, w.sm_scale,
                              np.array([L], np.int32), np.array([0], np.int64), qc, qs,
                              np.concatenate([kc, kn]), np.concatenate([ks, ksn]),
                              np.concatenate([vc, vn]), np.concatenate([vs, vsn]), *rows, 1)

    for i in range(args.warmup):
        step(i % w.q_heads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i % w.q_heads)
    dt = (time.perf_counter() - t0) / args.steps
    units = L / w.q_heads
    value = units / dt
    sample = (f"per step: sequence 0, one of 24 query heads, fp64 attention over the first {L} "
              f"keys + quantisation of the new token ({units:.1f} KV-token units), 1 thread")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def spill_restore(g, dev, stream, reps=5):
    """Page spill and restore of every page the cache uses (8196 pages, 302 MB) to and from a
    page-locked host arena, against a plain contiguous copy of the same bytes over the same link.
    The restore writes each page back to its own id, so the cache is unchanged."""
    import numpy as np
    import torch

    import bit_kv_cache_03_gb300 as kv
    c = g.cache
    w = g.w
    bt = c.block_table.cpu().numpy()
    used = np.concatenate([bt[s, :(int(w.seq_lens[s]) + 63) // 64] for s in range(w.num_seqs)])
    n = len(used)
    pb = kv.kv_nvfp4_page_bytes(c.layout)
    ids = torch.from_numpy(used.astype(np.int32)).to(dev)
    arena = torch.empty(n * pb, dtype=torch.uint8).pin_memory()
    scratch = torch.empty(n * pb, dtype=torch.uint8, device=dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / 1e3 / reps

    t_spill = timed(lambda: kv.kv_nvfp4_spill_pages(c.layout, c.pool, c.num_pages, ids, n, arena,
                                                    c.status))
    t_restore = timed(lambda: kv.kv_nvfp4_restore_pages(c.layout, arena, ids, n, c.pool,
                                                        c.num_pages, c.status))
    t_d2h = timed(lambda: arena.copy_(scratch, non_blocking=True))
    t_h2d = timed(lambda: scratch.copy_(arena, non_blocking=True))
    assert g.status() == 0, f"device status {g.status():#x}"
    b = n * pb
    return {"pages": n, "bytes": b,
            "spill_pages_per_s": n / t_spill, "spill_gbs": b / t_spill / 1e9,
            "restore_pages_per_s": n / t_restore, "restore_gbs": b / t_restore / 1e9,
            "copy_d2h_gbs": b / t_d2h / 1e9, "copy_h2d_gbs": b / t_h2d / 1e9,
            "spill_frac_of_copy": t_d2h / t_spill, "restore_frac_of_copy": t_h2d / t_restore,
            "note": "scattered pool pages <-> page-locked host arena by one kernel launch; copy = "
                    "one contiguous cudaMemcpyAsync of the same bytes"}


CMP_NAMES = {0: "bf16", 1: "int8", 2: "nvfp4k_fp16v"}
CMP_ROW_BYTES = {0: 512, 1: 264, 2: 328}  # K + V bytes per token per KV head


def comparators(w, dev, stream, peak, reps=200):
    """The comparator formats (bf16, int8, NVFP4 K + fp16 V) on the same workload: decode call
    time, KV-tokens/s and HBM fraction of their own algorithmic bytes."""
    import numpy as np
    import torch

    import bit_kv_cache_03_gb300 as kv
    L = kv.make_layout(w.q_heads, w.kv_heads, 128, 64, w.rot_dim)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table, np.int32)).to(dev)
    rope = torch.empty(max(1, w.max_pos * w.rot_dim), dtype=torch.float32, device=dev)
    kv.kv_nvfp4_rope_table_init(rope, w.max_pos, w.rot_dim, w.theta, w.pos_scale)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    cached = []
    for s_, c in enumerate(w.cached_lens):
        k, v, pos = w.cached_tokens(s_, 0, c)
        cached.append((bf(k), bf(v), torch.full((c,), s_, dtype=torch.int32, device=dev),
                       torch.from_numpy(pos).to(dev), c))
    q, k, v, sid, pos = w.new_tokens()
    T = q.shape[0]
    qn, kn, vn = bf(q), bf(k), bf(v)
    sidn, posn = torch.from_numpy(sid).to(dev), torch.from_numpy(pos).to(dev)
    q_out = torch.empty(T * w.q_heads * 128, dtype=torch.bfloat16, device=dev)
    out = torch.empty(T * w.q_heads * 128, dtype=torch.float32, device=dev)
    kv_tokens = int(w.seq_lens.sum())
    n_pages = int(sum((int(l) + 63) // 64 for l in w.seq_lens))
    res = {}
    for fmt in (0, 1, 2):
        pool = torch.empty(w.pool_pages * kv.kv_cmp_page_bytes(L, fmt), dtype=torch.uint8, device=dev)
        for (kc, vc, sc, pc, c) in cached:
            kv.kv_cmp_append(L, fmt, None, kc, vc, sc, pc, c, rope, w.max_pos, bt, w.num_seqs,
                             w.max_pages, w.pool_pages, pool, None, status)
        kv.kv_cmp_append(L, fmt, qn, kn, vn, sidn, posn, T, rope, w.max_pos, bt, w.num_seqs,
                         w.max_pages, w.pool_pages, pool, q_out, status)
        nws = kv.kv_cmp_plan_workspace_bytes(L, w.seq_lens, w.q_len, w.causal, CHUNK)
        ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=dev)
        plan = kv.kv_cmp_plan(L, w.seq_lens, w.q_len, w.causal, CHUNK, ws, nws)

        def call():
            kv.kv_cmp_decode_attn(L, fmt, plan, ws, q_out, w.sm_scale, pool, w.pool_pages, bt,
                                  w.max_pages, out, status)

        for _ in range(10):
            call()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t = e0.elapsed_time(e1) / 1e3 / reps
        b = (kv_tokens * w.kv_heads * CMP_ROW_BYTES[fmt] + T * w.q_heads * 256 + n_pages * 4 +
             T * w.q_heads * 128 * 4)
        res[CMP_NAMES[fmt]] = {"bytes_per_token_kv_head": CMP_ROW_BYTES[fmt],
                               "attn_us": t * 1e6, "kv_tokens_per_s": kv_tokens / t,
                               "hbm_gbs": b / t / 1e9, "hbm_frac_of_measured": b / t / 1e9 / peak}
        del pool, ws
    assert int(status.item()) == 0, f"comparator status {int(status.item()):#x}"
    return res


def decode_step_bytes(w, n_pages=None):
    """Algorithmic bytes of one kv_nvfp4_decode_step: every cached and new K/V row read (144 B per
    token and KV head), the new Q/K/V rows read in bf16 and their codes written, the block-table
    entries of the visited pages, and the fp32 output."""
    T = w.num_seqs * w.q_len
    if n_pages is None:
        n_pages = int(sum((int(l) + 63) // 64 for l in w.seq_lens))
    rows = w.q_heads + 2 * w.kv_heads
    return (w.kv_tokens * w.kv_heads * 144 + T * rows * 256 + T * rows * 72 + n_pages * 4 +
            T * w.q_heads * 128 * 4)


def attn_call_bytes(w):
    """Algorithmic bytes of one kv_nvfp4_decode_attn: the cache (144 B per token and KV head),
    the quantised Q rows, the block-table entries and the fp32 output."""
    T = w.num_seqs * w.q_len
    n_pages = int(sum((int(l) + 63) // 64 for l in w.seq_lens))
    return w.kv_tokens * w.kv_heads * 144 + T * w.q_heads * 72 + n_pages * 4 + T * w.q_heads * 512


def unquantized_cosine(g, rows):
    """Cosine similarity between the step's output rows and unquantised attention of the same rows:
    the bf16 Q/K/V rows, RoPE with the same fp32 table (each product rounded, then added), no
    Hadamard rotation and no quantisation, scores, softmax and P.V in float64 (torch on the GPU,
    for this report only)."""
    import numpy as np
    import torch
    w = g.w
    dev = g.dev
    rs, rt, rh = (np.asarray(a) for a in rows)
    out = g.out.view(w.num_seqs, w.q_len, w.q_heads, 128)
    rot, half = w.rot_dim, w.rot_dim // 2
    table = g.cache.rope.view(-1, rot) if rot else None

    def rope(x, pos):
        if not rot:
            return x
        t = table[pos]
        c, s_ = t[:, :half], t[:, half:rot]
        a, b = x[:, :half], x[:, half:rot]
        return torch.cat([a * c - b * s_, b * c + a * s_, x[:, rot:]], 1)

    def f32(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
        return t.view(torch.bfloat16).float()

    got, ref = [], []
    for s in np.unique(rs):
        L = int(w.seq_lens[s])
        sel = np.nonzero(rs == s)[0]
        K = f32(w.k_rows(int(s), 0, L))
        V = f32(w.v_rows(int(s), 0, L))
        Q = f32(w.q_rows(int(s), L - w.q_len, w.q_len))
        kpos = torch.arange(L, device=dev)
        for kvh in range(w.kv_heads):
            idx = sel[rh[sel] // w.group == kvh]
            if len(idx) == 0:
                continue
            kr = rope(K[:, kvh], kpos).double()
            qpos = torch.from_numpy((L - w.q_len + rt[idx]).astype(np.int64)).to(dev)
            qr = rope(Q[torch.from_numpy(rt[idx].astype(np.int64)).to(dev),
                        torch.from_numpy(rh[idx].astype(np.int64)).to(dev)], qpos).double()
            sc = (qr @ kr.T) * w.sm_scale
            if w.causal:
                sc = sc.masked_fill(kpos[None, :] > qpos[:, None], float("-inf"))
            ref.append(torch.softmax(sc, dim=1) @ V[:, kvh].double())
            got.append(out[int(s)][torch.from_numpy(rt[idx].astype(np.int64)).to(dev),
                                   torch.from_numpy(rh[idx].astype(np.int64)).to(dev)].double())
        del K, V
    a, b = torch.cat(got).ravel(), torch.cat(ref).ravel()
    return float((a @ b) / (a.norm() * b.norm()))


def all_rows(w):
    import numpy as np
    rs, rt, rh = np.meshgrid(np.arange(w.num_seqs), np.arange(w.q_len), np.arange(w.q_heads),
                             indexing="ij")
    return rs.ravel(), rt.ravel(), rh.ravel()


def timed_calls(fn, n, stream, dev):
    """n calls back to back between two CUDA events on the launching stream: seconds per call."""
    import torch
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / 1e3 / n


def decode_config(w, chunk, dev, stream, steps, warmup, peak):
    """One decode workload timed as the headline is: kv_nvfp4_decode_step back to back."""
    from kvrun import GpuRun
    g = GpuRun(w, device=dev)
    g.cache.plan(w.seq_lens, w.q_len, w.causal, chunk)

    def step():
        g.cache.decode_step(g.q, g.k, g.v, g.out, g.q_codes, g.q_scales, sm_scale=w.sm_scale)

    for _ in range(warmup):
        step()
    t = timed_calls(step, steps, stream, dev)
    assert g.status() == 0, f"{w.name}: device status {g.status():#x}"
    b = decode_step_bytes(w)
    return g, {"call": "kv_nvfp4_decode_step", "chunk_tokens": chunk, "steps": steps,
               "step_us": t * 1e6, "kv_tokens": w.kv_tokens, "kv_tokens_per_s": w.kv_tokens / t,
               "hbm_gbs": b / t / 1e9, "hbm_frac_of_measured": b / t / 1e9 / peak,
               "algorithmic_bytes": b}


def tile_config(w, chunk, dev, stream, reps, peak, bf16):
    """A many-row workload (speculative verify, prefill chunk): the append of its new tokens (with
    Q) and the attention call on the tile kernel, each timed back to back."""
    from kvrun import GpuRun
    g = GpuRun(w, device=dev)
    g.step(chunk_tokens=chunk)  # append the new tokens with Q, plan, attend

    def attend():
        g.cache.attend(g.q_codes, g.q_scales, g.out, sm_scale=w.sm_scale)

    def append():
        g.cache.append(g.k, g.v, g.sid, g.pos, q=g.q, q_codes=g.q_codes, q_scales=g.q_scales)

    for _ in range(3):
        append()
        attend()
    t_app = timed_calls(append, max(3, min(reps, 50)), stream, dev)
    t = timed_calls(attend, reps, stream, dev)
    assert g.status() == 0, f"{w.name}: device status {g.status():#x}"
    T = w.num_seqs * w.q_len
    vis = 0  # (query row, visible key) pairs: Q.K^T and P.V take 2 x 128 flops each per pair
    for L in w.seq_lens:
        L = int(L)
        vis += (sum(L - w.q_len + i + 1 for i in range(w.q_len)) if w.causal
                else L * w.q_len) * w.q_heads
    ab = attn_call_bytes(w)
    app_b = T * (w.q_heads + 2 * w.kv_heads) * (256 + 72)
    pv_tflops = 2 * 128 * vis / t / 1e12
    return g, {"call": "kv_nvfp4_append (new tokens, with Q) + kv_nvfp4_decode_attn (tile kernel)",
               "chunk_tokens": chunk, "reps": reps, "append_us": t_app * 1e6,
               "append_tokens_per_s": T / t_app, "append_gbs": app_b / t_app / 1e9,
               "attn_us": t * 1e6, "step_us": (t + t_app) * 1e6, "query_rows": T * w.q_heads,
               "kv_tokens": w.kv_tokens, "kv_tokens_per_s": w.kv_tokens / t,
               "hbm_gbs": ab / t / 1e9, "hbm_frac_of_measured": ab / t / 1e9 / peak,
               "qk_plus_pv_tflops": 2 * pv_tflops, "pv_tflops": pv_tflops,
               "pv_frac_of_bf16": pv_tflops / bf16, "bf16_peak_tflops": bf16}


def cpu_baseline_rows():
    """The oracle, as it stands, on this host's cores: quantize-append tokens/s and the attention
    step of each workload, on all cores and on one. A full pass is timed where it takes seconds;
    otherwise a seeded sample of query rows, extrapolated to the whole step and marked so. The
    cached rows' quantisation is state, not step work: done before the clock starts."""
    import numpy as np

    import oracle
    import synth
    from kvrun import OracleRun
    allc = oracle.num_threads()
    res = {"nproc": os.cpu_count(), "threads_all": allc, "rows": []}

    def rows_sample(w, n, seed):
        """n query rows drawn uniformly (seeded) from all of the step's rows."""
        return (synth.uniform_int(seed, 300, n, w.num_seqs), synth.uniform_int(seed, 301, n, w.q_len),
                synth.uniform_int(seed, 302, n, w.q_heads))

    def add(what, threads, unit, value, seconds, extrapolated):
        res["rows"].append({"what": what, "threads": threads, "unit": unit, "value": value,
                            "seconds": seconds, "extrapolated": extrapolated})

    # quantize-append: RoPE + Hadamard + NVFP4 of 24 Q and 4 K rows, NVFP4 of 4 V rows per token
    w = synth.steady_decode()
    n = 2048
    table = oracle.rope_table(w.max_pos, w.rot_dim, w.theta, w.pos_scale)
    q, k, v = w.q_rows(0, 0, n), w.k_rows(0, 0, n), w.v_rows(0, 0, n)
    qpos = np.repeat(np.arange(n, dtype=np.int32), w.q_heads)
    kpos = np.repeat(np.arange(n, dtype=np.int32), w.kv_heads)
    for th in (1, allc):
        t0 = time.perf_counter()
        oracle.quantize_rows(q.reshape(-1, 128), qpos, True, table, w.rot_dim, th)
        oracle.quantize_rows(k.reshape(-1, 128), kpos, True, table, w.rot_dim, th)
        oracle.quantize_rows(v.reshape(-1, 128), None, False, None, 0, th)
        dt = time.perf_counter() - t0
        add(f"quantize-append, {n} tokens x (24 Q + 4 K + 4 V rows)", th, "tokens/s", n / dt, dt,
            False)

    def step(w, rows, threads, label):
        o = OracleRun(w, nthreads=allc)  # the cache, quantised before the clock
        qn, kn, vn, _, pos = w.new_tokens()
        total = w.num_seqs * w.q_len * w.q_heads
        rs = rows[0] if rows is not None else None
        n_rows = total if rows is None else len(rs)
        t0 = time.perf_counter()
        oracle.quantize_rows(qn.reshape(-1, 128), np.repeat(pos, w.q_heads), True, o.table,
                             w.rot_dim, threads)
        oracle.quantize_rows(kn.reshape(-1, 128), np.repeat(pos, w.kv_heads), True, o.table,
                             w.rot_dim, threads)
        oracle.quantize_rows(vn.reshape(-1, 128), None, False, None, 0, threads)
        t_new = time.perf_counter() - t0
        t0 = time.perf_counter()
        o.nthreads = threads
        o.attention(rows)
        t_att = time.perf_counter() - t0
        dt = t_new + t_att * total / n_rows
        add(f"{label}: quantise the new tokens + fp64 attention of "
            f"{'all ' if rows is None else ''}{n_rows} of {total} query rows", threads,
            "KV-tokens/s", w.kv_tokens / dt, t_new + t_att, rows is not None)
        return w.kv_tokens / dt

    c1 = synth.tiny_decode()
    step(c1, None, 1, c1.name)
    step(c1, None, allc, c1.name)
    c2 = synth.steady_decode()
    main = step(c2, None, allc, c2.name)
    step(c2, rows_sample(c2, 1, 0), 1, c2.name)
    c3 = synth.ragged_decode()
    step(c3, None, allc, c3.name)
    step(c3, rows_sample(c3, 1, 0), 1, c3.name)
    c4 = synth.spec_verify()
    step(c4, None, allc, c4.name)
    c5 = synth.prefill_chunk()
    step(c5, rows_sample(c5, max(16, allc), 0), allc, c5.name)
    return main, res


def run_cuda(args, world, rank, local):
    import numpy as np
    import torch

    import bit_kv_cache_03_gb300 as kv
    import synth
    from kvrun import GpuRun

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.profile_tile:
        # short run of one many-row shape for the profiler: populate, then warm-up + timed calls
        from kvrun import GpuRun as _G
        wt = synth.spec_verify() if args.profile_tile == "verify" else synth.prefill_chunk()
        gt = _G(wt, device=dev)
        gt.step(chunk_tokens=128 if args.profile_tile == "verify" else 1024)
        for _ in range(args.warmup + args.steps):
            gt.cache.attend(gt.q_codes, gt.q_scales, gt.out, sm_scale=wt.sm_scale)
        torch.cuda.synchronize(dev)
        assert gt.status() == 0
        print(json.dumps({"profile_run": True, "workload": wt.name, "steps": args.steps}))
        return
    if args.profile_append:
        # short run of the bulk append (16,384 tokens with Q, K, V) for the profiler
        wa = synth.steady_decode()
        Ta = 16384
        qa = torch.randn(Ta, wa.q_heads, 128, device=dev).to(torch.bfloat16)
        ka = torch.randn(Ta, wa.kv_heads, 128, device=dev).to(torch.bfloat16)
        va = torch.randn(Ta, wa.kv_heads, 128, device=dev).to(torch.bfloat16)
        sida = torch.zeros(Ta, dtype=torch.int32, device=dev)
        posa = torch.arange(Ta, dtype=torch.int32, device=dev)
        ca = kv.PagedNVFP4Cache(Ta // 64, np.arange(Ta // 64, dtype=np.int32)[None], Ta,
                                wa.q_heads, wa.kv_heads, wa.rot_dim, device=dev)
        qca, qsa = ca.quantized_q_buffers(Ta)
        for _ in range(args.warmup + args.steps):
            ca.append(ka, va, sida, posa, q=qa, q_codes=qca, q_scales=qsa)
        torch.cuda.synchronize(dev)
        assert int(ca.status.item()) == 0
        print(json.dumps({"profile_run": True, "workload": "append_16384_tokens",
                          "steps": args.steps}))
        return
    w = synth.steady_decode()
    if args.seqs != 4:
        w = synth.Workload(f"steady_decode_{args.seqs}x128k", [131072] * args.seqs, q_len=1,
                           pool_pages=40000)
    g = GpuRun(w, device=dev)
    stream = torch.cuda.current_stream(dev)
    g.cache.plan(w.seq_lens, w.q_len, w.causal, CHUNK)

    if args.profile:
        # short run for the profiler: warm-up and the timed steps only
        for _ in range(args.warmup + args.steps):
            g.cache.decode_step(g.q, g.k, g.v, g.out, g.q_codes, g.q_scales, sm_scale=w.sm_scale)
        torch.cuda.synchronize(dev)
        assert g.status() == 0
        print(json.dumps({"profile_run": True, "seqs": w.num_seqs, "steps": args.steps}))
        return

    # ---- bulk append throughput (tokens with Q, K, V: the prefill-chunk shape) ----
    Tb = 16384
    qb = torch.randn(Tb, w.q_heads, 128, device=dev).to(torch.bfloat16)
    kb = torch.randn(Tb, w.kv_heads, 128, device=dev).to(torch.bfloat16)
    vb = torch.randn(Tb, w.kv_heads, 128, device=dev).to(torch.bfloat16)
    sidb = torch.zeros(Tb, dtype=torch.int32, device=dev)
    posb = torch.arange(Tb, dtype=torch.int32, device=dev)
    qcb, qsb = g.cache.quantized_q_buffers(Tb)
    spare = kv.PagedNVFP4Cache(Tb // 64, np.arange(Tb // 64, dtype=np.int32)[None], Tb,
                               w.q_heads, w.kv_heads, w.rot_dim, device=dev)
    for _ in range(3):
        spare.append(kb, vb, sidb, posb, q=qb, q_codes=qcb, q_scales=qsb)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    e0.record(stream)
    for _ in range(reps):
        spare.append(kb, vb, sidb, posb, q=qb, q_codes=qcb, q_scales=qsb)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    append_s = e0.elapsed_time(e1) / 1e3 / reps
    append_tps = Tb / append_s
    append_bytes = Tb * ((w.q_heads + 2 * w.kv_heads) * 256 + (w.q_heads + 2 * w.kv_heads) * 72)
    del spare, qb, kb, vb

    # ---- timed decode steps (device-resident inputs) ----
    def fused_step():
        g.cache.decode_step(g.q, g.k, g.v, g.out, g.q_codes, g.q_scales, sm_scale=w.sm_scale)

    def two_call_step():
        g.cache.append(g.k, g.v, g.sid, g.pos, q=g.q, q_codes=g.q_codes, q_scales=g.q_scales)
        g.cache.attend(g.q_codes, g.q_scales, g.out, sm_scale=w.sm_scale)

    def attn_only():
        g.cache.attend(g.q_codes, g.q_scales, g.out, sm_scale=w.sm_scale)

    def back_to_back(fn, n):
        # no event between the kernels of a step, so each kernel's launch overlaps the previous
        # one's tail as it would in a serving loop
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / 1e3

    side_steps = max(10, min(args.steps, 5000))
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the warm-up and the timed region
    for fn in (two_call_step, attn_only):
        for _ in range(args.warmup):
            fn()
    # the W warm-up steps directly before the timed steps, so the GPU is not idle in between
    for _ in range(args.warmup):
        fused_step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    elapsed = back_to_back(fused_step, args.steps)
    two_call_avg = back_to_back(two_call_step, side_steps) / side_steps
    attn_avg = back_to_back(attn_only, side_steps) / side_steps
    fused_step()  # leave the step's output and quantised Q in place
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    step_avg = elapsed / args.steps
    assert g.status() == 0, f"device status {g.status():#x}"

    # ---- end to end through the public API, host buffers ----
    q_h = torch.from_numpy(np.ascontiguousarray(w.new_tokens()[0]).view(np.int16)).pin_memory()
    k_h = torch.from_numpy(np.ascontiguousarray(w.new_tokens()[1]).view(np.int16)).pin_memory()
    v_h = torch.from_numpy(np.ascontiguousarray(w.new_tokens()[2]).view(np.int16)).pin_memory()
    out_h = torch.empty(g.out.numel(), dtype=torch.float32).pin_memory()
    q_d = torch.empty_like(q_h, device=dev)
    k_d = torch.empty_like(k_h, device=dev)
    v_d = torch.empty_like(v_h, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h))
    d2h = out_h.numel() * 4
    # steady state: 2,000 calls (~0.13 s) whatever the timed-step count, so that the first call's
    # host latency (plan build and launches before the GPU starts, ~25 us) does not stand in for
    # per-step cost; the same loop over the timed-step count is reported beside it
    e2e_steps = 2000
    e2e_short_steps = max(1, min(args.steps, e2e_steps))

    seq_lens_h = np.ascontiguousarray(w.seq_lens, np.int32)

    def e2e_step():
        # one library call: pinned H2D of the new tokens, plan build and upload, the fused step,
        # D2H of the output
        g.cache.decode_step_host(seq_lens_h, w.q_len, q_h, k_h, v_h, q_d, k_d, v_d, g.out, out_h,
                                 causal=w.causal, chunk_tokens=CHUNK, sm_scale=w.sm_scale)

    for _ in range(5):
        e2e_step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_elapsed = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_short_steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_short_elapsed = time.perf_counter() - t0

    spill = spill_restore(g, dev, stream)
    cmp = None if args.no_comparators else comparators(w, dev, stream, measured_peaks()[0])

    # ---- every workload of the parity tests, in the launch configuration timed here ----
    peak0 = measured_peaks()[0]
    bf16, _ = measured_bf16_tflops()
    configs = {}
    c2 = {"call": "kv_nvfp4_decode_step", "chunk_tokens": CHUNK, "steps": args.steps,
          "step_us": None, "note": "the headline line's own workload and numbers"}
    try:
        c2["cosine_vs_unquantized"] = unquantized_cosine(g, all_rows(w))
        c2["cosine_rows"] = w.num_seqs * w.q_len * w.q_heads
    except RuntimeError as e:  # reporting only: never fails the bench
        c2["cosine_error"] = str(e)[:200]
    configs[w.name] = c2
    if not args.no_configs:
        # split-K chunks of one page: the plan then deals every CTA its share to the page (the
        # ragged lengths with 1024-token chunks left CTAs between 49 and 80 pages)
        for wc, chunk in ((synth.tiny_decode(), 64), (synth.ragged_decode(), 64)):
            gc, r = decode_config(wc, chunk, dev, stream, max(args.steps, 20), args.warmup, peak0)
            r["cosine_vs_unquantized"] = unquantized_cosine(gc, all_rows(wc))
            r["cosine_rows"] = wc.num_seqs * wc.q_len * wc.q_heads
            if wc.name == "tiny_decode_4k":
                r["note"] = "2.4 MB of KV: L2-resident, so this is a latency figure"
            configs[wc.name] = r
            del gc
            torch.cuda.empty_cache()
    if not args.no_tile_workloads:
        from kvrun import sample_rows
        # verify: chunks of one key block (two pages) balance the CTAs to the block
        for wc, chunk, reps, n_cos in ((synth.spec_verify(), 128, 200, None),
                                       (synth.prefill_chunk(), 1024, 5, 64)):
            gc, r = tile_config(wc, chunk, dev, stream, reps, peak0, bf16)
            rows = all_rows(wc) if n_cos is None else sample_rows(wc, n_cos, seed=0)
            r["cosine_vs_unquantized"] = unquantized_cosine(gc, rows)
            r["cosine_rows"] = len(rows[0])
            configs[wc.name] = r
            del gc
            torch.cuda.empty_cache()

    elapsed, e2e_elapsed, e2e_short_elapsed = max_over_ranks(
        [elapsed, e2e_elapsed, e2e_short_elapsed], dev)
    if rank != 0:
        return

    kv_tokens = int(w.seq_lens.sum())
    value = replica_throughput(world, kv_tokens, args.steps, elapsed)
    e2e_value = replica_throughput(world, kv_tokens, e2e_steps, e2e_elapsed)
    e2e_short_value = replica_throughput(world, kv_tokens, e2e_short_steps, e2e_short_elapsed)
    n_pages = int(sum((int(l) + 63) // 64 for l in w.seq_lens))
    T = w.num_seqs * w.q_len
    # one attention call: every cached K/V row, the quantised Q, the block table, the fp32 output
    attn_bytes = (kv_tokens * w.kv_heads * 144 + T * w.q_heads * 72 + n_pages * 4 +
                  T * w.q_heads * 128 * 4)
    # one step call: the same, with the new rows read in bf16 and their K/V (and Q) codes written
    step_bytes = (kv_tokens * w.kv_heads * 144 + T * (w.q_heads + 2 * w.kv_heads) * 256 +
                  T * (w.q_heads + 2 * w.kv_heads) * 72 + n_pages * 4 + T * w.q_heads * 128 * 4)
    peak, peak_kind = measured_peaks()
    achieved = step_bytes / step_avg / 1e9
    attn_gbs = attn_bytes / attn_avg / 1e9
    traffic = decode_traffic_profile()
    c2.update({"step_us": step_avg * 1e6, "kv_tokens": kv_tokens,
               "kv_tokens_per_s": kv_tokens / step_avg, "hbm_gbs": achieved,
               "hbm_frac_of_measured": achieved / peak, "algorithmic_bytes": step_bytes})
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "kv_tokens_per_step": kv_tokens,
                   "kv_bytes_per_step": kv_tokens * w.kv_heads * 144,
                   "l2": "inputs larger than L2 (302 MB of KV per step vs 129 MB L2), no flush",
                   "chunk_tokens": CHUNK, "parallelism": "replicas" if world > 1 else "1 GPU"},
        "step_us": step_avg * 1e6,
        "two_call_step_us": two_call_avg * 1e6,
        "attn_only_us": attn_avg * 1e6,
        "hbm_gbs_attn_only": attn_gbs,
        "hbm_frac_attn_only_of_measured": attn_gbs / peak,
        "hbm_frac_step_of_nominal_7900": achieved / 7900.0,
        "append_tokens_per_s": append_tps,
        "append_gbs": append_bytes / append_s / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "decode_kernel<6,fused> + merge_kernel (one kv_nvfp4_decode_step "
                               "call; CUDA events around the %d back-to-back timed steps)"
                               % args.steps,
                     "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": step_bytes},
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "value_over_timed_step_count": e2e_short_value,
                "timed_step_count": e2e_short_steps,
                "includes": "one kv_nvfp4_decode_step_host call per step: pinned H2D of the new "
                            "Q/K/V, plan build and upload, the fused step, D2H of the output"},
        "gpu_launches": 2 * args.steps,  # per timed step: the attention kernel, split-K merge
        "spill": spill,
        "comparators": cmp,
        "configs": configs,
    }
    if not args.no_cpu_baseline:
        main_value, detail = cpu_baseline_rows()
        line["cpu_baseline"] = {
            "value": main_value, "unit": UNIT, "cores": detail["threads_all"], "kind": "oracle",
            "sample": "the headline step in full on all host threads: the 4 new tokens quantised "
                      "(Q, K, V) and the fp64 attention of all 96 query rows over 524,292 keys; "
                      "the cached rows are quantised before the clock",
            "nproc": detail["nproc"], "rows": detail["rows"]}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-tile", choices=["verify", "prefill"], default=None,
                    help="short run of the verify or prefill-chunk attention call (profiling)")
    ap.add_argument("--profile-append", action="store_true",
                    help="short run of the 16,384-token bulk append (profiling)")
    ap.add_argument("--no-tile-workloads", action="store_true",
                    help="skip timing the verify and prefill-chunk shapes (tile kernel)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the tiny and ragged decode workloads")
    ap.add_argument("--no-comparators", action="store_true",
                    help="skip the bf16 / int8 / NVFP4 K + fp16 V comparator timings")
    ap.add_argument("--seqs", type=int, default=4, help="sequences of 131072 tokens (profiling)")
    ap.add_argument("--profile", action="store_true",
                    help="warm-up + steps only, no extra measurements (for ncu)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    import __graft_entry__
    __graft_entry__.build()
    run_cuda(args, world, rank, local)


if __name__ == "__main__":
    main()
