"""Device buffers of one attention layer's NVFP4 paged cache, allocated by PyTorch.

PyTorch provides memory and streams only; every computation goes through the C ABI.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import (kv_nvfp4_append, kv_nvfp4_decode_attn, kv_nvfp4_decode_step,
               kv_nvfp4_decode_step_host, kv_nvfp4_plan, kv_nvfp4_plan_workspace_bytes,
               kv_nvfp4_pool_bytes, kv_nvfp4_rope_table_init, make_layout)


class PagedNVFP4Cache:
    """Page pool, block table, RoPE table and status word for one layer on one GPU."""

    def __init__(self, num_pages, block_table, max_pos, num_q_heads=24, num_kv_heads=4,
                 rot_dim=32, theta=1e7, pos_scale=1.0, device="cuda"):
        self.layout = make_layout(num_q_heads, num_kv_heads, 128, 64, rot_dim)
        self.device = torch.device(device)
        self.num_pages = int(num_pages)
        self.pool = torch.empty(kv_nvfp4_pool_bytes(self.layout, self.num_pages),
                                dtype=torch.uint8, device=self.device)
        bt = np.ascontiguousarray(block_table, np.int32)
        self.num_seqs, self.max_pages = bt.shape
        self.block_table = torch.from_numpy(bt).to(self.device)
        self.max_pos = int(max_pos)
        self.rot_dim = rot_dim
        self.rope = torch.empty(max(1, self.max_pos * rot_dim), dtype=torch.float32,
                                device=self.device)
        if rot_dim > 0:
            kv_nvfp4_rope_table_init(self.rope, self.max_pos, rot_dim, theta, pos_scale)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.workspace = None
        self.plan_info = None

    # -- fused quantize-append --------------------------------------------------------------
    def append(self, k, v, seq_ids, positions, q=None, q_codes=None, q_scales=None, stream=None):
        T = int(k.shape[0])
        kv_nvfp4_append(self.layout, q, k, v, seq_ids, positions, T, self.rope, self.max_pos,
                        self.block_table, self.num_seqs, self.max_pages, self.num_pages,
                        self.pool, q_codes, q_scales, self.status, stream)

    def quantized_q_buffers(self, T):
        H = self.layout.num_q_heads
        return (torch.empty(T * H * 64, dtype=torch.uint8, device=self.device),
                torch.empty(T * H * 8, dtype=torch.uint8, device=self.device))

    # -- split-K plan + attention -----------------------------------------------------------
    def plan(self, seq_lens, q_len, causal=True, chunk_tokens=1024, stream=None):
        need = kv_nvfp4_plan_workspace_bytes(self.layout, seq_lens, q_len, causal, chunk_tokens)
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        self.plan_info = kv_nvfp4_plan(self.layout, seq_lens, q_len, causal, chunk_tokens,
                                       self.workspace, self.workspace.numel(), stream)
        return self.plan_info

    def attend(self, q_codes, q_scales, out, sm_scale=None, stream=None):
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(128)
        kv_nvfp4_decode_attn(self.layout, self.plan_info, self.workspace, q_codes, q_scales,
                             sm_scale, self.pool, self.num_pages, self.block_table, self.max_pages,
                             out, self.status, stream)

    # -- append of the step's new tokens + attention, one launch ------------------------------
    def decode_step(self, q, k, v, out, q_codes=None, q_scales=None, sm_scale=None, stream=None):
        """New tokens of every sequence (sequence-major rows, at the last q_len positions of the
        lengths given to the last plan) appended and attended in one kernel launch."""
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(128)
        kv_nvfp4_decode_step(self.layout, self.plan_info, self.workspace, q, k, v, self.rope,
                             self.max_pos, self.block_table, self.max_pages, self.num_pages,
                             self.pool, q_codes, q_scales, sm_scale, out, self.status, stream)

    # -- one decode step from host buffers -------------------------------------------------------
    def decode_step_host(self, seq_lens, q_len, h_q, h_k, h_v, d_q, d_k, d_v, d_out, h_out,
                         causal=True, chunk_tokens=1024, sm_scale=None, stream=None):
        """Plan, host-to-device copies of the new tokens, the fused step and the device-to-host
        copy of the output, enqueued by one library call (the workspace must already be large
        enough: call plan() once with the same shape first)."""
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(128)
        kv_nvfp4_decode_step_host(self.layout, seq_lens, q_len, causal, chunk_tokens,
                                  self.workspace, self.workspace.numel(), h_q, h_k, h_v, d_q, d_k,
                                  d_v, self.rope, self.max_pos, self.block_table, self.max_pages,
                                  self.num_pages, self.pool, sm_scale, d_out, h_out, self.status,
                                  stream)
