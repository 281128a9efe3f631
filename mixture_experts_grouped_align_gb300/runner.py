"""Convenience wrapper: one MoE layer resident on a CUDA device.

Holds the weights, the alignment buffers and the workspace, and runs one step of the
path -- bucket padding (W4A16 MXFP4 only), routing + alignment, the forward -- through
the C ABI.  Marshalling only: every step runs in the library's kernels.
"""
from __future__ import annotations

import torch

from . import (Ctx, moe_align, moe_align_capacity, moe_bucket, moe_bucket_pad, moe_forward,
               moe_forward_workspace_size)

BLOCK_M = 128


class DeviceLayer:
    """Weights (torch uint8 / bf16 device tensors in the C ABI layouts) + buffers for up
    to ``max_rows`` token rows."""

    def __init__(self, quant, E, K, I, k, w1, w1_scale, b1, w2, w2_scale, b2, max_rows,
                 device="cuda", block_m=BLOCK_M, pad=True):
        self.quant, self.E, self.K, self.I, self.k = quant, E, K, I, k
        self.w1, self.w1_scale, self.b1 = w1, w1_scale, b1
        self.w2, self.w2_scale, self.b2 = w2, w2_scale, b2
        self.block_m = block_m
        self.pad = pad and quant == "mxfp4"
        rows = moe_bucket(max_rows) if self.pad and max_rows > 0 else max_rows
        self.max_rows = rows
        self.device = device
        P = rows * k
        self.cap, self.cap_blocks = moe_align_capacity(P, E, block_m)
        dev = device
        self.topk_ids = torch.empty((rows, k), dtype=torch.int32, device=dev)
        self.topk_w = torch.empty((rows, k), dtype=torch.float32, device=dev)
        self.sorted = torch.empty(self.cap, dtype=torch.int32, device=dev)
        self.expert_ids = torch.empty(max(self.cap_blocks, 1), dtype=torch.int32, device=dev)
        self.ntpp = torch.zeros(4, dtype=torch.int32, device=dev)
        self.expert_offsets = torch.empty(E + 1 + (-(E + 1)) % 4, dtype=torch.int32, device=dev)
        self.x_pad = torch.zeros((rows, K), dtype=torch.bfloat16, device=dev)
        self.logits_pad = torch.zeros((rows, E), dtype=torch.float32, device=dev)
        self.ws_bytes = moe_forward_workspace_size(rows, k, K, I, self.cap)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self._ctx_cache = {}

    def ctx(self, stream=None, events=None):
        key = (stream, None if events is None else tuple(id(e) for e in events))
        c = self._ctx_cache.get(key)
        if c is None:
            c = Ctx(stream=stream, workspace=self.workspace, dev_status=self.status, events=events)
            if len(self._ctx_cache) > 64:
                self._ctx_cache.clear()
            self._ctx_cache[key] = c
        return c

    def rows_for(self, T):
        return moe_bucket(T) if (self.pad and T > 0) else T

    def step(self, x, logits, T, y, stream=None, events=None):
        """x [T, K] bf16, logits [T, E] fp32 on the device -> y [T, K] bf16.  ``events``
        (4 torch.cuda.Event) are recorded around the forward's kernels."""
        ctx = self.ctx(stream)
        if self.pad:
            _, T_rows = moe_bucket_pad(T, self.quant, x, self.x_pad, self.K * 2, logits,
                                       self.logits_pad, self.E, ctx)
            xs, ls = self.x_pad, self.logits_pad
        else:
            T_rows, xs, ls = T, x, logits
        cap, _ = moe_align_capacity(T_rows * self.k, self.E, self.block_m)
        moe_align(ls, self.topk_ids, self.topk_w, T_rows, self.k, self.E, self.block_m,
                  self.sorted, cap, self.expert_ids, self.ntpp, self.expert_offsets, ctx)
        moe_forward(self.quant, self.E, self.K, self.I, self.w1, self.w1_scale, self.b1, self.w2,
                    self.w2_scale, self.b2, xs, None, T_rows, T, self.k, self.topk_w, self.sorted,
                    self.expert_ids, self.ntpp, self.expert_offsets, self.block_m, cap, y,
                    self.ctx(stream, events) if events else ctx)
        return T_rows
