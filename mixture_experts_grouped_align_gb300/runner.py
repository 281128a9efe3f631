"""Convenience wrapper: one MoE layer resident on a CUDA device.

Holds the weights, the alignment buffers and the workspace, and runs one step of the
path -- bucket padding (W4A16 MXFP4 only), routing + alignment, the forward -- through
the C ABI.  Marshalling only: every step runs in the library's kernels.

``prewarm`` captures one CUDA graph of routing + alignment + forward per token bucket (the
bucket values up to the layer's row capacity: 97 of them for 20000 rows), so that a serving
loop never captures or sets up kernels on the hot path; ``step_bucketed`` pads a batch to
its bucket and replays that bucket's graph ("Bound Triton MoE JIT specializations via
token-dim bucketing and warmup", TensorRT-LLM PR 15311, Description: bucketing bounds the
set of specializations and a prewarm builds all of them up front).
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
                 device="cuda", block_m=BLOCK_M, pad=True, activation="swiglu"):
        self.quant, self.E, self.K, self.I, self.k = quant, E, K, I, k
        self.activation = activation
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
        self.graphs = {}  # bucket rows -> torch.cuda.CUDAGraph (prewarm)
        self._graph_stream = None
        self._y_graph = None

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

    def step(self, x, logits, T, y, stream=None, events=None, x_scale=None):
        """x [T, K] bf16 (MXFP8: E4M3 codes with x_scale [T, K/32] E8M0), logits [T, E] fp32
        on the device -> y [T, K] bf16.  ``events`` (4 torch.cuda.Event) are recorded around
        the forward's kernels."""
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
                    self.w2_scale, self.b2, xs, x_scale, T_rows, T, self.k, self.topk_w, self.sorted,
                    self.expert_ids, self.ntpp, self.expert_offsets, self.block_m, cap, y,
                    self.ctx(stream, events) if events else ctx, activation=self.activation)
        return T_rows

    # ------------------------------------------------------------------ bucket graphs
    def buckets(self, max_tokens=None):
        """The bucket values up to ``max_tokens`` (default: the row capacity), ascending."""
        hi = self.max_rows if max_tokens is None else min(max_tokens, self.max_rows)
        out, b = [], 1
        while b <= hi:
            out.append(b)
            b = moe_bucket(b + 1)
        return out

    def _bucket_body(self, b, stream):
        """Routing + alignment + forward of ``b`` padded rows from x_pad / logits_pad into
        the graph output buffer (every row of the bucket is computed; callers slice)."""
        ctx = self.ctx(stream)
        cap, _ = moe_align_capacity(b * self.k, self.E, self.block_m)
        moe_align(self.logits_pad, self.topk_ids, self.topk_w, b, self.k, self.E, self.block_m,
                  self.sorted, cap, self.expert_ids, self.ntpp, self.expert_offsets, ctx)
        moe_forward(self.quant, self.E, self.K, self.I, self.w1, self.w1_scale, self.b1, self.w2,
                    self.w2_scale, self.b2, self.x_pad, None, b, b, self.k, self.topk_w, self.sorted,
                    self.expert_ids, self.ntpp, self.expert_offsets, self.block_m, cap, self._y_graph, ctx,
                    activation=self.activation)

    def prewarm(self, max_tokens=None):
        """Captures the graph of every bucket up to ``max_tokens``; returns the bucket list."""
        if not self.pad:
            raise ValueError("bucket graphs need a padded (W4A16 MXFP4) layer")
        if self._graph_stream is None:
            self._graph_stream = torch.cuda.Stream(device=self.device)
            self._y_graph = torch.empty((self.max_rows, self.K), dtype=torch.bfloat16, device=self.device)
        s = self._graph_stream
        s.wait_stream(torch.cuda.current_stream())
        todo = [b for b in self.buckets(max_tokens) if b not in self.graphs]
        with torch.cuda.stream(s):
            for b in todo:  # one eager run of each shape first: launch setup stays out of capture
                self._bucket_body(b, s)
        s.synchronize()
        for b in todo:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                self._bucket_body(b, s)
            self.graphs[b] = g
        torch.cuda.synchronize()
        return self.buckets(max_tokens)

    def step_bucketed(self, x, logits, T):
        """Pads x [T, K] / logits [T, E] to bucket(T) rows and replays that bucket's graph;
        returns y [T, K] (a view of the graph's output buffer, valid until the next call)."""
        b = moe_bucket(T)
        g = self.graphs.get(b)
        if g is None:
            raise KeyError(f"no graph for bucket {b}: call prewarm() first")
        s = self._graph_stream
        s.wait_stream(torch.cuda.current_stream())
        moe_bucket_pad(T, self.quant, x, self.x_pad, self.K * 2, logits, self.logits_pad, self.E,
                       self.ctx(s))
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.current_stream().wait_stream(s)
        return self._y_graph[:T]
