"""Grouped expert GEMMs, SwiGLU and the top-k combine, in float64.  (Test infrastructure.)

The expert layer (per real token t and top-k slot j, e = id[t, j]):

    gu   = x_t . W1[e]^T + b1[e]          W1[e]: [2I, K], rows 0..I-1 gate, I..2I-1 up
    h    = silu(gu[:I]) * gu[I:]          silu(g) = g / (1 + exp(-g))
    o_tj = h . W2[e]^T + b2[e]            W2[e]: [K, I]
    y_t  = sum_j w[t, j] * o_tj

With MXFP8 weights the activations are MXFP8 too, and h is quantised to MXFP8 (mx_quant.py)
before GEMM2.

The non-gated variant ("tune the Nemotron MTP decode row on S5000 with a checked-in
recipe", torchada PR 115, the table of added files: the Nemotron shape's activation is
relu2_no_mul, with GEMM1 N = 1856) has one GEMM1 matrix and no gate-times-up product:

    a    = x_t . W1[e]^T + b1[e]          W1[e]: [I, K]
    h    = relu(a)^2                      relu(a) = max(a, 0)

Reading taken: "relu2" is the square of the rectified value and "no_mul" is the absence of
the gate product, so GEMM1's N is I itself (1856 on that page).

Weights are decoded exactly (formats.py) and nothing is rounded in between.  The grouped
GEMM itself -- one launch over all experts, rows taken from the alignment, optional
per-expert bias [E, N] -- is the operation of "Add MoE GEMM variants and weight-gradient
kernel" (aiter PR 5310), Summary (moe_gemm_mxfp8); the gate|up layout, SwiGLU and the
routing-weighted combine are the plain reading of the layer the three pages serve
(the pages print no formula for them).  Bias is added before SwiGLU (b1) and before the
routing weight (b2).

Every matrix product below is numpy's float64 matmul; rows are grouped by expert only so
that each expert's weights are decoded once.
"""
import numpy as np

from . import formats


def silu(g):
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def relu2(a):
    """max(a, 0)^2."""
    r = np.maximum(a, 0.0)
    return r * r


ACTIVATIONS = ("swiglu", "relu2")


class ExpertWeights:
    """Decodes one expert's weights on demand from the raw ABI layouts.

    w1 [E, 2I, K(/2)] (+ w1_scale [E, 2I, K/32]), b1 [E, 2I] bf16 bits or None,
    w2 [E, K, I(/2)]  (+ w2_scale [E, K, I/32]),  b2 [E, K]  bf16 bits or None.
    With activation "relu2" GEMM1 has I rows: w1 [E, I, K(/2)], b1 [E, I].
    """

    def __init__(self, fmt, w1, w1_scale, b1, w2, w2_scale, b2, activation="swiglu"):
        if activation not in ACTIVATIONS:
            raise ValueError(activation)
        self.fmt = fmt
        self.activation = activation
        self.w1, self.w1_scale, self.b1 = w1, w1_scale, b1
        self.w2, self.w2_scale, self.b2 = w2, w2_scale, b2

    def _get(self, w, s, e):
        return formats.dequant(self.fmt, np.asarray(w[e]), None if s is None else np.asarray(s[e]))

    def gemm1(self, e):
        b = None if self.b1 is None else formats.bf16_decode(np.asarray(self.b1[e]))
        return self._get(self.w1, self.w1_scale, e), b

    def gemm2(self, e):
        b = None if self.b2 is None else formats.bf16_decode(np.asarray(self.b2[e]))
        return self._get(self.w2, self.w2_scale, e), b


def expert_ffn(x_rows, w1, b1, w2, b2):
    """float64 rows [n, K] through one expert: GEMM1 (+b1), SwiGLU, GEMM2 (+b2)."""
    gu = x_rows @ w1.T
    if b1 is not None:
        gu = gu + b1
    inter = w1.shape[0] // 2
    h = silu(gu[:, :inter]) * gu[:, inter:]
    o = h @ w2.T
    if b2 is not None:
        o = o + b2
    return o


def expert_ffn_relu2(x_rows, w1, b1, w2, b2):
    """float64 rows [n, K] through one non-gated expert: GEMM1 (+b1), relu^2, GEMM2 (+b2)."""
    a = x_rows @ w1.T
    if b1 is not None:
        a = a + b1
    o = relu2(a) @ w2.T
    if b2 is not None:
        o = o + b2
    return o


def moe_pairs(x, topk_ids, weights: ExpertWeights, tokens=None):
    """Unweighted expert outputs o[t, j] (float64 [T, k, K]) for the tokens listed
    (default all); rows of tokens not listed stay zero."""
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    K = x.shape[1]
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    o = np.zeros((T, k, K))
    ffn = expert_ffn if getattr(weights, "activation", "swiglu") == "swiglu" else expert_ffn_relu2
    sub = ids[tok]
    for e in np.unique(sub):
        rr, jj = np.nonzero(sub == e)
        t = tok[rr]
        w1, b1 = weights.gemm1(e)
        w2, b2 = weights.gemm2(e)
        o[t, jj] = ffn(x[t], w1, b1, w2, b2)
    return o


def moe_pairs_mxfp8(x, topk_ids, weights: ExpertWeights, tokens=None):
    """MXFP8 layer, unweighted pair outputs: as moe_pairs, with h brought to MXFP8 (E4M3
    codes, one E8M0 scale per 32 features; mx_quant.mx_quantize) before GEMM2 -- GEMM2's
    operands are MXFP8 on both sides.  ``x`` is the decoded activation (float64)."""
    from . import mx_quant
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    K = x.shape[1]
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    o = np.zeros((T, k, K))
    sub = ids[tok]
    for e in np.unique(sub):
        rr, jj = np.nonzero(sub == e)
        t = tok[rr]
        w1, b1 = weights.gemm1(e)
        w2, b2 = weights.gemm2(e)
        gu = x[t] @ w1.T
        if b1 is not None:
            gu = gu + b1
        inter = w1.shape[0] // 2
        h = silu(gu[:, :inter]) * gu[:, inter:]
        hq, hs = mx_quant.mx_quantize(h)
        r = formats.dequant_mxfp8(hq, hs) @ w2.T
        if b2 is not None:
            r = r + b2
        o[t, jj] = r
    return o


def combine(o_pairs, topk_w, tokens=None):
    """y_t = sum_j w[t, j] * o[t, j] (float64)."""
    w = np.asarray(topk_w, dtype=np.float64)
    y = np.einsum("tj,tjk->tk", w, o_pairs)
    return y if tokens is None else y[np.asarray(tokens)]


def moe_layer(x, topk_ids, topk_w, weights: ExpertWeights, tokens=None):
    """The layer output y [T or len(tokens), K] in float64 (MXFP8 weights: h quantised to
    MXFP8 between the GEMMs)."""
    pairs = moe_pairs_mxfp8 if weights.fmt == "mxfp8" else moe_pairs
    return combine(pairs(x, topk_ids, weights, tokens), topk_w, tokens)


def grouped_gemm(a, topk_ids, w_of_expert, per_pair: bool, pairs=None):
    """One grouped GEMM: out[p] = a[src(p)] . W[e_p]^T (+ bias[e_p]) for pair p.

    ``a`` float64 rows, indexed by token (src = p // k) or by pair (src = p);
    ``w_of_expert(e)`` returns (W [N, Kin] float64, bias [N] or None).
    Returns float64 [P, N] for the pairs listed (default all), others zero.
    """
    ids = np.asarray(topk_ids).reshape(-1)
    k = np.asarray(topk_ids).shape[1]
    P = ids.size
    sel = np.arange(P) if pairs is None else np.asarray(pairs)
    out = None
    for e in np.unique(ids[sel]):
        pp = sel[ids[sel] == e]
        W, b = w_of_expert(e)
        if out is None:
            out = np.zeros((P, W.shape[0]))
        src = pp if per_pair else pp // k
        r = a[src] @ W.T
        if b is not None:
            r = r + b
        out[pp] = r
    return out
