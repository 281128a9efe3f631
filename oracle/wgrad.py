"""Per-expert weight gradient.  (Test infrastructure.)

"Add MoE GEMM variants and weight-gradient kernel" (aiter PR 5310), Summary (moe_wgrad):
dW[e] = sum over the pairs routed to e of grad[p]^T (outer) input[src(p)], read directly
from the alignment (sorted_token_ids / expert_ids).  grad is pair-indexed [P, N]; input is
indexed per token (src = p // k) or per pair (src = p).  Routing weights do not enter (the
page's formula has none); an expert no pair reaches has dW[e] = 0; sentinel slots add
nothing (Tests & Benchmarks: constant input, linearity, zero-padded tokens).
"""
import numpy as np


def moe_wgrad(grad, inp, topk_ids, E: int, per_pair: bool, experts=None):
    """float64 dW[e] = grad[P_e]^T @ input[src(P_e)] for the experts listed (default all).

    Returns an array [len(experts), N, Kin].
    """
    ids = np.asarray(topk_ids)
    k = ids.shape[1]
    flat = ids.reshape(-1)
    ex = range(E) if experts is None else experts
    g = np.asarray(grad, dtype=np.float64)
    x = np.asarray(inp, dtype=np.float64)
    out = np.zeros((len(ex), g.shape[1], x.shape[1]))
    for i, e in enumerate(ex):
        pp = np.flatnonzero(flat == e)
        if pp.size:
            src = pp if per_pair else pp // k
            out[i] = g[pp].T @ x[src]
    return out
