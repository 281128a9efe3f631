"""Top-k routing of router logits.  (Test infrastructure.)

For every token (a row of logits [T, E], fp32) the k experts with the largest logits are
chosen, in descending order of logit; equal logits rank the lower expert index first.
The routing weights are the softmax over the k chosen logits -- equal to the full softmax
renormalised over the top-k -- computed in float64 and rounded to float32 (RNE).

The pages fix the workloads' routing only by name (softmax over the top-k, renormalised;
silu(gate)*up), so this is the plain reading of it.  A zero logit row (the pad rows of a
bucketed batch) ties everywhere and therefore routes to experts 0..k-1 with weight 1/k.
"""
import numpy as np


def route(logits, k: int):
    l32 = np.asarray(logits, dtype=np.float32)
    T, E = l32.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    for t in range(T):
        row = l32[t]
        # stable sort of the negated values: larger logit first, lower index on ties
        order = np.argsort(-row, kind="stable")[:k]
        sel = row[order].astype(np.float64)
        ex = np.exp(sel - sel.max())
        ids[t] = order
        w[t] = (ex / ex.sum()).astype(np.float32)
    return ids, w
