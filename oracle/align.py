"""Token-to-expert alignment (moe_align_block_size).  (Test infrastructure.)

Inputs: top-k expert ids [T, k]; flat pair index p = t*k + j.  With BM = block_m:

* c_e      = number of pairs routed to expert e;
* P_e      = ceil(c_e / BM) * BM, the count padded to whole blocks;
* O_e      = sum of P_e' over e' < e (padded offsets);
* sorted_token_ids[O_e + r] = the r-th pair index p (ascending) with id e; the remaining
  slots of each expert's padded range and every slot from sum(P_e) up to the capacity
  hold the sentinel P = T*k (one past the last pair);
* expert_ids[b] = e for blocks b in [O_e/BM, O_{e+1}/BM) and -1 for every block slot
  from sum(P_e)/BM up to the capacity -- the -1 sentinel blocks that the second review of
  "Add MoE GEMM variants and weight-gradient kernel" (aiter PR 5310) says every mapping
  has and kernels must skip;
* num_tokens_post_padded = sum(P_e);
* expert_offsets[e] = sum of c_e' over e' < e (unpadded; [E+1] entries), the per-expert
  token counts of the ``group_sizes`` interface on the same page (Summary) as differences.

Capacity: C = P + E*(BM-1) rounded up to BM (the most any routing can need), with C/BM
block slots.  Expert ids outside [0, E) are rejected.
"""
import numpy as np


def capacity(P: int, E: int, block_m: int):
    c = P + E * (block_m - 1)
    c = -(-c // block_m) * block_m
    return c, c // block_m


def moe_align(topk_ids, E: int, block_m: int, cap_tokens: int | None = None):
    ids = np.asarray(topk_ids, dtype=np.int64)
    flat = ids.reshape(-1)
    P = flat.size
    if P and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    cap, cap_blocks = capacity(P, E, block_m)
    if cap_tokens is not None:
        if cap_tokens < cap or cap_tokens % block_m:
            raise ValueError("capacity too small or not a multiple of block_m")
        cap, cap_blocks = cap_tokens, cap_tokens // block_m
    counts = np.array([int(np.count_nonzero(flat == e)) for e in range(E)], dtype=np.int64)
    padded = -(-counts // block_m) * block_m
    offs = np.concatenate([[0], np.cumsum(padded)])
    sorted_ids = np.full(cap, P, dtype=np.int32)
    expert_ids = np.full(cap_blocks, -1, dtype=np.int32)
    for e in range(E):
        members = np.flatnonzero(flat == e)   # ascending pair indices
        sorted_ids[offs[e]:offs[e] + members.size] = members
        expert_ids[offs[e] // block_m:offs[e + 1] // block_m] = e
    ntpp = np.int32(offs[-1])
    expert_offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return {"sorted_token_ids": sorted_ids, "expert_ids": expert_ids,
            "num_tokens_post_padded": ntpp, "expert_offsets": expert_offsets,
            "padded_offsets": offs.astype(np.int64), "counts": counts}
