"""Per-token FP8 grouped GEMM with a group-size row layout, in float64.  (Test infrastructure.)

"Add MoE GEMM variants and weight-gradient kernel" (aiter PR 5310), Summary,
moe_gemm_per_token: a grouped GEMM on FP8 operands whose per-token activation scales and
per-expert weight scales are applied after the FP8 dot product has been accumulated, with
the experts' rows described by a 1-D tensor of per-expert token counts (group_sizes).

Readings taken (the page prints no formula):
  * the rows of ``a`` are grouped by expert in expert order: expert e owns rows
    O_e .. O_e + g_e - 1 with O_e = g_0 + ... + g_{e-1};
  * one float scale per row of ``a`` and one float scale per expert's weight matrix;
  * out[m, n] = (sum_k a[m, k] * W[e, n, k]) * a_scale[m] * w_scale[e] + bias[e, n], the
    bias (optional, per expert) added after both scales, as on the MXFP8 variant of the
    same page;
  * a and W are E4M3 codes (the "fn" variant, decoded exactly by formats.e4m3_decode).

Rows past the sum of the group sizes belong to no expert and are not part of the result.
"""
import numpy as np

from . import formats


def group_offsets(group_sizes) -> np.ndarray:
    """O_e for e = 0..E (O_E = total rows), from the per-expert row counts."""
    g = np.asarray(group_sizes, dtype=np.int64)
    if (g < 0).any():
        raise ValueError("group sizes must be >= 0")
    return np.concatenate([[0], np.cumsum(g)])


def gemm_per_token(a_codes, a_scale, w_codes, w_scale, bias, group_sizes, rows=None):
    """float64 [sum(group_sizes), N] (rows listed in ``rows`` only, if given; others NaN)."""
    off = group_offsets(group_sizes)
    M = int(off[-1])
    E, N, _ = np.asarray(w_codes).shape
    out = np.full((M, N), np.nan)
    sel = np.arange(M) if rows is None else np.asarray(rows)
    a_scale = np.asarray(a_scale, dtype=np.float64)
    w_scale = np.asarray(w_scale, dtype=np.float64)
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        mine = sel[(sel >= lo) & (sel < hi)]
        if mine.size == 0:
            continue
        W = formats.e4m3_decode(np.asarray(w_codes[e]))           # [N, K]
        A = formats.e4m3_decode(np.asarray(a_codes)[mine])        # [rows, K]
        acc = A @ W.T
        r = acc * a_scale[mine][:, None] * w_scale[e]
        if bias is not None:
            r = r + formats.bf16_decode(np.asarray(bias[e]))[None, :]
        out[mine] = r
    return out
