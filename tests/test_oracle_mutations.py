"""Plausible mistakes planted in the oracle (on the CPU) must each fail some pin."""
import numpy as np
import pytest

import oracle_pins as pins
from oracle import align, bucket, formats, layer, mx_quant, per_token, route, wgrad


def _fails(checks):
    for c in checks:
        try:
            c()
        except (AssertionError, IndexError, ValueError):
            return True
    return False


def mut_e8m0_zero(monkeypatch):
    orig = formats.e8m0_decode
    monkeypatch.setattr(formats, "e8m0_decode", lambda c: np.where(np.asarray(c) == 0, 0.0, orig(c)))
    return [pins.check_e8m0_vs_torch]


def mut_nibble_order(monkeypatch):
    def unpack(p):
        p = np.asarray(p, dtype=np.uint8)
        out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
        out[..., 0::2] = p >> 4
        out[..., 1::2] = p & 0xF
        return out
    monkeypatch.setattr(formats, "unpack_e2m1", unpack)
    return [pins.check_mxfp4_dequant_layout]


def mut_e2m1_subnormal(monkeypatch):
    orig = formats.e2m1_decode
    monkeypatch.setattr(formats, "e2m1_decode", lambda c: np.where((np.asarray(c) & 7) == 1, 1.0, orig(c)))
    return [pins.check_e2m1_table]


def mut_e4m3_bias(monkeypatch):
    orig = formats.e4m3_decode
    monkeypatch.setattr(formats, "e4m3_decode", lambda c: orig(c) * 2.0)
    return [pins.check_e4m3_vs_torch]


def mut_bucket_floor2(monkeypatch):
    orig = bucket.bucket
    monkeypatch.setattr(bucket, "bucket", lambda m: max(2, orig(m)))
    return [lambda: pins.check_bucket_properties(2000), pins.check_bucket_count_20000]


def mut_bucket_16_per_octave(monkeypatch):
    def b(m):
        s = max(1, 1 << max(0, (int(m).bit_length() - 1) - 4))
        return -(-int(m) // s) * s
    monkeypatch.setattr(bucket, "bucket", b)
    return [pins.check_bucket_count_20000]


def mut_route_tie_high(monkeypatch):
    def r(logits, k):
        l = np.asarray(logits, dtype=np.float32)
        ids = np.argsort(-l[:, ::-1], axis=1, kind="stable")[:, :k]
        ids = l.shape[1] - 1 - ids
        sel = np.take_along_axis(l, ids, 1).astype(np.float64)
        ex = np.exp(sel - sel.max(1, keepdims=True))
        return ids.astype(np.int32), (ex / ex.sum(1, keepdims=True)).astype(np.float32)
    monkeypatch.setattr(route, "route", r)
    return [pins.check_route_brute]


def mut_route_full_softmax(monkeypatch):
    def r(logits, k):
        l = np.asarray(logits, dtype=np.float32)
        ids = np.argsort(-l, axis=1, kind="stable")[:, :k]
        ex = np.exp(l.astype(np.float64) - l.max(1, keepdims=True))
        full = ex / ex.sum(1, keepdims=True)
        return ids.astype(np.int32), np.take_along_axis(full, ids, 1).astype(np.float32)
    monkeypatch.setattr(route, "route", r)
    return [pins.check_route_brute]


def mut_align_unstable(monkeypatch):
    orig = align.moe_align

    def a(ids, E, bm, cap_tokens=None):
        r = orig(ids, E, bm, cap_tokens)
        s = r["sorted_token_ids"]
        P = np.asarray(ids).size
        for e in range(E):
            o = r["padded_offsets"][e]
            c = r["counts"][e]
            s[o:o + c] = s[o:o + c][::-1]
        return r
    monkeypatch.setattr(align, "moe_align", a)
    return [pins.check_align_golden, pins.check_align_brute]


def mut_align_sentinel_zero(monkeypatch):
    orig = align.moe_align

    def a(ids, E, bm, cap_tokens=None):
        r = orig(ids, E, bm, cap_tokens)
        r["expert_ids"][r["expert_ids"] < 0] = 0
        return r
    monkeypatch.setattr(align, "moe_align", a)
    return [pins.check_align_golden]


def mut_gate_up_swapped(monkeypatch):
    def ffn(x, w1, b1, w2, b2):
        gu = x @ w1.T + (0 if b1 is None else b1)
        i = w1.shape[0] // 2
        h = layer.silu(gu[:, i:]) * gu[:, :i]
        o = h @ w2.T
        return o + (0 if b2 is None else b2)
    monkeypatch.setattr(layer, "expert_ffn", ffn)
    return [pins.check_layer_dense_formulation]


def mut_dropped_b1(monkeypatch):
    orig = layer.expert_ffn
    monkeypatch.setattr(layer, "expert_ffn", lambda x, w1, b1, w2, b2: orig(x, w1, None, w2, b2))
    return [pins.check_layer_dense_formulation, pins.check_layer_single_expert_mlp]


def mut_w2_transposed(monkeypatch):
    def ffn(x, w1, b1, w2, b2):
        gu = x @ w1.T + (0 if b1 is None else b1)
        i = w1.shape[0] // 2
        h = layer.silu(gu[:, :i]) * gu[:, i:]
        o = h @ w2[:, ::-1].T  # wrong index order inside a row
        return o + (0 if b2 is None else b2)
    monkeypatch.setattr(layer, "expert_ffn", ffn)
    return [pins.check_layer_dense_formulation, pins.check_layer_single_expert_mlp]


def mut_combine_unweighted(monkeypatch):
    monkeypatch.setattr(layer, "combine", lambda o, w, tokens=None: o.sum(1) if tokens is None else o.sum(1)[tokens])
    return [pins.check_layer_dense_formulation, pins.check_layer_bias_only]


def mut_silu_sign(monkeypatch):
    monkeypatch.setattr(layer, "silu", lambda g: g / (1.0 + np.exp(g)))
    return [pins.check_layer_dense_formulation, pins.check_layer_constant_closed_form]


def mut_relu2_unsquared(monkeypatch):
    monkeypatch.setattr(layer, "relu2", lambda a: np.maximum(a, 0.0))
    return [pins.check_layer_relu2_single_expert_loops, pins.check_layer_relu2_closed_form]


def mut_relu2_sign(monkeypatch):
    monkeypatch.setattr(layer, "relu2", lambda a: np.minimum(a, 0.0) ** 2)
    return [pins.check_layer_relu2_single_expert_loops, pins.check_layer_relu2_closed_form]


def mut_relu2_dropped_b1(monkeypatch):
    orig = layer.expert_ffn_relu2
    monkeypatch.setattr(layer, "expert_ffn_relu2", lambda x, w1, b1, w2, b2: orig(x, w1, None, w2, b2))
    return [pins.check_layer_relu2_dense_formulation, pins.check_layer_relu2_single_expert_loops]


def mut_relu2_runs_swiglu(monkeypatch):
    orig = layer.moe_pairs

    def pairs(x, ids, W, tokens=None):
        if W.activation == "relu2":  # the non-gated weights read as gate|up halves
            W = layer.ExpertWeights(W.fmt, W.w1, W.w1_scale, W.b1, W.w2, W.w2_scale, W.b2)
        return orig(x, ids, W, tokens)
    monkeypatch.setattr(layer, "moe_pairs", pairs)
    return [pins.check_layer_relu2_closed_form]


def mut_gemm_src_per_pair(monkeypatch):
    orig = layer.grouped_gemm
    monkeypatch.setattr(layer, "grouped_gemm", lambda a, ids, f, per_pair, pairs=None: orig(a, ids, f, True, pairs) if not per_pair else orig(a, ids, f, False, pairs))
    return [pins.check_grouped_gemm_brute]


def mut_wgrad_transposed(monkeypatch):
    orig = wgrad.moe_wgrad

    def w(grad, inp, ids, E, per_pair, experts=None):
        r = orig(grad, inp, ids, E, per_pair, experts)
        return r[:, ::-1, :]
    monkeypatch.setattr(wgrad, "moe_wgrad", w)
    return [pins.check_wgrad_closed_forms]


def mut_wgrad_src_index(monkeypatch):
    def w(grad, inp, ids, E, per_pair, experts=None):
        ids = np.asarray(ids)
        k = ids.shape[1]
        flat = ids.reshape(-1)
        out = np.zeros((E, grad.shape[1], inp.shape[1]))
        for e in range(E):
            pp = np.flatnonzero(flat == e)
            src = pp if per_pair else pp % k    # wrong token index
            out[e] = np.asarray(grad, float)[pp].T @ np.asarray(inp, float)[src]
        return out
    monkeypatch.setattr(wgrad, "moe_wgrad", w)
    return [pins.check_wgrad_closed_forms]


def mut_per_token_offsets_inclusive(monkeypatch):
    # expert e's first row taken as g_0 + ... + g_e (an inclusive running sum)
    monkeypatch.setattr(per_token, "group_offsets",
                        lambda g: np.concatenate([np.cumsum(np.asarray(g, dtype=np.int64)), [int(np.sum(g))]]))
    return [pins.check_per_token_constant_closed_form, pins.check_per_token_brute]


def mut_per_token_scale_of_next_row(monkeypatch):
    orig = per_token.gemm_per_token

    def f(a, sa, w, sw, b, g, rows=None):
        return orig(a, np.roll(np.asarray(sa), 1), w, sw, b, g, rows)
    monkeypatch.setattr(per_token, "gemm_per_token", f)
    return [pins.check_per_token_constant_closed_form, pins.check_per_token_brute]


def mut_per_token_weight_scale_dropped(monkeypatch):
    orig = per_token.gemm_per_token

    def f(a, sa, w, sw, b, g, rows=None):
        return orig(a, sa, w, np.ones_like(np.asarray(sw, dtype=np.float64)), b, g, rows)
    monkeypatch.setattr(per_token, "gemm_per_token", f)
    return [pins.check_per_token_constant_closed_form, pins.check_per_token_brute]


def mut_mx_scale_ceil(monkeypatch):
    orig = mx_quant.block_exponent
    monkeypatch.setattr(mx_quant, "block_exponent", lambda amax: orig(amax) + 1)
    return [pins.check_mx_quantize_scale_rule]


def mut_mx_emax_7(monkeypatch):
    monkeypatch.setattr(mx_quant, "E4M3_EMAX", 7)
    return [pins.check_mx_quantize_scale_rule]


def mut_e4m3_ties_away(monkeypatch):
    mags = formats.e4m3_decode(np.arange(0x7F))

    def enc(v):
        v = np.asarray(v, dtype=np.float64)
        a = np.abs(v)
        code = np.abs(a[..., None] - mags).argmin(-1)       # first minimum: ties go down
        code = np.where(a >= 448, 0x7E, code) | np.where(np.signbit(v), 0x80, 0)
        return np.where(np.isnan(v), 0x7F, code).astype(np.uint8)
    monkeypatch.setattr(mx_quant, "e4m3_encode", enc)
    return [pins.check_e4m3_encode_vs_torch]


def mut_e4m3_no_saturation(monkeypatch):
    orig = mx_quant.e4m3_encode
    monkeypatch.setattr(mx_quant, "e4m3_encode",
                        lambda v: np.where(np.abs(np.asarray(v, dtype=np.float64)) > 464, 0x7F, orig(v)).astype(np.uint8))
    return [pins.check_e4m3_encode_saturates_and_round_trips]


def mut_mxfp8_layer_skips_quantiser(monkeypatch):
    monkeypatch.setattr(mx_quant, "mx_quantize",
                        lambda x: (np.zeros(np.shape(x), np.uint8), np.zeros(np.shape(x)[:-1] + (np.shape(x)[-1] // 32,), np.uint8)))
    return [pins.check_layer_mxfp8_constant_closed_form]



def mut_mxfp8_h_blocks_strided(monkeypatch):
    # h quantised with the wrong block grouping: block b holds features b, b + C/32, ...
    orig = mx_quant.mx_quantize

    def q(x):
        x = np.asarray(x, dtype=np.float64)
        C = x.shape[-1]
        xt = x.reshape(*x.shape[:-1], 32, C // 32).swapaxes(-1, -2).reshape(x.shape)
        c, s_ = orig(xt)
        c = c.reshape(*x.shape[:-1], C // 32, 32).swapaxes(-1, -2).reshape(x.shape)
        return c, s_
    monkeypatch.setattr(mx_quant, "mx_quantize", q)
    return [pins.check_layer_mxfp8_constant_closed_form, pins.check_layer_mxfp8_brute_rows]


def mut_mxfp8_h_scales_reversed(monkeypatch):
    # the scales of h applied to the blocks in reverse order
    orig = mx_quant.mx_quantize
    monkeypatch.setattr(mx_quant, "mx_quantize", lambda x: (orig(x)[0], orig(x)[1][..., ::-1].copy()))
    return [pins.check_layer_mxfp8_constant_closed_form, pins.check_layer_mxfp8_brute_rows]


def mut_mxfp8_h_quantised_over_tokens(monkeypatch):
    # h quantised along the token axis of each expert's rows (blocks run down the columns)
    orig = mx_quant.mx_quantize

    def q(x):
        x = np.asarray(x, dtype=np.float64)
        if x.ndim != 2:
            return orig(x)
        n, C = x.shape
        pad = (-n) % 32
        xp = np.concatenate([x, np.zeros((pad, C))], axis=0)
        c, s_ = orig(xp.T)
        codes = c.T[:n]
        scale_rows = np.repeat(s_.T, 32, axis=0)[:n]          # [n, C] one scale per element
        return codes, scale_rows[:, ::32].copy()
    monkeypatch.setattr(mx_quant, "mx_quantize", q)
    return [pins.check_layer_mxfp8_constant_closed_form, pins.check_layer_mxfp8_brute_rows]

MUTATIONS = [mut_e8m0_zero, mut_nibble_order, mut_e2m1_subnormal, mut_e4m3_bias,
             mut_bucket_floor2, mut_bucket_16_per_octave, mut_route_tie_high,
             mut_route_full_softmax, mut_align_unstable, mut_align_sentinel_zero,
             mut_gate_up_swapped, mut_dropped_b1, mut_w2_transposed, mut_combine_unweighted,
             mut_silu_sign, mut_relu2_unsquared, mut_relu2_sign, mut_relu2_dropped_b1,
             mut_relu2_runs_swiglu, mut_per_token_offsets_inclusive,
             mut_per_token_scale_of_next_row, mut_per_token_weight_scale_dropped,
             mut_mx_scale_ceil, mut_mx_emax_7, mut_e4m3_ties_away, mut_e4m3_no_saturation,
             mut_mxfp8_layer_skips_quantiser, mut_mxfp8_h_blocks_strided,
             mut_mxfp8_h_scales_reversed, mut_mxfp8_h_quantised_over_tokens,
             mut_gemm_src_per_pair, mut_wgrad_transposed, mut_wgrad_src_index]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutation, monkeypatch):
    checks = mutation(monkeypatch)
    assert _fails(checks), f"{mutation.__name__} was not caught"
