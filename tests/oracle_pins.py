"""Pins of the CPU oracle: checks against things other than the oracle itself.

Each ``check_*`` raises AssertionError on a mismatch.  ``test_oracle_pins.py`` runs them
on the oracle as it is; ``test_oracle_mutations.py`` plants plausible mistakes in the
oracle (on the CPU) and asserts that some check catches each one.
"""
import math
import os

import numpy as np
import torch

import oracle
from oracle import align, bucket, formats, layer, mx_quant, per_token, route, wgrad

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


# ----------------------------------------------------------------------------- formats

def check_e2m1_table():
    g = _golden("e2m1_e8m0_ocp.txt")
    want = np.array([float(v) for v in g["e2m1"]])
    got = formats.e2m1_decode(np.arange(16))
    assert np.array_equal(got, want), (got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def check_e8m0_vs_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(torch.float8_e8m0fnu).double().numpy()
    got = formats.e8m0_decode(np.arange(256))
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    g = _golden("e2m1_e8m0_ocp.txt")
    bits = int(g["e8m0_0x00_f32_bits"][0], 16)
    assert np.float32(got[0]).view(np.uint32) == bits
    assert got[127] == float(g["e8m0_0x7f"][0])
    assert np.isnan(got[255])


def check_e4m3_vs_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(torch.float8_e4m3fn).double().numpy()
    got = formats.e4m3_decode(np.arange(256))
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def check_bf16_vs_torch():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=4096).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = formats.bf16_decode(bits)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def check_mxfp4_dequant_layout():
    # one row of K=64: byte b packs element 2b (low nibble) and 2b+1 (high nibble);
    # elements 0..31 use scale byte 0, 32..63 scale byte 1
    packed = np.array([[0x21] + [0x00] * 15 + [0xF7] + [0x00] * 15], dtype=np.uint8)
    scales = np.array([[127 + 3, 127 - 2]], dtype=np.uint8)
    v = formats.dequant_mxfp4(packed, scales)[0]
    assert v[0] == 0.5 * 8 and v[1] == 1.0 * 8            # codes 1, 2 at scale 2^3
    assert v[32] == 6.0 * 0.25 and v[33] == -6.0 * 0.25   # codes 7, 15 at scale 2^-2
    assert np.count_nonzero(v) == 4


# ----------------------------------------------------------------------------- bucket

def check_bucket_properties(n_max=65536):
    fixed = []
    closure = set()
    prev = 0
    for m in range(1, n_max + 1):
        b = bucket.bucket(m)
        assert b >= m and 8 * (b - m) <= m, m          # rounds up by at most 12.5%
        assert bucket.bucket(b) == b, m                # fixed point
        assert b >= prev, m                            # monotonic
        prev = b
        if b == m:
            fixed.append(m)
        closure.add(b)
        # enumeration matches closure: the buckets <= bucket(m) are exactly the values
        # that bucket() takes on [1, m] plus the buckets between m and bucket(m)
        n_le = len(fixed) + (1 if b > m else 0)
        assert n_le == len(closure), m
        if m % 997 == 0 or m in (1, 15, 16, 17, 20000, n_max):
            assert set(bucket.bucket_iter(b)) == closure, m
    return fixed


def check_bucket_count_20000():
    assert len(bucket.bucket_iter(20000)) == 97
    its = bucket.bucket_iter(65536)
    assert its == sorted(set(its))
    assert its[:16] == list(range(1, 17))
    for j in range(4, 16):  # 8 buckets per power-of-two octave from 16 on
        assert len([b for b in its if 2 ** j <= b < 2 ** (j + 1)]) == 8


def check_pad_restriction():
    assert bucket.padded_rows(17, "mxfp4") == 18
    assert bucket.padded_rows(17, "bf16") == 17
    assert bucket.padded_rows(17, "mxfp8") == 17


# ----------------------------------------------------------------------------- route

def check_route_brute(seed=0):
    rng = np.random.default_rng(seed)
    for T, E, k in [(7, 5, 2), (4, 8, 8), (9, 16, 3), (3, 3, 1)]:
        lg = rng.standard_normal((T, E)).astype(np.float32)
        lg[0, :] = 0.0                           # full tie
        lg[1, E // 2:] = lg[1, 0]                # partial ties
        ids, w = route.route(lg, k)
        for t in range(T):
            order = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))[:k]
            assert list(ids[t]) == order, (t, list(ids[t]), order)
            vals = [float(lg[t, e]) for e in order]
            mx = max(vals)
            ex = [math.exp(v - mx) for v in vals]
            s = math.fsum(ex)
            want = np.array([v / s for v in ex], dtype=np.float32)
            assert np.max(np.abs(w[t].view(np.int32) - want.view(np.int32))) <= 1
            # equals the full softmax renormalised over the chosen experts
            full = np.exp(lg[t].astype(np.float64) - lg[t].max())
            full /= full.sum()
            ren = full[order] / full[order].sum()
            assert np.allclose(w[t], ren, rtol=1e-6, atol=0)
        assert list(ids[0]) == list(range(k))
        assert np.all(w[0] == np.float32(1.0 / k))


# ----------------------------------------------------------------------------- align

def check_align_golden():
    g = _golden("align_small.txt")
    T, k, E, bm = (int(g[n][0]) for n in ("T", "k", "E", "block_m"))
    ids = np.array([int(v) for v in g["topk_ids"]]).reshape(T, k)
    r = align.moe_align(ids, E, bm)
    assert r["sorted_token_ids"].tolist() == [int(v) for v in g["sorted_token_ids"]]
    assert r["expert_ids"].tolist() == [int(v) for v in g["expert_ids"]]
    assert int(r["num_tokens_post_padded"]) == int(g["num_tokens_post_padded"][0])
    assert r["expert_offsets"].tolist() == [int(v) for v in g["expert_offsets"]]


def _align_brute(ids, E, bm):
    T, k = ids.shape
    P = T * k
    pairs = sorted((int(ids[p // k, p % k]), p) for p in range(P))
    sorted_ids, expert_ids = [], []
    for e in range(E):
        mine = [p for (ee, p) in pairs if ee == e]
        if not mine:
            continue
        n_blocks = (len(mine) + bm - 1) // bm
        sorted_ids += mine + [P] * (n_blocks * bm - len(mine))
        expert_ids += [e] * n_blocks
    cap = P + E * (bm - 1)
    cap = (cap + bm - 1) // bm * bm
    ntpp = len(sorted_ids)
    sorted_ids += [P] * (cap - len(sorted_ids))
    expert_ids += [-1] * (cap // bm - len(expert_ids))
    return sorted_ids, expert_ids, ntpp


def check_align_brute(seed=1):
    rng = np.random.default_rng(seed)
    for T, k, E, bm in [(1, 1, 1, 1), (6, 2, 5, 4), (13, 3, 7, 8), (40, 4, 16, 16), (3, 2, 9, 128)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        r = align.moe_align(ids, E, bm)
        s, b, n = _align_brute(ids, E, bm)
        assert r["sorted_token_ids"].tolist() == s
        assert r["expert_ids"].tolist() == b
        assert int(r["num_tokens_post_padded"]) == n
        cnt = np.bincount(ids.reshape(-1), minlength=E)
        assert r["expert_offsets"].tolist() == [0] + np.cumsum(cnt).tolist()


def check_align_invariants(seed=2):
    rng = np.random.default_rng(seed)
    T, k, E, bm = 300, 4, 32, 16
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids = np.where(ids == 7, (ids + 1) % E, ids)    # expert 7 empty; a token may repeat 8
    r = align.moe_align(ids, E, bm)
    P = T * k
    s, b = r["sorted_token_ids"], r["expert_ids"]
    real = s[s < P]
    assert sorted(real.tolist()) == list(range(P))            # every pair exactly once
    n = int(r["num_tokens_post_padded"])
    assert n % bm == 0 and n <= s.size and np.all(s[n:] == P)
    assert np.all(b[n // bm:] == -1) and np.all(b[:n // bm] >= 0)
    assert np.all(np.diff(b[:n // bm]) >= 0)                  # blocks contiguous per expert
    assert 7 not in b.tolist()                                # empty expert has no block
    flat = ids.reshape(-1)
    for blk in range(n // bm):
        row = s[blk * bm:(blk + 1) * bm]
        assert np.all(flat[row[row < P]] == b[blk])
        rr = row[row < P]
        assert np.all(np.diff(rr) > 0)                        # ascending within expert


# ----------------------------------------------------------------------------- layer

def _rand_weights(rng, E, K, I, fmt="mxfp4", bias=True, scale=(-4, 0), activation="swiglu"):
    N1 = 2 * I if activation == "swiglu" else I
    if fmt == "mxfp4":
        w1 = rng.integers(0, 256, size=(E, N1, K // 2), dtype=np.uint8)
        s1 = (127 + rng.integers(scale[0], scale[1] + 1, size=(E, N1, K // 32))).astype(np.uint8)
        w2 = rng.integers(0, 256, size=(E, K, I // 2), dtype=np.uint8)
        s2 = (127 + rng.integers(scale[0], scale[1] + 1, size=(E, K, I // 32))).astype(np.uint8)
    else:
        from synth import to_bf16_bits
        w1 = to_bf16_bits(rng.standard_normal((E, N1, K)) * 0.05)
        w2 = to_bf16_bits(rng.standard_normal((E, K, I)) * 0.05)
        s1 = s2 = None
    from synth import to_bf16_bits
    b1 = to_bf16_bits(rng.standard_normal((E, N1)) * 0.1) if bias else None
    b2 = to_bf16_bits(rng.standard_normal((E, K)) * 0.1) if bias else None
    return layer.ExpertWeights(fmt, w1, s1, b1, w2, s2, b2, activation=activation)


def _dense_all_experts(x, ids, w, W: layer.ExpertWeights, E):
    """Every expert on every token, then mask by routing: an independent formulation."""
    T, K = x.shape
    W1 = np.stack([formats.dequant(W.fmt, W.w1[e], None if W.w1_scale is None else W.w1_scale[e]) for e in range(E)])
    W2 = np.stack([formats.dequant(W.fmt, W.w2[e], None if W.w2_scale is None else W.w2_scale[e]) for e in range(E)])
    if W.activation == "relu2":  # relu(a)^2 written as a * a * step(a)
        a = np.einsum("tk,eik->tei", x, W1)
        if W.b1 is not None:
            a = a + formats.bf16_decode(W.b1)[None]
        act = a * a * (a > 0)
    else:
        I = W1.shape[1] // 2
        gate = np.einsum("tk,eik->tei", x, W1[:, :I, :])
        up = np.einsum("tk,eik->tei", x, W1[:, I:, :])
        if W.b1 is not None:
            b1 = formats.bf16_decode(W.b1)
            gate = gate + b1[None, :, :I]
            up = up + b1[None, :, I:]
        act = gate * (1.0 / (1.0 + np.exp(-gate))) * up
    o = np.einsum("tei,eki->tek", act, W2)
    if W.b2 is not None:
        o = o + formats.bf16_decode(W.b2)[None]
    mask = np.zeros((T, E))
    for t in range(T):
        for j in range(ids.shape[1]):
            mask[t, ids[t, j]] += float(w[t, j])
    return np.einsum("te,tek->tk", mask, o)


def check_layer_dense_formulation(seed=3):
    rng = np.random.default_rng(seed)
    for fmt in ("mxfp4", "bf16"):
        T, K, I, E, k = 11, 64, 32, 5, 2
        W = _rand_weights(rng, E, K, I, fmt=fmt)
        from synth import to_bf16_bits
        x = formats.bf16_decode(to_bf16_bits(rng.standard_normal((T, K))))
        ids, w = route.route(rng.standard_normal((T, E)).astype(np.float32), k)
        y = layer.moe_layer(x, ids, w, W)
        yd = _dense_all_experts(x, ids, w, W, E)
        assert np.allclose(y, yd, rtol=1e-11, atol=1e-11), np.abs(y - yd).max()


def check_layer_single_expert_mlp(seed=4):
    """E=1, k=1: the layer is a plain dense MLP (per-row Python loops)."""
    rng = np.random.default_rng(seed)
    T, K, I = 3, 32, 32
    W = _rand_weights(rng, 1, K, I)
    from synth import to_bf16_bits
    x = formats.bf16_decode(to_bf16_bits(rng.standard_normal((T, K))))
    ids = np.zeros((T, 1), dtype=np.int32)
    w = np.ones((T, 1), dtype=np.float32)
    y = layer.moe_layer(x, ids, w, W)
    W1 = formats.dequant_mxfp4(W.w1[0], W.w1_scale[0])
    W2 = formats.dequant_mxfp4(W.w2[0], W.w2_scale[0])
    b1 = formats.bf16_decode(W.b1[0])
    b2 = formats.bf16_decode(W.b2[0])
    for t in range(T):
        h = []
        for i in range(I):
            g = math.fsum(x[t, c] * W1[i, c] for c in range(K)) + b1[i]
            u = math.fsum(x[t, c] * W1[I + i, c] for c in range(K)) + b1[I + i]
            h.append(g / (1.0 + math.exp(-g)) * u)
        for n in range(K):
            o = math.fsum(h[i] * W2[n, i] for i in range(I)) + b2[n]
            assert abs(o - y[t, n]) <= 1e-12 * max(1.0, abs(o)), (t, n, o, y[t, n])


def check_layer_constant_closed_form():
    """Constant activations a, constant codes and scales: closed form per stage."""
    T, K, I, E, k = 4, 64, 32, 3, 2
    a = 0.75
    c1, c2 = 0x3, 0xA          # E2M1 1.5 and -1.0
    s1, s2 = 127 - 3, 127 - 1
    w1 = np.full((E, 2 * I, K // 2), c1 | (c1 << 4), dtype=np.uint8)
    w2 = np.full((E, K, I // 2), c2 | (c2 << 4), dtype=np.uint8)
    W = layer.ExpertWeights("mxfp4", w1, np.full((E, 2 * I, K // 32), s1, np.uint8), None,
                            w2, np.full((E, K, I // 32), s2, np.uint8), None)
    x = np.full((T, K), a)
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2]], dtype=np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5], [1.0, 0.0], [0.125, 0.875]], dtype=np.float32)
    y = layer.moe_layer(x, ids, w, W)
    g = K * a * 1.5 * 2.0 ** -3
    h = g / (1.0 + math.exp(-g)) * g
    o = I * h * (-1.0) * 2.0 ** -1
    for t in range(T):
        assert np.allclose(y[t], float(w[t].astype(np.float64).sum()) * o, rtol=1e-14, atol=0)


def check_layer_bias_only():
    """Zero weights: o = b2[e], y = sum_j w_j b2[e_j] (b1 then has no effect)."""
    rng = np.random.default_rng(6)
    T, K, I, E, k = 5, 32, 32, 4, 2
    W = _rand_weights(rng, E, K, I)
    W.w1 = np.zeros_like(W.w1)
    W.w2 = np.zeros_like(W.w2)
    x = rng.standard_normal((T, K))
    ids, w = route.route(rng.standard_normal((T, E)).astype(np.float32), k)
    y = layer.moe_layer(x, ids, w, W)
    b2 = formats.bf16_decode(W.b2)
    want = np.einsum("tj,tjk->tk", w.astype(np.float64), b2[ids])
    assert np.allclose(y, want, rtol=1e-14, atol=1e-15)


def check_layer_relu2_dense_formulation(seed=10):
    rng = np.random.default_rng(seed)
    for fmt in ("mxfp4", "bf16"):
        T, K, I, E, k = 13, 64, 64, 6, 3
        W = _rand_weights(rng, E, K, I, fmt=fmt, activation="relu2")
        from synth import to_bf16_bits
        x = formats.bf16_decode(to_bf16_bits(rng.standard_normal((T, K))))
        ids, w = route.route(rng.standard_normal((T, E)).astype(np.float32), k)
        y = layer.moe_layer(x, ids, w, W)
        yd = _dense_all_experts(x, ids, w, W, E)
        assert np.allclose(y, yd, rtol=1e-11, atol=1e-11), np.abs(y - yd).max()


def check_layer_relu2_single_expert_loops(seed=11):
    """E=1, k=1, non-gated: a dense relu^2 MLP in per-element Python loops; the random bias
    gives pre-activations of both signs."""
    rng = np.random.default_rng(seed)
    T, K, I = 3, 32, 64
    W = _rand_weights(rng, 1, K, I, activation="relu2")
    from synth import to_bf16_bits
    x = formats.bf16_decode(to_bf16_bits(rng.standard_normal((T, K))))
    ids = np.zeros((T, 1), dtype=np.int32)
    w = np.ones((T, 1), dtype=np.float32)
    y = layer.moe_layer(x, ids, w, W)
    W1 = formats.dequant_mxfp4(W.w1[0], W.w1_scale[0])
    W2 = formats.dequant_mxfp4(W.w2[0], W.w2_scale[0])
    b1 = formats.bf16_decode(W.b1[0])
    b2 = formats.bf16_decode(W.b2[0])
    signs = set()
    for t in range(T):
        h = []
        for i in range(I):
            a = math.fsum(x[t, c] * W1[i, c] for c in range(K)) + b1[i]
            signs.add(a > 0)
            h.append(a * a if a > 0 else 0.0)
        for n in range(K):
            o = math.fsum(h[i] * W2[n, i] for i in range(I)) + b2[n]
            assert abs(o - y[t, n]) <= 1e-12 * max(1.0, abs(o)), (t, n, o, y[t, n])
    assert signs == {True, False}


def check_layer_relu2_closed_form():
    """Constant codes and scales, no bias: a positive constant activation gives h = g^2 per
    feature; its negation gives h = 0 and y = 0; and the layer is homogeneous of degree 2."""
    T, K, I, E = 4, 64, 32, 3
    c1, c2 = 0x3, 0xA          # E2M1 1.5 and -1.0
    s1, s2 = 127 - 3, 127 - 1
    w1 = np.full((E, I, K // 2), c1 | (c1 << 4), dtype=np.uint8)
    w2 = np.full((E, K, I // 2), c2 | (c2 << 4), dtype=np.uint8)
    W = layer.ExpertWeights("mxfp4", w1, np.full((E, I, K // 32), s1, np.uint8), None,
                            w2, np.full((E, K, I // 32), s2, np.uint8), None, activation="relu2")
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2]], dtype=np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5], [1.0, 0.0], [0.125, 0.875]], dtype=np.float32)
    a = 0.75
    y = layer.moe_layer(np.full((T, K), a), ids, w, W)
    g = K * a * 1.5 * 2.0 ** -3
    o = I * g * g * (-1.0) * 2.0 ** -1
    for t in range(T):
        assert np.allclose(y[t], float(w[t].astype(np.float64).sum()) * o, rtol=1e-14, atol=0)
    assert np.array_equal(layer.moe_layer(np.full((T, K), -a), ids, w, W), np.zeros((T, K)))
    rng = np.random.default_rng(12)
    Wr = _rand_weights(rng, E, K, I, bias=False, activation="relu2")
    x = rng.standard_normal((T, K))
    y1 = layer.moe_layer(x, ids, w, Wr)
    y3 = layer.moe_layer(3.0 * x, ids, w, Wr)
    assert np.allclose(y3, 9.0 * y1, rtol=1e-12, atol=1e-12)


def check_layer_empty_expert_no_effect(seed=7):
    rng = np.random.default_rng(seed)
    T, K, I, E, k = 9, 64, 32, 4, 2
    W = _rand_weights(rng, E + 1, K, I)
    x = rng.standard_normal((T, K))
    ids, w = route.route(rng.standard_normal((T, E)).astype(np.float32), k)
    y5 = layer.moe_layer(x, ids, w, W)                # expert 4 exists, gets nothing
    W4 = layer.ExpertWeights("mxfp4", W.w1[:E], W.w1_scale[:E], W.b1[:E], W.w2[:E],
                             W.w2_scale[:E], W.b2[:E])
    y4 = layer.moe_layer(x, ids, w, W4)
    assert np.array_equal(y5, y4)


def check_grouped_gemm_brute(seed=8):
    rng = np.random.default_rng(seed)
    T, k, E, N, Kin = 6, 3, 4, 5, 64
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    Ws = [rng.standard_normal((N, Kin)) for _ in range(E)]
    bs = [rng.standard_normal(N) for _ in range(E)]
    for per_pair in (False, True):
        a = rng.standard_normal((T * k if per_pair else T, Kin))
        out = layer.grouped_gemm(a, ids, lambda e: (Ws[e], bs[e]), per_pair)
        for p in range(T * k):
            e = ids[p // k, p % k]
            row = a[p if per_pair else p // k]
            for n in range(N):
                want = math.fsum(row[c] * Ws[e][n, c] for c in range(Kin)) + bs[e][n]
                assert abs(out[p, n] - want) <= 1e-12 * max(1, abs(want))


# ----------------------------------------------------------------------------- wgrad

def check_wgrad_closed_forms(seed=9):
    rng = np.random.default_rng(seed)
    T, k, E, N, Kin = 10, 2, 6, 4, 8
    ids = np.stack([rng.permutation(E - 1)[:k] for _ in range(T)]).astype(np.int32)  # expert E-1 empty
    # constant grad g and input a: dW[e] = n_e * g * a
    dW = wgrad.moe_wgrad(np.full((T * k, N), 0.5), np.full((T, Kin), -3.0), ids, E, per_pair=False)
    cnt = np.bincount(ids.reshape(-1), minlength=E)
    for e in range(E):
        assert np.all(dW[e] == cnt[e] * 0.5 * -3.0)
    assert np.all(dW[E - 1] == 0)
    # linearity in grad
    g1, g2 = rng.standard_normal((T * k, N)), rng.standard_normal((T * k, N))
    x = rng.standard_normal((T, Kin))
    lhs = wgrad.moe_wgrad(2.0 * g1 - 3.0 * g2, x, ids, E, False)
    rhs = 2.0 * wgrad.moe_wgrad(g1, x, ids, E, False) - 3.0 * wgrad.moe_wgrad(g2, x, ids, E, False)
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    # brute-force outer products; per-pair input equal to the token rows gives the same
    want = np.zeros((E, N, Kin))
    for p in range(T * k):
        want[ids[p // k, p % k]] += np.outer(g1[p], x[p // k])
    assert np.allclose(wgrad.moe_wgrad(g1, x, ids, E, False), want, rtol=1e-12, atol=1e-12)
    xp = x[np.arange(T * k) // k]
    assert np.allclose(wgrad.moe_wgrad(g1, xp, ids, E, True), want, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- per-token FP8

def _e4m3_codes(rng, shape):
    """Random finite E4M3 codes (0x7F / 0xFF are NaN)."""
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    return np.where((c & 0x7F) == 0x7F, c - 1, c).astype(np.uint8)


def check_per_token_constant_closed_form():
    """Constant codes (the page's constant-input round trip): every row is
    K * a * w * a_scale[m] * w_scale[e] (+ bias[e, n]), with an empty expert in between."""
    K, N = 64, 16
    g = np.array([3, 0, 5, 2])
    M = int(g.sum())
    a = np.full((M, K), 0x38, np.uint8)            # E4M3 1.0
    w = np.full((4, N, K), 0xB4, np.uint8)         # E4M3 -0.75
    sa = np.linspace(0.5, 2.0, M)
    sw = np.array([2.0, 3.0, 0.25, -1.0])
    from synth import to_bf16_bits
    b = to_bf16_bits(np.arange(4 * N, dtype=np.float64).reshape(4, N) * 0.125)
    y = per_token.gemm_per_token(a, sa, w, sw, b, g)
    exp_of = np.repeat(np.arange(4), g)
    want = K * 1.0 * -0.75 * sa[:, None] * sw[exp_of][:, None] + formats.bf16_decode(b)[exp_of]
    assert np.array_equal(y, want)
    y0 = per_token.gemm_per_token(a, sa, w, sw, None, g)
    assert np.array_equal(y0, np.broadcast_to(K * -0.75 * sa[:, None] * sw[exp_of][:, None], (M, N)))


def check_per_token_brute(seed=13):
    """Per-element Python loops on a ragged grouping: the row's expert comes from the
    running sum of the group sizes."""
    rng = np.random.default_rng(seed)
    E, N, K = 4, 6, 32
    g = np.array([2, 0, 3, 1])
    M = int(g.sum())
    a = _e4m3_codes(rng, (M, K))
    w = _e4m3_codes(rng, (E, N, K))
    sa = rng.uniform(0.1, 2.0, M)
    sw = rng.uniform(0.1, 2.0, E)
    from synth import to_bf16_bits
    b = to_bf16_bits(rng.standard_normal((E, N)))
    y = per_token.gemm_per_token(a, sa, w, sw, b, g)
    A = formats.e4m3_decode(a)
    W = formats.e4m3_decode(w)
    B = formats.bf16_decode(b)
    m = 0
    for e in range(E):
        for _ in range(int(g[e])):
            for n in range(N):
                dot = math.fsum(A[m, k] * W[e, n, k] for k in range(K))
                want = dot * sa[m] * sw[e] + B[e, n]
                assert abs(y[m, n] - want) <= 1e-12 * max(1.0, abs(want)), (m, n, y[m, n], want)
            m += 1


def check_per_token_scale_linearity(seed=14):
    """Scaling one row's activation scale scales that row only; scaling an expert's weight
    scale scales exactly that expert's rows (bias-free)."""
    rng = np.random.default_rng(seed)
    E, N, K = 3, 8, 32
    g = np.array([4, 3, 5])
    M = int(g.sum())
    a = _e4m3_codes(rng, (M, K))
    w = _e4m3_codes(rng, (E, N, K))
    sa = rng.uniform(0.5, 1.5, M)
    sw = rng.uniform(0.5, 1.5, E)
    y = per_token.gemm_per_token(a, sa, w, sw, None, g)
    sa2 = sa.copy()
    sa2[5] *= 4.0
    y2 = per_token.gemm_per_token(a, sa2, w, sw, None, g)
    assert np.allclose(y2[5], 4.0 * y[5], rtol=1e-14)
    assert np.array_equal(np.delete(y2, 5, 0), np.delete(y, 5, 0))
    sw2 = sw.copy()
    sw2[1] *= -2.0
    y3 = per_token.gemm_per_token(a, sa, w, sw2, None, g)
    rows1 = np.arange(4, 7)
    assert np.allclose(y3[rows1], -2.0 * y[rows1], rtol=1e-14)
    others = np.setdiff1d(np.arange(M), rows1)
    assert np.array_equal(y3[others], y[others])


# ----------------------------------------------------------------------------- MX quantiser

def check_e4m3_encode_vs_torch(seed=15):
    """Round-to-nearest-even E4M3 codes of in-range float32 values, including every exact
    midpoint between neighbouring codes, against torch's float8_e4m3fn conversion."""
    rng = np.random.default_rng(seed)
    mags = formats.e4m3_decode(np.arange(0x7F))
    mids = (mags[:-1] + mags[1:]) / 2
    v = np.concatenate([rng.uniform(-448, 448, 4000), rng.standard_normal(4000) * 2.0 ** rng.integers(-12, 6, 4000),
                        mids, -mids, mags, -mags]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mx_quant.e4m3_encode(v), want)


def check_e4m3_encode_saturates_and_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    assert np.array_equal(mx_quant.e4m3_encode(formats.e4m3_decode(codes)), codes.astype(np.uint8))
    big = np.array([448.0, 460.0, 464.0, 1e6, np.inf, -500.0, -np.inf])
    assert list(mx_quant.e4m3_encode(big)) == [0x7E] * 5 + [0xFE] * 2
    assert mx_quant.e4m3_encode(np.array([np.nan]))[0] == 0x7F


def check_mx_quantize_scale_rule(seed=16):
    """The block exponent is the smallest e with amax < 2^(e + 9) (an integer search, not a
    logarithm); fixed cases: amax 1 -> byte 119, 448 * 2^k -> 127 + k with the codes of 448,
    an all-zero block -> byte 0 and zero codes, a NaN block -> 0xFF and 0x7F codes."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((64, 96)) * 2.0 ** rng.integers(-30, 30, (64, 1))
    x[3, 32:64] = 0.0
    codes, scales = mx_quant.mx_quantize(x)
    amax = np.abs(x.reshape(64, 3, 32)).max(-1)
    for r in range(64):
        for b in range(3):
            if amax[r, b] == 0:
                assert scales[r, b] == 0 and not codes[r, 32 * b:32 * b + 32].any()
                continue
            e = -200
            while not amax[r, b] < 2.0 ** (e + 9):
                e += 1
            assert scales[r, b] == e + 127, (r, b)
    c1, s1 = mx_quant.mx_quantize(np.full((1, 32), 1.0))
    assert s1[0, 0] == 119 and (c1 == 0x78).all()          # 1.0 / 2^-8 = 256 = E4M3 0x78
    for k in (-5, 0, 7):
        ck, sk = mx_quant.mx_quantize(np.full((1, 32), 448.0 * 2.0 ** k))
        assert sk[0, 0] == 127 + k and (ck == 0x7E).all()
    xn = np.ones((1, 64))
    xn[0, 40] = np.nan
    cn, sn = mx_quant.mx_quantize(xn)
    assert sn[0, 1] == 0xFF and (cn[0, 32:] == 0x7F).all() and sn[0, 0] == 119


def check_mx_quantize_error_bound(seed=17):
    """Dequantised values are within half an E4M3 step (2^-4 relative) of the input for
    every element at least 2^-6 of its block's maximum (E4M3 normals under the scale) and
    at most 448 after scaling; above 448 (the block maximum can scale to 448..512) the
    element saturates to the code of 448."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((32, 128)) * np.exp(rng.uniform(-3, 3, (32, 128)))
    c, s = mx_quant.mx_quantize(x)
    d = formats.dequant_mxfp8(c, s)
    blk_max = np.repeat(np.abs(x.reshape(32, 4, 32)).max(-1), 32, axis=-1)
    scaled = np.abs(x) / np.repeat(formats.e8m0_decode(s), 32, axis=-1)
    sat = scaled > 448
    m = (np.abs(x) >= blk_max * 2.0 ** -6) & ~sat
    assert sat.any() and m.sum() > 0.5 * x.size
    assert np.all(np.abs(d - x)[m] <= np.abs(x)[m] * 2.0 ** -4 * (1 + 1e-12))
    assert np.all((c[sat] & 0x7F) == 0x7E)


def check_layer_mxfp8_constant_closed_form():
    """Constant E4M3 codes and scales: h = silu(g) * g is the same for every feature, so its
    block maximum is itself and it quantises to the code nearest h / 2^e; the output follows
    in closed form from that code."""
    T, K, I, E = 3, 64, 64, 2
    x = np.full((T, K), 0x38, np.uint8)                 # 1.0
    xs = np.full((T, K // 32), 127 - 4, np.uint8)        # x = 2^-4
    w1 = np.full((E, 2 * I, K), 0x30, np.uint8)         # 0.5
    w1s = np.full((E, 2 * I, K // 32), 127 - 2, np.uint8)
    w2 = np.full((E, K, I), 0xB8, np.uint8)             # -1.0
    w2s = np.full((E, K, I // 32), 127 - 3, np.uint8)
    W = layer.ExpertWeights("mxfp8", w1, w1s, None, w2, w2s, None)
    ids = np.array([[0, 1], [1, 0], [0, 1]], dtype=np.int32)
    wt = np.array([[0.75, 0.25], [0.5, 0.5], [1.0, 0.0]], dtype=np.float32)
    y = layer.moe_layer(formats.dequant_mxfp8(x, xs), ids, wt, W)
    g = K * 2.0 ** -4 * 0.5 * 2.0 ** -2                   # 0.5
    h = g / (1.0 + math.exp(-g)) * g
    e = math.frexp(h)[1] - 1 - 8
    hq = formats.e4m3_decode(mx_quant.e4m3_encode(np.array([h * 2.0 ** -e])))[0] * 2.0 ** e
    assert hq != h                                     # the quantisation step is visible
    o = I * hq * -1.0 * 2.0 ** -3
    for t in range(T):
        assert np.allclose(y[t], float(wt[t].astype(np.float64).sum()) * o, rtol=1e-14, atol=0)



def check_layer_mxfp8_brute_rows(seed=23):
    """Distinct features within and across 32-blocks: the MXFP8 layer against a brute force
    written pair by pair -- E4M3 codes decoded through torch's float8_e4m3fn cast, E8M0 as
    2^(byte - 127), every dot product a math.fsum, silu with math.exp, and each pair's h
    row quantised on its own, block by block (scale 2^(floor(log2 amax) - 8), codes by
    torch's E4M3 cast of the saturated quotient) -- so that quantising h along the wrong
    axis, with the wrong block grouping or with scales in the wrong block order changes
    the result."""
    rng = np.random.default_rng(seed)
    T, K, I, E, k = 5, 64, 96, 3, 2

    def draw(shape, lo, hi):
        v = np.clip(rng.standard_normal(shape) * 64.0, -448, 448).astype(np.float32)
        codes = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
        return codes, (127 + rng.integers(lo, hi + 1, shape[:-1] + (shape[-1] // 32,))).astype(np.uint8)

    x, xs = draw((T, K), -7, -5)
    w1, w1s = draw((E, 2 * I, K), -11, -8)
    w2, w2s = draw((E, K, I), -12, -9)
    b1 = rng.standard_normal((E, 2 * I)) * 0.1
    b2 = rng.standard_normal((E, K)) * 0.1
    b1 = torch.from_numpy(b1).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    b2 = torch.from_numpy(b2).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2], [2, 1]], dtype=np.int32)
    wt = np.array([[0.7, 0.3], [0.5, 0.5], [0.9, 0.1], [0.25, 0.75], [0.6, 0.4]], dtype=np.float32)

    def dec(codes, scales):
        c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        return c * np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32, axis=-1)

    def bf(b):
        return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()

    xd = dec(x, xs)
    want = np.zeros((T, K))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            W1, W2 = dec(w1[e], w1s[e]), dec(w2[e], w2s[e])
            gu = [math.fsum(xd[t, kk] * W1[n, kk] for kk in range(K)) + bf(b1[e])[n] for n in range(2 * I)]
            h = np.array([gu[f] / (1.0 + math.exp(-gu[f])) * gu[I + f] for f in range(I)])
            hd = np.empty(I)
            for b0 in range(0, I, 32):      # OCP rule, one block at a time, E4M3 by torch's cast
                blk = h[b0:b0 + 32]
                ex = math.frexp(float(np.abs(blk).max()))[1] - 1 - 8
                q = np.clip(blk * 2.0 ** -ex, -448.0, 448.0)
                hd[b0:b0 + 32] = torch.from_numpy(q).to(torch.float8_e4m3fn).to(torch.float64).numpy() * 2.0 ** ex
            o = [math.fsum(hd[f] * W2[c, f] for f in range(I)) + bf(b2[e])[c] for c in range(K)]
            want[t] += float(wt[t, j]) * np.array(o)
    W = layer.ExpertWeights("mxfp8", w1, w1s, b1, w2, w2s, b2)
    got = layer.moe_layer(formats.dequant_mxfp8(x, xs), ids, wt, W)
    # h itself must vary within and across blocks, or the check proves nothing
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())

ALL_CHECKS = [
    check_e2m1_table, check_e8m0_vs_torch, check_e4m3_vs_torch, check_bf16_vs_torch,
    check_mxfp4_dequant_layout, check_bucket_count_20000, check_pad_restriction,
    check_route_brute, check_align_golden, check_align_brute, check_align_invariants,
    check_layer_dense_formulation, check_layer_single_expert_mlp,
    check_layer_constant_closed_form, check_layer_bias_only,
    check_layer_relu2_dense_formulation, check_layer_relu2_single_expert_loops,
    check_layer_relu2_closed_form, check_layer_empty_expert_no_effect, check_grouped_gemm_brute,
    check_wgrad_closed_forms, check_per_token_constant_closed_form, check_per_token_brute,
    check_per_token_scale_linearity, check_e4m3_encode_vs_torch,
    check_e4m3_encode_saturates_and_round_trips, check_mx_quantize_scale_rule,
    check_mx_quantize_error_bound, check_layer_mxfp8_constant_closed_form,
    check_layer_mxfp8_brute_rows,
]
