"""moe_forward (GEMM1 + bias + SwiGLU -> GEMM2 + bias * routing weight -> combine) on the
GPU against the float64 oracle; padded vs unpadded real rows bit-identical."""
import numpy as np
import pytest

import synth
from oracle import bucket as obucket
from oracle import layer as olayer
from oracle import formats as ofmt
from oracle import route as oroute

from helpers import assert_close_bf16, bf16_to_np, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_grouped_align_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load()
    return m


def device_layer(moe, lay, w, max_rows, pad):
    from mixture_experts_grouped_align_gb300.runner import DeviceLayer
    return DeviceLayer(w.quant, w.E, w.K, w.I, w.k, dev(lay["w1"]), dev(lay["w1_scale"]),
                       dev(lay["b1"]), dev(lay["w2"]), dev(lay["w2_scale"]), dev(lay["b2"]),
                       max_rows=max_rows, pad=pad, activation=w.activation)


def run(moe, L, lay, T):
    x = dev(lay["x"][:T])
    lg = dev(lay["logits"][:T])
    y = torch.empty((max(T, 1), L.K), dtype=torch.bfloat16, device="cuda")
    L.status.zero_()
    rows = L.step(x, lg, T, y)
    torch.cuda.synchronize()
    assert int(L.status[0]) == 0
    return y[:T], rows


def oracle_y(lay, w, T, tokens=None):
    W = olayer.ExpertWeights(w.quant, lay["w1"], lay["w1_scale"], lay["b1"], lay["w2"],
                             lay["w2_scale"], lay["b2"], activation=w.activation)
    x = ofmt.bf16_decode(lay["x"][:T])
    ids, wt = oroute.route(lay["logits"][:T], w.k)
    return olayer.moe_layer(x, ids, wt, W, tokens)


@pytest.mark.parametrize("bias", [False, True])
def test_tiny_layer_full(moe, bias):
    w = synth.scaled(synth.TINY, bias=bias)
    lay = synth.make_layer(w)
    L = device_layer(moe, lay, w, w.T, pad=True)
    y, rows = run(moe, L, lay, w.T)
    assert rows == obucket.bucket(w.T)
    assert_close_bf16(bf16_to_np(y), oracle_y(lay, w, w.T), what="tiny")


def test_decode_mxfp4_full(moe):
    w = synth.DECODE_MXFP4
    lay = synth.make_layer(w)
    L = device_layer(moe, lay, w, w.T, pad=True)
    y, _ = run(moe, L, lay, w.T)
    assert_close_bf16(bf16_to_np(y), oracle_y(lay, w, w.T), what="decode_mxfp4")


@pytest.mark.parametrize("M", synth.DECODE_BF16_M)
def test_decode_bf16_tiny_m(moe, M):
    w = synth.decode_bf16_workload(M)
    lay = synth.make_layer(w)
    L = device_layer(moe, lay, w, M, pad=True)
    y, rows = run(moe, L, lay, M)
    assert rows == M  # bf16 mode: padding not allowed
    assert_close_bf16(bf16_to_np(y), oracle_y(lay, w, M), what=f"decode_bf16 M={M}")


@pytest.mark.parametrize("T", [1, 17, 250, 256, 257, 300, 1001])
def test_padded_equals_unpadded_and_oracle(moe, T):
    """Several tiles and a ragged tail; bucket-padded and unpadded runs give the same bits
    on every real row."""
    w = synth.Workload("ragged", T=T, K=256, I=256, E=16, k=4, quant="mxfp4", seed=11,
                       scale_exp=(-6, -2), bias=True)
    lay = synth.make_layer(w)
    Lp = device_layer(moe, lay, w, T, pad=True)
    Lu = device_layer(moe, lay, w, T, pad=False)
    yp, rows_p = run(moe, Lp, lay, T)
    yu, rows_u = run(moe, Lu, lay, T)
    assert rows_p == obucket.bucket(T) and rows_u == T
    assert torch.equal(yp.view(torch.int16), yu.view(torch.int16))
    assert_close_bf16(bf16_to_np(yp), oracle_y(lay, w, T), what=f"ragged T={T}")


@pytest.mark.parametrize("T,E,k", [(256, 4, 2), (250, 2, 1), (200, 8, 8)])
def test_few_experts_fill_whole_blocks_on_the_decode_path(moe, T, E, k):
    """Up to 256 rows with few experts: alignment blocks of up to 128 pairs (eight token
    groups, both accumulator halves) on the few-tokens kernels; padded = unpadded bit for
    bit, and the oracle."""
    w = synth.Workload("dense_blocks", T=T, K=320, I=256, E=E, k=k, quant="mxfp4", seed=17,
                       scale_exp=(-6, -2), bias=True)
    lay = synth.make_layer(w)
    Lp = device_layer(moe, lay, w, T, pad=True)
    Lu = device_layer(moe, lay, w, T, pad=False)
    yp, _ = run(moe, Lp, lay, T)
    yu, _ = run(moe, Lu, lay, T)
    assert torch.equal(yp.view(torch.int16), yu.view(torch.int16))
    assert_close_bf16(bf16_to_np(yp), oracle_y(lay, w, T), what=f"dense blocks T={T} E={E}")


@pytest.mark.parametrize("T", [300, 1001])
def test_bf16_layer_above_256_rows(moe, T):
    """bf16 weights above 256 rows (no padding in this mode): both GEMMs on the tcgen05
    kernel with bf16 operands (I and K multiples of 128), h in bf16."""
    w = synth.Workload("bf16_prefill", T=T, K=512, I=384, E=16, k=4, quant="bf16", seed=21, bias=True)
    lay = synth.make_layer(w)
    L = device_layer(moe, lay, w, T, pad=False)
    y, rows = run(moe, L, lay, T)
    assert rows == T
    assert_close_bf16(bf16_to_np(y), oracle_y(lay, w, T), what=f"bf16 layer T={T}")


def test_prefill_full_size_padded_vs_unpadded_and_sampled_oracle(moe):
    w = synth.prefill_workload()
    lay = synth.make_layer(w)
    T = w.T
    Lp = device_layer(moe, lay, w, T, pad=True)
    yp, rows = run(moe, Lp, lay, T)
    assert rows == obucket.bucket(T) and rows > T
    del Lp
    Lu = device_layer(moe, lay, w, T, pad=False)
    yu, _ = run(moe, Lu, lay, T)
    del Lu
    assert torch.equal(yp.view(torch.int16), yu.view(torch.int16))
    # sampled rows: tokens whose k experts all lie in a 12-expert subset (so that the
    # oracle decodes only those experts), plus the first and last tokens' own experts
    ids, _ = oroute.route(lay["logits"], w.k)
    rng = np.random.default_rng(0)
    subset = rng.choice(w.E, 12, replace=False)
    inside = np.flatnonzero(np.isin(ids, subset).all(axis=1))
    toks = np.concatenate([inside[:24], [0, T - 1]])
    yo = oracle_y(lay, w, T, tokens=toks)
    assert_close_bf16(bf16_to_np(yp)[toks], yo, what="prefill sampled rows")


def test_both_variants_agree_across_the_threshold(moe):
    """Rows 256 run the weight-streaming kernels, 257 the tensor-memory kernels: the first
    256 tokens agree within the floating-point bar (bit-identity is only promised within
    one variant)."""
    w = synth.Workload("threshold", T=257, K=256, I=256, E=16, k=4, quant="mxfp4", seed=12,
                       scale_exp=(-6, -2), bias=True)
    lay = synth.make_layer(w)
    L = device_layer(moe, lay, w, 257, pad=False)
    y257, _ = run(moe, L, lay, 257)
    y256, _ = run(moe, L, lay, 256)
    a, b = bf16_to_np(y257)[:256], bf16_to_np(y256)
    assert_close_bf16(a, oracle_y(lay, w, 256), what="tensor-memory path")
    assert_close_bf16(b, oracle_y(lay, w, 256), what="weight-streaming path")


def _run_status(moe, L, lay, T):
    x = dev(lay["x"][:T])
    lg = dev(lay["logits"][:T])
    y = torch.empty((T, L.K), dtype=torch.bfloat16, device="cuda")
    L.status.zero_()
    L.step(x, lg, T, y)
    torch.cuda.synchronize()
    return y, int(L.status[0])


@pytest.mark.parametrize("T", [64, 300])  # weight-streaming / tensor-memory path
def test_w4a16_nan_scale_reaches_exactly_its_tokens(moe, T):
    """An E8M0 0xFF (NaN) scale on one W1 block makes h -- and through GEMM2 every output --
    NaN for exactly the tokens routed to that expert (the oracle's decoding), and nothing
    else."""
    w = synth.Workload("nan_scale", T=T, K=256, I=256, E=16, k=4, quant="mxfp4", seed=21,
                       scale_exp=(-6, -2), bias=True)
    lay = synth.make_layer(w)
    lay["w1_scale"] = lay["w1_scale"].copy()
    lay["w1_scale"][3, 5, 2] = 0xFF  # expert 3, gate row 5, K block 2
    L = device_layer(moe, lay, w, T, pad=False)
    y, st = _run_status(moe, L, lay, T)
    assert st == 0
    got = bf16_to_np(y)
    ref = oracle_y(lay, w, T)
    nan_rows = np.isnan(ref).any(axis=1)
    assert nan_rows.any() and not nan_rows.all()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert_close_bf16(got[~nan_rows], ref[~nan_rows], what=f"nan scale T={T}")


@pytest.mark.parametrize("T", [64, 300])  # weight-streaming / tensor-memory path
def test_w4a16_scales_outside_the_f16_window_are_exact(moe, T):
    """Blocks with nonzero codes whose E8M0 scale is far below (2^-30) or above (2^+20) the
    window in which code * scale is an exact f16 (2^-23..2^13): the weight-streaming path
    scales f32 partial sums, the tensor-memory path shifts the row's decoded weights by a
    power of two and undoes it on the accumulator.  Both must succeed and match the oracle,
    whichever side of the 256-row threshold the batch falls on."""
    # no bias: with the up rows' weights scaled down, a bias would dominate up and push
    # h = silu(gate) * up beyond the float16 range of h (a legitimate MOE_ERR_RANGE)
    w = synth.Workload("tiny_scale", T=T, K=256, I=256, E=16, k=4, quant="mxfp4", seed=22,
                       scale_exp=(-6, -2), bias=False)
    lay = synth.make_layer(w)
    lay["w1_scale"] = lay["w1_scale"].copy()
    lay["w1"] = lay["w1"].copy()
    lay["w2_scale"] = lay["w2_scale"].copy()
    I = w.I
    lay["w1_scale"][2, 7, 1] = 127 - 30       # one block of a row far below the window
    lay["w1"][2, 7, 16:32] = 0x77             # nonzero codes in that block
    lay["w1_scale"][5, :I, :] += 20           # expert 5: gate rows above the window and up
    lay["w1_scale"][5, I:, :] -= 20           # rows below it (h = silu(gate) * up stays normal)
    lay["w2_scale"][3, 11, :] += 20           # a GEMM2 row above the window (output column 11)
    lay["w2_scale"][3, 12, 0] = 127 + 20      # one GEMM2 block above the window (column 12)
    L = device_layer(moe, lay, w, T, pad=False)
    y, st = _run_status(moe, L, lay, T)
    assert st == 0
    got, ref = bf16_to_np(y), oracle_y(lay, w, T)
    big = [11, 12]                            # the columns the large GEMM2 scales reach
    rest = np.setdiff1d(np.arange(w.K), big)
    assert_close_bf16(got[:, rest], ref[:, rest], what=f"scales outside the f16 window, T={T}")
    assert_close_bf16(got[:, big], ref[:, big], what=f"large GEMM2 scales, T={T}")


def test_w4a16_scale_spread_beyond_36_octaves_is_reported_on_the_tensor_memory_path(moe):
    """A weight row whose nonzero blocks span more than 36 octaves of scale cannot be put into
    one f16 window by a single shift: the tensor-memory path reports MOE_ERR_RANGE (-6) for
    it; the weight-streaming path stays exact."""
    w = synth.Workload("tiny_spread", T=300, K=256, I=256, E=16, k=4, quant="mxfp4", seed=23,
                       scale_exp=(-6, -2), bias=True)
    lay = synth.make_layer(w)
    lay["w1_scale"] = lay["w1_scale"].copy()
    lay["w1"] = lay["w1"].copy()
    lay["w1_scale"][2, 7, 0] = 127 + 6        # block 0: codes 0.5 * 2^6 (h stays in range)
    lay["w1"][2, 7, :16] = 0x11
    lay["w1_scale"][2, 7, 1] = 127 - 31       # 37 octaves below block 0 of the same row
    lay["w1"][2, 7, 16:32] = 0x77
    L = device_layer(moe, lay, w, 300, pad=False)
    _, st = _run_status(moe, L, lay, 300)
    assert st == -6
    y64, st64 = _run_status(moe, L, lay, 64)
    assert st64 == 0
    assert_close_bf16(bf16_to_np(y64), oracle_y(lay, w, 64), what="weight-streaming exact")


def test_bucket_graphs_replay_equal_eager_padded_steps(moe):
    """One CUDA graph per bucket (prewarm) replays the same bits as the eager padded step on
    every real row, for batches that share a bucket (stale pad rows are re-zeroed) and for
    batches in different buckets, including the largest."""
    w = synth.Workload("graphs", T=1100, K=256, I=256, E=16, k=4, quant="mxfp4", seed=13,
                       scale_exp=(-6, -2), bias=True)
    lay = synth.make_layer(w)
    Lg = device_layer(moe, lay, w, w.T, pad=True)
    Le = device_layer(moe, lay, w, w.T, pad=True)
    got = Lg.prewarm()
    assert got == obucket.bucket_iter(obucket.bucket(w.T))
    assert sorted(Lg.graphs) == got
    for T in [300, 290, 1, 17, 256, 257, 1001, 1100, 300]:
        x = dev(lay["x"][:T])
        lg = dev(lay["logits"][:T])
        Lg.status.zero_()
        yg = Lg.step_bucketed(x, lg, T).clone()
        torch.cuda.synchronize()
        assert int(Lg.status[0]) == 0
        ye, _ = run(moe, Le, lay, T)
        assert torch.equal(yg.view(torch.int16), ye.view(torch.int16)), f"T={T}"
    assert_close_bf16(bf16_to_np(yg), oracle_y(lay, w, 300), what="graph T=300")
    with pytest.raises(ValueError):
        device_layer(moe, lay, w, 64, pad=False).prewarm()


# ---------------------------------------------------------------- non-gated relu^2 layers

@pytest.mark.parametrize("M", [1, 7, 28])
def test_relu2_decode_bf16_nemotron_shape(moe, M):
    """The Nemotron decode shape with its non-gated relu^2 (GEMM1 N = 1856), bf16."""
    w = synth.decode_bf16_relu2_workload(M)
    lay = synth.make_layer(w)
    L = device_layer(moe, lay, w, M, pad=True)
    y, rows = run(moe, L, lay, M)
    assert rows == M
    assert_close_bf16(bf16_to_np(y), oracle_y(lay, w, M), what=f"relu2 bf16 M={M}")


@pytest.mark.parametrize("T,I", [(64, 512), (200, 320), (300, 320), (1001, 384)])
def test_relu2_w4a16_padded_equals_unpadded_and_oracle(moe, T, I):
    """W4A16 relu^2 on both variants (64 rows: weight streaming; 300 and 1001: tensor
    memory with slot-ordered h), feature counts that leave a partial and an empty 128-feature
    box in the last tile; padded and unpadded runs give the same bits on every real row."""
    w = synth.Workload("relu2", T=T, K=256, I=I, E=16, k=4, quant="mxfp4", seed=14,
                       scale_exp=(-6, -2), bias=True, activation="relu2")
    lay = synth.make_layer(w)
    Lp = device_layer(moe, lay, w, T, pad=True)
    Lu = device_layer(moe, lay, w, T, pad=False)
    yp, _ = run(moe, Lp, lay, T)
    yu, _ = run(moe, Lu, lay, T)
    assert torch.equal(yp.view(torch.int16), yu.view(torch.int16))
    assert_close_bf16(bf16_to_np(yp), oracle_y(lay, w, T), what=f"relu2 w4a16 T={T}")


def test_relu2_w4a16_long_k(moe):
    """K = 4160 (65 stages of 64, an odd count of four-stage code groups: the last group is
    one stage) through the tensor-memory kernel with the relu^2 epilogue."""
    w = synth.Workload("relu2_longk", T=300, K=4160, I=256, E=4, k=2, quant="mxfp4", seed=15,
                       scale_exp=(-7, -4), bias=True, activation="relu2")
    lay = synth.make_layer(w)
    L = device_layer(moe, lay, w, w.T, pad=False)
    y, _ = run(moe, L, lay, w.T)
    assert_close_bf16(bf16_to_np(y), oracle_y(lay, w, w.T), what="relu2 K=4160")


def test_relu2_graph_replay_equals_eager(moe):
    w = synth.Workload("relu2_graph", T=300, K=256, I=320, E=16, k=4, quant="mxfp4", seed=16,
                       scale_exp=(-6, -2), bias=True, activation="relu2")
    lay = synth.make_layer(w)
    Lg = device_layer(moe, lay, w, w.T, pad=True)
    Le = device_layer(moe, lay, w, w.T, pad=True)
    Lg.prewarm()
    for T in (300, 40):
        Lg.status.zero_()
        yg = Lg.step_bucketed(dev(lay["x"][:T]), dev(lay["logits"][:T]), T).clone()
        torch.cuda.synchronize()
        assert int(Lg.status[0]) == 0
        ye, _ = run(moe, Le, lay, T)
        assert torch.equal(yg.view(torch.int16), ye.view(torch.int16)), f"T={T}"


@pytest.mark.parametrize("block_m", [8, 32, 64, 256])
def test_mxfp4_small_batch_across_block_sizes(moe, block_m):
    """Up to 256 rows the MXFP4 SwiGLU layer runs the block-scaled kernels for alignment blocks
    of at most 128 slots (4- or 8-slot token tiles: one or several per block) and the
    weight-streaming kernels above; each matches the oracle, and padded and unpadded rows
    stay bit-identical."""
    from mixture_experts_grouped_align_gb300.runner import DeviceLayer
    w = synth.Workload("block_sizes", T=61, K=512, I=384, E=8, k=3, quant="mxfp4", seed=31,
                       scale_exp=(-5, -1), bias=True)
    lay = synth.make_layer(w)

    def layer(pad):
        return DeviceLayer(w.quant, w.E, w.K, w.I, w.k, dev(lay["w1"]), dev(lay["w1_scale"]),
                           dev(lay["b1"]), dev(lay["w2"]), dev(lay["w2_scale"]), dev(lay["b2"]),
                           max_rows=w.T, pad=pad, block_m=block_m)

    y_pad, rows = run(moe, layer(True), lay, w.T)
    y_raw, _ = run(moe, layer(False), lay, w.T)
    assert rows == obucket.bucket(w.T)
    assert torch.equal(y_pad.view(torch.int16), y_raw.view(torch.int16))
    assert_close_bf16(bf16_to_np(y_raw), oracle_y(lay, w, w.T), what=f"block_m={block_m}")


@pytest.mark.parametrize("T,E,k,block_m", [(40, 32, 2, 16), (40, 8, 4, 32)])  # 4- / 8-slot tiles
def test_decode_digit_planes_carry_large_and_wide_range_activations(moe, T, E, k, block_m):
    """The block-scaled decode path carries x as E2M1 digit planes under one scale per 32
    elements, so it takes activations far above the f16 range (here up to ~2^19, the
    weights' scales lowered by 2^-17 to match), blocks whose elements lie 2^10 and 2^30
    below the block's first one, an all-zero block and a block of magnitude ~2^-123 (below
    the planes' scale floor): no range error, and the oracle's result within the bar."""
    from mixture_experts_grouped_align_gb300.runner import DeviceLayer
    w = synth.Workload("digit_planes", T=T, K=512, I=256, E=E, k=k, quant="mxfp4", seed=41,
                       scale_exp=(-6, -2), bias=True)
    lay = synth.make_layer(w)
    rng = np.random.default_rng(41)
    xf = rng.standard_normal((T, w.K)).astype(np.float32) * np.float32(2.0 ** 17)
    blocks = xf.reshape(T, w.K // 32, 32)
    blocks[:, 1, 1:] *= np.float32(2.0 ** -10)
    blocks[:, 2, 1:] *= np.float32(2.0 ** -30)
    blocks[:, 3, :] = 0.0
    blocks[:, 4, :] *= np.float32(2.0 ** -140)
    lay["x"] = synth.to_bf16_bits(xf)
    assert np.abs(ofmt.bf16_decode(lay["x"])).max() > 65504
    lay["w1_scale"] = (lay["w1_scale"].astype(np.int32) - 17).astype(np.uint8)
    L = DeviceLayer(w.quant, w.E, w.K, w.I, w.k, dev(lay["w1"]), dev(lay["w1_scale"]), dev(lay["b1"]),
                    dev(lay["w2"]), dev(lay["w2_scale"]), dev(lay["b2"]), max_rows=T, pad=False,
                    block_m=block_m)
    y, _ = run(moe, L, lay, T)
    assert_close_bf16(bf16_to_np(y), oracle_y(lay, w, T), what=f"digit planes E={E} k={k}")
