"""moe_grouped_gemm (one launch over all experts, optional per-expert bias) on the GPU
against the float64 oracle, for MXFP8 (block-scaled E4M3 operands), MXFP4 and bf16."""
import numpy as np
import pytest

import synth
from oracle import align as oalign
from oracle import formats as ofmt
from oracle import layer as olayer

from helpers import assert_close_bf16, bf16_to_np, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
BM = 128


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_grouped_align_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load()
    return m


def align_dev(moe, ids, E, bm=BM):
    T, k = ids.shape
    cap, capb = moe.moe_align_capacity(T * k, E, bm)
    d = "cuda"
    tid = torch.from_numpy(ids.astype(np.int32)).to(d)
    srt = torch.empty(cap, dtype=torch.int32, device=d)
    eid = torch.empty(capb, dtype=torch.int32, device=d)
    ntpp = torch.empty(4, dtype=torch.int32, device=d)
    moe.moe_align(None, tid, None, T, k, E, bm, srt, cap, eid, ntpp, None)
    return srt, eid, ntpp, cap


def gemm_dev(moe, quant, E, N, Kin, a, a_scale, per_pair, w, w_scale, bias, ids, bm=BM, workspace=None):
    T, k = ids.shape
    srt, eid, ntpp, cap = align_dev(moe, ids, E, bm)
    out = torch.full((T * k, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm(quant, E, N, Kin, a, a_scale, per_pair, w, w_scale, bias, T, k, srt, eid,
                         ntpp, bm, cap, out, moe.Ctx(dev_status=st, workspace=workspace))
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    return out


def random_ids(rng, T, E, k, empty=()):
    allowed = np.array([e for e in range(E) if e not in set(empty)])
    return np.stack([rng.choice(allowed, k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T", [203, 600])   # weight-streaming path / tensor-memory path
@pytest.mark.parametrize("per_pair", [False, True])
@pytest.mark.parametrize("bias", [False, True])
def test_mxfp8_small(moe, T, per_pair, bias):
    rng = np.random.default_rng(3)
    E, k, N, Kin = 12, 3, 96, 320
    ids = random_ids(rng, T, E, k, empty=(5,))
    rows = T * k if per_pair else T
    a_c, a_s = synth.gen_mx_e4m3(rng, (rows, Kin))
    w_c, w_s = synth.gen_mx_e4m3(rng, (E, N, Kin), synth.scale_exp_for_std(0.05))
    b = synth.to_bf16_bits(rng.standard_normal((E, N)) * 0.1) if bias else None
    out = gemm_dev(moe, "mxfp8", E, N, Kin, dev(a_c), dev(a_s), per_pair, dev(w_c), dev(w_s),
                   dev(b), ids)
    A = ofmt.dequant_mxfp8(a_c, a_s)
    Wd = lambda e: (ofmt.dequant_mxfp8(w_c[e], w_s[e]), None if b is None else ofmt.bf16_decode(b[e]))
    ref = olayer.grouped_gemm(A, ids, Wd, per_pair)
    assert_close_bf16(bf16_to_np(out), ref, what="mxfp8 small")


@pytest.mark.parametrize("T", [77, 700])
@pytest.mark.parametrize("quant", ["mxfp4", "bf16"])
def test_w4a16_and_bf16_small(moe, T, quant):
    rng = np.random.default_rng(4)
    E, k, N, Kin = 9, 2, 64, 256
    ids = random_ids(rng, T, E, k)
    a = synth.to_bf16_bits(rng.standard_normal((T, Kin)))
    if quant == "mxfp4":
        w, ws = synth.gen_mxfp4_weight(rng, E, N, Kin, (-5, 0))
    else:
        w, ws = synth.gen_bf16_weight(rng, E, N, Kin, 0.05), None
    b = synth.to_bf16_bits(rng.standard_normal((E, N)) * 0.1)
    out = gemm_dev(moe, quant, E, N, Kin, dev(a), None, False, dev(w), dev(ws), dev(b), ids)
    Wd = lambda e: (ofmt.dequant(quant, w[e], None if ws is None else ws[e]), ofmt.bf16_decode(b[e]))
    ref = olayer.grouped_gemm(ofmt.bf16_decode(a), ids, Wd, False)
    assert_close_bf16(bf16_to_np(out), ref, what=quant)


@pytest.mark.parametrize("T,per_pair,bias", [(300, False, True), (700, True, False), (257, False, False)])
def test_bf16_above_threshold_tensor_path(moe, T, per_pair, bias):
    """bf16 above 256 rows with N a multiple of 128 and K of 64: the tcgen05 kernel (bf16
    operands, kind::f16, no scale factors), 224- or 256-wide tiles; the oracle on the
    decoded operands."""
    rng = np.random.default_rng(40 + T)
    E, k, N, Kin = 9, 2, 384, 320
    ids = random_ids(rng, T, E, k)
    a = synth.to_bf16_bits(rng.standard_normal((T * k if per_pair else T, Kin)))
    w = synth.gen_bf16_weight(rng, E, N, Kin, 0.05)
    b = synth.to_bf16_bits(rng.standard_normal((E, N)) * 0.1) if bias else None
    out = gemm_dev(moe, "bf16", E, N, Kin, dev(a), None, per_pair, dev(w), None, None if b is None else dev(b), ids)
    Wd = lambda e: (ofmt.bf16_decode(w[e]), None if b is None else ofmt.bf16_decode(b[e]))
    ref = olayer.grouped_gemm(ofmt.bf16_decode(a), ids, Wd, per_pair)
    assert_close_bf16(bf16_to_np(out), ref, what=f"bf16 T={T}")


def test_w4a16_weight_streaming_is_exact_for_any_scale(moe):
    """bf16 activations up to 256 rows run the weight-streaming kernel, which multiplies each
    32-block's f32 partial sum by its scale: a scale of 2^-30 on nonzero codes (outside what
    an f16 weight can hold) still gives the oracle's result."""
    rng = np.random.default_rng(23)
    T, E, k, N, Kin = 64, 9, 2, 64, 256
    ids = random_ids(rng, T, E, k)
    a = synth.to_bf16_bits(rng.standard_normal((T, Kin)))
    w, ws = synth.gen_mxfp4_weight(rng, E, N, Kin, (-5, 0))
    ws[:, :, 1] = 127 - 30
    w[:, :, 16:32] = 0x77
    out = gemm_dev(moe, "mxfp4", E, N, Kin, dev(a), None, False, dev(w), dev(ws), None, ids)
    Wd = lambda e: (ofmt.dequant("mxfp4", w[e], ws[e]), None)
    ref = olayer.grouped_gemm(ofmt.bf16_decode(a), ids, Wd, False)
    assert_close_bf16(bf16_to_np(out), ref, what="mxfp4 scale 2^-30")


def test_mxfp8_constant_roundtrip(moe):
    """Constant codes and scales: every output is Kin * a * w * 2^(sa + sw) exactly."""
    T, E, k, N, Kin = 16, 4, 2, 32, 128
    ids = np.array([[t % E, (t + 1) % E] for t in range(T)], dtype=np.int32)
    a_c = np.full((T, Kin), 0x38, np.uint8)          # E4M3 1.0
    a_s = np.full((T, Kin // 32), 127 - 2, np.uint8)
    w_c = np.full((E, N, Kin), 0xB4, np.uint8)        # E4M3 -0.75
    w_s = np.full((E, N, Kin // 32), 127 + 1, np.uint8)
    out = gemm_dev(moe, "mxfp8", E, N, Kin, dev(a_c), dev(a_s), False, dev(w_c), dev(w_s), None, ids)
    want = Kin * 1.0 * -0.75 * 2.0 ** (-2 + 1)
    assert np.all(bf16_to_np(out) == want)


def test_mxfp8_full_size_sampled(moe):
    """The 256-expert, hidden 7168 / intermediate 2048, top-8, T=8192 grouped GEMMs with Zipf
    routing; operands drawn on the device; sampled pairs of a few experts checked."""
    g = synth.make_mxfp8_gemm_wgrad(device="cuda")
    T, E, K, I, k = g["T"], g["E"], g["K"], g["I"], g["k"]
    ids = g["topk_ids"]
    out1 = gemm_dev(moe, "mxfp8", E, 2 * I, K, g["x_codes"], g["x_scale"], False, g["w1"],
                    g["w1_scale"], None, ids)
    out2 = gemm_dev(moe, "mxfp8", E, K, I, g["a2_codes"], g["a2_scale"], True, g["w2"],
                    g["w2_scale"], None, ids)
    flat = ids.reshape(-1)
    cnt = np.bincount(flat, minlength=E)
    rng = np.random.default_rng(1)
    experts = [int(np.argmax(cnt)), int(np.argsort(cnt)[E // 2])] + \
        [int(e) for e in rng.choice(np.flatnonzero(cnt), 2, replace=False)]
    for e in experts:
        pairs = np.flatnonzero(flat == e)
        pairs = pairs[rng.choice(pairs.size, min(16, pairs.size), replace=False)]
        W1 = ofmt.dequant_mxfp8(g["w1"][e].cpu().numpy(), g["w1_scale"][e].cpu().numpy())
        X = ofmt.dequant_mxfp8(g["x_codes"][pairs // k].cpu().numpy(), g["x_scale"][pairs // k].cpu().numpy())
        assert_close_bf16(bf16_to_np(out1[pairs]), X @ W1.T, what=f"gemm1 expert {e}")
        W2 = ofmt.dequant_mxfp8(g["w2"][e].cpu().numpy(), g["w2_scale"][e].cpu().numpy())
        A2 = ofmt.dequant_mxfp8(g["a2_codes"][pairs].cpu().numpy(), g["a2_scale"][pairs].cpu().numpy())
        assert_close_bf16(bf16_to_np(out2[pairs]), A2 @ W2.T, what=f"gemm2 expert {e}")
    assert np.all(cnt[g["cold"]] == 0)


@pytest.mark.parametrize("N", [256, 384])          # N tile 256 / N tile 128
@pytest.mark.parametrize("per_pair", [False, True])
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("Kin", [384, 1024])        # scale words per stage / per four stages
def test_mxfp8_block_scaled(moe, N, per_pair, bias, Kin):
    """Rows above the threshold, K a multiple of 128 and N of 128: the block-scaled MMA path.
    Ragged experts (two empty) over several 128-row tiles, three or eight K stages (K a
    multiple of 512 takes the scale words four stages at a time)."""
    rng = np.random.default_rng(13)
    T, E, k = 700, 12, 3
    ids = random_ids(rng, T, E, k, empty=(5, 9))
    rows = T * k if per_pair else T
    a_c, a_s = synth.gen_mx_e4m3(rng, (rows, Kin))
    w_c, w_s = synth.gen_mx_e4m3(rng, (E, N, Kin), synth.scale_exp_for_std(0.05))
    b = synth.to_bf16_bits(rng.standard_normal((E, N)) * 0.1) if bias else None
    out = gemm_dev(moe, "mxfp8", E, N, Kin, dev(a_c), dev(a_s), per_pair, dev(w_c), dev(w_s),
                   dev(b), ids)
    A = ofmt.dequant_mxfp8(a_c, a_s)
    Wd = lambda e: (ofmt.dequant_mxfp8(w_c[e], w_s[e]), None if b is None else ofmt.bf16_decode(b[e]))
    ref = olayer.grouped_gemm(A, ids, Wd, per_pair)
    assert_close_bf16(bf16_to_np(out), ref, what=f"mxfp8 block-scaled N={N}")


def test_mxfp8_block_scaled_constant_roundtrip(moe):
    """Constant codes and scales on the block-scaled path: every output is exactly
    Kin * a * w * 2^(sa + sw)."""
    T, E, k, N, Kin = 300, 4, 2, 256, 256
    ids = np.array([[t % E, (t + 1) % E] for t in range(T)], dtype=np.int32)
    a_c = np.full((T, Kin), 0x38, np.uint8)          # E4M3 1.0
    a_s = np.full((T, Kin // 32), 127 - 3, np.uint8)
    w_c = np.full((E, N, Kin), 0xB4, np.uint8)        # E4M3 -0.75
    w_s = np.full((E, N, Kin // 32), 127 + 2, np.uint8)
    out = gemm_dev(moe, "mxfp8", E, N, Kin, dev(a_c), dev(a_s), False, dev(w_c), dev(w_s), None, ids)
    want = Kin * 1.0 * -0.75 * 2.0 ** (-3 + 2)
    assert np.all(bf16_to_np(out) == want)


def test_mxfp8_block_scaled_scale_edges(moe):
    """E8M0 edge codes on the block-scaled path (the edge decoding of the second review on
    the aiter MoE GEMM page): 0x00 is 2^-127 -- here every weight scale of K block 2 is 0x00
    and every activation scale of that block is 2^125, so the block still weighs 2^-2 -- and
    0xFF is NaN, which must reach exactly the outputs whose dot product uses that block."""
    rng = np.random.default_rng(17)
    T, E, k, N, Kin = 300, 4, 2, 128, 256
    ids = random_ids(rng, T, E, k)
    a_c, a_s = synth.gen_mx_e4m3(rng, (T, Kin))
    w_c, w_s = synth.gen_mx_e4m3(rng, (E, N, Kin), synth.scale_exp_for_std(0.05))
    a_s[:, 2] = 127 + 125
    w_s[:, :, 2] = 0x00
    w_s[2, 3:5, 1] = 0xFF
    out = bf16_to_np(gemm_dev(moe, "mxfp8", E, N, Kin, dev(a_c), dev(a_s), False, dev(w_c), dev(w_s),
                              None, ids))
    A = ofmt.dequant_mxfp8(a_c, a_s)
    Wd = lambda e: (ofmt.dequant_mxfp8(w_c[e], w_s[e]), None)
    ref = olayer.grouped_gemm(A, ids, Wd, False)
    nan_ref = np.isnan(ref)
    assert nan_ref.any()
    assert np.array_equal(np.isnan(out), nan_ref)
    keep = ~nan_ref.any(axis=1)
    assert_close_bf16(out[keep], ref[keep], what="mxfp8 scale edges")


@pytest.mark.parametrize("per_pair,outside", [(False, False), (True, False), (False, True)])
def test_mxfp4_above_threshold_tensor_path_with_workspace(moe, per_pair, outside):
    """W4A16 above 256 rows: with moe_grouped_gemm_workspace_size() bytes of workspace the call
    converts A to f16 and runs the tcgen05 kernel (decoded weights in tensor memory); without it
    the weight-streaming kernel runs.  Both against the oracle: ragged experts over several
    128-row blocks, one empty expert, per-expert bias, Kin with a partial last scale group."""
    rng = np.random.default_rng(41)
    T, E, k, N, Kin = 760, 12, 3, 256, 576
    ids = random_ids(rng, T, E, k, empty=(4,))
    rows = T * k if per_pair else T
    a = synth.to_bf16_bits(rng.standard_normal((rows, Kin)))
    w, ws = synth.gen_mxfp4_weight(rng, E, N, Kin, (-6, -2))
    if outside:  # blocks whose scale puts code * scale outside the f16 window: the exact second pass
        ws[3, 5, 1] = 127 - 30
        w[3, 5, 16:32] = 0x77
        ws[7, :, 2] = 127 + 16
        w[7, :, 32:48] = 0x11
    b = synth.to_bf16_bits(rng.standard_normal((E, N)) * 0.1)
    need = moe.moe_grouped_gemm_workspace_size("mxfp4", T, k, N, Kin, per_pair)
    assert need >= rows * Kin * 2
    wsp = torch.empty(need, dtype=torch.uint8, device="cuda")
    Wd = lambda e: (ofmt.dequant("mxfp4", w[e], ws[e]), ofmt.bf16_decode(b[e]))
    ref = olayer.grouped_gemm(ofmt.bf16_decode(a), ids, Wd, per_pair)
    got_tc = gemm_dev(moe, "mxfp4", E, N, Kin, dev(a), None, per_pair, dev(w), dev(ws), dev(b), ids,
                      workspace=wsp)
    got_ws = gemm_dev(moe, "mxfp4", E, N, Kin, dev(a), None, per_pair, dev(w), dev(ws), dev(b), ids)
    if outside:  # expert 7's outputs are large: compare the two groups of pairs separately
        big = np.repeat((ids == 7).reshape(-1), 1)
        for sel, what in ((big, "expert 7"), (~big, "the others")):
            assert_close_bf16(bf16_to_np(got_tc)[sel], ref[sel], what=f"tensor-memory kernel, {what}")
            assert_close_bf16(bf16_to_np(got_ws)[sel], ref[sel], what=f"weight-streaming kernel, {what}")
        return
    assert_close_bf16(bf16_to_np(got_tc), ref, what="mxfp4 grouped GEMM, tensor-memory kernel")
    assert_close_bf16(bf16_to_np(got_ws), ref, what="mxfp4 grouped GEMM, weight-streaming kernel")
