"""Out-of-range reads on the forward path: every input buffer is followed by guard rows
that hold NaN (bf16 0xFFFF, E4M3 0x7F, E8M0 0xFF), a whole extra expert of NaN weights
sits after the last real one, and the workspace starts filled with NaN bytes.  A kernel
that reads past a tensor, reads an expert id it should have skipped (the -1 sentinel
blocks, second review of "Add MoE GEMM variants and weight-gradient kernel", aiter PR
5310), or reads scratch it did not write first, turns some output into NaN.  Every output
must stay finite and match the float64 oracle, on both kernel families of each format."""
import numpy as np
import pytest

import synth
from oracle import formats as ofmt
from oracle import layer as olayer
from oracle import route as oroute

from helpers import assert_close_bf16, bf16_to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
GUARD = 64  # guard rows after each buffer


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_grouped_align_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load()
    return m


def guarded(a, fill, extra_leading=0):
    """numpy array -> device tensor with the same bytes, followed by GUARD rows (and, for
    weights, `extra_leading` whole extra entries of the first axis) of the fill byte pattern;
    returns the full tensor and a view of the real part."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    shape = list(t.shape)
    if extra_leading:
        shape[0] += extra_leading
    else:
        shape[0] += GUARD
    full = torch.empty(shape, dtype=t.dtype, device="cuda")
    full.view(torch.uint8).fill_(fill)
    full[: t.shape[0]] = t.cuda()
    return full, full[: t.shape[0]]


def run_guarded(moe, w, lay, T):
    E, K, I, k = w.E, w.K, w.I, w.k
    mx8 = w.quant == "mxfp8"
    bm = 128
    if mx8:
        _, x = guarded(lay["x_codes"][:T], 0x7F)
        _, xs = guarded(lay["x_scale"][:T], 0xFF)
    else:
        _, x = guarded(lay["x"][:T], 0xFF)
        xs = None
    # weights: one extra expert of NaN scales (and NaN codes for E4M3) after the last
    wfill = 0x7F if mx8 else 0x00
    _, w1 = guarded(lay["w1"], wfill, extra_leading=1)
    _, w2 = guarded(lay["w2"], wfill, extra_leading=1)
    _, w1s = guarded(lay["w1_scale"], 0xFF, extra_leading=1)
    _, w2s = guarded(lay["w2_scale"], 0xFF, extra_leading=1)
    b1 = guarded(lay["b1"], 0xFF, extra_leading=1)[1] if lay["b1"] is not None else None
    b2 = guarded(lay["b2"], 0xFF, extra_leading=1)[1] if lay["b2"] is not None else None
    _, lg = guarded(lay["logits"][:T], 0xFF)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    topk_w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    cap, capb = moe.moe_align_capacity(T * k, E, bm)
    srt = torch.empty(cap, dtype=torch.int32, device="cuda")
    eid = torch.empty(capb, dtype=torch.int32, device="cuda")
    ntpp = torch.empty(4, dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    ctx_a = moe.Ctx(dev_status=status)
    moe.moe_align(lg, ids, topk_w, T, k, E, bm, srt, cap, eid, ntpp, None, ctx_a)
    ws = torch.full((moe.moe_forward_workspace_size(T, k, K, I, cap) + 4096,), 0xFF, dtype=torch.uint8,
                    device="cuda")
    y = torch.full((T + GUARD, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(w.quant, E, K, I, w1, w1s, b1, w2, w2s, b2, x, xs, T, T, k, topk_w, srt, eid, ntpp, None, bm,
                    cap, y[:T], moe.Ctx(workspace=ws, dev_status=status))
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    got = bf16_to_np(y[:T])
    assert np.all(np.isfinite(got)), "a guard row, the extra expert or stale scratch reached the output"
    assert bool(torch.isnan(y[T:].float()).all()), "rows past T_real were written"
    W = olayer.ExpertWeights(w.quant, lay["w1"], lay["w1_scale"], lay["b1"], lay["w2"], lay["w2_scale"], lay["b2"])
    ids_o, wt_o = oroute.route(lay["logits"][:T], k)
    xo = ofmt.dequant_mxfp8(lay["x_codes"][:T], lay["x_scale"][:T]) if mx8 else ofmt.bf16_decode(lay["x"][:T])
    assert_close_bf16(got, olayer.moe_layer(xo, ids_o, wt_o, W), what=f"{w.quant} T={T} with guard rows")


@pytest.mark.parametrize("T", [37, 300])   # weight-streaming / tensor-memory kernels
def test_mxfp4_forward_reads_nothing_past_its_buffers(moe, T):
    w = synth.Workload("poison_mxfp4", T=T, K=512, I=256, E=12, k=4, quant="mxfp4", seed=51,
                       scale_exp=(-6, -2), bias=True)
    run_guarded(moe, w, synth.make_layer(w), T)


@pytest.mark.parametrize("T", [37, 300])   # weight-streaming + quantiser / block-scaled kernels
def test_mxfp8_forward_reads_nothing_past_its_buffers(moe, T):
    w = synth.Workload("poison_mxfp8", T=T, K=512, I=256, E=12, k=4, quant="mxfp8", seed=52,
                       weight_std=0.05, bias=True)
    run_guarded(moe, w, synth.make_layer(w), T)


def test_bf16_forward_reads_nothing_past_its_buffers(moe):
    w = synth.Workload("poison_bf16", T=21, K=512, I=256, E=12, k=6, quant="bf16", seed=53, bias=True)
    lay = synth.make_layer(w)
    lay["w1_scale"] = np.zeros((w.E, 1), np.uint8)   # unused by bf16 weights; guarded() needs arrays
    lay["w2_scale"] = np.zeros((w.E, 1), np.uint8)
    run_guarded(moe, w, lay, w.T)
