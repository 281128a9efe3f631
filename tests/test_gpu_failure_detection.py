"""Failure detection of the tensor-memory kernels, without a GPU fault: with the stall
self-test switch on, the W4A16 and MXFP8 forward GEMMs above 256 rows and the deterministic
weight gradient (both feeds, the slot feed in clusters of four CTAs) launch with their copy
and MMA roles off, so their other roles wait on barriers nothing arrives on.  Every wait is
bounded: the kernels must give up after the short limit, report MOE_ERR_TIMEOUT in the
device status word and return, and the next normal call on the same context must succeed
and match the float64 oracle."""
import time

import numpy as np
import pytest

import synth
from oracle import formats, layer, route
from oracle import wgrad as owgrad

from helpers import assert_close_bf16, bf16_to_np, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
MOE_ERR_TIMEOUT = -7


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_grouped_align_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load()
    yield m
    m.moe_debug_stall_tensor_kernels(0)


def _layer(w):
    from mixture_experts_grouped_align_gb300.runner import DeviceLayer
    lay = synth.make_layer(w)
    L = DeviceLayer(w.quant, w.E, w.K, w.I, w.k, dev(lay["w1"]), dev(lay["w1_scale"]), dev(lay["b1"]),
                    dev(lay["w2"]), dev(lay["w2_scale"]), dev(lay["b2"]), max_rows=w.T)
    return lay, L


def _step(L, lay, w):
    y = torch.full((w.T, w.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    if w.quant == "mxfp8":
        L.step(dev(lay["x_codes"]), dev(lay["logits"]), w.T, y, x_scale=dev(lay["x_scale"]))
    else:
        L.step(dev(lay["x"]), dev(lay["logits"]), w.T, y)
    torch.cuda.synchronize()
    return y


def _oracle(lay, w):
    W = layer.ExpertWeights(w.quant, lay["w1"], lay["w1_scale"], lay["b1"], lay["w2"], lay["w2_scale"], lay["b2"])
    ids, wt = route.route(lay["logits"], w.k)
    x = formats.dequant_mxfp8(lay["x_codes"], lay["x_scale"]) if w.quant == "mxfp8" else formats.bf16_decode(lay["x"])
    return layer.moe_layer(x, ids, wt, W)


@pytest.mark.parametrize("quant", ["mxfp4", "mxfp4_decode", "mxfp8"])
def test_stalled_waits_time_out_and_the_context_recovers(moe, quant):
    if quant == "mxfp4":   # prefill_ts kernels (W4A16, decoded weights in tensor memory)
        w = synth.scaled(synth.TINY, T=300, bias=True)
    elif quant == "mxfp4_decode":  # decode_tc kernels (64 rows: E2M1 codes on the block-scaled MMA)
        w = synth.scaled(synth.TINY, T=64, bias=True)
    else:                  # mx8_gemm kernels (block-scaled MXFP8)
        w = synth.Workload("stall_mxfp8", T=300, K=512, I=512, E=8, k=2, quant="mxfp8", seed=7,
                           weight_std=0.05, bias=True)
    lay, L = _layer(w)
    _step(L, lay, w)                              # module loaded, kernels set up
    L.status.zero_()
    try:
        moe.moe_debug_stall_tensor_kernels(5_000)   # 5 us limit on every wait
        t0 = time.perf_counter()
        _step(L, lay, w)
        elapsed = time.perf_counter() - t0
    finally:
        moe.moe_debug_stall_tensor_kernels(0)
    assert int(L.status[0]) == MOE_ERR_TIMEOUT
    assert elapsed < 1.0, elapsed                 # gave up after the short limit, not 2 s
    # the context is still usable: a normal call succeeds and is correct
    L.status.zero_()
    y = _step(L, lay, w)
    assert int(L.status[0]) == 0
    assert_close_bf16(bf16_to_np(y), _oracle(lay, w), what=f"{quant} after the stalled call")


@pytest.mark.parametrize("slot", [False, True])
def test_wgrad_stalled_waits_time_out_and_recover(moe, slot):
    """N = 512 is four N tiles: with the slot feed the kernel runs in clusters of four."""
    rng = np.random.default_rng(21)
    T, E, k, N, Kin, bm = 300, 8, 2, 512, 256, 128
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    g = synth.to_bf16_bits(rng.standard_normal((T * k, N)))
    x = synth.to_bf16_bits(rng.standard_normal((T, Kin)))
    cap, capb = moe.moe_align_capacity(T * k, E, bm)
    srt = torch.empty(cap, dtype=torch.int32, device="cuda")
    eid = torch.empty(capb, dtype=torch.int32, device="cuda")
    ntpp = torch.empty(4, dtype=torch.int32, device="cuda")
    moe.moe_align(None, dev(ids), None, T, k, E, bm, srt, cap, eid, ntpp, None)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    ws = None
    if slot:
        ws = torch.empty(moe.moe_wgrad_workspace_size(E, N, Kin, bm, cap, 0), dtype=torch.uint8, device="cuda")
    ctx = moe.Ctx(dev_status=status, workspace=ws)
    dW = torch.empty((E, N, Kin), dtype=torch.float32, device="cuda")
    gd, xd = dev(g), dev(x)

    def call():
        moe.moe_wgrad(gd, xd, 0, T, k, E, N, Kin, srt, eid, ntpp, bm, cap, dW, 0, ctx)
        torch.cuda.synchronize()

    call()
    status.zero_()
    try:
        moe.moe_debug_stall_tensor_kernels(5_000)   # 5 us limit on every wait
        t0 = time.perf_counter()
        call()
        elapsed = time.perf_counter() - t0
    finally:
        moe.moe_debug_stall_tensor_kernels(0)
    assert int(status[0]) == MOE_ERR_TIMEOUT
    assert elapsed < 1.0, elapsed
    status.zero_()
    dW.fill_(float("nan"))
    call()
    assert int(status[0]) == 0
    ref = owgrad.moe_wgrad(formats.bf16_decode(g), formats.bf16_decode(x), ids, E, False)
    got = dW.cpu().numpy()
    assert np.linalg.norm(got - ref) <= 1e-5 * np.linalg.norm(ref)
