"""moe_forward_no_alloc: the forward for callers that cannot call cudaMalloc (a host
program that owns every device allocation, or a thread that must not enter the CUDA
allocator).  Its scratch is a fixed device array inside the library; these tests check it
through the C ABI against moe_forward with a caller workspace, on two calls in a row.

This file is collected last so that a run stopping at the first failure has already run
every other test."""
import numpy as np
import pytest

import synth

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


def _layer(moe, w, seed_shift):
    from mixture_experts_grouped_align_gb300.runner import DeviceLayer
    lay = synth.make_layer(synth.scaled(w, seed=w.seed + seed_shift))
    L = DeviceLayer(w.quant, w.E, w.K, w.I, w.k, dev(lay["w1"]), dev(lay["w1_scale"]),
                    dev(lay["b1"]), dev(lay["w2"]), dev(lay["w2_scale"]), dev(lay["b2"]),
                    max_rows=w.T, pad=False)
    return lay, L


def _both(moe, L, lay, T):
    """Routes + aligns once, then runs moe_forward (workspace) and moe_forward_no_alloc
    on the same alignment; returns both outputs."""
    if L.quant == "mxfp8":
        x, xs = dev(lay["x_codes"][:T]), dev(lay["x_scale"][:T])
    else:
        x, xs = dev(lay["x"][:T]), None
    lg = dev(lay["logits"][:T])
    cap, _ = moe.moe_align_capacity(T * L.k, L.E, L.block_m)
    ctx = L.ctx()
    moe.moe_align(lg, L.topk_ids, L.topk_w, T, L.k, L.E, L.block_m, L.sorted, cap,
                  L.expert_ids, L.ntpp, L.expert_offsets, ctx)
    args = (L.quant, L.E, L.K, L.I, L.w1, L.w1_scale, L.b1, L.w2, L.w2_scale, L.b2, x, xs, T,
            T, L.k, L.topk_w, L.sorted, L.expert_ids, L.ntpp, L.expert_offsets, L.block_m, cap)
    y_ws = torch.full((T, L.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_na = torch.full((T, L.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(*args, y_ws, ctx)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    moe.moe_forward_no_alloc(*args, y_na, moe.Ctx(dev_status=status))
    torch.cuda.synchronize()
    assert int(status[0]) == 0 and int(L.status[0]) == 0
    return y_ws, y_na


def _oracle(lay, w, T):
    from oracle import formats, layer, route
    W = layer.ExpertWeights(w.quant, lay["w1"], lay["w1_scale"], lay["b1"], lay["w2"], lay["w2_scale"],
                            lay["b2"])
    ids, wt = route.route(lay["logits"][:T], w.k)
    if w.quant == "mxfp8":
        x = formats.dequant_mxfp8(lay["x_codes"][:T], lay["x_scale"][:T])
    else:
        x = formats.bf16_decode(lay["x"][:T])
    return layer.moe_layer(x, ids, wt, W)


def test_no_alloc_matches_workspace_forward_on_two_calls(moe):
    w = synth.DECODE_MXFP4          # T=64, hidden 2880, intermediate 2880, 128 experts, top-4
    for shift, T in ((0, 64), (7, 37)):   # second call: other inputs, fewer tokens
        lay, L = _layer(moe, w, shift)
        y_ws, y_na = _both(moe, L, lay, T)
        a, b = bf16_to_np(y_na), bf16_to_np(y_ws)
        assert_close_bf16(a, b, what=f"no-alloc vs workspace (T={T})")
        assert torch.equal(y_na.view(torch.int16), y_ws.view(torch.int16))


def test_no_alloc_slot_ordered_path_against_oracle(moe):
    # Above 256 rows the W4A16 forward keeps x and h in alignment-slot order and carves the
    # scratch differently (cap_tokens rows of x and h): the tiny layer at 300 and 290 rows,
    # two calls in a row with different inputs, bit-exact against the workspace forward and
    # within the floating-point bar of the float64 oracle.
    for shift, T in ((0, 300), (3, 290)):
        w = synth.scaled(synth.TINY, T=T, bias=True)
        lay, L = _layer(moe, w, shift)
        y_ws, y_na = _both(moe, L, lay, T)
        assert torch.equal(y_na.view(torch.int16), y_ws.view(torch.int16)), f"T={T}"
        assert_close_bf16(bf16_to_np(y_na), _oracle(lay, synth.scaled(w, seed=w.seed + shift), T),
                          what=f"no-alloc vs oracle (T={T})")


@pytest.mark.parametrize("T", [300, 40])
def test_no_alloc_mxfp8_layer(moe, T):
    # The MXFP8 layer puts h codes and scales in the h region (300 rows: block-scaled kernels)
    # or fp32 h in the o region first (40 rows: weight-streaming kernels and the quantiser).
    w = synth.Workload("no_alloc_mxfp8", T=T, K=1024, I=512, E=8, k=2, quant="mxfp8", seed=11,
                       weight_std=0.05, bias=True)
    for shift in (0, 1):
        lay, L = _layer(moe, w, shift)
        y_ws, y_na = _both(moe, L, lay, T)
        assert torch.equal(y_na.view(torch.int16), y_ws.view(torch.int16)), f"T={T} call {shift}"


def test_no_alloc_empty_batch(moe):
    # no token: nothing is launched and the call succeeds, as moe_forward does
    w = synth.DECODE_MXFP4
    lay, L = _layer(moe, w, 0)
    cap, _ = moe.moe_align_capacity(0, L.E, L.block_m)
    y = torch.zeros((1, L.K), dtype=torch.bfloat16, device="cuda")
    args = (L.quant, L.E, L.K, L.I, L.w1, L.w1_scale, L.b1, L.w2, L.w2_scale, L.b2, L.x_pad, None, 0,
            0, L.k, L.topk_w, L.sorted, L.expert_ids, L.ntpp, L.expert_offsets, L.block_m, cap, y)
    assert moe.moe_forward(*args, L.ctx()) == 0
    assert moe.moe_forward_no_alloc(*args, moe.Ctx()) == 0
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(y.view(torch.int16))) == 0


def test_no_alloc_bf16_layer(moe):
    w = synth.decode_bf16_workload(28)
    lay, L = _layer(moe, w, 0)
    y_ws, y_na = _both(moe, L, lay, 28)
    assert_close_bf16(bf16_to_np(y_na), bf16_to_np(y_ws), what="no-alloc bf16")


def test_no_alloc_rejects_calls_beyond_the_array(moe):
    # 4096 rows of a 2880/2880 top-4 layer need far more than the fixed array
    need = moe.moe_forward_workspace_size(4096, 4, 2880, 2880, moe.moe_align_capacity(4096 * 4, 128, 128)[0])
    assert need > (16 << 20)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_no_alloc("mxfp4", 128, 2880, 2880, 16, 16, None, 16, 16, None, 16, None,
                                 4096, 4096, 4, 16, 16, 16, 16, None, 128, 1 << 20, 16,
                                 moe.Ctx(stream=0))
    assert ei.value.status == -3
    assert "scratch" in moe.load().moe_last_error().decode()
