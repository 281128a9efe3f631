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
    x, lg = dev(lay["x"][:T]), dev(lay["logits"][:T])
    cap, _ = moe.moe_align_capacity(T * L.k, L.E, L.block_m)
    ctx = L.ctx()
    moe.moe_align(lg, L.topk_ids, L.topk_w, T, L.k, L.E, L.block_m, L.sorted, cap,
                  L.expert_ids, L.ntpp, L.expert_offsets, ctx)
    args = (L.quant, L.E, L.K, L.I, L.w1, L.w1_scale, L.b1, L.w2, L.w2_scale, L.b2, x, None, T,
            T, L.k, L.topk_w, L.sorted, L.expert_ids, L.ntpp, L.expert_offsets, L.block_m, cap)
    y_ws = torch.full((T, L.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_na = torch.full((T, L.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(*args, y_ws, ctx)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    moe.moe_forward_no_alloc(*args, y_na, moe.Ctx(dev_status=status))
    torch.cuda.synchronize()
    assert int(status[0]) == 0 and int(L.status[0]) == 0
    return y_ws, y_na


def test_no_alloc_matches_workspace_forward_on_two_calls(moe):
    w = synth.DECODE_MXFP4          # T=64, hidden 2880, intermediate 2880, 128 experts, top-4
    for shift, T in ((0, 64), (7, 37)):   # second call: other inputs, fewer tokens
        lay, L = _layer(moe, w, shift)
        y_ws, y_na = _both(moe, L, lay, T)
        a, b = bf16_to_np(y_na), bf16_to_np(y_ws)
        assert_close_bf16(a, b, what=f"no-alloc vs workspace (T={T})")
        assert torch.equal(y_na.view(torch.int16), y_ws.view(torch.int16))


def test_no_alloc_bf16_layer(moe):
    w = synth.decode_bf16_workload(28)
    lay, L = _layer(moe, w, 0)
    y_ws, y_na = _both(moe, L, lay, 28)
    assert_close_bf16(bf16_to_np(y_na), bf16_to_np(y_ws), what="no-alloc bf16")


def test_no_alloc_rejects_calls_beyond_the_array(moe):
    # 4096 rows of a 2880/2880 top-4 layer need far more than the fixed array
    need = moe.moe_forward_workspace_size(4096, 4, 2880, 2880, moe.moe_align_capacity(4096 * 4, 128, 128)[0])
    assert need > (8 << 20)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_no_alloc("mxfp4", 128, 2880, 2880, 16, 16, None, 16, 16, None, 16, None,
                                 4096, 4096, 4, 16, 16, 16, 16, None, 128, 1 << 20, 16,
                                 moe.Ctx(stream=0))
    assert ei.value.status == -3
    assert "scratch" in moe.load().moe_last_error().decode()
