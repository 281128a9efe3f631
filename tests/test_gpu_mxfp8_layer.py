"""The MXFP8 layer (moe_forward with E4M3 operands and h quantised to MXFP8 between the
GEMMs) and the standalone quantiser on the GPU, against the float64 oracle."""
import numpy as np
import pytest

import synth
from oracle import formats as ofmt
from oracle import layer as olayer
from oracle import mx_quant as omx
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


def quant_inputs(seed=0):
    """float32 rows that exercise the rule: a wide range of block maxima, zero, NaN, inf,
    subnormal and saturating blocks, signed zeros and exact E4M3 midpoints."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((257, 96)) * 2.0 ** rng.integers(-40, 40, (257, 1))).astype(np.float32)
    x[0, :32] = 0.0
    x[0, 32:64] = -0.0
    x[1, 5] = np.nan
    x[2, 40] = np.inf
    x[3, :32] = np.float32(1e-40) * np.arange(1, 33)         # float32 subnormals
    mags = ofmt.e4m3_decode(np.arange(0x7F))
    mids = ((mags[:-1] + mags[1:]) / 2)[-32:]
    x[4, :32] = mids                                          # ties at the top of the range
    x[4, 32:64] = -mids * 2.0 ** -12
    x[5, :32] = 300.0
    x[5, 0] = 500.0                                           # maximum 500: the block saturates
    return x


def test_quantiser_bit_exact(moe):
    x = quant_inputs()
    rows, cols = x.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device="cuda")
    moe.moe_mx_quantize(dev(x), rows, cols, codes, scales)
    torch.cuda.synchronize()
    want_c, want_s = omx.mx_quantize(x.astype(np.float64))
    assert np.array_equal(scales.cpu().numpy(), want_s)
    assert np.array_equal(codes.cpu().numpy(), want_c)


def layer(moe, w, lay, T):
    from mixture_experts_grouped_align_gb300.runner import DeviceLayer
    L = DeviceLayer(w.quant, w.E, w.K, w.I, w.k, dev(lay["w1"]), dev(lay["w1_scale"]), dev(lay["b1"]),
                    dev(lay["w2"]), dev(lay["w2_scale"]), dev(lay["b2"]), max_rows=T, pad=True)
    y = torch.empty((T, w.K), dtype=torch.bfloat16, device="cuda")
    L.status.zero_()
    rows = L.step(dev(lay["x_codes"][:T]), dev(lay["logits"][:T]), T, y, x_scale=dev(lay["x_scale"][:T]))
    torch.cuda.synchronize()
    assert rows == T                       # MXFP8: no token-dimension padding
    assert int(L.status[0]) == 0
    return bf16_to_np(y)


def oracle_layer(w, lay, T):
    W = olayer.ExpertWeights("mxfp8", lay["w1"], lay["w1_scale"], lay["b1"], lay["w2"], lay["w2_scale"], lay["b2"])
    x = ofmt.dequant_mxfp8(lay["x_codes"][:T], lay["x_scale"][:T])
    ids, wt = oroute.route(lay["logits"][:T], w.k)
    return olayer.moe_layer(x, ids, wt, W)


@pytest.mark.parametrize("T,bias,K,I", [(64, True, 384, 256), (200, False, 384, 256), (300, True, 384, 256),
                                        (700, False, 384, 256), (600, True, 1024, 512)])
def test_mxfp8_layer(moe, T, bias, K, I):
    """Up to 256 rows the weight-streaming kernels with fp32 h and the standalone quantiser;
    above, the block-scaled kernel with the quantiser in its epilogue (K and I multiples of
    512: scale words four stages at a time)."""
    w = synth.Workload("mxfp8_layer", T=T, K=K, I=I, E=8, k=4, quant="mxfp8", seed=31,
                       weight_std=0.05, bias=bias)
    lay = synth.make_layer(w)
    assert_close_bf16(layer(moe, w, lay, T), oracle_layer(w, lay, T), what=f"mxfp8 layer T={T}")


def test_mxfp8_layer_paths_agree(moe):
    w = synth.Workload("mxfp8_layer", T=257, K=256, I=256, E=8, k=2, quant="mxfp8", seed=32,
                       weight_std=0.05, bias=True)
    lay = synth.make_layer(w)
    y257 = layer(moe, w, lay, 257)[:256]
    y256 = layer(moe, w, lay, 256)
    ref = oracle_layer(w, lay, 256)
    assert_close_bf16(y257, ref, what="block-scaled path")
    assert_close_bf16(y256, ref, what="weight-streaming path")


class _DeviceRows:
    """Rows of a device tensor brought to the host on indexing (codes, or codes decoded
    with their scales), so that the oracle reads only the rows it needs."""

    def __init__(self, codes, scales=None):
        self.codes, self.scales = codes, scales
        self.shape = tuple(codes.shape)

    def __getitem__(self, idx):
        i = torch.as_tensor(np.asarray(idx), device=self.codes.device)
        c = self.codes[i].cpu().numpy()
        return c if self.scales is None else ofmt.dequant_mxfp8(c, self.scales[i].cpu().numpy())


def test_mxfp8_layer_full_size_sampled(moe):
    """The whole MXFP8 layer at the size of the MXFP8 workload -- 256 experts, hidden 7168,
    intermediate 2048, top-8, T = 8192, Zipf(1.1) routing with cold experts, operands drawn
    on the device -- through moe_forward (block-scaled kernels, SwiGLU and the MXFP8
    quantiser fused in GEMM1's epilogue, the routing-weighted GEMM2, the combine).  Eight
    tokens routed to the hottest experts are checked against the oracle layer."""
    g = synth.make_mxfp8_gemm_wgrad(device="cuda")
    T, E, K, I, k, P = g["T"], g["E"], g["K"], g["I"], g["k"], g["P"]
    for n in ("grad1", "grad2", "x_bf16", "h_bf16", "a2_codes", "a2_scale"):
        g.pop(n)
    torch.cuda.empty_cache()
    ids = g["topk_ids"]
    rng = np.random.default_rng(5)
    wt = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    wt /= wt.sum(axis=1, keepdims=True)
    bm = 128
    cap, capb = moe.moe_align_capacity(P, E, bm)
    srt = torch.empty(cap, dtype=torch.int32, device="cuda")
    eid = torch.empty(capb, dtype=torch.int32, device="cuda")
    ntpp = torch.empty(4, dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    moe.moe_align(None, dev(ids), None, T, k, E, bm, srt, cap, eid, ntpp, None, moe.Ctx(dev_status=status))
    ws = torch.empty(moe.moe_forward_workspace_size(T, k, K, I, cap), dtype=torch.uint8, device="cuda")
    y = torch.full((T, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward("mxfp8", E, K, I, g["w1"], g["w1_scale"], None, g["w2"], g["w2_scale"], None,
                    g["x_codes"], g["x_scale"], T, T, k, dev(wt), srt, eid, ntpp, None, bm, cap, y,
                    moe.Ctx(workspace=ws, dev_status=status))
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    assert bool(torch.isfinite(y.float()).all())
    cnt = np.bincount(ids.reshape(-1), minlength=E)
    hot = cnt[ids].sum(axis=1)                       # tokens whose experts are the busiest
    tokens = np.sort(np.argsort(-hot, kind="stable")[:8])
    W = olayer.ExpertWeights("mxfp8", _DeviceRows(g["w1"]), _DeviceRows(g["w1_scale"]), None,
                             _DeviceRows(g["w2"]), _DeviceRows(g["w2_scale"]), None)
    ref = olayer.moe_layer(_DeviceRows(g["x_codes"], g["x_scale"]), ids, wt, W, tokens=tokens)
    got = bf16_to_np(y[torch.from_numpy(tokens).cuda()])
    assert_close_bf16(got, ref, what="MXFP8 layer, full size")
