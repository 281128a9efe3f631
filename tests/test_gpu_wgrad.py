"""moe_wgrad on the GPU against the float64 oracle (deterministic and accumulate modes).

Two bars: the relative Frobenius error of the whole dW, and a per-element bound -- every
element within ELEM of the absolute mass sum_p |grad[p, n] * input[src(p), c]| of its own
sum.  Products of bf16 values are exact in float32, so only the float32 accumulation
rounds: its typical error is about 2^-24 of that mass, and a dropped or doubled pair, a
wrong source row or a wrong expert moves an element by a whole term."""
import numpy as np
import pytest

import synth
from oracle import formats as ofmt
from oracle import wgrad as owgrad

from helpers import dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
BM = 128
REL = 1e-5  # float32 accumulation of exact bf16 products
ELEM = 1e-5  # per element, relative to the element's absolute mass


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


def wgrad_dev(moe, grad, inp, per_pair, ids, E, N, Kin, mode, bm=BM, fill=np.nan, slot=False):
    """slot=True gives the call moe_wgrad_workspace_size() bytes of workspace (NaN-filled), so
    that the tensor-core kernel reads slot-ordered copies by TMA (the test asserts it applies)."""
    T, k = ids.shape
    srt, eid, ntpp, cap = align_dev(moe, ids, E, bm)
    dW = torch.full((E, N, Kin), fill, dtype=torch.float32, device="cuda")
    ctx = None
    if slot:
        need = moe.moe_wgrad_workspace_size(E, N, Kin, bm, cap, mode)
        assert need > 0
        ws = torch.full((need // 2,), float("nan"), dtype=torch.bfloat16, device="cuda")
        ctx = moe.Ctx(workspace=ws)
    moe.moe_wgrad(grad, inp, per_pair, T, k, E, N, Kin, srt, eid, ntpp, bm, cap, dW, mode, ctx)
    torch.cuda.synchronize()
    return dW


def rel_err(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def check_wgrad(got, grad, inp, ids, E, per_pair, experts=None, what=""):
    """got [len(experts), N, Kin] against oracle.wgrad on the same (decoded) operands: the
    Frobenius bar and the per-element bar (the mass is the oracle applied to |grad|, |input|)."""
    ref = owgrad.moe_wgrad(grad, inp, ids, E, per_pair, experts)
    mass = owgrad.moe_wgrad(np.abs(grad), np.abs(inp), ids, E, per_pair, experts)
    assert rel_err(got, ref) <= REL, what
    excess = np.abs(got - ref) - ELEM * mass
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (what, worst, got[worst], ref[worst], mass[worst])
    return ref


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("per_pair", [False, True])
@pytest.mark.parametrize("bm", [128, 16])
def test_wgrad_small(moe, mode, per_pair, bm):
    rng = np.random.default_rng(7)
    T, E, k, N, Kin = 150, 6, 2, 128, 192
    ids = np.stack([rng.choice(E - 1, k, replace=False) for _ in range(T)]).astype(np.int32)  # E-1 empty
    g = synth.to_bf16_bits(rng.standard_normal((T * k, N)))
    x = synth.to_bf16_bits(rng.standard_normal((T * k if per_pair else T, Kin)))
    dW = wgrad_dev(moe, dev(g), dev(x), per_pair, ids, E, N, Kin, mode, bm=bm).cpu().numpy()
    check_wgrad(dW, ofmt.bf16_decode(g), ofmt.bf16_decode(x), ids, E, per_pair, what=f"mode {mode}")
    assert np.all(dW[E - 1] == 0)                   # empty expert written as zeros


@pytest.mark.parametrize("per_pair", [False, True])
@pytest.mark.parametrize("bm", [128, 64])
@pytest.mark.parametrize("N,Kin", [(128, 192), (256, 448), (384, 256), (512, 320), (1024, 768)])
def test_wgrad_slot_feed(moe, per_pair, bm, N, Kin):
    """The slot-ordered feed (workspace given): against the oracle, and bit-identical to the
    gather feed on the same inputs (the same MMAs over the same stages in the same order).
    The N tiles (1, 2, 3, 4, 8) run without clusters, in pairs and in fours; Kin = 192, 448,
    320 and 768 take 192-, 64-, 64- and 256-column tiles (one input box, which one CTA of a
    cluster loads for all four, up to four boxes, one per CTA); N <= Kin and N > Kin walk
    the tiles of an expert in the two orders."""
    rng = np.random.default_rng(17)
    T, E, k = 333, 7, 3
    ids = np.stack([rng.choice(E - 1, k, replace=False) for _ in range(T)]).astype(np.int32)  # E-1 empty
    g = synth.to_bf16_bits(rng.standard_normal((T * k, N)))
    x = synth.to_bf16_bits(rng.standard_normal((T * k if per_pair else T, Kin)))
    a = wgrad_dev(moe, dev(g), dev(x), per_pair, ids, E, N, Kin, 0, bm=bm, slot=True)
    b = wgrad_dev(moe, dev(g), dev(x), per_pair, ids, E, N, Kin, 0, bm=bm)
    assert torch.equal(a, b)
    dW = a.cpu().numpy()
    check_wgrad(dW, ofmt.bf16_decode(g), ofmt.bf16_decode(x), ids, E, per_pair, what="slot feed")
    assert np.all(dW[E - 1] == 0)


@pytest.mark.parametrize("N,Kin", [(64, 64), (128, 320)])   # mma.sync path / tcgen05 path
def test_wgrad_deterministic_repeatable_and_constant(moe, N, Kin):
    rng = np.random.default_rng(8)
    T, E, k = 500, 8, 2
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    g = dev(synth.to_bf16_bits(rng.standard_normal((T * k, N))))
    x = dev(synth.to_bf16_bits(rng.standard_normal((T, Kin))))
    a = wgrad_dev(moe, g, x, False, ids, E, N, Kin, 0)
    b = wgrad_dev(moe, g, x, False, ids, E, N, Kin, 0)
    assert torch.equal(a, b)
    # analytic constant-input check: grad = 0.5, input = -3 -> dW[e] = n_e * -1.5
    gc = torch.full((T * k, N), 0.5, dtype=torch.bfloat16, device="cuda")
    xc = torch.full((T, Kin), -3.0, dtype=torch.bfloat16, device="cuda")
    c = wgrad_dev(moe, gc, xc, False, ids, E, N, Kin, 0).cpu().numpy()
    cnt = np.bincount(ids.reshape(-1), minlength=E)
    for e in range(E):
        assert np.all(c[e] == cnt[e] * -1.5)


@pytest.mark.parametrize("N", [64, 128])
def test_wgrad_sentinel_rows_never_read(moe, N):
    """NaN rows directly after grad and input: sentinel slots must not touch them."""
    rng = np.random.default_rng(9)
    T, E, k, Kin = 40, 5, 2, 128
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    g = torch.full((T * k + 64, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    x = torch.full((T + 64, Kin), float("nan"), dtype=torch.bfloat16, device="cuda")
    gv = synth.to_bf16_bits(rng.standard_normal((T * k, N)))
    xv = synth.to_bf16_bits(rng.standard_normal((T, Kin)))
    g[:T * k] = dev(gv)
    x[:T] = dev(xv)
    for mode in (0, 1):
        dW = wgrad_dev(moe, g, x, False, ids, E, N, Kin, mode).cpu().numpy()
        assert np.all(np.isfinite(dW))
        check_wgrad(dW, ofmt.bf16_decode(gv), ofmt.bf16_decode(xv), ids, E, False, what=f"mode {mode}")


def test_wgrad_full_size_sampled(moe):
    """dW1 [256, 4096, 7168] and dW2 [256, 7168, 2048] of the MXFP8 training workload: a
    sample of rows and columns of three experts (the hottest, a cold one and a random one)
    against oracle.wgrad on the same sampled columns of grad and input; cold experts are
    exactly zero."""
    g = synth.make_mxfp8_gemm_wgrad(device="cuda")
    T, E, K, I, k = g["T"], g["E"], g["K"], g["I"], g["k"]
    ids = g["topk_ids"]
    flat = ids.reshape(-1)
    cnt = np.bincount(flat, minlength=E)
    rng = np.random.default_rng(2)
    experts = [int(np.argmax(cnt)), int(g["cold"][0]), int(rng.choice(np.flatnonzero(cnt)))]

    def host_bf16(t):
        return ofmt.bf16_decode(t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16))

    for (grad, inp, per_pair, N, Kin) in [(g["grad1"], g["x_bf16"], False, 2 * I, K),
                                          (g["grad2"], g["h_bf16"], True, K, I)]:
        rows = np.sort(rng.choice(N, 8, replace=False))
        cols = np.sort(rng.choice(Kin, 64, replace=False))
        gs = host_bf16(grad[:, torch.from_numpy(rows).cuda()])      # [P, 8]
        xs = host_bf16(inp[:, torch.from_numpy(cols).cuda()])       # [T or P, 64]
        for mode, slot in ((0, False), (0, True), (1, False)):
            dW = wgrad_dev(moe, grad, inp, per_pair, ids, E, N, Kin, mode, slot=slot)
            got = np.stack([dW[e][torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()
                            for e in experts])
            assert np.all(got[1] == 0) and cnt[experts[1]] == 0
            check_wgrad(got, gs, xs, ids, E, per_pair, experts, what=f"N={N} mode {mode} slot {slot}")
            del dW
            torch.cuda.empty_cache()
