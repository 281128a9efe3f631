"""moe_gemm_per_token on the GPU against the float64 oracle: ragged and empty expert
groups, both N tiles, the constant-input round trip, and group sizes that do not fit."""
import numpy as np
import pytest

import synth
from oracle import per_token as opt

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


def e4m3_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    return np.where((c & 0x7F) == 0x7F, c - 1, c).astype(np.uint8)


def run(moe, a, sa, w, sw, b, g, M, expect_status=0):
    E, N, K = w.shape
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    moe.moe_gemm_per_token(E, N, K, dev(a), dev(sa.astype(np.float32)), dev(w), dev(sw.astype(np.float32)),
                           None if b is None else dev(b), dev(np.asarray(g, dtype=np.int32)), M, out,
                           moe.Ctx(dev_status=st))
    torch.cuda.synchronize()
    assert int(st[0]) == expect_status
    return bf16_to_np(out)


@pytest.mark.parametrize("N,K,bias", [(256, 256, True), (128, 512, False), (384, 128, True)])
def test_ragged_groups(moe, N, K, bias):
    """Groups of 0, 1, 127, 128, 129, 300 and 50 rows (several tiles and ragged tails), with
    rows past the groups' sum left untouched."""
    rng = np.random.default_rng(N + K)
    g = np.array([0, 1, 127, 128, 129, 300, 0, 50])
    E, M = g.size, int(g.sum()) + 40
    a = e4m3_codes(rng, (M, K))
    w = e4m3_codes(rng, (E, N, K))
    sa = rng.uniform(2.0 ** -12, 2.0 ** -8, M)
    sw = rng.uniform(2.0 ** -10, 2.0 ** -6, E)
    b = synth.to_bf16_bits(rng.standard_normal((E, N))) if bias else None
    got = run(moe, a, sa.astype(np.float32), w, sw.astype(np.float32), b, g, M)
    used = int(g.sum())
    ref = opt.gemm_per_token(a, sa.astype(np.float32), w, sw.astype(np.float32), b, g)
    assert_close_bf16(got[:used], ref, what=f"per-token N={N} K={K}")
    assert np.isnan(got[used:]).all()


def test_constant_round_trip(moe):
    """The page's constant-input round trip: E4M3 1.0 x -0.75 over K gives K * -0.75 times
    the row's and the expert's scales, plus the bias."""
    K, N = 256, 128
    g = np.array([130, 0, 7, 128])
    E, M = g.size, int(g.sum())
    a = np.full((M, K), 0x38, np.uint8)
    w = np.full((E, N, K), 0xB4, np.uint8)
    sa = ((np.arange(M) % 7) + 1).astype(np.float32) * np.float32(2.0 ** -6)
    sw = np.array([0.5, 3.0, 0.25, -2.0], dtype=np.float32)
    b = synth.to_bf16_bits(np.tile(np.arange(N) * 0.5, (E, 1)))
    got = run(moe, a, sa, w, sw, b, g, M)
    ref = opt.gemm_per_token(a, sa, w, sw, b, g)
    assert_close_bf16(got, ref, what="constant round trip")


def test_group_sizes_past_m_are_reported(moe):
    rng = np.random.default_rng(5)
    K, N, M = 128, 128, 200
    g = np.array([150, 100])  # 250 rows claimed, 200 present
    a = e4m3_codes(rng, (M, K))
    w = e4m3_codes(rng, (2, N, K))
    sa = np.full(M, 2.0 ** -8, np.float32)
    sw = np.full(2, 2.0 ** -8, np.float32)
    got = run(moe, a, sa, w, sw, None, g, M, expect_status=-3)
    ref = opt.gemm_per_token(a, sa, w, sw, None, np.array([150, 50]))  # the rows that exist
    assert_close_bf16(got, ref, what="clamped groups")


def test_full_size_sampled(moe):
    """256 experts, N = 4096, K = 7168 (the DSv4-like GEMM1 shape of the MXFP8 workload),
    Zipf group sizes over 65,536 rows with cold experts; sampled rows against the oracle."""
    rng = np.random.default_rng(9)
    E, N, K = 256, 4096, 7168
    T, k = 8192, 8
    ids, _ = synth.zipf_topk_ids(rng, T, E, k)
    g = np.bincount(ids.reshape(-1), minlength=E)
    assert (g == 0).any()
    M = int(g.sum())
    a_t = torch.randint(0, 126, (M, K), dtype=torch.uint8, device="cuda")  # finite E4M3 codes
    w_t = torch.randint(0, 126, (E, N, K), dtype=torch.uint8, device="cuda")
    sa = rng.uniform(2.0 ** -10, 2.0 ** -8, M).astype(np.float32)
    sw = rng.uniform(2.0 ** -10, 2.0 ** -8, E).astype(np.float32)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    moe.moe_gemm_per_token(E, N, K, a_t, dev(sa), w_t, dev(sw), None, dev(g.astype(np.int32)), M, out,
                           moe.Ctx(dev_status=st))
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    off = np.concatenate([[0], np.cumsum(g)])
    experts = [e for e in rng.permutation(E) if g[e] > 0][:3]
    rows = np.concatenate([off[e] + rng.choice(g[e], min(4, g[e]), replace=False) for e in experts])
    a_np = a_t.cpu().numpy()
    w_np = {e: w_t[e].cpu().numpy() for e in experts}
    for m in rows:
        e = int(np.searchsorted(off, m, side="right") - 1)
        want = opt.gemm_per_token(a_np[m:m + 1], sa[m:m + 1], w_np[e][None], sw[e:e + 1], None, np.array([1]))
        assert_close_bf16(bf16_to_np(out[m:m + 1]), want, what=f"row {m} expert {e}")
