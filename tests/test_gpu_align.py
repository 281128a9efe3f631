"""Routing + alignment on the GPU against the oracle: bit-exact ids, sorted_token_ids,
expert_ids (with -1 sentinel blocks), num_tokens_post_padded and expert_offsets, and
bit-exact routing weights: both sides round the same float64 softmax (the same summation
order) to float32, so the weights are held to identical bits."""
import numpy as np
import pytest

import synth
from oracle import align as oalign
from oracle import route as oroute

from helpers import ulp_diff_f32

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


def gpu_align(moe, T, k, E, bm, logits=None, ids=None):
    P = T * k
    cap, capb = moe.moe_align_capacity(P, E, bm)
    d = "cuda"
    lg = torch.from_numpy(logits).to(d) if logits is not None else None
    tid = (torch.from_numpy(ids.astype(np.int32)).to(d) if ids is not None and T > 0
           else torch.empty((max(T, 1), k), dtype=torch.int32, device=d))
    tw = torch.empty((max(T, 1), k), dtype=torch.float32, device=d)
    srt = torch.full((cap + 16,), -7, dtype=torch.int32, device=d)
    eid = torch.full((capb + 16,), -7, dtype=torch.int32, device=d)
    ntpp = torch.full((4,), -7, dtype=torch.int32, device=d)
    eoff = torch.full((E + 1 + 8,), -7, dtype=torch.int32, device=d)
    status = torch.zeros(4, dtype=torch.int32, device=d)
    moe.moe_align(lg, tid, tw if lg is not None else None, T, k, E, bm, srt, cap, eid, ntpp, eoff,
                  moe.Ctx(dev_status=status))
    torch.cuda.synchronize()
    return {"ids": tid.cpu().numpy()[:T], "w": tw.cpu().numpy()[:T],
            "sorted": srt.cpu().numpy()[:cap], "eid": eid.cpu().numpy()[:capb],
            "ntpp": int(ntpp[0]), "eoff": eoff.cpu().numpy()[:E + 1], "status": int(status[0]),
            "srt_full": srt.cpu().numpy(), "eid_full": eid.cpu().numpy()}


def check_against_oracle(r, ids, E, bm):
    o = oalign.moe_align(ids, E, bm)
    assert np.array_equal(r["sorted"], o["sorted_token_ids"])
    assert np.array_equal(r["eid"], o["expert_ids"])
    assert r["ntpp"] == int(o["num_tokens_post_padded"])
    assert np.array_equal(r["eoff"], o["expert_offsets"])


def route_case(moe, T, E, k, bm, seed):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if T > 2:
        logits[1] = 0.0                       # full tie -> experts 0..k-1, weight 1/k
        logits[2, ::2] = logits[2, 1]         # partial ties
    r = gpu_align(moe, T, k, E, bm, logits=logits)
    ids, w = oroute.route(logits, k)
    assert np.array_equal(r["ids"], ids)
    ud = ulp_diff_f32(r["w"], w)
    bad = np.argwhere(ud > 0)
    assert bad.size == 0, (f"{bad.shape[0]} routing weights differ from the oracle; first at (t, j) = "
                           f"{tuple(bad[0])}: logits row {logits[bad[0][0]].tolist()}")
    check_against_oracle(r, ids, E, bm)
    assert r["status"] == 0
    return r


@pytest.mark.parametrize("T,E,k,bm", [
    (64, 8, 2, 128),        # tiny layer
    (64, 128, 4, 128),      # decode MXFP4 layer
    (1, 128, 6, 128), (7, 128, 6, 128), (14, 128, 6, 128), (21, 128, 6, 128), (28, 128, 6, 128),
    (600, 64, 8, 16),       # routed by the separate routing kernel (T > 512)
    (37, 1024, 32, 64),     # the limits: E = 1024, k = 32 (8-way float64 sum path)
    (5, 3, 3, 1),           # block_m = 1, k = E
    (1, 1, 1, 1),
])
def test_route_align_matches_oracle(moe, T, E, k, bm):
    route_case(moe, T, E, k, bm, seed=T * 1000 + E)


def test_prefill_size_route_align(moe):
    w = synth.prefill_workload()
    Tp = moe.moe_bucket(w.T)
    lay = synth.make_layer(w, T=w.T, with_logits=True)
    logits = np.zeros((Tp, w.E), dtype=np.float32)
    logits[:w.T] = lay["logits"]
    r = gpu_align(moe, Tp, w.k, w.E, 128, logits=logits)
    ids, wt = oroute.route(logits, w.k)
    assert np.array_equal(r["ids"], ids)
    assert ulp_diff_f32(r["w"], wt).max() == 0
    check_against_oracle(r, ids, w.E, 128)
    # pad rows (zero logits) route to experts 0..k-1 with weight 1/k
    assert np.all(r["ids"][w.T:] == np.arange(w.k))
    assert np.all(r["w"][w.T:] == np.float32(1.0 / w.k))


def test_given_ids_zipf_with_cold_experts(moe):
    g = synth.make_mxfp8_gemm_wgrad(T=8192, E=256, K=64, I=64)
    ids, cold = g["topk_ids"], g["cold"]
    r = gpu_align(moe, 8192, 8, 256, 128, ids=ids)
    check_against_oracle(r, ids, 256, 128)
    cnt = np.diff(r["eoff"])
    assert np.all(cnt[cold] == 0) and cold.size > 0
    assert not np.isin(cold, r["eid"]).any()


def test_empty_batch(moe):
    r = gpu_align(moe, 0, 4, 16, 128, ids=np.zeros((0, 4), dtype=np.int32))
    assert r["ntpp"] == 0
    assert np.all(r["eoff"] == 0)
    assert np.all(r["eid"] == -1)
    assert np.all(r["sorted"] == 0)


def test_invalid_expert_id_sets_status(moe):
    ids = np.array([[0, 1], [2, 9], [3, 1]], dtype=np.int32)   # 9 is out of range for E = 4
    r = gpu_align(moe, 3, 2, 4, 4, ids=ids)
    assert r["status"] == -5
    # the valid pairs are still aligned; the bad one is left out
    real = r["sorted"][r["sorted"] < 6]
    assert sorted(real.tolist()) == [0, 1, 2, 4, 5]


def test_capacity_tail_untouched_beyond_cap(moe):
    r = gpu_align(moe, 10, 2, 4, 4, ids=np.tile(np.array([[0, 1]], dtype=np.int32), (10, 1)))
    cap, capb = moe.moe_align_capacity(20, 4, 4)
    assert np.all(r["srt_full"][cap:] == -7)
    assert np.all(r["eid_full"][capb:] == -7)


@pytest.mark.parametrize("T,E,k,bm", [
    (4097, 8, 4, 128),      # 16388 pairs: just past the single-block size, a ragged last range
    (3000, 1024, 32, 64),   # E = 1024, k = 32: the largest shared-memory histograms
    (20000, 64, 2, 16),     # small blocks: many block ids, long sentinel tail
    (65536, 3, 1, 1),       # block_m = 1, a few hot experts
])
def test_multi_block_alignment(moe, T, E, k, bm):
    """Above 16384 pairs the alignment runs on a grid of blocks; its output is the same
    definition: bit-exact against the oracle over the whole capacity, beyond which nothing is
    written."""
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) if E > 64 else \
        rng.integers(0, E, size=(T, k)).astype(np.int32)
    if E > 4:
        ids[rng.random(T) < 0.3] = np.sort(rng.choice(max(E // 4, k), k, replace=False))  # skew to low ids
    r = gpu_align(moe, T, k, E, bm, ids=ids)
    check_against_oracle(r, ids, E, bm)
    assert r["status"] == 0
    cap, capb = moe.moe_align_capacity(T * k, E, bm)
    assert np.all(r["srt_full"][cap:] == -7)
    assert np.all(r["eid_full"][capb:] == -7)


def test_multi_block_invalid_expert_id(moe):
    T, E, k = 9000, 16, 2
    rng = np.random.default_rng(5)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[4321, 1] = E + 3
    ids[8999, 0] = -2
    r = gpu_align(moe, T, k, E, 128, ids=ids)
    assert r["status"] == -5
    keep = np.ones(T * k, dtype=bool)
    keep[[4321 * k + 1, 8999 * k]] = False
    real = r["sorted"][r["sorted"] < T * k]
    assert np.array_equal(np.sort(real), np.flatnonzero(keep))
