"""The activation carrier of the decode MXFP4 kernels, as a statement about numbers: a block
of 32 bf16 or f16 values written as eight base-4 digit planes, each plane an E2M1 code per
element under one E8M0 scale, sums back to every element no more than 2^8 (bf16) or 2^5
(f16) below the block's largest exactly, and to the others within 2^-16 of the largest; a
block with an infinity or NaN takes the NaN scale.  The decomposition is written out here
from its definition (round |v| to an integer X in units of 2^(emax-15), digit p of X in base
4 under scale 2^(emax-2p), emax floored at -113) and checked in exact float64 arithmetic;
the kernels' results against the oracle are the GPU tests' business."""
import math

import numpy as np
import pytest

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def planes(block):
    """-> (codes [8, 32] E2M1 codes, scale bytes [8]) of a block of 32 finite floats."""
    mx = float(np.max(np.abs(block)))
    emax = math.floor(math.log2(mx)) if mx > 0 else -127
    emax = max(emax, -113)
    X = np.rint(np.abs(block) * 2.0 ** (15 - emax)).astype(np.int64)  # float64: exact scaling
    assert X.max() < 2 ** 16
    codes = np.zeros((8, 32), np.int64)
    for p in range(8):
        d = (X >> (14 - 2 * p)) & 3
        codes[p] = np.where(d > 0, d | (np.signbit(block) * 8), 0)
    return codes, np.array([emax + 127 - 2 * p for p in range(8)])


def decode(codes, sbytes):
    v = E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    return np.sum(v * np.exp2(sbytes.astype(np.float64) - 127)[:, None], axis=0)


@pytest.mark.parametrize("dtype,window", [("bfloat16", 8), (np.float16, 5)])
def test_planes_sum_back_within_the_stated_window(dtype, window):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    if dtype == "bfloat16":
        def cast(a):
            return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)
        mant = rng.uniform(1.0, 2.0, size=(400, 32)) * rng.choice([-1.0, 1.0], size=(400, 32))
        blocks = cast(mant * np.exp2(rng.integers(-100, 100, size=(400, 1)) - rng.integers(0, 40, size=(400, 32))))
    else:
        mant = rng.uniform(1.0, 2.0, size=(400, 32)) * rng.choice([-1.0, 1.0], size=(400, 32))
        blocks = (mant * np.exp2(rng.integers(-10, 15, size=(400, 1)) - rng.integers(0, 20, size=(400, 32))))
        blocks = blocks.astype(np.float16).astype(np.float64)
    for b in blocks:
        codes, sb = planes(b)
        assert np.all((sb >= 0) & (sb <= 254))
        got = decode(codes, sb)
        mx = np.max(np.abs(b))
        emax = math.floor(math.log2(mx))
        near = np.abs(b) >= 2.0 ** (emax - window)
        assert np.array_equal(got[near], b[near])
        assert np.max(np.abs(got - b)) <= 2.0 ** -16 * mx


def test_edge_blocks():
    zero = np.zeros(32)
    codes, sb = planes(zero)
    assert not codes.any() and np.all(sb >= 0)
    # the largest bf16 magnitude: plane 0's scale byte is 254, the largest finite E8M0
    big = np.full(32, 3.3895313892515355e38)
    codes, sb = planes(big)
    assert sb[0] == 254 and np.array_equal(decode(codes, sb), big)
    # below the floor of the scales: what lies under 2^-128 is dropped, nothing else
    tiny = np.exp2(-np.arange(118, 150, dtype=np.float64))
    codes, sb = planes(tiny)
    assert np.all(sb >= 0)
    assert np.max(np.abs(decode(codes, sb) - tiny)) <= 2.0 ** -128
