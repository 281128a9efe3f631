"""The C ABI library loads, exports every symbol its header declares, and its host-side
logic (bucket math, capacity, workspace sizes, argument validation) is correct.  No GPU:
no call here launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import mixture_experts_grouped_align_gb300 as moe
from oracle import align as oalign
from oracle import bucket as obucket

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.load()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_binding_symbols():
    assert sorted(declared_functions()) == sorted(moe.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_bucket_matches_oracle_exhaustively(lib):
    got = [moe.moe_bucket(m) for m in range(1, 65537)]
    want = [obucket.bucket(m) for m in range(1, 65537)]
    assert got == want
    assert moe.moe_bucket(0) == -1
    assert moe.moe_bucket_count(20000) == 97
    for n in (1, 15, 16, 17, 100, 4096, 20000, 65536):
        assert moe.moe_bucket_count(n) == len(obucket.bucket_iter(n))


def test_bucket_pad_host_math_without_device_buffers(lib):
    st, tp = moe.moe_bucket_pad(59000, "mxfp4")
    assert st == 0 and tp == obucket.bucket(59000)
    st, tp = moe.moe_bucket_pad(59000, "bf16")
    assert st == moe.MOE_WARN_PAD_IGNORED and tp == 59000
    st, tp = moe.moe_bucket_pad(17, "mxfp8")
    assert st == moe.MOE_WARN_PAD_IGNORED and tp == 17
    st, tp = moe.moe_bucket_pad(0, "mxfp4")
    assert st == 0 and tp == 0


@pytest.mark.parametrize("P,E,bm", [(0, 1, 1), (256, 128, 128), (65536, 256, 128), (7, 5, 16)])
def test_capacity_matches_oracle(lib, P, E, bm):
    assert moe.moe_align_capacity(P, E, bm) == oalign.capacity(P, E, bm)


def test_workspace_size(lib):
    r = lambda v: (v + 255) // 256 * 256
    cap, _ = moe.moe_align_capacity(256, 128, 128)
    n = moe.moe_forward_workspace_size(64, 4, 2880, 2880, cap)
    P = 256  # up to 256 rows: h and x in pair / token order
    kq, sb = 23 * 64, 96  # K and I of 2880: 23 words of 128 K, 64 bytes each; 16-byte scale rows
    planes = r(64 * 8 * kq) + r(64 * sb) + r(P * 8 * kq) + r(P * sb) + r((P + 1) * 16)
    assert n == r(P * 2880 * 2) + r(P * 2880 * 4) + r(64 * 2880 * 2) + planes
    cap, _ = moe.moe_align_capacity(4 * 1000, 128, 128)
    n = moe.moe_forward_workspace_size(1000, 4, 2880, 2880, cap)
    assert n == r(cap * 2880 * 2) + r(4000 * 2880 * 4) + r(cap * 2880 * 2) + \
        2 * fix_bytes(cap // 128, 2880)  # slot order, and the marks of both GEMMs
    assert moe.moe_forward_workspace_size(-1, 4, 1, 1, 0) == 0


def test_argument_errors_are_reported_without_a_launch(lib):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_align(None, None, None, 4, 2, 8, 16, None, 64, None, None)
    assert ei.value.status == -1
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_align(None, 16, None, 4, 40, 8, 16, 16, 64, 16, 16)
    assert ei.value.status == -2            # k > 32 / k > E
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_align(None, 16, None, 4, 2, 8, 16, 16, 16, 16, 16)
    assert ei.value.status == -3            # capacity too small
    big = moe.Ctx(stream=0, workspace=16, workspace_bytes=1 << 40)  # checked, never touched
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward("mxfp8", 8, 256, 512, 16, 16, None, 16, 16, None, 16, 16, 4, 4, 2,
                        16, 16, 16, 16, None, 16, 256, 16, big, activation="relu2")
    assert ei.value.status == -2            # the MXFP8 layer takes SwiGLU only
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward("mxfp8", 8, 256, 512, 16, 16, None, 16, 16, None, 16, None, 4, 4, 2,
                        16, 16, 16, 16, None, 16, 256, 16, big)
    assert ei.value.status == -1            # MXFP8 activations need their scales
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward("mxfp8", 8, 256, 512, 16, 16, None, 16, 16, None, 16, 16, 4, 4, 2,
                        16, 16, 16, 16, None, 16, 256, 16, big)
    assert ei.value.status == -2            # few rows keep fp32 h in the o scratch: I <= K
    assert "I <= K" in lib.moe_last_error().decode()
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_mx_quantize(16, 4, 48, 16, 16, moe.Ctx(stream=0))
    assert ei.value.status == -1            # 48 columns: not whole 32-blocks
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward("mxfp4", 8, 256, 512, 16, 16, None, 16, 16, None, 16, None, 4, 4, 2,
                        16, 16, 16, 16, None, 16, 256, 16, moe.Ctx(stream=0), activation=5)
    assert ei.value.status == -1            # unknown activation
    assert "activation" in lib.moe_last_error().decode()
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_wgrad(16, 16, 0, 4, 2, 8, 100, 64, 16, 16, 16, 16, 256, 16, 0, moe.Ctx(stream=0))
    assert ei.value.status == -2            # N not a multiple of 64
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_grouped_gemm("bf16", 8, 64, 64, 8, None, 0, 16, None, None, 4, 2, 16, 16, 16, 16,
                             256, 16, moe.Ctx(stream=0))
    assert ei.value.status == -1            # misaligned pointer
    assert "aligned" in lib.moe_last_error().decode()
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_gemm_per_token(8, 192, 256, 16, 16, 16, 16, None, 16, 100, 16, moe.Ctx(stream=0))
    assert ei.value.status == -2            # N not a multiple of 128
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_gemm_per_token(8, 256, 256, 16, 16, 16, 16, None, None, 100, 16, moe.Ctx(stream=0))
    assert ei.value.status == -1            # no group sizes


def test_size_overflow_is_rejected_before_any_launch(lib):
    # T*k beyond int32 slot indices, including a T whose product with k overflows int64.
    for T, k in ((1 << 30, 2), (1 << 62, 8), ((1 << 31) - 1, 1)):
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_align(None, 16, None, T, k, 8, 16, 16, 16, 16, 16)
        if T * k >= 1 << 31:
            assert ei.value.status == -2 and "2^31" in lib.moe_last_error().decode()
        else:                                 # fits: then the capacity of 16 slots is short
            assert ei.value.status == -3
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_wgrad(16, 16, 0, 1 << 62, 4, 8, 64, 64, 16, 16, 16, 16, 256, 16, 0, moe.Ctx(stream=0))
    assert ei.value.status == -2
    # An [E, N, Kin] weight array past 64-bit element indexing.
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_grouped_gemm("bf16", 1024, (1 << 31) - 16, (1 << 31) - 32, 16, None, 0, 16, None,
                             None, 4, 2, 16, 16, 16, 16, 1 << 20, 16, moe.Ctx(stream=0))
    assert ei.value.status == -2 and "64-bit" in lib.moe_last_error().decode()
    big = moe.Ctx(stream=0, workspace=16, workspace_bytes=1 << 40)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward("bf16", 1024, (1 << 31) - 32, (1 << 31) - 32, 16, None, None, 16, None, None,
                        16, None, 4, 4, 2, 16, 16, 16, 16, None, 16, 256, 16, big)
    assert ei.value.status == -2 and "64-bit" in lib.moe_last_error().decode()


def fix_bytes(blocks, nout):
    """The marks of one tensor-memory GEMM: a 256-byte count, then one bit per tile (128
    output features per tile), rounded up to 256 bytes."""
    r = lambda v: (v + 255) // 256 * 256
    tiles = blocks * -(-nout // 128)
    return 256 + r(-(-tiles // 32) * 4)


def test_grouped_gemm_workspace_size(lib):
    r = lambda v: (v + 255) // 256 * 256
    blocks = lambda P: P + P // 128 + 1
    assert moe.moe_grouped_gemm_workspace_size("mxfp4", 256, 4, 5760, 2880, 0) == 0     # weight streaming
    assert moe.moe_grouped_gemm_workspace_size("mxfp4", 257, 4, 5760, 2880, 0) == \
        r(257 * 2880 * 2) + fix_bytes(blocks(257 * 4), 5760)
    assert moe.moe_grouped_gemm_workspace_size("mxfp4", 300, 4, 2880, 2880, 1) == \
        r(1200 * 2880 * 2) + fix_bytes(blocks(1200), 2880)
    assert moe.moe_grouped_gemm_workspace_size("mxfp8", 4096, 8, 4096, 7168, 0) == 0     # reads E4M3 as is
    assert moe.moe_grouped_gemm_workspace_size("bf16", 4096, 8, 4096, 7168, 0) == 0


def test_wgrad_workspace_size(lib):
    """Slot-ordered copies of grad [cap, N] and input [cap, Kin] bf16 and the experts' block
    ranges [E, 2] int32, each rounded up to 256 bytes, for the deterministic tensor-core
    wgrad; 0 wherever that kernel cannot read them."""
    r = lambda v: (v + 255) // 256 * 256
    cap = 98048                                     # 65536 pairs over 256 experts, block 128
    assert moe.moe_wgrad_workspace_size(256, 4096, 7168, 128, cap, 0) == \
        r(cap * 4096 * 2) + r(cap * 7168 * 2) + r(256 * 8)
    assert moe.moe_wgrad_workspace_size(256, 7168, 2048, 64, cap, 0) == \
        r(cap * 7168 * 2) + r(cap * 2048 * 2) + r(256 * 8)
    assert moe.moe_wgrad_workspace_size(256, 4096, 7168, 128, cap, 1) == 0   # accumulate mode
    assert moe.moe_wgrad_workspace_size(256, 4096, 7168, 16, cap, 0) == 0    # stages would cross experts
    assert moe.moe_wgrad_workspace_size(256, 64, 7168, 128, cap, 0) == 0     # N not a multiple of 128
    assert moe.moe_wgrad_workspace_size(2048, 128, 128, 128, cap, 0) == 0    # more than 1024 experts
    assert moe.moe_wgrad_workspace_size(8, 128, 128, 128, 0, 0) == 0
