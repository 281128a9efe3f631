"""Seeded synthetic inputs for the MoE expert layer.

This module is shared by the tests, the benchmark and the oracle's callers.  It holds
no arithmetic of the layer itself (no routing, alignment, bucketing, decoding, GEMM,
activation or combine): it only draws random codes, random values and their bf16 /
E4M3 encodings, with the shapes and distributions of the five workloads below.

Workloads (each named by what it is, with its sizes):

* ``tiny``            T=64, hidden 256, intermediate 512, 8 experts, top-2, W4A16 MXFP4,
                      E8M0 exponents 127+U{-4..0}, no bias, seed 0.
* ``decode_mxfp4``    T=64, hidden 2880, intermediate 2880, 128 experts, top-4, W4A16 MXFP4,
                      E8M0 exponents 127+U{-6..-2}, bf16 biases ~N(0, 0.02), seed 1.
* ``prefill_mxfp4``   the same layer; T is the sum of 16 request lengths drawn uniformly
                      from [3277, 4096] (the 0.8*ISL..ISL length rule of the TensorRT-LLM
                      bucketing page, ISL=4096), seed 2.
* ``decode_bf16``     128 experts, hidden 2688, GEMM1 N=1856 (intermediate 928), top-6,
                      bf16 weights ~N(0, 0.02), M in {1, 7, 14, 21, 28}, seed 3.
* ``mxfp8_wgrad``     256 experts, hidden 7168, intermediate 2048, top-8, T=8192; E4M3
                      operands with one E8M0 scale per 32 along K (codes and scale bytes
                      drawn directly, see gen_mx_e4m3), routing drawn from a
                      Zipf(1.1) law over a seeded expert permutation with 16 cold experts,
                      bf16 output gradients ~N(0, 1), seed 4.

Every generator uses numpy's PCG64 seeded generator, so the same seed gives the same
bytes on every machine.  Large operands can instead be drawn on a CUDA device with a
seeded torch generator (``device=`` argument); those are identical run to run on one
machine, and a caller hands the same device bytes to both sides of a comparison.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

try:  # torch is only needed for the bf16 / E4M3 encodings and device generation
    import torch
except ImportError:  # pragma: no cover
    torch = None


# --------------------------------------------------------------------------------------
# Workload descriptions
# --------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int              # real tokens (for decode_bf16: the M of the run)
    K: int              # hidden size
    I: int              # intermediate size (GEMM1 N = 2I gate|up; relu2: N = I)
    E: int              # experts
    k: int              # top-k
    quant: str          # "mxfp4" (W4A16), "bf16", "mxfp8"
    seed: int
    scale_exp: tuple = (0, 0)   # inclusive range of E8M0 exponent offsets (mxfp4)
    bias: bool = False
    weight_std: float = 0.02    # bf16 / mxfp8 weights
    lengths: tuple = ()         # request lengths when T is a sum of requests
    activation: str = "swiglu"  # "swiglu" or "relu2" (non-gated)

    @property
    def n1(self) -> int:
        """Rows of GEMM1 per expert."""
        return 2 * self.I if self.activation == "swiglu" else self.I


TINY = Workload("tiny", T=64, K=256, I=512, E=8, k=2, quant="mxfp4", seed=0,
                scale_exp=(-4, 0))
DECODE_MXFP4 = Workload("decode_mxfp4", T=64, K=2880, I=2880, E=128, k=4, quant="mxfp4",
                        seed=1, scale_exp=(-6, -2), bias=True)
DECODE_BF16_M = (1, 7, 14, 21, 28)
MXFP8_WGRAD = Workload("mxfp8_wgrad", T=8192, K=7168, I=2048, E=256, k=8, quant="mxfp8",
                       seed=4)
ZIPF_S = 1.1
ZIPF_COLD_EXPERTS = 16


def prefill_lengths(seed: int = 2, n_requests: int = 16, isl: int = 4096) -> tuple:
    """Request lengths uniform in [ceil(0.8*isl), isl] (inclusive)."""
    lo = math.ceil(0.8 * isl)
    rng = np.random.Generator(np.random.PCG64(seed))
    return tuple(int(v) for v in rng.integers(lo, isl + 1, size=n_requests))


def prefill_workload(seed: int = 2) -> Workload:
    lens = prefill_lengths(seed)
    return Workload("prefill_mxfp4", T=int(sum(lens)), K=2880, I=2880, E=128, k=4,
                    quant="mxfp4", seed=seed, scale_exp=(-6, -2), bias=True, lengths=lens)


def decode_bf16_workload(M: int, seed: int = 3) -> Workload:
    return Workload(f"decode_bf16_M{M}", T=M, K=2688, I=928, E=128, k=6, quant="bf16",
                    seed=seed)


def decode_bf16_relu2_workload(M: int, seed: int = 5) -> Workload:
    """The Nemotron decode shape with its own activation: non-gated relu^2, GEMM1 N = 1856."""
    return Workload(f"decode_bf16_relu2_M{M}", T=M, K=2688, I=1856, E=128, k=6, quant="bf16",
                    seed=seed, activation="relu2")


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some sizes changed (used for reduced parity cases)."""
    return dataclasses.replace(w, **changes)


def rng_for(seed: int, stream: int) -> np.random.Generator:
    """Independent PCG64 stream ``stream`` of seed ``seed``."""
    return np.random.Generator(np.random.PCG64([seed, stream]))


# --------------------------------------------------------------------------------------
# Encodings (library casts only)
# --------------------------------------------------------------------------------------

def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float array -> uint16 bf16 bit patterns, round-to-nearest-even (torch cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_e4m3_codes(a: np.ndarray) -> np.ndarray:
    """float array already within +-448 -> uint8 E4M3 ("fn") codes (torch cast, RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


# --------------------------------------------------------------------------------------
# Generators
# --------------------------------------------------------------------------------------

def gen_activations_bf16(rng, T, K):
    return to_bf16_bits(rng.standard_normal((T, K), dtype=np.float32))


def gen_logits(rng, T, E):
    return rng.standard_normal((T, E), dtype=np.float32)


def gen_mxfp4_weight(rng, E, N, K, scale_exp):
    """Packed E2M1 codes [E, N, K/2] (uniform over the 16 codes) + E8M0 [E, N, K/32]."""
    packed = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    lo, hi = scale_exp
    scales = (127 + rng.integers(lo, hi + 1, size=(E, N, K // 32))).astype(np.uint8)
    return packed, scales


def gen_bf16_weight(rng, E, N, K, std):
    return to_bf16_bits(rng.standard_normal((E, N, K), dtype=np.float32) * np.float32(std))


# MXFP8 operands are drawn directly as codes and scales: E4M3 codes are the torch cast of
# normal values of standard deviation E4M3_CODE_STD (truncated at the largest E4M3 value,
# 448, which a 7-sigma draw reaches), and each 32-element block gets its own E8M0 scale
# byte 127 + U{lo..hi}.  The decoded operand code * 2^(byte - 127) then has roughly the
# standard deviation E4M3_CODE_STD * 2^e of the workload's values.
E4M3_CODE_STD = 64.0
ACT_SCALE_EXP = (-7, -5)        # activations ~ N(0, 1): 64 * 2^-6 = 1


def scale_exp_for_std(std: float) -> tuple:
    """E8M0 exponent offsets whose middle value scales E4M3_CODE_STD codes to ``std``."""
    c = int(np.round(np.log2(std / E4M3_CODE_STD)))
    return (c - 1, c + 1)


def gen_mx_e4m3(rng, shape, scale_exp=ACT_SCALE_EXP):
    """E4M3 codes of ``shape`` (last axis a multiple of 32) and E8M0 scale bytes
    [..., shape[-1] / 32], drawn as described above (numpy PCG64 generator)."""
    shape = tuple(shape)
    v = rng.standard_normal(shape, dtype=np.float32) * np.float32(E4M3_CODE_STD)
    np.clip(v, -448.0, 448.0, out=v)
    codes = to_e4m3_codes(v)
    lo, hi = scale_exp
    scales = (127 + rng.integers(lo, hi + 1, size=shape[:-1] + (shape[-1] // 32,))).astype(np.uint8)
    return codes, scales


def zipf_topk_ids(rng, T, E, k, s=ZIPF_S, n_cold=ZIPF_COLD_EXPERTS):
    """Top-k distinct expert ids per token from a Zipf(s) law over a seeded permutation.

    ``n_cold`` seeded experts get probability zero.  Sampling without replacement uses
    the Gumbel-top-k construction on log-probabilities.
    """
    perm = rng.permutation(E)
    cold = perm[E - n_cold:] if n_cold else np.array([], dtype=np.int64)
    hot = perm[:E - n_cold]
    logp = np.full(E, -np.inf)
    ranks = np.arange(1, hot.size + 1, dtype=np.float64)
    logp[hot] = -s * np.log(ranks)
    g = rng.gumbel(size=(T, E))
    key = logp[None, :] + g
    ids = np.argsort(-key, axis=1, kind="stable")[:, :k]
    return ids.astype(np.int32), cold.astype(np.int32)


def make_layer(w: Workload, T: int | None = None, with_logits: bool = True):
    """Host inputs of one MoE layer: dict of numpy arrays.

    Keys: x (uint16 bf16 [T,K]) or x_codes/x_scale (mxfp8), logits (fp32 [T,E]),
    w1 / w1_scale / b1, w2 / w2_scale / b2 in the layouts of the C ABI:
    w1 [E, 2I, K(/2)] rows 0..I-1 gate and I..2I-1 up (relu2: w1 [E, I, K(/2)]);
    w2 [E, K, I(/2)].
    """
    T = w.T if T is None else T
    out = {"workload": w, "T": T}
    r_act, r_log, r_w1, r_w2, r_b = (rng_for(w.seed, s) for s in range(5))
    if w.quant == "mxfp8":
        out["x_codes"], out["x_scale"] = gen_mx_e4m3(r_act, (T, w.K))
    else:
        out["x"] = gen_activations_bf16(r_act, T, w.K)
    if with_logits:
        out["logits"] = gen_logits(r_log, T, w.E)
    if w.quant == "mxfp4":
        out["w1"], out["w1_scale"] = gen_mxfp4_weight(r_w1, w.E, w.n1, w.K, w.scale_exp)
        out["w2"], out["w2_scale"] = gen_mxfp4_weight(r_w2, w.E, w.K, w.I, w.scale_exp)
    elif w.quant == "bf16":
        out["w1"] = gen_bf16_weight(r_w1, w.E, w.n1, w.K, w.weight_std)
        out["w2"] = gen_bf16_weight(r_w2, w.E, w.K, w.I, w.weight_std)
        out["w1_scale"] = out["w2_scale"] = None
    elif w.quant == "mxfp8":
        se = scale_exp_for_std(w.weight_std)
        out["w1"], out["w1_scale"] = gen_mx_e4m3(r_w1, (w.E, w.n1, w.K), se)
        out["w2"], out["w2_scale"] = gen_mx_e4m3(r_w2, (w.E, w.K, w.I), se)
    else:
        raise ValueError(w.quant)
    if w.bias:
        out["b1"] = to_bf16_bits(r_b.standard_normal((w.E, w.n1), dtype=np.float32) * np.float32(0.02))
        out["b2"] = to_bf16_bits(r_b.standard_normal((w.E, w.K), dtype=np.float32) * np.float32(0.02))
    else:
        out["b1"] = out["b2"] = None
    return out


def pad_host_rows(a: np.ndarray, rows: int) -> np.ndarray:
    """Append zero rows so that ``a`` has ``rows`` rows (input preparation for tests)."""
    if a.shape[0] >= rows:
        return a
    pad = np.zeros((rows - a.shape[0],) + a.shape[1:], dtype=a.dtype)
    return np.concatenate([a, pad], axis=0)


# --------------------------------------------------------------------------------------
# The grouped-GEMM + wgrad workload with MXFP8 operands
# --------------------------------------------------------------------------------------

def make_mxfp8_gemm_wgrad(w: Workload = MXFP8_WGRAD, T: int | None = None, E: int | None = None,
                          K: int | None = None, I: int | None = None, device=None):
    """Operands of the MXFP8 grouped GEMMs and of the weight gradients.

    GEMM1: A = x (E4M3 [T,K] + E8M0 [T,K/32]) per token, W1 [E, 2I, K] -> out1 [P, 2I] bf16.
    GEMM2: A = a2 (E4M3 [P, I] + E8M0 [P, I/32]) per pair,  W2 [E, K, I] -> out2 [P, K] bf16.
    wgrad: dW1[e] = sum over pairs of expert e of grad1[p]^T x_bf16[p // k]   ([E, 2I, K])
           dW2[e] = sum over pairs of expert e of grad2[p]^T h_bf16[p]       ([E, K, I])

    With ``device`` set (a CUDA device) the large operands are drawn there with a
    seeded torch generator and returned as torch tensors; the small ones (routing) are
    numpy.  Without it everything is numpy on the host.
    """
    T = w.T if T is None else T
    E = w.E if E is None else E
    K = w.K if K is None else K
    I = w.I if I is None else I
    k = w.k
    P = T * k
    r_route = rng_for(w.seed, 10)
    ids, cold = zipf_topk_ids(r_route, T, E, k, n_cold=min(ZIPF_COLD_EXPERTS, max(E - k, 0) // 2))
    out = {"T": T, "E": E, "K": K, "I": I, "k": k, "P": P, "topk_ids": ids, "cold": cold}
    if device is None:
        rs = [rng_for(w.seed, 11 + i) for i in range(8)]
        se = scale_exp_for_std(w.weight_std)
        out["x_codes"], out["x_scale"] = gen_mx_e4m3(rs[0], (T, K))
        out["a2_codes"], out["a2_scale"] = gen_mx_e4m3(rs[1], (P, I))
        out["w1"], out["w1_scale"] = gen_mx_e4m3(rs[2], (E, 2 * I, K), se)
        out["w2"], out["w2_scale"] = gen_mx_e4m3(rs[3], (E, K, I), se)
        out["x_bf16"] = gen_activations_bf16(rs[4], T, K)
        out["h_bf16"] = gen_activations_bf16(rs[5], P, I)
        out["grad1"] = gen_activations_bf16(rs[6], P, 2 * I)
        out["grad2"] = gen_activations_bf16(rs[7], P, K)
        return out
    g = torch.Generator(device=device)

    def dev_mx(shape, scale_exp, sub):
        g.manual_seed(w.seed * 1000 + sub)
        v = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * E4M3_CODE_STD
        codes = v.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        del v
        lo, hi = scale_exp
        sc = torch.randint(127 + lo, 127 + hi + 1, shape[:-1] + (shape[-1] // 32,), generator=g,
                           device=device, dtype=torch.int32).to(torch.uint8)
        return codes.contiguous(), sc.contiguous()

    def dev_bf16(shape, sub):
        g.manual_seed(w.seed * 1000 + sub)
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)

    se = scale_exp_for_std(w.weight_std)
    out["x_codes"], out["x_scale"] = dev_mx((T, K), ACT_SCALE_EXP, 1)
    out["a2_codes"], out["a2_scale"] = dev_mx((P, I), ACT_SCALE_EXP, 2)
    # weights are drawn one expert slab at a time to bound the float32 temporaries
    w1c = torch.empty((E, 2 * I, K), dtype=torch.uint8, device=device)
    w1s = torch.empty((E, 2 * I, K // 32), dtype=torch.uint8, device=device)
    w2c = torch.empty((E, K, I), dtype=torch.uint8, device=device)
    w2s = torch.empty((E, K, I // 32), dtype=torch.uint8, device=device)
    step = 16
    for e0 in range(0, E, step):
        e1 = min(E, e0 + step)
        c, s = dev_mx((e1 - e0, 2 * I, K), se, 100 + e0)
        w1c[e0:e1].copy_(c), w1s[e0:e1].copy_(s)
        c, s = dev_mx((e1 - e0, K, I), se, 5000 + e0)
        w2c[e0:e1].copy_(c), w2s[e0:e1].copy_(s)
    out["w1"], out["w1_scale"], out["w2"], out["w2_scale"] = w1c, w1s, w2c, w2s
    out["x_bf16"] = dev_bf16((T, K), 3)
    out["h_bf16"] = dev_bf16((P, I), 4)
    out["grad1"] = dev_bf16((P, 2 * I), 5)
    out["grad2"] = dev_bf16((P, K), 6)
    return out
