"""Geometric token-dimension buckets, pad and slice.  (Test infrastructure.)

"Bound Triton MoE JIT specializations via token-dim bucketing and warmup" (TensorRT-LLM
PR 15311), Description: the MoE token count m is padded to a geometric bucket -- eight
buckets per power-of-two octave, at most 12.5% padding -- before the grouped GEMMs, and
the pad rows are sliced off before the reduction over ranks; 97 buckets cover
max_num_tokens = 20000.  Test Coverage lists the properties: rounds up by at most 12.5%,
is a fixed point on buckets, is monotonic, and the enumeration equals the closure.

Reading taken: bucket(m) = ceil(m / s) * s with s = max(1, 2^(floor(log2 m) - 3)).  For
m < 16 every m is its own bucket; from 16 on each octave [2^j, 2^(j+1)) holds 8 buckets
spaced 2^(j-3).  bucket_iter(N) lists every bucket <= N (97 of them for N = 20000).

Padding is allowed only for the W4A16 MXFP4 mode (bf16 activations, weights with static
block scales), where pad rows cannot change real rows; other modes leave m unpadded and
report it (Description, the paragraph on the W4A16 MXFP4 restriction).  Pad rows are
zero activations; their router logits are zero too.
"""
import numpy as np


def bucket(m: int) -> int:
    m = int(m)
    if m < 1:
        raise ValueError("bucket is defined for m >= 1")
    s = max(1, 1 << max(0, (m.bit_length() - 1) - 3))
    return -(-m // s) * s


def bucket_iter(n: int) -> list:
    return [b for b in range(1, int(n) + 1) if bucket(b) == b]


def pad_allowed(quant: str) -> bool:
    return quant == "mxfp4"


def padded_rows(m: int, quant: str) -> int:
    return bucket(m) if pad_allowed(quant) else int(m)


def pad_rows(a, rows: int):
    """``a`` with zero rows appended up to ``rows`` rows."""
    a = np.asarray(a)
    out = np.zeros((rows,) + a.shape[1:], dtype=a.dtype)
    out[:a.shape[0]] = a
    return out
