"""MXFP8 quantisation of a float tensor: E4M3 elements with one E8M0 scale per 32.
(Test infrastructure.)

The step the pages leave open between the GEMMs of an MXFP8 layer: "Add MoE GEMM variants
and weight-gradient kernel" (aiter PR 5310), Summary, gives moe_gemm_mxfp8 E4M3 operands
with one E8M0 microscale per 32 K elements, so the SwiGLU output h must be brought into that
format before GEMM2.  Reading taken, the scale rule of the OCP microscaling (MX)
specification for E4M3 elements (largest element exponent emax = 8):

  for each block of 32 consecutive values v along a row,
    amax = max |v|;  e = floor(log2(amax)) - 8, clamped to [-127, 127]  (e = -127 if amax = 0)
    scale byte = e + 127;  code_i = E4M3(v_i / 2^e)
  where E4M3(.) rounds to nearest, ties to the even code, and saturates magnitudes above
  448 to 448 (the "fn" format has no infinity); the sign of v (zero included) is kept.
  A block holding a NaN gets the NaN scale byte 0xFF and NaN codes 0x7F.

Every step here is exact in float64 except the one rounding of E4M3(.), so a float32 input
gives the same codes and scales whether the division is done in float32 or float64.
"""
import numpy as np

from . import formats

E4M3_EMAX = 8
# finite non-negative E4M3 magnitudes, indexed by code 0x00 .. 0x7E
_MAG = formats.e4m3_decode(np.arange(0x7F))


def e4m3_encode(v) -> np.ndarray:
    """Round-to-nearest-even, saturating E4M3 codes of float values (NaN -> 0x7F)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    # the largest code whose magnitude is <= a (0 for a < the smallest subnormal)
    lo = np.clip(np.searchsorted(_MAG, a, side="right") - 1, 0, 0x7E)
    hi = np.clip(lo + 1, 0, 0x7E)
    d_lo = a - _MAG[lo]
    d_hi = _MAG[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (lo % 2 == 1))
    code = np.where(pick_hi & (hi != lo), hi, lo)
    code = np.where(a >= _MAG[0x7E], 0x7E, code)  # saturation (448 and above)
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def block_exponent(amax) -> np.ndarray:
    """e = floor(log2(amax)) - 8 clamped to [-127, 127]; -127 for amax = 0."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        _, ex = np.frexp(amax)           # amax = m * 2^ex, 0.5 <= m < 1
    e = np.where(amax > 0, ex - 1 - E4M3_EMAX, -127)
    e = np.where(np.isinf(amax), 127, e)
    return np.clip(e, -127, 127).astype(np.int64)


def mx_quantize(x):
    """x [..., C] (C a multiple of 32) -> (codes [..., C] uint8, scales [..., C/32] uint8)."""
    x = np.asarray(x, dtype=np.float64)
    C = x.shape[-1]
    if C % 32:
        raise ValueError("the row length must be a multiple of 32")
    blk = x.reshape(*x.shape[:-1], C // 32, 32)
    nan_blk = np.isnan(blk).any(axis=-1)
    amax = np.where(nan_blk, 0.0, np.nanmax(np.abs(np.where(np.isnan(blk), 0.0, blk)), axis=-1))
    e = block_exponent(amax)
    codes = e4m3_encode(blk * np.ldexp(1.0, -e)[..., None])
    codes = np.where(nan_blk[..., None], 0x7F, codes).astype(np.uint8)
    scales = np.where(nan_blk, 255, e + 127).astype(np.uint8)
    return codes.reshape(x.shape), scales
