"""Element and scale formats, decoded exactly to float64.  (Test infrastructure.)

* E8M0 scale (one unsigned byte per 32 elements along K): value 2^(e-127); the byte
  0xFF is NaN and the byte 0x00 is 2^-127, not zero -- the decoding rule the second
  review of "Add MoE GEMM variants and weight-gradient kernel" (aiter PR 5310) states
  for E8M0 microscales.
* E2M1 (FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent field 0
  is subnormal (mantissa * 0.5).  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
* E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent field 0
  is subnormal (m * 2^-9); S.1111.111 is NaN; there is no infinity; max 448.
* bf16: the upper 16 bits of an IEEE binary32.

Packed E2M1 stores two elements per byte, the even K index in the low nibble (the
reading this project takes; the pages do not fix a nibble order).
"""
import numpy as np


def e8m0_decode(codes) -> np.ndarray:
    c = np.asarray(codes).astype(np.int64)
    val = np.ldexp(np.float64(1.0), c - 127)
    return np.where(c == 255, np.nan, val)


def e2m1_decode(codes) -> np.ndarray:
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = (c >> 3) & 1
    exp = (c >> 1) & 3
    man = c & 1
    mag = np.where(exp == 0, man * 0.5, np.ldexp(1.0 + man / 2.0, exp - 1))
    return np.where(sign == 1, -mag, mag).astype(np.float64)


def e4m3_decode(codes) -> np.ndarray:
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = (c >> 7) & 1
    exp = (c >> 3) & 0xF
    man = c & 7
    mag = np.where(exp == 0, man * 2.0 ** -9, np.ldexp(1.0 + man / 8.0, exp - 7))
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag).astype(np.float64)


def bf16_decode(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to NaN
        return b.view(np.float32).astype(np.float64)


def unpack_e2m1(packed) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] nibble codes (even index = low nibble)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def apply_block_scale(values: np.ndarray, scales) -> np.ndarray:
    """values [..., K] float64 times E8M0 scales [..., K/32] repeated over each 32-block."""
    s = e8m0_decode(scales)
    return values * np.repeat(s, 32, axis=-1)


def dequant_mxfp4(packed, scales) -> np.ndarray:
    # the 16 code values, then a gather: same numbers as decoding each code in place
    return apply_block_scale(e2m1_decode(np.arange(16))[unpack_e2m1(packed)], scales)


def dequant_mxfp8(codes, scales) -> np.ndarray:
    return apply_block_scale(e4m3_decode(np.arange(256))[np.asarray(codes, dtype=np.uint8)], scales)


def dequant(fmt: str, data, scales=None) -> np.ndarray:
    """Decode a weight or activation operand of format ``fmt`` to float64."""
    if fmt == "mxfp4":
        return dequant_mxfp4(data, scales)
    if fmt == "mxfp8":
        return dequant_mxfp8(data, scales)
    if fmt == "bf16":
        return bf16_decode(data)
    raise ValueError(fmt)
