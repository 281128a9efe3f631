"""Shared test helpers: tolerance checks and host <-> device marshalling."""
import numpy as np

try:
    import torch
except ImportError:  # pragma: no cover
    torch = None

# Floating-point bar for bf16 outputs against the float64 oracle: relative Frobenius error
# <= 5e-3, and every element within 2e-2 * rms(reference) beyond the half ulp that
# rounding the exact value to the bf16 output already costs (an element of magnitude
# above ~5 rms cannot be stored closer than 2^-9 of itself).
REL_FRO = 5e-3
ELEM_RMS = 2e-2


def bf16_half_ulp(ref):
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def assert_close_bf16(got, ref, rel_fro=REL_FRO, elem_rms=ELEM_RMS, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = got - ref
    nref = np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    rel = np.linalg.norm(diff) / nref if nref > 0 else np.linalg.norm(diff)
    beyond = np.maximum(np.abs(diff) - bf16_half_ulp(ref), 0.0)
    worst = np.max(beyond) if diff.size else 0.0
    assert rel <= rel_fro, f"{what}: relative Frobenius error {rel:.3e} > {rel_fro}"
    assert worst <= elem_rms * max(rms, 1e-30), \
        f"{what}: max |err| beyond the output half ulp {worst:.3e} > {elem_rms} * rms {rms:.3e}"
    return rel, worst / max(rms, 1e-30)


def bf16_to_np(t):
    """torch bf16 tensor (any device) -> float64 numpy."""
    return t.detach().to("cpu").view(torch.int16).numpy().view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)


def dev(a, device="cuda"):
    """numpy array -> torch device tensor with the same bytes (uint16 -> bf16)."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def ulp_diff_f32(a, b):
    ai = np.asarray(a, dtype=np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, dtype=np.float32).view(np.int32).astype(np.int64)
    return np.abs(ai - bi)
