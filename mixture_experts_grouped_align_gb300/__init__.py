"""Python binding of the GB300 MoE expert-layer library (libmoe_gb300.so).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.
Functions carry the C ABI's names (include/moe_gb300.h).  Tensor arguments may be torch
tensors (their device pointer is passed) or plain integers (raw device pointers) or None
(NULL).  PyTorch is used only for device memory and streams.

The library must have been built (``build()`` or ``python -m
mixture_experts_grouped_align_gb300.build``); loading fails loudly otherwise -- there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB, build  # noqa: F401

__all__ = [
    "MoeError", "load", "Ctx", "QUANT", "ACTIVATION", "moe_align_capacity", "moe_align", "moe_bucket",
    "moe_bucket_count", "moe_bucket_pad", "moe_forward_workspace_size", "moe_forward",
    "moe_forward_no_alloc", "moe_grouped_gemm", "moe_grouped_gemm_workspace_size", "moe_mx_quantize",
    "moe_gemm_per_token", "moe_wgrad", "moe_wgrad_workspace_size", "moe_debug_stall_tensor_kernels",
    "EXPORTED_SYMBOLS",
]

MOE_OK = 0
MOE_WARN_PAD_IGNORED = 1
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_WARN_PAD_IGNORED", -1: "MOE_ERR_INVALID_ARG",
                -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_CAPACITY", -4: "MOE_ERR_CUDA",
                -5: "MOE_ERR_INVALID_EXPERT", -6: "MOE_ERR_RANGE", -7: "MOE_ERR_TIMEOUT"}
QUANT = {"bf16": 0, "mxfp4": 1, "mxfp8": 2}
ACTIVATION = {"swiglu": 0, "relu2": 1}

EXPORTED_SYMBOLS = [
    "moe_last_error", "moe_align_capacity", "moe_align", "moe_bucket", "moe_bucket_count",
    "moe_bucket_pad", "moe_forward_workspace_size", "moe_forward", "moe_forward_no_alloc",
    "moe_grouped_gemm", "moe_grouped_gemm_workspace_size", "moe_mx_quantize", "moe_gemm_per_token", "moe_wgrad",
    "moe_wgrad_workspace_size", "moe_debug_stall_tensor_kernels",
]


class MoeError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class _Ctx(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("dev_status", ctypes.c_void_p),
                ("events", ctypes.POINTER(ctypes.c_void_p)), ("n_events", ctypes.c_int32)]


class _Weights(ctypes.Structure):
    _fields_ = [("quant", ctypes.c_int), ("E", ctypes.c_int32), ("K", ctypes.c_int32),
                ("I", ctypes.c_int32), ("w1", ctypes.c_void_p), ("w1_scale", ctypes.c_void_p),
                ("b1", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p),
                ("b2", ctypes.c_void_p), ("activation", ctypes.c_int32)]


_lib = None


def load(path: str | None = None):
    """Loads the library once.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(mixture_experts_grouped_align_gb300.build.build())")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "moe_last_error": (ctypes.c_char_p, []),
        "moe_align_capacity": (I32, [I64, I32, I32, P, P]),
        "moe_align": (I32, [P, P, P, I64, I32, I32, I32, P, I64, P, P, P, P]),
        "moe_bucket": (I64, [I64]),
        "moe_bucket_count": (I64, [I64]),
        "moe_bucket_pad": (I32, [I64, ctypes.c_int, P, P, P, I64, P, P, I32, P]),
        "moe_forward_workspace_size": (SZ, [I64, I32, I32, I32, I64]),
        "moe_forward": (I32, [P, P, P, I64, I64, I32, P, P, P, P, P, I32, I64, P, P]),
        "moe_forward_no_alloc": (I32, [P, P, P, I64, I64, I32, P, P, P, P, P, I32, I64, P, P]),
        "moe_grouped_gemm": (I32, [ctypes.c_int, I32, I32, I32, P, P, I32, P, P, P, I64, I32,
                                   P, P, P, I32, I64, P, P]),
        "moe_grouped_gemm_workspace_size": (SZ, [ctypes.c_int, I64, I32, I32, I32, I32]),
        "moe_mx_quantize": (I32, [P, I64, I32, P, P, P]),
        "moe_gemm_per_token": (I32, [I32, I32, I32, P, P, P, P, P, P, I64, P, P]),
        "moe_wgrad": (I32, [P, P, I32, I64, I32, I32, I32, I32, P, P, P, I32, I64, P, I32, P]),
        "moe_wgrad_workspace_size": (SZ, [I32, I32, I32, I32, I64, I32]),
        "moe_debug_stall_tensor_kernels": (None, [I64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _check(status):
    if status < 0:
        raise MoeError(status, load().moe_last_error().decode())
    return status


class Ctx:
    """Stream, workspace, device status word and profiling events of a call (all
    optional).  ``events`` is a list of torch.cuda.Event (or raw cudaEvent_t ints)."""

    def __init__(self, stream=None, workspace=None, workspace_bytes=None, dev_status=None,
                 events=None):
        s = stream
        if s is not None and not isinstance(s, int):
            s = s.cuda_stream
        if s is None:
            try:
                import torch
                s = torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
            except Exception:  # pragma: no cover
                s = 0
        nbytes = workspace_bytes
        if nbytes is None:
            nbytes = 0 if workspace is None or isinstance(workspace, int) else \
                workspace.numel() * workspace.element_size()
        ev_arr, n_ev = None, 0
        if events:
            handles = [e if isinstance(e, int) else e.cuda_event for e in events]
            ev_arr = (ctypes.c_void_p * len(handles))(*handles)
            n_ev = len(handles)
        self._c = _Ctx(s, _ptr(workspace), nbytes, _ptr(dev_status),
                       ctypes.cast(ev_arr, ctypes.POINTER(ctypes.c_void_p)) if ev_arr else None, n_ev)
        self._keep = (workspace, dev_status, events, ev_arr)

    @property
    def ref(self):
        return ctypes.byref(self._c)


def _ctx(ctx):
    return (ctx or Ctx()).ref


def moe_align_capacity(num_pairs: int, E: int, block_m: int):
    cap_t, cap_b = ctypes.c_int64(), ctypes.c_int64()
    _check(load().moe_align_capacity(num_pairs, E, block_m, ctypes.byref(cap_t), ctypes.byref(cap_b)))
    return cap_t.value, cap_b.value


def moe_align(logits, topk_ids, topk_w, T, k, E, block_m, sorted_token_ids, cap_tokens,
              expert_ids, num_tokens_post_padded, expert_offsets=None, ctx=None):
    return _check(load().moe_align(_ptr(logits), _ptr(topk_ids), _ptr(topk_w), T, k, E, block_m,
                                   _ptr(sorted_token_ids), cap_tokens, _ptr(expert_ids),
                                   _ptr(num_tokens_post_padded), _ptr(expert_offsets), _ctx(ctx)))


def moe_bucket(m: int) -> int:
    return load().moe_bucket(m)


def moe_bucket_count(max_tokens: int) -> int:
    return load().moe_bucket_count(max_tokens)


def moe_bucket_pad(T, quant, x=None, x_pad=None, row_bytes=0, logits=None, logits_pad=None, E=0,
                   ctx=None):
    """Returns (status, T_pad); status 1 = padding not allowed for this mode."""
    tp = ctypes.c_int64()
    q = QUANT[quant] if isinstance(quant, str) else quant
    st = _check(load().moe_bucket_pad(T, q, ctypes.byref(tp), _ptr(x), _ptr(x_pad), row_bytes,
                                      _ptr(logits), _ptr(logits_pad), E, _ctx(ctx)))
    return st, tp.value


def moe_forward_workspace_size(T_rows, k, K, I, cap_tokens) -> int:
    return load().moe_forward_workspace_size(T_rows, k, K, I, cap_tokens)


def _act(activation):
    return ACTIVATION[activation] if isinstance(activation, str) else int(activation)


def moe_forward(quant, E, K, I, w1, w1_scale, b1, w2, w2_scale, b2, x, x_scale, T_rows, T_real, k,
                topk_w, sorted_token_ids, expert_ids, num_tokens_post_padded, expert_offsets,
                block_m, cap_tokens, y, ctx, activation="swiglu"):
    q = QUANT[quant] if isinstance(quant, str) else quant
    W = _Weights(q, E, K, I, _ptr(w1), _ptr(w1_scale), _ptr(b1), _ptr(w2), _ptr(w2_scale), _ptr(b2),
                 _act(activation))
    return _check(load().moe_forward(ctypes.byref(W), _ptr(x), _ptr(x_scale), T_rows, T_real, k,
                                     _ptr(topk_w), _ptr(sorted_token_ids), _ptr(expert_ids),
                                     _ptr(num_tokens_post_padded), _ptr(expert_offsets), block_m,
                                     cap_tokens, _ptr(y), _ctx(ctx)))


def moe_forward_no_alloc(quant, E, K, I, w1, w1_scale, b1, w2, w2_scale, b2, x, x_scale, T_rows,
                         T_real, k, topk_w, sorted_token_ids, expert_ids, num_tokens_post_padded,
                         expert_offsets, block_m, cap_tokens, y, ctx=None, activation="swiglu"):
    """moe_forward with its scratch in the library's fixed device array (no workspace)."""
    q = QUANT[quant] if isinstance(quant, str) else quant
    W = _Weights(q, E, K, I, _ptr(w1), _ptr(w1_scale), _ptr(b1), _ptr(w2), _ptr(w2_scale), _ptr(b2),
                 _act(activation))
    return _check(load().moe_forward_no_alloc(
        ctypes.byref(W), _ptr(x), _ptr(x_scale), T_rows, T_real, k, _ptr(topk_w),
        _ptr(sorted_token_ids), _ptr(expert_ids), _ptr(num_tokens_post_padded),
        _ptr(expert_offsets), block_m, cap_tokens, _ptr(y), _ctx(ctx)))


def moe_grouped_gemm(quant, E, N, Kin, a, a_scale, a_per_pair, w, w_scale, bias, T, k,
                     sorted_token_ids, expert_ids, num_tokens_post_padded, block_m, cap_tokens,
                     out, ctx=None):
    q = QUANT[quant] if isinstance(quant, str) else quant
    return _check(load().moe_grouped_gemm(q, E, N, Kin, _ptr(a), _ptr(a_scale), int(a_per_pair),
                                          _ptr(w), _ptr(w_scale), _ptr(bias), T, k,
                                          _ptr(sorted_token_ids), _ptr(expert_ids),
                                          _ptr(num_tokens_post_padded), block_m, cap_tokens,
                                          _ptr(out), _ctx(ctx)))


def moe_grouped_gemm_workspace_size(quant, T, k, N, Kin, a_per_pair) -> int:
    q = QUANT[quant] if isinstance(quant, str) else quant
    return load().moe_grouped_gemm_workspace_size(q, T, k, N, Kin, int(a_per_pair))


def moe_mx_quantize(x, rows, cols, codes, scales, ctx=None):
    """fp32 [rows, cols] -> E4M3 codes [rows, cols] + E8M0 scales [rows, cols / 32]."""
    return _check(load().moe_mx_quantize(_ptr(x), rows, cols, _ptr(codes), _ptr(scales), _ctx(ctx)))


def moe_gemm_per_token(E, N, K, a, a_scale, w, w_scale, bias, group_sizes, M, out, ctx=None):
    """out[m] = (a[m] . w[e]^T) * a_scale[m] * w_scale[e] + bias[e] over group-size row ranges."""
    return _check(load().moe_gemm_per_token(E, N, K, _ptr(a), _ptr(a_scale), _ptr(w), _ptr(w_scale),
                                            _ptr(bias), _ptr(group_sizes), M, _ptr(out), _ctx(ctx)))


def moe_wgrad(grad, input, input_per_pair, T, k, E, N, Kin, sorted_token_ids, expert_ids,
              num_tokens_post_padded, block_m, cap_tokens, dW, mode=0, ctx=None):
    return _check(load().moe_wgrad(_ptr(grad), _ptr(input), int(input_per_pair), T, k, E, N, Kin,
                                   _ptr(sorted_token_ids), _ptr(expert_ids),
                                   _ptr(num_tokens_post_padded), block_m, cap_tokens, _ptr(dW),
                                   int(mode), _ctx(ctx)))


def moe_wgrad_workspace_size(E, N, Kin, block_m, cap_tokens, mode=0) -> int:
    return load().moe_wgrad_workspace_size(E, N, Kin, block_m, cap_tokens, int(mode))


def moe_debug_stall_tensor_kernels(stall_ns: int) -> None:
    """Failure-detection self-test switch: with stall_ns > 0 the tensor-memory kernels launch
    with their copy and MMA roles off, so their waits give up after stall_ns ns and report
    MOE_ERR_TIMEOUT; 0 restores normal operation."""
    load().moe_debug_stall_tensor_kernels(int(stall_ns))
