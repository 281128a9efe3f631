"""CPU oracle of the MoE expert-layer hot path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 restatement of what the layer computes, written from the
definitions on three pull-request pages:

* "Bound Triton MoE JIT specializations via token-dim bucketing and warmup"
  (TensorRT-LLM PR 15311): geometric token-dimension bucketing, pad-and-slice, and
  the W4A16-only restriction (Description; Test Coverage).
* "tune the Nemotron MTP decode row on S5000 with a checked-in recipe"
  (torchada PR 115): the tiny-M bf16 fused-MoE decode shape (What it does).
* "Add MoE GEMM variants and weight-gradient kernel" (ROCm aiter PR 5310):
  single-launch block-scaled grouped GEMM with E8M0 microscales and optional per-expert
  bias, and the weight gradient dW[e] = sum over tokens routed to e of grad^T x read
  from the alignment outputs (Summary; Notes; second review: sentinel handling,
  E8M0 decoding, bias indexing).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library and never imports it.

Modules: ``formats`` (E2M1 / E4M3 / E8M0 / bf16 decoding), ``route`` (top-k routing),
``align`` (token-to-expert alignment), ``bucket`` (token-dimension buckets and padding),
``layer`` (grouped GEMMs, SwiGLU, combine), ``wgrad`` (per-expert weight gradient).
Every function is pinned by ``tests/test_oracle_*.py`` against closed forms, library
routines, brute force on tiny inputs or properties the pages state.
"""
from . import formats, route, align, bucket, layer, wgrad  # noqa: F401
