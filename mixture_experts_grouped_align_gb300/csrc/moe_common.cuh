// Shared device helpers of the MoE kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moe_gb300.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

// First data-dependent error wins; nothing traps.
MOE_DEV void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// E8M0 scale byte -> float: 2^(e-127); 0x00 is 2^-127 (a float32 subnormal, bits
// 0x00400000), 0xFF is NaN.  A plain (e << 23) would give 0 and +inf for those two.
MOE_DEV float e8m0_to_f32(uint32_t e) {
  if (e == 0u) return __uint_as_float(0x00400000u);
  if (e == 255u) return __uint_as_float(0x7fc00000u);
  return __uint_as_float(e << 23);
}

// Two E2M1 codes (low nibble = first element) -> f16x2, exact (hardware conversion).
MOE_DEV uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(out) : "r"(byte));
  return out;
}

// Eight E2M1 codes (two per byte, low nibble first) -> four f16x2, exact (hardware
// conversions; the byte unpack costs nothing extra).
MOE_DEV void e2m1x8_to_f16x2(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2, uint32_t& o3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}

// Four E4M3 codes -> two f16x2, exact.
MOE_DEV void e4m3x4_to_f16x2(uint32_t w, uint32_t& o0, uint32_t& o1) {
  asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\tcvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
      : "=r"(o0), "=r"(o1)
      : "r"(w));
}

// Two E4M3 codes (low byte = first element) -> f16x2, exact (hardware conversion).
MOE_DEV uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t out;
  asm("{\n\t.reg .b16 h;\n\tcvt.u16.u32 h, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}"
      : "=r"(out) : "r"(two_bytes));
  return out;
}

// bf16x2 -> f16x2 (exact when |v| is in [2^-14, 65504] or zero; smaller magnitudes round
// to float16 subnormals).  *bad is set when a magnitude exceeds 65504.
MOE_DEV uint32_t bf16x2_to_f16x2(uint32_t v, bool* bad) {
  float lo = __uint_as_float(v << 16);
  float hi = __uint_as_float(v & 0xffff0000u);
  if (fabsf(lo) > 65504.f || fabsf(hi) > 65504.f) *bad = true;
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// f16x2 -> bf16x2 (round to nearest even).
MOE_DEV uint32_t f16x2_to_bf16x2(uint32_t v) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&b);
}

MOE_DEV float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

MOE_DEV uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// m16n8k16 tensor-core MMA, f16 inputs, f32 accumulate: D = A.B + C.
MOE_DEV void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                     const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// m16n8k16 tensor-core MMA, bf16 inputs, f32 accumulate.
MOE_DEV void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                      const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// Streaming read-only loads (weights are read once per layer).
MOE_DEV uint32_t ldg_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
MOE_DEV uint2 ldg_nc_u64(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
MOE_DEV uint4 ldg_nc_u128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// silu(g) = g * sigmoid(g) with the hardware exponential and reciprocal (relative error
// near 1e-6, far below the f16 / bf16 rounding of the value it feeds); 0 for g -> -inf.
MOE_DEV float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// relu(a)^2, exact up to the one rounding of the product; a NaN passes through.
MOE_DEV float relu2(float a) {
  const float r = a < 0.f ? 0.f : a;
  return r * r;
}

}  // namespace moe

// Host-side error reporting shared by the translation units.
namespace moe_host {
void set_error(const char* fmt, ...);
}
