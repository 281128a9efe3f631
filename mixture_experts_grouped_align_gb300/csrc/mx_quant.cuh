// MXFP8 quantisation of 32 float values: one E8M0 scale and 32 E4M3 codes, the OCP
// microscaling rule for E4M3 elements (largest element exponent 8): scale 2^e with
// e = floor(log2(amax)) - 8 clamped to [-127, 127] (-127 for an all-zero block), codes
// round-to-nearest-even of v / 2^e saturating at 448 (hardware conversion).  A block holding
// a NaN gets the NaN scale 0xFF and NaN codes 0x7F.  The division by 2^e is exact, so the
// codes depend only on the float32 inputs.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

#include "moe_common.cuh"

namespace mxq {

// Block exponent of a non-negative float32 maximum (inf -> 127).
MOE_DEV int block_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int ex = (int)((b >> 23) & 0xffu);
  int e;
  if (amax == 0.f) e = -127;
  else if (ex == 255) e = 127;
  else if (ex == 0) e = (31 - __clz((int)(b & 0x7fffffu))) - 149 - 8;  // subnormal maximum
  else e = ex - 127 - 8;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// v[0..31] -> codes (packed four per word, element 4 i + j in byte j of word i) and scale byte.
MOE_DEV void quant32(const float* v, uint32_t* codes, uint32_t& scale) {
  float amax = 0.f;
  bool nan = false;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    nan |= (v[i] != v[i]);
    amax = fmaxf(amax, fabsf(v[i]));
  }
  if (nan) {
    scale = 255u;
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = 0x7f7f7f7fu;
    return;
  }
  const int e = block_exponent(amax);
  scale = (uint32_t)(e + 127);
  // 2^-e: a normal float for e <= 126; 2^-127 (only for an infinite maximum) is subnormal
  const float inv = e >= 127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      w |= (uint32_t)__nv_cvt_float_to_fp8(v[4 * i + j] * inv, __NV_SATFINITE, __NV_E4M3) << (8 * j);
    codes[i] = w;
  }
}

}  // namespace mxq
