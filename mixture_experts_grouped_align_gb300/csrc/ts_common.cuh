// Helpers shared by the grouped GEMMs that decode W4A16 weights into tensor memory (the
// A operand of tcgen05.mma kind::f16): E2M1 codes times the E8M0 block scale to f16, the
// TMEM store of a decoded block, the TS-form MMA and the four-row TMA gather of token rows.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "tcgen05.cuh"

namespace ts {

// TMA gather of four 128-byte rows (rows y0..y3 of the tensor, bytes x..x+127) to dst.
MOE_DEV void tma_gather4(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y0, int32_t y1, int32_t y2,
                         int32_t y3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(tc::smem_addr(bar))
      : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T (kind::f16), issued by one thread.
MOE_DEV void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

MOE_DEV uint32_t hmul2_u32(uint32_t v, __half2 s) {
  __half2 h = __hmul2(*reinterpret_cast<__half2*>(&v), s);
  return *reinterpret_cast<uint32_t*>(&h);
}

// f16x2 holding 2^(s-127) in both halves: NaN for 0xFF; the exponent clamped to the f16
// range (a block whose nonzero codes need a scale outside 2^-23..2^13 is reported, and all-zero
// codes stay zero under any finite scale).
MOE_DEV __half2 scale_h2(uint32_t sb) {
  if (sb == 255u) return __half2half2(__ushort_as_half((unsigned short)0x7e00u));
  int se = (int)sb - 127;
  se = se < -24 ? -24 : (se > 15 ? 15 : se);
  const unsigned short bits = se >= -14 ? (unsigned short)((se + 15) << 10) : (unsigned short)(1u << (se + 24));
  return __half2half2(__ushort_as_half(bits));
}

// 16 E2M1 codes of one 32-element block (16 bytes, low nibble first) -> 16 f16x2 words scaled.
MOE_DEV void decode_block(const uint4 w, uint32_t sb, uint32_t* out, bool& bad) {
  const int se = (int)sb - 127;
  if ((w.x | w.y | w.z | w.w) && sb != 255u && (se < -23 || se > 13)) bad = true;
  const __half2 s2 = scale_h2(sb);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t o0, o1, o2, o3;
    moe::e2m1x8_to_f16x2(ws[q], o0, o1, o2, o3);
    out[4 * q + 0] = hmul2_u32(o0, s2);
    out[4 * q + 1] = hmul2_u32(o1, s2);
    out[4 * q + 2] = hmul2_u32(o2, s2);
    out[4 * q + 3] = hmul2_u32(o3, s2);
  }
}

// r[0..15] -> TMEM columns c..c+15 of this thread's lane (32 lanes x 16 columns per warp).
MOE_DEV void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

}  // namespace ts
