// Inline-PTX wrappers for the sm_100-family tensor-core path: mbarriers with bounded
// waits, tensor memory (TMEM) allocation and loads, tcgen05.mma and the shared-memory
// matrix descriptors of 128-byte-swizzled K-major tiles.
#pragma once

#include <stdint.h>

#include "moe_common.cuh"

namespace tc {

MOE_DEV uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

MOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

MOE_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

MOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

MOE_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Default limit of a bounded wait: 2 s, far beyond any stage of a healthy kernel.
constexpr uint64_t kWaitNs = 2000000000ull;

// Waits for the phase with the given parity to complete.  Gives up after about
// `budget_ns` nanoseconds (globaltimer) and returns false; never spins forever.
MOE_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > budget_ns) return false;
  }
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (tensor core) reads of the same memory.
MOE_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMEM

// One warp allocates `ncols` (power of two >= 32) TMEM columns; the base address is
// written to *dst (shared memory).
MOE_DEV void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
MOE_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 columns of 32-bit TMEM -> 32 registers per thread (thread i = lane i of
// the warp's 32-lane TMEM quarter, register j = column j).
MOE_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
MOE_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Registers -> TMEM: thread i writes lane i of the warp's 32-lane quarter, columns c..c+3
// (x4) or c..c+7 (x8) from r[0..].
MOE_DEV void tmem_st4(uint32_t taddr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r0),
               "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}
MOE_DEV void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// Waits until this thread's tcgen05.st writes have completed.
MOE_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- MMA

// Shared-memory matrix descriptor of a K-major operand tile stored in 128-byte swizzle
// atoms (8 rows x 128 B, 1024 B per atom, atoms of consecutive 8-row groups adjacent):
// start address >> 4 in bits 0-13, leading byte offset (unused for this layout) 16-29,
// stride byte offset (1024 B between 8-row groups) >> 4 in 32-45, the fixed value 1 in
// bits 46-48, swizzle mode 2 (128 B) in bits 61-63.
MOE_DEV uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                 // leading byte offset (16 B), ignored here
  d |= (uint64_t)(1024u >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1u << 46;                 // descriptor version for tcgen05
  d |= (uint64_t)2u << 61;                 // 128-byte swizzle
  return d;
}

// Descriptor of an MN-major operand tile in 128-byte swizzle atoms (64 MN elements x 8
// K rows, 1024 B each): leading byte offset = distance between atoms along MN, stride
// byte offset = distance between 8-row groups along K.
MOE_DEV uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: f32 accumulator, A and B both f16
// (ab_fmt 0) or both bf16 (ab_fmt 1), both K-major, N >> 3 in bits 17-22, M >> 4 in bits
// 24-28.
MOE_DEV uint32_t idesc_f16(int M, int N, uint32_t ab_fmt) {
  uint32_t d = 0;
  d |= 1u << 4;                // D format: f32
  d |= ab_fmt << 7;            // A format
  d |= ab_fmt << 10;           // B format
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

// D[tmem] (+)= A[smem] . B[smem]^T, issued by one thread.
MOE_DEV void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4.block_scale: E4M3 A and B, both
// K-major, f32 accumulator, UE8M0 scale factors; the scale-factor ids pick the byte of
// the 32-bit TMEM scale words this MMA uses (B in bits 4-5, A in bits 29-30), N >> 3 in
// bits 17-22, scale type UE8M0 in bit 23, M >> 4 in bits 24-28.
MOE_DEV uint32_t idesc_mx8(int M, int N, uint32_t sf_id_a, uint32_t sf_id_b) {
  uint32_t d = 0;
  d |= (sf_id_b & 3u) << 4;
  d |= (uint32_t)(N >> 3) << 17;
  d |= 1u << 23;
  d |= (uint32_t)(M >> 4) << 24;
  d |= (sf_id_a & 3u) << 29;
  return d;
}

// D[tmem] (+)= (A . SFA)[smem] . (B . SFB)[smem]^T with one E8M0 scale per 32 K elements
// of every A row and B row, read from TMEM; issued by one thread.
MOE_DEV void mma_mx8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa_tmem,
                        uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of tcgen05.mma.kind::mxf4.block_scale: E2M1 A and B (type code 1
// in bits 7-9 and 10-12), both K-major and packed two codes a byte, f32 accumulator, UE8M0
// scale factors (bit 23).  Each MMA covers K = 64, i.e. two 32-element scale blocks, whose
// factors are bytes sf_id and sf_id + 1 (sf_id 0 or 2) of the rows' TMEM scale words.
MOE_DEV uint32_t idesc_mxf4(int M, int N, uint32_t sf_id_a, uint32_t sf_id_b) {
  uint32_t d = 0;
  d |= (sf_id_b & 3u) << 4;
  d |= 1u << 7;
  d |= 1u << 10;
  d |= (uint32_t)(N >> 3) << 17;
  d |= 1u << 23;
  d |= (uint32_t)(M >> 4) << 24;
  d |= (sf_id_a & 3u) << 29;
  return d;
}

// D[tmem] (+)= (A . SFA)[smem] . (B . SFB)[smem]^T for packed E2M1 A and B, one E8M0 scale
// per 32 K elements of every row, read from TMEM; issued by one thread.
MOE_DEV void mma_mxf4_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa_tmem,
                         uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Arrives (once) on the mbarrier when every tcgen05 operation this thread issued before
// has completed.
MOE_DEV void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// mma_commit onto the mbarrier at the same shared-memory offset in every CTA of the cluster
// in cta_mask.
MOE_DEV void mma_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(cta_mask)
      : "memory");
}

// ---------------------------------------------------------------- clusters

MOE_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster (warp-converged): release this CTA's prior
// shared-memory writes (mbarrier inits included) to the cluster, then wait for the others.
MOE_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a tile of 128-byte rows stored in
// 128-byte swizzle atoms.
MOE_DEV uint32_t sw128_offset(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

}  // namespace tc
