// cp.async copies (global -> shared, asynchronous, no register cost for the bytes in flight)
// shared by the kernels that stream operands through shared-memory rings.
#pragma once

#include <stdint.h>

#include "tcgen05.cuh"

namespace cpa {

// 16 bytes, L2 only (.cg); both addresses 16-byte aligned.
MOE_DEV void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
// 16 bytes, or 16 zero bytes when !valid (source size 0: nothing is read).
MOE_DEV void cp_async16z(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz) : "memory");
}
// 4 bytes (.ca); both addresses 4-byte aligned.
MOE_DEV void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
// 4 bytes, or 4 zero bytes when !valid (source size 0: nothing is read).
MOE_DEV void cp_async4z(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(sz) : "memory");
}
MOE_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// Waits until at most N of this thread's committed groups are still in flight.
template <int N>
MOE_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
MOE_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
// Arrives on the mbarrier once every cp.async this thread issued before has landed (the
// barrier's expected count includes this arrival).
MOE_DEV void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_addr(bar)) : "memory");
}

}  // namespace cpa
