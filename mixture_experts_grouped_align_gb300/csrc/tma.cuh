// Tensor-memory-accelerator (TMA) copies: a host helper that encodes a 2-D byte tensor map
// and the device instructions that load one box of it into shared memory, completing on
// an mbarrier by transaction bytes.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tcgen05.cuh"

namespace tma {

// 2-D tensor of bytes: `outer` rows of `inner` bytes, consecutive rows `row_stride` bytes
// apart; boxes of box_inner x box_outer land in shared memory in the 128-byte swizzle
// (box_inner == 128) or unswizzled.  Returns false when the driver entry point is missing
// or the encoding is rejected (base not 16-byte aligned, stride not a multiple of 16, ...).
inline bool encode_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride,
                         uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (encode == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE,
                            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Arrives on the mbarrier and adds `bytes` to the transaction count its phase waits for.
MOE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Loads the box at (x = byte offset within a row, y = row) into shared memory at dst; the
// bytes complete on `bar`.  x must be a multiple of 16.
MOE_DEV void load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_addr(bar))
      : "memory");
}

// load_2d into the same shared-memory offset of every CTA of the cluster in cta_mask; each
// destination's mbarrier at the offset of `bar` receives the box's bytes.
MOE_DEV void load_2d_multicast(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar,
                               uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_addr(bar)), "h"(cta_mask)
      : "memory");
}

// L2 cache policies for the copies below: lines that should leave L2 first (data written
// once and not read again soon) or last (data read again by other tiles).
MOE_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// load_2d with an L2 cache policy for the lines it reads.
MOE_DEV void load_2d_hint(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar,
                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_addr(bar)), "l"(policy)
      : "memory");
}
// load_2d_multicast with an L2 cache policy.
MOE_DEV void load_2d_multicast_hint(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar,
                                    uint16_t cta_mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5, %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_addr(bar)), "h"(cta_mask), "l"(policy)
      : "memory");
}
// store_2d with an L2 cache policy for the lines it writes.
MOE_DEV void store_2d_hint(const CUtensorMap* map, int32_t x, int32_t y, uint32_t src, uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "l"(policy)
               : "memory");
}

// Stores the box at (x, y) of the tensor from shared memory at src (bulk-group completion).
MOE_DEV void store_2d(const CUtensorMap* map, int32_t x, int32_t y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
MOE_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the shared memory of every committed bulk store of this thread has been read.
MOE_DEV void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until the shared memory of all but the most recent committed bulk store of this
// thread has been read.
MOE_DEV void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Waits until every committed bulk store of this thread has completed.
MOE_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Starts bringing the box at (x, y) of the tensor into L2 (no shared memory, no completion).
MOE_DEV void prefetch_2d_l2(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

MOE_DEV void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace tma
