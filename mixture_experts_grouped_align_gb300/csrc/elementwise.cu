// Memory-bound helpers of the path: bucket padding (copy + zero tail), zero fill and the
// top-k combine.  All are grid-stride loops over 16-byte vectors with grids sized as a
// multiple of the SM count.
//
// Pad and slice: "Bound Triton MoE JIT specializations via token-dim bucketing and
// warmup" (TensorRT-LLM PR 15311), Description -- zero rows are appended up to the
// bucket before the grouped GEMMs and removed again before the reduction; the combine
// below only produces the real rows.
#include "moe_common.cuh"
#include "moe_launch.h"
#include "mx_quant.cuh"

namespace {

int grid_for(int64_t work, int threads) {
  const int sms = moe_launch::sm_count_current();
  int64_t need = (work + threads - 1) / threads;
  int64_t cap = (int64_t)sms * 8;
  return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

template <typename V>
__global__ void pad_rows_kernel(const V* __restrict__ src, V* __restrict__ dst, int64_t n_copy,
                                int64_t n_total) {
  const V zero{};
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < n_copy) {
      if (src) dst[i] = src[i];
    } else {
      dst[i] = zero;
    }
  }
}

__global__ void zero_kernel(float4* __restrict__ p, int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// y[t, n] = sum_{j < k} o[t*k + j, n] (j in order), rounded to bf16; 4 columns per thread.
__global__ void combine_kernel(const float4* __restrict__ o, int64_t T_real, int k, int K4,
                               uint2* __restrict__ y) {
  const int64_t n = T_real * K4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / K4;
    const int c = (int)(i - t * K4);
    const float4* src = o + (t * k) * K4 + c;
    float4 acc = __ldg(src);
    for (int j = 1; j < k; ++j) {
      float4 v = __ldg(src + (int64_t)j * K4);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    uint2 out;
    out.x = (uint32_t)moe::f32_to_bf16_bits(acc.x) | ((uint32_t)moe::f32_to_bf16_bits(acc.y) << 16);
    out.y = (uint32_t)moe::f32_to_bf16_bits(acc.z) | ((uint32_t)moe::f32_to_bf16_bits(acc.w) << 16);
    y[i] = out;
  }
}

// y = f16(x) for bf16 x, 8 elements per thread; |x| > 65504 is reported.
__global__ void bf16_to_f16_kernel(const uint4* __restrict__ x, uint4* __restrict__ y, int64_t n8,
                                   int32_t* status) {
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint4 v = __ldg(x + i);
    v.x = moe::bf16x2_to_f16x2(v.x, &bad);
    v.y = moe::bf16x2_to_f16x2(v.y, &bad);
    v.z = moe::bf16x2_to_f16x2(v.z, &bad);
    v.w = moe::bf16x2_to_f16x2(v.w, &bad);
    y[i] = v;
  }
  if (bad) moe::set_status(status, MOE_ERR_RANGE);
}

// y[s] = f16(x[sorted[s] / k]) for the alignment slots s < num_tokens_post_padded (a slot of
// the sentinel gets zeros): the token rows in slot order, so that a block of 128 slots is 128
// consecutive rows.  One warp per slot row (the pair id read once), four 16-byte chunks in
// flight per lane.  |x| > 65504 of a real row is reported.
__global__ void gather_rows_f16_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sorted,
                                       const int32_t* __restrict__ ntpp, int64_t P, int k, int per,
                                       int64_t slots, uint4* __restrict__ y, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t rows = slots < (int64_t)*ntpp ? slots : (int64_t)*ntpp;
  bool bad = false;
  for (int64_t s = warp0; s < rows; s += nwarps) {
    const int p = __ldg(sorted + s);
    const uint4* src = x + (int64_t)(p / k) * per;
    uint4* dst = y + s * per;
    for (int c0 = lane; c0 < per; c0 += 4 * 32) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 32 * j;
        v[j] = (p < P && c < per) ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 32 * j;
        if (c >= per) break;
        v[j].x = moe::bf16x2_to_f16x2(v[j].x, &bad);
        v[j].y = moe::bf16x2_to_f16x2(v[j].y, &bad);
        v[j].z = moe::bf16x2_to_f16x2(v[j].z, &bad);
        v[j].w = moe::bf16x2_to_f16x2(v[j].w, &bad);
        dst[c] = v[j];
      }
    }
  }
  if (bad) moe::set_status(status, MOE_ERR_RANGE);
}

// Rows of `per` 16-byte chunks into alignment-slot order: row s <- src row p / div of the
// pair p in slot s (zeros for the sentinel).  One warp per slot row, four chunks in flight
// per lane.
__global__ void gather_slot_rows_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ sorted,
                                        const int32_t* __restrict__ ntpp, int64_t P, int div, int per,
                                        int64_t slots, uint4* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t rows = slots < (int64_t)*ntpp ? slots : (int64_t)*ntpp;
  for (int64_t s = warp0; s < rows; s += nwarps) {
    const int p = __ldg(sorted + s);
    const uint4* row = src + (int64_t)(p / div) * per;
    uint4* dst = y + s * per;
    for (int c0 = lane; c0 < per; c0 += 4 * 32) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 32 * j;
        v[j] = (p < P && c < per) ? __ldg(row + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (c0 + 32 * j < per) dst[c0 + 32 * j] = v[j];
    }
  }
}

// One thread per 32-element block of a row: 128 bytes in, 32 codes and a scale byte out.
__global__ void mx_quantize_kernel(const float4* __restrict__ x, int64_t nblocks, uint4* __restrict__ codes,
                                   uint8_t* __restrict__ scales) {
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblocks; b += (int64_t)gridDim.x * blockDim.x) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 f = x[b * 8 + i];
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
    uint32_t c[8], s;
    mxq::quant32(v, c, s);
    codes[b * 2] = make_uint4(c[0], c[1], c[2], c[3]);
    codes[b * 2 + 1] = make_uint4(c[4], c[5], c[6], c[7]);
    scales[b] = (uint8_t)s;
  }
}

}  // namespace

namespace moe_launch {

cudaError_t gather_rows_f16(const void* x, const int32_t* sorted, const int32_t* ntpp, int64_t P, int k,
                            int64_t K, int64_t slots, void* y, int32_t* status, cudaStream_t stream) {
  const int64_t per = K / 8;
  if (slots == 0 || per == 0) return cudaSuccess;
  if (per >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  gather_rows_f16_kernel<<<grid_for(slots * 32, 256), 256, 0, stream>>>((const uint4*)x, sorted, ntpp, P, k,
                                                                         (int)per, slots, (uint4*)y, status);
  return cudaGetLastError();
}

cudaError_t gather_slot_rows(const void* src, int64_t row_bytes, const int32_t* sorted, const int32_t* ntpp,
                             int64_t P, int div, int64_t slots, void* y, cudaStream_t stream) {
  const int64_t per = row_bytes / 16;
  if (slots == 0 || per == 0) return cudaSuccess;
  if (per >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  gather_slot_rows_kernel<<<grid_for(slots * 32, 256), 256, 0, stream>>>((const uint4*)src, sorted, ntpp, P, div,
                                                                         (int)per, slots, (uint4*)y);
  return cudaGetLastError();
}

cudaError_t mx_quantize(const float* x, int64_t rows, int cols, uint8_t* codes, uint8_t* scales,
                        cudaStream_t stream) {
  const int64_t nblocks = rows * (cols / 32);
  if (nblocks == 0) return cudaSuccess;
  mx_quantize_kernel<<<grid_for(nblocks, 256), 256, 0, stream>>>((const float4*)x, nblocks, (uint4*)codes, scales);
  return cudaGetLastError();
}

cudaError_t bf16_to_f16(const void* x, void* y, int64_t n, int32_t* status, cudaStream_t stream) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  bf16_to_f16_kernel<<<grid_for(n8, 256), 256, 0, stream>>>((const uint4*)x, (uint4*)y, n8, status);
  return cudaGetLastError();
}

cudaError_t pad_rows(const void* src, void* dst, int64_t rows, int64_t rows_pad, int64_t row_bytes,
                     cudaStream_t stream) {
  const void* s = (src == dst) ? nullptr : src;
  if (row_bytes % 16 == 0) {
    int64_t per = row_bytes / 16;
    int64_t nt = rows_pad * per;
    pad_rows_kernel<uint4><<<grid_for(nt, 256), 256, 0, stream>>>(
        (const uint4*)s, (uint4*)dst, rows * per, nt);
  } else {
    int64_t per = row_bytes / 4;
    int64_t nt = rows_pad * per;
    pad_rows_kernel<uint32_t><<<grid_for(nt, 256), 256, 0, stream>>>(
        (const uint32_t*)s, (uint32_t*)dst, rows * per, nt);
  }
  return cudaGetLastError();
}

cudaError_t zero_f32(float* p, int64_t n, cudaStream_t stream) {
  zero_kernel<<<grid_for(n / 4, 256), 256, 0, stream>>>((float4*)p, n / 4);
  return cudaGetLastError();
}

cudaError_t combine(const float* o, int64_t T_real, int k, int K, void* y, cudaStream_t stream) {
  const int K4 = K / 4;
  const int64_t n = T_real * K4;
  if (n == 0) return cudaSuccess;
  combine_kernel<<<grid_for(n, 256), 256, 0, stream>>>((const float4*)o, T_real, k, K4, (uint2*)y);
  return cudaGetLastError();
}

}  // namespace moe_launch
