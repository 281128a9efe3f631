// Top-k routing and token-to-expert alignment (moe_align_block_size) kernels.
//
// Definitions: "Add MoE GEMM variants and weight-gradient kernel" (aiter PR 5310),
// Summary and second review (sorted_token_ids / expert_ids with -1 sentinel blocks);
// "tune the Nemotron MTP decode row on S5000 with a checked-in recipe" (torchada PR 115),
// What it does (moe_align_block_size as the native op feeding the fused-MoE kernel).
//
// Design: for decode sizes alignment runs in ONE thread block of 32 warps.  Each warp owns a contiguous
// range of pairs; pass 1 builds a private per-warp histogram in shared memory (no
// atomics: __match_any_sync groups lanes of equal expert and the group leader adds the
// group size), pass 2 scans the padded counts over experts and the per-warp counts over
// warps, pass 3 re-walks each range in order and scatters.  Because warps own ordered
// ranges and lanes are ranked inside each 32-pair step, the scatter is stable (ascending
// pair index within an expert) without any order-dependent atomics.  For small T the
// routing runs in the same block (one launch for the whole decode-size step); larger T
// routes with a grid of warps first, and above 16384 pairs the alignment itself runs on a
// grid of blocks (align_multi_kernel, below) with the same result.
#include "moe_common.cuh"
#include "moe_launch.h"

#include <limits.h>
#include <math.h>

namespace {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

struct AlignArgs {
  const float* logits;
  int32_t* ids;
  float* w;
  int64_t T;
  int k, E, bm;
  int32_t* sorted;
  int64_t cap;
  int32_t* expert_ids;
  int32_t* ntpp;
  int32_t* expert_offsets;
  int32_t* status;
  int route_here;
};

// (value, index) order of the top-k: larger value first, lower index on equal values.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return bi == INT_MAX || v > bv || (v == bv && i < bi);
}

// One warp selects one token's top-k: k rounds of a warp arg-max over the unchosen
// logits.  Lane j < k writes the j-th id and, for now, the chosen logit itself into the
// weight slot (the softmax replaces it).  The row is read once into registers (lane holds
// entries lane + 32 i); NPER is the compile-time bound on E / 32.
template <int NPER>
__device__ void select_topk(const float* __restrict__ row, int E, int k,
                            int32_t* __restrict__ ids_out, float* __restrict__ w_out, int lane) {
  float v[NPER];
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
  }
  uint32_t taken = 0;  // bit i <=> entry lane + 32*i already chosen
  float my_val = 0.f;
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    float best = -INFINITY;
    int bidx = INT_MAX;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && better(v[i], e, best, bidx)) {
        best = v[i];
        bidx = e;
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      float ov = __shfl_xor_sync(kFull, best, off);
      int oi = __shfl_xor_sync(kFull, bidx, off);
      if (oi != INT_MAX && better(ov, oi, best, bidx)) { best = ov; bidx = oi; }
    }
    if ((bidx & 31) == lane) taken |= 1u << (bidx >> 5);
    if (lane == j) { my_val = best; my_idx = bidx; }
  }
  if (lane < k) {
    ids_out[lane] = my_idx;
    w_out[lane] = my_val;
  }
}

__device__ void select_topk_any(const float* __restrict__ row, int E, int k, int32_t* __restrict__ ids_out,
                                float* __restrict__ w_out, int lane) {
  if (E <= 64) select_topk<2>(row, E, k, ids_out, w_out, lane);
  else if (E <= 128) select_topk<4>(row, E, k, ids_out, w_out, lane);
  else if (E <= 256) select_topk<8>(row, E, k, ids_out, w_out, lane);
  else select_topk<32>(row, E, k, ids_out, w_out, lane);
}

// One lane turns one token's k chosen logits (descending, in w[0..k)) into routing
// weights: softmax over them in float64, rounded to float32.  The float64 sum follows
// numpy's order for a short vector (a running sum below 8 terms, eight interleaved
// partial sums from 8 on) so that both sides round the same float64 value.  A lane per
// token keeps the (slow) float64 work on all 32 lanes of each instruction.
__device__ void softmax_topk(float* __restrict__ w, int k) {
  const double m = (double)w[0];
  double ex[32];
  for (int j = 0; j < k; ++j) ex[j] = exp((double)w[j] - m);
  double s;
  if (k < 8) {
    s = 0.0;
    for (int j = 0; j < k; ++j) s += ex[j];
  } else {
    double r[8];
    for (int i = 0; i < 8; ++i) r[i] = ex[i];
    int j = 8;
    for (; j + 8 <= k; j += 8)
      for (int i = 0; i < 8; ++i) r[i] += ex[j + i];
    s = ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
    for (; j < k; ++j) s += ex[j];
  }
  for (int j = 0; j < k; ++j) w[j] = __double2float_rn(ex[j] / s);
}

// The same softmax with a warp per token: lane j computes the j-th exponential, and every
// lane forms the float64 sum from the shuffled terms in exactly softmax_topk's order, so the
// bits are the same.  For a handful of tokens this replaces k dependent float64
// exponentials on one lane (float64 is slow on this part) by one per lane; for more tokens
// the warps' mostly idle float64 instructions crowd the SM's float64 pipe (measured: a
// 64-token step's alignment 28.7 -> 41.7 us), so the thread-per-token form stays there.
__device__ void softmax_topk_warp(float* __restrict__ w, int k, int lane) {
  const double m = (double)w[0];
  const double ex = lane < k ? exp((double)w[lane] - m) : 0.0;
  double s;
  if (k < 8) {
    s = 0.0;
    for (int j = 0; j < k; ++j) s += __shfl_sync(kFull, ex, j);
  } else {
    double r[8];
    for (int i = 0; i < 8; ++i) r[i] = __shfl_sync(kFull, ex, i);
    int j = 8;
    for (; j + 8 <= k; j += 8)
      for (int i = 0; i < 8; ++i) r[i] += __shfl_sync(kFull, ex, j + i);
    s = ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
    for (; j < k; ++j) s += __shfl_sync(kFull, ex, j);
  }
  if (lane < k) w[lane] = __double2float_rn(ex / s);
  __syncwarp();
}

// Routes tokens t0 .. t0 + n - 1 (n <= blockDim.x) with the whole thread block: a warp
// per token selects the top-k; then, for at most 8 tokens (one-token decode steps), the same
// warp computes the token's softmax, else (after a block barrier) a thread per token does.
__device__ void route_block(const float* __restrict__ logits, int64_t t0, int n, int E, int k,
                            int32_t* __restrict__ ids, float* __restrict__ w) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const bool warp_soft = n <= 8 && n <= nw;
  for (int i = warp; i < n; i += nw) {
    const int64_t t = t0 + i;
    select_topk_any(logits + t * E, E, k, ids + t * k, w + t * k, lane);
    if (warp_soft) {
      __syncwarp();  // the chosen logits, written by lanes 0..k-1
      softmax_topk_warp(w + t * k, k, lane);
    }
  }
  __syncthreads();
  if (!warp_soft && (int)threadIdx.x < n) softmax_topk(w + (t0 + threadIdx.x) * k, k);
  __syncthreads();
}

__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int64_t T,
                                                    int E, int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ w) {
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x;
  const int n = (int)((T - t0) < (int64_t)blockDim.x ? (T - t0) : (int64_t)blockDim.x);
  route_block(logits, t0, n, E, k, ids, w);
}

// Exclusive scan of v over threads 0..n-1 of the block (n <= 1024); returns the total.
__device__ int block_excl_scan(int v, int* warp_tot, int* out_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
    int xs = t;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(kFull, xs, off);
      if (lane >= off) xs += y;
    }
    warp_tot[lane] = xs - t;  // exclusive prefix of warp totals
    if (lane == 31) *out_total = xs;
  }
  __syncthreads();
  int r = warp_tot[warp] + x - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kAlignThreads, 1) align_kernel(AlignArgs a) {
  extern __shared__ int smem_i[];
  const int E = a.E, bm = a.bm, k = a.k;
  int* hist = smem_i;                     // [32][E]
  int* poff = hist + kAlignWarps * E;     // [E+1] padded offsets
  int* cnt = poff + (E + 1);              // [E]
  int* scratch = cnt + E;                 // [32 + 2]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (a.route_here) route_block(a.logits, 0, (int)a.T, E, k, a.ids, a.w);  // T <= 512
  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) hist[i] = 0;
  __syncthreads();

  const int P = (int)(a.T * k);
  const int chunk = (P + kAlignWarps - 1) / kAlignWarps;
  const int beg = min(P, warp * chunk), end = min(P, beg + chunk);
  int* myhist = hist + warp * E;

  // pass 1: per-warp histogram
  for (int base = beg; base < end; base += 32) {
    const int p = base + lane;
    int e = -1;
    if (p < end) {
      e = a.ids[p];
      if (e < 0 || e >= E) {
        moe::set_status(a.status, MOE_ERR_INVALID_EXPERT);
        e = -1;
      }
    }
    const int key = e >= 0 ? e : (0x40000000 | lane);
    const unsigned grp = __match_any_sync(kFull, key);
    if (e >= 0 && lane == __ffs(grp) - 1) myhist[e] += __popc(grp);
    __syncwarp();
  }
  __syncthreads();

  // pass 2: counts, padded offsets, per-warp bases
  int c = 0, padded = 0;
  if (tid < E) {
    for (int w = 0; w < kAlignWarps; ++w) c += hist[w * E + tid];
    padded = (c + bm - 1) / bm * bm;
  }
  int total_pad, total_cnt;
  int off_pad = block_excl_scan(tid < E ? padded : 0, scratch, scratch + 32);
  total_pad = scratch[32];
  __syncthreads();
  int off_cnt = block_excl_scan(tid < E ? c : 0, scratch, scratch + 33);
  total_cnt = scratch[33];
  if (tid < E) {
    poff[tid] = off_pad;
    cnt[tid] = c;
    int run = off_pad;
    for (int w = 0; w < kAlignWarps; ++w) {
      int t = hist[w * E + tid];
      hist[w * E + tid] = run;
      run += t;
    }
    if (a.expert_offsets) a.expert_offsets[tid] = off_cnt;
  }
  if (tid == 0) {
    poff[E] = total_pad;
    *a.ntpp = total_pad;
    if (a.expert_offsets) a.expert_offsets[E] = total_cnt;
  }
  __syncthreads();

  // pass 3: stable scatter (each warp walks its own range in order)
  for (int base = beg; base < end; base += 32) {
    const int p = base + lane;
    int e = -1;
    if (p < end) {
      e = a.ids[p];
      if (e < 0 || e >= E) e = -1;
    }
    const int key = e >= 0 ? e : (0x40000000 | lane);
    const unsigned grp = __match_any_sync(kFull, key);
    if (e >= 0) {
      const int rank = __popc(grp & ((1u << lane) - 1u));
      a.sorted[myhist[e] + rank] = p;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(grp) - 1) myhist[e] += __popc(grp);
    __syncwarp();
  }
  // sentinel fill of each expert's padding and of the tail up to the capacity: consecutive
  // threads take consecutive slots (coalesced stores); a slot below the padded total is
  // padding when it lies past its expert's pairs
  for (int64_t s = tid; s < a.cap; s += kAlignThreads) {
    bool pad = s >= total_pad;
    if (!pad) {
      int lo = 0, hi = E;  // last e with poff[e] <= s
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (poff[mid] <= s) lo = mid; else hi = mid;
      }
      pad = s >= (int64_t)poff[lo] + cnt[lo];
    }
    if (pad) a.sorted[s] = P;
  }
  // per-block expert ids; -1 past the last used block
  const int64_t cap_blocks = a.cap / bm;
  for (int64_t b = tid; b < cap_blocks; b += kAlignThreads) {
    int64_t s = b * bm;
    int eid = -1;
    if (s < total_pad) {
      int lo = 0, hi = E;  // last e with poff[e] <= s
      while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (poff[mid] <= s) lo = mid; else hi = mid;
      }
      eid = lo;
    }
    a.expert_ids[b] = eid;
  }
}

// The same alignment over many thread blocks, for large pair counts (prefill), without any
// scratch memory or inter-block communication: block b owns the pairs [b * chunk, (b + 1) *
// chunk).  Every block counts the whole id array (the expert totals, for the padded
// offsets) and, separately, the pairs before its own range (its starting rank inside each
// expert); then it scatters its own range exactly as the single-block kernel does, so the
// result is the same, bit for bit.  Sentinel slots and block expert ids are spread over
// all blocks; block 0 writes num_tokens_post_padded and the expert offsets.
__global__ void __launch_bounds__(kAlignThreads, 1) align_multi_kernel(AlignArgs a) {
  extern __shared__ int smem_i[];
  const int E = a.E, bm = a.bm, k = a.k;
  int* hist = smem_i;                     // [32][E] this block's range, per warp
  int* all = hist + kAlignWarps * E;      // [E] every pair
  int* before = all + E;                  // [E] pairs before this block's range
  int* poff = before + E;                 // [E+1] padded offsets
  int* scratch = poff + (E + 1);          // [32 + 2]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) hist[i] = 0;
  for (int i = tid; i < 2 * E; i += kAlignThreads) all[i] = 0;  // all, before
  __syncthreads();

  const int P = (int)(a.T * k);
  const int bchunk = (P + (int)gridDim.x - 1) / (int)gridDim.x;
  const int bbeg = min(P, (int)blockIdx.x * bchunk), bend = min(P, bbeg + bchunk);

  // totals and this block's starting ranks: one pass over every pair, eight loads in flight
  // per thread (the pass is bound by load latency, not by the shared-memory atomics)
  constexpr int kUnroll = 8;
  bool bad = false;
  for (int base = 0; base < P; base += kUnroll * kAlignThreads) {
    int ev[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int p = base + j * kAlignThreads + tid;
      ev[j] = p < P ? __ldg(a.ids + p) : -1;
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int p = base + j * kAlignThreads + tid;
      if (p >= P) continue;
      const int e = ev[j];
      if (e < 0 || e >= E) {
        bad = true;
        continue;
      }
      atomicAdd(&all[e], 1);
      if (p < bbeg) atomicAdd(&before[e], 1);
    }
  }
  if (bad && blockIdx.x == 0) moe::set_status(a.status, MOE_ERR_INVALID_EXPERT);
  // this block's range, per warp (for the stable in-block ranks)
  const int chunk = (bend - bbeg + kAlignWarps - 1) / kAlignWarps;
  const int beg = min(bend, bbeg + warp * chunk), end = min(bend, beg + chunk);
  int* myhist = hist + warp * E;
  for (int base = beg; base < end; base += 32) {
    const int p = base + lane;
    int e = -1;
    if (p < end) {
      e = a.ids[p];
      if (e < 0 || e >= E) e = -1;
    }
    const int key = e >= 0 ? e : (0x40000000 | lane);
    const unsigned grp = __match_any_sync(kFull, key);
    if (e >= 0 && lane == __ffs(grp) - 1) myhist[e] += __popc(grp);
    __syncwarp();
  }
  __syncthreads();

  // padded offsets over experts; each warp's base = expert offset + earlier blocks' pairs +
  // earlier warps' pairs of this block
  const int c = tid < E ? all[tid] : 0;
  const int padded = (c + bm - 1) / bm * bm;
  const int off_pad = block_excl_scan(tid < E ? padded : 0, scratch, scratch + 32);
  const int total_pad = scratch[32];
  __syncthreads();
  const int off_cnt = block_excl_scan(c, scratch, scratch + 33);
  const int total_cnt = scratch[33];
  if (tid < E) {
    poff[tid] = off_pad;
    int run = off_pad + before[tid];
    for (int w = 0; w < kAlignWarps; ++w) {
      const int t = hist[w * E + tid];
      hist[w * E + tid] = run;
      run += t;
    }
    if (blockIdx.x == 0 && a.expert_offsets) a.expert_offsets[tid] = off_cnt;
  }
  if (tid == 0) {
    poff[E] = total_pad;
    if (blockIdx.x == 0) {
      *a.ntpp = total_pad;
      if (a.expert_offsets) a.expert_offsets[E] = total_cnt;
    }
  }
  __syncthreads();

  // stable scatter of this block's range
  for (int base = beg; base < end; base += 32) {
    const int p = base + lane;
    int e = -1;
    if (p < end) {
      e = a.ids[p];
      if (e < 0 || e >= E) e = -1;
    }
    const int key = e >= 0 ? e : (0x40000000 | lane);
    const unsigned grp = __match_any_sync(kFull, key);
    if (e >= 0) {
      const int rank = __popc(grp & ((1u << lane) - 1u));
      a.sorted[myhist[e] + rank] = p;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(grp) - 1) myhist[e] += __popc(grp);
    __syncwarp();
  }
  // sentinel slots and block expert ids, spread over the grid
  const int64_t gtid = (int64_t)blockIdx.x * kAlignThreads + tid, gstride = (int64_t)gridDim.x * kAlignThreads;
  for (int64_t s = gtid; s < a.cap; s += gstride) {
    bool pad = s >= total_pad;
    if (!pad) {
      int lo = 0, hi = E;  // last e with poff[e] <= s
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (poff[mid] <= s) lo = mid; else hi = mid;
      }
      pad = s >= (int64_t)poff[lo] + all[lo];
    }
    if (pad) a.sorted[s] = P;
  }
  const int64_t cap_blocks = a.cap / bm;
  for (int64_t b = gtid; b < cap_blocks; b += gstride) {
    const int64_t s = b * bm;
    int eid = -1;
    if (s < total_pad) {
      int lo = 0, hi = E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (poff[mid] <= s) lo = mid; else hi = mid;
      }
      eid = lo;
    }
    a.expert_ids[b] = eid;
  }
}

}  // namespace

namespace moe_launch {

size_t align_smem_bytes(int E) { return sizeof(int) * ((size_t)kAlignWarps * E + 3 * E + 1 + 34); }

cudaError_t align(const float* logits, int32_t* ids, float* w, int64_t T, int k, int E, int bm,
                  int32_t* sorted, int64_t cap, int32_t* expert_ids, int32_t* ntpp,
                  int32_t* expert_offsets, int32_t* status, cudaStream_t stream) {
  AlignArgs a{logits, ids, w, T, k, E, bm, sorted, cap, expert_ids, ntpp, expert_offsets,
              status, 0};
  constexpr int64_t kFuseT = 512;
  if (logits) {
    if (T <= kFuseT) {
      a.route_here = 1;
    } else {
      const int64_t tok_per_block = 256;  // 8 warps; 32 tokens per warp, a thread per token
      route_kernel<<<(unsigned)((T + tok_per_block - 1) / tok_per_block), 256, 0, stream>>>(
          logits, T, E, k, ids, w);
      cudaError_t err = cudaGetLastError();
      if (err != cudaSuccess) return err;
    }
  }
  const size_t smem = align_smem_bytes(E);
  // Above kMultiPairs pairs (prefill) the grid version: one block per 4096 pairs, at most one
  // per SM.  Both kernels write the same bits, so the choice cannot break padded = unpadded.
  constexpr int64_t kMultiPairs = 16384;
  const int64_t P = T * k;
  if (P > kMultiPairs && !a.route_here) {
    cudaError_t err = cudaFuncSetAttribute(align_multi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    int64_t blocks = (P + 4095) / 4096;
    const int sms = sm_count_current();
    if (blocks > sms) blocks = sms;
    align_multi_kernel<<<(unsigned)blocks, kAlignThreads, smem, stream>>>(a);
    return cudaGetLastError();
  }
  cudaError_t err = cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  align_kernel<<<1, kAlignThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe_launch
