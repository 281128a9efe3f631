// Per-expert weight gradient dW[e] = sum over pairs p of expert e of grad[p]^T input[src(p)].
//
// "Add MoE GEMM variants and weight-gradient kernel" (aiter PR 5310), Summary (moe_wgrad):
// the gradient is read straight from the alignment outputs (sorted_token_ids /
// expert_ids) with no sort + pad + batched GEMM and no host synchronisation; Tests &
// Benchmarks: constant input, linearity, zero-padded tokens contribute nothing.
//
// Tile: a 64 (N) x 64 (Kin) block of dW[e] per thread block, accumulated in float32 by
// m16n8k16 bf16 tensor-core MMAs over the expert's token slots, 32 slots per stage.  Both
// operands are "transposed" relative to the MMA (the token index is the reduction index
// and is the slow index of grad and input), so tiles are staged token-major in shared
// memory with cp.async (sentinel slots are zero-filled) and read with ldmatrix.trans.
// Deterministic mode: one block per (expert, tile) walks all of the expert's slots in
// order and stores its tile (zeros for an expert with no pair).  Accumulate mode: one
// block per (alignment block, tile) adds its partial tile with float atomics into a dW the
// launcher zeroed first.
#include "moe_common.cuh"
#include "moe_launch.h"

namespace {

using namespace moe_launch;

constexpr int kTM = 64, kTN = 64, kTK = 32;  // N rows, Kin cols, token slots per stage
constexpr int kLd = 72;                       // shared row stride (bf16): 144 B, conflict-free
constexpr int kThreads = 128;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;  // 0 bytes read -> 16 zero bytes written
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;\n"); }

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

struct Tiles {
  uint16_t g[2][kTK][kLd];  // grad rows   [slot][n]
  uint16_t x[2][kTK][kLd];  // input rows  [slot][kin]
};

// Loads one stage: 32 slots x 64 columns of grad and of input (8 x 16 B per row).
__device__ __forceinline__ void load_stage(Tiles& t, int buf, const Wgrad& a, int64_t slot_beg,
                                           int64_t slot_end, int n0, int c0) {
  const uint16_t* grad = static_cast<const uint16_t*>(a.grad);
  const uint16_t* inp = static_cast<const uint16_t*>(a.input);
  for (int i = threadIdx.x; i < kTK * 8 * 2; i += kThreads) {
    const int which = i / (kTK * 8);
    const int r = (i / 8) % kTK, ch = i % 8;
    const int64_t s = slot_beg + r;
    int64_t p = a.P;
    if (s < slot_end) p = a.sorted[s];
    const bool valid = p < a.P;
    if (which == 0) {
      const uint16_t* src = valid ? grad + p * a.N + n0 + ch * 8 : grad;
      cp_async16(&t.g[buf][r][ch * 8], src, valid);
    } else {
      const int64_t row = a.input_per_pair ? p : p / a.k;
      const uint16_t* src = valid ? inp + row * a.Kin + c0 + ch * 8 : inp;
      cp_async16(&t.x[buf][r][ch * 8], src, valid);
    }
  }
}

template <bool ATOMIC>
__global__ void __launch_bounds__(kThreads) wgrad_kernel(Wgrad a) {
  __shared__ __align__(16) Tiles t;
  const int c0 = blockIdx.x * kTN;
  const int n0 = blockIdx.y * kTM;
  int64_t e, slot_beg, slot_end;
  const int ntpp = *a.ntpp;
  const int nblocks = ntpp / a.bm;
  if (ATOMIC) {
    const int64_t b = blockIdx.z;
    if (b >= nblocks) return;
    e = a.expert_ids[b];
    if (e < 0 || e >= a.E) return;
    slot_beg = b * a.bm;
    slot_end = slot_beg + a.bm;
  } else {
    e = blockIdx.z;
    // the expert's blocks: expert_ids is ascending over [0, nblocks)
    int lo = 0, hi = nblocks;
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if (a.expert_ids[mid] < e) lo = mid + 1; else hi = mid;
    }
    int lo2 = lo, hi2 = nblocks;
    while (lo2 < hi2) {
      int mid = (lo2 + hi2) >> 1;
      if (a.expert_ids[mid] <= e) lo2 = mid + 1; else hi2 = mid;
    }
    slot_beg = (int64_t)lo * a.bm;
    slot_end = (int64_t)lo2 * a.bm;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = (warp >> 1) * 32, wn = (warp & 1) * 32;
  float acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.f;

  const int64_t nst = (slot_end - slot_beg + kTK - 1) / kTK;
  if (nst > 0) {
    load_stage(t, 0, a, slot_beg, slot_end, n0, c0);
    cp_async_commit();
  }
  for (int64_t st = 0; st < nst; ++st) {
    const int buf = (int)(st & 1);
    if (st + 1 < nst) {
      load_stage(t, buf ^ 1, a, slot_beg + (st + 1) * kTK, slot_end, n0, c0);
      cp_async_commit();
      cp_async_wait_1();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
#pragma unroll
    for (int ks = 0; ks < kTK; ks += 16) {
      uint32_t af[2][4], bfr[2][4];
      const int li = lane >> 3, lr = lane & 7;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)  // matrix li: k half (li >> 1), m half (li & 1)
        ldsm_x4_t(af[mt], &t.g[buf][ks + (li >> 1) * 8 + lr][wm + mt * 16 + (li & 1) * 8]);
#pragma unroll
      for (int np = 0; np < 2; ++np)  // matrix li: k half (li & 1), n half (li >> 1)
        ldsm_x4_t(bfr[np], &t.x[buf][ks + (li & 1) * 8 + lr][wn + np * 16 + (li >> 1) * 8]);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          moe::mma_bf16(acc[mt][nt], af[mt], bfr[nt >> 1][(nt & 1) * 2],
                        bfr[nt >> 1][(nt & 1) * 2 + 1], acc[mt][nt]);
    }
    __syncthreads();
  }

  const int g = lane >> 2, q = lane & 3;
  float* out = a.dW + (e * a.N + n0) * (int64_t)a.Kin + c0;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = wm + mt * 16 + g + h * 8;
        const int c = wn + nt * 8 + 2 * q;
        float2 v = make_float2(acc[mt][nt][2 * h], acc[mt][nt][2 * h + 1]);
        float2* dst = reinterpret_cast<float2*>(out + (int64_t)r * a.Kin + c);
        if (ATOMIC) atomicAdd(dst, v); else *dst = v;
      }
}

}  // namespace

namespace moe_launch {

cudaError_t wgrad(const Wgrad& g, cudaStream_t stream) {
  dim3 block(kThreads);
  if (g.mode == 0 && wgrad_tc_tile(g) > 0) return wgrad_tc(g, stream);
  if (g.mode == 0) {
    dim3 grid(g.Kin / kTN, g.N / kTM, g.E);
    wgrad_kernel<false><<<grid, block, 0, stream>>>(g);
  } else {
    cudaError_t err = zero_f32(g.dW, (int64_t)g.E * g.N * g.Kin, stream);
    if (err != cudaSuccess) return err;
    if (g.cap_blocks == 0) return cudaSuccess;
    dim3 grid(g.Kin / kTN, g.N / kTM, (unsigned)g.cap_blocks);
    wgrad_kernel<true><<<grid, block, 0, stream>>>(g);
  }
  return cudaGetLastError();
}

}  // namespace moe_launch
