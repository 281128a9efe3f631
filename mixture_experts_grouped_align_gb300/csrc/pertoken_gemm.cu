// Per-token FP8 grouped GEMM with the rows of each expert given by group sizes.
//
// out[m, n] = bf16( (sum_k A[m, k] * W[e, n, k]) * a_scale[m] * w_scale[e] + bias[e, n] ) for
// the rows m of expert e, O_e <= m < O_e + g_e with O_e = g_0 + ... + g_{e-1} ("Add MoE GEMM
// variants and weight-gradient kernel", aiter PR 5310, Summary: moe_gemm_per_token -- per-token
// activation scales and per-expert weight scales applied after the FP8 dot product, a 1-D
// tensor of per-expert token counts instead of an alignment).  tcgen05.mma kind::f8f6f4 takes
// the E4M3 codes of both operands from shared memory and accumulates their exact products in
// f32; the two scales and the bias are applied in the epilogue.
//
// Per thread block (one per SM, 512 threads), persistent over (row block, N tile):
//   all threads first turn the group sizes into the running row offsets O_e and the running
//   counts of 128-row blocks, so that tile t's expert is a binary search away;
//   warp 0      allocates two TMEM accumulators (128 x BN f32 each, used in turn so that
//               a tile's epilogue overlaps the next tile's MMAs) and, on one lane, issues
//               the MMAs (M = 128, N = BN, K = 32; four per 128-wide K stage);
//   warps 8-15  copy each stage: one thread loads the BN weight rows of 128 bytes with a TMA
//               box into a 128-byte-swizzled K-major tile; all copy the block's activation
//               rows (contiguous: one expert's rows are consecutive) with cp.async into the
//               same layout, and hand the stage to the MMA two stages later;
//   warps 4-7   drain the accumulator (one TMEM lane = one row), apply the row's and the
//               expert's scales and the bias, and store bf16 rows.
// Experts with no rows produce no tile.  Group sizes that are negative or that add up to more
// than the M rows set MOE_ERR_CAPACITY in the status word; rows past M are never touched.
// Every mbarrier wait is bounded; one that runs out sets MOE_ERR_TIMEOUT, every role leaves
// its loop, the MMA lane drains its own work and the TMEM is freed.
#include "moe_common.cuh"
#include "cp_async.cuh"
#include "moe_launch.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace {

using namespace moe_launch;
using namespace cpa;

constexpr int kThreads = 512;
constexpr int kBM = 128, kBK = 128;        // tile rows, K elements (bytes) per stage
constexpr int kProd0 = 256, kNumProd = 256;
constexpr int kEpiWarp0 = 4;
constexpr int kTmemCols = 512;               // two accumulators of up to 256 columns
constexpr int kStages = 4;
constexpr int kLag = 2;                    // stages between a stage's copies and its hand-over
constexpr int kMaxE = 1024;

// One stage slot: A tile (128 rows x 128 B) | B tile (BN rows x 128 B); then the expert
// tables (row offsets and block offsets, E + 1 each) and the barriers.
struct PLayout {
  int a, b, slot, tables, bars, total;
};

__host__ __device__ inline PLayout playout(int BN) {
  PLayout L;
  L.a = 0;
  L.b = kBM * kBK;
  L.slot = L.b + BN * kBK;  // a multiple of 1024
  L.tables = kStages * L.slot;
  L.bars = L.tables + (kMaxE + 1) * 8 + (kMaxE + 1) * 4;
  L.bars = (L.bars + 15) & ~15;
  L.total = L.bars + 256 + 1024;
  return L;
}

struct PTArgs {
  const uint8_t* a;        // [M, K] E4M3
  const float* a_scale;    // [M]
  const void* w;           // [E, N, K] E4M3 (read through the tensor map)
  const float* w_scale;    // [E]
  const uint16_t* bias;    // [E, N] bf16 or null
  const int32_t* group_sizes;
  uint16_t* out;           // [M, N] bf16
  int32_t* status;
  int64_t M;
  int E, N, K, BN, n_tiles;
  int64_t tiles;           // upper bound of row blocks (ceil(M / 128) + E) * n_tiles
};

// D[tmem] (+)= A[smem] . B[smem]^T, E4M3 x E4M3 -> f32 (kind::f8f6f4), issued by one thread.
__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Tile t: row block b and N tile nt; the expert e of the block and its rows [r0, r1).
struct Tile {
  int e, nt;
  int64_t r0, r1;
};

__device__ __forceinline__ bool tile_of(const PTArgs& pa, int64_t t, const int64_t* roff, const int32_t* boff,
                                        int nblocks, Tile& tl) {
  const int64_t b = t / pa.n_tiles;
  if (b >= nblocks) return false;
  tl.nt = (int)(t - b * pa.n_tiles);
  int lo = 0, hi = pa.E;  // the last e with boff[e] <= b (experts without rows own no block)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (boff[mid] <= b) lo = mid;
    else hi = mid;
  }
  tl.e = lo;
  tl.r0 = roff[lo] + (b - boff[lo]) * (int64_t)kBM;
  tl.r1 = tl.r0 + kBM < roff[lo + 1] ? tl.r0 + kBM : roff[lo + 1];
  return true;
}

__global__ void __launch_bounds__(kThreads, 1) pertoken_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                                                     PTArgs pa) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = pa.BN;
  const PLayout L = playout(BN);
  int64_t* roff = reinterpret_cast<int64_t*>(smem + L.tables);  // [E + 1] row offsets
  int32_t* boff = reinterpret_cast<int32_t*>(roff + (kMaxE + 1));  // [E + 1] block offsets
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;  // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint64_t* drain = tempty + 2;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_s + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], kNumProd / 32 + 1);  // producer warps + the weight box
      tc::mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], 4);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(taddr_s, kTmemCols);
    tc::tmem_relinquish();
  } else if (warp == 1) {
    // running row and block offsets over the experts, 32 experts per step; a negative size
    // counts as zero, and rows past M are cut off (both reported)
    int64_t rows = 0;
    int32_t blocks = 0;
    bool bad = false;
    for (int e0 = 0; e0 < pa.E; e0 += 32) {
      const int e = e0 + lane;
      int64_t gsz = e < pa.E ? (int64_t)pa.group_sizes[e] : 0;
      if (gsz < 0) {
        bad = true;
        gsz = 0;
      }
      int64_t incl = gsz;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int64_t start = rows + incl - gsz;
      if (start > pa.M) start = pa.M;
      int64_t end = rows + incl;
      if (end > pa.M) {
        end = pa.M;
        bad = true;
      }
      const int32_t nb = (int32_t)((end - start + kBM - 1) / kBM);
      int32_t binc = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, binc, o);
        if (lane >= o) binc += v;
      }
      if (e < pa.E) {
        roff[e] = start;
        boff[e] = blocks + binc - nb;
      }
      rows += __shfl_sync(0xffffffffu, incl, 31);
      blocks += __shfl_sync(0xffffffffu, binc, 31);
    }
    if (lane == 0) {
      roff[pa.E] = rows < pa.M ? rows : pa.M;
      boff[pa.E] = blocks;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0) moe::set_status(pa.status, MOE_ERR_CAPACITY);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t taddr = *taddr_s;
  const int nblocks = boff[pa.E];
  const int nk = pa.K / kBK;
  const uint32_t smem_s = tc::smem_addr(smem);

  if (warp >= 8) {
    // ------------------------------------------------------------------ producers
    const int pt = tid - kProd0;
    const int c16 = pt & 7, r0 = pt >> 3;  // 16-byte chunk and first row of this thread's copies
    if (pt == 0) tma::prefetch_map(&tmap_w);
    uint32_t it = 0;
    int npend = 0;
    auto hand_over = [&](uint32_t h) {  // this thread's copies of stage h have landed
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&full[h % kStages]);
    };
    for (int64_t t = blockIdx.x; t < pa.tiles && !*abort_flag; t += gridDim.x) {
      Tile tl;
      if (!tile_of(pa, t, roff, boff, nblocks, tl)) break;  // tiles are in block order
      const uint8_t* aptr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t row = tl.r0 + r0 + 32 * i;
        aptr[i] = row < tl.r1 ? pa.a + row * pa.K + c16 * 16 : nullptr;
      }
      const int64_t brow0 = (int64_t)tl.e * pa.N + (int64_t)tl.nt * BN;
      for (int kc = 0; kc < nk; ++kc) {
        if (npend == kLag) {
          cp_async_wait<kLag - 1>();
          hand_over(it - kLag);
          --npend;
        }
        const int s = (int)(it % kStages);
        if (!tc::mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1)) {
          moe::set_status(pa.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const uint32_t sl = smem_s + s * L.slot;
        if (pt == 0) {
          tma::mbar_arrive_expect_tx(&full[s], (uint32_t)(BN * kBK));
          tma::load_2d(sl + L.b, &tmap_w, kc * kBK, (int32_t)brow0, &full[s]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (aptr[i]) cp_async16(sl + L.a + tc::sw128_offset(r0 + 32 * i, c16), aptr[i] + kc * kBK);
        cp_async_commit();
        ++it;
        ++npend;
      }
    }
    cp_async_wait<0>();
    while (npend > 0) {
      hand_over(it - npend);
      --npend;
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(kBM, BN, 0);  // format code 0: E4M3 for kind::f8f6f4
      uint32_t it = 0, acc_it = 0;
      for (int64_t t = blockIdx.x; t < pa.tiles && !*abort_flag; t += gridDim.x) {
        Tile tl;
        if (!tile_of(pa, t, roff, boff, nblocks, tl)) break;
        const uint32_t acc = acc_it & 1;
        if (!tc::mbar_wait(&tempty[acc], ((acc_it >> 1) & 1) ^ 1)) {
          moe::set_status(pa.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        bool ok = true;
        for (int kc = 0; kc < nk; ++kc) {
          const int s = (int)(it % kStages);
          if (!tc::mbar_wait(&full[s], (it / kStages) & 1)) {
            moe::set_status(pa.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t sl = smem_s + s * L.slot;
#pragma unroll
          for (int j = 0; j < kBK / 32; ++j)
            mma_f8_ss(taddr + acc * 256, tc::sdesc_sw128(sl + L.a + j * 32), tc::sdesc_sw128(sl + L.b + j * 32), idesc,
                      (kc | j) != 0);
          tc::mma_commit(&empty[s]);
          ++it;
        }
        if (!ok) break;
        tc::mma_commit(&tfull[acc]);
        ++acc_it;
      }
      tc::mma_commit(drain);
      if (!tc::mbar_wait(drain, 0)) moe::set_status(pa.status, MOE_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp - kEpiWarp0;
    const int r = quarter * 32 + lane;
    uint32_t acc_it = 0;
    for (int64_t t = blockIdx.x; t < pa.tiles && !*abort_flag; t += gridDim.x) {
      Tile tl;
      if (!tile_of(pa, t, roff, boff, nblocks, tl)) break;
      const int64_t row = tl.r0 + r;
      const bool valid = row < tl.r1;
      const float sa = valid ? pa.a_scale[row] : 0.f;
      const float sw = pa.w_scale[tl.e];
      const uint32_t acc = acc_it & 1;
      if (!tc::mbar_wait(&tfull[acc], (acc_it >> 1) & 1)) {
        moe::set_status(pa.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      const int n0 = tl.nt * BN;
      const uint32_t tb = taddr + acc * 256 + ((uint32_t)(quarter * 32) << 16);
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld32(tb + c0, v);
        tc::tmem_ld_wait();
        if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float o0 = __uint_as_float(v[2 * j]) * sa * sw, o1 = __uint_as_float(v[2 * j + 1]) * sa * sw;
            if (pa.bias) {
              o0 += moe::bf16_bits_to_f32(pa.bias[(int64_t)tl.e * pa.N + n0 + c0 + 2 * j]);
              o1 += moe::bf16_bits_to_f32(pa.bias[(int64_t)tl.e * pa.N + n0 + c0 + 2 * j + 1]);
            }
            pk[j] = (uint32_t)moe::f32_to_bf16_bits(o0) | ((uint32_t)moe::f32_to_bf16_bits(o1) << 16);
          }
          uint4* dst = reinterpret_cast<uint4*>(pa.out + row * pa.N + n0 + c0);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[acc]);
      ++acc_it;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, kTmemCols);
  }
}

int sm_count_pt() { return moe_launch::sm_count_current(); }

}  // namespace

namespace moe_launch {

cudaError_t pertoken_gemm(const PerTokenGemm& g, cudaStream_t stream) {
  if (g.E < 1 || g.E > kMaxE || g.N < 128 || g.N % 128 != 0 || g.K < kBK || g.K % kBK != 0 || g.M < 0)
    return cudaErrorInvalidValue;
  if (g.M == 0) return cudaSuccess;
  PTArgs pa;
  pa.a = static_cast<const uint8_t*>(g.a);
  pa.a_scale = g.a_scale;
  pa.w = g.w;
  pa.w_scale = g.w_scale;
  pa.bias = static_cast<const uint16_t*>(g.bias);
  pa.group_sizes = g.group_sizes;
  pa.out = static_cast<uint16_t*>(g.out);
  pa.status = g.status;
  pa.M = g.M;
  pa.E = g.E;
  pa.N = g.N;
  pa.K = g.K;
  pa.BN = (g.N % 256 == 0) ? 256 : 128;
  pa.n_tiles = g.N / pa.BN;
  pa.tiles = ((g.M + kBM - 1) / kBM + g.E) * pa.n_tiles;
  // weights as E * N rows of K bytes; boxes of 128 bytes x BN rows in the 128-byte swizzle
  CUtensorMap tmap;
  if (!tma::encode_2d_u8(&tmap, g.w, (uint64_t)g.K, (uint64_t)g.E * g.N, (uint64_t)g.K, kBK, pa.BN, true))
    return cudaErrorInvalidValue;
  const PLayout L = playout(pa.BN);
  cudaError_t err = cudaFuncSetAttribute(pertoken_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  int64_t grid = sm_count_pt();
  if (pa.tiles < grid) grid = pa.tiles;
  pertoken_gemm_kernel<<<(unsigned)grid, kThreads, L.total, stream>>>(tmap, pa);
  return cudaGetLastError();
}

}  // namespace moe_launch
