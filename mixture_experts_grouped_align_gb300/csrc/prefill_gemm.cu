// Grouped expert GEMM, tensor-memory variant (many rows per expert: prefill shapes).
//
// One persistent launch covers every (alignment block, N tile) of every expert ("Add MoE
// GEMM variants and weight-gradient kernel", aiter PR 5310, Summary: all expert GEMMs in
// a single launch).  Tiles whose block slot is past num_tokens_post_padded or carries
// the -1 sentinel are skipped by every role before anything is read (second review,
// sentinel handling).  Expert offsets into the weights are 64-bit (Notes).
//
// Per thread block (one per SM, 512 threads):
//   warp 0      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and, on one
//               lane, issues tcgen05.mma (kind::f16, M = 128, N = BN, K = 16) from
//               128-byte-swizzled K-major shared tiles, committing each stage back to
//               its producers and each finished accumulator to the epilogue;
//   warps 8-15  produce the stages: cp.async of the A rows (gathered through
//               sorted_token_ids) and of the raw MX weight bytes, then decode the
//               weights (E2M1 / E4M3 codes -> f16 with the hardware conversions, times
//               the block's E8M0 scale) into the B tile, one stage behind the copies.
//               Every thread copies exactly the raw bytes it later decodes: a cp.async
//               wait only covers the waiting thread's own copies;
//   warps 4-7   drain an accumulator with tcgen05.ld (one TMEM lane = one tile row)
//               and run the fused epilogue: bias + SwiGLU -> h (f16), bias * routing
//               weight -> o (fp32), or bias -> out (bf16), each row to its pair index.
// Every mbarrier wait is bounded; a wait that runs out sets MOE_ERR_TIMEOUT, every role
// leaves its loop, the MMA lane drains its own work and the TMEM is freed.
//
// f16 operands: a decoded weight is exact when its scale is within 2^-23..2^13 (E2M1)
// or 2^-15..2^7 (E4M3); a block with nonzero codes outside that range sets MOE_ERR_RANGE.
// Each output row depends on its own A row only and K is always reduced in the same
// order, so padded and unpadded batches give identical real rows.
#include "moe_common.cuh"
#include "moe_launch.h"
#include "tcgen05.cuh"

namespace {

using namespace moe_launch;

constexpr int kThreads = 512;
constexpr int kBM = 128, kBK = 64;
constexpr int kProd0 = 256, kNumProd = 256;  // producer threads: warps 8..15
constexpr int kEpiWarp0 = 4;                 // epilogue warps 4..7
constexpr int kTmemCols = 512;
constexpr int kSmemLimit = 227 * 1024;

struct PLayout {
  int a, b, braw, araw, slot, nslots, bars, total;
};

// Per-slot shared layout (bytes): A tile 128 x 128 B | B tile BN x 128 B | raw weight
// bytes of the stage | raw E4M3 activation bytes (MXFP8 A only).
__host__ __device__ inline PLayout playout(int wf, bool a_e4m3, int BN) {
  PLayout L;
  L.a = 0;
  L.b = kBM * 128;
  L.braw = L.b + BN * 128;
  const int braw_bytes = (wf == WF_MXFP4) ? BN * 32 : BN * 64;
  L.araw = L.braw + braw_bytes;
  const int araw_bytes = a_e4m3 ? kBM * 64 : 0;
  L.slot = ((L.araw + araw_bytes) + 1023) / 1024 * 1024;
  int n = (kSmemLimit - 1024 - 256) / L.slot;
  L.nslots = n > 4 ? 4 : n;
  L.bars = L.nslots * L.slot;
  L.total = L.bars + 256 + 1024;  // barriers, TMEM address, flags; 1024 B alignment slack
  return L;
}

struct PArgs {
  GroupedGemm g;
  int BN;        // N tile (output columns of the MMA), multiple of 32, <= 256
  int half;      // SwiGLU: gate columns per tile (BN / 2)
  int n_tiles;   // N tiles per block
  int64_t tiles; // block slots * n_tiles
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t v, __half2 s) {
  __half2 h = __hmul2(*reinterpret_cast<__half2*>(&v), s);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Decodes one (row, 32-element half-stage) unit of raw MX weight bytes in shared memory
// into 4 f16 chunks of the swizzled B (or A) tile.
template <int FMT>
__device__ __forceinline__ void dequant_unit(const uint8_t* raw, uint8_t* tile, int row, int half,
                                             uint32_t scale_byte, bool& bad) {
  const int se = (int)scale_byte - 127;
  const float sf = moe::e8m0_to_f32(scale_byte);
  const __half2 s2 = __float2half2_rn(sf);
  uint32_t out[16];
  uint32_t any = 0;
  if (FMT == WF_MXFP4) {
    const uint4 w = *reinterpret_cast<const uint4*>(raw);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    any = w.x | w.y | w.z | w.w;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int b = 0; b < 4; ++b) out[i * 4 + b] = hmul2_u32(moe::e2m1x2_to_f16x2((ws[i] >> (8 * b)) & 0xffu), s2);
    if (any && (se < -23 || se > 13)) bad = true;
  } else {
    const uint4 w0 = *reinterpret_cast<const uint4*>(raw);
    const uint4 w1 = *reinterpret_cast<const uint4*>(raw + 16);
    const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    any = w0.x | w0.y | w0.z | w0.w | w1.x | w1.y | w1.z | w1.w;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      out[i * 2] = hmul2_u32(moe::e4m3x2_to_f16x2(ws[i] & 0xffffu), s2);
      out[i * 2 + 1] = hmul2_u32(moe::e4m3x2_to_f16x2(ws[i] >> 16), s2);
    }
    if ((any & 0x7f7f7f7fu) && (se < -15 || se > 7)) bad = true;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(tile + tc::sw128_offset(row, half * 4 + q)) =
        make_uint4(out[q * 4], out[q * 4 + 1], out[q * 4 + 2], out[q * 4 + 3]);
}

// Tile index -> (block slot, N tile); false for a tile no role works on.
__device__ __forceinline__ bool tile_info(const PArgs& pa, int64_t t, int ntpp, int64_t& blk,
                                          int& nt, int64_t& e) {
  blk = t / pa.n_tiles;
  nt = (int)(t - blk * pa.n_tiles);
  if (blk * pa.g.bm >= ntpp) return false;
  e = pa.g.expert_ids[blk];
  return e >= 0 && e < pa.g.E;
}

template <int WF, int EPI, bool A_E4M3>
__global__ void __launch_bounds__(kThreads, 1) prefill_gemm_kernel(PArgs pa) {
  const GroupedGemm& a = pa.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const PLayout L = playout(WF, A_E4M3, pa.BN);
  const int S = L.nslots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + 4;
  uint64_t* tfull = empty + 4;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_s + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], kNumProd / 32);
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
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t taddr = *taddr_s;
  const int ntpp = *a.ntpp;
  const int Kin = a.Kin, nk = Kin / kBK, nkb = Kin / 32;
  const int BN = pa.BN;
  const uint32_t smem_s = tc::smem_addr(smem);
  bool bad = false;

  if (warp >= 8) {
    // ------------------------------------------------------------------ producers
    const int pt = tid - kProd0;
    const int64_t rb = (WF == WF_MXFP4) ? Kin / 2 : Kin;  // raw weight row bytes
    const int braw_row = (WF == WF_MXFP4) ? 32 : 64;     // raw bytes per row per stage
    const uint8_t* wbase = static_cast<const uint8_t*>(a.w);
    uint32_t it = 0;
    bool pending = false;
    int prev_slot = 0;
    uint32_t sc_b[2] = {0, 0}, sc_a = 0;  // scale bytes of the pending stage
    bool va = false;                      // the pending stage's A unit row is a real pair
    for (int64_t t = blockIdx.x; t < pa.tiles && !*abort_flag; t += gridDim.x) {
      int64_t blk, e;
      int nt;
      if (!tile_info(pa, t, ntpp, blk, nt, e)) continue;
      // this thread's 4 A rows (f16 A) / its A unit row (E4M3 A)
      int64_t arow[4];
      bool avalid[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = (pt >> 3) + 32 * i;
        const int p = a.sorted[blk * a.bm + r];
        avalid[i] = p < a.P;
        arow[i] = avalid[i] ? (a.act_per_pair ? (int64_t)p : (int64_t)(p / a.k)) : 0;
      }
      // B units (row, half): unit u = pt + 256 * i, row = u >> 1, half = u & 1
      int64_t brow[2];
      bool bvalid[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int u = pt + 256 * i;
        const int r = u >> 1;
        bvalid[i] = r < BN;
        int64_t n;
        if (EPI == EPI_SWIGLU)
          n = (r < pa.half) ? (int64_t)nt * pa.half + r : (int64_t)a.Nout + (int64_t)nt * pa.half + (r - pa.half);
        else
          n = (int64_t)nt * BN + r;
        brow[i] = e * a.Nw + n;
      }
      for (int kc = 0; kc < nk; ++kc) {
        const int slot = it % S;
        if (!tc::mbar_wait(&empty[slot], ((it / S) & 1) ^ 1)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const uint32_t sl_s = smem_s + slot * L.slot;
        // A rows
        if (!A_E4M3) {
          const uint16_t* act = static_cast<const uint16_t*>(a.act);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = (pt >> 3) + 32 * i, c = pt & 7;
            if (avalid[i])
              cp_async16(sl_s + L.a + tc::sw128_offset(r, c), act + arow[i] * Kin + kc * kBK + c * 8);
          }
        } else {
          // raw A of this thread's own decode unit (row pt/2, half pt%2): 32 B, so that
          // the thread that decodes the bytes is the one whose cp.async wait covers them
          const uint8_t* act = static_cast<const uint8_t*>(a.act);
          const int r = pt >> 1, h = pt & 1;
          const int p = a.sorted[blk * a.bm + r];
          if (p < a.P) {
            const int64_t ar = a.act_per_pair ? (int64_t)p : (int64_t)(p / a.k);
            const uint8_t* src = act + ar * Kin + kc * kBK + h * 32;
            cp_async16(sl_s + L.araw + r * 64 + h * 32, src);
            cp_async16(sl_s + L.araw + r * 64 + h * 32 + 16, src + 16);
          }
        }
        // raw B bytes of this thread's own decode units (row u/2, half u%2)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int u = pt + 256 * i;
          const int r = u >> 1, h = u & 1;
          if (r < BN) {
            const uint8_t* src = wbase + brow[i] * rb + (int64_t)kc * braw_row + h * (braw_row / 2);
            const uint32_t dst = sl_s + L.braw + r * braw_row + h * (braw_row / 2);
            cp_async16(dst, src);
            if (braw_row / 2 > 16) cp_async16(dst + 16, src + 16);
          }
        }
        cp_async_commit();
        // scale bytes of this stage (used one iteration later)
        uint32_t nsc_b[2] = {0, 0}, nsc_a = 0;
        bool nva = false;
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (bvalid[i]) nsc_b[i] = a.w_scale[brow[i] * nkb + 2 * kc + ((pt + 256 * i) & 1)];
        if (A_E4M3) {
          const int r = pt >> 1, h = pt & 1;
          const int p = a.sorted[blk * a.bm + r];
          if (p < a.P) {
            const int64_t ar = a.act_per_pair ? (int64_t)p : (int64_t)(p / a.k);
            nsc_a = a.act_scale[ar * nkb + 2 * kc + h];
            nva = true;
          }
        }
        if (pending) {  // decode the previous stage, then hand it to the MMA
          cp_async_wait<1>();
          uint8_t* ps = smem + prev_slot * L.slot;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int u = pt + 256 * i;
            const int r = u >> 1, h = u & 1;
            if (r < BN) dequant_unit<WF>(ps + L.braw + r * braw_row + h * (braw_row / 2), ps + L.b, r, h, sc_b[i], bad);
          }
          if (A_E4M3 && va) {
            const int r = pt >> 1, h = pt & 1;
            dequant_unit<WF_MXFP8>(ps + L.araw + r * 64 + h * 32, ps + L.a, r, h, sc_a, bad);
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&full[prev_slot]);
        }
        va = nva;
        pending = true;
        prev_slot = slot;
        sc_b[0] = nsc_b[0];
        sc_b[1] = nsc_b[1];
        sc_a = nsc_a;
        ++it;
      }
    }
    if (pending) {
      cp_async_wait<0>();
      uint8_t* ps = smem + prev_slot * L.slot;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int u = pt + 256 * i;
        const int r = u >> 1, h = u & 1;
        if (r < BN) dequant_unit<WF>(ps + L.braw + r * braw_row + h * (braw_row / 2), ps + L.b, r, h, sc_b[i], bad);
      }
      if (A_E4M3 && va) {
        const int r = pt >> 1, h = pt & 1;
        dequant_unit<WF_MXFP8>(ps + L.araw + r * 64 + h * 32, ps + L.a, r, h, sc_a, bad);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&full[prev_slot]);
    }
    cp_async_wait<0>();
  } else if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(kBM, BN, 0);
      uint32_t it = 0, acc_it = 0;
      for (int64_t t = blockIdx.x; t < pa.tiles && !*abort_flag; t += gridDim.x) {
        int64_t blk, e;
        int nt;
        if (!tile_info(pa, t, ntpp, blk, nt, e)) continue;
        const uint32_t acc = acc_it & 1;
        if (!tc::mbar_wait(&tempty[acc], ((acc_it >> 1) & 1) ^ 1)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d_tmem = taddr + acc * 256;
        bool ok = true;
        for (int kc = 0; kc < nk; ++kc) {
          const int slot = it % S;
          if (!tc::mbar_wait(&full[slot], (it / S) & 1)) {
            moe::set_status(a.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a_s = smem_s + slot * L.slot + L.a;
          const uint32_t b_s = smem_s + slot * L.slot + L.b;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc::mma_f16_ss(d_tmem, tc::sdesc_sw128(a_s + kk * 32), tc::sdesc_sw128(b_s + kk * 32), idesc,
                           (kc | kk) != 0);
          tc::mma_commit(&empty[slot]);
          ++it;
        }
        if (!ok) break;
        tc::mma_commit(&tfull[acc]);
        ++acc_it;
      }
      // drain: every MMA this thread issued has completed before the TMEM is freed
      tc::mma_commit(drain);
      if (!tc::mbar_wait(drain, 0)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp - kEpiWarp0;
    const int r = quarter * 32 + lane;
    uint32_t acc_it = 0;
    const uint16_t* bias = static_cast<const uint16_t*>(a.bias);
    for (int64_t t = blockIdx.x; t < pa.tiles && !*abort_flag; t += gridDim.x) {
      int64_t blk, e;
      int nt;
      if (!tile_info(pa, t, ntpp, blk, nt, e)) continue;
      const uint32_t acc = acc_it & 1;
      if (!tc::mbar_wait(&tfull[acc], (acc_it >> 1) & 1)) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      const int p = a.sorted[blk * a.bm + r];
      const bool valid = p < a.P;
      const uint32_t tb = taddr + acc * 256 + ((uint32_t)(quarter * 32) << 16);
      if (EPI == EPI_SWIGLU) {
        const int n0 = nt * pa.half;
        for (int c0 = 0; c0 < pa.half; c0 += 32) {
          uint32_t gv[32], uv[32];
          tc::tmem_ld32(tb + c0, gv);
          tc::tmem_ld32(tb + pa.half + c0, uv);
          tc::tmem_ld_wait();
          if (valid) {
            __half hv[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              float gt = __uint_as_float(gv[j]), up = __uint_as_float(uv[j]);
              if (bias) {
                gt += moe::bf16_bits_to_f32(bias[e * a.Nw + n0 + c0 + j]);
                up += moe::bf16_bits_to_f32(bias[e * a.Nw + a.Nout + n0 + c0 + j]);
              }
              hv[j] = __float2half_rn(moe::silu(gt) * up);
              if (__hisinf(hv[j]) || __hisnan(hv[j])) bad = true;
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(a.out) + (int64_t)p * a.Nout + n0 + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = reinterpret_cast<const uint4*>(hv)[q];
          }
        }
      } else {
        const int n0 = nt * BN;
        const float wgt = (EPI == EPI_WEIGHTED_F32 && valid) ? a.topk_w[p] : 1.f;
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(tb + c0, v);
          tc::tmem_ld_wait();
          if (valid) {
            float o[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              o[j] = __uint_as_float(v[j]);
              if (bias) o[j] += moe::bf16_bits_to_f32(bias[e * a.Nw + n0 + c0 + j]);
            }
            if (EPI == EPI_WEIGHTED_F32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + (int64_t)p * a.Nout + n0 + c0);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(o[4 * q] * wgt, o[4 * q + 1] * wgt, o[4 * q + 2] * wgt, o[4 * q + 3] * wgt);
            } else {
              uint32_t pk[16];
#pragma unroll
              for (int q = 0; q < 16; ++q)
                pk[q] = (uint32_t)moe::f32_to_bf16_bits(o[2 * q]) | ((uint32_t)moe::f32_to_bf16_bits(o[2 * q + 1]) << 16);
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + (int64_t)p * a.Nout + n0 + c0);
#pragma unroll
              for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[acc]);
      ++acc_it;
    }
  }
  if (bad) moe::set_status(a.status, MOE_ERR_RANGE);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, kTmemCols);
  }
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

template <int WF, int EPI, bool AE>
cudaError_t launch_t(const PArgs& pa, cudaStream_t stream) {
  const PLayout L = playout(WF, AE, pa.BN);
  cudaError_t err = cudaFuncSetAttribute(prefill_gemm_kernel<WF, EPI, AE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  int64_t grid = sm_count();
  if (pa.tiles < grid) grid = pa.tiles;
  if (grid <= 0) return cudaSuccess;
  prefill_gemm_kernel<WF, EPI, AE><<<(unsigned)grid, kThreads, L.total, stream>>>(pa);
  return cudaGetLastError();
}

}  // namespace

namespace moe_launch {

// N tile for the tensor-memory path, or 0 when the shape does not fit it.
int prefill_tile_n(const GroupedGemm& g) {
  if (g.bm != kBM || g.Kin % kBK != 0) return 0;
  if (g.epi == EPI_SWIGLU) {
    for (int h : {128, 96, 64, 32})
      if (g.Nout % h == 0) return 2 * h;
    return 0;
  }
  for (int bn = 256; bn >= 32; bn -= 32)
    if (g.Nout % bn == 0) return bn;
  return 0;
}

bool prefill_supported(const GroupedGemm& g) {
  if (g.wfmt == WF_BF16) return false;
  if (g.wfmt == WF_MXFP4 && g.act_fmt != ACT_F16) return false;
  if (g.wfmt == WF_MXFP8 && g.act_scale == nullptr) return false;
  return prefill_tile_n(g) > 0;
}

cudaError_t prefill_gemm(const GroupedGemm& g, cudaStream_t stream) {
  PArgs pa;
  pa.g = g;
  pa.BN = prefill_tile_n(g);
  if (pa.BN == 0) return cudaErrorInvalidValue;
  pa.half = pa.BN / 2;
  pa.n_tiles = (g.epi == EPI_SWIGLU) ? g.Nout / pa.half : g.Nout / pa.BN;
  pa.tiles = g.grid_blocks * pa.n_tiles;
#define MOE_CASE(WF, EP, AE) \
  if (g.wfmt == WF && g.epi == EP && (g.wfmt == WF_MXFP8) == AE) return launch_t<WF, EP, AE>(pa, stream);
  MOE_CASE(WF_MXFP4, EPI_SWIGLU, false)
  MOE_CASE(WF_MXFP4, EPI_WEIGHTED_F32, false)
  MOE_CASE(WF_MXFP4, EPI_PLAIN_BF16, false)
  MOE_CASE(WF_MXFP8, EPI_PLAIN_BF16, true)
  MOE_CASE(WF_MXFP8, EPI_SWIGLU, true)
  MOE_CASE(WF_MXFP8, EPI_WEIGHTED_F32, true)
#undef MOE_CASE
  return cudaErrorInvalidValue;
}

cudaError_t grouped_gemm(const GroupedGemm& g, int64_t rows, cudaStream_t stream) {
  if (rows > kPrefillRowsAbove && prefill_supported(g)) return prefill_gemm(g, stream);
  return decode_gemm(g, stream);
}

}  // namespace moe_launch
