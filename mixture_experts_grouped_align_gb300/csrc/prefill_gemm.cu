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
//               and run the fused epilogue: bias + SwiGLU or bias + relu^2 -> h (f16),
//               bias * routing weight -> o (fp32), or bias -> out (bf16), each row to
//               its pair index.
// Every mbarrier wait is bounded; a wait that runs out sets MOE_ERR_TIMEOUT, every role
// leaves its loop, the MMA lane drains its own work and the TMEM is freed.
//
// f16 operands: a decoded weight is exact when its scale is within 2^-23..2^13 (E2M1)
// or 2^-15..2^7 (E4M3); a block with nonzero codes outside that range sets MOE_ERR_RANGE.
// Each output row depends on its own A row only and K is always reduced in the same
// order, so padded and unpadded batches give identical real rows.
#include "moe_common.cuh"
#include "cp_async.cuh"
#include "moe_launch.h"
#include "tcgen05.cuh"

namespace {

using namespace moe_launch;
using namespace cpa;

constexpr int kThreads = 512;
constexpr int kBM = 128, kBK = 64;
constexpr int kProd0 = 256, kNumProd = 256;  // producer threads: warps 8..15
constexpr int kEpiWarp0 = 4;                 // epilogue warps 4..7
constexpr int kTmemCols = 512;
constexpr int kSmemLimit = 227 * 1024;

struct PLayout {
  // raw ring: what the producers copy (the f16 A tile in its final layout, or raw E4M3
  // A) plus the raw weight bytes; decoded ring: the decoded B tile (and decoded A).
  int raw_a, raw_b, raw_slot, nraw;
  int dec_b, dec_a, dec_slot, ndec;
  int raw_base, dec_base, bars, total;
};

constexpr int kLag = 3;  // stages between a stage's copies and its decode (nraw >= kLag + 1)

__host__ __device__ inline PLayout playout(int wf, bool a_e4m3, int BN) {
  PLayout L;
  const int braw_row = (wf == WF_MXFP4) ? 32 : 64;
  L.raw_a = 0;
  L.raw_b = a_e4m3 ? kBM * 64 : kBM * 128;
  L.raw_slot = ((L.raw_b + BN * braw_row) + 1023) / 1024 * 1024;
  L.dec_b = 0;
  L.dec_a = BN * 128;
  L.dec_slot = ((L.dec_a + (a_e4m3 ? kBM * 128 : 0)) + 1023) / 1024 * 1024;
  const int budget = kSmemLimit - 1024 - 256;
  L.ndec = 3;
  L.nraw = (budget - L.ndec * L.dec_slot) / L.raw_slot;
  if (L.nraw < kLag + 1) {
    L.ndec = 2;
    L.nraw = (budget - L.ndec * L.dec_slot) / L.raw_slot;
  }
  if (L.nraw > 8) L.nraw = 8;
  L.dec_base = 0;
  L.raw_base = L.ndec * L.dec_slot;
  L.bars = L.raw_base + L.nraw * L.raw_slot;
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

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t v, __half2 s) {
  __half2 h = __hmul2(*reinterpret_cast<__half2*>(&v), s);
  return *reinterpret_cast<uint32_t*>(&h);
}

// f16x2 holding 2^(s-127) in both halves (exact for the scales the f16 path accepts).
__device__ __forceinline__ __half2 scale_h2(uint32_t scale_byte) {
  return __float2half2_rn(moe::e8m0_to_f32(scale_byte));
}

// Decodes one (row, 32-element half-stage) unit of raw MX bytes in shared memory into
// the 4 f16 chunks of the swizzled tile whose byte offsets (within the slot) are dst[].
template <int FMT>
__device__ __forceinline__ void dequant_unit(const uint8_t* raw, uint8_t* slot, const uint32_t (&dst)[4],
                                             uint32_t scale_byte, bool& bad) {
  const int se = (int)scale_byte - 127;
  const __half2 s2 = scale_h2(scale_byte);
  if (FMT == WF_MXFP4) {
    const uint4 w = *reinterpret_cast<const uint4*>(raw);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    if ((w.x | w.y | w.z | w.w) && (se < -23 || se > 13)) bad = true;
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // chunk q = elements 8q..8q+7 = raw word q
      uint32_t o0, o1, o2, o3;
      moe::e2m1x8_to_f16x2(ws[q], o0, o1, o2, o3);
      *reinterpret_cast<uint4*>(slot + dst[q]) =
          make_uint4(hmul2_u32(o0, s2), hmul2_u32(o1, s2), hmul2_u32(o2, s2), hmul2_u32(o3, s2));
    }
  } else {
    const uint4 w0 = *reinterpret_cast<const uint4*>(raw);
    const uint4 w1 = *reinterpret_cast<const uint4*>(raw + 16);
    const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const uint32_t any = w0.x | w0.y | w0.z | w0.w | w1.x | w1.y | w1.z | w1.w;
    if ((any & 0x7f7f7f7fu) && (se < -15 || se > 7)) bad = true;
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // chunk q = elements 8q..8q+7 = raw words 2q, 2q+1
      uint32_t o0, o1, o2, o3;
      moe::e4m3x4_to_f16x2(ws[2 * q], o0, o1);
      moe::e4m3x4_to_f16x2(ws[2 * q + 1], o2, o3);
      *reinterpret_cast<uint4*>(slot + dst[q]) =
          make_uint4(hmul2_u32(o0, s2), hmul2_u32(o1, s2), hmul2_u32(o2, s2), hmul2_u32(o3, s2));
    }
  }
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
  const int NR = L.nraw, ND = L.ndec;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);  // [ND] decoded stage ready
  uint64_t* dec_empty = full + 3;                                // [ND]
  uint64_t* raw_empty = dec_empty + 3;                           // [NR]
  uint64_t* tfull = raw_empty + 8;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_s + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < ND; ++s) {
      tc::mbar_init(&full[s], kNumProd / 32);
      tc::mbar_init(&dec_empty[s], 1);
    }
    for (int s = 0; s < NR; ++s) tc::mbar_init(&raw_empty[s], 1);
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
    // Each thread owns fixed pieces of every stage: A chunks (rows pt/8 + 32i, chunk
    // pt%8) for f16 activations, or the A decode unit (row pt/2, half pt%2) for E4M3
    // activations, and the B decode units u = pt + 256i (row u/2, half u%2).  Stage s is
    // copied into raw slot s % NR and decoded kLag stages later into decoded slot s % ND,
    // so kLag stages of copies are in flight while the MMA works on decoded stages.
    const int pt = tid - kProd0;
    const int64_t rb = (WF == WF_MXFP4) ? Kin / 2 : Kin;  // raw weight row bytes
    constexpr int kBrawRow = (WF == WF_MXFP4) ? 32 : 64;   // raw bytes per row per stage
    constexpr int kBrawHalf = kBrawRow / 2;
    const uint8_t* wbase = static_cast<const uint8_t*>(a.w);
    uint32_t a_off[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a_off[i] = L.raw_a + tc::sw128_offset((pt >> 3) + 32 * i, pt & 7);
    const int ra = pt >> 1, ha = pt & 1;  // E4M3 A decode unit
    uint32_t a_dst[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) a_dst[q] = L.dec_a + tc::sw128_offset(ra, ha * 4 + q);
    const uint32_t a_raw = L.raw_a + ra * 64 + ha * 32;
    uint32_t b_dst[2][4], b_raw[2];
    bool bvalid[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int u = pt + 256 * i, r = u >> 1, h = u & 1;
      bvalid[i] = r < BN;
#pragma unroll
      for (int q = 0; q < 4; ++q) b_dst[i][q] = L.dec_b + tc::sw128_offset(r, h * 4 + q);
      b_raw[i] = L.raw_b + r * kBrawRow + h * kBrawHalf;
    }
    // stages whose copies are in flight, oldest first
    uint32_t pend_st[kLag] = {};
    uint32_t pend_sb[kLag][2] = {}, pend_sa[kLag] = {};
    bool pend_va[kLag] = {};
    int npend = 0;
    uint32_t it = 0;
    auto finish_oldest = [&]() {  // decode + hand over pend[0], shift the queue
      const uint32_t d = pend_st[0];
      const int ds = d % ND;
      if (!tc::mbar_wait(&dec_empty[ds], ((d / ND) & 1) ^ 1)) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      const uint8_t* rs = smem + L.raw_base + (d % NR) * L.raw_slot;
      uint8_t* dst = smem + L.dec_base + ds * L.dec_slot;
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (bvalid[i]) dequant_unit<WF>(rs + b_raw[i], dst, b_dst[i], pend_sb[0][i], bad);
      if (A_E4M3 && pend_va[0]) dequant_unit<WF_MXFP8>(rs + a_raw, dst, a_dst, pend_sa[0], bad);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&full[ds]);
#pragma unroll
      for (int j = 0; j + 1 < kLag; ++j) {
        pend_st[j] = pend_st[j + 1];
        pend_sb[j][0] = pend_sb[j + 1][0];
        pend_sb[j][1] = pend_sb[j + 1][1];
        pend_sa[j] = pend_sa[j + 1];
        pend_va[j] = pend_va[j + 1];
      }
      --npend;
    };
    for (int64_t t = blockIdx.x; t < pa.tiles && !*abort_flag; t += gridDim.x) {
      int64_t blk, e;
      int nt;
      if (!tile_info(pa, t, ntpp, blk, nt, e)) continue;
      // global pointers of this tile
      const uint16_t* aptr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int p = A_E4M3 ? (int)a.P : a.sorted[blk * a.bm + (pt >> 3) + 32 * i];
        aptr[i] = nullptr;
        if (p < a.P) {
          const int64_t ar = a.act_per_pair ? (int64_t)p : (int64_t)(p / a.k);
          aptr[i] = static_cast<const uint16_t*>(a.act) + ar * Kin + (pt & 7) * 8;
        }
      }
      const uint8_t* a8 = nullptr;   // E4M3 A unit row
      const uint8_t* as8 = nullptr;  // its scale row
      if (A_E4M3) {
        const int p = a.sorted[blk * a.bm + ra];
        if (p < a.P) {
          const int64_t ar = a.act_per_pair ? (int64_t)p : (int64_t)(p / a.k);
          a8 = static_cast<const uint8_t*>(a.act) + ar * Kin + ha * 32;
          as8 = a.act_scale + ar * nkb + ha;
        }
      }
      const uint8_t* bptr[2];
      const uint8_t* sptr[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int u = pt + 256 * i, r = u >> 1, h = u & 1;
        int64_t n;
        if (EPI == EPI_SWIGLU)
          n = (r < pa.half) ? (int64_t)nt * pa.half + r : (int64_t)a.Nout + (int64_t)nt * pa.half + (r - pa.half);
        else
          n = (int64_t)nt * BN + r;
        const int64_t brow = e * a.Nw + n;
        bptr[i] = wbase + brow * rb + h * kBrawHalf;
        sptr[i] = a.w_scale + brow * nkb + h;
      }
      for (int kc = 0; kc < nk && !*abort_flag; ++kc) {
        const int rsl = it % NR;
        if (!tc::mbar_wait(&raw_empty[rsl], ((it / NR) & 1) ^ 1)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const uint32_t sl_s = smem_s + L.raw_base + rsl * L.raw_slot;
        if (!A_E4M3) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (aptr[i]) cp_async16(sl_s + a_off[i], aptr[i] + kc * kBK);
        } else if (a8) {
          // raw A of this thread's own decode unit: the thread that decodes the bytes is
          // the one whose cp.async wait covers them
          cp_async16(sl_s + a_raw, a8 + kc * kBK);
          cp_async16(sl_s + a_raw + 16, a8 + kc * kBK + 16);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {  // raw B bytes of this thread's own decode units
          if (bvalid[i]) {
            cp_async16(sl_s + b_raw[i], bptr[i] + (int64_t)kc * kBrawRow);
            if (kBrawHalf > 16) cp_async16(sl_s + b_raw[i] + 16, bptr[i] + (int64_t)kc * kBrawRow + 16);
          }
        }
        cp_async_commit();
        uint32_t nsc_b[2] = {0, 0}, nsc_a = 0;  // scale bytes, used when the stage is decoded
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (bvalid[i]) nsc_b[i] = sptr[i][2 * kc];
        if (A_E4M3 && as8) nsc_a = as8[2 * kc];
        if (npend == kLag) {  // the oldest stage's copies have landed: decode, hand over
          cp_async_wait<kLag>();
          finish_oldest();
        }
#pragma unroll
        for (int j = 0; j < kLag; ++j)
          if (j == npend) {
            pend_st[j] = it;
            pend_sb[j][0] = nsc_b[0];
            pend_sb[j][1] = nsc_b[1];
            pend_sa[j] = nsc_a;
            pend_va[j] = A_E4M3 && (a8 != nullptr);
          }
        ++npend;
        ++it;
      }
    }
    cp_async_wait<0>();
    while (npend > 0) finish_oldest();
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
          const int ds = it % ND, rsl = it % NR;
          if (!tc::mbar_wait(&full[ds], (it / ND) & 1)) {
            moe::set_status(a.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t dec_s = smem_s + L.dec_base + ds * L.dec_slot;
          const uint32_t a_s = A_E4M3 ? dec_s + L.dec_a : smem_s + L.raw_base + rsl * L.raw_slot + L.raw_a;
          const uint32_t b_s = dec_s + L.dec_b;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc::mma_f16_ss(d_tmem, tc::sdesc_sw128(a_s + kk * 32), tc::sdesc_sw128(b_s + kk * 32), idesc,
                           (kc | kk) != 0);
          tc::mma_commit(&raw_empty[rsl]);
          tc::mma_commit(&dec_empty[ds]);
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
              if (__hisinf(hv[j])) bad = true;
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
            } else if (EPI == EPI_RELU2) {
              __half hv[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                hv[j] = __float2half_rn(moe::relu2(o[j]));
                if (__hisinf(hv[j])) bad = true;
              }
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(a.out) + (int64_t)p * a.Nout + n0 + c0);
#pragma unroll
              for (int q = 0; q < 4; ++q) dst[q] = reinterpret_cast<const uint4*>(hv)[q];
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

int sm_count() { return moe_launch::sm_count_current(); }

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
  if (g.wfmt == WF_MXFP8 && (g.act_scale == nullptr || g.epi == EPI_SWIGLU || g.epi == EPI_RELU2)) return false;
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
  MOE_CASE(WF_MXFP4, EPI_RELU2, false)
  MOE_CASE(WF_MXFP8, EPI_PLAIN_BF16, true)
  MOE_CASE(WF_MXFP8, EPI_WEIGHTED_F32, true)
#undef MOE_CASE
  return cudaErrorInvalidValue;
}

cudaError_t grouped_gemm(const GroupedGemm& g, int64_t rows, cudaStream_t stream) {
  if (g.act_by_slot || g.out_by_slot)  // slot-ordered rows: only the tensor-memory W4A16 kernel
    return ts_supported(g) ? prefill_ts(g, stream) : cudaErrorInvalidValue;
  if (rows > kPrefillRowsAbove && ts_supported(g)) return prefill_ts(g, stream);
  if (rows > kPrefillRowsAbove && mx8_supported(g)) return mx8_gemm(g, stream);
  if (rows > kPrefillRowsAbove && prefill_supported(g)) return prefill_gemm(g, stream);
  return decode_gemm(g, stream);
}

}  // namespace moe_launch
