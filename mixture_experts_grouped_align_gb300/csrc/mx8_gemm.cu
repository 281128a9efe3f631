// Grouped expert GEMM on MXFP8 operands with the block-scaled tensor-core MMA (and, with
// the template flag BF, on bf16 operands with the plain kind::f16 MMA and no scale factors:
// the same tiles, copies and epilogues, a bf16 h for SwiGLU).
//
// out[p, n] = bf16( sum_k A[row(p), k] * sa[row(p), k / 32] * W[e, n, k] * sw[e, n, k / 32]
//                   + bias[e, n] ): E4M3 activations and weights, one E8M0 scale per 32
// K elements of every activation row and weight row ("Add MoE GEMM variants and
// weight-gradient kernel", aiter PR 5310, Summary: single-launch MXFP8 grouped GEMM with
// E8M0 microscales and per-expert bias).  tcgen05.mma kind::mxf8f6f4 takes the E4M3 codes
// straight from shared memory and the E8M0 scales from tensor memory, so nothing is
// decoded: the products of codes and power-of-two scales are exact and accumulate in f32.
//
// Per thread block (one per SM, 512 threads), persistent over (alignment block, N tile):
//   warp 0      allocates the 512 TMEM columns (128 x BN f32 accumulators from column 0:
//               one of BN = 256, or two alternating ones of BN <= 224 so that the epilogue
//               of a tile overlaps the MMAs of the next; the scale factors of the stages in
//               448..511) and, on one lane, issues the MMAs (M = 128, N = BN, K = 32) of
//               each 128-wide K stage;
//   warps 8-15  copy each stage: one thread loads the BN weight rows of 128 bytes with a
//               TMA box into a 128-byte-swizzled K-major tile (completing on the stage's
//               barrier); all copy the 128 gathered activation rows into the same layout
//               and the stage's scale words with cp.async; two stages later they write the
//               scale words into TMEM (warps 8-11 the activation scales, 12-15 the weight
//               scales) and hand the stage to the MMA;
//   warps 4-7   drain the accumulator (one TMEM lane = one tile row) and run the epilogue
//               at the row's pair index: bias -> bf16; bias * routing weight -> f32; or, for
//               GEMM1 of an MXFP8 layer, bias + SwiGLU and the MXFP8 quantisation of h
//               (mx_quant.cuh: 32 features per E8M0 scale, all in the thread's registers).
// SwiGLU tiles hold 128 features: weight rows 0..127 of the B tile are their gate rows and
// 128..255 their up rows (two TMA boxes), so gate and up of a feature share a TMEM lane.
// A last 224-wide tile may reach past N: its extra weight rows are read (the next expert's,
// or zeros past the tensor), their scale words are zero-filled, and their outputs are not
// stored.
// Tiles past num_tokens_post_padded or of the -1 sentinel are skipped by every role before
// anything is read (second review of the same page).  Expert offsets are 64-bit (Notes).
// Every mbarrier wait is bounded; one that runs out sets MOE_ERR_TIMEOUT, every role leaves
// its loop, the copy threads wait for the copies they issued (cp.async groups and the
// weight boxes), the MMA lane drains its own work and the TMEM is freed.  In the stalled
// self-test (GroupedGemm::stall) the copy warps and the MMA lane do nothing, so the epilogue
// waits on a barrier no one arrives on and gives up after GroupedGemm::wait_ns with no copy
// or MMA in flight.
//
// Scale factors in TMEM (32-bit words, one byte per 32-element K block; the MMA of the
// stage's K block j selects byte j): the MMA reads the word of A row m at lane m, column
// m / 32 of the stage's A region (the word is written to all four columns of lane m), and
// the word of B row n in column n / 32 of the B region at lane n % 32 (written to that
// lane of every 32-lane quarter).
#include "moe_common.cuh"
#include "cp_async.cuh"
#include "moe_launch.h"
#include "mx_quant.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace {

using namespace moe_launch;
using namespace cpa;

constexpr int kThreads = 512;
constexpr int kBM = 128, kBK = 128;        // tile rows, K elements (bytes) per stage
constexpr int kProd0 = 256, kNumProd = 256;
constexpr int kEpiWarp0 = 4;
constexpr int kTmemCols = 512;
constexpr int kSfCol0 = 448;               // first TMEM column of the scale regions (4 x 16)
constexpr int kStages = 4;
constexpr int kLag = 2;                    // stages between a stage's copies and its hand-over

// One stage slot: A tile | B tile | A scale words (one per row) | B scale words (one copy
// per 32-lane quarter: [4][BN/32][32 lanes], lanes contiguous).  When Kin is a multiple of
// 512 the scale words instead arrive four stages at a time, 16 bytes per row, into two group
// buffers (A [128 rows][16 B], B [BN rows][16 B]): far fewer, larger copies.
struct MLayout {
  int a, b, sfa, sfb, slot, ga, gb, bars, stg, total;
};

// `staged`: the fp32 routing-weighted epilogue also takes a 32 x 32 fp32 box per epilogue
// warp, through which its rows leave as whole 128-byte lines.
__host__ __device__ inline MLayout mlayout(int BN, bool staged) {
  MLayout L;
  L.a = 0;
  L.b = kBM * kBK;
  L.sfa = L.b + BN * kBK;
  L.sfb = L.sfa + kBM * 4;
  L.slot = (L.sfb + 4 * 32 * (BN / 32) * 4 + 1023) / 1024 * 1024;
  L.ga = kStages * L.slot;
  L.gb = L.ga + 2 * kBM * 16;
  L.bars = L.gb + 2 * BN * 16;
  L.stg = L.bars + 256;
  L.total = L.stg + (staged ? 4 * 32 * 128 : 0) + 1024;
  return L;
}

// TMEM columns of a stage's scale words: A (4 columns at +0), B (BN / 32 <= 8 columns at +8).
__device__ __forceinline__ uint32_t sfa_col(int s) { return kSfCol0 + 16 * s; }
__device__ __forceinline__ uint32_t sfb_col(int s) { return kSfCol0 + 16 * s + 8; }

struct MArgs {
  GroupedGemm g;
  int BN;
  int nacc;        // accumulators in TMEM: 2 (alternating, BN <= 224) or 1 (BN = 256)
  int n_tiles;
  int64_t tiles;
};

__device__ __forceinline__ bool tile_info(const MArgs& ma, int64_t t, int ntpp, int64_t& blk, int& nt,
                                          int64_t& e) {
  blk = t / ma.n_tiles;
  nt = (int)(t - blk * ma.n_tiles);
  if (blk * ma.g.bm >= ntpp) return false;
  e = ma.g.expert_ids[blk];
  return e >= 0 && e < ma.g.E;
}

__device__ __forceinline__ int64_t act_row(const GroupedGemm& a, int p) {
  return a.act_per_pair ? (int64_t)p : (int64_t)(p / a.k);
}

// Weight row of B-tile row n in N tile nt (SwiGLU: gate rows, then up rows of 128 features).
template <int EPI>
__device__ __forceinline__ int64_t b_row(const GroupedGemm& a, int64_t e, int nt, int BN, int n) {
  if (EPI == EPI_SWIGLU)
    return e * a.Nw + (n < 128 ? (int64_t)nt * 128 + n : (int64_t)a.Nout + (int64_t)nt * 128 + (n - 128));
  return e * a.Nw + (int64_t)nt * BN + n;
}

// BF: bf16 weights and activations (kind::f16, no scale factors); otherwise MXFP8.
template <int EPI, bool BF>
__global__ void __launch_bounds__(kThreads, 1) mx8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, MArgs ma) {
  const GroupedGemm& a = ma.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = ma.BN, NBW = BN / 32;  // B scale words per lane
  const MLayout L = mlayout(BN, EPI == EPI_WEIGHTED_F32);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;  // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint64_t* drain = tempty + 2;
  uint64_t* gb_full = drain + 1;  // [2] B scale group landed (every B-scale thread's copies)
  uint64_t* tma_full = gb_full + 2;  // [kStages] the stage's weight box landed
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(tma_full + kStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_s + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], kNumProd / 32);  // producer warps
      tc::mbar_init(&tma_full[s], 1);          // the weight box
      tc::mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], 4);
    }
    tc::mbar_init(drain, 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(&gb_full[i], kNumProd / 2);
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
  // bytes of an operand row (a stage takes 128 of them: 128 E4M3 or 64 bf16 elements)
  const int64_t rbytes = BF ? (int64_t)a.Kin * 2 : (int64_t)a.Kin;
  const int nk = (int)(rbytes / kBK), nkb = a.Kin / 32;
  const uint32_t smem_s = tc::smem_addr(smem);
  // the limit of every wait (a caller's short limit only in the stalled self-test)
  const uint64_t wb = a.wait_ns > 0 ? (uint64_t)a.wait_ns : tc::kWaitNs;

  if (warp >= 8 && !a.stall) {
    // ------------------------------------------------------------------ producers
    const int pt = tid - kProd0, wp = pt >> 5, q = wp & 3;
    const int c16 = pt & 7, r0 = pt >> 3;  // 16-byte chunk and first row of this thread's copies
    const uint8_t* abase = static_cast<const uint8_t*>(a.act);
    if (pt == 0) tma::prefetch_map(&tmap_w);
    uint32_t it = 0;
    int npend = 0;
    // scale words by groups of four stages (16-byte rows) when Kin % 512 == 0: a tile's stage
    // count is then a multiple of four, so stage it belongs to group it / 4
    const bool grouped = !BF && (nkb % 16) == 0;
    const int tb = pt - 128;  // B-scale copier index (warps 12-15)
    // hand stage h over to the MMA: its copies (this thread's own) have landed
    auto hand_over = [&](uint32_t h) -> bool {
      const int hs = (int)(h % kStages);
      const uint8_t* sl = smem + hs * L.slot;
      tc::fence_proxy_async_smem();
      if (BF) {
        // no scale factors: the landed copies are all the stage needs
      } else if (wp < 4) {
        const uint32_t wv = grouped
            ? *reinterpret_cast<const uint32_t*>(smem + L.ga + ((h >> 2) & 1) * kBM * 16 + (q * 32 + lane) * 16 + (h & 3) * 4)
            : *reinterpret_cast<const uint32_t*>(sl + L.sfa + (q * 32 + lane) * 4);
        tc::tmem_st4(taddr + ((uint32_t)(q * 32) << 16) + sfa_col(hs), wv, wv, wv, wv);
      } else {
        uint32_t v[8];
        if (grouped) {  // rows 32 j + lane of the group, copied by all four B-scale warps
          const uint32_t g = h >> 2;
          if ((h & 3) == 0 && !tc::mbar_wait(&gb_full[g & 1], (g >> 1) & 1, wb)) {
            moe::set_status(a.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            return false;
          }
          const uint8_t* gsrc = smem + L.gb + (g & 1) * BN * 16 + (h & 3) * 4;
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = j < NBW ? *reinterpret_cast<const uint32_t*>(gsrc + (32 * j + lane) * 16) : 0u;
        } else {
          const uint32_t* src = reinterpret_cast<const uint32_t*>(sl + L.sfb) + q * NBW * 32 + lane;
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = j < NBW ? src[j * 32] : 0u;
        }
        tc::tmem_st8(taddr + ((uint32_t)(q * 32) << 16) + sfb_col(hs), v);
      }
      if (!BF) tc::tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&full[hs]);
      return true;
    };
    for (int64_t t = blockIdx.x; t < ma.tiles && !*abort_flag; t += gridDim.x) {
      int64_t blk, e;
      int nt;
      if (!tile_info(ma, t, ntpp, blk, nt, e)) continue;
      const uint8_t* aptr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int p = a.sorted[blk * a.bm + r0 + 32 * i];
        aptr[i] = p < a.P ? abase + act_row(a, p) * rbytes + c16 * 16 : nullptr;
      }
      const uint8_t* sfsrc = nullptr;  // A: this lane's row (B rows: b_row below)
      if (!BF && wp < 4) {
        const int p = a.sorted[blk * a.bm + q * 32 + lane];
        if (p < a.P) sfsrc = a.act_scale + act_row(a, p) * nkb;
      }
      for (int kc = 0; kc < nk; ++kc) {
        // hand the oldest stage over before waiting for a free slot, so that the MMA has two
        // stages queued while this one's copies fly
        if (npend == kLag) {
          cp_async_wait<kLag - 1>();
          if (!hand_over(it - kLag)) break;
          --npend;
        }
        const int s = (int)(it % kStages);
        if (!tc::mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, wb)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const uint32_t sl = smem_s + s * L.slot;
        if (pt == 0) {
          tma::mbar_arrive_expect_tx(&tma_full[s], (uint32_t)(BN * kBK));
          if (EPI == EPI_SWIGLU) {  // gate rows, then up rows: two boxes of 128
            tma::load_2d(sl + L.b, &tmap_w, kc * kBK, (int32_t)b_row<EPI>(a, e, nt, BN, 0), &tma_full[s]);
            tma::load_2d(sl + L.b + 128 * kBK, &tmap_w, kc * kBK, (int32_t)b_row<EPI>(a, e, nt, BN, 128),
                         &tma_full[s]);
          } else {
            tma::load_2d(sl + L.b, &tmap_w, kc * kBK, (int32_t)b_row<EPI>(a, e, nt, BN, 0), &tma_full[s]);
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (aptr[i]) cp_async16(sl + L.a + tc::sw128_offset(r0 + 32 * i, c16), aptr[i] + kc * kBK);
        if (BF) {
          // bf16: no scale words
        } else if (grouped) {
          if ((kc & 3) == 0) {  // this group's four stages of scale words, 16 bytes per row
            const uint32_t gsel = (it >> 2) & 1;
            if (wp < 4) {
              if (sfsrc) cp_async16(smem_s + L.ga + gsel * kBM * 16 + (q * 32 + lane) * 16, sfsrc + kc * 4);
            } else {
              for (int n = tb; n < BN; n += 128) {
                const bool live = EPI == EPI_SWIGLU || (int64_t)nt * BN + n < a.Nout;
                cp_async16z(smem_s + L.gb + gsel * BN * 16 + n * 16,
                            live ? a.w_scale + b_row<EPI>(a, e, nt, BN, n) * nkb + kc * 4 : a.w_scale, live);
              }
              cp_async_arrive_noinc(&gb_full[gsel]);
            }
          }
        } else if (wp < 4) {
          if (sfsrc) cp_async4(sl + L.sfa + (q * 32 + lane) * 4, sfsrc + kc * 4);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < NBW) {
              const bool live = EPI == EPI_SWIGLU || (int64_t)nt * BN + 32 * j + lane < a.Nout;
              cp_async4z(sl + L.sfb + ((q * NBW + j) * 32 + lane) * 4,
                         live ? a.w_scale + b_row<EPI>(a, e, nt, BN, 32 * j + lane) * nkb + kc * 4 : a.w_scale,
                         live);
            }
        }
        cp_async_commit();
        ++it;
        ++npend;
      }
    }
    cp_async_wait<0>();
    while (npend > 0 && !*abort_flag) {
      if (!hand_over(it - npend)) break;
      --npend;
    }
    // Leaving early (a role gave up): the weight boxes already issued still land in this
    // block's shared memory, so wait for each of them (the last kStages issued hold every
    // slot's last armed phase) before exiting.
    if (pt == 0 && *abort_flag)
      for (uint32_t j = it > (uint32_t)kStages ? it - kStages : 0; j < it; ++j)
        if (!tc::mbar_wait(&tma_full[j % kStages], (j / kStages) & 1, wb)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
  } else if (warp == 0 && !a.stall) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t idesc[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) idesc[j] = tc::idesc_mx8(kBM, BN, j, j);
      const uint32_t idesc_bf = tc::idesc_f16(kBM, BN, 1);
      uint32_t it = 0, acc_it = 0;
      for (int64_t t = blockIdx.x; t < ma.tiles && !*abort_flag; t += gridDim.x) {
        int64_t blk, e;
        int nt;
        if (!tile_info(ma, t, ntpp, blk, nt, e)) continue;
        const uint32_t acc = ma.nacc == 2 ? (acc_it & 1) : 0;
        const uint32_t use = ma.nacc == 2 ? (acc_it >> 1) : acc_it;  // earlier uses of this accumulator
        if (!tc::mbar_wait(&tempty[acc], (use & 1) ^ 1, wb)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d_tmem = taddr + acc * (uint32_t)BN;
        bool ok = true;
        for (int kc = 0; kc < nk; ++kc) {
          const int s = (int)(it % kStages);
          if (!tc::mbar_wait(&full[s], (it / kStages) & 1, wb) || !tc::mbar_wait(&tma_full[s], (it / kStages) & 1, wb)) {
            moe::set_status(a.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t sl = smem_s + s * L.slot;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (BF)  // 16 bf16 of K per MMA: 32 bytes of the 128-byte rows, like 32 E4M3
              tc::mma_f16_ss(d_tmem, tc::sdesc_sw128(sl + L.a + j * 32), tc::sdesc_sw128(sl + L.b + j * 32),
                             idesc_bf, (kc | j) != 0);
            else
            tc::mma_mx8_ss(d_tmem, tc::sdesc_sw128(sl + L.a + j * 32), tc::sdesc_sw128(sl + L.b + j * 32), idesc[j],
                           taddr + sfa_col(s), taddr + sfb_col(s), (kc | j) != 0);
          tc::mma_commit(&empty[s]);
          ++it;
        }
        if (!ok) break;
        tc::mma_commit(&tfull[acc]);
        ++acc_it;
      }
      tc::mma_commit(drain);
      if (!tc::mbar_wait(drain, 0, wb)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp - kEpiWarp0;
    const int r = quarter * 32 + lane;
    const uint16_t* bias = static_cast<const uint16_t*>(a.bias);
    uint32_t acc_it = 0;
    for (int64_t t = blockIdx.x; t < ma.tiles && !*abort_flag; t += gridDim.x) {
      int64_t blk, e;
      int nt;
      if (!tile_info(ma, t, ntpp, blk, nt, e)) continue;
      const uint32_t acc = ma.nacc == 2 ? (acc_it & 1) : 0;
      const uint32_t use = ma.nacc == 2 ? (acc_it >> 1) : acc_it;
      if (!tc::mbar_wait(&tfull[acc], use & 1, wb)) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      const int p = a.sorted[blk * a.bm + r];
      const bool valid = p < a.P;
      const uint32_t tb = taddr + acc * (uint32_t)BN + ((uint32_t)(quarter * 32) << 16);
      if (EPI == EPI_SWIGLU) {  // 128 features: h = silu(gate) * up, quantised 32 at a time
        const int f0 = nt * 128;
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t gv[32], uv[32];
          tc::tmem_ld32(tb + c0, gv);
          tc::tmem_ld32(tb + 128 + c0, uv);
          tc::tmem_ld_wait();
          if (valid) {
            float h[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              float gt = __uint_as_float(gv[j]), up = __uint_as_float(uv[j]);
              if (bias) {
                gt += moe::bf16_bits_to_f32(bias[e * a.Nw + f0 + c0 + j]);
                up += moe::bf16_bits_to_f32(bias[e * a.Nw + a.Nout + f0 + c0 + j]);
              }
              h[j] = moe::silu(gt) * up;
            }
            if (BF) {  // bf16 weights: h in bf16 (RNE)
              uint32_t pk[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                pk[j] = (uint32_t)moe::f32_to_bf16_bits(h[2 * j]) | ((uint32_t)moe::f32_to_bf16_bits(h[2 * j + 1]) << 16);
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + (int64_t)p * a.Nout + f0 + c0);
#pragma unroll
              for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
              continue;
            }
            uint32_t code[8], sc;
            mxq::quant32(h, code, sc);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + (int64_t)p * a.Nout + f0 + c0);
            dst[0] = make_uint4(code[0], code[1], code[2], code[3]);
            dst[1] = make_uint4(code[4], code[5], code[6], code[7]);
            a.out_scale[(int64_t)p * (a.Nout / 32) + (f0 + c0) / 32] = (uint8_t)sc;
          }
        }
      } else {
        const int n0 = nt * BN;
        const float wgt = (EPI == EPI_WEIGHTED_F32 && valid) ? a.topk_w[p] : 1.f;
        // N is a multiple of 128 and n0 of 32: a 32-column chunk is wholly in N or past it
        const int cols = a.Nout - n0 < BN ? a.Nout - n0 : BN;
        for (int c0 = 0; c0 < cols; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(tb + c0, v);
          tc::tmem_ld_wait();
          if (EPI == EPI_WEIGHTED_F32) {
            // this lane's row of the chunk into the box (16-byte chunks swizzled by row), then
            // four rows per instruction out of it: eight lanes store a row's 128 bytes
            const uint32_t box = smem_s + L.stg + quarter * 32 * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float o4[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                o4[i] = __uint_as_float(v[4 * j + i]);
                if (bias) o4[i] += moe::bf16_bits_to_f32(bias[e * a.Nw + n0 + c0 + 4 * j + i]);
                o4[i] *= wgt;
              }
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(box + lane * 128 + ((j ^ (lane & 7)) << 4)),
                           "f"(o4[0]), "f"(o4[1]), "f"(o4[2]), "f"(o4[3])
                           : "memory");
            }
            __syncwarp();
            const int cc = lane & 7;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = (lane >> 3) + 4 * i;
              const int pr = __shfl_sync(0xffffffffu, p, rr);
              float4 w4;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(w4.x), "=f"(w4.y), "=f"(w4.z), "=f"(w4.w)
                           : "r"(box + rr * 128 + ((cc ^ (rr & 7)) << 4))
                           : "memory");
              if (pr < a.P)
                *reinterpret_cast<float4*>(static_cast<float*>(a.out) + (int64_t)pr * a.Nout + n0 + c0 + 4 * cc) = w4;
            }
            __syncwarp();
          } else if (valid) {
            float o[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              o[j] = __uint_as_float(v[j]);
              if (bias) o[j] += moe::bf16_bits_to_f32(bias[e * a.Nw + n0 + c0 + j]);
            }
            {
              uint32_t pk[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                pk[j] = (uint32_t)moe::f32_to_bf16_bits(o[2 * j]) | ((uint32_t)moe::f32_to_bf16_bits(o[2 * j + 1]) << 16);
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + (int64_t)p * a.Nout + n0 + c0);
#pragma unroll
              for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
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
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, kTmemCols);
  }
}

int sm_count_mx8() { return moe_launch::sm_count_current(); }

template <int EPI, bool BF>
cudaError_t launch_mx8(const MArgs& ma, const CUtensorMap& tmap, cudaStream_t stream) {
  const MLayout L = mlayout(ma.BN, EPI == EPI_WEIGHTED_F32);
  cudaError_t err =
      cudaFuncSetAttribute(mx8_gemm_kernel<EPI, BF>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  int64_t grid = sm_count_mx8();
  if (ma.tiles < grid) grid = ma.tiles;
  if (grid <= 0) return cudaSuccess;
  mx8_gemm_kernel<EPI, BF><<<(unsigned)grid, kThreads, L.total, stream>>>(tmap, ma);
  return cudaGetLastError();
}

}  // namespace

namespace moe_launch {

bool mx8_supported(const GroupedGemm& g) {
  const bool bf = g.wfmt == WF_BF16;
  if (bf) {
    // bf16 weights and activations: SwiGLU writes bf16 h (no quantiser)
    if (g.act_fmt != ACT_BF16) return false;
    if (g.epi != EPI_PLAIN_BF16 && g.epi != EPI_WEIGHTED_F32 && g.epi != EPI_SWIGLU) return false;
  } else {
    if (g.wfmt != WF_MXFP8 || g.act_scale == nullptr) return false;
    if (g.epi != EPI_PLAIN_BF16 && g.epi != EPI_WEIGHTED_F32 && !(g.epi == EPI_SWIGLU && g.out_scale)) return false;
  }
  if (g.act_by_slot || g.out_by_slot) return false;
  const int64_t rbytes = bf ? (int64_t)g.Kin * 2 : (int64_t)g.Kin;
  if (g.bm != kBM || g.Kin <= 0 || rbytes % kBK != 0) return false;
  if (g.Nout % 128 != 0) return false;
  if ((int64_t)g.E * g.Nw >= ((int64_t)1 << 31)) return false;  // TMA row coordinates are 32-bit
  // 16-byte copies of activation and weight rows, 4-byte copies of scale words
  const uintptr_t al16 = reinterpret_cast<uintptr_t>(g.act) | reinterpret_cast<uintptr_t>(g.w);
  const uintptr_t al4 = bf ? 0 : (reinterpret_cast<uintptr_t>(g.act_scale) | reinterpret_cast<uintptr_t>(g.w_scale));
  return (al16 & 15) == 0 && (al4 & 3) == 0;
}

cudaError_t mx8_gemm(const GroupedGemm& g, cudaStream_t stream) {
  if (!mx8_supported(g)) return cudaErrorInvalidValue;
  MArgs ma;
  ma.g = g;
  const bool sw = g.epi == EPI_SWIGLU;
  // SwiGLU: 128 features (gate and up rows) per tile, one accumulator.  The routing-weighted
  // fp32 epilogue (twice the output bytes of the bf16 one) overlaps the next tile's MMAs:
  // 224 rows per tile (the last one may reach past N) in two accumulators; measured on the
  // 7168-wide GEMM2 of the MXFP8 layer, 2.33 -> 2.19 ms.  The bf16 epilogue keeps one
  // accumulator of 256 rows (224 measured slower there: 2.44 -> 2.71 ms on N = 4096).
  ma.BN = sw ? 256 : (g.epi == EPI_WEIGHTED_F32 ? 224 : (g.Nout % 256 == 0 ? 256 : 128));
  ma.nacc = ma.BN <= 224 ? 2 : 1;
  ma.n_tiles = sw ? g.Nout / 128 : (g.Nout + ma.BN - 1) / ma.BN;
  ma.tiles = g.grid_blocks * ma.n_tiles;
  // weights as E * Nw rows of Kin (E4M3) or 2 Kin (bf16) bytes; boxes of 128 bytes x BN rows
  // in the 128-byte swizzle
  const bool bf = g.wfmt == WF_BF16;
  const uint64_t rbytes = bf ? (uint64_t)g.Kin * 2 : (uint64_t)g.Kin;
  CUtensorMap tmap;
  if (!tma::encode_2d_u8(&tmap, g.w, rbytes, (uint64_t)g.E * g.Nw, rbytes, kBK, sw ? 128 : ma.BN, true))
    return cudaErrorInvalidValue;
  if (bf) {
    if (g.epi == EPI_SWIGLU) return launch_mx8<EPI_SWIGLU, true>(ma, tmap, stream);
    if (g.epi == EPI_WEIGHTED_F32) return launch_mx8<EPI_WEIGHTED_F32, true>(ma, tmap, stream);
    return launch_mx8<EPI_PLAIN_BF16, true>(ma, tmap, stream);
  }
  if (g.epi == EPI_SWIGLU) return launch_mx8<EPI_SWIGLU, false>(ma, tmap, stream);
  if (g.epi == EPI_WEIGHTED_F32) return launch_mx8<EPI_WEIGHTED_F32, false>(ma, tmap, stream);
  return launch_mx8<EPI_PLAIN_BF16, false>(ma, tmap, stream);
}

}  // namespace moe_launch
