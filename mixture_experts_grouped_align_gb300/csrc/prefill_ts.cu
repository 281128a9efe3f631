// Grouped expert GEMM for W4A16 prefill shapes with the weights as the tensor-memory
// operand of tcgen05.mma.
//
// D[f, t] = sum_k W[e, f, k] * x[row(t), k] over one alignment block of 128 pairs t and 128
// output features f of the block's expert e ("Add MoE GEMM variants and weight-gradient
// kernel", aiter PR 5310, Summary: all expert GEMMs in one launch; "Bound Triton MoE JIT
// specializations via token-dim bucketing and warmup", TensorRT-LLM PR 15311, Description:
// the W4A16 MXFP4 path, E2M1 weights with one E8M0 scale per 32 K elements, 16-bit
// activations).  Tiles past num_tokens_post_padded or of the -1 sentinel are skipped by every
// role before anything is read (second review of the aiter page); expert offsets are 64-bit.
//
// Why this shape.  The weights must be decoded (E2M1 codes times the block scale, to f16)
// before an f16 MMA can use them.  Writing the decoded weights to shared memory and reading
// them back as an MMA operand costs more shared-memory bandwidth than the MMA leaves free;
// decoded into tensor memory they cost none: tcgen05.mma reads its A operand (M = 128
// weight rows x K) straight from TMEM and only the token tile B (N = 128 rows x K) from
// shared memory.  SwiGLU pairs gate row f and up row f in the same TMEM lane: the two
// matrices are two MMAs into two accumulators G and U.
//
// Every tile is two 128-row weight matrices against one token tile of 128 slots: the gate and
// up rows of 128 features for SwiGLU, else 256 consecutive features; reading the token tile
// once for both halves its L2 traffic per flop.  Per thread block (one per SM, 640 threads),
// persistent over (alignment block, feature tile):
//   warp 0      allocates the 512 TMEM columns (the two 128-column accumulators in 0..255,
//               the decoded weight stages in 256..511);
//   warps 2-3   issue the MMAs, one lane each, warp 2 + m for weight matrix m (M = 128,
//               N = 128, K = 16);
//   warp 1      loads each 64-wide K stage of the token tile with TMA (one box of 128 slot
//               rows when the rows are in slot order, else gathered four rows per
//               instruction) and the raw E2M1 codes 128 bytes (four stages) per weight row;
//   warps 8-15  decode: one thread per weight row (= TMEM lane) turns the stage's codes into
//               f16 (hardware conversion, times the block's E8M0 scale, read a group ahead)
//               and writes them into the stage's TMEM columns with tcgen05.st;
//   warps 4-7 and 16-19 drain the accumulators (one TMEM lane = one feature, one column =
//               one pair; each group of four takes half of the columns), release them before
//               computing the last chunk, and run the fused epilogue: bias + SwiGLU or
//               bias + relu^2 -> h (f16, through a shared staging tile and TMA stores when h
//               is in slot order), bias * routing weight -> o (fp32), or bias -> out (bf16).
// Every mbarrier wait is bounded; one that runs out sets MOE_ERR_TIMEOUT, every role leaves
// its loop, the copy warp waits for the loads it has issued, the MMA lane drains its own work
// and the TMEM is freed.  In the stalled self-test (GroupedGemm::stall) the copy warp and the
// MMA lanes do nothing, so the decoders and the epilogue wait on barriers no one arrives on
// and give up after GroupedGemm::wait_ns with no copy or MMA in flight.
//
// f16 operands: a decoded weight code * 2^se is exact when se is within -23..13.  The main
// launch decodes every block that way and only marks a tile (a bit in GroupedGemm::fix_bits,
// counted in fix_count) when one of its blocks with nonzero codes has a scale outside that
// window; a second launch of the same kernel (FIX) then does exactly the marked tiles again,
// with every weight row decoded as code * 2^(se - c) for one shift c per row (its largest
// block scale mapped to 2^13) and the row's accumulator multiplied by 2^c in the epilogue:
// a power of two, so the result is the same as with exact f16 weights.  It exits at once
// when no tile is marked, so weights with ordinary scales cost one empty launch.  Only a
// row whose nonzero blocks span more than 36 octaves of scale still has a block outside
// the window; it sets MOE_ERR_RANGE (as does any out-of-window block when the caller gives
// no room for the marks).  Each output
// depends on its own token row only and K is always reduced in the same order, so padded
// and unpadded batches give identical real rows.
#include "moe_common.cuh"
#include "moe_launch.h"
#include "tcgen05.cuh"
#include "tma.cuh"
#include "ts_common.cuh"

namespace {

using namespace moe_launch;
using ts::decode_block;
using ts::mma_ts;
using ts::tma_gather4;
using ts::tmem_st16;

constexpr int kThreads = 640;
constexpr int kTM = 128;    // weight rows (features) per tile: MMA M
constexpr int kTN = 128;    // pairs per tile (one alignment block): MMA N
constexpr int kBK = 64;     // K elements per stage
// Shared-memory stages (token tile + raw codes) and TMEM stages (decoded weights) form two
// rings: copies may run further ahead of the MMA than the TMEM columns allow decoding to.
// Every tile is two 128-row weight matrices against one token tile: the gate and up rows of
// 128 features for SwiGLU, else 256 consecutive features.  The token tile is read once for
// both, which halves its L2 traffic per flop.
constexpr int kMats = 2;
// (fewer stages where the h staging tile takes shared memory: 128 x 128 f16 for SwiGLU,
// 128 x 256 for relu^2)
__host__ __device__ constexpr int smem_stages(int epi) { return epi == EPI_SWIGLU ? 5 : (epi == EPI_RELU2 ? 4 : 7); }
__host__ __device__ constexpr int stage_out_bytes(int epi) {
  return epi == EPI_SWIGLU ? kTN * kTM * 2 : (epi == EPI_RELU2 ? kMats * kTN * kTM * 2 : 0);
}
constexpr int kTmemStages = 4;
// epilogue warps 4-7 take token columns 0-63, warps 16-19 columns 64-127 (warp % 4 = TMEM
// lane quarter); decoders are warps 8-15
constexpr int kMmaWarp0 = 2, kEpiWarp0 = 4, kEpiWarp1 = 16, kDecWarp0 = 8;
constexpr int kEpiCols = kTN / 2;
constexpr int kTmemCols = 512;
constexpr int kAcol0 = 256;  // first TMEM column of the decoded weight stages
constexpr int kMaxKin = 1 << 16;  // a sanity bound: every loop and coordinate takes far more
// The raw codes of a weight row are loaded 128 bytes (four K stages) per TMA box, into a
// ring of their own.
constexpr int kGroup = 4;
constexpr int kRawSlots = 3;

struct TArgs {
  GroupedGemm g;
  int m_tiles;       // feature tiles per block: ceil(Nout / 128) for SwiGLU, else ceil(Nout / 256)
  int64_t tiles;     // block slots * m_tiles
};

// Shared memory: token-tile stages (16 KB each) | raw-code slots (2 x 128 rows x 128 B,
// 128-byte swizzle) | h output staging (128 slots x 128 f16 per matrix) | barriers.
struct TLayout {
  int slot, raw, raw_slot, stg, bars, shift, total;
};

__host__ __device__ inline TLayout tlayout(int epi) {
  TLayout L;
  L.slot = kTN * 128;
  L.raw = smem_stages(epi) * L.slot;
  L.raw_slot = kMats * kTM * 128;
  L.stg = L.raw + kRawSlots * L.raw_slot;
  L.bars = L.stg + stage_out_bytes(epi);
  L.shift = L.bars + 512;  // [2 tiles][kMats][kTM] int8 row shifts
  L.total = L.shift + 2 * kMats * kTM + 1024;
  return L;
}

template <bool FIX = false>
__device__ __forceinline__ bool tile_info(const TArgs& ta, int64_t t, int ntpp, int64_t& blk, int& mt,
                                          int64_t& e) {
  blk = t / ta.m_tiles;
  mt = (int)(t - blk * ta.m_tiles);
  if (blk * ta.g.bm >= ntpp) return false;
  if (FIX && ((ta.g.fix_bits[t >> 5] >> (t & 31)) & 1u) == 0) return false;  // only the marked tiles
  e = ta.g.expert_ids[blk];
  return e >= 0 && e < ta.g.E;
}

// Marks tile t for the FIX launch (counted once).
__device__ __forceinline__ void mark_tile(const GroupedGemm& a, int64_t t) {
  const uint32_t bit = 1u << (t & 31);
  if ((atomicOr(&a.fix_bits[t >> 5], bit) & bit) == 0) atomicAdd(a.fix_count, 1);
}

// First tile of this block's sequence at or after t that some role works on (or >= tiles).
template <bool FIX>
__device__ __forceinline__ int64_t next_tile(const TArgs& ta, int64_t t, int ntpp) {
  int64_t blk, e;
  int mt;
  while (t < ta.tiles && !tile_info<FIX>(ta, t, ntpp, blk, mt, e)) t += gridDim.x;
  return t;
}

// E8M0 byte of a block scale divided by 2^c (the row's shift): NaN (0xFF) stays NaN, and a
// byte pushed below 0x00 is clamped there (a block with nonzero codes is then reported by
// decode_block).
__device__ __forceinline__ uint32_t shifted_scale(uint32_t sb, int c) {
  if (sb == 255u || c == 0) return sb;
  const int v = (int)sb - c;
  return (uint32_t)(v < 0 ? 0 : (v > 254 ? 254 : v));
}

// 2^c as a float for -149 <= c <= 127 (1 for c = 0).
__device__ __forceinline__ float pow2f(int c) {
  if (c >= -126) return __uint_as_float((uint32_t)(c + 127) << 23);
  return __uint_as_float(1u << (c + 149));
}

// TMEM column of stage s, matrix m, in the decoded-weight region.
__device__ __forceinline__ uint32_t a_col(int s, int m) { return kAcol0 + s * 32 * kMats + 32 * m; }

// Output feature of row r of matrix m in feature tile mt, and the weight row that holds it.
template <bool SWIGLU>
__device__ __forceinline__ int64_t tile_feature(int mt, int m, int r) {
  return SWIGLU ? (int64_t)mt * kTM + r : (int64_t)mt * (kMats * kTM) + m * kTM + r;
}
template <bool SWIGLU>
__device__ __forceinline__ int64_t tile_wrow(const GroupedGemm& a, int64_t e, int mt, int m, int r) {
  return e * a.Nw + (SWIGLU ? (int64_t)m * a.Nout : 0) + tile_feature<SWIGLU>(mt, m, r);
}

template <int EPI, bool FIX>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_ts_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_h, TArgs ta) {
  constexpr bool SW = (EPI == EPI_SWIGLU);
  const GroupedGemm& a = ta.g;
  if (FIX && *a.fix_count == 0) return;  // no marked tile: nothing to do again
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr bool R2 = (EPI == EPI_RELU2);
  const TLayout L = tlayout(EPI);
  constexpr int S1 = smem_stages(EPI), S2 = kTmemStages;
  uint64_t* ld_full = reinterpret_cast<uint64_t*>(smem + L.bars);  // [S1] token tile + raw codes landed
  uint64_t* empty = ld_full + S1;                                   // [S1] shared stage consumed by the MMA
  uint64_t* a_full = empty + S1;                                    // [S2] decoded weights in TMEM
  uint64_t* a_empty = a_full + S2;                                  // [S2] TMEM stage consumed by the MMA
  uint64_t* raw_full = a_empty + S2;                                // [kRawSlots] raw codes landed
  uint64_t* raw_empty = raw_full + kRawSlots;                       // [kRawSlots] decoded by all
  uint64_t* tfull = raw_empty + kRawSlots;                          // [2]
  uint64_t* tempty = tfull + 2;                                     // [2]
  uint64_t* drain = tempty + 2;
  uint64_t* epi_bar = drain + 1;  // the eight epilogue warps meet here (bounded, unlike bar.sync)
  uint64_t* shift_full = epi_bar + 1;  // [2] FIX: a tile's row shifts written (by tile parity)
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(shift_full + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_s + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < S1; ++s) {
      tc::mbar_init(&ld_full[s], 1);
      tc::mbar_init(&empty[s], kMats);
    }
    for (int s = 0; s < S2; ++s) {
      tc::mbar_init(&a_full[s], 8);
      tc::mbar_init(&a_empty[s], kMats);
    }
    for (int s = 0; s < kRawSlots; ++s) {
      tc::mbar_init(&raw_full[s], 1);
      tc::mbar_init(&raw_empty[s], 8);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&tfull[i], kMats);
      tc::mbar_init(&tempty[i], 8);
    }
    tc::mbar_init(drain, kMats);
    tc::mbar_init(epi_bar, 8);
    tc::mbar_init(&shift_full[0], 8);
    tc::mbar_init(&shift_full[1], 8);
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
  const uint32_t smem_s = tc::smem_addr(smem);
  bool bad = false;
  // the limit of every wait (a caller's short limit only in the stalled self-test)
  const uint64_t wb = a.wait_ns > 0 ? (uint64_t)a.wait_ns : tc::kWaitNs;

  if (warp == 1 && !a.stall) {
    // ------------------------------------------------------------------ TMA loads
    if (lane == 0) {
      tma::prefetch_map(&tmap_x);
      tma::prefetch_map(&tmap_w);
    }
    const int64_t rows_total = a.act_per_pair ? a.P : a.P / a.k;
    const uint32_t stage_bytes = kTN * 128;
    const uint32_t raw_bytes = kMats * kTM * 128;
    uint32_t it = 0, gi = 0;
    for (int64_t t = blockIdx.x; t < ta.tiles && !*abort_flag; t += gridDim.x) {
      int64_t blk, e;
      int mt;
      if (!tile_info<FIX>(ta, t, ntpp, blk, mt, e)) continue;
      // token rows of slots 4 lane .. 4 lane + 3 (this lane's gather); an empty slot reads
      // past the end of the activations (zeros).  Rows already in slot order need no gather.
      int32_t y[4] = {0, 0, 0, 0};
      if (!a.act_by_slot) {
        const int4 p4 = *reinterpret_cast<const int4*>(a.sorted + blk * a.bm + 4 * lane);
        const int pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          y[j] = (int32_t)(pv[j] < a.P ? (a.act_per_pair ? (int64_t)pv[j] : (int64_t)(pv[j] / a.k)) : rows_total);
      }
      bool ok = true;
      for (int kc = 0; kc < nk; ++kc) {
        if (kc % kGroup == 0) {  // raw codes of stages kc .. kc + 3: 128 bytes of every row
          const int rs = (int)(gi % kRawSlots);
          if (lane == 0) ok = tc::mbar_wait(&raw_empty[rs], ((gi / kRawSlots) & 1) ^ 1, wb);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (lane == 0) {
            const uint32_t rsl = smem_s + L.raw + rs * L.raw_slot;
            tma::mbar_arrive_expect_tx(&raw_full[rs], raw_bytes);
#pragma unroll
            for (int m = 0; m < kMats; ++m)
              tma::load_2d(rsl + m * kTM * 128, &tmap_w, (kc / kGroup) * 128, (int32_t)tile_wrow<SW>(a, e, mt, m, 0),
                           &raw_full[rs]);
          }
          ++gi;
        }
        const int s = (int)(it % S1);
        if (lane == 0) ok = tc::mbar_wait(&empty[s], ((it / S1) & 1) ^ 1, wb);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t sl = smem_s + s * L.slot;
        if (lane == 0) tma::mbar_arrive_expect_tx(&ld_full[s], stage_bytes);
        __syncwarp();
        if (a.act_by_slot) {  // the block's 128 slot rows: one box
          if (lane == 0) tma::load_2d(sl, &tmap_x, kc * 128, (int32_t)(blk * a.bm), &ld_full[s]);
        } else {  // rows 4 lane .. 4 lane + 3 of the token tile: every lane issues its own gather
          tma_gather4(sl + lane * 512, &tmap_x, kc * 128, y[0], y[1], y[2], y[3], &ld_full[s]);
        }
        ++it;
      }
      if (!ok) {
        if (lane == 0) moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
    }
    // Leaving early (another role gave up): the loads already issued still land in this
    // block's shared memory, so wait for each armed stage and code group before exiting.
    // Every slot's last armed phase is one of the last S1 stages (kRawSlots groups) issued.
    if (*abort_flag && lane == 0) {
      for (uint32_t j = it > (uint32_t)S1 ? it - S1 : 0; j < it; ++j)
        if (!tc::mbar_wait(&ld_full[j % S1], (j / S1) & 1, wb)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
      for (uint32_t j = gi > (uint32_t)kRawSlots ? gi - kRawSlots : 0; j < gi; ++j)
        if (!tc::mbar_wait(&raw_full[j % kRawSlots], (j / kRawSlots) & 1, wb)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
    }
  } else if (warp >= kDecWarp0 && warp < kDecWarp0 + 8) {
    // ------------------------------------------------------------------ decoders
    const int dj = warp - kDecWarp0, q = dj & 3, part = dj >> 2;
    const int m = part;          // matrix (SwiGLU: gate, up; else the two feature halves)
    const int r = 32 * q + lane;  // tile row = TMEM lane
    const int ngroups = (nk + kGroup - 1) / kGroup;
    // The eight E8M0 bytes of this row's K group g (blocks 8g .. 8g + 7), read from global
    // memory one group ahead into registers; 127 (scale 1) for a row past the features.
    auto load_scales = [&](int64_t e, int mt, int g, uint32_t (&w)[2]) {
      w[0] = w[1] = 0x7f7f7f7fu;
      if (tile_feature<SW>(mt, m, r) >= a.Nout) return;
      const uint8_t* src = a.w_scale + tile_wrow<SW>(a, e, mt, m, r) * nkb + 8 * g;
      uint32_t v[2] = {0u, 0u};
#pragma unroll
      for (int bb = 0; bb < 8; ++bb)
        if (8 * g + bb < nkb) v[bb >> 2] |= (uint32_t)__ldg(src + bb) << (8 * (bb & 3));
      w[0] = v[0];
      w[1] = v[1];
    };
    // The shift c of this row for the tile (0 when every block scale is in the f16 window;
    // else the largest block scale is mapped to 2^13), written for the epilogue at
    // shift[tile parity][m][r].
    auto row_shift = [&](int64_t e, int mt) -> int {
      if (tile_feature<SW>(mt, m, r) >= a.Nout) return 0;
      const uint8_t* src = a.w_scale + tile_wrow<SW>(a, e, mt, m, r) * nkb;
      int mx = 0, mn = 254;
      for (int b = 0; b < nkb; ++b) {
        const int sb = __ldg(src + b);
        if (sb != 255) {
          mx = sb > mx ? sb : mx;
          mn = sb < mn ? sb : mn;
        }
      }
      return (mx <= 127 + 13 && mn >= 127 - 23) ? 0 : mx - (127 + 13);
    };
    int8_t* shift_s = reinterpret_cast<int8_t*>(smem + L.shift);
    uint32_t tseq = 0;
    uint32_t it = 0, gi = 0;
    int64_t t = next_tile<FIX>(ta, blockIdx.x, ntpp);
    int64_t blk = 0, e = 0;
    int mt = 0;
    uint32_t sc_next[2] = {0x7f7f7f7fu, 0x7f7f7f7fu};
    if (t < ta.tiles) {
      tile_info<FIX>(ta, t, ntpp, blk, mt, e);
      load_scales(e, mt, 0, sc_next);
    }
    while (t < ta.tiles && !*abort_flag) {
      // the next tile in this block's sequence, read now for the scale prefetch of its first group
      const int64_t tn = t + gridDim.x;
      const int64_t blk_n = tn / ta.m_tiles;
      const int mt_n = (int)(tn - blk_n * ta.m_tiles);
      const bool live_n = tn < ta.tiles && blk_n * a.bm < ntpp &&
                          (!FIX || ((a.fix_bits[tn >> 5] >> (tn & 31)) & 1u) != 0);
      const int64_t e_n = live_n ? (int64_t)a.expert_ids[blk_n] : -1;
      const bool next_ok = e_n >= 0 && e_n < a.E;
      int csh = 0;
      if (FIX) {  // this row's shift, for the decoding below and (through shift_full) the epilogue
        csh = row_shift(e, mt);
        csh = csh < -128 ? -128 : (csh > 127 ? 127 : csh);
        shift_s[((tseq & 1) * kMats + m) * kTM + r] = (int8_t)csh;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&shift_full[tseq & 1]);
      }
      ++tseq;
      bool oow = false;  // a block with nonzero codes outside the f16 window
      bool ok = true;
      uint32_t sc0 = 0u, sc1 = 0u;
      int rs = 0;
      for (int kc = 0; kc < nk; ++kc) {
        const int kg = kc % kGroup, g = kc / kGroup;
        if (kg == 0) {  // a new group of raw codes: its scales are the prefetched ones
          rs = (int)(gi % kRawSlots);
          sc0 = sc_next[0];
          sc1 = sc_next[1];
          if (g + 1 < ngroups) load_scales(e, mt, g + 1, sc_next);
          else if (next_ok) load_scales(e_n, mt_n, 0, sc_next);
          if (!tc::mbar_wait(&raw_full[rs], (gi / kRawSlots) & 1, wb)) {
            ok = false;
            break;
          }
        }
        const int s2 = (int)(it % S2);
        if (!tc::mbar_wait(&a_empty[s2], ((it / S2) & 1) ^ 1, wb)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();  // the MMA that read this TMEM stage before has completed
        // row r of the slot, bytes 32 kg + 16 h of the row, in the 128-byte swizzle
        const uint8_t* rowp = smem + L.raw + rs * L.raw_slot + m * kTM * 128 + r * 128;
        const uint32_t dst = taddr + ((uint32_t)(32 * q) << 16) + a_col(s2, m);
        const uint32_t scw = (kg >> 1) ? sc1 : sc0;  // scale bytes of blocks 2 kg, 2 kg + 1
        const int sh = 16 * (kg & 1);
        {
          uint32_t v[32];
          const uint4 w0 = *reinterpret_cast<const uint4*>(rowp + (((2 * kg) ^ (r & 7)) << 4));
          const uint4 w1 = *reinterpret_cast<const uint4*>(rowp + (((2 * kg + 1) ^ (r & 7)) << 4));
          if (FIX) {
            decode_block(w0, shifted_scale((scw >> sh) & 0xffu, csh), v, oow);
            decode_block(w1, shifted_scale((scw >> (sh + 8)) & 0xffu, csh), v + 16, oow);
          } else {
            decode_block(w0, (scw >> sh) & 0xffu, v, oow);
            decode_block(w1, (scw >> (sh + 8)) & 0xffu, v + 16, oow);
          }
          tmem_st16(dst, v);
          tmem_st16(dst + 16, v + 16);
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&a_full[s2]);
        if (kg == kGroup - 1 || kc == nk - 1) {  // this group's raw codes are decoded
          if (lane == 0) tc::mbar_arrive(&raw_empty[rs]);
          ++gi;
        }
        ++it;
      }
      if (!ok) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      // an out-of-window block: the FIX launch does the tile again (or, out of room for the
      // marks or in that launch itself, the block cannot be exact: reported)
      if (oow) {
        if (!FIX && a.fix_bits) mark_tile(a, t);
        else bad = true;
      }
      if (next_ok) {
        t = tn;
        blk = blk_n;
        mt = mt_n;
        e = e_n;
      } else {  // no live next tile, or an expert id the roles skip: search on
        t = next_tile<FIX>(ta, tn, ntpp);
        if (t < ta.tiles) {
          tile_info<FIX>(ta, t, ntpp, blk, mt, e);
          load_scales(e, mt, 0, sc_next);
        }
      }
    }
  } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kMats && !a.stall) {
    // ------------------------------------------------------------------ MMA issuers
    // one thread per weight matrix, in two warps on different SM sub-partitions: the waits,
    // commits and issues of a stage cost the issuing thread about as long as the tensor core
    // needs for the stage's MMAs, so one thread alone would pace the tensor core
    const int m = warp - kMmaWarp0;
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(kTM, kTN, 0);
      uint32_t it = 0, acc_it = 0;
      for (int64_t t = blockIdx.x; t < ta.tiles && !*abort_flag; t += gridDim.x) {
        int64_t blk, e;
        int mt;
        if (!tile_info<FIX>(ta, t, ntpp, blk, mt, e)) continue;
        const int acc = 0;  // one accumulator set (two 128-column accumulators)
        if (!tc::mbar_wait(&tempty[acc], (acc_it & 1) ^ 1, wb)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        bool ok = true;
        for (int kc = 0; kc < nk; ++kc) {
          const int s = (int)(it % S1), s2 = (int)(it % S2);
          if (!tc::mbar_wait(&ld_full[s], (it / S1) & 1, wb) || !tc::mbar_wait(&a_full[s2], (it / S2) & 1, wb)) {
            moe::set_status(a.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t bs = smem_s + s * L.slot;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_ts(taddr + m * 128, taddr + a_col(s2, m) + kk * 8, tc::sdesc_sw128(bs + kk * 32), idesc,
                   (kc | kk) != 0);
          tc::mma_commit(&empty[s]);
          tc::mma_commit(&a_empty[s2]);
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
  } else if ((warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) || warp >= kEpiWarp1) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int cbase = warp >= kEpiWarp1 ? kEpiCols : 0;  // this warp's token columns
    const uint16_t* bias = static_cast<const uint16_t*>(a.bias);
    // SwiGLU or relu^2 into slot-ordered h: the tile goes through shared memory and leaves
    // as one TMA store per 128 features, and the accumulators are released before the last
    // chunk is computed
    const bool staged = (SW || R2) && a.out_by_slot;
    __half* stg = reinterpret_cast<__half*>(smem + L.stg);
    const uint32_t stg_s = smem_s + L.stg;
    uint32_t acc_it = 0, eb_it = 0;
    // all four epilogue warps reach this point (a wait that runs out aborts the kernel)
    auto epi_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(epi_bar);
      const bool ok = tc::mbar_wait(epi_bar, eb_it & 1, wb);
      ++eb_it;
      if (!ok) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      return ok;
    };
    for (int64_t t = blockIdx.x; t < ta.tiles && !*abort_flag; t += gridDim.x) {
      int64_t blk, e;
      int mt;
      if (!tile_info<FIX>(ta, t, ntpp, blk, mt, e)) continue;
      const int acc = 0;  // one accumulator set
      int pls[kEpiCols / 32];  // pair of token column cbase + 32 i + lane, read while the MMAs run
      float wls[kEpiCols / 32];
#pragma unroll
      for (int i = 0; i < kEpiCols / 32; ++i) pls[i] = a.sorted[blk * a.bm + cbase + 32 * i + lane];
      const int64_t slot0 = blk * a.bm;
#pragma unroll
      for (int i = 0; i < kEpiCols / 32; ++i)
        wls[i] = (EPI == EPI_WEIGHTED_F32 && pls[i] < a.P) ? a.topk_w[pls[i]] : 1.f;
      if (!tc::mbar_wait(&tfull[acc], acc_it & 1, wb)) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      // this lane's features: SwiGLU gate (accumulator 0) and up (1) of feature fA; otherwise
      // feature fA in accumulator 0 and fB in accumulator 1
      const int64_t fA = tile_feature<SW>(mt, 0, 32 * q + lane), fB = tile_feature<SW>(mt, 1, 32 * q + lane);
      const bool vA = fA < a.Nout, vB = fB < a.Nout;
      // FIX: 2^c of the two rows of this lane (their weights were decoded with 2^-c)
      float fsA = 1.f, fsB = 1.f;
      if (FIX) {
        if (!tc::mbar_wait(&shift_full[acc_it & 1], (acc_it >> 1) & 1, wb)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const int8_t* shift_s = reinterpret_cast<const int8_t*>(smem + L.shift) + (acc_it & 1) * kMats * kTM;
        fsA = pow2f(shift_s[32 * q + lane]);
        fsB = pow2f(shift_s[kTM + 32 * q + lane]);
      }
      float b0 = 0.f, b1 = 0.f;
      if (bias) {
        if (vA) b0 = moe::bf16_bits_to_f32(bias[e * a.Nw + fA]);
        if (SW && vA) b1 = moe::bf16_bits_to_f32(bias[e * a.Nw + a.Nout + fA]);
        if (!SW && vB) b1 = moe::bf16_bits_to_f32(bias[e * a.Nw + fB]);
      }
      const uint32_t tb = taddr + ((uint32_t)(32 * q) << 16);
      if (staged) {  // the previous tile's store has finished reading the staging buffer
        if (warp == kEpiWarp0 && lane == 0) tma::bulk_wait_read_all();
        if (!epi_sync()) break;
      }
#pragma unroll
      for (int cc = 0; cc < kEpiCols; cc += 32) {
        const int c0 = cbase + cc;
        const int pl = pls[cc / 32];
        uint32_t v0[32], v1[32];
        tc::tmem_ld32(tb + c0, v0);
        tc::tmem_ld32(tb + 128 + c0, v1);
        tc::tmem_ld_wait();
        if (cc == kEpiCols - 32) {  // this warp's accumulator columns are drained
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&tempty[acc]);
        }
        if (SW) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int p = __shfl_sync(0xffffffffu, pl, j);
            const float gt = __uint_as_float(v0[j]) * fsA + b0, up = __uint_as_float(v1[j]) * fsB + b1;
            const __half hv = __float2half_rn(moe::silu(gt) * up);
            if (p < a.P && vA && __hisinf(hv)) bad = true;
            if (staged) {
              stg[(c0 + j) * kTM + 32 * q + lane] = hv;
            } else if (p < a.P && vA) {
              const int64_t row = a.out_by_slot ? slot0 + c0 + j : (int64_t)p;
              static_cast<__half*>(a.out)[row * a.Nout + fA] = hv;
            }
          }
        } else if (R2) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int p = __shfl_sync(0xffffffffu, pl, j);
            const __half hA = __float2half_rn(moe::relu2(__uint_as_float(v0[j]) * fsA + b0));
            const __half hB = __float2half_rn(moe::relu2(__uint_as_float(v1[j]) * fsB + b1));
            if (p < a.P && ((vA && __hisinf(hA)) || (vB && __hisinf(hB)))) bad = true;
            if (staged) {
              stg[(c0 + j) * kTM + 32 * q + lane] = hA;
              stg[kTN * kTM + (c0 + j) * kTM + 32 * q + lane] = hB;
            } else if (p < a.P) {
              const int64_t row = a.out_by_slot ? slot0 + c0 + j : (int64_t)p;
              if (vA) static_cast<__half*>(a.out)[row * a.Nout + fA] = hA;
              if (vB) static_cast<__half*>(a.out)[row * a.Nout + fB] = hB;
            }
          }
        } else {
          const float wl = wls[cc / 32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int p = __shfl_sync(0xffffffffu, pl, j);
            const float wp = __shfl_sync(0xffffffffu, wl, j);
            if (p < a.P) {
              const int64_t row = a.out_by_slot ? slot0 + c0 + j : (int64_t)p;
              const float o0 = __uint_as_float(v0[j]) * fsA + b0, o1 = __uint_as_float(v1[j]) * fsB + b1;
              if (EPI == EPI_WEIGHTED_F32) {
                if (vA) static_cast<float*>(a.out)[row * a.Nout + fA] = o0 * wp;
                if (vB) static_cast<float*>(a.out)[row * a.Nout + fB] = o1 * wp;
              } else {
                if (vA) static_cast<uint16_t*>(a.out)[row * a.Nout + fA] = moe::f32_to_bf16_bits(o0);
                if (vB) static_cast<uint16_t*>(a.out)[row * a.Nout + fB] = moe::f32_to_bf16_bits(o1);
              }
            }
          }
        }
      }
      if (staged) {  // the tile's h rows [slot0, slot0 + 128) x its features, 128 per box
        tc::fence_proxy_async_smem();
        if (!epi_sync()) break;
        if (warp == kEpiWarp0 && lane == 0) {
          if (SW) {
            tma::store_2d(&tmap_h, mt * kTM * 2, (int32_t)slot0, stg_s);
          } else {
#pragma unroll
            for (int m = 0; m < kMats; ++m)  // a box past the last feature is not stored
              if (tile_feature<false>(mt, m, 0) < a.Nout)
                tma::store_2d(&tmap_h, (int32_t)tile_feature<false>(mt, m, 0) * 2, (int32_t)slot0,
                              stg_s + m * kTN * kTM * 2);
          }
          tma::bulk_commit();
        }
      }
      ++acc_it;
    }
    if (staged && warp == kEpiWarp0 && lane == 0) tma::bulk_wait_all();
  }
  if (bad) moe::set_status(a.status, MOE_ERR_RANGE);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, kTmemCols);
  }
}

int sm_count_ts() { return moe_launch::sm_count_current(); }

template <int EPI, bool FIX>
cudaError_t launch_ts1(const TArgs& ta, const CUtensorMap& mx, const CUtensorMap& mw, const CUtensorMap& mh,
                       cudaStream_t stream) {
  const TLayout L = tlayout(EPI);
  cudaError_t err =
      cudaFuncSetAttribute(prefill_ts_kernel<EPI, FIX>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  int64_t grid = sm_count_ts();
  if (ta.tiles < grid) grid = ta.tiles;
  if (grid <= 0) return cudaSuccess;
  prefill_ts_kernel<EPI, FIX><<<(unsigned)grid, kThreads, L.total, stream>>>(mx, mw, mh, ta);
  return cudaGetLastError();
}

// The main launch, then (with room for the marks) the launch that does the marked tiles
// again; the caller zeroed the marks and their count.
template <int EPI>
cudaError_t launch_ts(const TArgs& ta, const CUtensorMap& mx, const CUtensorMap& mw, const CUtensorMap& mh,
                      cudaStream_t stream) {
  cudaError_t err = launch_ts1<EPI, false>(ta, mx, mw, mh, stream);
  if (err != cudaSuccess || ta.g.fix_bits == nullptr) return err;
  return launch_ts1<EPI, true>(ta, mx, mw, mh, stream);
}

}  // namespace

namespace moe_launch {

// An upper bound of the tiles of any epilogue: 128 features per tile (SwiGLU; the others
// take 256 per tile).
int64_t ts_fix_tiles(int64_t blocks, int64_t nout) { return blocks * ((nout + kTM - 1) / kTM); }

size_t ts_fix_bytes(int64_t blocks, int64_t nout) {
  const int64_t words = (ts_fix_tiles(blocks, nout) + 31) / 32;
  return (size_t)(256 + (words * 4 + 255) / 256 * 256);
}

bool ts_supported(const GroupedGemm& g) {
  if (g.wfmt != WF_MXFP4 || g.act_fmt != ACT_F16) return false;
  if (g.epi != EPI_SWIGLU && g.epi != EPI_RELU2 && g.epi != EPI_WEIGHTED_F32 && g.epi != EPI_PLAIN_BF16)
    return false;
  if (g.bm != kTN || g.Kin <= 0 || g.Kin % kBK != 0 || g.Kin > kMaxKin) return false;
  const int64_t rows_total = g.act_by_slot ? g.grid_blocks * g.bm : (g.act_per_pair ? g.P : g.P / g.k);
  if (rows_total >= ((int64_t)1 << 31) - 1 || (int64_t)g.E * g.Nw >= ((int64_t)1 << 31)) return false;
  // TMA sources and destinations 16-byte aligned
  uintptr_t al16 = reinterpret_cast<uintptr_t>(g.act) | reinterpret_cast<uintptr_t>(g.w);
  if (g.out_by_slot) al16 |= reinterpret_cast<uintptr_t>(g.out);
  if ((al16 & 15) != 0) return false;
  return tlayout(g.epi).total <= 227 * 1024;
}

cudaError_t prefill_ts(const GroupedGemm& g, cudaStream_t stream) {
  if (!ts_supported(g)) return cudaErrorInvalidValue;
  TArgs ta;
  ta.g = g;
  const int tile_features = g.epi == EPI_SWIGLU ? kTM : kMats * kTM;
  ta.m_tiles = (g.Nout + tile_features - 1) / tile_features;
  ta.tiles = g.grid_blocks * ta.m_tiles;
  const int64_t rows_total = g.act_by_slot ? g.grid_blocks * g.bm : (g.act_per_pair ? g.P : g.P / g.k);
  // token rows of Kin f16 in 128-byte swizzle: 128 slot rows per box when the rows are in
  // slot order, else gathered one row at a time; weight rows of Kin / 2 bytes of E2M1 codes
  // (boxes of four stages' 128 bytes x 128 rows, 128-byte swizzle)
  CUtensorMap mx, mw;
  if (!tma::encode_2d_u8(&mx, g.act, (uint64_t)g.Kin * 2, (uint64_t)rows_total, (uint64_t)g.Kin * 2, 128,
                         g.act_by_slot ? kTN : 1, true))
    return cudaErrorInvalidValue;
  if (!tma::encode_2d_u8(&mw, g.w, (uint64_t)g.Kin / 2, (uint64_t)g.E * g.Nw, (uint64_t)g.Kin / 2, 128, kTM,
                         true))
    return cudaErrorInvalidValue;
  // SwiGLU or relu^2 output in slot order: h rows of Nout f16, stored 128 slots x 128
  // features per box
  CUtensorMap mh = mx;
  if ((g.epi == EPI_SWIGLU || g.epi == EPI_RELU2) && g.out_by_slot &&
      !tma::encode_2d_u8(&mh, g.out, (uint64_t)g.Nout * 2, (uint64_t)(g.grid_blocks * g.bm), (uint64_t)g.Nout * 2,
                         kTM * 2, kTN, false))
    return cudaErrorInvalidValue;
  if (g.epi == EPI_SWIGLU) return launch_ts<EPI_SWIGLU>(ta, mx, mw, mh, stream);
  if (g.epi == EPI_RELU2) return launch_ts<EPI_RELU2>(ta, mx, mw, mh, stream);
  if (g.epi == EPI_WEIGHTED_F32) return launch_ts<EPI_WEIGHTED_F32>(ta, mx, mw, mh, stream);
  return launch_ts<EPI_PLAIN_BF16>(ta, mx, mw, mh, stream);
}

}  // namespace moe_launch
