// MXFP4 expert layer of up to 256 rows (the decode regime) on the block-scaled tensor-core
// MMA for 4-bit operands, tcgen05.mma.kind::mxf4.
//
// The layer is bound by reading the weights once from HBM ("tune the Nemotron MTP decode
// row on S5000 with a checked-in recipe", torchada PR 115: the small-M bucket dominates the
// step), so nothing may cost instructions per weight byte.  Here the E2M1 weight codes are
// the MMA's A operand exactly as stored, two codes a byte: TMA boxes of 128 bytes x 64 rows
// land in the 128-byte-swizzled K-major tile the MMA reads, and the weights' E8M0 block
// scales go to tensor memory as the MMA's A scale factors ("Add MoE GEMM variants and
// weight-gradient kernel", aiter PR 5310: MXFP4 weights with one E8M0 scale per 32
// elements, decoded as 2^(e-127) in its second review).  No weight is ever decoded in
// registers, and one thread moves every byte a CTA reads.
//
// The other operand must then be E2M1 too, so the activations enter as E2M1 digit planes:
// the 32 elements of a scale block are written as integers X below 2^16 in units of
// u = 2^(emax-15) (emax = floor(log2) of the block's largest magnitude), and plane p holds
// the base-4 digit (X >> (14 - 2p)) & 3 of every element, with its sign, as the E2M1 value
// digit / 2 under the scale 2^(emax - 2p).  The eight planes sum to X u: exactly the value
// for every bf16 element no more than 2^8 below its block's largest and every f16 element
// no more than 2^5 below it (their ulps are multiples of u); a smaller element is rounded to
// a multiple of u, an error below 2^-16 of the largest.  Digit plane j of token t is B row
// 8 t + j of a unit's token tile (4 or 8 slots), so one MMA of N = 32 or 64 columns gives
// every plane's partial sum, and the epilogue adds the planes in a fixed order.
//
// One launch covers every expert (the aiter page, Summary: all expert GEMMs in one launch).
// A unit is (alignment block, token tile, 128 weight rows); only tiles that hold a
// pair become units (a block past num_tokens_post_padded or with the -1 expert sentinel is
// never read: the page's second review, sentinel handling), and each CTA takes a contiguous
// range of units.  Roles: one thread issues the TMA boxes of stages of two 256-K sub-tiles
// into a ring, one thread issues the MMAs into one of two accumulators, and four epilogue
// warps drain the other and write the scale factors of the unit two ahead into tensor
// memory.  Every wait is bounded; a wait that runs out sets MOE_ERR_TIMEOUT and the block
// leaves cleanly, after the boxes it has asked for have landed.
#include "moe_common.cuh"
#include "tma.cuh"
#include "moe_launch.h"

namespace {

using namespace moe_launch;

constexpr int kThreads = 192;           // warps 0-3 epilogue, 4 TMA producer, 5 MMA
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kSub = 2;                 // 256-K sub-tiles per stage (one handshake each)
constexpr int kPlanes = 8;              // E2M1 digit planes per activation row
constexpr int kRowsA = 128;             // weight rows per unit (MMA M)
constexpr int kBoxRowsA = 64;           // weight rows per TMA box
constexpr int kAStage = kRowsA * 128;   // 256 K of 128 rows: two codes a byte
constexpr int kMaxWords = 24;           // 128-K scale words per unit: Kin <= 3072
constexpr int kMaxStages = 6;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kScaleCol0 = 128;    // accumulators at columns 0 and 64
constexpr uint32_t kScaleBufCols = 8 * kMaxWords;  // per buffer: 4 A + 4 B columns a scale word
constexpr unsigned kFull = 0xffffffffu;

// A unit's token tile: TOK slots (4 or 8), whose digit-plane rows are the MMA's N = 8 TOK
// B rows, 128 bytes each per sub-tile.
template <int TOK>
struct TokTile {
  static constexpr int kTok = TOK;
  static constexpr int kTilesPerBallot = 32 / TOK;
  static constexpr int kBRows = TOK * kPlanes;
  static constexpr int kBStage = kBRows * 128;
  static_assert(kBRows == 32 || kBRows == 64, "one or two 32-column TMEM loads; MMA N of M = 128 a multiple of 16");
  static_assert((kAStage + kBStage) % 1024 == 0, "MMA slots must keep the 1024-byte swizzle atoms aligned");
};
static_assert(kScaleCol0 + 2 * kScaleBufCols <= kTmemCols, "tensor memory columns");

// Splits this lane's value v, one of the 32 elements of a scale block held by the warp (one
// per lane), into its eight E2M1 digit codes (plane p in bits 4p..4p+3) and the block's
// E8M0 scale byte for plane 0, emax + 127 (plane p's is 2p less): v = sum over p of
// code_p x 2^(sb - 2p - 127), up to the rounding of elements far below the block's largest.
// emax is floored at -113, so that every plane's scale is a valid E8M0 byte (a block whose
// largest magnitude is below 2^-113 loses what lies below 2^-128).  A block holding an
// infinity or a NaN gets the NaN scale 0xFF (every product with it is NaN).
MOE_DEV uint32_t split_digits(float v, uint32_t& sb) {
  const uint32_t bits = __float_as_uint(v), mag = bits & 0x7fffffffu;
  const uint32_t mx = __reduce_max_sync(kFull, mag);
  if (mx >= 0x7f800000u) {
    sb = 0xffu;
    return 0u;
  }
  int emax = (int)(mx >> 23) - 127;
  emax = emax < -113 ? -113 : emax;
  sb = (uint32_t)(emax + 127);
  // |v| / u = |v| x 2^(15 - emax): a power-of-two product (2^-112 .. 2^128 is split in two
  // factors to stay in range), then rounded to the nearest integer, ties to even
  const int sh = 15 - emax;
  const int s1 = sh > 64 ? 64 : sh, s2 = sh - s1;
  const float y = __uint_as_float(mag) * __uint_as_float((uint32_t)(127 + s1) << 23) *
                  __uint_as_float((uint32_t)(127 + s2) << 23);
  const uint32_t X = __float2uint_rn(y);
  const uint32_t sgn = (bits >> 31) << 3;
  uint32_t w = 0;
#pragma unroll
  for (int p = 0; p < kPlanes; ++p) {
    const uint32_t dg = (X >> (14 - 2 * p)) & 3u;
    w |= (dg ? (dg | sgn) : 0u) << (4 * p);
  }
  return w;
}

// Writes the eight digit planes of a warp's 32 elements (lane = element) as packed bytes:
// element 2i in the low nibble of byte i of the 16-byte run at dst + plane x pitch.
MOE_DEV void store_planes(uint32_t w, int lane, uint8_t* dst, int64_t pitch) {
  const uint32_t wn = __shfl_down_sync(kFull, w, 1);
  if ((lane & 1) == 0) {
    uint8_t* d = dst + (lane >> 1);
#pragma unroll
    for (int p = 0; p < kPlanes; ++p) d[p * pitch] = (uint8_t)(((w >> (4 * p)) & 15u) | (((wn >> (4 * p)) & 15u) << 4));
  }
}

// ---------------------------------------------------------------- prep: items and x planes

struct PrepArgs {
  // activation rows -> planes
  const uint16_t* x;      // [rows, K] bf16
  int64_t rows;
  int K;
  uint8_t* q;             // [rows, 8, kq] packed E2M1 digits
  int kq;
  uint8_t* sc;            // [rows, sstride] E8M0 of plane 0 (byte K/32 - 1 is the last one written)
  int sstride;
  // units
  const int32_t* sorted;
  const int32_t* expert_ids;
  const int32_t* ntpp;
  int64_t P;
  int E, bm;
  int64_t blocks;         // alignment blocks the launch may visit
  int4* items;            // (alignment block, token tile, slots to the last pair + 1, expert)
  int32_t* n_items;
};

constexpr int kPrepThreads = 1024;

// Block 0 lists the units' (alignment block, TOK-slot token tile) items; the other blocks
// split the rows of x into eight digit planes.
template <int TOK>
__global__ void __launch_bounds__(kPrepThreads) dt_prep_kernel(PrepArgs pa) {
  constexpr int kTok = TokTile<TOK>::kTok, kTilesPerBallot = TokTile<TOK>::kTilesPerBallot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (blockIdx.x == 0) {
    // rounds of 128 alignment blocks, four per warp, every slot load of a round in flight at
    // once; a block of at most 128 slots is read by one ballot per 32 slots (32 / TOK tiles each)
    __shared__ int wcount[32];
    __shared__ int base_s;
    if (tid == 0) base_s = 0;
    __syncthreads();
    const int ntpp = *pa.ntpp;
    int64_t used = ((int64_t)ntpp + pa.bm - 1) / pa.bm;
    if (used > pa.blocks) used = pa.blocks;
    if (used < 0) used = 0;
    for (int64_t b0 = 0; b0 < used; b0 += 128) {
      int ex[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t b = b0 + warp + 32 * j;
        ex[j] = -1;
        if (b < used) {
          const int e = pa.expert_ids[b];
          if (e >= 0 && e < pa.E) ex[j] = e;
        }
      }
      bool v[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int s = lane + 32 * i;
          v[j][i] = ex[j] >= 0 && s < pa.bm && pa.sorted[(b0 + warp + 32 * j) * pa.bm + s] < pa.P;
        }
      uint32_t mk[4][4];
      int count = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          mk[j][i] = __ballot_sync(kFull, v[j][i]);
#pragma unroll
          for (int t = 0; t < kTilesPerBallot; ++t) count += ((mk[j][i] >> (kTok * t)) & ((1u << kTok) - 1)) != 0;
        }
      if (lane == 0) wcount[warp] = count;
      __syncthreads();
      int before = 0, total = 0;
      for (int w = 0; w < 32; ++w) {
        const int c = wcount[w];
        if (w < warp) before += c;
        total += c;
      }
      int idx = base_s + before;
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int t = 0; t < kTilesPerBallot; ++t) {
            const uint32_t mm = (mk[j][i] >> (kTok * t)) & ((1u << kTok) - 1);
            if (mm) {
              if (lane == 0 && idx < pa.P)  // a valid alignment has at most P such tiles
                pa.items[idx] = make_int4((int)(b0 + warp + 32 * j), kTilesPerBallot * i + t, 32 - __clz((int)mm), ex[j]);
              ++idx;
            }
          }
      __syncthreads();
      if (tid == 0) base_s += total;
      __syncthreads();
    }
    if (tid == 0) *pa.n_items = base_s < pa.P ? base_s : (int32_t)pa.P;
    return;
  }
  // x rows: one warp per (row, 32-element block), one element per lane
  const int nb = pa.K / 32;
  const int64_t tasks = pa.rows * nb;
  const int64_t nw = (int64_t)(gridDim.x - 1) * (kPrepThreads / 32);
  for (int64_t t = (int64_t)(blockIdx.x - 1) * (kPrepThreads / 32) + warp; t < tasks; t += nw) {
    const int64_t row = t / nb;
    const int blk = (int)(t - row * nb);
    const float v = moe::bf16_bits_to_f32(pa.x[row * pa.K + blk * 32 + lane]);
    uint32_t sb;
    const uint32_t w = split_digits(v, sb);
    store_planes(w, lane, pa.q + row * kPlanes * (int64_t)pa.kq + blk * 16, pa.kq);
    if (lane == 0) pa.sc[row * pa.sstride + blk] = (uint8_t)sb;
  }
}

// ---------------------------------------------------------------- the GEMM

struct DtArgs {
  GroupedGemm g;          // MXFP4 weights; EPI_SWIGLU (GEMM1) or EPI_WEIGHTED_F32 (GEMM2)
  const uint8_t* bsc;     // activation scales (plane 0): row r at bsc + r * sb_tok, a byte per 32 K
  int sb_tok;
  uint8_t* hq;            // GEMM1 output: h digit planes [P, 8, hkq]
  uint8_t* hsc;           // GEMM1 output: h scales [P, hsb]
  int hkq, hsb;
  const int4* items;
  const int32_t* n_items;
  int n_rt;               // weight-row tiles of 128 rows per item
  int nsub;               // 256-K sub-tiles per unit: ceil(Kin / 256)
  int nwords;             // 128-K scale words per unit: ceil(Kin / 128)
  int stages;             // ring slots (each kSub sub-tiles)
};

struct DtLayout {
  int mring, sub, slot, stg, ex, bars, total;
};
// `stages` ring slots of kSub sub-tiles (each an A tile of 128 weight rows and the B tile of
// tok tokens x 8 planes, 128 bytes a row), per epilogue warp a staging area for a unit's
// scales (its 32 weight rows' scale bytes, then tok token scale rows), the SwiGLU exchange
// of up values, barriers.
__host__ __device__ inline DtLayout dt_layout(int stages, int Kin, int sb_tok, int tok) {
  DtLayout L;
  L.mring = 0;
  L.sub = kAStage + tok * kPlanes * 128;
  L.slot = kSub * L.sub;
  L.stg = L.mring + stages * L.slot;
  L.ex = L.stg + 4 * (Kin + tok * sb_tok);
  L.bars = L.ex + 2 * 2 * tok * 32 * 4;
  L.total = L.bars + 8 * (2 * stages + 11) + 8;  // barriers, TMEM address, abort flag
  return L;
}

// Weight row (within the expert) of A row m of row tile rt; -1 past the matrix.  SwiGLU
// tiles hold 64 features: rows 0-63 their gate rows, rows 64-127 their up rows.
template <int EPI>
MOE_DEV int64_t a_row(const GroupedGemm& a, int rt, int m) {
  if (EPI == EPI_SWIGLU) {
    const int f = rt * 64 + (m & 63);
    return f < a.Nout ? (m < 64 ? (int64_t)f : (int64_t)a.Nout + f) : -1;
  }
  const int r = rt * 128 + m;
  return r < a.Nout ? (int64_t)r : -1;
}

MOE_DEV int64_t b_row(const GroupedGemm& a, int p) { return a.act_per_pair ? (int64_t)p : (int64_t)(p / a.k); }

// TMEM columns of unit buffer `buf`: the A scale words of 128-K word w at colA + 4 w (one
// word per lane, the same in the four columns: row m is read at lane m, column m / 32), the
// B ones at colB + 4 w (B row n at lane n % 32, column n / 32, in every lane quarter: the
// rows of quarter q read the copy in quarter q).
MOE_DEV uint32_t scale_col_a(uint32_t buf) { return kScaleCol0 + buf * kScaleBufCols; }
MOE_DEV uint32_t scale_col_b(uint32_t buf) { return kScaleCol0 + buf * kScaleBufCols + 4 * kMaxWords; }

// The four plane-0 scale bytes in v turned into plane p's: 2p less, the NaN scale kept.
MOE_DEV uint32_t plane_scales(uint32_t v, int p) {
  const uint32_t nan = __vcmpeq4(v, 0xffffffffu);
  return (__vsub4(v, 0x02020202u * (uint32_t)p) & ~nan) | (v & nan);
}

// Epilogue warp q writes the scale factors of one unit into TMEM buffer buf: the scale bytes
// of its 32 weight rows (a contiguous run of Kin bytes) and the tokens' scale rows are staged
// in its own shared area with 16-byte loads, then every lane writes its row's A words and
// the B words of B rows lane and 32 + lane (B row 8 t + j: token t, digit plane j) into the
// warp's lane quarter.
template <int EPI, int TOK>
MOE_DEV void write_scales(const DtArgs& d, uint8_t* stg, uint32_t taddr, int q, int lane, int64_t u, uint32_t buf) {
  constexpr int kTok = TokTile<TOK>::kTok, kBRows = TokTile<TOK>::kBRows;
  const GroupedGemm& a = d.g;
  const int64_t ii = u / d.n_rt;
  const int rt = (int)(u - ii * d.n_rt);
  const int4 item = d.items[ii];
  const int kb = a.Kin / 32;
  const int64_t r0 = a_row<EPI>(a, rt, q * 32);
  if (r0 >= 0) {
    const uint4* src = reinterpret_cast<const uint4*>(a.w_scale + ((int64_t)item.w * a.Nw + r0) * kb);
    for (int c = lane; c < a.Kin / 16; c += 32) reinterpret_cast<uint4*>(stg)[c] = __ldg(src + c);
  }
  uint8_t* stb = stg + a.Kin;
  const int64_t slot0 = (int64_t)item.x * a.bm + item.y * kTok;
  const int sbw = d.sb_tok / 16;
  for (int c = lane; c < item.z * sbw; c += 32) {
    const int j = c / sbw, cc = c - j * sbw;
    const int p = a.sorted[slot0 + j];
    if (p < a.P)
      reinterpret_cast<uint4*>(stb + j * d.sb_tok)[cc] =
          __ldg(reinterpret_cast<const uint4*>(d.bsc + b_row(a, p) * d.sb_tok) + cc);
  }
  __syncwarp();
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;
  const uint8_t* ra = stg + lane * kb;
  const uint32_t ca = taddr + lane_base + scale_col_a(buf), cb = taddr + lane_base + scale_col_b(buf);
  const uint8_t* rb0 = stb + (lane >> 3) * d.sb_tok;
  const uint8_t* rb1 = stb + (kBRows > 32 ? 4 + (lane >> 3) : 0) * d.sb_tok;
  const int pl = lane & 7;
  for (int w = 0; w < d.nwords; ++w) {
    const int o = 4 * w;
    uint32_t wa = 0;
    if (o + 2 <= kb) wa = *reinterpret_cast<const uint16_t*>(ra + o);
    if (o + 4 <= kb) wa |= (uint32_t)*reinterpret_cast<const uint16_t*>(ra + o + 2) << 16;
    tc::tmem_st4(ca + 4 * w, wa, wa, wa, wa);
    const uint32_t v0 = plane_scales(*reinterpret_cast<const uint32_t*>(rb0 + o), pl);
    const uint32_t v1 = kBRows > 32 ? plane_scales(*reinterpret_cast<const uint32_t*>(rb1 + o), pl) : 0u;
    tc::tmem_st4(cb + 4 * w, v0, v1, 0u, 0u);
  }
  tc::tmem_st_wait();
  tc::tc_fence_before();
  __syncwarp();  // the staging area is read before the next unit's loads refill it
}

template <int EPI, int TOK>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b, DtArgs d) {
  constexpr int kTok = TokTile<TOK>::kTok, kBRows = TokTile<TOK>::kBRows;
  const GroupedGemm& a = d.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const DtLayout L = dt_layout(d.stages, a.Kin, d.sb_tok, TOK);
  const int S = d.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);  // [S] MMA slot filled
  uint64_t* empty = full + S;                                   // [S] MMA slot read
  uint64_t* tfull = empty + S;   // [2] accumulator done (and the unit's scale columns free)
  uint64_t* tempty = tfull + 2;  // [2] accumulator drained
  uint64_t* sready = tempty + 2; // [2] the unit's scale factors written
  uint64_t* xfull = sready + 2;  // [2] up values staged (SwiGLU)
  uint64_t* xempty = xfull + 2;  // [2] up values read
  uint64_t* drain = xempty + 2;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_s + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], 4);
      tc::mbar_init(&sready[i], 4);
      tc::mbar_init(&xfull[i], 2);
      tc::mbar_init(&xempty[i], 2);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(taddr_s, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t taddr = *taddr_s;
  const int64_t n_units = (int64_t)(*d.n_items) * d.n_rt;
  const int64_t u0 = n_units * blockIdx.x / gridDim.x, u1 = n_units * (blockIdx.x + 1) / gridDim.x;
  const uint32_t smem_s = tc::smem_addr(smem);
  const int nsub = d.nsub, nst2 = (d.nsub + kSub - 1) / kSub;
  const uint64_t wb = a.wait_ns > 0 ? (uint64_t)a.wait_ns : tc::kWaitNs;
  bool bad = false;

  if (warp == kProdWarp && !a.stall) {
    // ------------------------------------------------------------------ TMA producer
    // Per stage and sub-tile: the unit's 128 weight rows as two boxes of 64 rows x 128 bytes
    // (256 K; a box wholly past the matrix is skipped, bytes past a row's end read as zero)
    // and, per token of the tile, its eight digit-plane rows as one box of 8 x 128 bytes.
    // Lanes 0-7 look up the tile's tokens; lane 0 issues every box.
    if (lane == 0) {
      tma::prefetch_map(&tmap_a);
      tma::prefetch_map(&tmap_b);
    }
    uint32_t ws = 0, wph = 0;  // slot (and its phase) of the next stage issued
    int64_t issued = 0;
    int64_t cur_ii = -1;
    int32_t brow = -1;         // lane j < 8: the first digit-plane row of token j, or -1
    int64_t arow0 = 0, arow1 = 0;
    bool box1 = true;
    for (int64_t u = u0; u < u1; ++u) {
      if (__any_sync(kFull, *abort_flag != 0)) break;  // the same decision in every lane
      const int64_t ii = u / d.n_rt;
      const int rt = (int)(u - ii * d.n_rt);
      const int4 item = d.items[ii];
      if (ii != cur_ii) {  // a new (alignment block, token tile): its tokens' plane rows
        cur_ii = ii;
        brow = -1;
        if (lane < kTok && lane < item.z) {
          const int p = a.sorted[(int64_t)item.x * a.bm + item.y * kTok + lane];
          if (p < a.P) brow = (int32_t)(b_row(a, p) * kPlanes);
        }
      }
      int32_t rows_b[kTok];
#pragma unroll
      for (int j = 0; j < kTok; ++j) rows_b[j] = __shfl_sync(kFull, brow, j);
      const int64_t ebase = (int64_t)item.w * a.Nw;
      if (EPI == EPI_SWIGLU) {
        arow0 = ebase + (int64_t)rt * 64;
        arow1 = ebase + a.Nout + (int64_t)rt * 64;
        box1 = true;
      } else {
        arow0 = ebase + (int64_t)rt * 128;
        arow1 = arow0 + kBoxRowsA;
        box1 = rt * 128 + kBoxRowsA < a.Nout;
      }
      int nb = 0;
#pragma unroll
      for (int j = 0; j < kTok; ++j) nb += rows_b[j] >= 0;
      for (int st = 0; st < nst2; ++st) {
        bool ok = true;
        if (lane == 0) {
          ok = tc::mbar_wait(&empty[ws], wph ^ 1, wb);
          if (ok) {
            const int nh = nsub - st * kSub < kSub ? nsub - st * kSub : kSub;
            const uint32_t bytes = (uint32_t)nh * (uint32_t)((box1 ? 2 : 1) * kBoxRowsA * 128 + nb * kPlanes * 128);
            tma::mbar_arrive_expect_tx(&full[ws], bytes);
            for (int h = 0; h < nh; ++h) {
              const int ss = st * kSub + h;
              const uint32_t sl = smem_s + L.mring + ws * L.slot + h * L.sub;
              tma::load_2d(sl, &tmap_a, ss * 128, (int32_t)arow0, &full[ws]);
              if (box1) tma::load_2d(sl + kBoxRowsA * 128, &tmap_a, ss * 128, (int32_t)arow1, &full[ws]);
#pragma unroll
              for (int j = 0; j < kTok; ++j)
                if (rows_b[j] >= 0) tma::load_2d(sl + kAStage + j * kPlanes * 128, &tmap_b, ss * 128, rows_b[j], &full[ws]);
            }
            ++issued;
          }
        }
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        if (!ok) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        if (++ws == (uint32_t)S) {
          ws = 0;
          wph ^= 1;
        }
      }
    }
    // no box may land after the block has left: wait for the last S stages asked for
    // (already complete unless the MMA side gave up)
    if (lane == 0) {
      const int64_t n = issued < S ? issued : S;
      for (int64_t i = 1; i <= n; ++i) {
        const int64_t k = issued - i;  // stage number; slot k % S, phase parity (k / S) & 1
        if (!tc::mbar_wait(&full[k % S], (uint32_t)((k / S) & 1), wb)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp && !a.stall) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc0 = tc::idesc_mxf4(kRowsA, kBRows, 0, 0), idesc1 = tc::idesc_mxf4(kRowsA, kBRows, 2, 2);
      const uint64_t adesc0 = tc::sdesc_sw128(smem_s), bdesc0 = tc::sdesc_sw128(smem_s + kAStage);
      uint32_t ms = 0, mph = 0;  // MMA slot and its phase
      for (int64_t u = u0; u < u1 && !*abort_flag; ++u) {
        const uint32_t li = (uint32_t)(u - u0), buf = li & 1, use = li >> 1;
        if (!tc::mbar_wait(&tempty[buf], (use & 1) ^ 1, wb) || !tc::mbar_wait(&sready[buf], use & 1, wb)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d_tmem = taddr + buf * 64;
        const uint32_t ca = taddr + scale_col_a(buf), cb = taddr + scale_col_b(buf);
        bool ok = true;
        for (int st = 0; st < nst2; ++st) {
          const int s = (int)ms;
          if (!tc::mbar_wait(&full[s], mph, wb)) {
            moe::set_status(a.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int h = 0; h < kSub; ++h) {
            const int ss = st * kSub + h;
            // descriptors advance by address >> 4: 32 bytes (64 K) per MMA
            const uint64_t so = (uint64_t)((L.mring + s * L.slot + h * L.sub) >> 4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int kk = ss * 4 + j;  // 64-K step of the unit
              if (kk * 64 < a.Kin)
                tc::mma_mxf4_ss(d_tmem, adesc0 + so + 2 * j, bdesc0 + so + 2 * j, (j & 1) ? idesc1 : idesc0,
                                ca + 4 * (kk >> 1), cb + 4 * (kk >> 1), kk != 0);
            }
          }
          tc::mma_commit(&empty[s]);
          if (++ms == (uint32_t)S) {
            ms = 0;
            mph ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(&tfull[buf]);
      }
      tc::mma_commit(drain);
      if (!tc::mbar_wait(drain, 0, wb)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp, m = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint16_t* bias = static_cast<const uint16_t*>(a.bias);
    float* ex = reinterpret_cast<float*>(smem + L.ex);
    uint8_t* stg = smem + L.stg + q * (a.Kin + kTok * d.sb_tok);
    // the scale factors of the first two units; each later unit's once the unit two before
    // it (same buffer) has been drained
    for (int64_t u = u0; u < u0 + 2 && u < u1; ++u) write_scales<EPI, TOK>(d, stg, taddr, q, lane, u, (uint32_t)(u - u0) & 1);
    if (lane == 0)
      for (int64_t u = u0; u < u0 + 2 && u < u1; ++u) tc::mbar_arrive(&sready[(u - u0) & 1]);
    for (int64_t u = u0; u < u1; ++u) {
      if (__any_sync(kFull, *abort_flag != 0)) break;  // the same decision in every lane
      const uint32_t li = (uint32_t)(u - u0), buf = li & 1, use = li >> 1;
      const int64_t ii = u / d.n_rt;
      const int rt = (int)(u - ii * d.n_rt);
      const int4 item = d.items[ii];
      const int64_t slot0 = (int64_t)item.x * a.bm + item.y * kTok;
      const int nreal = item.z;
      const int64_t e = item.w;
      if (!__all_sync(kFull, tc::mbar_wait(&tfull[buf], use & 1, wb))) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      // columns 8 t + j: token t's digit plane j
      uint32_t r[kBRows / 32][32];
      tc::tmem_ld32(taddr + lane_base + buf * 64, r[0]);
      if (kBRows > 32) tc::tmem_ld32(taddr + lane_base + buf * 64 + 32, r[kBRows / 32 - 1]);
      tc::tmem_ld_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[buf]);
      if (u + 2 < u1) {
        write_scales<EPI, TOK>(d, stg, taddr, q, lane, u + 2, buf);
        if (lane == 0) tc::mbar_arrive(&sready[buf]);
      }
      // the planes' partial sums, least significant first
      float acc[kTok];
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        float s = __uint_as_float(r[t >> 2][(t & 3) * kPlanes + kPlanes - 1]);
#pragma unroll
        for (int j = kPlanes - 2; j >= 0; --j) s += __uint_as_float(r[t >> 2][(t & 3) * kPlanes + j]);
        acc[t] = s;
      }
      if (EPI == EPI_SWIGLU) {
        float* xs = ex + (buf * 2 + (q & 1)) * kTok * 32;
        if (q >= 2) {  // up rows: hand the values to the warp holding the same features' gate rows
          if (!__all_sync(kFull, tc::mbar_wait(&xempty[buf], (use & 1) ^ 1, wb))) {
            moe::set_status(a.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
#pragma unroll
          for (int j = 0; j < kTok; ++j) xs[j * 32 + lane] = acc[j];
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&xfull[buf]);
          continue;
        }
        if (!__all_sync(kFull, tc::mbar_wait(&xfull[buf], use & 1, wb))) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        float up[kTok];
#pragma unroll
        for (int j = 0; j < kTok; ++j) up[j] = xs[j * 32 + lane];
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&xempty[buf]);
        const int f = rt * 64 + m;  // this lane's feature (q < 2)
        const float bg = bias ? moe::bf16_bits_to_f32(bias[e * a.Nw + f]) : 0.f;
        const float bu = bias ? moe::bf16_bits_to_f32(bias[e * a.Nw + a.Nout + f]) : 0.f;
#pragma unroll
        for (int j = 0; j < kTok; ++j) {
          if (j >= nreal) break;
          const int p = a.sorted[slot0 + j];
          if (p >= a.P) continue;
          const float hval = moe::silu(acc[j] + bg) * (up[j] + bu);
          const __half hv = __float2half_rn(hval);
          if (__hisinf(hv)) bad = true;  // an overflow of f16 h (NaN only comes from NaN inputs)
          uint32_t sb;
          const uint32_t w = split_digits(__half2float(hv), sb);
          store_planes(w, lane, d.hq + (int64_t)p * kPlanes * d.hkq + (rt * 64 + q * 32) / 2, d.hkq);
          if (lane == 0) d.hsc[(int64_t)p * d.hsb + f / 32] = (uint8_t)sb;
        }
      } else {
        const int n = rt * 128 + m;
        if (n < a.Nout) {
          const float b = bias ? moe::bf16_bits_to_f32(bias[e * a.Nw + n]) : 0.f;
          float* out = static_cast<float*>(a.out);
#pragma unroll
          for (int j = 0; j < kTok; ++j) {
            if (j >= nreal) break;
            const int p = a.sorted[slot0 + j];
            if (p < a.P) out[(int64_t)p * a.Nout + n] = (acc[j] + b) * a.topk_w[p];
          }
        }
      }
    }
  }
  if (bad) moe::set_status(a.status, MOE_ERR_RANGE);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kMmaWarp) tc::tmem_dealloc(taddr, kTmemCols);
}

}  // namespace

namespace {

int dt_nwords(int Kin) { return (Kin + 127) / 128; }
int dt_kq(int Kin) { return dt_nwords(Kin) * 64; }  // bytes of a digit-plane row
int dt_sb(int Kin) { return (dt_nwords(Kin) * 4 + 15) / 16 * 16; }
size_t r256(size_t v) { return (v + 255) / 256 * 256; }

constexpr int kSmemMax = 227 * 1024;

// Ring slots: as many as fit, up to kMaxStages.
int dt_stages(int Kin, int tok) {
  const DtLayout L0 = dt_layout(0, Kin, dt_sb(Kin), tok);
  const int s = (kSmemMax - 1024 - L0.total) / (L0.slot + 16);
  return s < kMaxStages ? s : kMaxStages;
}

// Slots per token tile.  A tile of 4 slots halves the B rows of a stage, which lets a fifth
// ring slot (of 40 KB) fit beside the others; but an expert with more than 4 pairs in an
// alignment block then streams its weights once per tile.  With at most 3 pairs per expert
// on average (the decode regime) the deeper ring wins (GEMM1 of the 64-token decode layer:
// 0.205 -> 0.190 ms); denser batches keep 8-slot tiles.
int dt_tok(const GroupedGemm& g) { return g.P <= 3 * (int64_t)g.E ? 4 : 8; }

template <int EPI, int TOK>
cudaError_t launch_dt(const CUtensorMap& ma, const CUtensorMap& mb, const DtArgs& d, cudaStream_t stream) {
  const int smem = dt_layout(d.stages, d.g.Kin, d.sb_tok, TOK).total + 1024;
  cudaError_t err =
      cudaFuncSetAttribute(decode_tc_kernel<EPI, TOK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  decode_tc_kernel<EPI, TOK><<<(unsigned)moe_launch::sm_count_current(), kThreads, smem, stream>>>(ma, mb, d);
  return cudaGetLastError();
}

}  // namespace

namespace moe_launch {

bool decode_tc_supported(const GroupedGemm& g1, const GroupedGemm& g2) {
  auto ok = [](const GroupedGemm& g, int epi) {
    if (g.wfmt != WF_MXFP4 || g.epi != epi || g.act_by_slot || g.out_by_slot) return false;
    // scale rows of an even number of bytes, tensor memory for every scale word
    if (g.Kin % 64 != 0 || g.Kin > 128 * kMaxWords) return false;
    if (epi == EPI_SWIGLU ? (g.Nout % 64 != 0 || g.Nw != 2 * (int64_t)g.Nout)
                          : (g.Nout % 32 != 0 || g.Nw != (int64_t)g.Nout))
      return false;
    if (g.bm % 8 != 0 || g.bm > 128) return false;
    // TMA boxes of the weight rows: a 16-byte aligned base, rows of at least one box (128
    // bytes) and at least two boxes of rows, row coordinates below 2^31
    if (reinterpret_cast<uintptr_t>(g.w) % 16 != 0 || g.Kin < 256 || (int64_t)g.E * g.Nw < 2 * kBoxRowsA ||
        (int64_t)g.E * g.Nw >= (int64_t)1 << 31)
      return false;
    return dt_stages(g.Kin, 8) >= 2;
  };
  // both GEMMs read the one unit list: the same token tiles
  return ok(g1, EPI_SWIGLU) && ok(g2, EPI_WEIGHTED_F32) && g2.Kin == g1.Nout && g1.P == g2.P &&
         dt_tok(g1) == dt_tok(g2);
}

size_t decode_tc_workspace_bytes(int64_t T_rows, int k, int K, int I) {
  if (T_rows <= 0 || k < 1 || K < 1 || I < 1) return 0;
  const int64_t P = T_rows * k;
  return r256((size_t)T_rows * kPlanes * dt_kq(K)) + r256((size_t)T_rows * dt_sb(K)) +
         r256((size_t)P * kPlanes * dt_kq(I)) + r256((size_t)P * dt_sb(I)) + r256((size_t)(P + 1) * 16);
}

DecodeTcBufs decode_tc_carve(void* ws, int64_t T_rows, int k, int K, int I) {
  const int64_t P = T_rows * k;
  uint8_t* p = static_cast<uint8_t*>(ws);
  DecodeTcBufs b;
  b.xq = p;
  p += r256((size_t)T_rows * kPlanes * dt_kq(K));
  b.xs = p;
  p += r256((size_t)T_rows * dt_sb(K));
  b.hq = p;
  p += r256((size_t)P * kPlanes * dt_kq(I));
  b.hs = p;
  p += r256((size_t)P * dt_sb(I));
  b.items = reinterpret_cast<int4*>(p);
  b.n_items = reinterpret_cast<int32_t*>(p + (size_t)P * 16);
  return b;
}

cudaError_t decode_tc_prep(const GroupedGemm& g1, const void* x, int64_t T_rows, const DecodeTcBufs& b,
                           cudaStream_t stream) {
  PrepArgs pa{};
  pa.x = static_cast<const uint16_t*>(x);
  pa.rows = T_rows;
  pa.K = g1.Kin;
  pa.q = b.xq;
  pa.kq = dt_kq(g1.Kin);
  pa.sc = b.xs;
  pa.sstride = dt_sb(g1.Kin);
  pa.sorted = g1.sorted;
  pa.expert_ids = g1.expert_ids;
  pa.ntpp = g1.ntpp;
  pa.P = g1.P;
  pa.E = g1.E;
  pa.bm = g1.bm;
  pa.blocks = g1.grid_blocks;
  pa.items = b.items;
  pa.n_items = b.n_items;
  const int64_t warps = T_rows * (g1.Kin / 32);
  int64_t blocks = (warps + kPrepThreads / 32 - 1) / (kPrepThreads / 32);
  const int64_t cap = 2 * (int64_t)sm_count_current();
  if (blocks > cap) blocks = cap;
  if (dt_tok(g1) == 4)
    dt_prep_kernel<4><<<(unsigned)(1 + blocks), kPrepThreads, 0, stream>>>(pa);
  else
    dt_prep_kernel<8><<<(unsigned)(1 + blocks), kPrepThreads, 0, stream>>>(pa);
  return cudaGetLastError();
}

cudaError_t decode_tc_gemm(const GroupedGemm& g, const DecodeTcBufs& b, cudaStream_t stream) {
  DtArgs d{};
  d.g = g;
  d.sb_tok = dt_sb(g.Kin);
  d.items = b.items;
  d.n_items = b.n_items;
  d.nsub = (g.Kin + 255) / 256;
  d.nwords = dt_nwords(g.Kin);
  const int tok = dt_tok(g);
  d.stages = dt_stages(g.Kin, tok);
  // weight rows of Kin / 2 bytes (boxes of 128 bytes x 64 rows) and digit-plane rows of the
  // activations, eight per token row (boxes of 128 bytes x 8 rows), both 128-byte swizzled
  const int64_t act_rows = g.act_per_pair ? g.P : g.P / g.k;
  CUtensorMap ma, mb;
  if (!tma::encode_2d_u8(&ma, g.w, (uint64_t)g.Kin / 2, (uint64_t)g.E * g.Nw, (uint64_t)g.Kin / 2, 128, kBoxRowsA,
                         true))
    return cudaErrorInvalidValue;
  const uint8_t* bq = g.epi == EPI_SWIGLU ? b.xq : b.hq;
  if (!tma::encode_2d_u8(&mb, bq, (uint64_t)g.Kin / 2, (uint64_t)act_rows * kPlanes, (uint64_t)dt_kq(g.Kin), 128,
                         kPlanes, true))
    return cudaErrorInvalidValue;
  if (g.epi == EPI_SWIGLU) {
    d.bsc = b.xs;
    d.hq = b.hq;
    d.hsc = b.hs;
    d.hkq = dt_kq(g.Nout);
    d.hsb = dt_sb(g.Nout);
    d.n_rt = g.Nout / 64;
    return tok == 4 ? launch_dt<EPI_SWIGLU, 4>(ma, mb, d, stream) : launch_dt<EPI_SWIGLU, 8>(ma, mb, d, stream);
  }
  d.bsc = b.hs;
  d.n_rt = (g.Nout + 127) / 128;
  return tok == 4 ? launch_dt<EPI_WEIGHTED_F32, 4>(ma, mb, d, stream)
                  : launch_dt<EPI_WEIGHTED_F32, 8>(ma, mb, d, stream);
}

}  // namespace moe_launch
