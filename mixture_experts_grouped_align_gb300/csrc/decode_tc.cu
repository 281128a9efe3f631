// MXFP4 expert layer of up to 256 rows (the decode regime) on the block-scaled tensor-core
// MMA, tcgen05.mma.kind::mxf8f6f4.
//
// The layer is bound by reading the weights once from HBM ("tune the Nemotron MTP decode
// row on S5000 with a checked-in recipe", torchada PR 115: the small-M bucket dominates the
// step), so nothing may cost instructions per weight byte.  Here the E2M1 weight codes are
// the MMA's A operand exactly as stored: 8-byte cp.async copies (16 codes each) land in the
// low half of each 16-byte chunk of a 128-byte-swizzled tile -- the layout in which the MMA
// reads 4-bit operands -- and the weights' E8M0 block scales go to tensor memory as the
// MMA's A scale factors ("Add MoE GEMM variants and weight-gradient kernel", aiter PR 5310:
// MXFP4 weights with one E8M0 scale per 32 elements, decoded as 2^(e-127) in its second
// review).  No weight is ever decoded in registers.
//
// The activations enter as E4M3 planes: each row of x (bf16) is written as two planes and
// each row of h (f16) as three, sharing one E8M0 scale per 32 elements, such that the planes
// sum to the value exactly -- a bf16 significand is 8 bits, an f16 one 11, an E4M3 one 4, and
// every residual is representable -- for every bf16 element no more than 2^9 below its
// block's largest and every f16 element no more than 2^6 below it; a smaller element keeps
// an error below 2^-17 of the largest.  Plane j of token t is B row 8 j + t of an 8-token
// unit, so one MMA of N = 16 (x) or 32 (h; rows 24-31 unused) columns gives every plane's
// partial sum, and the epilogue adds the planes in a fixed order.
//
// One launch covers every expert (the aiter page, Summary: all expert GEMMs in one launch).
// A unit is (alignment block, 8-slot token tile, 128 weight rows); only tiles that hold a
// pair become units (a block past num_tokens_post_padded or with the -1 expert sentinel is
// never read: the page's second review, sentinel handling), and each CTA takes a contiguous
// range of units.  Roles: eight producer warps issue the copies of stages of two 128-K
// sub-tiles (one handshake a stage: the MMA side of a handshake costs a fixed few hundred
// cycles, so the stage carries sixteen MMAs' worth of bytes), one thread issues the MMAs into
// one of two accumulators, and four epilogue warps drain the other and write the scale
// factors of the unit two ahead into tensor memory.  Every wait is bounded; a wait that runs
// out sets MOE_ERR_TIMEOUT and the block leaves cleanly.
#include <cuda_fp8.h>

#include "moe_common.cuh"
#include "cp_async.cuh"
#include "moe_launch.h"

namespace {

using namespace moe_launch;
using namespace cpa;

constexpr int kThreads = 416;           // warps 0-3 epilogue, 4-11 producers, 12 MMA
constexpr int kProdWarp0 = 4;
constexpr int kProdWarps = 8;
constexpr int kMmaWarp = 12;
constexpr int kSub = 2;                 // 128-K sub-tiles per stage (one handshake each)
constexpr int kLag = 2;                 // stages a producer thread keeps in flight
constexpr int kTok = 8;                 // token rows (slots) per unit
constexpr int kTilesPerBallot = 32 / kTok;
constexpr int kRowsA = 128;             // weight rows per unit (MMA M)
constexpr int kAStage = kRowsA * 128;   // 128 K of 128 rows: 16 codes per 16-byte chunk
constexpr int kMaxNst = 24;             // 128-K sub-tiles per unit: Kin <= 3072
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kScaleCol0 = 128;    // accumulators at columns 0 and 64
constexpr uint32_t kScaleBufCols = 8 * kMaxNst;  // per buffer: 4 A + 4 B columns a 128-K sub-tile
constexpr unsigned kFull = 0xffffffffu;

// B rows of a sub-tile: planes x kTok rounded up to the MMA's N granularity (16)
__host__ __device__ constexpr int b_rows(int planes) { return (planes * kTok + 15) / 16 * 16; }
static_assert((kAStage + b_rows(2) * 128) % 1024 == 0 && (kAStage + b_rows(3) * 128) % 1024 == 0,
              "MMA slots must keep the 1024-byte swizzle atoms aligned");
static_assert(kScaleCol0 + 2 * kScaleBufCols <= kTmemCols, "tensor memory columns");

MOE_DEV uint32_t f32_to_e4m3(float v) {
  return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}
MOE_DEV float e4m3_to_f32(uint32_t c) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

// Splits this lane's value v, one of the 32 elements of a scale block held by the warp (one
// per lane), into `planes` E4M3 codes and the block's E8M0 scale byte: v = 2^(sb-127) x (sum
// of the planes' values).  The scale puts the block's largest magnitude in [128, 256); each
// plane is the round-to-nearest-even of what the earlier planes left.  A block holding an
// infinity or a NaN gets the NaN scale 0xFF (every product with it is NaN).
MOE_DEV void split_planes(float v, int planes, uint32_t (&code)[3], uint32_t& sb) {
  const uint32_t mag = __float_as_uint(v) & 0x7fffffffu;
  const uint32_t mx = __reduce_max_sync(kFull, mag);
  code[0] = code[1] = code[2] = 0u;
  if (mx >= 0x7f800000u) {
    sb = 0xffu;
    return;
  }
  // floor(log2(max)) for a normal maximum; a zero or subnormal maximum takes the floor of
  // the scale range below
  const int emax = (int)(mx >> 23) - 127;
  int s = emax + 120;  // scale 2^(emax - 7)
  s = s < 1 ? 1 : (s > 253 ? 253 : s);
  sb = (uint32_t)s;
  float r = v * __uint_as_float((uint32_t)(254 - s) << 23);  // v / 2^(s-127): exact
#pragma unroll
  for (int p = 0; p < 3; ++p)
    if (p < planes) {
      code[p] = f32_to_e4m3(r);
      r -= e4m3_to_f32(code[p]);
    }
}

// ---------------------------------------------------------------- prep: items and x planes

struct PrepArgs {
  // activation rows -> planes
  const uint16_t* x;      // [rows, K] bf16
  int64_t rows;
  int K;
  uint8_t* q;             // [rows, 2, kp] E4M3
  int kp;
  uint8_t* sc;            // [rows, sstride] E8M0 (byte K/32 - 1 is the last one written)
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

// Block 0 lists the units' (alignment block, token tile) items; the other blocks split the
// rows of x into two planes.
__global__ void __launch_bounds__(kPrepThreads) dt_prep_kernel(PrepArgs pa) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (blockIdx.x == 0) {
    // rounds of 128 alignment blocks, four per warp, every slot load of a round in flight at
    // once; a block of at most 128 slots is read by one ballot per 32 slots (two tiles each)
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
    uint32_t code[3], sb;
    split_planes(v, 2, code, sb);
    uint8_t* dst = pa.q + row * 2 * (int64_t)pa.kp + blk * 32 + lane;
    dst[0] = (uint8_t)code[0];
    dst[pa.kp] = (uint8_t)code[1];
    if (lane == 0) pa.sc[row * pa.sstride + blk] = (uint8_t)sb;
  }
}

// ---------------------------------------------------------------- the GEMM

struct DtArgs {
  GroupedGemm g;          // MXFP4 weights; EPI_SWIGLU (GEMM1) or EPI_WEIGHTED_F32 (GEMM2)
  const uint8_t* bq;      // activation planes: row r, plane j at bq + (r * planes + j) * kp
  const uint8_t* bsc;     // activation scales: row r at bsc + r * sb_tok, one byte per 32 K
  int planes, kp, sb_tok;
  uint8_t* hq;            // GEMM1 output: h planes [P, 3, hkp]
  uint8_t* hsc;           // GEMM1 output: h scales [P, hsb]
  int hkp, hsb;
  const int4* items;
  const int32_t* n_items;
  int n_rt;               // weight-row tiles of 128 rows per item
  int nst;                // 128-K sub-tiles per unit: ceil(Kin / 128)
  int stages;             // ring slots (each kSub sub-tiles)
};

struct DtLayout {
  int mring, sub, slot, stg, ex, bars, total;
};
// `stages` ring slots of kSub sub-tiles (each an A tile in the 4-bit padded layout and the
// planes' B rows), per epilogue warp a staging area for a unit's scales (its 32 weight rows'
// scale bytes, then kTok token scale rows), the SwiGLU exchange of up values, barriers.
__host__ __device__ inline DtLayout dt_layout(int stages, int planes, int Kin, int sb_tok) {
  DtLayout L;
  L.mring = 0;
  L.sub = kAStage + b_rows(planes) * 128;
  L.slot = kSub * L.sub;
  L.stg = L.mring + stages * L.slot;
  L.ex = L.stg + 4 * (Kin + kTok * sb_tok);
  L.bars = L.ex + 2 * 2 * kTok * 32 * 4;
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

// TMEM columns of unit buffer `buf`: the A scale words of stage st at colA + 4 st (one word
// per lane, the same in the four columns: row m is read at lane m, column m / 32), the B
// ones at colB + 4 st (B row n at lane n % 32, column n / 32).
MOE_DEV uint32_t scale_col_a(uint32_t buf) { return kScaleCol0 + buf * kScaleBufCols; }
MOE_DEV uint32_t scale_col_b(uint32_t buf) { return kScaleCol0 + buf * kScaleBufCols + 4 * kMaxNst; }

// Epilogue warp q writes the scale factors of one unit into TMEM buffer buf: the scale bytes
// of its 32 weight rows (a contiguous run of Kin bytes) and the tokens' scale rows are
// staged in its own shared area with 16-byte loads, then every lane writes its row's words.
template <int EPI>
MOE_DEV void write_scales(const DtArgs& d, uint8_t* stg, uint32_t taddr, int q, int lane, int64_t u, uint32_t buf) {
  const GroupedGemm& a = d.g;
  const int64_t ii = u / d.n_rt;
  const int rt = (int)(u - ii * d.n_rt);
  const int4 item = d.items[ii];
  const int64_t slot0 = (int64_t)item.x * a.bm + item.y * kTok;
  const int kb = a.Kin / 32;
  const int64_t r0 = a_row<EPI>(a, rt, q * 32);
  if (r0 >= 0) {
    const uint4* src = reinterpret_cast<const uint4*>(a.w_scale + ((int64_t)item.w * a.Nw + r0) * kb);
    for (int c = lane; c < a.Kin / 16; c += 32) reinterpret_cast<uint4*>(stg)[c] = __ldg(src + c);
  }
  const int sbw = d.sb_tok / 16;
  uint8_t* stb = stg + a.Kin;
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
  const uint8_t* rb = stb + (lane & (kTok - 1)) * d.sb_tok;
  const uint32_t ca = taddr + lane_base + scale_col_a(buf), cb = taddr + lane_base + scale_col_b(buf);
  for (int st = 0; st < d.nst; ++st) {
    const int o = 4 * st;
    uint32_t w = 0;
    if (o + 2 <= kb) w = *reinterpret_cast<const uint16_t*>(ra + o);
    if (o + 4 <= kb) w |= (uint32_t)*reinterpret_cast<const uint16_t*>(ra + o + 2) << 16;
    tc::tmem_st4(ca + 4 * st, w, w, w, w);
    const uint32_t v = *reinterpret_cast<const uint32_t*>(rb + o);
    tc::tmem_st4(cb + 4 * st, v, v, 0u, 0u);
  }
  tc::tmem_st_wait();
  tc::tc_fence_before();
  __syncwarp();  // the staging area is read before the next unit's loads refill it
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(DtArgs d) {
  const GroupedGemm& a = d.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const DtLayout L = dt_layout(d.stages, d.planes, a.Kin, d.sb_tok);
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
      tc::mbar_init(&full[s], kProdWarps);
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
  const int nst = d.nst, nst2 = (d.nst + kSub - 1) / kSub;
  const uint64_t wb = a.wait_ns > 0 ? (uint64_t)a.wait_ns : tc::kWaitNs;
  bool bad = false;

  if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps && !a.stall) {
    // ------------------------------------------------------------------ producers
    // Per stage a thread copies 8 bytes (16 codes) of four weight rows straight into the low
    // half of 16-byte chunks of the MMA slot (rows 32 i + pt / 8, chunk pt % 8 of the
    // 128-byte-swizzled tile: the MMA's 4-bit operand layout) and at most two 16-byte chunks
    // of B rows (c = 256 i + pt: row c / 8, chunk c % 8); once its copies of a stage have
    // landed it hands the stage over.  Row pointers are set per unit.
    const int pt = tid - kProdWarp0 * 32;
    const int ar = pt >> 3, ch = pt & 7;
    const uint32_t aoff = tc::sw128_offset(ar, ch);  // + 4096 i for row 32 i + ar
    const uint8_t* wcodes = static_cast<const uint8_t*>(a.w);
    const int64_t wrow_bytes = a.Kin / 2;
    uint32_t hs = 0;  // slot of the next stage handed over
    auto hand_over = [&]() {
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&full[hs]);
      if (++hs == (uint32_t)S) hs = 0;
    };
    uint32_t ws = 0, wph = 0;  // slot (and its phase) of the next stage issued
    int npend = 0;
    int64_t cur_ii = -1;
    int4 item = make_int4(0, 0, 0, 0);
    const uint8_t* bsrc[2] = {nullptr, nullptr};
    bool ok = true;
    for (int64_t u = u0; u < u1 && ok && !*abort_flag; ++u) {
      const int64_t ii = u / d.n_rt;
      const int rt = (int)(u - ii * d.n_rt);
      if (ii != cur_ii) {  // a new (alignment block, token tile): its B rows
        cur_ii = ii;
        item = d.items[ii];
        const int64_t slot0 = (int64_t)item.x * a.bm + item.y * kTok;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int n = (i * 256 + pt) >> 3, j = n % kTok, pl = n / kTok;
          bsrc[i] = nullptr;
          if (pl < d.planes && j < item.z) {
            const int p = a.sorted[slot0 + j];
            if (p < a.P) bsrc[i] = d.bq + (b_row(a, p) * d.planes + pl) * (int64_t)d.kp + ch * 16;
          }
        }
      }
      const uint8_t* arow[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t r = a_row<EPI>(a, rt, 32 * i + ar);
        arow[i] = r >= 0 ? wcodes + ((int64_t)item.w * a.Nw + r) * wrow_bytes + ch * 8 : nullptr;
      }
      for (int st = 0; st < nst2; ++st) {
        if (npend == kLag) {
          cp_async_wait<kLag - 1>();
          hand_over();
          --npend;
        }
        if (!tc::mbar_wait(&empty[ws], wph ^ 1, wb)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
#pragma unroll
        for (int h = 0; h < kSub; ++h) {
          const int ss = st * kSub + h;  // 128-K sub-stage
          const uint32_t sl = smem_s + L.mring + ws * L.slot + h * L.sub;
          if (ss * 128 + ch * 16 + 16 <= a.Kin) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (arow[i]) cp_async8(sl + aoff + 4096 * i, arow[i] + ss * 64);
          }
          if (ss < nst) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
              if (bsrc[i]) cp_async16(sl + kAStage + tc::sw128_offset((i * 256 + pt) >> 3, ch), bsrc[i] + ss * 128);
          }
        }
        cp_async_commit();
        ++npend;
        if (++ws == (uint32_t)S) {
          ws = 0;
          wph ^= 1;
        }
      }
    }
    cp_async_wait<0>();
    while (npend > 0 && !*abort_flag) {
      hand_over();
      --npend;
    }
  } else if (warp == kMmaWarp && !a.stall) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const int N = b_rows(d.planes);
      uint32_t idesc[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) idesc[j] = tc::idesc_mx8(kRowsA, N, j, j) | (tc::kTypeE2M1 << 7);
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
            // descriptors advance by address >> 4: 32 bytes of K per MMA
            const uint64_t so = (uint64_t)((L.mring + s * L.slot + h * L.sub) >> 4);
            const int rem = (a.Kin - ss * 128) / 32, nk = rem < 4 ? rem : 4;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (j < nk)
                tc::mma_mx8_ss(d_tmem, adesc0 + so + 2 * j, bdesc0 + so + 2 * j, idesc[j], ca + 4 * ss, cb + 4 * ss,
                               (ss | j) != 0);
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
    for (int64_t u = u0; u < u0 + 2 && u < u1; ++u) write_scales<EPI>(d, stg, taddr, q, lane, u, (uint32_t)(u - u0) & 1);
    if (lane == 0)
      for (int64_t u = u0; u < u0 + 2 && u < u1; ++u) tc::mbar_arrive(&sready[(u - u0) & 1]);
    for (int64_t u = u0; u < u1 && !*abort_flag; ++u) {
      const uint32_t li = (uint32_t)(u - u0), buf = li & 1, use = li >> 1;
      const int64_t ii = u / d.n_rt;
      const int rt = (int)(u - ii * d.n_rt);
      const int4 item = d.items[ii];
      const int64_t slot0 = (int64_t)item.x * a.bm + item.y * kTok;
      const int nreal = item.z;
      const int64_t e = item.w;
      if (!tc::mbar_wait(&tfull[buf], use & 1, wb)) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      uint32_t r[32];
      tc::tmem_ld32(taddr + lane_base + buf * 64, r);
      tc::tmem_ld_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[buf]);
      if (u + 2 < u1) {
        write_scales<EPI>(d, stg, taddr, q, lane, u + 2, buf);
        if (lane == 0) tc::mbar_arrive(&sready[buf]);
      }
      float acc[kTok];
#pragma unroll
      for (int j = 0; j < kTok; ++j) {
        acc[j] = __uint_as_float(r[j]) + __uint_as_float(r[kTok + j]);
        if (d.planes == 3) acc[j] += __uint_as_float(r[2 * kTok + j]);
      }
      if (EPI == EPI_SWIGLU) {
        float* xs = ex + (buf * 2 + (q & 1)) * kTok * 32;
        if (q >= 2) {  // up rows: hand the values to the warp holding the same features' gate rows
          if (!tc::mbar_wait(&xempty[buf], (use & 1) ^ 1, wb)) {
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
        if (!tc::mbar_wait(&xfull[buf], use & 1, wb)) {
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
          uint32_t code[3], sb;
          split_planes(__half2float(hv), 3, code, sb);
          uint8_t* dst = d.hq + (int64_t)p * 3 * d.hkp + f;
          dst[0] = (uint8_t)code[0];
          dst[d.hkp] = (uint8_t)code[1];
          dst[2 * d.hkp] = (uint8_t)code[2];
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

int dt_nst(int Kin) { return (Kin + 127) / 128; }
int dt_kp(int Kin) { return dt_nst(Kin) * 128; }
int dt_sb(int Kin) { return (dt_nst(Kin) * 4 + 15) / 16 * 16; }
size_t r256(size_t v) { return (v + 255) / 256 * 256; }

constexpr int kSmemMax = 227 * 1024;

// Stage slots: up to kLag + 2 (kLag stages in flight, two for the MMA: a stage handed over is
// reused two stages later, which hides the MMA's completion).  The copies go through L1
// (8-byte cp.async.ca): the carve-out below leaves L1 whatever shared memory does not take.
int dt_stages(int planes, int Kin) {
  const DtLayout L0 = dt_layout(0, planes, Kin, dt_sb(Kin));
  const int s = (kSmemMax - 1024 - L0.total) / (L0.slot + 16);
  return s < kLag + 2 ? s : kLag + 2;
}

template <int EPI>
cudaError_t launch_dt(const DtArgs& d, cudaStream_t stream) {
  const int smem = dt_layout(d.stages, d.planes, d.g.Kin, d.sb_tok).total + 1024;
  cudaError_t err = cudaFuncSetAttribute(decode_tc_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  // the smallest shared-memory carve-out that holds the layout: the rest of the SM's 256 KB
  // stays L1, which holds the 8-byte copies in flight
  const int pct = (smem * 100 + kSmemMax - 1) / kSmemMax;
  err = cudaFuncSetAttribute(decode_tc_kernel<EPI>, cudaFuncAttributePreferredSharedMemoryCarveout, pct);
  if (err != cudaSuccess) return err;
  decode_tc_kernel<EPI><<<(unsigned)moe_launch::sm_count_current(), kThreads, smem, stream>>>(d);
  return cudaGetLastError();
}

}  // namespace

namespace moe_launch {

bool decode_tc_supported(const GroupedGemm& g1, const GroupedGemm& g2) {
  auto ok = [](const GroupedGemm& g, int epi) {
    if (g.wfmt != WF_MXFP4 || g.epi != epi || g.act_by_slot || g.out_by_slot) return false;
    // scale rows of an even number of bytes, tensor memory for every stage's scales
    if (g.Kin % 64 != 0 || g.Kin > 128 * kMaxNst) return false;
    if (epi == EPI_SWIGLU ? (g.Nout % 64 != 0 || g.Nw != 2 * (int64_t)g.Nout)
                          : (g.Nout % 32 != 0 || g.Nw != (int64_t)g.Nout))
      return false;
    if (g.bm % kTok != 0 || g.bm > 128) return false;
    return dt_stages(epi == EPI_SWIGLU ? 2 : 3, g.Kin) >= 2;
  };
  return ok(g1, EPI_SWIGLU) && ok(g2, EPI_WEIGHTED_F32) && g2.Kin == g1.Nout && g1.P == g2.P;
}

size_t decode_tc_workspace_bytes(int64_t T_rows, int k, int K, int I) {
  if (T_rows <= 0 || k < 1 || K < 1 || I < 1) return 0;
  const int64_t P = T_rows * k;
  return r256((size_t)T_rows * 2 * dt_kp(K)) + r256((size_t)T_rows * dt_sb(K)) +
         r256((size_t)P * 3 * dt_kp(I)) + r256((size_t)P * dt_sb(I)) + r256((size_t)(P + 1) * 16);
}

DecodeTcBufs decode_tc_carve(void* ws, int64_t T_rows, int k, int K, int I) {
  const int64_t P = T_rows * k;
  uint8_t* p = static_cast<uint8_t*>(ws);
  DecodeTcBufs b;
  b.xq = p;
  p += r256((size_t)T_rows * 2 * dt_kp(K));
  b.xs = p;
  p += r256((size_t)T_rows * dt_sb(K));
  b.hq = p;
  p += r256((size_t)P * 3 * dt_kp(I));
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
  pa.kp = dt_kp(g1.Kin);
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
  dt_prep_kernel<<<(unsigned)(1 + blocks), kPrepThreads, 0, stream>>>(pa);
  return cudaGetLastError();
}

cudaError_t decode_tc_gemm(const GroupedGemm& g, const DecodeTcBufs& b, cudaStream_t stream) {
  DtArgs d{};
  d.g = g;
  d.kp = dt_kp(g.Kin);
  d.sb_tok = dt_sb(g.Kin);
  d.items = b.items;
  d.n_items = b.n_items;
  d.nst = dt_nst(g.Kin);
  if (g.epi == EPI_SWIGLU) {
    d.bq = b.xq;
    d.bsc = b.xs;
    d.planes = 2;
    d.hq = b.hq;
    d.hsc = b.hs;
    d.hkp = dt_kp(g.Nout);
    d.hsb = dt_sb(g.Nout);
    d.n_rt = g.Nout / 64;
    d.stages = dt_stages(2, g.Kin);
    return launch_dt<EPI_SWIGLU>(d, stream);
  }
  d.bq = b.hq;
  d.bsc = b.hs;
  d.planes = 3;
  d.n_rt = (g.Nout + 127) / 128;
  d.stages = dt_stages(3, g.Kin);
  return launch_dt<EPI_WEIGHTED_F32>(d, stream);
}

}  // namespace moe_launch
