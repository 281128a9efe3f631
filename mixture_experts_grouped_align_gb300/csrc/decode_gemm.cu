// Grouped expert GEMM, weight-streaming variant (few rows per expert: decode shapes).
//
// One launch covers every expert ("Add MoE GEMM variants and weight-gradient kernel",
// aiter PR 5310, Summary: all expert GEMMs in a single launch).  The launch grid is
// (block slot of the alignment) x (16 output rows).  A thread block whose block slot is
// past num_tokens_post_padded, or whose expert id is the -1 sentinel, returns before it
// reads any weight, scale or bias (second review of the same page, sentinel handling).
//
// Why this shape: with few tokens per expert the layer is bound by reading the weights
// once from HBM ("tune the Nemotron MTP decode row on S5000 with a checked-in recipe",
// torchada PR 115: the M <= 28 decode bucket dominates the step).  The kernel streams
// each weight row exactly once per 8-token tile with coalesced 4/8/16-byte read-only
// loads, turns MXFP4 / E4M3 codes into float16 in registers with the hardware
// conversions (exact), and feeds m16n8k16 tensor-core MMAs with the weights as the
// 16-row operand and up to 8 tokens as the 8-column operand.  The four warps of a block
// each take a quarter of K and are summed in a fixed order, so every output element has
// one fixed reduction order whatever the number of tokens (padded and unpadded batches
// give identical bits).
//
// K permutation: inside a 32-element K block, lane quad q supplies logical MMA columns
// {2q, 2q+1, 2q+8, 2q+9} from physical elements 8q..8q+3 (first MMA) and 8q+4..8q+7
// (second MMA), for both operands -- a dot product does not depend on the order of its
// terms, and this lets every lane read 8 consecutive elements of one weight row.
// A 32-element K block is exactly one E8M0 scale block, so the two MMAs of a block give a
// partial sum that is multiplied by the block's scale (per weight row, and per token for
// MXFP8 activations) and added to the float32 accumulator.
#include "moe_common.cuh"
#include "cp_async.cuh"
#include "moe_launch.h"

namespace {

using namespace moe_launch;
using namespace cpa;

constexpr int kWarps = 4;   // warps per block, each a quarter of K
constexpr int kTok = 8;     // tokens per tile (MMA N)
constexpr int kRows = 16;   // output rows per block (MMA M)
constexpr unsigned kFull = 0xffffffffu;

// Weight streaming: each warp copies its K quarter of the block's weight rows through a
// ring of R shared-memory stages with cp.async (16-byte chunks, no register cost for
// the bytes in flight); stage = D scale blocks of every row, plus the same K range of
// the tile's token rows.  Row strides are padded so that the lanes' shared loads of one
// block hit distinct banks.
template <int WF>
struct Pipe;
template <>
struct Pipe<WF_MXFP4> {  // 16 B per 32-element block; lane reads 4 B (8 codes)
  static constexpr int BPB = 16, D = 4, R = 3, RS = 80;
};
template <>
struct Pipe<WF_MXFP8> {  // 32 B per block; lane reads 8 B
  static constexpr int BPB = 32, D = 2, R = 4, RS = 96;
};
template <>
struct Pipe<WF_BF16> {   // 64 B per block; lane reads 16 B
  static constexpr int BPB = 64, D = 2, R = 3, RS = 192;
};

struct Smem {
  int ring, wsc, red, total;  // byte offsets
  int ring_warp, sw;          // bytes of one warp's ring; floats per scale row
};

// Token rows in a ring slot: D blocks of 32 activations (E4M3 for MXFP8 weights, else 16
// bits), row stride padded by 16 bytes.
template <int WF>
__host__ __device__ constexpr int act_block_bytes() { return WF == WF_MXFP8 ? 32 : 64; }
template <int WF>
__host__ __device__ constexpr int act_row_stride() { return Pipe<WF>::D * act_block_bytes<WF>() + 16; }

// One ring slot: weight rows | 2 scale words per row | decoded scales (D per row) | token rows.
__host__ __device__ constexpr int slot_bytes(int WF, int nrows, int RS, int D) {
  return nrows * RS + ((WF != WF_BF16) ? nrows * 2 * 4 + nrows * D * 4 : 0);
}
template <int WF>
__host__ __device__ constexpr int act_offset(int nmat) {
  return slot_bytes(WF, nmat * kRows, Pipe<WF>::RS, Pipe<WF>::D);
}
template <int WF>
__host__ __device__ constexpr int ring_slot_total(int nmat) {
  return act_offset<WF>(nmat) + kTok * act_row_stride<WF>();
}

template <int WF, int R>
__host__ __device__ inline Smem smem_layout(int nmat, int Kin) {
  Smem s;
  s.ring_warp = R * ring_slot_total<WF>(nmat);
  s.sw = 0;
  (void)Kin;
  int off = 0;
  s.ring = off;  off += kWarps * s.ring_warp;
  s.wsc = off;
  s.red = off;   off += 2 * kWarps * nmat * 4 * 32 * 4;  // double-buffered cross-warp partials
  s.total = off;
  return s;
}

template <int WF>
struct Fmt;
template <>
struct Fmt<WF_MXFP4> {
  using W = uint32_t;  // 8 codes of one row: physical K 8q..8q+7 of a 32-block
  static __device__ __forceinline__ W lds(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
  // half 0: elements 0..3 of the lane's 8 -> (pair 0,1), (pair 2,3); half 1: elements 4..7
  static __device__ __forceinline__ void pairs(W w, int half, uint32_t& p0, uint32_t& p1) {
    p0 = moe::e2m1x2_to_f16x2((w >> (16 * half)) & 0xffu);
    p1 = moe::e2m1x2_to_f16x2((w >> (16 * half + 8)) & 0xffu);
  }
};
template <>
struct Fmt<WF_MXFP8> {
  using W = uint2;
  static __device__ __forceinline__ W lds(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
  static __device__ __forceinline__ void pairs(W w, int half, uint32_t& p0, uint32_t& p1) {
    const uint32_t v = half ? w.y : w.x;
    p0 = moe::e4m3x2_to_f16x2(v & 0xffffu);
    p1 = moe::e4m3x2_to_f16x2(v >> 16);
  }
};
template <>
struct Fmt<WF_BF16> {
  using W = uint4;
  static __device__ __forceinline__ W lds(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
  static __device__ __forceinline__ void pairs(W w, int half, uint32_t& p0, uint32_t& p1) {
    p0 = half ? w.z : w.x;
    p1 = half ? w.w : w.y;
  }
};

template <int WF>
__host__ __device__ inline int64_t wrow_bytes(int Kin) {
  return WF == WF_MXFP4 ? Kin / 2 : (WF == WF_MXFP8 ? Kin : (int64_t)Kin * 2);
}

// Work units are (alignment block, 16-row tile) pairs, block-major; a thread block owns
// a contiguous run of the units that num_tokens_post_padded makes live, so that each
// warp streams its weight K-slice through the ring without draining between units.
struct Unit {
  int64_t blk, e;
  int rt, nsub;
};

// Unit u; the block's expert and sub-tile count are reused from `prev` when it is in the
// same block (consecutive units mostly are), so the alignment arrays are read once per block.
__device__ __forceinline__ Unit load_unit(const GroupedGemm& a, int64_t u, int row_tiles,
                                          const Unit& prev) {
  Unit x;
  x.blk = u / row_tiles;
  x.rt = (int)(u - x.blk * row_tiles);
  if (x.blk == prev.blk) {
    x.e = prev.e;
    x.nsub = prev.nsub;
    return x;
  }
  x.e = a.expert_ids[x.blk];
  // real pairs form a prefix of every block: count them, 8 tokens per sub-tile
  int cnt = 0;
  const int lane = threadIdx.x & 31;
  for (int s0 = 0; s0 < a.bm; s0 += 32) {
    const int s = s0 + lane;
    const bool v = s < a.bm && a.sorted[x.blk * a.bm + s] < a.P;
    cnt += __popc(__ballot_sync(0xffffffffu, v));
  }
  x.nsub = (x.e >= 0 && x.e < a.E) ? (cnt + kTok - 1) / kTok : 0;
  return x;
}

// Weight row of unit row r (0..31): SwiGLU pairs gate row f with up row Nout + f; the
// routing-weighted GEMM takes 32 consecutive rows per unit (two 16-row MMA tiles against one
// copy of the token rows); the others 16.
__device__ __forceinline__ int64_t unit_row(const GroupedGemm& a, const Unit& x, int r) {
  if (a.epi == EPI_WEIGHTED_F32) return x.e * a.Nw + (int64_t)x.rt * (2 * kRows) + r;
  return x.e * a.Nw + ((r >= kRows) ? a.Nout : 0) + (int64_t)x.rt * kRows + (r & (kRows - 1));
}

// Weight-row matrices per unit and output rows per unit.
__host__ __device__ constexpr int unit_mats(int epi) { return (epi == EPI_SWIGLU || epi == EPI_WEIGHTED_F32) ? 2 : 1; }
__host__ __device__ constexpr int unit_out_rows(int epi) { return epi == EPI_WEIGHTED_F32 ? 2 * kRows : kRows; }

// E8M0 byte -> float bits: 2^(s-127); 0x00 -> 2^-127 (subnormal), 0xFF -> NaN.
__device__ __forceinline__ float e8m0_fast(uint32_t s) {
  uint32_t b = s << 23;
  b = (s == 0u) ? 0x00400000u : b;
  b = (s == 255u) ? 0x7fc00000u : b;
  return __uint_as_float(b);
}

template <int WF>
struct Lane;  // per-format lane mapping of the ring copies
template <>
struct Lane<WF_MXFP4> {  // 4 chunks per lane: rows lane/4 + 8i, block lane%4
  static constexpr int NPL = 4;
  static __device__ __forceinline__ int row(int lane, int i) { return (lane >> 2) + 8 * i; }
  static __device__ __forceinline__ int blk(int lane) { return lane & 3; }
  static __device__ __forceinline__ int sub(int lane) { return 0; }
};
template <>
struct Lane<WF_MXFP8> {  // rows lane/4 + 8i, block (lane%4)/2, 16-byte half lane%2
  static constexpr int NPL = 4;
  static __device__ __forceinline__ int row(int lane, int i) { return (lane >> 2) + 8 * i; }
  static __device__ __forceinline__ int blk(int lane) { return (lane & 3) >> 1; }
  static __device__ __forceinline__ int sub(int lane) { return lane & 1; }
};
template <>
struct Lane<WF_BF16> {   // rows lane/8 + 4i, block (lane%8)/4, 16-byte quarter lane%4
  static constexpr int NPL = 8;
  static __device__ __forceinline__ int row(int lane, int i) { return (lane >> 3) + 4 * i; }
  static __device__ __forceinline__ int blk(int lane) { return (lane & 7) >> 2; }
  static __device__ __forceinline__ int sub(int lane) { return lane & 3; }
};

template <int WF, int NMAT>
__host__ __device__ constexpr int ring_slot_bytes() {
  return ring_slot_total<WF>(NMAT);
}

// Token-row copies of one stage: chunk c = lane + 32 i is token c / (D * CPB), block
// (c / CPB) % D, 16-byte piece c % CPB of that block.
template <int WF>
struct ActCopy {
  static constexpr int CPB = act_block_bytes<WF>() / 16;
  static constexpr int PER_TOK = Pipe<WF>::D * CPB;
  static constexpr int N = (kTok * PER_TOK + 31) / 32;  // chunks per lane
};

// Issue side of the ring: the unit being copied and this lane's row addresses in it.
template <int WF, int NMAT>
struct Issuer {
  static constexpr int NPL = Lane<WF>::NPL * NMAT / 2;  // rows per lane (chunks / 32)
  static constexpr int NACT = ActCopy<WF>::N;
  int64_t iu, u_end;
  Unit ix;
  int isub, ist;
  uint32_t issued;
  const uint8_t* wrow[NPL];   // weight row start of this lane's rows
  int64_t srow[2];            // scale row offsets of this lane's two scale words (MX)
  const uint8_t* arow[NACT];  // token row start (plus block / piece offset) of this lane's chunks
  int64_t act_blk;            // (block, sub-tile) the token rows were bound for
  int act_sub;

  __device__ __forceinline__ void bind(const GroupedGemm& a, int64_t rb, int lane) {
    const uint8_t* wb = static_cast<const uint8_t*>(a.w);
#pragma unroll
    for (int i = 0; i < NPL; ++i) wrow[i] = wb + unit_row(a, ix, Lane<WF>::row(lane, i)) * rb;
    const int nkb = a.Kin / 32;
#pragma unroll
    for (int i = 0; i < 2; ++i) srow[i] = unit_row(a, ix, (lane >> 1) + 16 * i) * nkb;
  }

  // Token rows of sub-tile isub of the current unit's block (read once per block and
  // sub-tile: consecutive units of a block share them).
  __device__ __forceinline__ void bind_act(const GroupedGemm& a, int lane) {
    if (ix.blk == act_blk && isub == act_sub) return;
    act_blk = ix.blk;
    act_sub = isub;
    using AC = ActCopy<WF>;
    const int s = isub * kTok + lane;
    int p = (int)a.P;
    if (lane < kTok && s < a.bm) p = a.sorted[ix.blk * a.bm + s];
    const int64_t abytes = (WF == WF_MXFP8) ? 1 : 2;
#pragma unroll
    for (int i = 0; i < NACT; ++i) {
      const int c = lane + 32 * i;
      const int t = c / AC::PER_TOK, rem = c % AC::PER_TOK;
      const int pt = __shfl_sync(0xffffffffu, p, t & (kTok - 1));
      arow[i] = nullptr;
      if (t < kTok && pt < a.P) {
        const int64_t r = a.act_per_pair ? (int64_t)pt : (int64_t)(pt / a.k);
        arow[i] = static_cast<const uint8_t*>(a.act) + r * a.Kin * abytes +
                  (rem / AC::CPB) * act_block_bytes<WF>() + (rem % AC::CPB) * 16;
      }
    }
  }
};

template <int WF, int NMAT, int R>
__device__ __forceinline__ void issue_next(const GroupedGemm& a, Issuer<WF, NMAT>& c, uint32_t ring_s,
                                           int64_t rb, int kb0, int kb1, int nst, int row_tiles,
                                           int lane) {
  using PP = Pipe<WF>;
  using LN = Lane<WF>;
  using AC = ActCopy<WF>;
  constexpr int NROWS = NMAT * kRows;
  constexpr bool MX = (WF != WF_BF16);
  constexpr int SLOT = ring_slot_bytes<WF, NMAT>();
  constexpr int AOFF = act_offset<WF>(NMAT);
  if (c.iu < c.u_end) {
    const int kbs = kb0 + c.ist * PP::D;
    const uint32_t slot = ring_s + (c.issued % R) * SLOT;
    const int j = LN::blk(lane), sub = LN::sub(lane);
    if (kbs + j < kb1) {
#pragma unroll
      for (int i = 0; i < Issuer<WF, NMAT>::NPL; ++i)
        cp_async16(slot + LN::row(lane, i) * PP::RS + j * PP::BPB + sub * 16,
                   c.wrow[i] + (int64_t)(kbs + j) * PP::BPB + sub * 16);
    }
    if (MX) {  // the two 4-byte words that hold this stage's scale bytes of every row
      const int wi = lane & 1;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = (lane >> 1) + 16 * i;
        if (r < NROWS) {
          const int64_t wa = ((c.srow[i] + kbs) & ~int64_t(3)) + 4 * wi;
          if (wa < c.srow[i] + kb1) cp_async4(slot + NROWS * PP::RS + (r * 2 + wi) * 4, a.w_scale + wa);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < Issuer<WF, NMAT>::NACT; ++i) {  // this stage's K range of the token rows
      const int ci = lane + 32 * i;
      const int t = ci / AC::PER_TOK, rem = ci % AC::PER_TOK;
      if (c.arow[i] != nullptr && kbs + rem / AC::CPB < kb1)
        cp_async16(slot + AOFF + t * act_row_stride<WF>() + (rem / AC::CPB) * act_block_bytes<WF>() +
                       (rem % AC::CPB) * 16,
                   c.arow[i] + (int64_t)kbs * act_block_bytes<WF>());
    }
    if (++c.ist == nst) {
      c.ist = 0;
      if (++c.isub == c.ix.nsub) {
        c.isub = 0;
        do {
          ++c.iu;
          if (c.iu < c.u_end) c.ix = load_unit(a, c.iu, row_tiles, c.ix);
        } while (c.iu < c.u_end && c.ix.nsub == 0);
        if (c.iu < c.u_end) c.bind(a, rb, lane);
      }
      if (c.iu < c.u_end) c.bind_act(a, lane);
    }
  }
  cp_async_commit();
  ++c.issued;
}

// R: stages in each warp's ring.  Fewer stages leave room for more resident warps, which
// hide the conversion and MMA latencies better when there are many units; more stages keep
// more bytes in flight per warp when there are few.
template <int WF, int EPI, int R>
__global__ void __launch_bounds__(kWarps * 32, 4) decode_gemm_kernel(GroupedGemm a) {
  constexpr int NMAT = unit_mats(EPI);
  constexpr int NROWS = NMAT * kRows;
  constexpr bool MX = (WF != WF_BF16);
  constexpr bool ACT_E4M3 = (WF == WF_MXFP8);
  using F = Fmt<WF>;
  using W = typename F::W;
  using PP = Pipe<WF>;
  constexpr int SLOT = ring_slot_bytes<WF, NMAT>();
  constexpr int AOFF = act_offset<WF>(NMAT);

  extern __shared__ __align__(16) uint8_t smem[];
  const Smem L = smem_layout<WF, R>(NMAT, a.Kin);
  float* red = reinterpret_cast<float*>(smem + L.red);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int Kin = a.Kin, nkb = Kin / 32;
  const int kb0 = warp * nkb / kWarps, kb1 = (warp + 1) * nkb / kWarps, nb = kb1 - kb0;
  const int nst = (nb + PP::D - 1) / PP::D;
  const int64_t rb = wrow_bytes<WF>(Kin);
  uint8_t* ring = smem + L.ring + warp * L.ring_warp;
  const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring));

  // this block's run of live units
  const int row_tiles = a.Nout / unit_out_rows(EPI);
  const int64_t n_units = ((int64_t)*a.ntpp / a.bm) * row_tiles;
  const int64_t per = (n_units + gridDim.x - 1) / gridDim.x;
  const int64_t u_begin = blockIdx.x * per;
  const int64_t u_end = u_begin + per < n_units ? u_begin + per : n_units;
  if (u_begin >= u_end) return;

  Issuer<WF, NMAT> cur;
  cur.iu = u_begin;
  cur.u_end = u_end;
  Unit none;
  none.blk = -1;
  none.e = -1;
  none.rt = 0;
  none.nsub = 0;
  cur.ix = load_unit(a, cur.iu, row_tiles, none);
  cur.isub = 0;
  cur.ist = 0;
  cur.issued = 0;
  cur.act_blk = -1;
  cur.act_sub = 0;
  while (cur.ix.nsub == 0 && ++cur.iu < u_end) cur.ix = load_unit(a, cur.iu, row_tiles, cur.ix);
  if (cur.iu < u_end) {
    cur.bind(a, rb, lane);
    cur.bind_act(a, lane);
  }
#pragma unroll 1
  for (int s = 0; s < R - 1; ++s) issue_next<WF, NMAT, R>(a, cur, ring_s, rb, kb0, kb1, nst, row_tiles, lane);

  bool bad = false;
  uint32_t consumed = 0, red_buf = 0;
  Unit cx = none;
  for (int64_t cu = u_begin; cu < u_end; ++cu) {
    cx = load_unit(a, cu, row_tiles, cx);
    if (cx.nsub == 0) continue;
    // scale-byte offsets of the rows this lane decodes (rows lane/D + (32/D) i)
    uint32_t soff = 0;
    if (MX) {
#pragma unroll
      for (int i = 0; i < NROWS * PP::D / 32; ++i) {
        const int r = lane / PP::D + (32 / PP::D) * i;
        soff |= (uint32_t)((unit_row(a, cx, r) * nkb) & 3) << (8 * i);
      }
    }
    for (int csub = 0; csub < cx.nsub; ++csub) {
      const int64_t slot0 = cx.blk * a.bm + csub * kTok;
      int pr = (int)a.P;
      if (lane < kTok && csub * kTok + lane < a.bm) pr = a.sorted[slot0 + lane];
      const int p0 = __shfl_sync(kFull, pr, 0);
      // token column g: its row is in the ring when valid; an invalid column holds stale
      // bytes, which only reach that column's outputs (never stored, never flagged)
      const bool gvalid = __shfl_sync(kFull, pr, g) < a.P;
      bool xbad = false;
      int pc0 = __shfl_sync(kFull, pr, 2 * q), pc1 = __shfl_sync(kFull, pr, 2 * q + 1);
      if (pc0 >= a.P) pc0 = p0;
      if (pc1 >= a.P) pc1 = p0;
      const int64_t crow0 = a.act_per_pair ? (int64_t)pc0 : (int64_t)(pc0 / a.k);
      const int64_t crow1 = a.act_per_pair ? (int64_t)pc1 : (int64_t)(pc1 / a.k);

      float acc[NMAT][4];
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;

      for (int st = 0; st < nst; ++st) {
        issue_next<WF, NMAT, R>(a, cur, ring_s, rb, kb0, kb1, nst, row_tiles, lane);
        cp_async_wait<R - 1>();
        __syncwarp();
        const uint8_t* slot = ring + (consumed % R) * SLOT;
        float* sf = reinterpret_cast<float*>(ring + (consumed % R) * SLOT + NROWS * PP::RS + NROWS * 8);
        const int kbs = kb0 + st * PP::D;
        const uint8_t* xs = slot + AOFF + g * act_row_stride<WF>() + q * (act_block_bytes<WF>() / 4);
        if (MX) {  // decode this stage's scale bytes (row r, block j) to floats
          const uint32_t* words = reinterpret_cast<const uint32_t*>(slot + NROWS * PP::RS);
#pragma unroll
          for (int i = 0; i < NROWS * PP::D / 32; ++i) {
            const int r = lane / PP::D + (32 / PP::D) * i, j = lane % PP::D;
            const uint2 w2 = *reinterpret_cast<const uint2*>(words + 2 * r);
            const uint32_t off = (((soff >> (8 * i)) & 3u) + (uint32_t)kbs) & 3u;
            const uint32_t byte = __byte_perm(w2.x, w2.y, off + j) & 0xffu;
            sf[r * PP::D + j] = e8m0_fast(byte);
          }
          __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < PP::D; ++j) {
          const int kk = kbs + j;
          if (kk < kb1) {
            uint4 xv;
            if (ACT_E4M3) {
              const uint2 raw = *reinterpret_cast<const uint2*>(xs + j * act_block_bytes<WF>());
              xv.x = moe::e4m3x2_to_f16x2(raw.x & 0xffffu);
              xv.y = moe::e4m3x2_to_f16x2(raw.x >> 16);
              xv.z = moe::e4m3x2_to_f16x2(raw.y & 0xffffu);
              xv.w = moe::e4m3x2_to_f16x2(raw.y >> 16);
            } else {
              xv = *reinterpret_cast<const uint4*>(xs + j * act_block_bytes<WF>());
              if (MX && a.act_fmt == ACT_BF16) {  // bf16 activations for the f16 MMA
                xv.x = moe::bf16x2_to_f16x2(xv.x, &xbad);
                xv.y = moe::bf16x2_to_f16x2(xv.y, &xbad);
                xv.z = moe::bf16x2_to_f16x2(xv.z, &xbad);
                xv.w = moe::bf16x2_to_f16x2(xv.w, &xbad);
              } else if (!MX && a.act_fmt == ACT_F16) {
                xv.x = moe::f16x2_to_bf16x2(xv.x);
                xv.y = moe::f16x2_to_bf16x2(xv.y);
                xv.z = moe::f16x2_to_bf16x2(xv.z);
                xv.w = moe::f16x2_to_bf16x2(xv.w);
              }
            }
            float xs0 = 1.f, xs1 = 1.f;
            if (ACT_E4M3) {
              xs0 = moe::e8m0_to_f32(a.act_scale[crow0 * nkb + kk]);
              xs1 = moe::e8m0_to_f32(a.act_scale[crow1 * nkb + kk]);
            }
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
              const uint8_t* r0 = slot + (m * kRows + g) * PP::RS + j * PP::BPB + q * (PP::BPB / 4);
              const W w0 = F::lds(r0);
              const W w1 = F::lds(r0 + 8 * PP::RS);
              uint32_t A1[4], A2[4];
              if constexpr (WF == WF_MXFP4) {
                moe::e2m1x8_to_f16x2(w0, A1[0], A1[2], A2[0], A2[2]);
                moe::e2m1x8_to_f16x2(w1, A1[1], A1[3], A2[1], A2[3]);
              } else {
                F::pairs(w0, 0, A1[0], A1[2]);
                F::pairs(w1, 0, A1[1], A1[3]);
                F::pairs(w0, 1, A2[0], A2[2]);
                F::pairs(w1, 1, A2[1], A2[3]);
              }
              if (MX) {
                const float zero[4] = {0.f, 0.f, 0.f, 0.f};
                float t[4];
                moe::mma_f16(t, A1, xv.x, xv.y, zero);
                moe::mma_f16(t, A2, xv.z, xv.w, t);
                const float s0 = sf[(m * kRows + g) * PP::D + j];
                const float s1 = sf[(m * kRows + g + 8) * PP::D + j];
                if (ACT_E4M3) {
                  acc[m][0] = fmaf(t[0] * s0, xs0, acc[m][0]);
                  acc[m][1] = fmaf(t[1] * s0, xs1, acc[m][1]);
                  acc[m][2] = fmaf(t[2] * s1, xs0, acc[m][2]);
                  acc[m][3] = fmaf(t[3] * s1, xs1, acc[m][3]);
                } else {
                  acc[m][0] = fmaf(t[0], s0, acc[m][0]);
                  acc[m][1] = fmaf(t[1], s0, acc[m][1]);
                  acc[m][2] = fmaf(t[2], s1, acc[m][2]);
                  acc[m][3] = fmaf(t[3], s1, acc[m][3]);
                }
              } else {
                moe::mma_bf16(acc[m], A1, xv.x, xv.y, acc[m]);
                moe::mma_bf16(acc[m], A2, xv.z, xv.w, acc[m]);
              }
            }
          }
        }
        __syncwarp();
        ++consumed;
      }
      if (xbad && gvalid) bad = true;

      // fixed-order sum over the four K quarters (double-buffered partials), epilogue
      float* rb_ = red + red_buf * (kWarps * NMAT * 4 * 32);
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) rb_[((warp * NMAT + m) * 4 + i) * 32 + lane] = acc[m][i];
      __syncthreads();
      if (warp == 0) {
        float v[NMAT][4];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float s = rb_[((0 * NMAT + m) * 4 + i) * 32 + lane];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) s += rb_[((w * NMAT + m) * 4 + i) * 32 + lane];
            v[m][i] = s;
          }
        const int pcol0 = __shfl_sync(kFull, pr, 2 * q), pcol1 = __shfl_sync(kFull, pr, 2 * q + 1);
        const uint16_t* bias = static_cast<const uint16_t*>(a.bias);
        const int64_t e = cx.e;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int p = (i & 1) ? pcol1 : pcol0;
          if (p >= a.P) continue;
          const int n = cx.rt * kRows + g + ((i >> 1) << 3);
          if (EPI == EPI_SWIGLU) {
            float gt = v[0][i], up = v[NMAT - 1][i];
            if (bias) {
              gt += moe::bf16_bits_to_f32(bias[e * a.Nw + n]);
              up += moe::bf16_bits_to_f32(bias[e * a.Nw + a.Nout + n]);
            }
            const float hval = moe::silu(gt) * up;
            if (ACT_E4M3) {  // MXFP8 layer: fp32, quantised to MXFP8 before GEMM2
              static_cast<float*>(a.out)[(int64_t)p * a.Nout + n] = hval;
            } else if (MX) {  // f16 for the f16 MMA of GEMM2; an overflow is reported
              const __half hv = __float2half_rn(hval);
              if (__hisinf(hv)) bad = true;  // an overflow (NaN only comes from NaN inputs)
              static_cast<__half*>(a.out)[(int64_t)p * a.Nout + n] = hv;
            } else {   // bf16 for the bf16 MMA of GEMM2
              static_cast<uint16_t*>(a.out)[(int64_t)p * a.Nout + n] = moe::f32_to_bf16_bits(hval);
            }
          } else if (EPI == EPI_RELU2) {
            float av = v[0][i];
            if (bias) av += moe::bf16_bits_to_f32(bias[e * a.Nw + n]);
            const float hval = moe::relu2(av);
            if (ACT_E4M3) {
              static_cast<float*>(a.out)[(int64_t)p * a.Nout + n] = hval;
            } else if (MX) {
              const __half hv = __float2half_rn(hval);
              if (__hisinf(hv)) bad = true;
              static_cast<__half*>(a.out)[(int64_t)p * a.Nout + n] = hv;
            } else {
              static_cast<uint16_t*>(a.out)[(int64_t)p * a.Nout + n] = moe::f32_to_bf16_bits(hval);
            }
          } else if (EPI == EPI_WEIGHTED_F32) {  // rows rt * 32 + 16 m + (g, g + 8)
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
              const int nm = cx.rt * (2 * kRows) + m * kRows + g + ((i >> 1) << 3);
              float o = v[m][i];
              if (bias) o += moe::bf16_bits_to_f32(bias[e * a.Nw + nm]);
              static_cast<float*>(a.out)[(int64_t)p * a.Nout + nm] = o * a.topk_w[p];
            }
          } else {
            float o = v[0][i];
            if (bias) o += moe::bf16_bits_to_f32(bias[e * a.Nw + n]);
            static_cast<uint16_t*>(a.out)[(int64_t)p * a.Nout + n] = moe::f32_to_bf16_bits(o);
          }
        }
      }
      red_buf ^= 1;
    }
  }
  cp_async_wait<0>();
  if (bad) moe::set_status(a.status, MOE_ERR_RANGE);
}

int sm_count_dec() { return moe_launch::sm_count_current(); }

// Resident blocks of the R-stage variant on the whole GPU (0 on error).
template <int WF, int EPI, int R>
int64_t resident_blocks(const GroupedGemm& g) {
  const Smem L = smem_layout<WF, R>(unit_mats(EPI), g.Kin);
  if (cudaFuncSetAttribute(decode_gemm_kernel<WF, EPI, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total) !=
      cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_gemm_kernel<WF, EPI, R>, kWarps * 32, L.total) !=
      cudaSuccess)
    return 0;
  return (int64_t)sm_count_dec() * (per_sm < 1 ? 1 : per_sm);
}

template <int WF, int EPI, int R>
cudaError_t launch_t(const GroupedGemm& g, cudaStream_t stream) {
  const Smem L = smem_layout<WF, R>(unit_mats(EPI), g.Kin);
  // enough resident blocks to keep every SM streaming; each owns a run of live units
  int64_t grid = resident_blocks<WF, EPI, R>(g);
  if (grid <= 0) return cudaErrorInvalidValue;
  const int64_t units = g.grid_blocks * (g.Nout / unit_out_rows(EPI));
  if (units < grid) grid = units;
  if (grid <= 0) return cudaSuccess;
  decode_gemm_kernel<WF, EPI, R><<<(unsigned)grid, kWarps * 32, L.total, stream>>>(g);
  return cudaGetLastError();
}

// Ring depth: two stages for MXFP4 codes (measured faster on the 64-token decode layer).
// For bf16 weights, two stages when every unit fits in two rounds of the two-stage
// variant's resident blocks (a one-token step: the smaller ring lets one more block per SM
// in and shortens the longest run), else three; MXFP8 keeps its four.
template <int WF, int EPI>
cudaError_t launch_r(const GroupedGemm& g, cudaStream_t stream) {
  if (WF == WF_MXFP4) return launch_t<WF, EPI, 2>(g, stream);
  if (WF == WF_BF16) {
    const int64_t units = g.grid_blocks * (g.Nout / unit_out_rows(EPI));
    if (units <= 2 * resident_blocks<WF, EPI, 2>(g)) return launch_t<WF, EPI, 2>(g, stream);
    return launch_t<WF, EPI, 3>(g, stream);
  }
  return launch_t<WF, EPI, Pipe<WF>::R>(g, stream);
}

}  // namespace

namespace moe_launch {

size_t decode_gemm_smem_bytes(const GroupedGemm& g) {
  const int nmat = unit_mats(g.epi);
  if (g.wfmt == WF_MXFP4) return smem_layout<WF_MXFP4, 2>(nmat, g.Kin).total;
  if (g.wfmt == WF_MXFP8) return smem_layout<WF_MXFP8, Pipe<WF_MXFP8>::R>(nmat, g.Kin).total;
  return smem_layout<WF_BF16, 3>(nmat, g.Kin).total;
}

cudaError_t decode_gemm(const GroupedGemm& g, cudaStream_t stream) {
#define MOE_CASE(WF, EP) \
  if (g.wfmt == WF && g.epi == EP) return launch_r<WF, EP>(g, stream);
  MOE_CASE(WF_MXFP4, EPI_SWIGLU)
  MOE_CASE(WF_MXFP4, EPI_WEIGHTED_F32)
  MOE_CASE(WF_MXFP4, EPI_PLAIN_BF16)
  MOE_CASE(WF_MXFP4, EPI_RELU2)
  MOE_CASE(WF_BF16, EPI_SWIGLU)
  MOE_CASE(WF_BF16, EPI_WEIGHTED_F32)
  MOE_CASE(WF_BF16, EPI_PLAIN_BF16)
  MOE_CASE(WF_BF16, EPI_RELU2)
  MOE_CASE(WF_MXFP8, EPI_SWIGLU)
  MOE_CASE(WF_MXFP8, EPI_RELU2)
  MOE_CASE(WF_MXFP8, EPI_WEIGHTED_F32)
  MOE_CASE(WF_MXFP8, EPI_PLAIN_BF16)
#undef MOE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe_launch
