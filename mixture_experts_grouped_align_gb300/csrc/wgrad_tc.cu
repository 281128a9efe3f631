// Per-expert weight gradient on the tensor-memory path (deterministic mode).
//
// dW[e] = sum over the pairs p routed to e of grad[p]^T (outer) input[src(p)], read
// straight from the alignment outputs ("Add MoE GEMM variants and weight-gradient
// kernel", aiter PR 5310, Summary: moe_wgrad; Tests & Benchmarks: zero-padded tokens add
// nothing).  One persistent launch; a tile is a 128 (N) x BN (Kin) block of one dW[e],
// expert-major so that an expert's rows stay in L2 across its tiles.
//
// The token index is the reduction index and the slow index of both grad [P, N] and
// input [., Kin], so both operands are staged token-major, exactly as they lie in
// memory, into MN-major 128-byte-swizzle atoms (64 MN elements x 8 tokens) and fed to
// tcgen05.mma (kind::f16, bf16, M = 128, N = BN, K = 16) with both operands MN-major.
// Two feeds of the same stages:
//   gather feed (no workspace): warps 8-15 copy each stage's token rows from grad and
//     input with cp.async (16 B, sentinel slots zero-filled); warps 4-7 drain the
//     accumulators with plain stores through a padded staging tile.
//   slot feed (grad and input already copied into slot order): one thread loads a stage as
//     2 + BN/64 TMA boxes of 64 slots x 128 bytes, which land in exactly the atom layout;
//     warps 4-11 (two per TMEM lane quarter, one half of the columns each) drain the
//     accumulators through swizzled 32 x 32 staging boxes that leave by TMA stores.
// Warp 0 owns TMEM (two 128 x 256 fp32 accumulators) and issues the MMAs.  Both feeds run
// the same MMAs on the same stages in the same order, so they give identical bits.
// Every mbarrier wait is bounded; a wait that runs out sets MOE_ERR_TIMEOUT and every
// role leaves its loop.  Each tile sums its tokens in one fixed order: repeatable bits.
#include "moe_common.cuh"
#include "cp_async.cuh"
#include "moe_launch.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace {

using namespace moe_launch;
using namespace cpa;

constexpr int kThreads = 512;
constexpr int kTM = 128;          // dW rows (N) per tile
constexpr int kTok = 64;          // token slots per stage
constexpr int kProd0 = 256, kNumProd = 256;
constexpr int kEpiWarp0 = 4;
constexpr int kTmemCols = 512;
constexpr int kAtom = 1024;       // 64 MN elements x 8 tokens x 2 B
constexpr int kAtomCol = 8 * kAtom;  // one MN atom column over the stage's 64 tokens
constexpr int kMaxStages = 4;

constexpr int kStageLd = 36;                 // gather feed: staging row stride (floats), conflict-free
constexpr int kStage = 4 * 32 * kStageLd;    // floats of its epilogue staging (4 warps)
constexpr int kBox = 32 * 128;               // slot feed: one 32 x 32 fp32 store box (bytes)
constexpr int kSlotEpiWarps = 8;

struct WLayout {
  int a, b, slot, nslots, stg, zero, bars, eb, total;
};

// Stages (A = 2 MN atom columns (128 n) | B = BN/64 atom columns) | epilogue staging (slot
// feed: two store boxes per epilogue warp and one zero box) | barriers | expert block
// ranges (8 KB).  Offsets from a 1024-byte aligned base.
__host__ __device__ inline WLayout wlayout(int BN, bool slot_feed) {
  WLayout L;
  L.a = 0;
  L.b = 2 * kAtomCol;
  L.slot = L.b + (BN / 64) * kAtomCol;
  const int staging = slot_feed ? (2 * kSlotEpiWarps + 1) * kBox : kStage * 4;
  int n = (227 * 1024 - 1024 - 256 - 8 * 1024 - staging) / L.slot;
  L.nslots = n > kMaxStages ? kMaxStages : n;
  L.stg = L.nslots * L.slot;
  L.zero = L.stg + 2 * kSlotEpiWarps * kBox;
  L.bars = L.stg + staging;
  L.eb = L.bars + 256;
  L.total = L.eb + 8 * 1024 + 1024;
  return L;
}

struct WArgs {
  Wgrad g;
  int BN;          // Kin columns per tile (multiple of 64, <= 256)
  int n_tiles;     // N / 128
  int c_tiles;     // Kin / BN
  int nt_fast;     // 1: N tiles vary fastest within an expert (every grad column live at once)
  int64_t tiles;   // E * n_tiles * c_tiles
};

// Byte offset of (token t, 16-byte chunk c of a row of 64 MN elements) in an atom column.
__device__ __forceinline__ uint32_t mn_offset(int t, int c) {
  return (uint32_t)((t >> 3) * kAtom + (t & 7) * 128 + ((c ^ (t & 7)) << 4));
}

struct TileInfo {
  int64_t e;
  int nt, ct;
  int64_t slot_beg, slot_end;  // the expert's token slots
};

// Tile t -> expert, N tile, Kin tile and the expert's slot range (from the per-expert
// block ranges the thread block built in shared memory).  Within an expert the tile index
// whose operand is narrower over all tiles varies fastest, so that the tiles running at
// once share the wider operand's columns and their rows stay small in L2.
__device__ __forceinline__ TileInfo tile_info(const WArgs& wa, int64_t t, const int* eb) {
  const Wgrad& a = wa.g;
  TileInfo ti;
  const int64_t per_e = (int64_t)wa.n_tiles * wa.c_tiles;
  ti.e = t / per_e;
  const int rem = (int)(t - ti.e * per_e);
  if (wa.nt_fast) {
    ti.ct = rem / wa.n_tiles;
    ti.nt = rem - ti.ct * wa.n_tiles;
  } else {
    ti.nt = rem / wa.c_tiles;
    ti.ct = rem - ti.nt * wa.c_tiles;
  }
  ti.slot_beg = (int64_t)eb[2 * ti.e] * a.bm;
  ti.slot_end = (int64_t)eb[2 * ti.e + 1] * a.bm;
  return ti;
}

template <bool SLOT>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_i,
                    const __grid_constant__ CUtensorMap tm_d, WArgs wa) {
  const Wgrad& a = wa.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = wa.BN;
  const WLayout L = wlayout(BN, SLOT);
  const int S = L.nslots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_s + 1);
  int* eb = reinterpret_cast<int*>(smem + L.eb);  // [E][2]: first, end block

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nblocks = *a.ntpp / a.bm;
  for (int i = tid; i < 2 * a.E; i += kThreads) eb[i] = 0;
  if (SLOT) {  // the zero box that the stores of an expert with no pair read
    for (int i = tid; i < kBox / 16; i += kThreads)
      *reinterpret_cast<uint4*>(smem + L.zero + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    tc::fence_proxy_async_smem();
  }
  __syncthreads();
  for (int b = tid; b < nblocks; b += kThreads) {  // used blocks: ascending expert ids
    const int e = a.expert_ids[b];
    if (e < 0 || e >= a.E) continue;
    if (b == 0 || a.expert_ids[b - 1] != e) eb[2 * e] = b;
    if (b == nblocks - 1 || a.expert_ids[b + 1] != e) eb[2 * e + 1] = b + 1;
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      // gather feed: one completion arrival per producer thread; slot feed: the TMA thread
      tc::mbar_init(&full[s], SLOT ? 1 : kNumProd);
      tc::mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], SLOT ? kSlotEpiWarps : 4);
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
  const uint32_t smem_s = tc::smem_addr(smem);

  if (!SLOT && warp >= 8) {
    // ------------------------------------------------------------------ gather feed
    const int pt = tid - kProd0;
    const int t = pt >> 2, sub = pt & 3;  // token row of the stage, chunk phase
    const uint16_t* grad = static_cast<const uint16_t*>(a.grad);
    const uint16_t* inp = static_cast<const uint16_t*>(a.input);
    uint32_t a_off[4], b_off[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = sub + 4 * i;
      a_off[i] = L.a + (j >> 3) * kAtomCol + mn_offset(t, j & 7);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = sub + 4 * i;
      b_off[i] = L.b + (j >> 3) * kAtomCol + mn_offset(t, j & 7);
    }
    const int nbj = BN / 32;  // B chunks per thread
    // Each thread's copies of a stage complete on the stage's barrier by themselves
    // (cp.async.mbarrier.arrive.noinc), so no producer waits for its own copies and every
    // free slot can have a stage in flight; the MMA lane makes the landed bytes visible to
    // the tensor core with a proxy fence after its wait.
    // A cursor over (tile, stage) pairs of this block, one step ahead of the copies: the
    // pair id of the next stage's token row is loaded before this stage waits for its slot.
    int64_t tt = blockIdx.x, st = 0, nst = 0;
    TileInfo ti{};
    auto seek = [&]() {  // the first tile from tt on with a stage (an expert with pairs)
      for (; tt < wa.tiles; tt += gridDim.x) {
        ti = tile_info(wa, tt, eb);
        nst = (ti.slot_end - ti.slot_beg + kTok - 1) / kTok;
        if (nst > 0) return;
      }
    };
    auto pair_at = [&]() -> int64_t {
      const int64_t s = ti.slot_beg + st * kTok + t;
      return s < ti.slot_end ? (int64_t)a.sorted[s] : a.P;
    };
    seek();
    int64_t p_next = tt < wa.tiles ? pair_at() : a.P;
    uint32_t it = 0;
    while (tt < wa.tiles && !*abort_flag) {
      const int64_t p = p_next;
      const int64_t n0 = (int64_t)ti.nt * kTM, c0 = (int64_t)ti.ct * BN;
      if (++st == nst) {
        st = 0;
        tt += gridDim.x;
        seek();
      }
      if (tt < wa.tiles) p_next = pair_at();
      const int slot = it % S;
      if (!tc::mbar_wait(&empty[slot], ((it / S) & 1) ^ 1)) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      const uint32_t sl = smem_s + slot * L.slot;
      const bool valid = p < a.P;
      const int64_t srow = a.input_per_pair ? p : p / a.k;
      const uint16_t* gsrc = valid ? grad + p * a.N + n0 + sub * 8 : grad;
      const uint16_t* isrc = valid ? inp + srow * a.Kin + c0 + sub * 8 : inp;
#pragma unroll
      for (int i = 0; i < 4; ++i) cp_async16z(sl + a_off[i], gsrc + (valid ? 32 * i : 0), valid);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i < nbj) cp_async16z(sl + b_off[i], isrc + (valid ? 32 * i : 0), valid);
      cp_async_arrive_noinc(&full[slot]);
      ++it;
    }
    cp_async_wait_all();
  } else if (SLOT && warp == 1) {
    // ------------------------------------------------------------------ slot feed (TMA)
    if (lane == 0) {
      tma::prefetch_map(&tm_g);
      tma::prefetch_map(&tm_i);
      const uint32_t stage_tx = (uint32_t)(2 + BN / 64) * kAtomCol;
      uint32_t it = 0;
      for (int64_t tt = blockIdx.x; tt < wa.tiles && !*abort_flag; tt += gridDim.x) {
        const TileInfo ti = tile_info(wa, tt, eb);
        const int64_t nst = (ti.slot_end - ti.slot_beg) / kTok;  // block_m is a multiple of kTok
        const int32_t xg = (int32_t)((int64_t)ti.nt * kTM * 2), xi = (int32_t)((int64_t)ti.ct * BN * 2);
        bool ok = true;
        for (int64_t st = 0; st < nst; ++st) {
          const int slot = it % S;
          if (!tc::mbar_wait(&empty[slot], ((it / S) & 1) ^ 1)) {
            ok = false;
            break;
          }
          const uint32_t sl = smem_s + slot * L.slot;
          const int32_t y = (int32_t)(ti.slot_beg + st * kTok);
          tma::mbar_arrive_expect_tx(&full[slot], stage_tx);
          // 64 slots x 64 bf16 per box, 128-byte swizzled: one MN atom column
          tma::load_2d(sl + L.a, &tm_g, xg, y, &full[slot]);
          tma::load_2d(sl + L.a + kAtomCol, &tm_g, xg + 128, y, &full[slot]);
          for (int j = 0; j < BN / 64; ++j) tma::load_2d(sl + L.b + j * kAtomCol, &tm_i, xi + 128 * j, y, &full[slot]);
          ++it;
        }
        if (!ok) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
      }
      // Leaving early: the loads already issued still land in this block's shared memory,
      // so wait for the last armed phase of every slot before exiting.
      if (*abort_flag)
        for (uint32_t j = it > (uint32_t)S ? it - S : 0; j < it; ++j)
          if (!tc::mbar_wait(&full[j % S], (j / S) & 1)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(kTM, BN, 1) | (1u << 15) | (1u << 16);
      uint32_t it = 0, acc_it = 0;
      for (int64_t tt = blockIdx.x; tt < wa.tiles && !*abort_flag; tt += gridDim.x) {
        const TileInfo ti = tile_info(wa, tt, eb);
        const int64_t nst = (ti.slot_end - ti.slot_beg + kTok - 1) / kTok;
        if (nst == 0) continue;  // the epilogue writes zeros itself
        const uint32_t acc = acc_it & 1;
        if (!tc::mbar_wait(&tempty[acc], ((acc_it >> 1) & 1) ^ 1)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d_tmem = taddr + acc * 256;
        bool ok = true;
        for (int64_t st = 0; st < nst; ++st) {
          const int slot = it % S;
          if (!tc::mbar_wait(&full[slot], (it / S) & 1)) {
            moe::set_status(a.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (!SLOT) tc::fence_proxy_async_smem();  // the producers' landed copies, for the tensor core
          tc::tc_fence_after();
          const uint32_t a_s = smem_s + slot * L.slot + L.a;
          const uint32_t b_s = smem_s + slot * L.slot + L.b;
#pragma unroll
          for (int k4 = 0; k4 < kTok / 16; ++k4)
            tc::mma_f16_ss(d_tmem, tc::sdesc_sw128_mn(a_s + k4 * 2 * kAtom, kAtomCol, kAtom),
                           tc::sdesc_sw128_mn(b_s + k4 * 2 * kAtom, kAtomCol, kAtom), idesc,
                           (st | k4) != 0);
          tc::mma_commit(&empty[slot]);
          ++it;
        }
        if (!ok) break;
        tc::mma_commit(&tfull[acc]);
        ++acc_it;
      }
      tc::mma_commit(drain);
      if (!tc::mbar_wait(drain, 0)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (!SLOT && warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------------ epilogue (gather feed)
    // TMEM lane = dW row.  Each 32 x 32 chunk goes through shared memory so that the
    // stores to dW are whole 128-byte row segments (4 rows per store instruction).
    const int quarter = warp - kEpiWarp0;
    float* stg = reinterpret_cast<float*>(smem + L.stg) + quarter * 32 * kStageLd;
    const int rr = lane >> 3, cc = (lane & 7) * 4;  // store phase: row rr + 4i, columns cc..cc+3
    uint32_t acc_it = 0;
    for (int64_t tt = blockIdx.x; tt < wa.tiles && !*abort_flag; tt += gridDim.x) {
      const TileInfo ti = tile_info(wa, tt, eb);
      float* tile = a.dW + ((ti.e * a.N) + (int64_t)ti.nt * kTM + quarter * 32) * (int64_t)a.Kin +
                    (int64_t)ti.ct * BN;
      if (ti.slot_end == ti.slot_beg) {  // an expert with no pair: dW[e] = 0
        for (int r = 0; r < 32; ++r)
          for (int c = lane * 4; c < BN; c += 128)
            *reinterpret_cast<float4*>(tile + (int64_t)r * a.Kin + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const uint32_t acc = acc_it & 1;
      if (!tc::mbar_wait(&tfull[acc], (acc_it >> 1) & 1)) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      const uint32_t tb = taddr + acc * 256 + ((uint32_t)(quarter * 32) << 16);
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld32(tb + c0, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(stg + lane * kStageLd + 4 * q) = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = rr + 4 * i;
          *reinterpret_cast<float4*>(tile + (int64_t)r * a.Kin + c0 + cc) =
              *reinterpret_cast<const float4*>(stg + r * kStageLd + cc);
        }
        __syncwarp();
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[acc]);
      ++acc_it;
    }
  } else if (SLOT && warp >= kEpiWarp0 && warp < kEpiWarp0 + kSlotEpiWarps) {
    // ------------------------------------------------------------------ epilogue (slot feed)
    // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (= its 32 dW rows) and half (w - 4) / 4 of
    // the tile's columns, 32 at a time: registers -> a 128-byte swizzled 32 x 32 box in
    // shared memory (two per warp, alternating) -> one TMA store.
    const int ew = warp - kEpiWarp0, quarter = warp & 3, half = ew >> 2;
    const int cols = BN / 2;
    const uint32_t stg0 = smem_s + L.stg + ew * 2 * kBox;
    uint32_t nstore = 0, acc_it = 0;
    for (int64_t tt = blockIdx.x; tt < wa.tiles && !*abort_flag; tt += gridDim.x) {
      const TileInfo ti = tile_info(wa, tt, eb);
      const int32_t row0 = (int32_t)(ti.e * a.N + (int64_t)ti.nt * kTM + quarter * 32);
      const int32_t col0 = ti.ct * BN + half * cols;
      if (ti.slot_end == ti.slot_beg) {  // an expert with no pair: dW[e] = 0
        if (lane == 0) {
          for (int c = 0; c < cols; c += 32) tma::store_2d(&tm_d, (col0 + c) * 4, row0, smem_s + L.zero);
          tma::bulk_commit();
        }
        continue;
      }
      const uint32_t acc = acc_it & 1;
      if (!tc::mbar_wait(&tfull[acc], (acc_it >> 1) & 1)) {
        moe::set_status(a.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      const uint32_t tb = taddr + acc * 256 + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(half * cols);
      for (int c = 0; c < cols; c += 32) {
        uint32_t v[32];
        tc::tmem_ld32(tb + c, v);
        tc::tmem_ld_wait();
        // the store that last read this box (two stores ago) has finished reading it
        if (lane == 0) tma::bulk_wait_read_1();
        __syncwarp();
        const uint32_t box = stg0 + (nstore & 1) * kBox;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(box + lane * 128 + ((q ^ (lane & 7)) << 4)),
                       "r"(v[4 * q]), "r"(v[4 * q + 1]), "r"(v[4 * q + 2]), "r"(v[4 * q + 3])
                       : "memory");
        tc::fence_proxy_async_smem();  // these writes, for the TMA engine
        __syncwarp();
        if (lane == 0) {
          tma::store_2d(&tm_d, (col0 + c) * 4, row0, box);
          tma::bulk_commit();
        }
        ++nstore;
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[acc]);
      ++acc_it;
    }
    if (lane == 0) tma::bulk_wait_all();
    __syncwarp();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, kTmemCols);
  }
}

int sm_count_w() { return moe_launch::sm_count_current(); }

}  // namespace

namespace moe_launch {

// Kin tile of the tensor-memory wgrad, or 0 when the shape does not fit it.
int wgrad_tc_tile(const Wgrad& g) {
  // the per-expert block ranges live in 8 KB of shared memory: at most 1024 experts
  if (g.mode != 0 || g.N % kTM != 0 || g.Kin % 64 != 0 || g.E > 1024) return 0;
  for (int bn : {256, 192, 128, 64})
    if (g.Kin % bn == 0) return bn;
  return 0;
}

bool wgrad_tc_slot_feed(const Wgrad& g) {
  // whole 64-slot stages never cross into the next expert's slots; TMA row coordinates
  // (slots, and dW rows e * N + n) are 32-bit
  return wgrad_tc_tile(g) > 0 && g.bm % kTok == 0 && g.cap < ((int64_t)1 << 31) &&
         (int64_t)g.E * g.N < ((int64_t)1 << 31) && (int64_t)g.Kin * 4 < ((int64_t)1 << 31);
}

cudaError_t wgrad_tc(const Wgrad& g, cudaStream_t stream) {
  WArgs wa;
  wa.g = g;
  wa.BN = wgrad_tc_tile(g);
  if (wa.BN == 0) return cudaErrorInvalidValue;
  wa.n_tiles = g.N / kTM;
  wa.c_tiles = g.Kin / wa.BN;
  wa.nt_fast = g.N <= g.Kin ? 1 : 0;
  wa.tiles = (int64_t)g.E * wa.n_tiles * wa.c_tiles;
  const bool slot = g.grad_s != nullptr && g.input_s != nullptr;
  if (slot && !wgrad_tc_slot_feed(g)) return cudaErrorInvalidValue;
  const WLayout L = wlayout(wa.BN, slot);
  int64_t grid = sm_count_w();
  if (wa.tiles < grid) grid = wa.tiles;
  if (grid <= 0) return cudaSuccess;
  CUtensorMap mg{}, mi{}, md{};
  if (slot) {
    // slot-ordered rows: boxes of 64 slots x 128 bytes, 128-byte swizzle (one MN atom
    // column); dW rows of Kin fp32, stored 32 rows x 128 bytes per box
    if (!tma::encode_2d_u8(&mg, g.grad_s, (uint64_t)g.N * 2, (uint64_t)g.cap, (uint64_t)g.N * 2, 128, kTok, true) ||
        !tma::encode_2d_u8(&mi, g.input_s, (uint64_t)g.Kin * 2, (uint64_t)g.cap, (uint64_t)g.Kin * 2, 128, kTok,
                           true) ||
        !tma::encode_2d_u8(&md, g.dW, (uint64_t)g.Kin * 4, (uint64_t)g.E * g.N, (uint64_t)g.Kin * 4, 128, 32, true))
      return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(wgrad_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (err != cudaSuccess) return err;
    wgrad_tc_kernel<true><<<(unsigned)grid, kThreads, L.total, stream>>>(mg, mi, md, wa);
  } else {
    cudaError_t err = cudaFuncSetAttribute(wgrad_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (err != cudaSuccess) return err;
    wgrad_tc_kernel<false><<<(unsigned)grid, kThreads, L.total, stream>>>(mg, mi, md, wa);
  }
  return cudaGetLastError();
}

}  // namespace moe_launch
