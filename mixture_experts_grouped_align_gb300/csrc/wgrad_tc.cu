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
//     accumulators through swizzled 32 x 32 staging boxes, read back row-contiguous for
//     whole-line stores (marked to leave L2 first).  The experts' slot ranges come from a
//     small kernel (global memory), which leaves shared memory to four 48 KB stages.
//     Launched in clusters of C CTAs that take the C N tiles of one (expert, Kin tile): the
//     input boxes, the same for all of them, are loaded once per cluster and multicast
//     (each CTA issues its share), and every CTA's MMA commit frees the stage in all of
//     them, which halves (C = 4) the operand bytes the L2 serves per output.
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
constexpr int kBox = 32 * 128;               // slot feed: one 32 x 32 fp32 staging box (bytes)
constexpr int kSlotEpiWarps = 8;

struct WLayout {
  int a, b, slot, nslots, stg, bars, eb, total;
};

// Stages (A = 2 MN atom columns (128 n) | B = BN/64 atom columns) | epilogue staging (slot
// feed: one box per epilogue warp) | barriers | gather feed: expert block ranges (8 KB).
// Offsets from a 1024-byte aligned base.
__host__ __device__ inline WLayout wlayout(int BN, bool slot_feed) {
  WLayout L;
  L.a = 0;
  L.b = 2 * kAtomCol;
  L.slot = L.b + (BN / 64) * kAtomCol;
  const int staging = slot_feed ? kSlotEpiWarps * kBox : kStage * 4;
  const int ranges = slot_feed ? 0 : 8 * 1024;
  int n = (227 * 1024 - 1024 - 256 - ranges - staging) / L.slot;
  L.nslots = n > kMaxStages ? kMaxStages : n;
  L.stg = L.nslots * L.slot;
  L.bars = L.stg + staging;
  L.eb = L.bars + 256;
  L.total = L.eb + ranges + 1024;
  return L;
}

struct WArgs {
  Wgrad g;
  int BN;          // Kin columns per tile (multiple of 64, <= 256)
  int n_tiles;     // N / 128
  int c_tiles;     // Kin / BN
  int groups;      // n_tiles / C: the cluster's C CTAs take N tiles C g .. C g + C - 1
  int nt_fast;     // 1: N tile groups vary fastest within an expert (every grad column live at once)
  int64_t tiles;   // E * groups * c_tiles (one per cluster)
};

// Byte offset of (token t, 16-byte chunk c of a row of 64 MN elements) in an atom column.
__device__ __forceinline__ uint32_t mn_offset(int t, int c) {
  return (uint32_t)((t >> 3) * kAtom + (t & 7) * 128 + ((c ^ (t & 7)) << 4));
}

// 16-byte global store with an L2 cache policy.
__device__ __forceinline__ void st_global_v4_hint(float* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                                  uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d),
               "l"(policy)
               : "memory");
}

struct TileInfo {
  int64_t e;
  int nt, ct;
  int64_t slot_beg, slot_end;  // the expert's token slots
};

// Cluster tile t -> expert, this CTA's N tile, Kin tile and the expert's slot range (from
// the per-expert block ranges the thread block built in shared memory).  Within an expert
// the tile index whose operand is narrower over all tiles varies fastest, so that the
// tiles running at once share the wider operand's columns and their rows stay small in L2.
__device__ __forceinline__ TileInfo tile_info(const WArgs& wa, int64_t t, const int* eb, int C, int rank) {
  const Wgrad& a = wa.g;
  TileInfo ti;
  const int64_t per_e = (int64_t)wa.groups * wa.c_tiles;
  ti.e = t / per_e;
  const int rem = (int)(t - ti.e * per_e);
  int grp;
  if (wa.nt_fast) {
    ti.ct = rem / wa.groups;
    grp = rem - ti.ct * wa.groups;
  } else {
    grp = rem / wa.c_tiles;
    ti.ct = rem - grp * wa.c_tiles;
  }
  ti.nt = grp * C + rank;
  ti.slot_beg = (int64_t)eb[2 * ti.e] * a.bm;
  ti.slot_end = (int64_t)eb[2 * ti.e + 1] * a.bm;
  return ti;
}

template <bool SLOT, int C>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_i, WArgs wa) {
  const Wgrad& a = wa.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  static_assert(C == 1 || SLOT, "clusters share the slot feed's boxes");
  const int BN = wa.BN;
  const WLayout L = wlayout(BN, SLOT);
  // this CTA's cluster (C consecutive blocks) and its rank in it; the loops walk cluster tiles
  const int rank = C > 1 ? (int)tc::cluster_ctarank() : 0;
  const int64_t cid = blockIdx.x / C, ncl = gridDim.x / C;
  const uint16_t cmask = (uint16_t)((1u << C) - 1u);
  const int S = L.nslots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_s + 1);
  // [E][2]: first, end block of every expert (slot feed: computed before the launch)
  int* eb = SLOT ? a.ranges : reinterpret_cast<int*>(smem + L.eb);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (!SLOT) {
    const int nblocks = *a.ntpp / a.bm;
    for (int i = tid; i < 2 * a.E; i += kThreads) eb[i] = 0;
    __syncthreads();
    for (int b = tid; b < nblocks; b += kThreads) {  // used blocks: ascending expert ids
      const int e = a.expert_ids[b];
      if (e < 0 || e >= a.E) continue;
      if (b == 0 || a.expert_ids[b - 1] != e) eb[2 * e] = b;
      if (b == nblocks - 1 || a.expert_ids[b + 1] != e) eb[2 * e + 1] = b + 1;
    }
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      // gather feed: one completion arrival per producer thread; slot feed: the TMA thread
      tc::mbar_init(&full[s], SLOT ? 1 : kNumProd);
      tc::mbar_init(&empty[s], C);  // the MMA commit of every CTA of the cluster
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
  if (C > 1) tc::cluster_sync();  // every CTA's barriers exist before a peer signals them
  tc::tc_fence_after();
  const uint32_t taddr = *taddr_s;
  const uint32_t smem_s = tc::smem_addr(smem);
  // the limit of every wait (a caller's short limit only in the stalled self-test)
  const uint64_t wb = a.wait_ns > 0 ? (uint64_t)a.wait_ns : tc::kWaitNs;

  if (!SLOT && warp >= 8 && !a.stall) {
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
        ti = tile_info(wa, tt, eb, 1, 0);
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
      if (!tc::mbar_wait(&empty[slot], ((it / S) & 1) ^ 1, wb)) {
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
  } else if (SLOT && warp == 1 && !a.stall) {
    // ------------------------------------------------------------------ slot feed (TMA)
    if (lane == 0) {
      tma::prefetch_map(&tm_g);
      tma::prefetch_map(&tm_i);
      const uint32_t stage_tx = (uint32_t)(2 + BN / 64) * kAtomCol;
      // the operand rows are read again by the expert's other tiles: kept in L2 over the dW
      // lines, which the stores mark to leave first
      const uint64_t keep = tma::policy_evict_last();
      uint32_t it = 0;
      for (int64_t tt = cid; tt < wa.tiles && !*abort_flag; tt += ncl) {
        const TileInfo ti = tile_info(wa, tt, eb, C, rank);
        const int64_t nst = (ti.slot_end - ti.slot_beg) / kTok;  // block_m is a multiple of kTok
        const int32_t xg = (int32_t)((int64_t)ti.nt * kTM * 2), xi = (int32_t)((int64_t)ti.ct * BN * 2);
        // the first stages of this CTA's next tile, into L2 while this one streams: the ring
        // then starts the next tile on L2 hits instead of HBM round trips
        if (tt + ncl < wa.tiles) {
          const TileInfo tn = tile_info(wa, tt + ncl, eb, C, rank);
          const int64_t pst = (tn.slot_end - tn.slot_beg) / kTok;
          const int32_t pg = (int32_t)((int64_t)tn.nt * kTM * 2), pi = (int32_t)((int64_t)tn.ct * BN * 2);
          for (int64_t st = 0; st < pst && st < kMaxStages; ++st) {
            const int32_t y = (int32_t)(tn.slot_beg + st * kTok);
            tma::prefetch_2d_l2(&tm_g, pg, y);
            tma::prefetch_2d_l2(&tm_g, pg + 128, y);
            for (int j = rank; j < BN / 64; j += C) tma::prefetch_2d_l2(&tm_i, pi + 128 * j, y);
          }
        }
        bool ok = true;
        for (int64_t st = 0; st < nst; ++st) {
          const int slot = it % S;
          if (!tc::mbar_wait(&empty[slot], ((it / S) & 1) ^ 1, wb)) {
            ok = false;
            break;
          }
          const uint32_t sl = smem_s + slot * L.slot;
          const int32_t y = (int32_t)(ti.slot_beg + st * kTok);
          tma::mbar_arrive_expect_tx(&full[slot], stage_tx);
          // 64 slots x 64 bf16 per box, 128-byte swizzled: one MN atom column
          tma::load_2d_hint(sl + L.a, &tm_g, xg, y, &full[slot], keep);
          tma::load_2d_hint(sl + L.a + kAtomCol, &tm_g, xg + 128, y, &full[slot], keep);
          // input boxes: this CTA's share, into every CTA of the cluster
          for (int j = rank; j < BN / 64; j += C) {
            if (C > 1)
              tma::load_2d_multicast_hint(sl + L.b + j * kAtomCol, &tm_i, xi + 128 * j, y, &full[slot], cmask, keep);
            else
              tma::load_2d_hint(sl + L.b + j * kAtomCol, &tm_i, xi + 128 * j, y, &full[slot], keep);
          }
          ++it;
        }
        if (!ok) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
      }
      // Leaving early: the loads already issued still land in this block's shared memory,
      // so wait for the last armed phase of every slot before exiting.  In a cluster, the
      // normal end waits instead until every CTA's MMAs have released this CTA's last
      // stages, so that no peer's commit arrives after this CTA is gone.
      if (*abort_flag) {
        for (uint32_t j = it > (uint32_t)S ? it - S : 0; j < it; ++j)
          if (!tc::mbar_wait(&full[j % S], (j / S) & 1, wb)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
      } else if (C > 1) {
        for (uint32_t j = it > (uint32_t)S ? it - S : 0; j < it; ++j)
          if (!tc::mbar_wait(&empty[j % S], (j / S) & 1, wb)) moe::set_status(a.status, MOE_ERR_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp == 0 && !a.stall) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(kTM, BN, 1) | (1u << 15) | (1u << 16);
      uint32_t it = 0, acc_it = 0;
      for (int64_t tt = cid; tt < wa.tiles && !*abort_flag; tt += ncl) {
        const TileInfo ti = tile_info(wa, tt, eb, C, rank);
        const int64_t nst = (ti.slot_end - ti.slot_beg + kTok - 1) / kTok;
        if (nst == 0) continue;  // the epilogue writes zeros itself
        const uint32_t acc = acc_it & 1;
        if (!tc::mbar_wait(&tempty[acc], ((acc_it >> 1) & 1) ^ 1, wb)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d_tmem = taddr + acc * 256;
        bool ok = true;
        for (int64_t st = 0; st < nst; ++st) {
          const int slot = it % S;
          if (!tc::mbar_wait(&full[slot], (it / S) & 1, wb)) {
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
          if (C > 1)
            tc::mma_commit_multicast(&empty[slot], cmask);  // the stage is free in every CTA
          else
            tc::mma_commit(&empty[slot]);
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
  } else if (!SLOT && warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------------ epilogue (gather feed)
    // TMEM lane = dW row.  Each 32 x 32 chunk goes through shared memory so that the
    // stores to dW are whole 128-byte row segments (4 rows per store instruction).
    const int quarter = warp - kEpiWarp0;
    float* stg = reinterpret_cast<float*>(smem + L.stg) + quarter * 32 * kStageLd;
    const int rr = lane >> 3, cc = (lane & 7) * 4;  // store phase: row rr + 4i, columns cc..cc+3
    uint32_t acc_it = 0;
    for (int64_t tt = blockIdx.x; tt < wa.tiles && !*abort_flag; tt += gridDim.x) {
      const TileInfo ti = tile_info(wa, tt, eb, 1, 0);
      float* tile = a.dW + ((ti.e * a.N) + (int64_t)ti.nt * kTM + quarter * 32) * (int64_t)a.Kin +
                    (int64_t)ti.ct * BN;
      if (ti.slot_end == ti.slot_beg) {  // an expert with no pair: dW[e] = 0
        for (int r = 0; r < 32; ++r)
          for (int c = lane * 4; c < BN; c += 128)
            *reinterpret_cast<float4*>(tile + (int64_t)r * a.Kin + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const uint32_t acc = acc_it & 1;
      if (!tc::mbar_wait(&tfull[acc], (acc_it >> 1) & 1, wb)) {
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
    // shared memory -> read back four rows at a time, each row's 128 bytes by eight lanes,
    // and stored as whole lines.
    const int ew = warp - kEpiWarp0, quarter = warp & 3, half = ew >> 2;
    const int cols = BN / 2;
    const uint32_t box = smem_s + L.stg + ew * kBox;
    const uint64_t stream_out = tma::policy_evict_first();  // dW is not read again here
    const int cc = lane & 7, r0 = lane >> 3;                 // store phase: rows r0 + 4 i, chunk cc
    uint32_t acc_it = 0;
    for (int64_t tt = cid; tt < wa.tiles && !*abort_flag; tt += ncl) {
      const TileInfo ti = tile_info(wa, tt, eb, C, rank);
      float* tile = a.dW + (ti.e * a.N + (int64_t)ti.nt * kTM + quarter * 32) * (int64_t)a.Kin +
                    (int64_t)ti.ct * BN + half * cols;
      if (ti.slot_end == ti.slot_beg) {  // an expert with no pair: dW[e] = 0
        for (int c = 0; c < cols; c += 32)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_global_v4_hint(tile + (int64_t)(r0 + 4 * i) * a.Kin + c + 4 * cc, 0u, 0u, 0u, 0u, stream_out);
        continue;
      }
      const uint32_t acc = acc_it & 1;
      if (!tc::mbar_wait(&tfull[acc], (acc_it >> 1) & 1, wb)) {
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
#pragma unroll
        for (int q = 0; q < 8; ++q)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(box + lane * 128 + ((q ^ (lane & 7)) << 4)),
                       "r"(v[4 * q]), "r"(v[4 * q + 1]), "r"(v[4 * q + 2]), "r"(v[4 * q + 3])
                       : "memory");
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = r0 + 4 * i;
          uint32_t w0, w1, w2, w3;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                       : "r"(box + r * 128 + ((cc ^ (r & 7)) << 4))
                       : "memory");
          st_global_v4_hint(tile + (int64_t)r * a.Kin + c + 4 * cc, w0, w1, w2, w3, stream_out);
        }
        __syncwarp();
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[acc]);
      ++acc_it;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (C > 1) tc::cluster_sync();  // no CTA leaves while a peer may still signal it
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(taddr, kTmemCols);
  }
}

int sm_count_w() { return moe_launch::sm_count_current(); }

// ranges[e] = (first, end) alignment block of expert e, (0, 0) for an expert with no block:
// one block of threads, the same rule the gather-feed kernel applies in shared memory.
__global__ void expert_ranges_kernel(const int32_t* __restrict__ expert_ids, const int32_t* __restrict__ ntpp, int bm,
                                     int E, int32_t* __restrict__ ranges) {
  const int nblocks = *ntpp / bm;
  for (int i = threadIdx.x; i < 2 * E; i += blockDim.x) ranges[i] = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < nblocks; b += blockDim.x) {  // used blocks: ascending expert ids
    const int e = expert_ids[b];
    if (e < 0 || e >= E) continue;
    if (b == 0 || expert_ids[b - 1] != e) ranges[2 * e] = b;
    if (b == nblocks - 1 || expert_ids[b + 1] != e) ranges[2 * e + 1] = b + 1;
  }
}

cudaError_t expert_ranges(const Wgrad& g, cudaStream_t stream) {
  if (g.ranges == nullptr) return cudaErrorInvalidValue;
  expert_ranges_kernel<<<1, 1024, 0, stream>>>(g.expert_ids, g.ntpp, g.bm, g.E, g.ranges);
  return cudaGetLastError();
}

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
  // (slots) are 32-bit
  return wgrad_tc_tile(g) > 0 && g.bm % kTok == 0 && g.cap < ((int64_t)1 << 31);
}

// The slot-fed kernel in clusters of C CTAs: persistent, as many whole clusters as fit on
// the GPU at once (at most one per cluster tile).  *no_fit when no cluster of C fits.
template <int C>
cudaError_t launch_slot(const CUtensorMap& mg, const CUtensorMap& mi, WArgs wa, int smem,
                        cudaStream_t stream, bool* no_fit) {
  auto kern = wgrad_tc_kernel<true, C>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  wa.groups = wa.n_tiles / C;
  wa.tiles = (int64_t)wa.g.E * wa.groups * wa.c_tiles;
  int64_t nclusters = sm_count_w() / C;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  if (C > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(nclusters * C));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      *no_fit = true;
      return cudaSuccess;
    }
    nclusters = n;
  }
  if (wa.tiles < nclusters) nclusters = wa.tiles;
  if (nclusters <= 0) return cudaSuccess;
  cfg.gridDim = dim3((unsigned)(nclusters * C));
  return cudaLaunchKernelEx(&cfg, kern, mg, mi, wa);
}

cudaError_t wgrad_tc(const Wgrad& g, cudaStream_t stream) {
  WArgs wa;
  wa.g = g;
  wa.BN = wgrad_tc_tile(g);
  if (wa.BN == 0) return cudaErrorInvalidValue;
  wa.n_tiles = g.N / kTM;
  wa.c_tiles = g.Kin / wa.BN;
  wa.groups = wa.n_tiles;
  wa.nt_fast = g.N <= g.Kin ? 1 : 0;
  wa.tiles = (int64_t)g.E * wa.n_tiles * wa.c_tiles;
  const bool slot = g.grad_s != nullptr && g.input_s != nullptr;
  if (slot && !wgrad_tc_slot_feed(g)) return cudaErrorInvalidValue;
  const WLayout L = wlayout(wa.BN, slot);
  CUtensorMap mg{}, mi{};
  if (slot) {
    // slot-ordered rows: boxes of 64 slots x 128 bytes, 128-byte swizzle (one MN atom column)
    if (!tma::encode_2d_u8(&mg, g.grad_s, (uint64_t)g.N * 2, (uint64_t)g.cap, (uint64_t)g.N * 2, 128, kTok, true) ||
        !tma::encode_2d_u8(&mi, g.input_s, (uint64_t)g.Kin * 2, (uint64_t)g.cap, (uint64_t)g.Kin * 2, 128, kTok,
                           true))
      return cudaErrorInvalidValue;
    cudaError_t rerr = expert_ranges(g, stream);
    if (rerr != cudaSuccess) return rerr;
    // the largest cluster that divides the N tiles and fits
    bool no_fit = false;
    if (wa.n_tiles % 4 == 0) {
      cudaError_t err = launch_slot<4>(mg, mi, wa, L.total, stream, &no_fit);
      if (err != cudaSuccess || !no_fit) return err == cudaSuccess ? cudaGetLastError() : err;
    }
    no_fit = false;
    if (wa.n_tiles % 2 == 0) {
      cudaError_t err = launch_slot<2>(mg, mi, wa, L.total, stream, &no_fit);
      if (err != cudaSuccess || !no_fit) return err == cudaSuccess ? cudaGetLastError() : err;
    }
    cudaError_t err = launch_slot<1>(mg, mi, wa, L.total, stream, &no_fit);
    return err == cudaSuccess ? cudaGetLastError() : err;
  }
  int64_t grid = sm_count_w();
  if (wa.tiles < grid) grid = wa.tiles;
  if (grid <= 0) return cudaSuccess;
  cudaError_t err =
      cudaFuncSetAttribute(wgrad_tc_kernel<false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  wgrad_tc_kernel<false, 1><<<(unsigned)grid, kThreads, L.total, stream>>>(mg, mi, wa);
  return cudaGetLastError();
}

}  // namespace moe_launch
