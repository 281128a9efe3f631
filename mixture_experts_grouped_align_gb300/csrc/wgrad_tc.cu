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
// tcgen05.mma (kind::f16, bf16, M = 128, N = BN, K = 16) with both operands MN-major:
// the producers only copy (cp.async, 16 B), sentinel slots are zero-filled.
//   warp 0     TMEM (two 128 x 256 fp32 accumulators) and the MMA lane;
//   warps 4-7  epilogue: TMEM -> dW rows (fp32), or zeros for an expert with no pair;
//   warps 8-15 producers, one stage (64 token slots) at a time.
// Every mbarrier wait is bounded; a wait that runs out sets MOE_ERR_TIMEOUT and every
// role leaves its loop.  Each tile sums its tokens in one fixed order: repeatable bits.
#include "moe_common.cuh"
#include "cp_async.cuh"
#include "moe_launch.h"
#include "tcgen05.cuh"

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

constexpr int kStageLd = 36;                 // staging row stride (floats): conflict-free
constexpr int kStage = 4 * 32 * kStageLd;    // floats of epilogue staging (4 warps)

struct WLayout {
  int a, b, slot, nslots, bars, total;
};

// Stage: A = 2 MN atom columns (128 n) | B = BN/64 atom columns.
__host__ __device__ inline WLayout wlayout(int BN) {
  WLayout L;
  L.a = 0;
  L.b = 2 * kAtomCol;
  L.slot = L.b + (BN / 64) * kAtomCol;
  int n = (227 * 1024 - 1024 - 256 - 8 * 1024 - kStage * 4) / L.slot;
  L.nslots = n > 4 ? 4 : n;
  L.bars = L.nslots * L.slot;
  // barriers etc. | expert block ranges (8 KB) | epilogue staging (4 x 32 x 36 floats) | slack
  L.total = L.bars + 256 + 8 * 1024 + kStage * 4 + 1024;
  return L;
}

struct WArgs {
  Wgrad g;
  int BN;          // Kin columns per tile (multiple of 64, <= 256)
  int n_tiles;     // N / 128
  int c_tiles;     // Kin / BN
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
// block ranges the thread block built in shared memory).
__device__ __forceinline__ TileInfo tile_info(const WArgs& wa, int64_t t, const int* eb) {
  const Wgrad& a = wa.g;
  TileInfo ti;
  const int64_t per_e = (int64_t)wa.n_tiles * wa.c_tiles;
  ti.e = t / per_e;
  const int rem = (int)(t - ti.e * per_e);
  ti.nt = rem / wa.c_tiles;
  ti.ct = rem - ti.nt * wa.c_tiles;
  ti.slot_beg = (int64_t)eb[2 * ti.e] * a.bm;
  ti.slot_end = (int64_t)eb[2 * ti.e + 1] * a.bm;
  return ti;
}

__global__ void __launch_bounds__(kThreads, 1) wgrad_tc_kernel(WArgs wa) {
  const Wgrad& a = wa.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = wa.BN;
  const WLayout L = wlayout(BN);
  const int S = L.nslots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + 4;
  uint64_t* tfull = empty + 4;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(taddr_s + 1);
  int* eb = reinterpret_cast<int*>(smem + L.bars + 256);  // [E][2]: first, end block

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nblocks = *a.ntpp / a.bm;
  for (int i = tid; i < 2 * a.E; i += kThreads) eb[i] = 0;
  __syncthreads();
  for (int b = tid; b < nblocks; b += kThreads) {  // used blocks: ascending expert ids
    const int e = a.expert_ids[b];
    if (e < 0 || e >= a.E) continue;
    if (b == 0 || a.expert_ids[b - 1] != e) eb[2 * e] = b;
    if (b == nblocks - 1 || a.expert_ids[b + 1] != e) eb[2 * e + 1] = b + 1;
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], kNumProd);  // one completion arrival per producer thread
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
  const uint32_t smem_s = tc::smem_addr(smem);

  if (warp >= 8) {
    // ------------------------------------------------------------------ producers
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
    uint32_t it = 0;
    for (int64_t tt = blockIdx.x; tt < wa.tiles && !*abort_flag; tt += gridDim.x) {
      const TileInfo ti = tile_info(wa, tt, eb);
      const int64_t n0 = (int64_t)ti.nt * kTM, c0 = (int64_t)ti.ct * BN;
      const int64_t nst = (ti.slot_end - ti.slot_beg + kTok - 1) / kTok;
      for (int64_t st = 0; st < nst; ++st) {
        const int slot = it % S;
        if (!tc::mbar_wait(&empty[slot], ((it / S) & 1) ^ 1)) {
          moe::set_status(a.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const uint32_t sl = smem_s + slot * L.slot;
        const int64_t s = ti.slot_beg + st * kTok + t;
        int64_t p = a.P;
        if (s < ti.slot_end) p = a.sorted[s];
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
    }
    cp_async_wait_all();
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
          tc::fence_proxy_async_smem();  // the producers' landed copies, for the tensor core
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
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------------ epilogue
    // TMEM lane = dW row.  Each 32 x 32 chunk goes through shared memory so that the
    // stores to dW are whole 128-byte row segments (4 rows per store instruction).
    const int quarter = warp - kEpiWarp0;
    float* stg = reinterpret_cast<float*>(smem + L.bars + 256 + 8 * 1024) + quarter * 32 * kStageLd;
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

cudaError_t wgrad_tc(const Wgrad& g, cudaStream_t stream) {
  WArgs wa;
  wa.g = g;
  wa.BN = wgrad_tc_tile(g);
  if (wa.BN == 0) return cudaErrorInvalidValue;
  wa.n_tiles = g.N / kTM;
  wa.c_tiles = g.Kin / wa.BN;
  wa.tiles = (int64_t)g.E * wa.n_tiles * wa.c_tiles;
  const WLayout L = wlayout(wa.BN);
  cudaError_t err = cudaFuncSetAttribute(wgrad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  int64_t grid = sm_count_w();
  if (wa.tiles < grid) grid = wa.tiles;
  if (grid <= 0) return cudaSuccess;
  wgrad_tc_kernel<<<(unsigned)grid, kThreads, L.total, stream>>>(wa);
  return cudaGetLastError();
}

}  // namespace moe_launch
