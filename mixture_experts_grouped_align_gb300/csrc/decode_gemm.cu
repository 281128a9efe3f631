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
#include "moe_launch.h"

namespace {

using namespace moe_launch;

constexpr int kWarps = 4;   // warps per block, each a quarter of K
constexpr int kTok = 8;     // tokens per tile (MMA N)
constexpr int kRows = 16;   // output rows per block (MMA M)
constexpr unsigned kFull = 0xffffffffu;

// Activation rows in shared memory use a stride of S 16-bit elements with S = 32 mod 64,
// so that the 8-lane phases of a 16-byte shared load (two token rows) hit disjoint banks.
__host__ __device__ inline int xs_stride(int Kin) { return (Kin % 64 == 32) ? Kin : Kin + 32; }

struct Smem {
  int wsc, xs, xsc, red, total;  // byte offsets
};

__host__ __device__ inline Smem smem_layout(int nmat, int Kin, bool act_scaled) {
  const int nkb = Kin / 32;
  Smem s;
  int off = 0;
  s.wsc = off;  off += ((nmat * kRows * nkb + 15) / 16) * 16;          // weight scale bytes
  s.xs = off;   off += kTok * xs_stride(Kin) * 2;                       // activations, 16-bit
  s.xsc = off;  off += act_scaled ? ((kTok * nkb + 15) / 16) * 16 : 0;  // activation scales
  s.red = off;  off += kWarps * nmat * 4 * 32 * 4;                      // cross-warp partials
  s.total = off;
  return s;
}

template <int WF>
struct Fmt;
template <>
struct Fmt<WF_MXFP4> {
  using W = uint32_t;  // 8 codes of one row: physical K 8q..8q+7 of a 32-block
  static constexpr int kUnroll = 8;
  static __device__ __forceinline__ W load(const uint8_t* row, int kb, int q) {
    return moe::ldg_nc_u32(row + kb * 16 + q * 4);
  }
  // half 0: elements 0..3 of the lane's 8 -> (pair 0,1), (pair 2,3); half 1: elements 4..7
  static __device__ __forceinline__ void pairs(W w, int half, uint32_t& p0, uint32_t& p1) {
    p0 = moe::e2m1x2_to_f16x2((w >> (16 * half)) & 0xffu);
    p1 = moe::e2m1x2_to_f16x2((w >> (16 * half + 8)) & 0xffu);
  }
};
template <>
struct Fmt<WF_MXFP8> {
  using W = uint2;
  static constexpr int kUnroll = 4;
  static __device__ __forceinline__ W load(const uint8_t* row, int kb, int q) {
    return moe::ldg_nc_u64(row + kb * 32 + q * 8);
  }
  static __device__ __forceinline__ void pairs(W w, int half, uint32_t& p0, uint32_t& p1) {
    const uint32_t v = half ? w.y : w.x;
    p0 = moe::e4m3x2_to_f16x2(v & 0xffffu);
    p1 = moe::e4m3x2_to_f16x2(v >> 16);
  }
};
template <>
struct Fmt<WF_BF16> {
  using W = uint4;
  static constexpr int kUnroll = 4;
  static __device__ __forceinline__ W load(const uint8_t* row, int kb, int q) {
    return moe::ldg_nc_u128(row + kb * 64 + q * 16);
  }
  static __device__ __forceinline__ void pairs(W w, int half, uint32_t& p0, uint32_t& p1) {
    p0 = half ? w.z : w.x;
    p1 = half ? w.w : w.y;
  }
};

template <int WF>
__host__ __device__ inline int64_t wrow_bytes(int Kin) {
  return WF == WF_MXFP4 ? Kin / 2 : (WF == WF_MXFP8 ? Kin : (int64_t)Kin * 2);
}

template <int WF, int EPI>
__global__ void __launch_bounds__(kWarps * 32) decode_gemm_kernel(GroupedGemm a) {
  constexpr int NMAT = (EPI == EPI_SWIGLU) ? 2 : 1;
  constexpr bool MX = (WF != WF_BF16);
  constexpr bool ACT_SCALED = (WF == WF_MXFP8);
  using F = Fmt<WF>;
  using W = typename F::W;
  constexpr int U = F::kUnroll;

  extern __shared__ __align__(16) uint8_t smem[];
  const Smem L = smem_layout(NMAT, a.Kin, ACT_SCALED);
  uint8_t* wsc = smem + L.wsc;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs);
  uint8_t* xsc = smem + L.xsc;
  float* red = reinterpret_cast<float*>(smem + L.red);

  const int row_tiles = a.Nout / kRows;
  const int64_t blk = blockIdx.x / row_tiles;
  const int rt = blockIdx.x - (int)(blk * row_tiles);
  // sentinel / unused block slots leave before touching weights, scales or bias
  if (blk * a.bm >= *a.ntpp) return;
  const int64_t e = a.expert_ids[blk];
  if (e < 0) return;
  if (e >= a.E) {
    if (threadIdx.x == 0 && blockIdx.x % row_tiles == 0) moe::set_status(a.status, MOE_ERR_INVALID_EXPERT);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int Kin = a.Kin, nkb = Kin / 32, S = xs_stride(Kin);
  const int kb0 = warp * nkb / kWarps, kb1 = (warp + 1) * nkb / kWarps, nb = kb1 - kb0;
  const int64_t rb = wrow_bytes<WF>(Kin);
  const uint8_t* wbase = static_cast<const uint8_t*>(a.w);

  auto wrow = [&](int m, int i) -> int64_t {  // matrix m (0 gate/main, 1 up), tile row i
    return e * a.Nw + (m ? a.Nout : 0) + (int64_t)rt * kRows + i;
  };
  if (MX) {  // this warp's K slice of the block's weight scales
    for (int idx = lane; idx < NMAT * kRows * nb; idx += 32) {
      const int r = idx / nb, c = idx - r * nb;
      wsc[r * nkb + kb0 + c] = a.w_scale[wrow(r / kRows, r % kRows) * nkb + kb0 + c];
    }
  }
  const uint8_t* rowp[NMAT][2];
#pragma unroll
  for (int m = 0; m < NMAT; ++m) {
    rowp[m][0] = wbase + wrow(m, g) * rb;
    rowp[m][1] = wbase + wrow(m, g + 8) * rb;
  }

  const int64_t slot0 = blk * a.bm;
  bool bad = false;
  for (int st = 0; st < a.bm; st += kTok) {
    int pr = (int)a.P;
    if (lane < kTok && st + lane < a.bm) pr = a.sorted[slot0 + st + lane];
    int ptok[kTok];
#pragma unroll
    for (int j = 0; j < kTok; ++j) ptok[j] = __shfl_sync(kFull, pr, j);
    if (ptok[0] >= a.P) break;  // uniform over the block: all warps read the same slots

    // stage this warp's K slice of the tile's activations as 16-bit values
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kTok; ++j) {
      const bool valid = ptok[j] < a.P;
      const int64_t arow = a.act_per_pair ? (int64_t)ptok[j] : (int64_t)(ptok[j] / a.k);
      uint16_t* dst = xs + j * S + kb0 * 32;
      for (int c = lane; c < nb * 4; c += 32) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (valid) {
          if (WF == WF_MXFP8) {
            const uint2 raw = *reinterpret_cast<const uint2*>(
                static_cast<const uint8_t*>(a.act) + arow * Kin + kb0 * 32 + c * 8);
            v.x = moe::e4m3x2_to_f16x2(raw.x & 0xffffu);
            v.y = moe::e4m3x2_to_f16x2(raw.x >> 16);
            v.z = moe::e4m3x2_to_f16x2(raw.y & 0xffffu);
            v.w = moe::e4m3x2_to_f16x2(raw.y >> 16);
          } else {
            const uint4 raw = *reinterpret_cast<const uint4*>(
                static_cast<const uint16_t*>(a.act) + arow * Kin + kb0 * 32 + c * 8);
            if (WF == WF_BF16) {  // bf16 MMA operand
              if (a.act_fmt == ACT_F16) {
                v.x = moe::f16x2_to_bf16x2(raw.x);
                v.y = moe::f16x2_to_bf16x2(raw.y);
                v.z = moe::f16x2_to_bf16x2(raw.z);
                v.w = moe::f16x2_to_bf16x2(raw.w);
              } else {
                v = raw;
              }
            } else {              // f16 MMA operand
              if (a.act_fmt == ACT_F16) {
                v = raw;
              } else {
                v.x = moe::bf16x2_to_f16x2(raw.x, &bad);
                v.y = moe::bf16x2_to_f16x2(raw.y, &bad);
                v.z = moe::bf16x2_to_f16x2(raw.z, &bad);
                v.w = moe::bf16x2_to_f16x2(raw.w, &bad);
              }
            }
          }
        }
        *reinterpret_cast<uint4*>(dst + c * 8) = v;
      }
      if (ACT_SCALED) {
        for (int c = lane; c < nb; c += 32)
          xsc[j * nkb + kb0 + c] = valid ? a.act_scale[arow * nkb + kb0 + c] : (uint8_t)127;
      }
    }
    __syncwarp();

    float acc[NMAT][4];
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;

    for (int kb = kb0; kb < kb1; kb += U) {
      W wr[U][NMAT][2];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (kb + u < kb1) {
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            wr[u][m][0] = F::load(rowp[m][0], kb + u, q);
            wr[u][m][1] = F::load(rowp[m][1], kb + u, q);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int kk = kb + u;
        if (kk < kb1) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + g * S + kk * 32 + q * 8);
          float xsc0 = 1.f, xsc1 = 1.f;
          if (ACT_SCALED) {
            xsc0 = moe::e8m0_to_f32(xsc[(2 * q) * nkb + kk]);
            xsc1 = moe::e8m0_to_f32(xsc[(2 * q + 1) * nkb + kk]);
          }
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            uint32_t A[4];
            if (MX) {
              const float zero[4] = {0.f, 0.f, 0.f, 0.f};
              float t[4];
              F::pairs(wr[u][m][0], 0, A[0], A[2]);
              F::pairs(wr[u][m][1], 0, A[1], A[3]);
              moe::mma_f16(t, A, xv.x, xv.y, zero);
              F::pairs(wr[u][m][0], 1, A[0], A[2]);
              F::pairs(wr[u][m][1], 1, A[1], A[3]);
              moe::mma_f16(t, A, xv.z, xv.w, t);
              const float s0 = moe::e8m0_to_f32(wsc[(m * kRows + g) * nkb + kk]);
              const float s1 = moe::e8m0_to_f32(wsc[(m * kRows + g + 8) * nkb + kk]);
              if (ACT_SCALED) {
                acc[m][0] = fmaf(t[0] * s0, xsc0, acc[m][0]);
                acc[m][1] = fmaf(t[1] * s0, xsc1, acc[m][1]);
                acc[m][2] = fmaf(t[2] * s1, xsc0, acc[m][2]);
                acc[m][3] = fmaf(t[3] * s1, xsc1, acc[m][3]);
              } else {
                acc[m][0] = fmaf(t[0], s0, acc[m][0]);
                acc[m][1] = fmaf(t[1], s0, acc[m][1]);
                acc[m][2] = fmaf(t[2], s1, acc[m][2]);
                acc[m][3] = fmaf(t[3], s1, acc[m][3]);
              }
            } else {
              F::pairs(wr[u][m][0], 0, A[0], A[2]);
              F::pairs(wr[u][m][1], 0, A[1], A[3]);
              moe::mma_bf16(acc[m], A, xv.x, xv.y, acc[m]);
              F::pairs(wr[u][m][0], 1, A[0], A[2]);
              F::pairs(wr[u][m][1], 1, A[1], A[3]);
              moe::mma_bf16(acc[m], A, xv.z, xv.w, acc[m]);
            }
          }
        }
      }
    }

    // fixed-order sum over the four K quarters, then the epilogue (warp 0)
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[((warp * NMAT + m) * 4 + i) * 32 + lane] = acc[m][i];
    __syncthreads();
    if (warp == 0) {
      float v[NMAT][4];
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float s = red[((0 * NMAT + m) * 4 + i) * 32 + lane];
#pragma unroll
          for (int w = 1; w < kWarps; ++w) s += red[((w * NMAT + m) * 4 + i) * 32 + lane];
          v[m][i] = s;
        }
      const int pc[2] = {__shfl_sync(kFull, pr, 2 * q), __shfl_sync(kFull, pr, 2 * q + 1)};
      const uint16_t* bias = static_cast<const uint16_t*>(a.bias);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int p = pc[i & 1];
        if (p >= a.P) continue;
        const int n = rt * kRows + g + ((i >> 1) << 3);
        if (EPI == EPI_SWIGLU) {
          float gt = v[0][i], up = v[NMAT - 1][i];
          if (bias) {
            gt += moe::bf16_bits_to_f32(bias[e * a.Nw + n]);
            up += moe::bf16_bits_to_f32(bias[e * a.Nw + a.Nout + n]);
          }
          // h is kept as float16 (11-bit significand); an overflow is reported
          const __half hv = __float2half_rn(moe::silu(gt) * up);
          if (__hisinf(hv) || __hisnan(hv)) bad = true;
          static_cast<__half*>(a.out)[(int64_t)p * a.Nout + n] = hv;
        } else if (EPI == EPI_WEIGHTED_F32) {
          float o = v[0][i];
          if (bias) o += moe::bf16_bits_to_f32(bias[e * a.Nw + n]);
          static_cast<float*>(a.out)[(int64_t)p * a.Nout + n] = o * a.topk_w[p];
        } else {
          float o = v[0][i];
          if (bias) o += moe::bf16_bits_to_f32(bias[e * a.Nw + n]);
          static_cast<uint16_t*>(a.out)[(int64_t)p * a.Nout + n] = moe::f32_to_bf16_bits(o);
        }
      }
    }
    __syncthreads();
  }
  if (bad) moe::set_status(a.status, MOE_ERR_RANGE);
}

template <int WF, int EPI>
cudaError_t launch_t(const GroupedGemm& g, cudaStream_t stream) {
  const Smem L = smem_layout(EPI == EPI_SWIGLU ? 2 : 1, g.Kin, WF == WF_MXFP8);
  cudaError_t err = cudaFuncSetAttribute(decode_gemm_kernel<WF, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  const int64_t grid = g.grid_blocks * (g.Nout / kRows);
  if (grid <= 0) return cudaSuccess;
  decode_gemm_kernel<WF, EPI><<<(unsigned)grid, kWarps * 32, L.total, stream>>>(g);
  return cudaGetLastError();
}

}  // namespace

namespace moe_launch {

size_t decode_gemm_smem_bytes(const GroupedGemm& g) {
  return smem_layout(g.epi == EPI_SWIGLU ? 2 : 1, g.Kin, g.wfmt == WF_MXFP8).total;
}

cudaError_t decode_gemm(const GroupedGemm& g, cudaStream_t stream) {
#define MOE_CASE(WF, EP) \
  if (g.wfmt == WF && g.epi == EP) return launch_t<WF, EP>(g, stream);
  MOE_CASE(WF_MXFP4, EPI_SWIGLU)
  MOE_CASE(WF_MXFP4, EPI_WEIGHTED_F32)
  MOE_CASE(WF_MXFP4, EPI_PLAIN_BF16)
  MOE_CASE(WF_BF16, EPI_SWIGLU)
  MOE_CASE(WF_BF16, EPI_WEIGHTED_F32)
  MOE_CASE(WF_BF16, EPI_PLAIN_BF16)
  MOE_CASE(WF_MXFP8, EPI_SWIGLU)
  MOE_CASE(WF_MXFP8, EPI_WEIGHTED_F32)
  MOE_CASE(WF_MXFP8, EPI_PLAIN_BF16)
#undef MOE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe_launch
