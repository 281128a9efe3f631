// Internal launchers of the MoE kernels (host side; not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe_launch {

// Streaming multiprocessors of the current device (cached per device index; 1 if the
// query fails).
int sm_count_current();

// ---- route + align (route_align.cu)
size_t align_smem_bytes(int E);
cudaError_t align(const float* logits, int32_t* ids, float* w, int64_t T, int k, int E, int bm,
                  int32_t* sorted, int64_t cap, int32_t* expert_ids, int32_t* ntpp,
                  int32_t* expert_offsets, int32_t* status, cudaStream_t stream);

// ---- pad rows (elementwise.cu)
cudaError_t pad_rows(const void* src, void* dst, int64_t rows, int64_t rows_pad, int64_t row_bytes,
                     cudaStream_t stream);
cudaError_t zero_f32(float* p, int64_t n, cudaStream_t stream);
cudaError_t combine(const float* o, int64_t T_real, int k, int K, void* y, cudaStream_t stream);
cudaError_t bf16_to_f16(const void* x, void* y, int64_t n, int32_t* status, cudaStream_t stream);
// MXFP8 quantisation of fp32 rows ([rows, cols], cols % 32 == 0) -> E4M3 codes [rows, cols]
// and E8M0 scales [rows, cols / 32] (mx_quant.cuh).
cudaError_t mx_quantize(const float* x, int64_t rows, int cols, uint8_t* codes, uint8_t* scales,
                        cudaStream_t stream);
// Token rows of bf16 x gathered into alignment-slot order as f16 ([slots, K]).
cudaError_t gather_rows_f16(const void* x, const int32_t* sorted, const int32_t* ntpp, int64_t P, int k,
                            int64_t K, int64_t slots, void* y, int32_t* status, cudaStream_t stream);
// Rows of row_bytes (a multiple of 16) copied into alignment-slot order: y[s] = src[p / div]
// for slot s < num_tokens_post_padded holding pair p < P, zeros for a sentinel slot.
cudaError_t gather_slot_rows(const void* src, int64_t row_bytes, const int32_t* sorted, const int32_t* ntpp,
                             int64_t P, int div, int64_t slots, void* y, cudaStream_t stream);

// ---- grouped GEMMs on the weight-streaming (decode) path (decode_gemm.cu)
enum WFmt { WF_BF16 = 0, WF_MXFP4 = 1, WF_MXFP8 = 2 };
// SwiGLU and relu^2 write h (f16 for MX weights, bf16 for bf16 weights); relu^2 reads one
// weight matrix (Nw = Nout), SwiGLU two (gate rows then up rows, Nw = 2 * Nout).
enum Epi { EPI_SWIGLU = 0, EPI_WEIGHTED_F32 = 1, EPI_PLAIN_BF16 = 2, EPI_RELU2 = 3 };
enum ActFmt { ACT_BF16 = 0, ACT_F16 = 1 };

struct GroupedGemm {
  int wfmt;                 // WFmt
  int epi;                  // Epi
  const void* w;            // [E, Nw, Kin] in wfmt
  const uint8_t* w_scale;   // [E, Nw, Kin/32] E8M0 (mx formats)
  const void* bias;         // [E, Nw] bf16 or null
  const void* act;          // rows [*, Kin]: bf16, f16 (act_fmt) or E4M3 (wfmt mxfp8)
  int act_fmt;              // ActFmt of 16-bit activations
  const uint8_t* act_scale; // [*, Kin/32] (mxfp8)
  int act_per_pair;         // act row = p (1) or p / k (0)
  int act_by_slot;          // 1: act row = alignment slot (rows already in sorted order)
  int out_by_slot;          // 1: output row = alignment slot instead of the pair p
  int64_t Nw;               // weight rows per expert (SwiGLU: 2 * Nout)
  int Kin;                  // reduction length
  int Nout;                 // output columns
  int k;                    // top-k
  int64_t P;                // number of pairs = sentinel value
  int E;                    // experts (guards the expert ids read from the alignment)
  const int32_t* sorted;
  const int32_t* expert_ids;
  const int32_t* ntpp;
  int bm;
  int64_t grid_blocks;      // block slots to launch for
  const float* topk_w;      // [P] (EPI_WEIGHTED_F32)
  void* out;                // [P, Nout]: f16 / bf16 (SWIGLU, RELU2), bf16 (PLAIN) or f32 (WEIGHTED);
                            // MXFP8 weights: f32 h (SWIGLU, RELU2), or E4M3 codes of h when
                            // out_scale is set (SWIGLU on the block-scaled kernel)
  uint8_t* out_scale;       // [P, Nout / 32] E8M0 scales of an MXFP8 h, or null
  int32_t* status;
  int64_t wait_ns;          // limit of the tensor-memory kernels' waits (0: the 2 s default)
  int stall;                // stalled self-test: the copy and MMA roles do nothing
  // W4A16 tensor-memory kernel: tiles with a weight block scale outside the f16 window are
  // marked here (one bit per tile, zeroed by the caller) and done again with shifted
  // weights by a second launch; null: such blocks are reported (MOE_ERR_RANGE)
  uint32_t* fix_bits;
  int32_t* fix_count;
};

// Bytes of the marks of one W4A16 tensor-memory GEMM over at most `blocks` alignment blocks
// and `nout` output features (256-byte aligned: the count, then one bit per tile).
size_t ts_fix_bytes(int64_t blocks, int64_t nout);
// Tiles of that GEMM: feature tiles per block (128 features, two matrices per tile).
int64_t ts_fix_tiles(int64_t blocks, int64_t nout);

// Stall limit set by moe_debug_stall_tensor_kernels (0: normal operation), and its
// application to one GEMM's arguments.
int64_t debug_stall_ns();
void apply_debug_stall(GroupedGemm& g);
size_t decode_gemm_smem_bytes(const GroupedGemm& g);
cudaError_t decode_gemm(const GroupedGemm& g, cudaStream_t stream);


// ---- the MXFP4 layer of up to 256 rows on the block-scaled MMA (decode_tc.cu): x and h split
// into eight E2M1 digit planes each, one E8M0 scale per 32 elements (plane 0's; plane j's is
// 2j less); GEMM1 writes h's planes.  kq(n) = 64 * ceil(n / 128) bytes a plane row.
struct DecodeTcBufs {
  uint8_t* xq;       // [T_rows, 8, kq(K)] x planes, two codes a byte
  uint8_t* xs;       // [T_rows, sb(K)] x scales
  uint8_t* hq;       // [P, 8, kq(I)] h planes
  uint8_t* hs;       // [P, sb(I)] h scales
  int4* items;       // [P] (alignment block, 4- or 8-slot tile, slots to its last pair + 1, expert)
  int32_t* n_items;
};
// Whether GEMM1 (SwiGLU, MXFP4 weights) and GEMM2 (routing-weighted) of a layer fit the kernel.
bool decode_tc_supported(const GroupedGemm& g1, const GroupedGemm& g2);
size_t decode_tc_workspace_bytes(int64_t T_rows, int k, int K, int I);
DecodeTcBufs decode_tc_carve(void* ws, int64_t T_rows, int k, int K, int I);
// x (bf16 [T_rows, K]) -> planes, and the units' items (g1's alignment).
cudaError_t decode_tc_prep(const GroupedGemm& g1, const void* x, int64_t T_rows, const DecodeTcBufs& b,
                           cudaStream_t stream);
// GEMM1 (g.epi EPI_SWIGLU: x planes -> h planes) or GEMM2 (EPI_WEIGHTED_F32: h planes -> o).
cudaError_t decode_tc_gemm(const GroupedGemm& g, const DecodeTcBufs& b, cudaStream_t stream);

// ---- grouped GEMMs on the tensor-memory (prefill) path (prefill_gemm.cu)
int prefill_tile_n(const GroupedGemm& g);
bool prefill_supported(const GroupedGemm& g);
cudaError_t prefill_gemm(const GroupedGemm& g, cudaStream_t stream);

// ---- W4A16 grouped GEMM with the decoded weights in tensor memory (prefill_ts.cu)
bool ts_supported(const GroupedGemm& g);
cudaError_t prefill_ts(const GroupedGemm& g, cudaStream_t stream);

// ---- MXFP8 grouped GEMM on the block-scaled tensor-core MMA (mx8_gemm.cu)
bool mx8_supported(const GroupedGemm& g);
cudaError_t mx8_gemm(const GroupedGemm& g, cudaStream_t stream);

// ---- per-token FP8 grouped GEMM over group sizes (pertoken_gemm.cu)
struct PerTokenGemm {
  int E, N, K;
  int64_t M;                   // rows of a and out
  const void* a;               // [M, K] E4M3, rows grouped by expert in expert order
  const float* a_scale;        // [M]
  const void* w;               // [E, N, K] E4M3
  const float* w_scale;        // [E]
  const void* bias;            // [E, N] bf16 or null
  const int32_t* group_sizes;  // [E] rows per expert (device)
  void* out;                   // [M, N] bf16
  int32_t* status;
};
// N and K multiples of 128, 1 <= E <= 1024.
cudaError_t pertoken_gemm(const PerTokenGemm& g, cudaStream_t stream);

// Row counts above this bucket value use the tensor-memory path.  A bucket value (a
// fixed point of the bucket map) keeps a batch and its bucket-padded copy on the same
// side of the threshold, so both run the same kernel.
constexpr int64_t kPrefillRowsAbove = 256;

// Runs one grouped GEMM on the path its row count and shape select.
cudaError_t grouped_gemm(const GroupedGemm& g, int64_t rows, cudaStream_t stream);

// ---- weight gradient (wgrad.cu)
struct Wgrad {
  const void* grad;   // [P, N] bf16
  const void* input;  // [T or P, Kin] bf16
  int input_per_pair;
  int64_t P;
  int k, E, N, Kin;
  const int32_t* sorted;
  const int32_t* expert_ids;
  const int32_t* ntpp;
  int bm;
  int64_t cap_blocks;
  float* dW;
  int mode;
  int32_t* status;
  // slot-ordered copies of grad [cap, N] and input [cap, Kin] (gather_slot_rows), or null:
  // with them the tensor-memory kernel loads whole 64-slot tiles by TMA
  const void* grad_s;
  const void* input_s;
  int64_t cap;
  int32_t* ranges;  // [E][2] first, end alignment block of each expert (slot feed scratch)
  int64_t wait_ns;  // limit of every wait of the tensor-memory kernel (0: the default)
  int stall;        // failure-detection self-test: its copy and MMA roles off
};
cudaError_t wgrad(const Wgrad& g, cudaStream_t stream);
void apply_debug_stall(Wgrad& g);

// ---- weight gradient on the tensor-memory path (wgrad_tc.cu)
int wgrad_tc_tile(const Wgrad& g);
// Whether the tensor-memory kernel can read the slot-ordered copies (block_m a multiple of
// the 64-slot stage, dW rows addressable by TMA).
bool wgrad_tc_slot_feed(const Wgrad& g);
cudaError_t wgrad_tc(const Wgrad& g, cudaStream_t stream);

}  // namespace moe_launch
