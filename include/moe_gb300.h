/*
 * moe_gb300.h -- C ABI of the Mixture-of-Experts expert-layer hot path on GB300 (sm_103a).
 *
 * The path: top-k routing -> token-to-expert alignment (moe_align) -> geometric
 * token-dimension bucketing and padding (moe_bucket_pad) -> grouped GEMM1 + bias + SwiGLU
 * (or relu^2) -> grouped GEMM2 + bias * routing weight -> top-k combine (moe_forward; in
 * MXFP8 with h quantised between the GEMMs, moe_mx_quantize); a single grouped GEMM over
 * given operands (moe_grouped_gemm); a per-token-scaled FP8 grouped GEMM over per-expert
 * group sizes (moe_gemm_per_token); and the per-expert weight gradient (moe_wgrad).
 *
 * Sources of the definitions (pull-request pages):
 *  [BUCKET] "Bound Triton MoE JIT specializations via token-dim bucketing and warmup",
 *           TensorRT-LLM PR 15311 -- Description; Test Coverage.
 *  [DECODE] "tune the Nemotron MTP decode row on S5000 with a checked-in recipe",
 *           torchada PR 115 -- What it does (tiny-M bf16 fused-MoE decode shape).
 *  [AITER]  "Add MoE GEMM variants and weight-gradient kernel", ROCm aiter PR 5310 --
 *           Summary; Notes; second review (sentinel handling, E8M0 decoding, bias indexing).
 *
 * Conventions for every call
 *  - All device buffers are owned by the caller.  The library never allocates device
 *    memory; scratch comes from ctx->workspace (size from the *_workspace_size calls).
 *  - Work is enqueued on ctx->stream (a cudaStream_t; NULL = the legacy default stream).
 *    No call synchronises the host with the device.
 *  - Every device pointer must be 16-byte aligned and every tensor dense row-major with
 *    exactly the shape stated (a per-expert bias is a contiguous [E, N] array; strided
 *    biases are not accepted -- the bias-stride defect named in [AITER]'s second review
 *    is ruled out by contract).
 *  - Integers that index pairs or weight elements are 64-bit inside the kernels: with
 *    E = 256 an expert offset times the per-expert weight size exceeds INT32_MAX ([AITER],
 *    Notes).
 *  - The return value reports argument and launch errors only.  Errors that depend on
 *    the data (an expert id outside [0, E), an activation outside the decode path's
 *    float16 range) are written to the optional device word ctx->dev_status, first error
 *    wins; the caller reads it after synchronising.  No kernel traps.
 *  - moe_last_error() returns a thread-local description of the last failed call.
 *  - The library keeps no state; calls are thread-safe.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status;
#define MOE_OK 0
#define MOE_WARN_PAD_IGNORED 1    /* moe_bucket_pad: padding not allowed for this mode   */
#define MOE_ERR_INVALID_ARG (-1)  /* null pointer, bad size, misalignment               */
#define MOE_ERR_UNSUPPORTED (-2)  /* a size or mode this build does not implement       */
#define MOE_ERR_CAPACITY (-3)     /* an output or workspace buffer is too small         */
#define MOE_ERR_CUDA (-4)         /* a CUDA launch or runtime error                     */
/* device status codes (ctx->dev_status) */
#define MOE_ERR_INVALID_EXPERT (-5) /* a top-k id outside [0, E)                        */
#define MOE_ERR_RANGE (-6)          /* an activation or h value beyond float16's 65504   */
#define MOE_ERR_TIMEOUT (-7)        /* a bounded wait inside a kernel ran out            */

typedef enum {
  MOE_Q_BF16 = 0,        /* bf16 weights, bf16 activations                              */
  MOE_Q_MXFP4_W4A16 = 1, /* E2M1 weights, two per byte (even K index in the low nibble),
                            one E8M0 scale per 32 along K; bf16 activations            */
  MOE_Q_MXFP8 = 2        /* E4M3 weights and activations, one E8M0 scale per 32 along K */
} moe_quant;

typedef struct {
  void* stream;            /* cudaStream_t                                                  */
  void* workspace;         /* device scratch, caller-owned, 256-byte aligned                */
  size_t workspace_bytes;  /* its size                                                      */
  int32_t* dev_status;     /* optional device int32 (set to 0 by the caller); may be NULL   */
  void** events;           /* optional host array of cudaEvent_t recorded on the stream
                              around each kernel of a call (profiling); may be NULL.
                              moe_forward: [0] before GEMM1 (after x's f16 copy or
                              planes), [1] after GEMM1, [2] after GEMM2, [3] after the
                              combine (needs n_events >= 4);
                              moe_grouped_gemm, moe_wgrad: [0] before, [1] after.      */
  int32_t n_events;
} moe_ctx;

/* Thread-local text of the last error returned on this thread ("" if none). */
const char* moe_last_error(void);

/* ------------------------------------------------------------------------------------ *
 * Alignment: routing + moe_align_block_size                                             *
 * ------------------------------------------------------------------------------------ */

/* Capacity of the alignment outputs for num_pairs = T*k pairs:
 *   cap_tokens = round_up(num_pairs + E*(block_m-1), block_m), cap_blocks = cap_tokens/block_m
 * -- the most slots any routing can need (each expert's count padded up to whole
 * blocks). */
moe_status moe_align_capacity(int64_t num_pairs, int32_t E, int32_t block_m,
                              int64_t* cap_tokens, int64_t* cap_blocks);

/* Routing and alignment (one call).
 *
 * Routing (when logits != NULL): logits [T, E] fp32 -> topk_ids [T, k] int32 (the k largest
 * logits in descending order; equal logits rank the lower expert id first) and topk_w
 * [T, k] fp32 = softmax over the k chosen logits, computed in float64 and rounded to
 * float32.  When logits == NULL, topk_ids is an input and topk_w is not touched (may be
 * NULL).
 *
 * Alignment ([AITER] Summary and second review; [DECODE] What it does): with pair index
 * p = t*k + j, c_e pairs routed to expert e, P_e = c_e rounded up to block_m and
 * O_e = sum_{e'<e} P_e':
 *   sorted_token_ids[cap_tokens]: slots O_e .. O_e+c_e-1 hold expert e's pair indices in
 *       ascending order; every other slot holds the sentinel T*k;
 *   expert_ids[cap_tokens/block_m]: block b holds the expert owning slots
 *       b*block_m .. (b+1)*block_m-1, and -1 for every block at or past
 *       num_tokens_post_padded/block_m (kernels skip -1 blocks at once);
 *   num_tokens_post_padded[1] = sum_e P_e;
 *   expert_offsets[E+1] (may be NULL) = unpadded prefix sums of c_e (differences are the
 *       per-expert group sizes).
 * Limits: 1 <= k <= 32, k <= E <= 1024, 1 <= block_m <= 1024, 0 <= T, T*k < 2^31.
 * cap_tokens must be >= moe_align_capacity() and a multiple of block_m
 * (MOE_ERR_CAPACITY).  Out-of-range ids set MOE_ERR_INVALID_EXPERT in dev_status and are
 * left out of the outputs.  Needs no workspace. */
moe_status moe_align(const float* logits, int32_t* topk_ids, float* topk_w,
                     int64_t T, int32_t k, int32_t E, int32_t block_m,
                     int32_t* sorted_token_ids, int64_t cap_tokens,
                     int32_t* expert_ids, int32_t* num_tokens_post_padded,
                     int32_t* expert_offsets, const moe_ctx* ctx);

/* ------------------------------------------------------------------------------------ *
 * Token-dimension bucketing ([BUCKET] Description, Test Coverage)                        *
 * ------------------------------------------------------------------------------------ */

/* bucket(m) = ceil(m / s) * s with s = max(1, 2^(floor(log2 m) - 3)): eight buckets per
 * power-of-two octave from 16 on, every m < 16 its own bucket, at most 12.5% padding.
 * Returns -1 for m < 1. */
int64_t moe_bucket(int64_t m);

/* Number of buckets <= max_tokens (97 for 20000). */
int64_t moe_bucket_count(int64_t max_tokens);

/* T_pad = bucket(T) for MOE_Q_MXFP4_W4A16; for every other mode padding is not allowed
 * (dynamic activation scales would let pad rows change real outputs), *T_pad = T and the
 * call returns MOE_WARN_PAD_IGNORED.  T == 0 gives T_pad = 0.
 * Device part (optional): when x_pad != NULL, rows [0, T) of x ([T, row_bytes]) are copied
 * to x_pad ([T_pad, row_bytes]; x == x_pad skips the copy) and rows [T, T_pad) are zeroed;
 * likewise logits [T, E] fp32 -> logits_pad [T_pad, E] when logits_pad != NULL (zero pad
 * logits route pad rows to experts 0..k-1 with weight 1/k).  row_bytes must be a multiple
 * of 16. */
moe_status moe_bucket_pad(int64_t T, moe_quant quant, int64_t* T_pad,
                          const void* x, void* x_pad, int64_t row_bytes,
                          const float* logits, float* logits_pad, int32_t E,
                          const moe_ctx* ctx);

/* ------------------------------------------------------------------------------------ *
 * Forward: grouped GEMM1 + SwiGLU -> grouped GEMM2 -> combine                           *
 * ------------------------------------------------------------------------------------ */

/* Activation between the GEMMs.  MOE_ACT_RELU2 is the non-gated relu2_no_mul of [DECODE]
 * (the Nemotron recipe in its table of added files: GEMM1 N = 1856 = I, no gate product). */
typedef enum {
  MOE_ACT_SWIGLU = 0,     /* h = silu(gate) * up; GEMM1 has 2I rows (gate | up)           */
  MOE_ACT_RELU2 = 1       /* h = max(a, 0)^2;     GEMM1 has I rows                        */
} moe_activation;

/* N1 = 2I for MOE_ACT_SWIGLU, I for MOE_ACT_RELU2. */
typedef struct {
  moe_quant quant;
  int32_t E, K, I;        /* experts, hidden size, intermediate size                      */
  const void* w1;         /* [E, N1, K] (MXFP4: [E, N1, K/2] bytes); SwiGLU: rows 0..I-1
                             gate, rows I..2I-1 up                                        */
  const uint8_t* w1_scale;/* [E, N1, K/32] E8M0 (NULL for bf16)                           */
  const void* b1;         /* [E, N1] bf16 or NULL                                         */
  const void* w2;         /* [E, K, I] (MXFP4: [E, K, I/2] bytes)                         */
  const uint8_t* w2_scale;/* [E, K, I/32] E8M0 (NULL for bf16)                            */
  const void* b2;         /* [E, K] bf16 or NULL                                          */
  int32_t activation;     /* moe_activation (a zero-initialised struct is SwiGLU)         */
} moe_weights;

/* Workspace bytes moe_forward needs for T_rows rows of top-k with an alignment of
 * cap_tokens slots (moe_align_capacity): h [rows_h, I] (f16 for MXFP4 weights, bf16 for bf16
 * weights), o [T_rows*k, K] fp32 and x as f16 [rows_x, K], each 256-byte aligned.  rows_h =
 * T_rows*k and rows_x = T_rows up to 256 rows; above that h and x may be kept in
 * alignment-slot order and rows_h = rows_x = cap_tokens, and two small regions (one bit per
 * output tile of each GEMM) follow, which mark tiles whose weight scales need the exact
 * second pass.  Up to 256 rows five more regions follow, for the block-scaled MXFP4 kernels:
 * x as eight E2M1 digit planes [T_rows, 8, kq(K)] bytes (two codes a byte) and their E8M0
 * scales [T_rows, sb(K)], h as eight planes [T_rows*k, 8, kq(I)] and scales [T_rows*k,
 * sb(I)], and a unit list [T_rows*k + 1, 16 bytes], where kq(n) = 64 * ceil(n / 128) and
 * sb(n) = 16 * ceil(ceil(n / 128) / 4).  Returns 0 for a negative argument. */
size_t moe_forward_workspace_size(int64_t T_rows, int32_t k, int32_t K, int32_t I, int64_t cap_tokens);

/* One MoE expert layer over the alignment of moe_align: both grouped GEMMs run as single
 * launches over every expert, each with an optional contiguous per-expert bias ([AITER]
 * Summary: the grouped GEMM over all experts in one launch with per-expert bias), and
 * token-dimension pad rows are computed like any other row but sliced off before the
 * top-k reduction, so only rows t < T_real reach y ([BUCKET] Description: padded rows are
 * removed ahead of the combine).  Blocks whose expert id is the -1 sentinel are skipped
 * before any weight is read ([AITER] second review: return at once on the sentinel).
 *
 * For every real token t < T_real (the others, e.g. bucket pad rows, are computed and
 * then sliced off):
 * Exactness of the W4A16 tensor-core path (above 256 rows): weights are decoded to float16
 * as code * 2^(E8M0 - 127), exact while that exponent lies in -23..13; a tile with a
 * nonzero block outside that window is computed again by a second pass with each weight row
 * shifted by a power of two (undone on its fp32 accumulator), so any E8M0 scale gives the
 * exact products the weight-streaming path gives below 256 rows.  Only a weight row whose
 * nonzero blocks span more than 36 octaves of scale is reported (MOE_ERR_RANGE).
 *
 *   gu = x_t . W1[e]^T + b1[e];  h = silu(gu[:I]) * gu[I:]  (SwiGLU) or
 *        h = max(gu, 0)^2  (relu^2; a NaN stays NaN)  (fp32, then rounded to the operand
 *        type of GEMM2: f16 RNE for MXFP4 weights -- |h| > 65504 sets MOE_ERR_RANGE, and so
 *        does |x| > 65504 where x is converted to f16: above 256 rows and for relu^2 -- and
 *        bf16 RNE for bf16 weights).  Up to 256 rows the MXFP4 SwiGLU layer (K and I
 *        multiples of 64, 256..3072) runs the block-scaled kernels: x and the f16 h enter
 *        the MMA as eight E2M1 digit planes (base-4 digits under one E8M0 scale per 32
 *        elements and plane), which sum to each value exactly for elements no more than
 *        2^8 (x) or 2^5 (h) below their block's largest, and within 2^-16 of that largest
 *        for the rest
 *   o_tj = w[t,j] * (h . W2[e]^T + b2[e])                    (fp32)
 *   y_t  = sum_{j=0..k-1} o_tj, in order of j, rounded to bf16 RNE.
 * x: [T_rows, K] bf16 (BF16 and MXFP4_W4A16 modes).  topk_w [T_rows, k]; the alignment
 * arrays come from moe_align over T_rows rows with the same block_m and cap_tokens.
 * y: [T_real, K] bf16.  K and I must be multiples of 32 (and of 16 output rows).
 * MXFP8 (SwiGLU only): x is E4M3 codes [T_rows, K] with x_scale [T_rows, K/32] E8M0, the
 * weights E4M3 with E8M0 scales; h is computed in fp32 and quantised to MXFP8 by the rule of
 * moe_mx_quantize before GEMM2, whose operands are then MXFP8 on both sides.  Below the
 * tensor-memory threshold (or for shapes the block-scaled kernel does not take: I or K not
 * a multiple of 128) this mode needs I <= K.  No pair-count-dependent split of K is
 * made and every output row depends only on its own input row, so padded and unpadded
 * calls give bit-identical real rows. */
moe_status moe_forward(const moe_weights* W, const void* x, const uint8_t* x_scale,
                       int64_t T_rows, int64_t T_real, int32_t k,
                       const float* topk_w, const int32_t* sorted_token_ids,
                       const int32_t* expert_ids, const int32_t* num_tokens_post_padded,
                       const int32_t* expert_offsets, int32_t block_m, int64_t cap_tokens,
                       void* y, const moe_ctx* ctx);

/* Size of the fixed device scratch array used by moe_forward_no_alloc (16 MiB). */
#define MOE_NO_ALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* moe_forward without a caller workspace; the pages have no counterpart to this call.
 *
 * For callers that cannot call cudaMalloc: code embedded in a host program that owns
 * every device allocation (it hands the plug-in its input and output buffers only), or
 * threads that must not enter the CUDA allocator, which can synchronise the device and
 * fail under memory pressure.  Arguments and results are exactly those of moe_forward;
 * ctx->workspace and ctx->workspace_bytes are ignored.  The scratch (h, o and the f16
 * copy of x) lives in a file-scope device array of MOE_NO_ALLOC_SCRATCH_BYTES inside
 * the library; every GPU that loads the library holds it until the process exits.
 *  - A call whose moe_forward_workspace_size exceeds the array returns MOE_ERR_CAPACITY
 *    (e.g. the 64-token, 2880/2880, top-4 layer needs about 4.8 MB and fits).
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress).  The first call on a device also loads the library's device
 *    code there; make that first call before any stream capture.
 *  - An empty batch (T_rows == 0) returns MOE_OK, as moe_forward does; invalid arguments
 *    are reported by moe_forward's own checks.
 *  - Every call shares the one array, which keeps the last call's contents.  Nothing in
 *    it has to start at zero: each call writes every scratch element it reads.  Calls
 *    that can overlap on the GPU (other streams, other host threads) race on the array:
 *    serialise them.
 *  - The call itself allocates no memory (no cudaMalloc, cudaFree or allocating library
 *    routine). */
moe_status moe_forward_no_alloc(const moe_weights* W, const void* x, const uint8_t* x_scale,
                                int64_t T_rows, int64_t T_real, int32_t k,
                                const float* topk_w, const int32_t* sorted_token_ids,
                                const int32_t* expert_ids,
                                const int32_t* num_tokens_post_padded,
                                const int32_t* expert_offsets, int32_t block_m,
                                int64_t cap_tokens, void* y, const moe_ctx* ctx);

/* ------------------------------------------------------------------------------------ *
 * One grouped GEMM over all experts in a single launch ([AITER] Summary: moe_gemm_mxfp8) *
 * ------------------------------------------------------------------------------------ */

/* Workspace bytes that let moe_grouped_gemm run W4A16 (MOE_Q_MXFP4_W4A16) weights on the
 * tensor cores: above 256 token rows the tcgen05 kernel reads A as float16, and the call
 * converts A into the workspace first (rows x Kin x 2 bytes, rows = T*k if a_per_pair else
 * T), followed by one bit per output tile that marks tiles whose weight scales need the
 * exact second pass (see moe_forward).  0 for the other modes, for T <= 256, or for invalid
 * sizes. */
size_t moe_grouped_gemm_workspace_size(moe_quant quant, int64_t T, int32_t k, int32_t N, int32_t Kin,
                                       int32_t a_per_pair);

/* out[p, :] = A[src(p), :] . W[e_p]^T + bias[e_p]   for every pair p < T*k, in bf16 RNE.
 * A: [T, Kin] (a_per_pair == 0, src = p / k) or [T*k, Kin] (a_per_pair != 0, src = p);
 *    bf16 for MOE_Q_BF16 / MOE_Q_MXFP4_W4A16, E4M3 bytes + a_scale [rows, Kin/32] E8M0
 *    for MOE_Q_MXFP8.
 * W: [E, N, Kin] (MXFP4: [E, N, Kin/2] bytes) + w_scale [E, N, Kin/32]; bias [E, N] bf16
 *    or NULL.  out: [T*k, N] bf16, indexed by pair.
 * N must be a multiple of 16 and Kin of 32.
 * Kernels: MXFP8 above 256 token rows runs the block-scaled tensor-core kernel (K and N
 * multiples of 128); bf16 above 256 rows the same tcgen05 kernel with bf16 operands (block_m
 * 128, K a multiple of 64, N of 128); W4A16 above 256 rows runs the tcgen05 kernel with
 * decoded weights in tensor memory when ctx->workspace holds
 * moe_grouped_gemm_workspace_size() bytes (block_m 128, Kin a multiple of 64; |A| <= 65504,
 * else MOE_ERR_RANGE in dev_status); every other call runs the weight-streaming kernel,
 * which needs no workspace.  The kernel
 * choice depends on T only through the bucket value 256, and each kernel reduces K in one
 * fixed order. */
moe_status moe_grouped_gemm(moe_quant quant, int32_t E, int32_t N, int32_t Kin,
                            const void* a, const uint8_t* a_scale, int32_t a_per_pair,
                            const void* w, const uint8_t* w_scale, const void* bias,
                            int64_t T, int32_t k,
                            const int32_t* sorted_token_ids, const int32_t* expert_ids,
                            const int32_t* num_tokens_post_padded, int32_t block_m,
                            int64_t cap_tokens, void* out, const moe_ctx* ctx);

/* ------------------------------------------------------------------------------------ *
 * MXFP8 quantisation (the step between the GEMMs of an MXFP8 layer)                      *
 * ------------------------------------------------------------------------------------ */

/* x [rows, cols] fp32 (cols a multiple of 32) -> codes [rows, cols] E4M3 and scales
 * [rows, cols / 32] E8M0, per 32 consecutive values of a row, by the OCP microscaling rule
 * for E4M3 elements: e = floor(log2(max |v|)) - 8 clamped to [-127, 127] (-127 for an
 * all-zero block), scale byte e + 127, code = E4M3(v / 2^e) rounded to nearest even and
 * saturated at 448, signs (zero included) kept.  A block holding a NaN gets scale 0xFF and
 * codes 0x7F.  [AITER] Summary gives the GEMM operands this format (moe_gemm_mxfp8); the
 * rule itself is the reading this library takes where the pages stop.  moe_forward applies
 * it to h in MXFP8 mode. */
moe_status moe_mx_quantize(const float* x, int64_t rows, int32_t cols, uint8_t* codes, uint8_t* scales,
                           const moe_ctx* ctx);

/* ------------------------------------------------------------------------------------ *
 * Per-token FP8 grouped GEMM over group sizes ([AITER] Summary: moe_gemm_per_token)      *
 * ------------------------------------------------------------------------------------ */

/* The rows of a are grouped by expert in expert order: expert e owns rows
 * O_e .. O_e + group_sizes[e] - 1, O_e = group_sizes[0] + ... + group_sizes[e-1]. For each
 * such row m:
 *   out[m, n] = bf16 RNE( (sum_k a[m, k] * w[e, n, k]) * a_scale[m] * w_scale[e] + bias[e, n] )
 * with the dot product of the E4M3 codes accumulated in fp32 before either scale.
 * a: [M, K] E4M3 codes; a_scale: [M] fp32; w: [E, N, K] E4M3; w_scale: [E] fp32;
 * bias: [E, N] bf16 or NULL; group_sizes: [E] int32 in device memory; out: [M, N] bf16.
 * Rows past the sum of the group sizes are not written.  Negative sizes, or sizes adding up
 * to more than M, set MOE_ERR_CAPACITY in ctx->dev_status (the sizes are read as clamped to
 * the M rows).  Limits: 1 <= E <= 1024, N and K multiples of 128, M < 2^31,
 * E * N < 2^31.  Needs no workspace. */
moe_status moe_gemm_per_token(int32_t E, int32_t N, int32_t K, const uint8_t* a, const float* a_scale,
                              const uint8_t* w, const float* w_scale, const void* bias,
                              const int32_t* group_sizes, int64_t M, void* out, const moe_ctx* ctx);

/* ------------------------------------------------------------------------------------ *
 * Weight gradient ([AITER] Summary: moe_wgrad; Tests & Benchmarks)                      *
 * ------------------------------------------------------------------------------------ */

/* Workspace bytes for moe_wgrad's slot-ordered copies (cap_tokens x N and cap_tokens x Kin
 * bf16) and the experts' block ranges (E x 2 int32), each 256-byte aligned: mode 0 with N a
 * multiple of 128, Kin of 64, block_m of 64 and E <= 1024; 0 otherwise (moe_wgrad then
 * needs none). */
size_t moe_wgrad_workspace_size(int32_t E, int32_t N, int32_t Kin, int32_t block_m, int64_t cap_tokens,
                                int32_t mode);

/* dW[e] = sum over pairs p routed to e of grad[p, :]^T (outer) input[src(p), :], fp32
 * accumulation, read straight from the alignment outputs (sentinel slots add nothing).
 * grad: [T*k, N] bf16 indexed by pair; input: [T, Kin] bf16 (input_per_pair == 0,
 * src = p / k) or [T*k, Kin] (input_per_pair != 0, src = p).  dW: [E, N, Kin] fp32.
 * mode 0: deterministic -- every dW[e] is written, zeros for experts with no pair, and
 *         repeated calls give identical bits.
 * mode 1: accumulate -- the library zeroes dW, then adds token-chunk partial sums with
 *         atomics (summation order varies between runs).
 * N and Kin must be multiples of 64.  Needs no workspace; with ctx->workspace holding
 * moe_wgrad_workspace_size() bytes, mode 0 first copies grad and input rows into slot order
 * there and the tensor-core kernel loads whole stages of them by TMA -- the same sums in the
 * same order, so the same bits as without a workspace. */
moe_status moe_wgrad(const void* grad, const void* input, int32_t input_per_pair,
                     int64_t T, int32_t k, int32_t E, int32_t N, int32_t Kin,
                     const int32_t* sorted_token_ids, const int32_t* expert_ids,
                     const int32_t* num_tokens_post_padded, int32_t block_m,
                     int64_t cap_tokens, float* dW, int32_t mode, const moe_ctx* ctx);

/* ------------------------------------------------------------------------------------ *
 * Diagnostics: failure detection of the bounded waits                                    *
 * ------------------------------------------------------------------------------------ */

/* Self-test switch of the tensor-memory kernels' failure detection (their waits on
 * mbarriers are bounded and report MOE_ERR_TIMEOUT instead of hanging).  With stall_ns > 0,
 * every later launch of the W4A16 and MXFP8 tensor-memory grouped GEMMs in this process
 * (moe_forward above 256 rows, moe_grouped_gemm in MXFP8) runs with its copy and MMA roles
 * switched off: the other roles wait on barriers that nothing arrives on, give up after
 * stall_ns nanoseconds, write MOE_ERR_TIMEOUT to ctx->dev_status, free their tensor memory
 * and return; no copy or MMA is in flight when they give up, and the context stays usable.
 * Outputs of calls made meanwhile are undefined.  stall_ns <= 0 restores normal operation
 * (2 s limits).  Process-wide; not for use while other threads run the library.  The pages
 * have no counterpart to this call. */
void moe_debug_stall_tensor_kernels(int64_t stall_ns);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
