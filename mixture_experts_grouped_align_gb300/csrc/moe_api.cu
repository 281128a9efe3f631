// The C ABI (include/moe_gb300.h): argument validation, workspace carving and launches.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "moe_common.cuh"
#include "moe_launch.h"

namespace moe_host {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

}  // namespace moe_host

namespace moe_launch {

namespace {
std::atomic<int64_t> g_debug_stall_ns{0};
}  // namespace

int64_t debug_stall_ns() { return g_debug_stall_ns.load(std::memory_order_relaxed); }

// The wait limit and stall flag every GroupedGemm and Wgrad of a call carries.
void apply_debug_stall(GroupedGemm& g) {
  const int64_t ns = debug_stall_ns();
  g.wait_ns = ns > 0 ? ns : 0;
  g.stall = ns > 0 ? 1 : 0;
}
void apply_debug_stall(Wgrad& g) {
  const int64_t ns = debug_stall_ns();
  g.wait_ns = ns > 0 ? ns : 0;
  g.stall = ns > 0 ? 1 : 0;
}

int sm_count_current() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  if (dev >= 0 && dev < kMaxDev) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev >= 0 && dev < kMaxDev && n > 1) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace moe_launch

namespace {

using moe_host::set_error;

#define MOE_REQUIRE(cond, code, ...) \
  do {                               \
    if (!(cond)) {                   \
      set_error(__VA_ARGS__);        \
      return code;                   \
    }                                \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status cuda_status(cudaError_t err, const char* what) {
  if (err == cudaSuccess) return MOE_OK;
  set_error("%s: %s", what, cudaGetErrorString(err));
  return MOE_ERR_CUDA;
}

cudaStream_t stream_of(const moe_ctx* ctx) {
  return ctx ? static_cast<cudaStream_t>(ctx->stream) : nullptr;
}
int32_t* status_of(const moe_ctx* ctx) { return ctx ? ctx->dev_status : nullptr; }

// Records profiling event i of the caller (if it gave at least `need` events).
void rec(const moe_ctx* ctx, int i, int need) {
  if (ctx && ctx->events && ctx->n_events >= need && ctx->events[i])
    cudaEventRecord(static_cast<cudaEvent_t>(ctx->events[i]), stream_of(ctx));
}

// T*k pairs index int32 slots: true when 0 <= T and T*k <= INT32_MAX, without forming an
// overflowing product for huge T.
bool pairs_fit(int64_t T, int32_t k) { return T >= 0 && k >= 1 && T <= INT32_MAX / k; }

// An [E, N, Kin] weight array (elements) is indexed with int64 inside the kernels.
bool weights_fit(int32_t E, int64_t N, int64_t Kin) {
  return E >= 1 && N >= 1 && Kin >= 1 && N <= (INT64_MAX / 4) / Kin / E;
}

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

int64_t bucket_of(int64_t m) {
  if (m < 1) return -1;
  int lg = 63 - __builtin_clzll((unsigned long long)m);
  int sh = lg - 3 > 0 ? lg - 3 : 0;
  int64_t s = (int64_t)1 << sh;
  return (m + s - 1) / s * s;
}

moe_status check_align_outputs(int64_t P, int32_t E, int32_t block_m, const int32_t* sorted,
                               const int32_t* expert_ids, const int32_t* ntpp, int64_t cap_tokens) {
  MOE_REQUIRE(sorted && expert_ids && ntpp, MOE_ERR_INVALID_ARG, "null alignment pointer");
  MOE_REQUIRE(aligned16(sorted) && aligned16(expert_ids) && aligned16(ntpp), MOE_ERR_INVALID_ARG,
              "alignment pointers must be 16-byte aligned");
  MOE_REQUIRE(block_m >= 1 && block_m <= 1024, MOE_ERR_INVALID_ARG, "block_m must be in [1, 1024]");
  int64_t need = P + (int64_t)E * (block_m - 1);
  need = (need + block_m - 1) / block_m * block_m;
  MOE_REQUIRE(cap_tokens >= need && cap_tokens % block_m == 0, MOE_ERR_CAPACITY,
              "cap_tokens %lld < required %lld or not a multiple of block_m", (long long)cap_tokens,
              (long long)need);
  return MOE_OK;
}

// Block slots a grouped launch must cover: at most ceil(P / bm) + min(E, P) are used.
int64_t used_blocks_bound(int64_t P, int32_t E, int32_t bm, int64_t cap_tokens) {
  int64_t b = (P + bm - 1) / bm + (E < P ? E : P);
  int64_t cap_blocks = cap_tokens / bm;
  return b < cap_blocks ? b : cap_blocks;
}

}  // namespace

extern "C" {

const char* moe_last_error(void) { return moe_host::g_err; }

moe_status moe_align_capacity(int64_t num_pairs, int32_t E, int32_t block_m, int64_t* cap_tokens,
                              int64_t* cap_blocks) {
  MOE_REQUIRE(cap_tokens && cap_blocks, MOE_ERR_INVALID_ARG, "null output pointer");
  MOE_REQUIRE(num_pairs >= 0 && E >= 1 && block_m >= 1, MOE_ERR_INVALID_ARG,
              "need num_pairs >= 0, E >= 1, block_m >= 1");
  int64_t c = num_pairs + (int64_t)E * (block_m - 1);
  c = (c + block_m - 1) / block_m * block_m;
  *cap_tokens = c;
  *cap_blocks = c / block_m;
  return MOE_OK;
}

moe_status moe_align(const float* logits, int32_t* topk_ids, float* topk_w, int64_t T, int32_t k,
                     int32_t E, int32_t block_m, int32_t* sorted_token_ids, int64_t cap_tokens,
                     int32_t* expert_ids, int32_t* num_tokens_post_padded, int32_t* expert_offsets,
                     const moe_ctx* ctx) {
  MOE_REQUIRE(T >= 0, MOE_ERR_INVALID_ARG, "T must be >= 0");
  MOE_REQUIRE(k >= 1 && k <= 32 && E >= k && E <= 1024, MOE_ERR_UNSUPPORTED,
              "need 1 <= k <= 32 and k <= E <= 1024 (k=%d, E=%d)", k, E);
  MOE_REQUIRE(pairs_fit(T, k), MOE_ERR_UNSUPPORTED, "T*k must be < 2^31");
  MOE_REQUIRE(topk_ids && aligned16(topk_ids), MOE_ERR_INVALID_ARG,
              "topk_ids must be a 16-byte aligned device pointer");
  if (logits) {
    MOE_REQUIRE(topk_w && aligned16(topk_w) && aligned16(logits), MOE_ERR_INVALID_ARG,
                "routing needs 16-byte aligned logits and topk_w");
  }
  MOE_REQUIRE(!expert_offsets || aligned16(expert_offsets), MOE_ERR_INVALID_ARG,
              "expert_offsets must be 16-byte aligned");
  moe_status st = check_align_outputs(T * k, E, block_m, sorted_token_ids, expert_ids,
                                      num_tokens_post_padded, cap_tokens);
  if (st != MOE_OK) return st;
  return cuda_status(moe_launch::align(logits, topk_ids, topk_w, T, k, E, block_m, sorted_token_ids,
                                       cap_tokens, expert_ids, num_tokens_post_padded,
                                       expert_offsets, status_of(ctx), stream_of(ctx)),
                     "moe_align");
}

int64_t moe_bucket(int64_t m) { return bucket_of(m); }

int64_t moe_bucket_count(int64_t max_tokens) {
  // 1..15 are their own buckets; from 16 on every octave [2^j, 2^(j+1)) holds 8 buckets.
  int64_t n = 0;
  for (int64_t b = 1; b <= max_tokens;) {
    ++n;
    int64_t nb = bucket_of(b + 1);
    b = nb;
  }
  return n;
}

moe_status moe_bucket_pad(int64_t T, moe_quant quant, int64_t* T_pad, const void* x, void* x_pad,
                          int64_t row_bytes, const float* logits, float* logits_pad, int32_t E,
                          const moe_ctx* ctx) {
  MOE_REQUIRE(T_pad, MOE_ERR_INVALID_ARG, "T_pad is null");
  MOE_REQUIRE(T >= 0, MOE_ERR_INVALID_ARG, "T must be >= 0");
  const bool allowed = (quant == MOE_Q_MXFP4_W4A16);
  const int64_t tp = (allowed && T > 0) ? bucket_of(T) : T;
  *T_pad = tp;
  cudaStream_t s = stream_of(ctx);
  if (x_pad) {
    MOE_REQUIRE(x && row_bytes > 0 && row_bytes % 16 == 0 && aligned16(x) && aligned16(x_pad),
                MOE_ERR_INVALID_ARG, "x / x_pad must be 16-byte aligned with row_bytes % 16 == 0");
    moe_status st = cuda_status(moe_launch::pad_rows(x, x_pad, T, tp, row_bytes, s), "pad x");
    if (st != MOE_OK) return st;
  }
  if (logits_pad) {
    MOE_REQUIRE(logits && E >= 1 && aligned16(logits) && aligned16(logits_pad),
                MOE_ERR_INVALID_ARG, "logits / logits_pad must be 16-byte aligned, E >= 1");
    moe_status st =
        cuda_status(moe_launch::pad_rows(logits, logits_pad, T, tp, (int64_t)E * 4, s), "pad logits");
    if (st != MOE_OK) return st;
  }
  if (!allowed) {
    set_error("token-dimension padding is only allowed for MOE_Q_MXFP4_W4A16");
    return MOE_WARN_PAD_IGNORED;
  }
  return MOE_OK;
}

// Scratch of moe_forward: h ([rows_h, I], 16-bit), o ([P, K] fp32) and the f16 copy of x
// ([rows_x, K]).  Above the tensor-memory threshold h and x may be kept in alignment-slot
// order, with one row per slot of the capacity.
static void forward_scratch_rows(int64_t T_rows, int32_t k, int64_t cap_tokens, int64_t* rows_h,
                                 int64_t* rows_x) {
  const int64_t P = T_rows * k;
  const bool slots = T_rows > moe_launch::kPrefillRowsAbove && cap_tokens > P;
  *rows_h = slots ? cap_tokens : P;
  *rows_x = slots ? cap_tokens : T_rows;
}

// Bytes of the two GEMMs' marks of out-of-window weight tiles (the slot-ordered tensor-memory
// path only; see moe_launch::GroupedGemm::fix_bits).
static size_t forward_fix_bytes(int64_t T_rows, int32_t k, int32_t K, int32_t I, int64_t cap_tokens) {
  int64_t rows_h, rows_x;
  forward_scratch_rows(T_rows, k, cap_tokens, &rows_h, &rows_x);
  if (rows_h <= T_rows * k) return 0;  // pair order: the weight-streaming kernels
  const int64_t blocks = cap_tokens / 128;
  return moe_launch::ts_fix_bytes(blocks, I) + moe_launch::ts_fix_bytes(blocks, K);
}

size_t moe_forward_workspace_size(int64_t T_rows, int32_t k, int32_t K, int32_t I, int64_t cap_tokens) {
  if (T_rows < 0 || k < 1 || K < 1 || I < 1 || cap_tokens < 0) return 0;
  const int64_t P = T_rows * k;
  int64_t rows_h, rows_x;
  forward_scratch_rows(T_rows, k, cap_tokens, &rows_h, &rows_x);
  // up to 256 rows: the planes of x and h and the unit list of the block-scaled MXFP4 kernel
  const size_t dt = T_rows <= moe_launch::kPrefillRowsAbove ? moe_launch::decode_tc_workspace_bytes(T_rows, k, K, I) : 0;
  return round256((size_t)rows_h * I * 2) + round256((size_t)P * K * 4) + round256((size_t)rows_x * K * 2) +
         forward_fix_bytes(T_rows, k, K, I, cap_tokens) + dt;
}

// The MXFP8 layer: GEMM1 + SwiGLU, h quantised to MXFP8 (E4M3 codes and one E8M0 scale per
// 32 features), GEMM2 on MXFP8 operands, combine.  Above the threshold the block-scaled kernel
// quantises h in its epilogue; otherwise the weight-streaming kernels run and h goes through
// fp32 in the o scratch (which needs I <= K) and the standalone quantiser.  The workspace
// regions are those of the other modes: h codes and scales in the h region, o as before.
static moe_status forward_mxfp8(const moe_weights* W, const void* x, const uint8_t* x_scale, int64_t T_rows,
                                int64_t T_real, int32_t k, const float* topk_w, const int32_t* sorted_token_ids,
                                const int32_t* expert_ids, const int32_t* num_tokens_post_padded,
                                int32_t block_m, int64_t cap_tokens, void* y, const moe_ctx* ctx) {
  const int32_t E = W->E, K = W->K, I = W->I;
  MOE_REQUIRE(W->activation == MOE_ACT_SWIGLU, MOE_ERR_UNSUPPORTED, "the MXFP8 layer takes SwiGLU");
  MOE_REQUIRE(x_scale && W->w1_scale && W->w2_scale, MOE_ERR_INVALID_ARG, "MXFP8 needs x_scale and weight scales");
  MOE_REQUIRE(aligned16(x_scale), MOE_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  const int64_t P = T_rows * k;
  int64_t rows_h, rows_x;
  forward_scratch_rows(T_rows, k, cap_tokens, &rows_h, &rows_x);
  uint8_t* ws = static_cast<uint8_t*>(ctx->workspace);
  uint8_t* hq = ws;                                   // [P, I] E4M3 codes of h
  uint8_t* hs = ws + (size_t)P * I;                   // [P, I / 32] E8M0 scales of h
  float* o = reinterpret_cast<float*>(ws + round256((size_t)rows_h * I * 2));
  cudaStream_t s = stream_of(ctx);
  const int64_t blocks = used_blocks_bound(P, E, block_m, cap_tokens);

  moe_launch::GroupedGemm g1{};
  g1.wfmt = moe_launch::WF_MXFP8;
  g1.epi = moe_launch::EPI_SWIGLU;
  g1.w = W->w1; g1.w_scale = W->w1_scale; g1.bias = W->b1;
  g1.act = x; g1.act_fmt = moe_launch::ACT_BF16; g1.act_scale = x_scale; g1.act_per_pair = 0;
  g1.Nw = 2 * (int64_t)I; g1.Kin = K; g1.Nout = I; g1.k = k; g1.P = P; g1.E = E;
  g1.sorted = sorted_token_ids; g1.expert_ids = expert_ids; g1.ntpp = num_tokens_post_padded;
  g1.bm = block_m; g1.grid_blocks = blocks; g1.topk_w = topk_w; g1.out = hq; g1.out_scale = hs;
  g1.status = status_of(ctx);
  moe_launch::apply_debug_stall(g1);
  moe_launch::GroupedGemm g2 = g1;
  g2.epi = moe_launch::EPI_WEIGHTED_F32;
  g2.w = W->w2; g2.w_scale = W->w2_scale; g2.bias = W->b2;
  g2.act = hq; g2.act_scale = hs; g2.act_per_pair = 1;
  g2.Nw = K; g2.Kin = I; g2.Nout = K; g2.out = o; g2.out_scale = nullptr;
  const bool tc1 = T_rows > moe_launch::kPrefillRowsAbove && moe_launch::mx8_supported(g1);
  const bool tc2 = T_rows > moe_launch::kPrefillRowsAbove && moe_launch::mx8_supported(g2);
  if (!tc1) {
    MOE_REQUIRE(I <= K, MOE_ERR_UNSUPPORTED, "the MXFP8 weight-streaming path keeps fp32 h in the o scratch: needs I <= K");
    MOE_REQUIRE(moe_launch::decode_gemm_smem_bytes(g1) <= 227 * 1024, MOE_ERR_UNSUPPORTED, "K too large for the decode path");
  }
  if (!tc2)
    MOE_REQUIRE(moe_launch::decode_gemm_smem_bytes(g2) <= 227 * 1024, MOE_ERR_UNSUPPORTED, "I too large for the decode path");
  rec(ctx, 0, 4);
  moe_status st;
  if (tc1) {
    st = cuda_status(moe_launch::mx8_gemm(g1, s), "moe_forward GEMM1");
  } else {
    moe_launch::GroupedGemm gf = g1;
    gf.out = o;  // fp32 h, quantised next
    gf.out_scale = nullptr;
    st = cuda_status(moe_launch::decode_gemm(gf, s), "moe_forward GEMM1");
    if (st == MOE_OK) st = cuda_status(moe_launch::mx_quantize(o, P, I, hq, hs, s), "moe_forward quantise h");
  }
  if (st != MOE_OK) return st;
  rec(ctx, 1, 4);
  st = cuda_status(tc2 ? moe_launch::mx8_gemm(g2, s) : moe_launch::decode_gemm(g2, s), "moe_forward GEMM2");
  if (st != MOE_OK) return st;
  rec(ctx, 2, 4);
  st = cuda_status(moe_launch::combine(o, T_real, k, K, y, s), "moe_forward combine");
  rec(ctx, 3, 4);
  return st;
}

moe_status moe_forward(const moe_weights* W, const void* x, const uint8_t* x_scale, int64_t T_rows,
                       int64_t T_real, int32_t k, const float* topk_w,
                       const int32_t* sorted_token_ids, const int32_t* expert_ids,
                       const int32_t* num_tokens_post_padded, const int32_t* expert_offsets,
                       int32_t block_m, int64_t cap_tokens, void* y, const moe_ctx* ctx) {
  (void)expert_offsets;
  MOE_REQUIRE(W && ctx, MOE_ERR_INVALID_ARG, "null weights or context");
  MOE_REQUIRE(W->quant == MOE_Q_BF16 || W->quant == MOE_Q_MXFP4_W4A16 || W->quant == MOE_Q_MXFP8,
              MOE_ERR_INVALID_ARG, "unknown quant mode");
  const int32_t E = W->E, K = W->K, I = W->I;
  MOE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= E, MOE_ERR_INVALID_ARG, "bad E or k");
  MOE_REQUIRE(W->activation == MOE_ACT_SWIGLU || W->activation == MOE_ACT_RELU2, MOE_ERR_INVALID_ARG,
              "unknown activation");
  const bool relu2 = W->activation == MOE_ACT_RELU2;
  MOE_REQUIRE(K >= 32 && I >= 32 && K % 32 == 0 && I % 32 == 0, MOE_ERR_UNSUPPORTED,
              "K and I must be positive multiples of 32");
  MOE_REQUIRE(T_rows >= 0 && T_real >= 0 && T_real <= T_rows, MOE_ERR_INVALID_ARG,
              "need 0 <= T_real <= T_rows");
  MOE_REQUIRE(pairs_fit(T_rows, k), MOE_ERR_UNSUPPORTED, "T_rows*k must be < 2^31");
  MOE_REQUIRE(weights_fit(E, 2 * (int64_t)I, K) && weights_fit(E, K, I), MOE_ERR_UNSUPPORTED,
              "weight arrays too large for 64-bit indexing");
  const bool fp4 = (W->quant == MOE_Q_MXFP4_W4A16);
  MOE_REQUIRE(W->w1 && W->w2 && x && topk_w && y, MOE_ERR_INVALID_ARG, "null tensor pointer");
  MOE_REQUIRE(!fp4 || (W->w1_scale && W->w2_scale), MOE_ERR_INVALID_ARG, "MXFP4 needs scales");
  MOE_REQUIRE(aligned16(W->w1) && aligned16(W->w2) && aligned16(x) && aligned16(topk_w) &&
                  aligned16(y) && aligned16(W->b1) && aligned16(W->b2) &&
                  aligned16(W->w1_scale) && aligned16(W->w2_scale),
              MOE_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  const int64_t P = T_rows * k;
  moe_status st = check_align_outputs(P, E, block_m, sorted_token_ids, expert_ids,
                                      num_tokens_post_padded, cap_tokens);
  if (st != MOE_OK) return st;
  const size_t need = moe_forward_workspace_size(T_rows, k, K, I, cap_tokens);
  MOE_REQUIRE(ctx->workspace && ctx->workspace_bytes >= need && aligned16(ctx->workspace),
              MOE_ERR_CAPACITY, "workspace of %zu bytes needed", need);
  if (T_rows == 0) return MOE_OK;
  if (W->quant == MOE_Q_MXFP8)
    return forward_mxfp8(W, x, x_scale, T_rows, T_real, k, topk_w, sorted_token_ids, expert_ids,
                         num_tokens_post_padded, block_m, cap_tokens, y, ctx);

  int64_t rows_h, rows_x;
  forward_scratch_rows(T_rows, k, cap_tokens, &rows_h, &rows_x);
  uint8_t* ws = static_cast<uint8_t*>(ctx->workspace);
  void* h = ws;
  float* o = reinterpret_cast<float*>(ws + round256((size_t)rows_h * I * 2));
  void* x16 = ws + round256((size_t)rows_h * I * 2) + round256((size_t)P * K * 4);
  cudaStream_t s = stream_of(ctx);
  const int wf = fp4 ? moe_launch::WF_MXFP4 : moe_launch::WF_BF16;
  const int64_t blocks = used_blocks_bound(P, E, block_m, cap_tokens);

  moe_launch::GroupedGemm g1{};
  g1.wfmt = wf;
  g1.epi = relu2 ? moe_launch::EPI_RELU2 : moe_launch::EPI_SWIGLU;
  g1.w = W->w1; g1.w_scale = W->w1_scale; g1.bias = W->b1;
  g1.act = fp4 ? x16 : x;  // the f16 MMA of the MXFP4 path reads x converted once to f16
  g1.act_fmt = fp4 ? moe_launch::ACT_F16 : moe_launch::ACT_BF16;
  g1.act_scale = nullptr; g1.act_per_pair = 0;
  g1.Nw = relu2 ? (int64_t)I : 2 * (int64_t)I; g1.Kin = K; g1.Nout = I; g1.k = k; g1.P = P; g1.E = E;
  g1.sorted = sorted_token_ids; g1.expert_ids = expert_ids; g1.ntpp = num_tokens_post_padded;
  g1.bm = block_m; g1.grid_blocks = blocks; g1.topk_w = topk_w; g1.out = h;
  g1.status = status_of(ctx);
  moe_launch::apply_debug_stall(g1);
  MOE_REQUIRE(moe_launch::decode_gemm_smem_bytes(g1) <= 227 * 1024, MOE_ERR_UNSUPPORTED,
              "K too large for the decode path");
  moe_launch::GroupedGemm g2 = g1;
  g2.epi = moe_launch::EPI_WEIGHTED_F32;
  g2.w = W->w2; g2.w_scale = W->w2_scale; g2.bias = W->b2;
  g2.act = h; g2.act_fmt = fp4 ? moe_launch::ACT_F16 : moe_launch::ACT_BF16; g2.act_per_pair = 1;
  g2.Nw = K; g2.Kin = I; g2.Nout = K; g2.out = o;
  // Above the threshold the MXFP4 path keeps x and h in alignment-slot order: a block of 128
  // slots is then 128 consecutive rows, which the tensor-memory kernel loads as one box.
  uint8_t* fix = nullptr;  // marks of out-of-window weight tiles (tensor-memory kernels)
  size_t fix_bytes = 0;
  if (fp4 && rows_x == rows_h && rows_h > P) {
    moe_launch::GroupedGemm s1 = g1, s2 = g2;
    s1.act_by_slot = 1; s1.out_by_slot = 1;
    s2.act_by_slot = 1;
    if (blocks * block_m <= rows_h && moe_launch::ts_supported(s1) && moe_launch::ts_supported(s2)) {
      g1 = s1;
      g2 = s2;
      const int64_t cap_blocks = cap_tokens / 128;
      fix = static_cast<uint8_t*>(x16) + round256((size_t)rows_x * K * 2);
      const size_t f1 = moe_launch::ts_fix_bytes(cap_blocks, I);
      fix_bytes = f1 + moe_launch::ts_fix_bytes(cap_blocks, K);
      g1.fix_count = reinterpret_cast<int32_t*>(fix);
      g1.fix_bits = reinterpret_cast<uint32_t*>(fix + 256);
      g2.fix_count = reinterpret_cast<int32_t*>(fix + f1);
      g2.fix_bits = reinterpret_cast<uint32_t*>(fix + f1 + 256);
    }
  }
  // Up to 256 rows, MXFP4 with SwiGLU: the block-scaled kernel reads the E2M1 codes as they
  // are stored, with x and h split into E2M1 digit planes
  if (fp4 && !relu2 && !g1.act_by_slot && T_rows <= moe_launch::kPrefillRowsAbove &&
      moe_launch::decode_tc_supported(g1, g2)) {
    const size_t off = round256((size_t)rows_h * I * 2) + round256((size_t)P * K * 4) +
                       round256((size_t)rows_x * K * 2) + forward_fix_bytes(T_rows, k, K, I, cap_tokens);
    const moe_launch::DecodeTcBufs b = moe_launch::decode_tc_carve(ws + off, T_rows, k, K, I);
    st = cuda_status(moe_launch::decode_tc_prep(g1, x, T_rows, b, s), "moe_forward x planes");
    if (st != MOE_OK) return st;
    rec(ctx, 0, 4);
    st = cuda_status(moe_launch::decode_tc_gemm(g1, b, s), "moe_forward GEMM1");
    if (st != MOE_OK) return st;
    rec(ctx, 1, 4);
    st = cuda_status(moe_launch::decode_tc_gemm(g2, b, s), "moe_forward GEMM2");
    if (st != MOE_OK) return st;
    rec(ctx, 2, 4);
    st = cuda_status(moe_launch::combine(o, T_real, k, K, y, s), "moe_forward combine");
    rec(ctx, 3, 4);
    return st;
  }
  if (fix) {
    st = cuda_status(cudaMemsetAsync(fix, 0, fix_bytes, s), "moe_forward marks");
    if (st != MOE_OK) return st;
  }
  if (fp4 && g1.act_by_slot) {
    st = cuda_status(moe_launch::gather_rows_f16(x, sorted_token_ids, num_tokens_post_padded, P, k, K,
                                                 blocks * block_m, x16, status_of(ctx), s),
                     "moe_forward x");
    if (st != MOE_OK) return st;
  } else if (fp4) {
    st = cuda_status(moe_launch::bf16_to_f16(x, x16, T_rows * K, status_of(ctx), s), "moe_forward x");
    if (st != MOE_OK) return st;
  }
  rec(ctx, 0, 4);  // after x's f16 copy: the events bracket the GEMM kernels alone
  st = cuda_status(moe_launch::grouped_gemm(g1, T_rows, s), "moe_forward GEMM1");
  if (st != MOE_OK) return st;
  rec(ctx, 1, 4);
  st = cuda_status(moe_launch::grouped_gemm(g2, T_rows, s), "moe_forward GEMM2");
  if (st != MOE_OK) return st;
  rec(ctx, 2, 4);
  st = cuda_status(moe_launch::combine(o, T_real, k, K, y, s), "moe_forward combine");
  rec(ctx, 3, 4);
  return st;
}

// Block slots a grouped GEMM over P pairs can launch for, whatever E: every used block holds
// a pair, and the launch covers at most P / bm + min(E, P) of them.
static int64_t grouped_blocks_bound(int64_t P) { return P + P / 128 + 1; }

size_t moe_grouped_gemm_workspace_size(moe_quant quant, int64_t T, int32_t k, int32_t N, int32_t Kin,
                                       int32_t a_per_pair) {
  // the W4A16 tensor-memory kernel reads the activations as f16: one converted copy of A, and
  // the marks of out-of-window weight tiles
  if (quant != MOE_Q_MXFP4_W4A16 || T <= moe_launch::kPrefillRowsAbove || k < 1 || N < 1 || Kin < 1) return 0;
  if (!pairs_fit(T, k)) return 0;
  const int64_t rows = a_per_pair ? T * k : T;
  return round256((size_t)rows * Kin * 2) + moe_launch::ts_fix_bytes(grouped_blocks_bound(T * k), N);
}

moe_status moe_grouped_gemm(moe_quant quant, int32_t E, int32_t N, int32_t Kin, const void* a,
                            const uint8_t* a_scale, int32_t a_per_pair, const void* w,
                            const uint8_t* w_scale, const void* bias, int64_t T, int32_t k,
                            const int32_t* sorted_token_ids, const int32_t* expert_ids,
                            const int32_t* num_tokens_post_padded, int32_t block_m,
                            int64_t cap_tokens, void* out, const moe_ctx* ctx) {
  MOE_REQUIRE(quant == MOE_Q_BF16 || quant == MOE_Q_MXFP4_W4A16 || quant == MOE_Q_MXFP8,
              MOE_ERR_INVALID_ARG, "unknown quant mode");
  MOE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= E && T >= 0, MOE_ERR_INVALID_ARG,
              "bad E, k or T");
  MOE_REQUIRE(N >= 16 && N % 16 == 0 && Kin >= 32 && Kin % 32 == 0, MOE_ERR_UNSUPPORTED,
              "N must be a multiple of 16 and Kin of 32");
  MOE_REQUIRE(weights_fit(E, N, Kin), MOE_ERR_UNSUPPORTED, "weight array too large for 64-bit indexing");
  MOE_REQUIRE(pairs_fit(T, k), MOE_ERR_UNSUPPORTED, "T*k must be < 2^31");
  const bool mx8 = quant == MOE_Q_MXFP8, fp4 = quant == MOE_Q_MXFP4_W4A16;
  MOE_REQUIRE(a && w && out, MOE_ERR_INVALID_ARG, "null tensor pointer");
  MOE_REQUIRE(!(mx8 || fp4) || w_scale, MOE_ERR_INVALID_ARG, "MX weights need w_scale");
  MOE_REQUIRE(!mx8 || a_scale, MOE_ERR_INVALID_ARG, "MXFP8 activations need a_scale");
  MOE_REQUIRE(aligned16(a) && aligned16(w) && aligned16(out) && aligned16(bias) &&
                  aligned16(a_scale) && aligned16(w_scale),
              MOE_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  const int64_t P = T * k;
  moe_status st = check_align_outputs(P, E, block_m, sorted_token_ids, expert_ids,
                                      num_tokens_post_padded, cap_tokens);
  if (st != MOE_OK) return st;
  if (P == 0) return MOE_OK;
  moe_launch::GroupedGemm g{};
  g.wfmt = mx8 ? moe_launch::WF_MXFP8 : (fp4 ? moe_launch::WF_MXFP4 : moe_launch::WF_BF16);
  g.epi = moe_launch::EPI_PLAIN_BF16;
  g.w = w; g.w_scale = w_scale; g.bias = bias;
  g.act = a; g.act_fmt = moe_launch::ACT_BF16; g.act_scale = a_scale; g.act_per_pair = a_per_pair ? 1 : 0;
  g.Nw = N; g.Kin = Kin; g.Nout = N; g.k = k; g.P = P; g.E = E;
  g.sorted = sorted_token_ids; g.expert_ids = expert_ids; g.ntpp = num_tokens_post_padded;
  g.bm = block_m; g.grid_blocks = used_blocks_bound(P, E, block_m, cap_tokens);
  g.topk_w = nullptr; g.out = out; g.status = status_of(ctx);
  moe_launch::apply_debug_stall(g);
  // W4A16 above the tensor-memory threshold, with a workspace for the f16 copy of A: the
  // tcgen05 kernel (decoded weights in tensor memory) where it takes the shape
  const size_t ws_need = moe_grouped_gemm_workspace_size(quant, T, k, N, Kin, a_per_pair);
  if (ws_need > 0 && ctx && ctx->workspace && ctx->workspace_bytes >= ws_need && aligned16(ctx->workspace)) {
    moe_launch::GroupedGemm gt = g;
    gt.act = ctx->workspace;
    gt.act_fmt = moe_launch::ACT_F16;
    const int64_t rows = a_per_pair ? P : T;
    uint8_t* fix = static_cast<uint8_t*>(ctx->workspace) + round256((size_t)rows * Kin * 2);
    gt.fix_count = reinterpret_cast<int32_t*>(fix);
    gt.fix_bits = reinterpret_cast<uint32_t*>(fix + 256);
    if (moe_launch::ts_supported(gt)) {
      rec(ctx, 0, 2);
      st = cuda_status(cudaMemsetAsync(fix, 0, moe_launch::ts_fix_bytes(grouped_blocks_bound(P), N), stream_of(ctx)),
                       "moe_grouped_gemm marks");
      if (st == MOE_OK)
        st = cuda_status(moe_launch::bf16_to_f16(a, ctx->workspace, rows * Kin, status_of(ctx), stream_of(ctx)),
                         "moe_grouped_gemm activations");
      if (st == MOE_OK) st = cuda_status(moe_launch::prefill_ts(gt, stream_of(ctx)), "moe_grouped_gemm");
      rec(ctx, 1, 2);
      return st;
    }
  }
  MOE_REQUIRE(moe_launch::decode_gemm_smem_bytes(g) <= 227 * 1024, MOE_ERR_UNSUPPORTED,
              "Kin too large for the decode path");
  rec(ctx, 0, 2);
  st = cuda_status(moe_launch::grouped_gemm(g, T, stream_of(ctx)), "moe_grouped_gemm");
  rec(ctx, 1, 2);
  return st;
}

moe_status moe_mx_quantize(const float* x, int64_t rows, int32_t cols, uint8_t* codes, uint8_t* scales,
                           const moe_ctx* ctx) {
  MOE_REQUIRE(rows >= 0 && cols >= 32 && cols % 32 == 0, MOE_ERR_INVALID_ARG,
              "need rows >= 0 and cols a positive multiple of 32");
  MOE_REQUIRE(x && codes && scales, MOE_ERR_INVALID_ARG, "null tensor pointer");
  MOE_REQUIRE(aligned16(x) && aligned16(codes) && aligned16(scales), MOE_ERR_INVALID_ARG,
              "all pointers must be 16-byte aligned");
  return cuda_status(moe_launch::mx_quantize(x, rows, cols, codes, scales, stream_of(ctx)), "moe_mx_quantize");
}

moe_status moe_gemm_per_token(int32_t E, int32_t N, int32_t K, const uint8_t* a, const float* a_scale,
                              const uint8_t* w, const float* w_scale, const void* bias,
                              const int32_t* group_sizes, int64_t M, void* out, const moe_ctx* ctx) {
  MOE_REQUIRE(E >= 1 && E <= 1024 && M >= 0, MOE_ERR_INVALID_ARG, "need 1 <= E <= 1024 and M >= 0");
  MOE_REQUIRE(N >= 128 && N % 128 == 0 && K >= 128 && K % 128 == 0, MOE_ERR_UNSUPPORTED,
              "N and K must be positive multiples of 128");
  MOE_REQUIRE(M < ((int64_t)1 << 31) && (int64_t)E * N < ((int64_t)1 << 31), MOE_ERR_UNSUPPORTED,
              "M and E*N must be < 2^31");
  MOE_REQUIRE(a && a_scale && w && w_scale && group_sizes && out, MOE_ERR_INVALID_ARG, "null tensor pointer");
  MOE_REQUIRE(aligned16(a) && aligned16(a_scale) && aligned16(w) && aligned16(w_scale) && aligned16(bias) &&
                  aligned16(group_sizes) && aligned16(out),
              MOE_ERR_INVALID_ARG, "all pointers must be 16-byte aligned");
  if (M == 0) return MOE_OK;
  moe_launch::PerTokenGemm g{};
  g.E = E; g.N = N; g.K = K; g.M = M;
  g.a = a; g.a_scale = a_scale; g.w = w; g.w_scale = w_scale; g.bias = bias;
  g.group_sizes = group_sizes; g.out = out; g.status = status_of(ctx);
  rec(ctx, 0, 2);
  moe_status st = cuda_status(moe_launch::pertoken_gemm(g, stream_of(ctx)), "moe_gemm_per_token");
  rec(ctx, 1, 2);
  return st;
}

// The slot-ordered copies of grad and input that let the tensor-memory wgrad load whole
// stages by TMA: [cap_tokens, N] and [cap_tokens, Kin] bf16, then the experts' block ranges
// [E][2] int32, each 256-byte aligned.
static moe_launch::Wgrad wgrad_shape(int32_t E, int32_t N, int32_t Kin, int32_t block_m, int64_t cap_tokens,
                                     int32_t mode) {
  moe_launch::Wgrad g{};
  g.E = E; g.N = N; g.Kin = Kin; g.bm = block_m; g.cap = cap_tokens; g.mode = mode;
  return g;
}

size_t moe_wgrad_workspace_size(int32_t E, int32_t N, int32_t Kin, int32_t block_m, int64_t cap_tokens,
                                int32_t mode) {
  if (E < 1 || N < 64 || Kin < 64 || block_m < 1 || cap_tokens < 1) return 0;
  if (!moe_launch::wgrad_tc_slot_feed(wgrad_shape(E, N, Kin, block_m, cap_tokens, mode))) return 0;
  return round256((size_t)cap_tokens * N * 2) + round256((size_t)cap_tokens * Kin * 2) + round256((size_t)E * 8);
}

moe_status moe_wgrad(const void* grad, const void* input, int32_t input_per_pair, int64_t T,
                     int32_t k, int32_t E, int32_t N, int32_t Kin, const int32_t* sorted_token_ids,
                     const int32_t* expert_ids, const int32_t* num_tokens_post_padded,
                     int32_t block_m, int64_t cap_tokens, float* dW, int32_t mode,
                     const moe_ctx* ctx) {
  MOE_REQUIRE(mode == 0 || mode == 1, MOE_ERR_INVALID_ARG, "mode must be 0 or 1");
  MOE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= E && T >= 0, MOE_ERR_INVALID_ARG,
              "bad E, k or T");
  MOE_REQUIRE(N >= 64 && N % 64 == 0 && Kin >= 64 && Kin % 64 == 0, MOE_ERR_UNSUPPORTED,
              "N and Kin must be multiples of 64");
  MOE_REQUIRE(N / 64 <= 65535 && Kin / 64 <= 65535, MOE_ERR_UNSUPPORTED, "N or Kin too large");
  MOE_REQUIRE(pairs_fit(T, k), MOE_ERR_UNSUPPORTED, "T*k must be < 2^31");
  MOE_REQUIRE(grad && input && dW, MOE_ERR_INVALID_ARG, "null tensor pointer");
  MOE_REQUIRE(aligned16(grad) && aligned16(input) && aligned16(dW), MOE_ERR_INVALID_ARG,
              "all pointers must be 16-byte aligned");
  const int64_t P = T * k;
  moe_status st = check_align_outputs(P, E, block_m, sorted_token_ids, expert_ids,
                                      num_tokens_post_padded, cap_tokens);
  if (st != MOE_OK) return st;
  const int64_t cap_blocks = cap_tokens / block_m;
  MOE_REQUIRE(mode == 0 || cap_blocks <= 65535, MOE_ERR_UNSUPPORTED,
              "accumulate mode supports at most 65535 block slots");
  moe_launch::Wgrad g{};
  g.grad = grad; g.input = input; g.input_per_pair = input_per_pair ? 1 : 0;
  g.P = P; g.k = k; g.E = E; g.N = N; g.Kin = Kin;
  g.sorted = sorted_token_ids; g.expert_ids = expert_ids; g.ntpp = num_tokens_post_padded;
  g.bm = block_m; g.cap_blocks = cap_blocks; g.dW = dW; g.mode = mode; g.status = status_of(ctx);
  g.cap = cap_tokens;
  moe_launch::apply_debug_stall(g);
  rec(ctx, 0, 2);
  // With a workspace: grad and input copied into slot order first, then the tensor-memory
  // kernel loads whole 64-slot stages by TMA (the same MMAs in the same order: same bits).
  const size_t ws_need = moe_wgrad_workspace_size(E, N, Kin, block_m, cap_tokens, mode);
  if (ws_need > 0 && ctx && ctx->workspace && ctx->workspace_bytes >= ws_need && aligned16(ctx->workspace)) {
    uint8_t* ws = static_cast<uint8_t*>(ctx->workspace);
    void* grad_s = ws;
    void* input_s = ws + round256((size_t)cap_tokens * N * 2);
    st = cuda_status(moe_launch::gather_slot_rows(grad, (int64_t)N * 2, sorted_token_ids, num_tokens_post_padded,
                                                  P, 1, cap_tokens, grad_s, stream_of(ctx)),
                     "moe_wgrad grad rows");
    if (st == MOE_OK)
      st = cuda_status(moe_launch::gather_slot_rows(input, (int64_t)Kin * 2, sorted_token_ids,
                                                    num_tokens_post_padded, P, input_per_pair ? 1 : k, cap_tokens,
                                                    input_s, stream_of(ctx)),
                       "moe_wgrad input rows");
    if (st != MOE_OK) return st;
    g.grad_s = grad_s;
    g.input_s = input_s;
    g.ranges = reinterpret_cast<int32_t*>(ws + round256((size_t)cap_tokens * N * 2) +
                                          round256((size_t)cap_tokens * Kin * 2));
  }
  st = cuda_status(moe_launch::wgrad(g, stream_of(ctx)), "moe_wgrad");
  rec(ctx, 1, 2);
  return st;
}

void moe_debug_stall_tensor_kernels(int64_t stall_ns) {
  moe_launch::g_debug_stall_ns.store(stall_ns > 0 ? stall_ns : 0, std::memory_order_relaxed);
}

}  // extern "C"
