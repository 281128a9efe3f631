/* A plain C program built against include/moe_gb300.h and linked with libmoe_gb300.so.
 * It calls only the host-side entry points (bucket math, capacities, workspace sizes,
 * argument validation), so it runs without a GPU.  It prints one line per check and exits
 * non-zero on the first mismatch.  Expected values are written out from the definitions
 * stated in the header: bucket(m) = ceil(m/s)*s with s = max(1, 2^(floor(log2 m)-3));
 * cap = round_up(P + E*(bm-1), bm). */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "moe_gb300.h"

static int failures = 0;

#define CHECK(cond, ...)                   \
  do {                                     \
    if (!(cond)) {                         \
      printf("FAIL %s:%d: ", __FILE__, __LINE__); \
      printf(__VA_ARGS__);                 \
      printf("\n");                        \
      ++failures;                          \
    }                                      \
  } while (0)

static int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

int main(void) {
  /* bucket values at the edges of the octaves */
  static const int64_t m_in[] = {1, 15, 16, 17, 18, 19, 20, 31, 32, 33, 35, 4097, 20000, 58879, 65536};
  static const int64_t b_out[] = {1, 15, 16, 18, 18, 20, 20, 32, 32, 36, 36, 4608, 20480, 61440, 65536};
  for (size_t i = 0; i < sizeof(m_in) / sizeof(m_in[0]); ++i)
    CHECK(moe_bucket(m_in[i]) == b_out[i], "moe_bucket(%lld) = %lld, want %lld", (long long)m_in[i],
          (long long)moe_bucket(m_in[i]), (long long)b_out[i]);
  CHECK(moe_bucket(0) == -1, "moe_bucket(0) must be -1");
  CHECK(moe_bucket_count(20000) == 97, "moe_bucket_count(20000) = %lld", (long long)moe_bucket_count(20000));
  CHECK(moe_bucket_count(16) == 16, "moe_bucket_count(16) = %lld", (long long)moe_bucket_count(16));

  /* alignment capacity */
  int64_t ct = 0, cb = 0;
  CHECK(moe_align_capacity(256, 128, 128, &ct, &cb) == MOE_OK, "moe_align_capacity failed");
  CHECK(ct == round_up(256 + 128 * 127, 128) && cb == ct / 128, "capacity %lld/%lld", (long long)ct,
        (long long)cb);
  CHECK(moe_align_capacity(65536, 256, 128, &ct, &cb) == MOE_OK && ct == 98048 && cb == 766,
        "capacity of 65536 pairs over 256 experts: %lld/%lld", (long long)ct, (long long)cb);
  CHECK(moe_align_capacity(-1, 4, 16, &ct, &cb) == MOE_ERR_INVALID_ARG, "negative pairs accepted");
  CHECK(strlen(moe_last_error()) > 0, "no error text after a failed call");

  /* workspace of the 64-token decode layer: h f16 [P, I] + o fp32 [P, K] + x f16 [T, K], then
   * x digit planes [T, 8, 1472] + x scales [T, 96] + h planes [P, 8, 1472] + h scales [P, 96] +
   * the unit list [P + 1, 16] of the block-scaled kernel */
  CHECK(moe_align_capacity(256, 128, 128, &ct, &cb) == MOE_OK, "capacity");
  size_t ws = moe_forward_workspace_size(64, 4, 2880, 2880, ct);
  size_t want = (size_t)round_up(256 * 2880 * 2, 256) + (size_t)round_up(256 * 2880 * 4, 256) +
                (size_t)round_up(64 * 2880 * 2, 256) + (size_t)round_up(64 * 8 * 1472, 256) +
                (size_t)round_up(64 * 96, 256) + (size_t)round_up(256 * 8 * 1472, 256) +
                (size_t)round_up(256 * 96, 256) + (size_t)round_up(257 * 16, 256);
  CHECK(ws == want, "workspace %zu, want %zu", ws, want);

  /* wgrad's slot-ordered copies [cap, N] + [cap, Kin] bf16 and expert ranges [E, 2] int32 */
  CHECK(moe_wgrad_workspace_size(256, 4096, 7168, 128, 98048, 0) ==
            (size_t)round_up(98048LL * 4096 * 2, 256) + (size_t)round_up(98048LL * 7168 * 2, 256) +
                (size_t)round_up(256 * 8, 256),
        "wgrad workspace %zu", moe_wgrad_workspace_size(256, 4096, 7168, 128, 98048, 0));
  CHECK(moe_wgrad_workspace_size(256, 4096, 7168, 128, 98048, 1) == 0, "accumulate mode needs no workspace");

  /* bucket padding host math: W4A16 pads, the other modes warn and keep T */
  int64_t tp = 0;
  CHECK(moe_bucket_pad(58879, MOE_Q_MXFP4_W4A16, &tp, NULL, NULL, 0, NULL, NULL, 0, NULL) == MOE_OK &&
            tp == 61440, "pad of 58879 rows: %lld", (long long)tp);
  CHECK(moe_bucket_pad(17, MOE_Q_MXFP8, &tp, NULL, NULL, 0, NULL, NULL, 0, NULL) == MOE_WARN_PAD_IGNORED &&
            tp == 17, "MXFP8 padding must be refused");

  /* argument validation returns before any launch */
  moe_ctx ctx;
  memset(&ctx, 0, sizeof(ctx));
  CHECK(moe_align(NULL, NULL, NULL, 4, 2, 8, 16, NULL, 0, NULL, NULL, NULL, &ctx) == MOE_ERR_INVALID_ARG,
        "null topk_ids accepted");
  CHECK(moe_forward(NULL, NULL, NULL, 0, 0, 1, NULL, NULL, NULL, NULL, NULL, 16, 0, NULL, &ctx) ==
            MOE_ERR_INVALID_ARG, "null weights accepted");
  CHECK(moe_wgrad(NULL, NULL, 0, 4, 2, 8, 64, 64, NULL, NULL, NULL, 16, 0, NULL, 2, &ctx) ==
            MOE_ERR_INVALID_ARG, "bad wgrad mode accepted");

  printf("%s: %d failure(s)\n", failures ? "FAIL" : "ok", failures);
  return failures ? 1 : 0;
}
