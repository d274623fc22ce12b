/* A plain C11 user of libquail: includes only quail.h, links only libquail.so, and calls
 * the host-side entry points (no GPU needed). Prints one line per check; exit status 0
 * when every check holds. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "quail.h"

static int failures = 0;
#define CHECK(cond, what)                                       \
  do {                                                          \
    if (cond) {                                                 \
      printf("ok %s\n", what);                                  \
    } else {                                                    \
      printf("FAILED %s\n", what);                              \
      ++failures;                                               \
    }                                                           \
  } while (0)

int main(void) {
  CHECK(strncmp(quail_version(), "quail-gb300", 11) == 0, "version");
  CHECK(strcmp(quail_status_string(QUAIL_ERR_TIMEOUT), "QUAIL_ERR_TIMEOUT") == 0,
        "status string");

  /* descriptor of a small join; the workspace holds at least the schedule */
  quail_cascade_desc d;
  memset(&d, 0, sizeof d);
  d.num_anchors = 2;
  d.num_suffixes = 3;
  d.total_anchor_tokens = 100;
  d.total_suffix_tokens = 40;
  d.max_anchor_len = 60;
  d.max_suffix_len = 20;
  d.num_q_heads = 32;
  d.num_kv_heads = 8;
  d.head_dim = 128;
  d.kv_anchor_dtype = QUAIL_BF16;
  const size_t ws_bf16 = quail_cascade_workspace_size(&d);
  d.kv_anchor_dtype = QUAIL_FP8_E4M3;
  const size_t ws_fp8 = quail_cascade_workspace_size(&d);
  CHECK(ws_bf16 > 0 && ws_bf16 % 256 == 0, "workspace size");
  CHECK(ws_fp8 >= ws_bf16 + (size_t)4 * 100 * 8 * 128, "fp8 workspace holds the staged anchors");
  /* argument errors come back synchronously, before any device work */
  CHECK(quail_cascade_attn(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                           NULL, NULL, NULL, 0, NULL) == QUAIL_ERR_INVALID_ARG,
        "null descriptor rejected");

  /* shard three anchors over two ranks: work 19, 3 and 0 visible pairs */
  const int32_t ao[4] = {0, 3, 3, 10}, asp[4] = {0, 2, 3, 3}, so[4] = {0, 1, 4, 6};
  int32_t rank_of[3];
  int64_t pairs[2];
  CHECK(quail_shard_anchors(3, ao, asp, so, 2, rank_of, pairs) == QUAIL_OK, "shard call");
  CHECK(rank_of[0] == 0 && rank_of[1] == 1 && rank_of[2] == 1, "shard plan");
  CHECK(pairs[0] == 19 && pairs[1] == 3, "shard loads");
  /* rank 1's sub-batch: anchors 1 and 2 (0 and 7 tokens) with suffixes 2 (2 tokens) */
  quail_shard_sizes sz;
  CHECK(quail_shard_batch(3, ao, asp, so, rank_of, 1, &sz, NULL, NULL, NULL, NULL, NULL,
                          NULL) == QUAIL_OK &&
            sz.num_anchors == 2 && sz.num_suffixes == 1 && sz.anchor_tokens == 7 &&
            sz.suffix_tokens == 2,
        "sub-batch sizes");
  int32_t sao[3], sasp[3], sso[2], anc[2];
  int64_t arows[7], srows[2];
  CHECK(quail_shard_batch(3, ao, asp, so, rank_of, 1, &sz, sao, sasp, sso, anc, arows,
                          srows) == QUAIL_OK &&
            sao[1] == 0 && sao[2] == 7 && sasp[1] == 1 && sasp[2] == 1 && sso[1] == 2 &&
            anc[0] == 1 && anc[1] == 2 && arows[0] == 3 && srows[0] == 4 && srows[1] == 5,
        "sub-batch arrays");

  /* cache plan: anchors of 4, 4 and 2 tokens, capacity 8, accesses 0 1 2 0 1 */
  const int64_t size[3] = {4, 4, 2};
  const int32_t acc[5] = {0, 1, 2, 0, 1};
  uint8_t hit[5];
  quail_kv_plan_stats st;
  CHECK(quail_kv_plan(3, size, 5, acc, 8, QUAIL_KV_FURTHEST_NEXT_USE, hit, &st) == QUAIL_OK,
        "kv plan call");
  /* anchor 2 is never used again, so it is bypassed: both later accesses hit */
  CHECK(st.hits == 2 && st.regret_tokens == 0 && st.compulsory_tokens == 10, "kv plan stats");
  CHECK(quail_kv_plan(3, size, 5, acc, 8, QUAIL_KV_LRU, hit, &st) == QUAIL_OK &&
            st.regret_tokens > 0,
        "lru regrets");
  /* kernel choice for head_dim 128: the three modes, anything else rejected */
  CHECK(quail_set_cta_pairs(QUAIL_CTA_PAIRS_OFF) == QUAIL_OK &&
            quail_set_cta_pairs(QUAIL_CTA_PAIRS_ALWAYS) == QUAIL_OK &&
            quail_set_cta_pairs(7) == QUAIL_ERR_INVALID_ARG &&
            quail_set_cta_pairs(QUAIL_CTA_PAIRS_AUTO) == QUAIL_OK,
        "cta pair modes");
  return failures == 0 ? 0 : 1;
}
