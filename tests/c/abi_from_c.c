/* A plain C caller of the library (no Python, no torch): the boundary is usable
 * from C as declared in include/hs.h.  Runs without a GPU: it exercises only the
 * host-side checks that come before any device work.  Exit status 0 = all good. */
#include <stdio.h>
#include <string.h>

#include "hs.h"

static int fails = 0;
#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      fprintf(stderr, "check failed: %s (line %d)\n", #c, __LINE__); \
      ++fails;                                                \
    }                                                         \
  } while (0)

int main(void) {
  hs_config_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n_layers = 1;
  cfg.max_requests = 2;
  cfg.max_context = 4096;
  cfg.h_q = 32;
  cfg.h_kv = 8;
  cfg.d_qk = 128;
  cfg.d_v = 128;
  cfg.d_idx = 128;
  cfg.top_k = 256;
  cfg.hot_slots = 512;
  cfg.replacement = HS_REPLACE_LRU;

  hs_handle_t* h = NULL;
  /* top_k above hot_slots: rejected before any device work, nothing allocated */
  cfg.top_k = 1024;
  CHECK(hs_create(&cfg, &h) == HS_ERR_CONFIG);
  CHECK(h == NULL);
  CHECK(strlen(hs_last_error(NULL)) > 0);
  cfg.top_k = 256;
  /* an unknown replacement policy */
  cfg.replacement = 7;
  CHECK(hs_create(&cfg, &h) == HS_ERR_CONFIG);
  cfg.replacement = HS_REPLACE_RANDOM;
  /* null arguments */
  CHECK(hs_create(NULL, &h) == HS_ERR_INVALID);
  CHECK(hs_create(&cfg, NULL) == HS_ERR_INVALID);
  CHECK(hs_stats(NULL, NULL) == HS_ERR_INVALID);
  /* the status names */
  CHECK(strcmp(hs_status_string(HS_OK), "HS_OK") == 0);
  CHECK(strcmp(hs_status_string(HS_ERR_CONFIG), "HS_ERR_CONFIG") == 0);
  /* the entry point that allocates nothing rejects bad shapes on the host */
  CHECK(hs_indexer_topk_static(65, 16, 128, 8, NULL, NULL, NULL, NULL, 0, NULL) != HS_OK);
  CHECK(hs_indexer_topk_static_error(0, NULL) == HS_ERR_INVALID);
  hs_destroy(NULL); /* a no-op */
  if (fails == 0) printf("abi_from_c: ok\n");
  return fails == 0 ? 0 : 1;
}
