/* Plain C11 client of the C ABI (include/ltk.h): compiles as C, links against
 * libltk.so and calls the host-only entry points -- no GPU needed.  Prints
 * "abi ok" and exits 0 when every check holds; otherwise names the failing
 * check and exits 1. */
#include <stdio.h>
#include <string.h>

#include "ltk.h"

static int failures = 0;

static void expect(int cond, const char* what) {
  if (!cond) {
    fprintf(stderr, "FAILED: %s\n", what);
    ++failures;
  }
}

int main(void) {
  expect(ltk_abi_version() == LTK_ABI_VERSION, "abi version");
  expect(strcmp(ltk_status_string(LTK_OK), "ok") == 0, "status string of LTK_OK");

  ltk_config cfg;
  expect(ltk_config_init(&cfg, 64, 128, 2048, 8192, 1LL << 20) == LTK_OK, "config init");
  expect(cfg.relu == 1 && cfg.causal == 1 && cfg.dtype == LTK_BF16, "indexer defaults");

  unsigned long long bytes = 0;
  expect(ltk_workspace_bytes(&cfg, &bytes) == LTK_OK && bytes > (1ULL << 30), "workspace bytes");

  ltk_config bad = cfg;
  bad.k = 0;
  expect(ltk_workspace_bytes(&bad, &bytes) == LTK_ERR_ARG, "k = 0 rejected");
  bad = cfg;
  bad.n_bins = 100;
  expect(ltk_workspace_bytes(&bad, &bytes) == LTK_ERR_ARG, "n_bins not a power of two rejected");

  ltk_config one;
  expect(ltk_config_init(&one, 1, 768, 1000, 1024, 8388608LL) == LTK_OK, "retrieval config");
  expect(one.relu == 0 && one.causal == 0, "retrieval defaults: plain inner product, no mask");

  /* calls without a handle are rejected on the host, before any CUDA work */
  ltk_handle* h = NULL;
  expect(ltk_create(NULL, &h) == LTK_ERR_ARG && h == NULL, "create without a config");
  expect(ltk_indexer_topk(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 10, NULL, 0, 1, NULL, NULL,
                          NULL) == LTK_ERR_ARG, "fused call without a handle");
  ltk_stats st;
  expect(ltk_get_stats(NULL, &st) == LTK_ERR_ARG, "stats without a handle");
  expect(ltk_decoupled_topk_noalloc(7, 1, NULL, NULL, NULL, NULL, NULL, NULL, 1, 10, 1, NULL, NULL,
                                    NULL, NULL) == LTK_ERR_ARG, "allocation-free call with a bad dtype");
  expect(ltk_decoupled_topk_noalloc(LTK_BF16, 1, NULL, NULL, NULL, NULL, NULL, NULL, 4096, 4096, 1,
                                    NULL, NULL, NULL, NULL) == LTK_ERR_ARG,
         "allocation-free call beyond its static array");
  expect(ltk_litedsa_pack(NULL, 4, 8, 0, NULL, NULL, NULL, NULL) == LTK_ERR_ARG, "LiteDSA group 0");
  expect(ltk_litedsa_pack(NULL, 4, 8192, 8, NULL, NULL, NULL, NULL) == LTK_ERR_UNSUPPORTED,
         "LiteDSA group beyond 16384 keys");
  ltk_destroy(NULL);

  if (failures == 0) printf("abi ok\n");
  return failures == 0 ? 0 : 1;
}
