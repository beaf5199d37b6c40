/* A plain C consumer of libmoe: includes include/moe_layer.h, links libmoe.so and calls the
 * entry points whose work ends before any CUDA call (status names, NULL handles, argument
 * checks). Built and run by tests/test_abi.py on a machine without a GPU. Exit status 0 on
 * success, else the number of the first failed check. */
#include <stdio.h>
#include <string.h>

#include "moe_layer.h"

static int check(int ok, int id) {
  if (!ok) fprintf(stderr, "check %d failed\n", id);
  return ok ? 0 : id;
}

int main(void) {
  static const char* names[] = {"MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_OOM",
                                "MOE_ERR_CUDA", "MOE_ERR_TIMEOUT", "MOE_ERR_DEVICE_CHECK"};
  int rc = 0;
  for (int s = 0; s <= 6 && !rc; ++s) rc = check(strcmp(moe_status_string((moe_status)s), names[s]) == 0, 1 + s);
  if (rc) return rc;
  if ((rc = check(strcmp(moe_status_string((moe_status)42), "MOE_ERR_UNKNOWN") == 0, 10))) return rc;

  moe_layer_destroy(NULL);                                   /* a no-op */
  moe_config cfg;
  moe_weights w;
  memset(&cfg, 0, sizeof cfg);                               /* hidden = 0 */
  memset(&w, 0, sizeof w);
  moe_layer* layer = (moe_layer*)&cfg;                       /* must come back NULL */
  if ((rc = check(moe_layer_create(&cfg, &w, NULL, &layer) == MOE_ERR_INVALID_ARG, 11))) return rc;
  if ((rc = check(layer == NULL, 12))) return rc;
  cfg.hidden = 6144; cfg.inter = 2048; cfg.n_experts = 256; cfg.top_k = 8; cfg.n_group = 8;
  cfg.topk_group = 4; cfg.max_tokens = 64; cfg.routed_scaling_factor = 2.5f;
  cfg.weight_format = 7;                                     /* no such format */
  if ((rc = check(moe_layer_create(&cfg, &w, NULL, &layer) == MOE_ERR_UNSUPPORTED, 13))) return rc;
  if ((rc = check(moe_layer_create(NULL, &w, NULL, &layer) == MOE_ERR_INVALID_ARG, 14))) return rc;
  if ((rc = check(moe_layer_forward(NULL, NULL, 1, NULL, NULL) == MOE_ERR_INVALID_ARG, 15))) return rc;
  if ((rc = check(moe_layer_status(NULL) == MOE_ERR_INVALID_ARG, 16))) return rc;
  if ((rc = check(moe_route_noalloc(NULL, 0, -1, 256, NULL, 0, NULL, 16, 4, 2, 4, 2.5f, NULL, NULL, NULL,
                                    NULL, NULL) == MOE_ERR_INVALID_ARG, 17)))
    return rc;
  printf("ok\n");
  return 0;
}
