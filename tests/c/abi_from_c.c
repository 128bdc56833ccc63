/* The library used from plain C (C11, no C++ and no CUDA headers): the header compiles as C
 * and the host-side entry points behave as documented.  Nothing here touches a GPU:
 * every call below either runs on the host or is refused before any launch.
 * Prints "ok" and returns 0, or names the first failed check and returns 1. */
#include <stdio.h>
#include <string.h>

#include "dit.h"

#define CHECK(cond)                                           \
  do {                                                        \
    if (!(cond)) {                                            \
      printf("failed: %s (line %d)\n", #cond, __LINE__);      \
      return 1;                                               \
    }                                                         \
  } while (0)

int main(void) {
  dit_config cfg;
  memset(&cfg, 0, sizeof cfg);
  CHECK(dit_config_klein(&cfg) == DIT_OK);
  CHECK(cfg.hidden == 3072 && cfg.heads == 24 && cfg.head_dim == 128 && cfg.mlp_hidden == 9216);
  CHECK(cfg.n_dual == 5 && cfg.n_single == 20 && cfg.in_channels == 128 && cfg.txt_dim == 7680);
  CHECK(cfg.axes_dim[0] == 32 && cfg.axes_dim[3] == 32 && cfg.rope_theta == 2000.0f);

  /* workspace sizes: defined for a valid shape, growing with the tokens and the batch */
  dit_shape small = {1, 512, 4096, 0}, more = {1, 512, 8192, 0}, two = {2, 512, 4096, 0};
  size_t a = 0, b = 0, c = 0;
  CHECK(dit_workspace_size(&cfg, &small, &a) == DIT_OK && a > 0);
  CHECK(dit_workspace_size(&cfg, &more, &b) == DIT_OK && b > a);
  CHECK(dit_workspace_size(&cfg, &two, &c) == DIT_OK && c > a);

  /* refused shapes and configurations */
  dit_shape bad = {0, 512, 4096, 0}, huge = {1, 512, 1 << 20, 0};
  CHECK(dit_workspace_size(&cfg, &bad, &a) == DIT_ERR_INVALID_ARG);
  CHECK(dit_workspace_size(&cfg, &huge, &a) == DIT_ERR_UNSUPPORTED);
  CHECK(dit_workspace_size(NULL, &small, &a) == DIT_ERR_INVALID_ARG);
  dit_config odd = cfg;
  odd.head_dim = 64;
  CHECK(dit_workspace_size(&odd, &small, &a) == DIT_ERR_UNSUPPORTED);

  /* token ids of a small joint sequence: text rows (0, 0, 0, i), the target grid
   * (0, r, c, 0), then reference 0 at t = 10 */
  dit_shape s = {1, 2, 4, 2};
  const int ref_grid[2] = {1, 2};
  int32_t ids[8 * 4];
  CHECK(dit_token_ids(&s, 2, 2, ref_grid, 1, ids) == DIT_OK);
  CHECK(ids[0] == 0 && ids[3] == 0 && ids[4 + 3] == 1);             /* text rows */
  CHECK(ids[2 * 4 + 1] == 0 && ids[5 * 4 + 1] == 1 && ids[5 * 4 + 2] == 1); /* grid (1, 1) */
  CHECK(ids[6 * 4] == 10 && ids[7 * 4 + 2] == 1);                    /* reference, t = 10 */
  CHECK(dit_token_ids(&s, 3, 2, ref_grid, 1, ids) == DIT_ERR_INVALID_ARG); /* 6 != n_img */

  /* entry points that would launch are refused on bad arguments before touching memory */
  void* fake = (void*)(uintptr_t)0x10000;
  CHECK(dit_attention(1, 2, 10, fake, fake, fake, fake, 200, fake, 256, NULL) == DIT_ERR_INVALID_ARG);
  CHECK(dit_linear(1, 10, 64, 60, fake, fake, fake, 64, DIT_EPI_STORE, NULL, 0, fake, 256, NULL) ==
        DIT_ERR_INVALID_ARG);
  CHECK(dit_adaln(1, 4, 300, fake, 4, 0, 0, fake, fake, fake, fake, 0, 1e-6f, fake, NULL) == DIT_ERR_UNSUPPORTED);

  CHECK(strlen(dit_status_string(DIT_ERR_TIMEOUT)) > 0);
  printf("ok\n");
  return 0;
}
