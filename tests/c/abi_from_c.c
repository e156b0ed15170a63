/* Plain C99 user of the C ABI: compiles against include/fm.h, links libfm.so
 * and calls the entry points that need no GPU (size helpers, index widths,
 * argument validation).  Prints "ok" and exits 0 when every check holds. */
#include <stdio.h>

#include "fm.h"

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
      return 1;                                                  \
    }                                                            \
  } while (0)

int main(void) {
  void* fake = (void*)0x10000; /* never dereferenced: validation fails first */
  CHECK(fm_version() > 0);
  CHECK(fm_num_kv_tiles_bound(8192, 10, 128) == 8192 / 128 + 10);
  CHECK(fm_attn_fwd_workspace_size(8192, 10, 32, 128) % 256 == 0);
  CHECK(fm_attn_index_bits(131072, 32, 8, 128, 0) == 32);
  CHECK(fm_attn_index_bits(131072, 32, 8, 128, FM_FLAG_FORCE_INT64) == 64);
  CHECK(fm_rope_index_bits((int64_t)1 << 21, 8, 128, 1024, 1024, 0) == 64);
  /* head_dim 96 is not supported; a NULL q is an invalid argument */
  CHECK(fm_rope_qk_varlen(fake, fake, 16, 1, 1, 96, 96, 96, (const int32_t*)fake, 1, 1e4, 0, 0,
                          NULL) == FM_ERR_UNSUPPORTED);
  CHECK(fm_rope_qk_varlen(NULL, fake, 16, 1, 1, 64, 64, 64, (const int32_t*)fake, 1, 1e4, 0, 0,
                          NULL) == FM_ERR_INVALID_ARG);
  CHECK(fm_attn_fwd_varlen_rope(fake, fake, fake, 256, 4, 2, 128, (const int32_t*)fake, 2, 0.0,
                                NULL, 0, NULL, 1, 0.0f, 128, 128, fake, (float*)fake, NULL, NULL,
                                fake, 1 << 20, 0, NULL) == FM_ERR_INVALID_ARG);
  /* a plan needs a workspace of fm_attn_fwd_workspace_size bytes */
  CHECK(fm_attn_fwd_plan(8192, 32, 8, (const int32_t*)fake, 8, NULL, 0, NULL, 1, 128, 128, fake,
                         64, NULL) == FM_ERR_WORKSPACE);
  printf("ok %s\n", fm_status_string(FM_ERR_WORKSPACE));
  return 0;
}
