/* Calls the library through include/oasis.h from plain C99, with no GPU work:
 * the version string, then calls whose arguments the library must reject
 * before launching anything.  Prints one "name status" line per call. */
#include <stddef.h>
#include <stdio.h>

#include "oasis.h"

static void report(const char* name, oasis_status st) { printf("%s %d\n", name, (int)st); }

int main(void) {
  printf("version %s\n", oasis_version());

  oasis_shape ok = {2, 32, 8, 128, 16, 256, 4, 32, 32};
  oasis_shape bad_d = ok;
  bad_d.d = 64;
  oasis_shape bad_group = ok;
  bad_group.Hq = 30;

  /* NULL device pointers: invalid; unsupported head dim; ragged GQA group */
  report("score_null", oasis_score_blocks(&ok, NULL, NULL, NULL, NULL, NULL, NULL));
  report("score_d64", oasis_score_blocks(&bad_d, NULL, NULL, NULL, NULL, NULL, NULL));
  report("topk_group", oasis_topk_select(&bad_group, NULL, NULL, NULL, NULL, NULL, NULL, NULL));
  report("shape_null", oasis_fetch_diff_capped(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 2, NULL, NULL, NULL));
  printf("workspace %zu\n", oasis_attn_workspace_bytes(&ok));
  printf("workspace_bad %zu\n", oasis_attn_workspace_bytes(&bad_d));
  return 0;
}
