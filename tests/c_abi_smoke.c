/* Plain C use of the library's ABI (include/sagebwd.h): no C++, no torch, no GPU.
 * Prints the sizes the entry points report and the statuses they return for
 * invalid problems, one "name value" pair per line; the test compares them
 * with the Python binding's answers. */
#include <stdio.h>
#include <string.h>

#include "sagebwd.h"

static sagebwd_problem make(int B, int Hq, int Hkv, int N, int d, int causal) {
  sagebwd_problem p;
  memset(&p, 0, sizeof p);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.d = d;
  p.causal = causal;
  p.smooth_k = 1;
  p.qk_subexp = 1; /* the library's default Q/K granularity */
  return p;
}

int main(void) {
  sagebwd_problem p = make(1, 12, 2, 16384, 128, 1);
  printf("version %d\n", (int)sagebwd_version());
  printf("saved %zu\n", sagebwd_saved_bytes(&p));
  printf("ws0 %zu\n", sagebwd_workspace_bytes(&p, 0));
  printf("ws1 %zu\n", sagebwd_workspace_bytes(&p, 1));
  sagebwd_problem bad_d = make(1, 2, 2, 128, 96, 0);
  printf("bad_d_saved %zu\n", sagebwd_saved_bytes(&bad_d));
  sagebwd_problem bad_g = make(1, 3, 2, 128, 64, 0);
  printf("bad_g_saved %zu\n", sagebwd_saved_bytes(&bad_g));
  /* argument checks return before any launch: a null pointer and a misaligned one */
  char buf[64];
  printf("fwd_null %d\n", (int)sagebwd_fwd(&p, NULL, buf, buf, buf, (float*)buf, buf, buf, NULL));
  printf("fwd_misaligned %d\n",
         (int)sagebwd_fwd(&p, buf + 1, buf + 1, buf + 1, buf + 1, (float*)(buf + 1), buf + 1, buf + 1, NULL));
  printf("status_string_2 %s\n", sagebwd_status_string(SAGEBWD_ERR_UNSUPPORTED));
  return 0;
}
