/* The public header as plain C11: every declaration compiles without C++,
 * and the pure host functions link and answer without a GPU. */
#include <stdio.h>
#include <string.h>

#include "qs.h"

int main(void) {
  qs_cache_bytes_t b;
  if (qs_cache_bytes(2, 3, 128, 128, 4, &b) != QS_OK) return 1;
  if (b.k_upper != (size_t)2 * 3 * 4 * 128 * 64 || b.arrive != (size_t)2 * 3 * 4) return 2;
  if (qs_cache_bytes(1, 1, 64, 128, 1, &b) != QS_ERR_UNSUPPORTED) return 3;
  if (qs_cache_bytes(1, 1, 128, 128, 1, NULL) != QS_ERR_ARG) return 4;
  if (strcmp(qs_status_string(QS_OK), "ok") != 0) return 5;
  qs_cache c;
  memset(&c, 0, sizeof c);
  if (qs_state_reset(&c, NULL) != QS_ERR_ARG) return 6; /* null arrays */
  if (qs_state_reset(NULL, NULL) != QS_ERR_ARG) return 7;
  puts("abi ok");
  return 0;
}
