/* A plain C99 caller of the library: sizes and lays out the metadata of a pool descriptor and prints an error
 * string. It needs no GPU, so it runs on any machine that can load libhs.so. */
#include <stdio.h>

#include "hs.h"

int main(void) {
  hs_pool_desc d = {0};
  hs_meta_layout lay;
  d.layers = 2;
  d.max_batch = 3;
  d.ctx = 1000;
  d.slots = 64;
  d.topk_max = 32;
  d.row_bytes = 656;
  if (hs_get_meta_layout(&d, &lay) != HS_OK) return 1;
  printf("%zu %zu %zu %zu\n", hs_meta_bytes(&d), lay.tok2slot, lay.slot_stamp, lay.total);
  printf("%s\n", hs_error_string(HS_ERR_INVALID_ARG));
  d.row_bytes = 650; /* not a multiple of 16 */
  printf("%d %zu\n", hs_get_meta_layout(&d, &lay), hs_meta_bytes(&d));
  return 0;
}
