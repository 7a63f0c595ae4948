/* A plain C11 caller of the C ABI (include/pda.h): compiled and run by
 * tests/test_abi.py. Only host-side paths are used, so no GPU is needed:
 * the pure planner, the tail-piece cut, status strings, and argument checks
 * that return before any CUDA call. */
#include <stdio.h>
#include <string.h>

#include "pda.h"

int main(void) {
  if (pda_choose_splits(16, 8, 64, 16, 152, 4) < 1) return 1;
  if (strlen(pda_status_string(PDA_ERR_INVALID_ARG)) == 0) return 2;
  /* no sequences: nothing to do */
  if (pda_decode(NULL, NULL, NULL, NULL, NULL, NULL, 0, 8, 2, 128, 16, 4, 0.1f, 0.05f, 0.05f, NULL) != PDA_OK) return 3;
  /* head size 64 is outside the supported set */
  if (pda_decode(NULL, NULL, NULL, NULL, NULL, NULL, 2, 8, 2, 64, 16, 4, 0.1f, 0.05f, 0.05f, NULL) !=
      PDA_ERR_UNSUPPORTED)
    return 4;
  /* host buffers with a table entry outside a 4-block pool: refused on the host */
  static uint16_t q[8 * 128], out[8 * 128];
  static uint8_t k[4 * 2 * 128 * 16], v[4 * 2 * 128 * 16];
  const int32_t table[2] = {0, 9};
  const int32_t lens[1] = {20};
  if (pda_decode_host(out, q, k, v, table, lens, 1, 8, 2, 128, 16, 2, 4, 0.1f, 0.05f, 0.05f, NULL) !=
      PDA_ERR_INVALID_ARG)
    return 5;
  /* the tail-piece cut of the 256 x 4096-token batch: 5 shrinking pieces */
  int sizes[8] = {0};
  if (pda_tail_pieces(256, 224, 456, 16, sizes, 8) != 5 || sizes[0] != 126 || sizes[4] != 17) return 6;
  if (pda_tail_pieces(256, 456, 456, 16, sizes, 8) != -1) return 7;
  puts("ok");
  return 0;
}
