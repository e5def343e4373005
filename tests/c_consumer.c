/*
 * A plain C99 consumer of the library: compiled against include/pa.h with
 * gcc -std=c99 -pedantic -Werror and linked to libpagedattn.so by the ABI
 * tests, then run on the host.  It uses only calls that need no GPU: the
 * version, the workspace and partition sizing, the block manager (allocate,
 * a batch append, fork with a copy-on-write, free, the table export, running
 * out of blocks) and one argument rejection by pa_decode.  Prints "ok" and
 * exits 0 when every check holds.
 */
#include <stdio.h>
#include <string.h>

#include "pa.h"

static int failures = 0;

#define CHECK(cond)                                                       \
  do {                                                                    \
    if (!(cond)) {                                                        \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond);  \
      ++failures;                                                         \
    }                                                                     \
  } while (0)

int main(void) {
  pa_block_manager* bm;
  int64_t ids[3], counts[3], slots[3], copies[6];
  int32_t n_copies = -1;
  int32_t tables[12], lens[3];
  int32_t want_tables[12] = {0, 1, -1, -1, 2, 3, -1, -1, 0, 4, -1, -1};

  CHECK(pa_version() >= 100);

  /* Sizing: 8 blocks (128 tokens) never split; 100 blocks in 512-token
   * partitions need a workspace. */
  CHECK(pa_decode_workspace_size(4, 8, 2, 128, 8, 16, 0) == 0);
  CHECK(pa_decode_workspace_size(4, 8, 2, 128, 100, 16, 512) > 0);
  CHECK(pa_decode_partition_size(4, 2, 100, 16, 512) == 512);

  /* Eight 16-token blocks, handed out from the front of the free list. */
  bm = pa_bm_create(8, 16);
  CHECK(bm != NULL);
  CHECK(pa_bm_allocate(bm, 1, 20) == PA_OK);   /* blocks 0, 1 */
  CHECK(pa_bm_allocate(bm, 2, 16) == PA_OK);   /* block 2 */
  CHECK(pa_bm_num_free(bm) == 5);

  /* One token each: sequence 1 writes position 20 (block 1, offset 4);
   * sequence 2 fills block 2 and spills into a new block 3. */
  ids[0] = 1; ids[1] = 2;
  counts[0] = 1; counts[1] = 1;
  CHECK(pa_bm_append_batch(bm, ids, counts, 2, slots, copies, &n_copies) == PA_OK);
  CHECK(n_copies == 0);
  CHECK(slots[0] == 1 * 16 + 4);
  CHECK(slots[1] == 3 * 16 + 0);

  /* A fork shares blocks 0 and 1; the child's next token goes to a copy of
   * the shared partial block 1 (block 4), at offset 5. */
  CHECK(pa_bm_fork(bm, 1, 3) == PA_OK);
  CHECK(pa_bm_ref_count(bm, 1) == 2);
  CHECK(pa_bm_append(bm, 3, 1, slots, copies, &n_copies) == PA_OK);
  CHECK(n_copies == 1 && copies[0] == 1 && copies[1] == 4);
  CHECK(slots[0] == 4 * 16 + 5);
  CHECK(pa_bm_ref_count(bm, 1) == 1);

  ids[0] = 1; ids[1] = 2; ids[2] = 3;
  CHECK(pa_bm_block_tables(bm, ids, 3, 4, tables, lens) == PA_OK);
  CHECK(memcmp(tables, want_tables, sizeof(tables)) == 0);
  CHECK(lens[0] == 21 && lens[1] == 17 && lens[2] == 22);

  /* Releasing the child returns block 4 only; asking for more blocks than
   * are free changes nothing. */
  CHECK(pa_bm_free(bm, 3) == PA_OK);
  CHECK(pa_bm_ref_count(bm, 0) == 1);
  CHECK(pa_bm_num_free(bm) == 4);
  CHECK(pa_bm_allocate(bm, 9, 5 * 16) == PA_ERR_OUT_OF_BLOCKS);
  CHECK(pa_bm_num_free(bm) == 4);
  CHECK(strlen(pa_last_error()) > 0);
  pa_bm_destroy(bm);

  /* Host validation: a null output is rejected before anything is launched. */
  CHECK(pa_decode(NULL, (const void*)0x10000, (const void*)0x10000, (const void*)0x10000,
                  (const int32_t*)0x10000, (const int32_t*)0x10000, 4, 8, 64, 8, 2, 128, 16,
                  0.1f, PA_F16, PA_F16, 1.0f, 0, NULL, 0, NULL) == PA_ERR_INVALID_ARG);
  CHECK(strlen(pa_last_error()) > 0);

  if (failures) return 1;
  printf("ok\n");
  return 0;
}
