/* A C11 program that includes include/ringred.h and links libringred.so: the
 * boundary is plain C.  Run on a machine without a GPU it exercises only the
 * calls that need none (versions, chunk table, argument checks) and prints one
 * line per check; the test compares them with what the header promises. */
#include <stdint.h>
#include <stdio.h>

#include "ringred.h"

int main(void) {
  printf("abi %d\n", ring_abi_version());
  /* the chunk table of (10, 4): 2 2 2 4 at 0 2 4 6 */
  for (int c = 0; c < 4; c++)
    printf("chunk %d %zu %zu\n", c, ring_chunk_count(10, 4, c), ring_chunk_offset(10, 4, c));
  /* argument errors are detected before anything touches a device */
  uintptr_t fake_in[2] = {0x10000, 0x20000}, fake_out[2] = {0x30000, 0x40000};
  const void *in[2] = {(const void *)fake_in[0], (const void *)fake_in[1]};
  void *out[2] = {(void *)fake_out[0], (void *)fake_out[1]};
  printf("bad_rank_count %d\n", (int)ring_allreduce(in, out, 0, 100, RR_FP32, NULL));
  printf("bad_dtype %d\n", (int)ring_allreduce(in, out, 2, 100, (rr_dtype)7, NULL));
  printf("unsupported_pair %d\n", (int)ring_allreduce_ex(in, out, 2, 100, RR_FP16, RR_BF16, 0, NULL));
  void *alias_out[2] = {(void *)fake_in[1], (void *)fake_out[1]};
  printf("alias %d\n", (int)ring_allreduce(in, alias_out, 2, 100, RR_FP32, NULL));
  printf("empty %d\n", (int)ring_allreduce(in, out, 2, 0, RR_FP32, NULL));
  printf("status %s\n", ring_status_string(RR_ERR_ALIAS));
  return 0;
}
