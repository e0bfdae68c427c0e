/* A plain C99 program using the library through include/moelora.h only:
 * workspace sizing, status strings and the argument checks that return
 * before anything is enqueued.  It touches no device memory, so it runs on a
 * machine without a GPU; tests/test_c_consumer.py builds and runs it. */
#include <stdio.h>
#include <stdint.h>
#include "moelora.h"

static int fails = 0;

static void expect(int cond, const char* what) {
  if (!cond) {
    printf("FAIL %s\n", what);
    ++fails;
  }
}

int main(void) {
  moelora_dims decode = {16, 4, 32, 2880, 2880, 8, 32};
  moelora_dims bad_rank = {16, 4, 32, 2880, 2880, 8, 24};
  moelora_dims empty = {0, 4, 32, 2880, 2880, 8, 32};
  moelora_linear_dims dense = {8, 8192, 28672, 32, 16};
  void* fake = (void*)(uintptr_t)0x7f0000000000ull;   /* never dereferenced */
  size_t ws = moelora_workspace_bytes(&decode);

  expect(ws > 0, "workspace bytes of the decode layer");
  expect(moelora_workspace_bytes(&bad_rank) == 0, "rank 24 has no workspace");
  expect(moelora_linear_workspace_bytes(&dense) > 0, "workspace bytes of the dense linear");
  expect(moelora_align_capacity(&decode, 16) == 16 * 4 + 32 * 15, "align capacity");
  expect(moe_lora_forward(&empty, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                          fake, fake, ws, NULL) == MOELORA_OK, "empty batch is a no-op");
  expect(moe_lora_forward(&bad_rank, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                          fake, fake, ws, NULL) == MOELORA_ERR_UNSUPPORTED, "rank 24 is unsupported");
  expect(moe_lora_forward(&decode, NULL, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                          fake, fake, ws, NULL) == MOELORA_ERR_INVALID_ARG, "null x");
  expect(moe_lora_forward(&decode, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                          fake, fake, ws - 1, NULL) == MOELORA_ERR_WORKSPACE, "workspace too small");
  for (int s = MOELORA_OK; s >= MOELORA_ERR_DEVICE_CHECK; --s)
    expect(moelora_status_string(s) != NULL && moelora_status_string(s)[0] != '\0', "status string");
  printf("%s %zu\n", fails ? "FAILED" : "OK", ws);
  return fails != 0;
}
