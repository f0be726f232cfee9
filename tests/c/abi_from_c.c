/* The library's boundary used from plain C99: the header compiles as C, the
 * entry points link, and every host-side check answers without a GPU
 * (nothing below reaches a launch).  Exit status 0 when all checks hold. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "moe_fp4.h"

static int failures = 0;

static void expect(int cond, const char* what) {
  if (!cond) {
    fprintf(stderr, "FAILED: %s\n", what);
    ++failures;
  }
}

int main(void) {
  moe_fp4_dims decode = {32, 4096, 2048, 256, 8};
  moe_fp4_dims bad_k = {16, 256, 128, 8, 9};
  moe_fp4_dims bad_d = {16, 100, 128, 8, 2};
  const size_t ws = moe_fp4_workspace_bytes(&decode);
  expect(ws > 0, "workspace bytes of the decode layer");
  expect(moe_fp4_host_workspace_bytes(&decode) > ws, "host workspace adds staging");
  expect(moe_fp4_workspace_bytes(&bad_k) == 0, "k > E rejected");
  expect(moe_fp4_workspace_bytes(&bad_d) == 0, "d not a multiple of 128 rejected");
  expect(moe_fp4_workspace_bytes(NULL) == 0, "null dims rejected");

  /* never dereferenced: each call fails its host-side checks first */
  void* fake = (void*)(uintptr_t)0x100000;
  float* fake_f = (float*)fake;
  int32_t* fake_i = (int32_t*)fake;
  const uint8_t* fake_u8 = (const uint8_t*)fake;
  expect(moe_fp4_forward(&decode, fake, fake_f, fake_u8, fake_u8, fake_u8, fake_u8, NULL, NULL, NULL, NULL, NULL,
                         NULL, 0u, fake, ws, NULL) == MOE_FP4_ERR_INVALID_ARG, "null out");
  expect(moe_fp4_forward(&decode, fake, fake_f, fake_u8, fake_u8, fake_u8, fake_u8, fake_f, NULL, NULL, NULL, NULL,
                         NULL, MOE_FP4_FLAG_FORCE_GEMV | MOE_FP4_FLAG_FORCE_TC, fake, ws, NULL) ==
             MOE_FP4_ERR_INVALID_ARG, "both path flags");
  expect(moe_fp4_forward(&decode, fake, fake_f, fake_u8, fake_u8, fake_u8, fake_u8, fake_f, NULL, NULL, NULL, NULL,
                         NULL, 0u, fake, 64, NULL) == MOE_FP4_ERR_WORKSPACE, "workspace too small");
  expect(moe_fp4_route(&decode, fake_f, NULL, fake_f, fake_i, fake_i, fake, ws, NULL) == MOE_FP4_ERR_INVALID_ARG,
         "route without topk_ids");
  expect(moe_fp4_mxfp8_quantize(NULL, 0, 64, NULL, NULL, NULL) == MOE_FP4_OK, "quantiser: zero rows");
  expect(moe_fp4_mxfp8_quantize(fake, 4, 48, (uint8_t*)fake, (uint8_t*)fake, NULL) == MOE_FP4_ERR_INVALID_ARG,
         "quantiser: K not a multiple of 32");
  expect(moe_fp4_check(NULL, NULL) == MOE_FP4_ERR_INVALID_ARG, "check without workspace");
  expect(strlen(moe_fp4_status_string(MOE_FP4_ERR_DEVICE)) > 0, "status string");
  expect(MOE_FP4_NUM_STAGE_EVENTS == 6, "stage event count");
  if (failures == 0) printf("C ABI checks passed\n");
  return failures == 0 ? 0 : 1;
}
