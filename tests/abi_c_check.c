/* Compiled as plain C99 by tests/test_abi_cpu.py against include/flce.h and
 * linked with libflce.so: the header is valid C, its structs have the layout
 * the binding assumes, and the entry points that need no GPU answer. Prints
 * "ok" and exits 0 on success. */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "flce.h"

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      printf("failed: %s (line %d)\n", #cond, __LINE__);         \
      return 1;                                                  \
    }                                                            \
  } while (0)

int main(void) {
  flce_options o;
  size_t bytes = 0;
  memset(&o, 0x5a, sizeof(o));
  flce_default_options(&o);
  CHECK(sizeof(flce_options) == 64);
  CHECK(o.ignore_index == -100 && o.reduction == FLCE_REDUCTION_MEAN && o.grad_scale == 1.0f);
  CHECK(o.dw_dtype == FLCE_DTYPE_F32 && o.timeout_ns == 0 && o.trace_events == NULL);
  CHECK(flce_workspace_size(8192, 4096, 128256, &o, &bytes) == FLCE_OK);
  CHECK(bytes > ((size_t)256 << 20) && bytes < ((size_t)600 << 20));
  CHECK(flce_workspace_size(8192, 4100, 128256, &o, &bytes) == FLCE_ERR_ALIGN);
  CHECK(flce_workspace_size(0, 4096, 128256, &o, &bytes) == FLCE_ERR_SHAPE);
  CHECK(flce_workspace_size(8, 64, 100, &o, NULL) == FLCE_ERR_NULL);
  CHECK(flce_ce_workspace_size(8192, 128256, NULL, &bytes) == FLCE_OK && bytes > 0);
  {
    /* the forward-only size leaves out the G chunk and accumulators, and not D */
    size_t fwd = 0, fwd2 = 0, full = 0;
    CHECK(flce_forward_workspace_size(8192, 4096, 128256, &o, &fwd) == FLCE_OK);
    CHECK(flce_forward_workspace_size(8192, 64, 128256, &o, &fwd2) == FLCE_OK && fwd2 == fwd);
    CHECK(flce_workspace_size(8192, 4096, 128256, &o, &full) == FLCE_OK && fwd < full);
    CHECK(flce_forward_workspace_size(8192, 4100, 128256, &o, &fwd) == FLCE_ERR_ALIGN);
  }
  CHECK(flce_forward_backward(NULL, NULL, NULL, 8, 64, 100, &o, NULL, NULL, NULL, NULL, NULL, 0,
                              NULL, NULL) == FLCE_ERR_NULL);
  {
    /* the shard, FP8 and quantiser entry points reject bad arguments on the host */
    float m[4], s[4], zt[4];
    CHECK(flce_forward_shard((const uint16_t*)0x1000, (const uint16_t*)0x2000,
                             (const int32_t*)0x3000, 64, 128, 500, 501, 1000, &o, m, s, zt,
                             (void*)0x7000, (size_t)1 << 30, NULL, NULL) == FLCE_ERR_SHAPE);
    CHECK(flce_forward_shard((const uint16_t*)0x1000, (const uint16_t*)0x2000,
                             (const int32_t*)0x3000, 64, 128, 500, 500, 1000, &o, NULL, s, zt,
                             (void*)0x7000, (size_t)1 << 30, NULL, NULL) == FLCE_ERR_NULL);
    CHECK(flce_backward_shard((const uint16_t*)0x1000, (const uint16_t*)0x2000,
                              (const int32_t*)0x3000, 64, 128, 500, 500, 1000, &o, NULL,
                              (float*)0x9000, NULL, (void*)0x7000, (size_t)1 << 30, NULL,
                              NULL) == FLCE_ERR_NULL);
    CHECK(flce_forward_fp8((const uint8_t*)0x1000, NULL, (const uint8_t*)0x2000,
                           (const float*)0x8004, (const int32_t*)0x3000, 64, 128, 1000, &o,
                           (float*)0x4000, NULL, (void*)0x5000, (size_t)1 << 30, NULL,
                           NULL) == FLCE_ERR_NULL);
    CHECK(flce_quantize_e4m3((const uint16_t*)0x1000, 12, (uint8_t*)0x2000, (float*)0x3000,
                             NULL) == FLCE_ERR_ALIGN);
  }
  CHECK(flce_status_string(FLCE_OK) != NULL && flce_status_string(FLCE_ERR_TIMEOUT) != NULL);
  CHECK(flce_status_string(12345) != NULL);
  printf("ok\n");
  return 0;
}
