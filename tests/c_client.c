/* A C program that uses the library only through include/mla_decode.h: it
 * sizes a workspace, checks host-side argument rejection and reads the status
 * strings.  Needs no GPU (no call here reaches the device). */
#include <stdio.h>
#include <string.h>

#include "mla_decode.h"

static int fails = 0;
#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      ++fails;                                                   \
    }                                                            \
  } while (0)

int main(void) {
  mla_decode_dims d;
  memset(&d, 0, sizeof(d));
  d.batch = 64;
  d.q_len = 1;
  d.num_heads = 16;
  d.qk_nope = 128;
  d.qk_rope = 64;
  d.kv_lora = 512;
  d.v_head = 128;
  d.page_size = 64;
  d.num_pages = 4096;
  d.max_pages_per_seq = 64;

  size_t bytes = 0;
  CHECK(mla_decode_workspace_size_ex(&d, 152, &bytes) == MLA_DECODE_OK);
  /* q_lat (bf16), q_lo (E4M3 bytes) and o_lat (bf16) for 1024 rows, plus 304
     partial slots of 16 rows (bf16 o, fp32 lse). */
  CHECK(bytes >= (size_t)1024 * (576 * 2 + 512 + 512 * 2) + (size_t)304 * 16 * (512 * 2 + 4));

  mla_decode_dims bad = d;
  bad.kv_lora = 256;
  CHECK(mla_decode_workspace_size_ex(&bad, 152, &bytes) == MLA_DECODE_UNSUPPORTED);
  bad = d;
  bad.q_len = 9;
  CHECK(mla_decode_workspace_size_ex(&bad, 152, &bytes) == MLA_DECODE_UNSUPPORTED);
  CHECK(mla_decode_workspace_size_ex(&d, 152, NULL) == MLA_DECODE_INVALID_ARG);

  /* A whole run with a null output is rejected before anything is enqueued. */
  void* p = (void*)4096;
  CHECK(mla_decode_run(&d, p, p, (const int32_t*)p, (const int32_t*)p, p, p, 0.07f, NULL,
                       (float*)p, p, (size_t)1 << 30, NULL) == MLA_DECODE_INVALID_ARG);
  CHECK(mla_decode_run_fp8w(&d, p, p, (const int32_t*)p, (const int32_t*)p,
                            (const uint8_t*)p, NULL, (const uint8_t*)p, (const float*)p, 0.07f,
                            p, (float*)p, p, (size_t)1 << 30, NULL) == MLA_DECODE_INVALID_ARG);
  CHECK(mla_decode_check(NULL, NULL) == MLA_DECODE_INVALID_ARG);

  /* The softmax scale must be finite and > 0. */
  const float bad_scales[3] = {0.0f, -0.07f, 1.0f / 0.0f};
  for (int i = 0; i < 3; ++i) {
    CHECK(mla_decode_run(&d, p, p, (const int32_t*)p, (const int32_t*)p, p, p, bad_scales[i], p,
                         (float*)p, p, (size_t)1 << 30, NULL) == MLA_DECODE_INVALID_ARG);
    CHECK(mla_decode_attend(&d, p, (const int32_t*)p, (const int32_t*)p, bad_scales[i], (float*)p,
                            p, (size_t)1 << 30, NULL) == MLA_DECODE_INVALID_ARG);
    CHECK(mla_decode_combine(&d, bad_scales[i], (float*)p, p, (size_t)1 << 30, NULL) ==
          MLA_DECODE_INVALID_ARG);
    CHECK(mla_decode_run_static_scratch(&d, p, p, (const int32_t*)p, (const int32_t*)p, p, p,
                                        bad_scales[i], p, (float*)p, NULL) ==
          MLA_DECODE_INVALID_ARG);
  }

  for (int s = 0; s <= 6; ++s) CHECK(strcmp(mla_decode_status_string(s), "unknown status") != 0);
  CHECK(strcmp(mla_decode_status_string(42), "unknown status") == 0);

  if (fails == 0) printf("c client: ok\n");
  return fails == 0 ? 0 : 1;
}
