/* A plain C consumer of libfp8mm: includes the public header, links the shared
 * library and exercises the host-side paths that need no GPU (version, status
 * strings, argument validation, empty problems).  Built and run by
 * tests/test_abi.py::test_plain_c_consumer. */
#include <stdint.h>
#include <stdio.h>

#include "fp8mm.h"

static int failures = 0;

static void expect(const char* what, int got, int want) {
  if (got != want) {
    printf("FAIL %s: got %d (%s), want %d\n", what, got, fp8mm_status_string(got), want);
    ++failures;
  }
}

int main(void) {
  const int v = fp8mm_version();
  printf("libfp8mm version %d.%d\n", v >> 16, v & 0xFFFF);
  if ((v >> 16) != 1) ++failures;

  void* fake = (void*)(uintptr_t)(1u << 20);   /* never dereferenced: validation fails first */
  float* fs = (float*)fake;
  uint8_t* f8 = (uint8_t*)fake;

  /* GEMM: empty problem, K not a multiple of 16, misaligned A */
  expect("gemm M=0", fp8_scaled_mm(fake, fake, fs, fs, FP8MM_SCALE_A_ROW | FP8MM_SCALE_B_COL, NULL, fake,
                                   FP8MM_DTYPE_BF16, 0, 256, 512, 512, 512, 0, NULL), FP8MM_OK);
  expect("gemm K%16", fp8_scaled_mm(fake, fake, fs, fs, FP8MM_SCALE_A_ROW | FP8MM_SCALE_B_COL, NULL, fake,
                                    FP8MM_DTYPE_BF16, 64, 256, 72, 80, 80, 0, NULL), FP8MM_EINVAL);
  expect("gemm misaligned", fp8_scaled_mm(f8 + 8, f8 + (1 << 24), fs, fs, FP8MM_SCALE_A_ROW | FP8MM_SCALE_B_COL,
                                          NULL, f8 + (2 << 24), FP8MM_DTYPE_BF16, 64, 256, 512, 512, 512, 0, NULL),
         FP8MM_EALIGN);
  /* quant: empty batch, bad group */
  expect("quant M=0", per_token_group_quant_fp8(NULL, FP8MM_DTYPE_BF16, NULL, NULL, 0, 2048, 128,
                                                FP8MM_SCALE_FP32, 0, 0, NULL), FP8MM_OK);
  expect("quant group", per_token_group_quant_fp8(fake, FP8MM_DTYPE_BF16, f8, fake, 4, 2048, 96,
                                                  FP8MM_SCALE_FP32, 0, 0, NULL), FP8MM_EINVAL);
  expect("int8 group", per_token_group_quant_int8(fake, FP8MM_DTYPE_BF16, (int8_t*)fake, fs, 4, 2048, 96, 0, 0,
                                                  NULL), FP8MM_EINVAL);
  expect("static numel", static_per_tensor_quant_fp8(fake, FP8MM_DTYPE_BF16, fs, f8, 24, NULL), FP8MM_EINVAL);
  printf("%s\n", failures ? "c consumer FAILED" : "c consumer ok");
  return failures ? 1 : 0;
}
