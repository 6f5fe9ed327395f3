// Host-side probe of the GEMM planner: compiles the library's own sources into one
// translation unit (device code to PTX only; nothing runs on a GPU) and answers
// queries read from stdin, one per line:
//   config M N deterministic group_a sms   ->  "bn stages"
//   splits M N num_kb sms                  ->  "S"
//   det N num_kb                           ->  "bn S" (deterministic tile width, K ranges)
// Built and run by tests/test_tile_table.py.
#include "../../fp8_scaled_gemm_mm_gb300/csrc/api.cu"
#include "../../fp8_scaled_gemm_mm_gb300/csrc/gemm.cu"

#include <cstdio>
#include <cstring>

int main() {
  char op[16];
  while (std::scanf("%15s", op) == 1) {
    if (std::strcmp(op, "config") == 0) {
      long long M, N;
      int det, group, sms;
      if (std::scanf("%lld %lld %d %d %d", &M, &N, &det, &group, &sms) != 5) return 2;
      const fp8mm::Config c = fp8mm::pick_config(M, N, det != 0, group != 0, sms);
      std::printf("%d %d\n", c.bn, c.stages);
    } else if (std::strcmp(op, "splits") == 0) {
      long long M, N;
      int num_kb, sms;
      if (std::scanf("%lld %lld %d %d", &M, &N, &num_kb, &sms) != 4) return 2;
      std::printf("%d\n", fp8mm::pick_splits(M, N, num_kb, sms));
    } else if (std::strcmp(op, "det") == 0) {
      long long N;
      int num_kb;
      if (std::scanf("%lld %d", &N, &num_kb) != 2) return 2;
      std::printf("%d %d\n", fp8mm::det_bn(N), fp8mm::det_splits(N, num_kb));
    } else {
      return 2;
    }
  }
  return 0;
}
