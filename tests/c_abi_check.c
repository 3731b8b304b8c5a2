/*
 * A plain C caller of the library's C ABI (include/moe.h), built with gcc
 * and linked against libmoe.so by tests/test_abi.py.  It uses only calls
 * that are answered on the host (no GPU needed): the version, workspace
 * sizes, the expert capacity, the launch plan and the argument validation
 * that every entry point runs before it touches the device.  Prints "ok"
 * and exits 0 when every check holds; otherwise names the failed check.
 */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "moe.h"

static int failures = 0;

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #cond); \
      ++failures;                                                \
    }                                                            \
  } while (0)

static moe_shape shape(int T, int H, int F, int E, int k, double cf) {
  moe_shape s;
  memset(&s, 0, sizeof s);
  s.T = T;
  s.H = H;
  s.F = F;
  s.E = E;
  s.k = k;
  s.capacity_factor = cf;
  s.gating = MOE_GATE_TOPK_SOFTMAX;
  s.expert_act = MOE_EXPERT_GELU;
  return s;
}

int main(void) {
  CHECK((moe_version() >> 16) == 1);

  /* workspace of the decode shape: status block, per-tile counts, h and Y,
   * and the fp32 partials of the small-batch second GEMM (T*k = 64 rows) */
  moe_shape d = shape(32, 4096, 14336, 8, 2, -1.0);
  const size_t want = 1024 + 1024 + (size_t)64 * 14336 * 2 + (size_t)64 * 4096 * 2 +
                      (size_t)4 * 64 * 4096 * 4;
  CHECK(moe_workspace_size(&d) == want);
  CHECK(moe_route_workspace_size(&d) == 1024 + 1024);

  /* capacity: ceil(1.2 * 8192 * 4 / 64) = 615; no limit: -1 */
  moe_shape sk = shape(8192, 2048, 1408, 64, 4, 1.2);
  CHECK(moe_expert_capacity(&sk) == 615);
  sk.capacity_factor = NAN;
  CHECK(moe_expert_capacity(&sk) == -1);

  /* launch plan: small batches and up to 128 tiles route in one launch;
   * k = 1 combines inside the second GEMM */
  int32_t in_router = -1, in_gemm = -1;
  CHECK(moe_forward_plan(&d, &in_router, &in_gemm) == MOE_OK && in_router == 1 && in_gemm == 0);
  moe_shape big = shape(40000, 256, 256, 8, 1, -1.0);
  CHECK(moe_forward_plan(&big, &in_router, &in_gemm) == MOE_OK && in_router == 0 && in_gemm == 1);

  /* validation before anything is enqueued */
  moe_shape bad = shape(64, 100, 256, 8, 2, -1.0); /* H not a multiple of 8 */
  CHECK(moe_workspace_size(&bad) == 0);
  CHECK(moe_forward(&bad, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                    NULL, 0, NULL) == MOE_ERR_UNSUPPORTED);
  CHECK(strstr(moe_last_error_string(), "H = 100") != NULL);
  moe_shape bad_e = shape(64, 128, 256, 300, 2, -1.0);
  CHECK(moe_route(&bad_e, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) ==
        MOE_ERR_UNSUPPORTED);
  moe_shape ok = shape(64, 128, 256, 6, 2, -1.0); /* any E in 1..256 */
  CHECK(moe_workspace_size(&ok) > 0);
  CHECK(moe_forward(&ok, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                    NULL, moe_workspace_size(&ok), NULL) == MOE_ERR_INVALID_ARG);
  CHECK(strstr(moe_last_error_string(), "ws") != NULL);
  /* the allocation-free entry point refuses shapes beyond its scratch */
  moe_shape prefill = shape(4096, 4096, 14336, 8, 2, -1.0);
  CHECK(moe_expert_ffn_combine_noalloc(&prefill, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                                       NULL) == MOE_ERR_UNSUPPORTED);
  CHECK(strstr(moe_last_error_string(), "scratch") != NULL);
  CHECK(moe_noalloc_device_status(NULL, NULL) == MOE_ERR_INVALID_ARG);
  CHECK(moe_route_plan(&d, NULL, NULL) == MOE_ERR_INVALID_ARG);

  if (failures) return 1;
  printf("ok\n");
  return 0;
}
