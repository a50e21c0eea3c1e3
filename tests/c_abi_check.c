/* The C ABI of libmuon used from plain C (no Python, no CUDA headers): plan a
 * parameter set, query groups and slices, assign slices to replicas, check
 * the argument errors and the host-side fault switches, all host-only calls.  Prints "ok" and exits 0
 * when every check holds; otherwise prints the failed check and exits 1. */
#define _POSIX_C_SOURCE 200112L
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "muon.h"

static int fails = 0;
#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      printf("failed: %s (line %d)\n", #c, __LINE__);         \
      ++fails;                                                \
    }                                                         \
  } while (0)

int main(void) {
  /* 74 bf16 [24,10240] matrices, an fp32 [1408,2048] stack of 3, a
   * transposed bf16 [2048,1408] matrix */
  muon_shape shapes[76];
  for (int i = 0; i < 74; ++i) {
    shapes[i].ndim = 2;
    shapes[i].dims[0] = 24;
    shapes[i].dims[1] = 10240;
    shapes[i].dims[2] = 0;
    shapes[i].dtype = MUON_BF16;
  }
  shapes[74].ndim = 3;
  shapes[74].dims[0] = 3;
  shapes[74].dims[1] = 1408;
  shapes[74].dims[2] = 2048;
  shapes[74].dtype = MUON_F32;
  shapes[75].ndim = 2;
  shapes[75].dims[0] = 2048;
  shapes[75].dims[1] = 1408;
  shapes[75].dims[2] = 0;
  shapes[75].dtype = MUON_BF16;

  muon_options opt;
  muon_options_default(&opt);
  CHECK(opt.mode == MUON_MODE_TC16 && opt.skinny_max_m == 64 &&
        opt.scale_mode == MUON_SCALE_SQRT_RATIO);

  muon_plan_t* plan = NULL;
  CHECK(muon_plan(shapes, 76, &opt, &plan) == MUON_OK && plan != NULL);

  int ng = 0, ns = 0;
  CHECK(muon_plan_num_groups(plan, &ng) == MUON_OK && ng == 3);
  CHECK(muon_plan_num_slices(plan, &ns) == MUON_OK && ns == 78);
  muon_group_info gi;
  CHECK(muon_plan_group(plan, 0, &gi) == MUON_OK);
  CHECK(gi.m == 24 && gi.n == 10240 && gi.count == 74 && gi.tr == 0 &&
        gi.kernel == MUON_KERNEL_SKINNY && gi.cluster == 2 && gi.scale == 1.0f);
  CHECK(muon_plan_group(plan, 2, &gi) == MUON_OK);
  CHECK(gi.M == 2048 && gi.N == 1408 && gi.m == 1408 && gi.tr == 1 &&
        gi.kernel == MUON_KERNEL_DENSE);
  int g = -1, idx = -1;
  CHECK(muon_plan_slice(plan, 74, 2, &g, &idx) == MUON_OK && g == 1 && idx == 2);
  size_t ws = 0;
  CHECK(muon_plan_workspace_bytes(plan, &ws) == MUON_OK && ws > 256 && ws % 256 == 0);
  int launches = 0;
  /* one fused launch for the skinny group; per dense group front, finalize,
   * normalize and three products per step, the last of which applies the
   * update (transposed groups too) */
  CHECK(muon_plan_launches(plan, 5, &launches) == MUON_OK && launches == 1 + 18 + 18);

  /* the other update scale: s = 0.2 sqrt(max(M, N)) */
  muon_options opt2 = opt;
  opt2.scale_mode = MUON_SCALE_RMS_MATCH;
  muon_plan_t* plan2 = NULL;
  CHECK(muon_plan(shapes, 76, &opt2, &plan2) == MUON_OK && plan2 != NULL);
  CHECK(muon_plan_group(plan2, 0, &gi) == MUON_OK &&
        gi.scale == (float)(0.2 * 101.19288512538813) /* sqrt(10240) */);
  CHECK(muon_plan_group(plan2, 2, &gi) == MUON_OK &&
        gi.scale == (float)(0.2 * 45.254833995939045) /* sqrt(2048) */);
  muon_plan_destroy(plan2);
  opt2.scale_mode = 7;
  CHECK(muon_plan(shapes, 76, &opt2, &plan2) == MUON_ERR_INVALID_ARG);

  /* host-side fault switches: status codes, no device work */
  setenv("MUON_FAULT", "alloc", 1);
  plan2 = NULL;
  CHECK(muon_plan(shapes, 76, &opt, &plan2) == MUON_ERR_NOMEM && plan2 == NULL);
  setenv("MUON_FAULT", "launch", 1);
  {
    void* fake[76];
    float* fakef[76];
    for (int i = 0; i < 76; ++i) {
      fake[i] = (void*)(uintptr_t)(0x10000 + 256 * i);
      fakef[i] = (float*)fake[i];
    }
    CHECK(muon_step(plan, fake, (const void* const*)fake, fakef, 0.02f, 0.95f, 0.1f, 1, 5, NULL,
                    (void*)(uintptr_t)0x100000, ws, NULL) == MUON_ERR_CUDA);
  }
  unsetenv("MUON_FAULT");

  /* host-state allocator: argument checks, the fault switch, frees of NULL
     and of an address it did not return.  With no device the registration
     fails and nothing is held; with one, the memory is aligned and zeroed. */
  {
    void* hp = (void*)(uintptr_t)1;
    CHECK(muon_host_alloc(0, &hp) == MUON_ERR_INVALID_ARG && hp == NULL);
    CHECK(muon_host_alloc(4096, NULL) == MUON_ERR_INVALID_ARG);
    CHECK(muon_host_free(NULL) == MUON_OK);
    CHECK(muon_host_free((void*)(uintptr_t)0x123000) == MUON_ERR_INVALID_ARG);
    setenv("MUON_FAULT", "alloc", 1);
    hp = (void*)(uintptr_t)1;
    CHECK(muon_host_alloc(4096, &hp) == MUON_ERR_NOMEM && hp == NULL);
    unsetenv("MUON_FAULT");
    muon_status hs = muon_host_alloc(4096, &hp);
    if (hs == MUON_OK) {
      CHECK(hp != NULL && (uintptr_t)hp % 4096 == 0 && ((unsigned char*)hp)[4095] == 0);
      CHECK(muon_host_free(hp) == MUON_OK);
      CHECK(muon_host_free(hp) == MUON_ERR_INVALID_ARG);
    } else {
      CHECK(hs == MUON_ERR_CUDA && hp == NULL);
    }
  }

  /* replicas: every slice has one owner, the loads sum up */
  int owner[78];
  double load[4];
  CHECK(muon_plan_partition(plan, 4, 5, 1.88e15, 6.78e12, owner, load) == MUON_OK);
  int count[4] = {0, 0, 0, 0};
  for (int s = 0; s < 78; ++s) {
    CHECK(owner[s] >= 0 && owner[s] < 4);
    if (owner[s] >= 0 && owner[s] < 4) ++count[owner[s]];
  }
  for (int r = 0; r < 4; ++r) CHECK(count[r] > 0 && load[r] > 0.0);

  /* argument errors are status codes, before any device work */
  CHECK(muon_plan(NULL, 1, NULL, &plan) == MUON_ERR_INVALID_ARG);
  shapes[0].ndim = 1;
  muon_plan_t* bad = NULL;
  CHECK(muon_plan(shapes, 1, NULL, &bad) == MUON_ERR_UNSUPPORTED_SHAPE && bad == NULL);
  CHECK(muon_step(plan, NULL, NULL, NULL, 0.02f, 0.95f, 0.1f, 1, 5, NULL, NULL, 0, NULL) ==
        MUON_ERR_INVALID_ARG);
  CHECK(muon_plan_partition(plan, 0, 5, 1.0, 1.0, owner, NULL) == MUON_ERR_INVALID_ARG);
  CHECK(strcmp(muon_status_string(MUON_ERR_WORKSPACE), "workspace too small for the plan") == 0);
  CHECK(strcmp(muon_status_string(MUON_ERR_NOMEM), "host memory allocation failed") == 0);

  muon_plan_destroy(plan);
  if (fails) return 1;
  printf("ok\n");
  return 0;
}
