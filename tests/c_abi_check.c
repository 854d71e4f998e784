/* A plain C (C11) caller of the library's C ABI, built and run by
 * tests/test_abi.py without a GPU: the header must compile as C, and the
 * host-only entry points must answer through the shared library.  Prints one
 * "key=value" line per check and exits nonzero on the first failure. */
#include <stdio.h>
#include <string.h>

#include "dsmem_hist.h"

static int fail(const char* what) {
  fprintf(stderr, "FAIL %s (last error: %s)\n", what, dsmem_hist_last_error());
  return 1;
}

int main(void) {
  const int version = dsmem_hist_version();
  printf("version=%d\n", version);
  if (version < 100) return fail("version");
  if (strncmp(dsmem_hist_strerror(DSMEM_HIST_EINVAL), "DSMEM_HIST_EINVAL", 17) != 0)
    return fail("strerror");

  /* Bad arguments are refused before any CUDA call. */
  uint32_t bins[4];
  if (dsmem_hist(NULL, 16, 4, bins, NULL) != DSMEM_HIST_EINVAL) return fail("null keys");
  if (dsmem_hist((const int32_t*)bins, -1, 4, bins, NULL) != DSMEM_HIST_EINVAL) return fail("n < 0");
  if (dsmem_hist((const int32_t*)bins, 4, 0, bins, NULL) != DSMEM_HIST_EINVAL) return fail("num_bins");

  /* The planner's plain three-argument form: a NULL `out` is refused before
   * any CUDA call; with a valid `out` it answers OK on a GPU and an error
   * code (never a crash) on a machine without one. */
  dsmem_hist_plan_t here;
  if (dsmem_hist_plan(262144, (int64_t)1 << 28, NULL) != DSMEM_HIST_EINVAL) return fail("plan NULL out");
  const int rc_here = dsmem_hist_plan(262144, (int64_t)1 << 28, &here);
  printf("plan_rc=%d\n", rc_here);
  if (rc_here != DSMEM_HIST_OK && rc_here != DSMEM_HIST_ECUDA && rc_here != DSMEM_HIST_EUNSUPPORTED)
    return fail("plan rc");
  if (rc_here == DSMEM_HIST_OK && here.cluster_size < 2) return fail("plan on this device");

  /* The planner for a described GB300: 262,144 bins take clusters of 8
   * CTAs x 32,768 counters in one pass, on the key-shipping kernel. */
  dsmem_hist_device_t dev;
  memset(&dev, 0, sizeof dev);
  dev.cc_major = 10;
  dev.cc_minor = 3;
  dev.sm_count = 152;
  dev.max_smem_per_block_optin = 232448;
  dev.max_smem_per_sm = 233472;
  dev.max_threads_per_sm = 2048;
  dev.max_cluster_size = 16;
  dsmem_hist_plan_t plan;
  memset(&plan, 0, sizeof plan);
  if (dsmem_hist_plan_for_device(&dev, 262144, (int64_t)1 << 28, NULL, 15, &plan) != DSMEM_HIST_OK)
    return fail("plan_for_device");
  printf("cluster_size=%d bins_per_cta=%d passes=%d kernel=%d block_threads=%d num_clusters=%d\n",
         plan.cluster_size, plan.bins_per_cta, plan.passes, plan.kernel, plan.block_threads,
         plan.num_clusters);
  if (plan.cluster_size != 8 || plan.bins_per_cta != 32768 || plan.passes != 1 ||
      plan.kernel != DSMEM_HIST_KERNEL_SHIP || plan.block_threads != DSMEM_HIST_SHIP_THREADS ||
      plan.num_clusters != 15)
    return fail("plan fields");
  printf("ok\n");
  return 0;
}
