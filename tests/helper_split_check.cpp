// CPU check of the idle-SM helper's split and share controller
// (cluster_distributed_shared_gb300/csrc/helper_split.h), driven with
// synthetic reports.  Prints "ok" and exits 0 when every check holds.
#include <math.h>
#include <stdint.h>
#include <stdio.h>

#include "helper_split.h"

using namespace dsmh;

static int failures = 0;

#define CHECK(cond)                                                   \
  do {                                                                \
    if (!(cond)) {                                                    \
      printf("FAIL %s:%d: %s\n", __FILE__, __LINE__, #cond);          \
      ++failures;                                                     \
    }                                                                 \
  } while (0)

// A stream that launches, gets each launch's report back before the next
// launch (the host synchronises between calls), and feeds it to the
// controller.  Returns the share after `steps` reports of `target`.
static double settle(double start, float target, int steps, HelperShare* out = nullptr) {
  HelperShare h;
  h.share = start;
  uint32_t launch = 0;
  for (int i = 0; i < steps; ++i) {
    ++launch;  // the launch that ran at h.share
    CHECK(helper_report_current(h, launch));
    CHECK(helper_share_step(h, target, launch));
  }
  if (out) *out = h;
  return h.share;
}

int main() {
  // The prior: the idle SMs' pace relative to the clusters'.
  CHECK(fabs(helper_prior(120, 32) - 32 * 0.42 / (120 + 32 * 0.42)) < 1e-12);
  CHECK(helper_prior(120, 32) > 0.09 && helper_prior(120, 32) < 0.11);  // about 10% at P = 8
  CHECK(helper_prior(152, 0) == 0.0);

  // A fixed target is approached from either side without overshoot (the
  // step never exceeds three quarters) and reached within 1e-3.
  {
    HelperShare h;
    const double s = settle(0.1, 0.3f, 20, &h);
    CHECK(fabs(s - 0.3) < 1e-3);
    CHECK(h.last_sign == 1);
    CHECK(h.gain == kHelperGainMax);
    double prev = 0.1;
    HelperShare g;
    g.share = 0.1;
    for (uint32_t i = 1; i <= 10; ++i) {
      helper_share_step(g, 0.3f, i);
      CHECK(g.share > prev && g.share <= 0.3 + 1e-12);  // monotone, never past the target
      prev = g.share;
    }
    CHECK(fabs(settle(0.5, 0.2f, 30) - 0.2) < 1e-3);
  }
  // The first step takes three quarters of the way.
  {
    HelperShare h;
    h.share = 0.1;
    CHECK(helper_share_step(h, 0.5f, 1));
    CHECK(fabs(h.share - (0.1 + 0.75 * 0.4)) < 1e-6);
  }
  // Clamps: the share stays within [0.01, 0.6] whatever the target.
  CHECK(fabs(settle(0.1, 0.95f, 40) - kHelperShareMax) < 1e-12);
  CHECK(fabs(settle(0.1, 0.0001f, 40) - kHelperShareMin) < 1e-12);
  // Targets outside (0, 1) are ignored.
  {
    HelperShare h;
    h.share = 0.2;
    CHECK(!helper_share_step(h, 0.0f, 1));
    CHECK(!helper_share_step(h, 1.0f, 1));
    CHECK(!helper_share_step(h, -0.5f, 1));
    CHECK(!helper_share_step(h, NAN, 1));
    CHECK(h.share == 0.2 && h.gain == 0.0 && h.valid_from == 0);
  }
  // Damping: a target that alternates around a value halves the step at
  // every change of direction, down to the floor, and the share's swing
  // shrinks with it.
  {
    HelperShare h;
    h.share = 0.3;
    double swing_first = 0.0, swing_last = 0.0;
    for (uint32_t i = 1; i <= 40; ++i) {
      const double before = h.share;
      helper_share_step(h, (i & 1) ? 0.4f : 0.2f, i);
      const double swing = fabs(h.share - before);
      if (i == 2) swing_first = swing;
      swing_last = swing;
    }
    CHECK(h.gain == kHelperGainMin);
    CHECK(swing_last < 0.25 * swing_first);
    CHECK(fabs(h.share - 0.3) < 0.02);  // it stays near the middle
  }
  // The step grows again by a quarter while the direction holds.
  {
    HelperShare h;
    h.share = 0.3;
    helper_share_step(h, 0.2f, 1);  // gain 0.75, down
    helper_share_step(h, 0.4f, 2);  // up: 0.375
    CHECK(fabs(h.gain - 0.375) < 1e-12);
    helper_share_step(h, 0.5f, 3);  // up again: 0.46875
    CHECK(fabs(h.gain - 0.46875) < 1e-12);
  }
  // Only current reports count: once the share moves, reports of launches
  // made before the move (up to the last count handed out) are stale.
  {
    HelperShare h;
    h.share = 0.1;
    // Launches 1..5 are enqueued at share 0.1; launch 1's report arrives.
    CHECK(helper_report_current(h, 1));
    CHECK(helper_share_step(h, 0.3f, 5));
    CHECK(h.valid_from == 6);
    for (uint32_t launch = 2; launch <= 5; ++launch) CHECK(!helper_report_current(h, launch));
    CHECK(helper_report_current(h, 6));
    CHECK(helper_report_current(h, 7));
    // A report that leaves the share where it is keeps the window open.
    HelperShare g;
    g.share = kHelperShareMax;
    g.valid_from = 3;
    CHECK(helper_share_step(g, 0.9f, 10));
    CHECK(g.share == kHelperShareMax && g.valid_from == 3);
    // Launch counts wrap around 2^32 without breaking the window.
    HelperShare w;
    w.share = 0.2;
    w.valid_from = 0xFFFFFFF0u;
    CHECK(helper_report_current(w, 0xFFFFFFF0u));
    CHECK(helper_report_current(w, 5u));  // past the wrap
    CHECK(!helper_report_current(w, 0xFFFFFFEFu));
  }
  // The split: the clusters' tiles are whole rounds, at most their share,
  // and the helper gets the rest.
  {
    const uint64_t per_round = 120 * 28 * 2;  // P = 8: 120 CTAs x 28 warps x 2 tiles
    const uint32_t ntiles = 268435456u / 128u;
    for (int k = 0; k <= 100; ++k) {
      const double share = k / 100.0;
      const uint32_t c = helper_cluster_tiles(ntiles, share, per_round);
      CHECK(c % per_round == 0);
      CHECK(c <= ntiles);
      CHECK(static_cast<double>(c) <= ntiles * (1.0 - share) + 1e-6);
      CHECK(static_cast<double>(c) > ntiles * (1.0 - share) - per_round);
    }
    CHECK(helper_cluster_tiles(ntiles, 1.0, per_round) == 0);
    CHECK(helper_cluster_tiles(ntiles, 2.0, per_round) == 0);  // clamped to 1
    CHECK(helper_cluster_tiles(ntiles, -1.0, per_round) == ntiles / per_round * per_round);
    CHECK(helper_cluster_tiles(100, 0.0, per_round) == 0);     // less than a round
    CHECK(helper_cluster_tiles(0, 0.3, per_round) == 0);
    CHECK(helper_cluster_tiles(ntiles, 0.3, 0) == 0);
  }
  if (failures) {
    printf("%d checks failed\n", failures);
    return 1;
  }
  printf("ok\n");
  return 0;
}
