// How a single-pass ship launch splits its tiles between the cluster kernel
// and the global-atomic helper on the SMs its clusters leave idle, and how a
// stream's share for the helper follows the launches' reports.  Pure host
// arithmetic (no CUDA calls), so that the CPU tests can drive it with
// synthetic reports.
#pragma once

#include <stdint.h>

namespace dsmh {

// The helper's speed per idle SM relative to a cluster SM's (global atomics
// against the ship kernel, measured on uniform keys); it sets the helper's
// share of the tiles until a stream has reported how the split went.
constexpr double kHelperRelativeRate = 0.42;
// Bounds of the share, and of the step a report moves it by.
constexpr double kHelperShareMin = 0.01, kHelperShareMax = 0.6;
constexpr double kHelperGainMin = 0.05, kHelperGainMax = 0.75;

// The share the idle SMs would finish in the time the clusters take for
// theirs: idle * r / (active + idle * r).
inline double helper_prior(int active_sms, int idle_sms) {
  const double idle = idle_sms * kHelperRelativeRate;
  return idle / (active_sms + idle);
}

// One stream's learned share for one kernel kind.
struct HelperShare {
  double share = 0.0;       // 0: nothing learned yet
  double gain = 0.0;        // step towards a report; 0: no report taken yet
  int last_sign = 0;        // direction of the last correction
  uint32_t valid_from = 0;  // first launch (count) made at the current share
};

// A report counts only if its launch ran with the current share: calls
// enqueued far ahead of the GPU see reports of launches made with an older
// share, and acting on those made the share overshoot.
inline bool helper_report_current(const HelperShare& h, uint32_t launch) {
  return static_cast<int32_t>(launch - h.valid_from) >= 0;
}

// Moves the share part of the way to a report's target (the share at which
// helper and clusters would have finished together), within
// [kHelperShareMin, kHelperShareMax].  The step starts at kHelperGainMax,
// halves (down to kHelperGainMin) whenever the correction changes direction
// and grows by a quarter while it keeps its direction: where the helper's
// pace depends on which tiles it gets (runs in the last half of the keys and
// uniform keys before them: the target then moves several times as far as
// the share), full steps made the share swing around its optimum.  A target
// outside (0, 1) is ignored (returns false).  When the share moves, reports
// of launches up to `last_launch` (the latest count handed out) no longer
// count.
inline bool helper_share_step(HelperShare& h, float target, uint32_t last_launch) {
  if (!(target > 0.0f && target < 1.0f)) return false;
  const double before = h.share;
  const int sign = target > h.share ? 1 : -1;
  if (h.gain <= 0.0)
    h.gain = kHelperGainMax;
  else if (h.last_sign != 0 && sign != h.last_sign)
    h.gain = h.gain * 0.5 < kHelperGainMin ? kHelperGainMin : h.gain * 0.5;
  else
    h.gain = h.gain * 1.25 > kHelperGainMax ? kHelperGainMax : h.gain * 1.25;
  h.last_sign = sign;
  h.share += h.gain * (target - h.share);
  h.share = h.share < kHelperShareMin ? kHelperShareMin
                                      : (h.share > kHelperShareMax ? kHelperShareMax : h.share);
  if (h.share != before) h.valid_from = last_launch + 1u;
  return true;
}

// The cluster kernel's tiles at helper share `share` (clamped to [0, 1]):
// ntiles * (1 - share), rounded down to whole rounds of per_round tiles.  The
// helper takes the rest, so with share 0 it gets only the last partial round.
inline uint32_t helper_cluster_tiles(uint32_t ntiles, double share, uint64_t per_round) {
  share = share < 0.0 ? 0.0 : (share > 1.0 ? 1.0 : share);
  if (per_round == 0) return 0;
  return static_cast<uint32_t>(static_cast<uint64_t>(static_cast<double>(ntiles) * (1.0 - share)) /
                               per_round * per_round);
}

}  // namespace dsmh
