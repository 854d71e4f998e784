// Cluster-shape planner: pure host logic, no CUDA calls.
//
// Inputs: the bin count, the key count, the device's shared-memory and
// cluster limits ("Thread Block Clusters and Distributed Shared Memory":
// clusters of up to 8 CTAs portably, 16 as an opt-in; "@dynshared": more than
// 48 KB of shared memory per CTA only as dynamic shared memory requested at
// launch) and, when known, the occupancy answer for the chosen shape.
//
// Policy:
//   S_max   = slice cap / 4 counters, rounded down to a multiple of 4
//   P       = smallest power of two >= 2 with P * S_max >= num_bins, capped
//             at the device's largest cluster (forced P taken as given)
//   passes  = ceil(num_bins / (P * S_max)); S = ceil(ceil(num_bins / passes) / P)
//             rounded up to a multiple of 4 (the page's kernel needs
//             P * S == num_bins exactly; here the last CTA's slice may have
//             a few never-hit counters instead, and no bin is dropped)
//   kernel  = SHIP (keys shipped to owners as 16-bit indices, local atomics)
//             when P >= 2 and the slice plus its staging fit one CTA: 8 keys
//             per thread per round if that fits, else 4, with staging rows
//             holding twice the expected entries per column (at least 1.5
//             times); else DIRECT
//   threads = kShipThreads (896) for SHIP; for DIRECT 1024 when only one CTA fits an SM,
//             else 512
//   C       = min(resident clusters, clusters needed so each CTA gets at
//             least kMinShipRoundsPerCta rounds (SHIP) or kMinStepsPerCta
//             unrolled steps (DIRECT) of keys, clusters whose partial rows
//             fit kMaxAutoScratchBytes), at least 1
//   helper  = one more partial row, for the global-atomic helper kernel on
//             the SMs the clusters leave idle, when the plan is a
//             single-pass SHIP plan of at least kHelperMinKeys keys and at
//             least kHelperMinIdleSms SMs stay idle
#include <stdint.h>

#include "internal.h"

namespace dsmh {

uint64_t owner_magic(uint32_t S) { return ((uint64_t{1} << 40) / S) + 1; }

// Shared memory the ship kernel needs beside the slice; the kernel lays it
// out in this order: 32 padding counters after the slice, three cursor sets
// u32[P + 1][32], inbox headers u32[2][16] plus a 16-bit sink per lane,
// three mbarriers and a flag (256 bytes), then two staging buffers and two
// inbox buffers of P blocks of `rows` rows of 64 bytes.
uint32_t ship_staging_bytes(int cluster_size, int rows) {
  const uint32_t P = static_cast<uint32_t>(cluster_size), q = static_cast<uint32_t>(rows);
  return 4u * 32u + 3u * 4u * 32u * (P + 1u) + 256u + 4u * P * 64u * q;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

static int ctas_per_sm(const dsmem_hist_device_t* dev, int smem_bytes, int threads) {
  int by_smem = dev->max_smem_per_sm / (smem_bytes + kSmemReservedPerCta);
  int by_threads = dev->max_threads_per_sm / threads;
  int c = by_smem < by_threads ? by_smem : by_threads;
  return c < 32 ? c : 32;
}

int plan_shape(const dsmem_hist_device_t* dev, int32_t num_bins, int64_t n,
               const dsmem_hist_request_t* req, int32_t max_active_clusters,
               dsmem_hist_plan_t* out, const char** why) {
  static const dsmem_hist_request_t kNoRequest = {0, 0, 0, -1, 0, -1};
  if (!req) req = &kNoRequest;
  *why = "";
  if (!dev || !out) { *why = "null device or plan pointer"; return DSMEM_HIST_EINVAL; }
  if (num_bins < 1) { *why = "num_bins must be >= 1"; return DSMEM_HIST_EINVAL; }
  if (n < 0) { *why = "n must be >= 0"; return DSMEM_HIST_EINVAL; }
  if (dev->cc_major < 9) {
    *why = "thread-block clusters need compute capability 9.0 or newer";
    return DSMEM_HIST_EUNSUPPORTED;
  }
  if (dev->sm_count < 1 || dev->max_smem_per_block_optin < 1024 || dev->max_threads_per_sm < 64) {
    *why = "device description incomplete";
    return DSMEM_HIST_EINVAL;
  }

  int slice_cap = kDefaultSliceCapBytes;
  if (req->max_slice_bytes > 0) slice_cap = req->max_slice_bytes;
  if (slice_cap > dev->max_smem_per_block_optin) slice_cap = dev->max_smem_per_block_optin;
  if (slice_cap > dev->max_smem_per_sm - kSmemReservedPerCta)
    slice_cap = dev->max_smem_per_sm - kSmemReservedPerCta;
  const int64_t s_max = (slice_cap / 4) & ~int64_t{3};
  if (s_max < 4) { *why = "slice cap below 16 bytes"; return DSMEM_HIST_EINVAL; }

  const int max_cluster = dev->max_cluster_size < 1 ? 1 : dev->max_cluster_size;
  int P;
  if (req->cluster_size != 0) {
    if (req->cluster_size < 1 || req->cluster_size > 16) {
      *why = "cluster_size must be in [1, 16]";
      return DSMEM_HIST_EINVAL;
    }
    if (req->cluster_size > max_cluster) {
      *why = "requested cluster size exceeds the device's largest cluster";
      return DSMEM_HIST_EUNSUPPORTED;
    }
    P = req->cluster_size;
  } else {
    P = max_cluster >= 2 ? 2 : 1;
    while (2 * P <= max_cluster && P * s_max < num_bins) P *= 2;
  }

  const int64_t passes = ceil_div(num_bins, P * s_max);
  int64_t S = ceil_div(ceil_div(num_bins, passes), P);
  S = (S + 3) & ~int64_t{3};
  int smem = static_cast<int>(4 * S);

  if (req->block_threads != 0 &&
      (req->block_threads < 64 || req->block_threads > 1024 || (req->block_threads & 31))) {
    *why = "block_threads must be a multiple of 32 in [64, 1024]";
    return DSMEM_HIST_EINVAL;
  }
  if (req->kernel < -1 || req->kernel > DSMEM_HIST_KERNEL_SHIP) {
    *why = "kernel must be -1, DSMEM_HIST_KERNEL_DIRECT or DSMEM_HIST_KERNEL_SHIP";
    return DSMEM_HIST_EINVAL;
  }
  // Kernel choice: shipping whenever the cluster has remote owners and its
  // staging fits beside the slice (kShipThreads threads), else direct increments.
  int kernel = DSMEM_HIST_KERNEL_DIRECT, kpt = 0, nq = 0;
  const bool ship_ok_threads = req->block_threads == 0 || req->block_threads == kShipThreads;
  if (req->kernel == DSMEM_HIST_KERNEL_SHIP ||
      (req->kernel < 0 && P >= 2 && ship_ok_threads && n < kShipMaxKeys)) {
    if (n >= kShipMaxKeys) {
      *why = "the ship kernel takes fewer than 2^38 keys per call";
      return DSMEM_HIST_EINVAL;
    }
    if (P < 2 || !ship_ok_threads) {
      if (req->kernel == DSMEM_HIST_KERNEL_SHIP) {
        *why = "the ship kernel needs cluster_size >= 2 and its fixed block size";
        return DSMEM_HIST_EINVAL;
      }
    } else {
      // Staging rows per owner block: twice the expected entries per column
      // and round, or as many as fit down to 1.5 times; 8 keys per thread
      // and round before 4.
      for (int k = 8; k >= 4 && !kernel; k -= 4) {
        const int64_t expect = static_cast<int64_t>(kShipThreads / 32) * k;  // per column and round, times P
        const int64_t want = ceil_div(2 * expect, P), least = ceil_div(3 * expect, 2 * P);
        const int64_t room = static_cast<int64_t>(dev->max_smem_per_block_optin) - 4 * S -
                             ship_staging_bytes(P, 0);
        const int64_t room_sm = static_cast<int64_t>(dev->max_smem_per_sm) - kSmemReservedPerCta - 4 * S -
                                ship_staging_bytes(P, 0);
        const int64_t fit = (room < room_sm ? room : room_sm) / (4 * 64 * P);
        const int64_t q = want < fit ? want : fit;
        if (q >= least && q >= 1) {
          kernel = DSMEM_HIST_KERNEL_SHIP;
          kpt = k;
          nq = static_cast<int>(q);
          smem = static_cast<int>(4 * S + ship_staging_bytes(P, nq));
        }
      }
      if (!kernel && req->kernel == DSMEM_HIST_KERNEL_SHIP) {
        *why = "slice plus ship staging exceed the shared memory of one CTA";
        return DSMEM_HIST_EUNSUPPORTED;
      }
    }
  }

  int threads;
  if (kernel == DSMEM_HIST_KERNEL_SHIP) {
    threads = kShipThreads;
  } else if (req->block_threads != 0) {
    threads = req->block_threads;
  } else {
    threads = ctas_per_sm(dev, smem, 512) <= 1 ? 1024 : 512;
  }
  const int per_sm = ctas_per_sm(dev, smem, threads);
  if (per_sm < 1) {
    *why = "shape does not fit one SM";
    return DSMEM_HIST_EUNSUPPORTED;
  }

  const int64_t stride = (static_cast<int64_t>(num_bins) + 3) & ~int64_t{3};
  int64_t mac = max_active_clusters;
  if (mac <= 0) mac = static_cast<int64_t>(dev->sm_count) * per_sm / P;
  if (mac < 1) {
    *why = "no cluster of this shape can be resident";
    return DSMEM_HIST_EUNSUPPORTED;
  }
  int64_t C;
  if (req->num_clusters != 0) {
    if (req->num_clusters < 1 || req->num_clusters > (1 << 20)) {
      *why = "num_clusters must be in [1, 2^20]";
      return DSMEM_HIST_EINVAL;
    }
    C = req->num_clusters;
  } else {
    const int64_t keys_per_cluster =
        kernel == DSMEM_HIST_KERNEL_SHIP
            ? static_cast<int64_t>(P) * threads * kpt * kMinShipRoundsPerCta
            : static_cast<int64_t>(P) * threads * kKeysPerThreadStep * kMinStepsPerCta;
    const int64_t need = ceil_div(n > 0 ? n : 1, keys_per_cluster);
    C = need < mac ? need : mac;
    // Bound the partial rows' scratch for very large bin counts.
    const int64_t by_scratch = kMaxAutoScratchBytes / (4 * stride);
    if (C > by_scratch) C = by_scratch;
    if (C < 1) C = 1;
  }

  out->cluster_size = P;
  out->bins_per_cta = static_cast<int32_t>(S);
  out->passes = static_cast<int32_t>(passes);
  out->block_threads = threads;
  out->num_clusters = static_cast<int32_t>(C);
  out->smem_bytes = smem;
  // Direct kernel: __match_any_sync aggregation only on request (it costs
  // about as much as a remote increment on GB300).  Ship kernel: whole-tile
  // aggregation of runs is always on.
  out->aggregate = kernel == DSMEM_HIST_KERNEL_SHIP ? 1 : (req->aggregate > 0 ? 1 : 0);
  out->kernel = kernel;
  out->keys_per_thread = kpt;
  out->sub_vectors = nq;
  out->ctas_per_sm = per_sm;
  out->max_active_clusters = max_active_clusters > 0 ? max_active_clusters : 0;
  out->hot_bin = -1;
  if (req->hot_bin_valid > 0 && kernel == DSMEM_HIST_KERNEL_SHIP) {
    if (req->hot_bin < 0 || req->hot_bin >= num_bins) {
      *why = "hot_bin must lie in [0, num_bins)";
      return DSMEM_HIST_EINVAL;
    }
    out->hot_bin = req->hot_bin;
  }
  out->partial_stride = stride;
  const int64_t idle = static_cast<int64_t>(dev->sm_count) - C * P;
  const bool helper = kernel == DSMEM_HIST_KERNEL_SHIP && passes == 1 && n >= kHelperMinKeys &&
                      idle >= kHelperMinIdleSms;
  set_partial_rows(out, helper);
  return DSMEM_HIST_OK;
}

}  // namespace dsmh
