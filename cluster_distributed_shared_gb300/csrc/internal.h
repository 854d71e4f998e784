// Internal interfaces between the kernel translation unit and the host layer
// of libdsmemhist.  Not installed; the public C ABI is include/dsmem_hist.h.
#pragma once

#include <stdint.h>
#include <cuda_runtime_api.h>

#include "dsmem_hist.h"


namespace dsmh {

// Keys every thread handles per unrolled step of the streaming loop: four
// 16-byte vectors of four int32 keys.
constexpr int kVecPerThread = 4;
constexpr int kKeysPerThreadStep = 4 * kVecPerThread;
// The planner gives every CTA of the direct kernel at least this many
// unrolled steps of work, and every CTA of the ship kernel at least this many
// rounds (kShipThreads * keys_per_thread keys each).
constexpr int kMinStepsPerCta = 4;
constexpr int kMinShipRoundsPerCta = 2;
// Default cap on one CTA's counter slice: 128 KiB leaves room for a second
// small allocation per SM while keeping the slice count at the published
// cluster sizes (2 x 32768 bins, 8 x 32768, 16 x 32768).
constexpr int kDefaultSliceCapBytes = 128 * 1024;
// Scratch bound the planner keeps the partial rows under when it picks C.
constexpr int64_t kMaxAutoScratchBytes = int64_t{1} << 30;
// The ship kernel indexes 512-byte warp tiles with 32-bit integers (and adds
// up to three rounds of tiles to them): it takes fewer keys than this.
constexpr int64_t kShipMaxKeys = int64_t{1} << 38;
// Threads per CTA of the ship kernel.
constexpr int kShipThreads = DSMEM_HIST_SHIP_THREADS;
// Shared memory the runtime reserves per CTA on sm_90 and later.
constexpr int kSmemReservedPerCta = 1024;

// Arguments of one cluster-histogram launch (passed by value).
struct ClusterHistArgs {
  const int32_t* keys;
  int64_t n;
  uint32_t* partials;   // [num_clusters][stride] u32, one row per cluster
  uint32_t num_bins;
  uint32_t S;           // counters per CTA slice (multiple of 4)
  uint64_t magic;       // floor(2^40 / S) + 1: owner = (rel * magic) >> 40
  uint32_t passes;      // bin ranges of P*S bins
  uint64_t stride;      // partial row stride (u32 elements, multiple of 4)
  uint32_t head;        // keys before the first 16-byte boundary of `keys` (0..3, <= n)
  uint32_t accumulate;  // 1: add the slice into the partial row, 0: overwrite it
  uint32_t sub_vectors; // ship kernel: rows of each owner's staging block
  // Ship kernel error channel and wait bound.  `status` (may be null) is this
  // call's word in pinned, host-mapped memory: a bounded inbox wait that gives
  // up sets bit 0 there (and in the device-wide status word), so the next call
  // on the same stream can report it without a device synchronisation.
  uint32_t* status;
  long long wait_cycles;    // bound of one inbox wait (clock64 cycles)
  uint32_t withhold_last;   // test only: senders skip the last round's arrival and stores
  uint32_t hot_bin;         // ship kernel: the plan's hot bin, 0xFFFFFFFF for none
  // Helper and mop-up kernels (single-pass ship launches with a helper; the
  // cluster kernel itself is launched on the first cluster_tiles tiles only,
  // 128 keys each after `head`, and reads none of these): the helper's range
  // is [cluster_tiles, cluster_tiles + helper_tiles), and `queue` (zeroed
  // before the launches) counts its claimed tiles.
  uint32_t cluster_tiles;
  uint32_t helper_tiles;
  uint32_t* queue;
  // The mop-up kernel's first CTA writes (helper_seq << 32) | (bits of a
  // float: the helper's share at which both sides would have finished
  // together) to this pinned, host-mapped word (may be null), from which the
  // next launch on the stream sets the helper's share.  The zeroed
  // kHelperQueueBytes at `queue`: u32 tile counter, u32 report flag, u64
  // globaltimer of the helper's start, u64 globaltimer of its end, u32
  // helper CTAs finished.
  unsigned long long* helper_report;
  uint32_t helper_seq;
};
constexpr int64_t kHelperQueueBytes = 32;

// The global-atomic helper on the SMs a ship launch leaves idle: tiles per
// claim and tiles loaded at a time (a claim counted in two batches gives the
// next claim twice as long to return), threads per CTA, the direct-mapped
// cache of frequent keys in its shared memory (slots of a key and a count),
// and the fewest keys for which a launch takes a helper.
constexpr uint32_t kHelperTiles = 16;
constexpr uint32_t kHelperBatch = 8;
constexpr int kHelperThreads = 1024;
constexpr int kHelperSlotsLog2 = 13;
constexpr uint32_t kHelperSlots = 1u << kHelperSlotsLog2;
constexpr int kHelperSmemBytes = 8 << kHelperSlotsLog2;
constexpr uint32_t kNoKey = 0xFFFFFFFFu;
constexpr int64_t kHelperMinKeys = int64_t{1} << 24;
// Fewest idle SMs for which a plan takes the helper.
constexpr int64_t kHelperMinIdleSms = 4;

// A plan's partial rows (one per cluster, plus the helper's) and its
// scratch: the rows, then (with the helper) kHelperQueueBytes of tile
// counter and timing.
inline void set_partial_rows(dsmem_hist_plan_t* p, bool helper) {
  p->partial_rows = p->num_clusters + (helper ? 1 : 0);
  p->workspace_bytes = static_cast<int64_t>(p->partial_rows) * p->partial_stride * 4 +
                       (helper ? kHelperQueueBytes : 0);
}

// The mop-up kernel after a ship launch with a helper: threads per CTA and
// tiles per claim (two per warp).
constexpr int kMopThreads = 512;
constexpr uint32_t kMopTiles = 2 * (kMopThreads / 32);

// Streams per device with their own status words (later streams share the
// last slot).
constexpr int kStatusSlots = 64;

// Default bound of one inbox wait: ~1e8 cycles, about 50 ms at 2 GHz.
constexpr long long kDefaultWaitCycles = 100000000ll;

// Launches (all asynchronous on `stream`).
cudaError_t launch_cluster_hist(const dsmem_hist_plan_t& plan, const ClusterHistArgs& args,
                                cudaStream_t stream);
// With hot_word and seq_word non-null and hot_min > 0 the reduction also
// stamps *seq_word with seq and writes (seq << 32) | bin to *hot_word (both
// pinned, host-mapped) for a bin holding at least hot_min keys, if any does.
cudaError_t launch_reduce_partials(const uint32_t* partials, uint64_t stride,
                                   uint32_t num_clusters, uint32_t num_bins, uint32_t* bins,
                                   cudaStream_t stream, uint32_t hot_min = 0,
                                   unsigned long long* hot_word = nullptr,
                                   uint32_t* seq_word = nullptr, uint32_t seq = 0);
// The helper: `ctas` CTAs of kHelperThreads threads and kHelperSmemBytes of
// shared memory (prepare_ship_helper sets the limit once per device) count
// the tiles of args' helper range they claim from args.queue into `row`.
cudaError_t prepare_ship_helper();
// The mop-up: `ctas` CTAs report the split, count the ragged tail, and
// count the helper's tiles still unclaimed into `row`.
cudaError_t launch_ship_mop_up(const ClusterHistArgs& args, uint32_t* row, int ctas,
                               cudaStream_t stream);
cudaError_t launch_ship_helper(const ClusterHistArgs& args, uint32_t* row, int ctas,
                               cudaStream_t stream);
cudaError_t launch_global_atomic(const int32_t* keys, int64_t n, uint32_t num_bins,
                                 uint32_t* bins, cudaStream_t stream);
// Work-free control kernel with a plan's grid, cluster and shared memory.
cudaError_t launch_cluster_control(const dsmem_hist_plan_t& plan, uint32_t* sink,
                                   cudaStream_t stream);

// Ship kernel (cluster_ship.cu; its staging size is computed by the planner).
uint32_t ship_staging_bytes(int cluster_size, int rows);
cudaError_t prepare_ship_kernel(int keys_per_thread, int smem_bytes);
cudaError_t query_ship_active_clusters(int keys_per_thread, int cluster_size, int smem_bytes,
                                       int* out);
cudaError_t launch_cluster_ship(const dsmem_hist_plan_t& plan, const ClusterHistArgs& args,
                                cudaStream_t stream);
// Reads (synchronously) and clears the ship kernel's device status word on
// the current device: bit 0 = a bounded inbox wait gave up.
cudaError_t read_and_clear_ship_status(uint32_t* out);

// Sets the kernel attributes a shape needs (dynamic shared memory above
// 48 KiB, non-portable cluster sizes) on the current device.
cudaError_t prepare_cluster_kernel(int aggregate, int smem_bytes);
// Occupancy query: clusters of this shape that can be resident at once.
cudaError_t query_max_active_clusters(int aggregate, int cluster_size, int block_threads,
                                      int smem_bytes, int* out);
// Largest co-schedulable cluster size (cudaOccupancyMaxPotentialClusterSize)
// for the direct and the ship kernel at a given shape.
cudaError_t query_max_potential_cluster_size(int aggregate, int block_threads, int smem_bytes,
                                             int* out);
cudaError_t query_ship_potential_cluster_size(int keys_per_thread, int smem_bytes, int* out);

// The whole histogram with partial rows in caller-supplied device memory of
// at most max_rows_bytes (api.cpp; used by static_scratch.cu).
int run_with_fixed_scratch(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
                           uint32_t* scratch, int64_t max_rows_bytes, cudaStream_t stream);
// Records a message for dsmem_hist_last_error and returns `code`.
int record_error(int code, const char* what);

// Planner (pure host logic, planner.cpp).
int plan_shape(const dsmem_hist_device_t* dev, int32_t num_bins, int64_t n,
               const dsmem_hist_request_t* req, int32_t max_active_clusters,
               dsmem_hist_plan_t* out, const char** why);
uint64_t owner_magic(uint32_t S);

}  // namespace dsmh
