// C ABI of libdsmemhist: argument checks, per-device state, scratch from a
// stream-ordered memory pool, and the launch sequence
//   cluster_hist_kernel  (zero slices, stream keys, DSMEM increments, flush)
//   reduce_partials      (sum the clusters' partial rows into `bins`).
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>
#include <vector>
#include <string>
#include <tuple>

#include <cuda_runtime_api.h>

#include "dsmem_hist.h"
#include "helper_split.h"
#include "internal.h"

namespace dsmh {
namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(DSMEM_HIST_ECUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

struct DeviceState {
  bool ready = false;
  dsmem_hist_device_t dev = {};
  cudaMemPool_t pool = nullptr;
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ev_copied[2] = {nullptr, nullptr};
  cudaEvent_t ev_consumed[2] = {nullptr, nullptr};
  // Largest dynamic shared memory set so far per kernel variant: direct
  // (aggregate 0/1), ship (4 / 8 keys per thread).
  int prepared_direct[2] = {0, 0};
  int prepared_ship[2] = {0, 0};
  // (kernel, variant, P, threads, smem) -> resident clusters
  std::map<std::tuple<int, int, int, int, int>, int> occupancy;
  // (kernel, variant, threads, smem) -> largest co-schedulable cluster size
  std::map<std::tuple<int, int, int, int>, int> potential;
  std::mutex host_call;  // serialises dsmem_hist_host on this device
  // The helper kernel's streams (lowest priority, so the clusters launched
  // first keep their SMs) and their fork and join events, one set per
  // caller-stream slot, so that calls on different streams do not queue
  // behind each other's helpers; helper_call serialises their use.  Calls
  // without a stream slot use the last set.
  struct HelperStream {
    cudaStream_t stream = nullptr;         // the helper's, lowest priority
    cudaStream_t cluster_stream = nullptr; // the cluster kernel's, highest priority
    cudaEvent_t fork = nullptr, clusters_done = nullptr, join = nullptr;
  };
  HelperStream helper_streams[kStatusSlots + 1] = {};
  bool helper_prepared = false;
  std::mutex helper_call;
  // Per stream slot, under helper_call: the helper's learned share beside
  // the default and beside the hot-bin kernel (the best shares differ), the
  // last report taken, and the last sequence number handed out (2 * launch
  // count + kind).
  HelperShare helper[kStatusSlots][2] = {};
  uint32_t helper_taken[kStatusSlots] = {};
  uint32_t helper_seq[kStatusSlots] = {};
  // Per-stream words in pinned, host-mapped memory (h_status on the host,
  // d_status the same memory for the device), kStatusSlots of each kind: the
  // ship kernel's u32 status words; u32 sequence stamps, the number of the
  // latest histogram whose reduction has run on the slot; and u64 hot-bin
  // words, (seq << 32) | bin for a bin that held a sixth or more of the keys
  // of histogram seq.
  uint32_t* h_status = nullptr;
  uint32_t* d_status = nullptr;
  std::map<cudaStream_t, int> status_slot;
  // Per slot, host side: the last sequence number handed out, the bin count
  // of the latest histogram, and the first sequence number that had it (every
  // histogram from that one on had the same bin count).
  uint32_t slot_seq[kStatusSlots] = {};
  int32_t slot_bins[kStatusSlots] = {};
  uint32_t slot_bins_since[kStatusSlots] = {};
};

// Bytes of the host-mapped block: status words, sequence stamps, hot-bin words.
constexpr size_t kMappedBytes = kStatusSlots * (2 * sizeof(uint32_t) + 2 * sizeof(unsigned long long));
// The hot-bin kernel is chosen when one bin held at least 1/kHotShareDen of
// the keys of the previous histogram on the same stream.
constexpr int64_t kHotShareDen = 6;

// One stream's words; all null when the device has none (see stream_slot).
struct SlotRef {
  int slot = -1;
  uint32_t* h_status = nullptr;
  uint32_t* d_status = nullptr;
  uint32_t* h_seq = nullptr;
  uint32_t* d_seq = nullptr;
  unsigned long long* h_hot = nullptr;
  unsigned long long* d_hot = nullptr;
  unsigned long long* h_helper = nullptr;  // the helper's progress report
  unsigned long long* d_helper = nullptr;
};

// What the reduction of a histogram reports for later calls on its stream.
struct HotReport {
  uint32_t min_count = 0;  // 0: nothing
  unsigned long long* word = nullptr;
  uint32_t* seq_word = nullptr;
  uint32_t seq = 0;
};

std::mutex g_mutex;
std::map<int, DeviceState*> g_devices;

bool trace_enabled() {
  static int on = -1;
  if (on < 0) {
    const char* v = getenv("DSMEM_HIST_TRACE");
    on = (v && *v && strcmp(v, "0") != 0) ? 1 : 0;
  }
  return on == 1;
}

int env_int(const char* name, int fallback) {
  const char* v = getenv(name);
  if (!v || !*v) return fallback;
  return atoi(v);
}

// Per-device state for the current device; g_mutex must be held.
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  DeviceState*& st = g_devices[dev];
  if (!st) st = new DeviceState();
  if (!st->ready) {
    cudaDeviceProp p;
    if ((e = cudaGetDeviceProperties(&p, dev)) != cudaSuccess)
      return fail_cuda(e, "cudaGetDeviceProperties");
    st->dev.cc_major = p.major;
    st->dev.cc_minor = p.minor;
    st->dev.sm_count = p.multiProcessorCount;
    st->dev.max_smem_per_block_optin = static_cast<int32_t>(p.sharedMemPerBlockOptin);
    st->dev.max_smem_per_sm = static_cast<int32_t>(p.sharedMemPerMultiprocessor);
    st->dev.max_threads_per_sm = p.maxThreadsPerMultiProcessor;
    int cluster_launch = 0;
    cudaDeviceGetAttribute(&cluster_launch, cudaDevAttrClusterLaunch, dev);
    st->dev.max_cluster_size = (p.major >= 9 && cluster_launch) ? 16 : 1;
    st->ready = true;
  }
  *out = st;
  return DSMEM_HIST_OK;
}

// Test hooks, read at every call (documented in the header): a shorter
// bound for the ship kernel's inbox waits, a launch whose senders withhold
// their last round (so that owners' waits run out with nothing in flight),
// and a scratch allocation that fails.
long long wait_cycles_setting() {
  const char* v = getenv("DSMEM_HIST_TEST_WAIT_CYCLES");
  if (!v || !*v) return kDefaultWaitCycles;
  const long long c = atoll(v);
  return c < 1000 ? 1000 : (c > kDefaultWaitCycles ? kDefaultWaitCycles : c);
}
bool env_flag(const char* name) {
  const char* v = getenv(name);
  return v && *v && strcmp(v, "0") != 0;
}
bool injected_alloc_failure() { return env_flag("DSMEM_HIST_TEST_FAIL_ALLOC"); }

// This stream's words (host and device views); g_mutex must be held.  With
// may_alloc false, a device whose words were never allocated gets none.
int stream_slot(DeviceState* st, cudaStream_t stream, bool may_alloc, SlotRef* r) {
  *r = SlotRef{};
  if (!st->h_status) {
    if (!may_alloc) return DSMEM_HIST_OK;
    void* p = nullptr;
    cudaError_t e = cudaHostAlloc(&p, kMappedBytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) return fail_cuda(e, "cudaHostAlloc (status words)");
    memset(p, 0, kMappedBytes);
    void* dp = nullptr;
    if ((e = cudaHostGetDevicePointer(&dp, p, 0)) != cudaSuccess) {
      cudaFreeHost(p);
      return fail_cuda(e, "cudaHostGetDevicePointer (status words)");
    }
    st->h_status = static_cast<uint32_t*>(p);
    st->d_status = static_cast<uint32_t*>(dp);
  }
  auto it = st->status_slot.find(stream);
  int slot;
  if (it != st->status_slot.end()) {
    slot = it->second;
  } else {
    slot = std::min<int>(static_cast<int>(st->status_slot.size()), kStatusSlots - 1);
    st->status_slot[stream] = slot;
  }
  r->slot = slot;
  r->h_status = st->h_status + slot;
  r->d_status = st->d_status + slot;
  r->h_seq = st->h_status + kStatusSlots + slot;
  r->d_seq = st->d_status + kStatusSlots + slot;
  r->h_hot = reinterpret_cast<unsigned long long*>(st->h_status + 2 * kStatusSlots) + slot;
  r->d_hot = reinterpret_cast<unsigned long long*>(st->d_status + 2 * kStatusSlots) + slot;
  r->h_helper = reinterpret_cast<unsigned long long*>(st->h_status + 4 * kStatusSlots) + slot;
  r->d_helper = reinterpret_cast<unsigned long long*>(st->d_status + 4 * kStatusSlots) + slot;
  return DSMEM_HIST_OK;
}

// The hot bin for a histogram of n keys into num_bins bins on this stream
// slot, or -1.  It comes from the latest histogram whose reduction has run on
// the slot (its sequence stamp): if every histogram since had the same bin
// count, the bin it reported as holding a sixth or more of its keys.  Reports arrive
// asynchronously, so in a loop of calls this is one a few calls back; one
// with no hot bin switches the choice off again.  Also sets up *report for
// this call's reduction.  g_mutex must be held.
int32_t choose_hot_bin(DeviceState* st, const SlotRef& r, int64_t n, int32_t num_bins,
                       HotReport* report) {
  *report = HotReport{};
  if (r.slot < 0 || !r.h_hot) return -1;
  const uint32_t done = *reinterpret_cast<volatile uint32_t*>(r.h_seq);
  const unsigned long long w = *reinterpret_cast<volatile unsigned long long*>(r.h_hot);
  int32_t hot = -1;
  if (done != 0 && st->slot_bins[r.slot] == num_bins && done >= st->slot_bins_since[r.slot] &&
      static_cast<uint32_t>(w >> 32) == done && static_cast<uint32_t>(w) < static_cast<uint32_t>(num_bins))
    hot = static_cast<int32_t>(static_cast<uint32_t>(w));
  uint32_t seq = st->slot_seq[r.slot] + 1;
  if (seq == 0) {  // after 2^32 calls: start over
    seq = 1;
    st->slot_bins[r.slot] = 0;
  }
  st->slot_seq[r.slot] = seq;
  if (st->slot_bins[r.slot] != num_bins) {
    st->slot_bins[r.slot] = num_bins;
    st->slot_bins_since[r.slot] = seq;
  }
  const int64_t min_count = (n + kHotShareDen - 1) / kHotShareDen;
  if (n > 0 && min_count <= 0xFFFFFFFFll) {
    report->min_count = static_cast<uint32_t>(min_count);
    report->word = r.d_hot;
    report->seq_word = r.d_seq;
    report->seq = seq;
  }
  return hot;
}

// Takes the automatic choice into a ship-kernel plan (tracing it).
void use_hot_bin(dsmem_hist_plan_t* plan, int32_t chosen, const SlotRef& r) {
  if (chosen < 0 || plan->kernel != DSMEM_HIST_KERNEL_SHIP) return;
  plan->hot_bin = chosen;
  if (trace_enabled())
    fprintf(stderr, "[dsmem_hist] stream slot %d: bin %d held a sixth or more of the keys of a "
            "recent histogram -> hot-bin kernel\n", r.slot, chosen);
}

// Reports (once) a bounded wait that gave up in an earlier launch on this
// stream, as seen from the host without synchronising.
int take_pending_timeout(uint32_t* h) {
  if (!h || *reinterpret_cast<volatile uint32_t*>(h) == 0u) return DSMEM_HIST_OK;
  *reinterpret_cast<volatile uint32_t*>(h) = 0u;
  return fail(DSMEM_HIST_ETIMEOUT,
              "an earlier ship-kernel launch on this stream had a bounded inbox wait give up, so "
              "its histogram was wrong; this call enqueued nothing (call again)");
}

int ensure_pool(DeviceState* st) {
  if (st->pool) return DSMEM_HIST_OK;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaMemPoolProps props = {};
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  cudaError_t e = cudaMemPoolCreate(&st->pool, &props);
  if (e != cudaSuccess) {
    st->pool = nullptr;
    return fail_cuda(e, "cudaMemPoolCreate");
  }
  // Keep freed scratch in the pool between calls instead of returning it to
  // the driver at every synchronisation.
  uint64_t keep = UINT64_MAX;
  cudaMemPoolSetAttribute(st->pool, cudaMemPoolAttrReleaseThreshold, &keep);
  return DSMEM_HIST_OK;
}

// Sets the dynamic shared-memory attribute a plan's kernel needs (once per
// size increase).  g_mutex must be held.
int prepare_locked(DeviceState* st, const dsmem_hist_plan_t& p) {
  cudaError_t e = cudaSuccess;
  if (p.kernel == DSMEM_HIST_KERNEL_SHIP) {
    const int v = p.keys_per_thread == 8 ? 1 : 0;
    if (p.smem_bytes > st->prepared_ship[v]) {
      if ((e = prepare_ship_kernel(p.keys_per_thread, p.smem_bytes)) != cudaSuccess)
        return fail_cuda(e, "cudaFuncSetAttribute");
      st->prepared_ship[v] = p.smem_bytes;
    }
  } else if (p.smem_bytes > st->prepared_direct[p.aggregate]) {
    if ((e = prepare_cluster_kernel(p.aggregate, p.smem_bytes)) != cudaSuccess)
      return fail_cuda(e, "cudaFuncSetAttribute");
    st->prepared_direct[p.aggregate] = p.smem_bytes;
  }
  return DSMEM_HIST_OK;
}

// The helper's share for the next launch on the stream of `sr`: the share it
// has learned, else `prior`.  Each launch with a helper reports, from the
// mop-up kernel's first CTA, the share at which the helper and the
// clusters would have finished together (report_helper_share in the ship
// kernel's source); a new report of a launch made at the current share moves
// the share part of the way to it (helper_share_step).  Shares are kept
// apart for the default (kind 0) and the hot-bin kernel (kind 1); a report's
// sequence number carries its kind in bit 0 and the launch count above it.
// st->helper_call must be held.
double helper_share(DeviceState* st, const SlotRef* sr, int kind, double prior) {
  if (!sr || sr->slot < 0 || !sr->h_helper) return prior;
  const int slot = sr->slot;
  for (HelperShare& h : st->helper[slot])
    if (h.share <= 0.0) h.share = prior;
  const unsigned long long w = *reinterpret_cast<volatile unsigned long long*>(sr->h_helper);
  const uint32_t seq = static_cast<uint32_t>(w >> 32), bits = static_cast<uint32_t>(w);
  HelperShare& h = st->helper[slot][seq & 1u];
  if (seq != 0 && seq != st->helper_taken[slot] && helper_report_current(h, seq >> 1)) {
    st->helper_taken[slot] = seq;
    float target = 0.0f;
    memcpy(&target, &bits, sizeof target);
    const double before = h.share;
    if (helper_share_step(h, target, st->helper_seq[slot] >> 1) && trace_enabled())
      fprintf(stderr, "[dsmem_hist] stream slot %d: helper launch %u (kind %u) reports share %.4f "
              "-> share %.4f -> %.4f\n", slot, seq >> 1, seq & 1u, target, before, h.share);
  }
  return st->helper[slot][kind].share;
}

// Launches a plan.  With `st` non-null and a helper row in the plan
// (partial_rows > num_clusters), the ship kernel is launched on the first
// tiles and the global-atomic helper, on the SMs the clusters leave idle,
// takes the rest: its share starts at what the idle SMs would finish in the
// time the clusters take for theirs and then follows the stream's reports
// (helper_share); the clusters' tiles are rounded down to whole rounds.
// The cluster kernel and the helper run on two library streams forked from
// and joined back into `stream`; the tile counter and (unless accumulating)
// the helper's row are zeroed on `stream` before the fork.  The mop-up
// kernel follows the cluster kernel on `stream`.
cudaError_t launch_plan(const dsmem_hist_plan_t& plan, ClusterHistArgs args, cudaStream_t stream,
                        DeviceState* st = nullptr, const SlotRef* sr = nullptr) {
  if (plan.kernel != DSMEM_HIST_KERNEL_SHIP) return launch_cluster_hist(plan, args, stream);
  const uint32_t ntiles = static_cast<uint32_t>(((args.n - args.head) >> 2) >> 5);
  args.cluster_tiles = ntiles;
  args.helper_tiles = 0;
  args.queue = nullptr;
  if (!st || plan.partial_rows <= plan.num_clusters) return launch_cluster_ship(plan, args, stream);

  cudaError_t e;
  std::lock_guard<std::mutex> g(st->helper_call);
  if (!st->helper_prepared) {
    if ((e = prepare_ship_helper()) != cudaSuccess) return e;
    st->helper_prepared = true;
  }
  DeviceState::HelperStream& hs = st->helper_streams[sr && sr->slot >= 0 ? sr->slot : kStatusSlots];
  if (!hs.stream) {
    int least = 0, greatest = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess ||
        (e = cudaStreamCreateWithPriority(&hs.stream, cudaStreamNonBlocking, least)) != cudaSuccess ||
        (e = cudaStreamCreateWithPriority(&hs.cluster_stream, cudaStreamNonBlocking, greatest)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hs.fork, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hs.clusters_done, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hs.join, cudaEventDisableTiming)) != cudaSuccess)
      return e;
  }
  const int active = plan.num_clusters * plan.cluster_size;
  const int idle = st->dev.sm_count > active ? st->dev.sm_count - active : 0;
  const int kind = args.hot_bin != 0xFFFFFFFFu ? 1 : 0;
  double share = helper_share(st, sr, kind, helper_prior(active, idle));
  if (const char* v = getenv("DSMEM_HIST_HELPER_SHARE")) share = atof(v);  // sweeps
  const uint64_t per_round = static_cast<uint64_t>(active) * (kShipThreads / 32) * (plan.keys_per_thread / 4);
  args.cluster_tiles = helper_cluster_tiles(ntiles, share, per_round);
  args.helper_tiles = ntiles - args.cluster_tiles;
  uint32_t* row = args.partials + static_cast<size_t>(plan.num_clusters) * args.stride;
  args.queue = args.partials + static_cast<size_t>(plan.partial_rows) * args.stride;
  if (sr && sr->slot >= 0 && sr->d_helper) {
    // A new sequence number tells this launch's report from older ones;
    // bit 0 is the kernel kind.
    const int slot = sr->slot;
    uint32_t seq = st->helper_seq[slot] + 2u;
    if (seq < 2u) seq = 2u;
    st->helper_seq[slot] = seq;
    args.helper_report = sr->d_helper;
    args.helper_seq = seq | static_cast<uint32_t>(kind);
  }
  // The counter and the helper's row are zeroed on `stream` before the
  // fork.  Then the cluster kernel goes on the highest-priority stream and
  // the helper on the lowest, both forked from `stream`: when both are ready
  // to start, the clusters' CTAs are dispatched first, and the helper's CTAs
  // fill the SMs they leave idle.  (When the helper's CTAs, or a memset's,
  // got to SMs a cluster needed first, that cluster waited for the helper,
  // and some streams settled at 1.72 instead of 1.31 ms on the run-heavy
  // workload.)  The mop-up kernel follows the cluster kernel on `stream` and
  // takes the helper's tiles it has not claimed by then.  The cluster kernel
  // sees only its own tiles (and the unaligned head).
  ClusterHistArgs cargs = args;
  cargs.n = static_cast<int64_t>(args.head) + (static_cast<int64_t>(args.cluster_tiles) << 7);
  if ((e = cudaMemsetAsync(args.queue, 0, kHelperQueueBytes, stream)) != cudaSuccess ||
      (!args.accumulate &&
       (e = cudaMemsetAsync(row, 0, sizeof(uint32_t) * args.stride, stream)) != cudaSuccess) ||
      (e = cudaEventRecord(hs.fork, stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hs.cluster_stream, hs.fork, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hs.stream, hs.fork, 0)) != cudaSuccess ||
      (e = launch_cluster_ship(plan, cargs, hs.cluster_stream)) != cudaSuccess ||
      (e = cudaEventRecord(hs.clusters_done, hs.cluster_stream)) != cudaSuccess ||
      (e = launch_ship_helper(args, row, idle, hs.stream)) != cudaSuccess ||
      (e = cudaEventRecord(hs.join, hs.stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(stream, hs.clusters_done, 0)) != cudaSuccess ||
      (e = launch_ship_mop_up(args, row, st->dev.sm_count, stream)) != cudaSuccess)
    return e;
  return cudaStreamWaitEvent(stream, hs.join, 0);
}

// Plans for the current device, confirming the shape with the occupancy
// API; in automatic mode a cluster size the device cannot hold is halved
// (more passes) until one fits.  g_mutex must be held.
int plan_locked(DeviceState* st, int32_t num_bins, int64_t n, const dsmem_hist_request_t* req_in,
                dsmem_hist_plan_t* out) {
  dsmem_hist_request_t req = {0, 0, 0, -1, 0, -1, 0, 0};
  if (req_in) req = *req_in;
  // Environment overrides for sweeps (only where the caller left a field open).
  if (req.cluster_size == 0) req.cluster_size = env_int("DSMEM_HIST_CLUSTER", 0);
  if (req.block_threads == 0) req.block_threads = env_int("DSMEM_HIST_BLOCK", 0);
  if (req.num_clusters == 0) req.num_clusters = env_int("DSMEM_HIST_GRID", 0);
  if (req.aggregate < 0) req.aggregate = env_int("DSMEM_HIST_AGGREGATE", -1);
  if (req.kernel < 0) req.kernel = env_int("DSMEM_HIST_KERNEL", -1);

  dsmem_hist_device_t dev = st->dev;
  for (;;) {
    const char* why = "";
    int rc = plan_shape(&dev, num_bins, n, &req, 0, out, &why);
    if (rc != DSMEM_HIST_OK) return fail(rc, "plan: %s", why);
    cudaError_t e;
    if ((rc = prepare_locked(st, *out))) return rc;
    const bool ship = out->kernel == DSMEM_HIST_KERNEL_SHIP;
    const int variant = ship ? out->keys_per_thread : out->aggregate;
    if (req.cluster_size == 0) {
      // An automatic cluster size stays within the largest cluster this shape
      // can be co-scheduled with (cudaOccupancyMaxPotentialClusterSize).
      auto pkey = std::make_tuple(out->kernel, variant, out->block_threads, out->smem_bytes);
      auto pit = st->potential.find(pkey);
      int pcs = 0;
      if (pit != st->potential.end()) {
        pcs = pit->second;
      } else {
        e = ship ? query_ship_potential_cluster_size(out->keys_per_thread, out->smem_bytes, &pcs)
                 : query_max_potential_cluster_size(out->aggregate, out->block_threads,
                                                    out->smem_bytes, &pcs);
        if (e != cudaSuccess) {
          cudaGetLastError();
          pcs = 0;
        }
        st->potential[pkey] = pcs;
      }
      if (pcs >= 1 && pcs < out->cluster_size && pcs < dev.max_cluster_size) {
        dev.max_cluster_size = pcs;
        continue;
      }
    }
    auto key = std::make_tuple(out->kernel, variant, out->cluster_size, out->block_threads,
                               out->smem_bytes);
    auto it = st->occupancy.find(key);
    int mac = 0;
    if (it != st->occupancy.end()) {
      mac = it->second;
    } else {
      e = ship ? query_ship_active_clusters(out->keys_per_thread, out->cluster_size,
                                            out->smem_bytes, &mac)
               : query_max_active_clusters(out->aggregate, out->cluster_size, out->block_threads,
                                           out->smem_bytes, &mac);
      if (e != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of a refused shape
        mac = 0;
      }
      st->occupancy[key] = mac;
    }
    if (mac > 0) {
      rc = plan_shape(&dev, num_bins, n, &req, mac, out, &why);
      if (rc != DSMEM_HIST_OK) return fail(rc, "plan: %s", why);
      break;
    }
    if (out->kernel == DSMEM_HIST_KERNEL_SHIP && req.kernel < 0) {
      req.kernel = DSMEM_HIST_KERNEL_DIRECT;  // shipping shape not resident: try direct
      continue;
    }
    if (req.cluster_size != 0 || out->cluster_size <= 1)
      return fail(DSMEM_HIST_EUNSUPPORTED,
                  "cluster of %d CTAs x %d threads x %d B shared memory cannot be resident",
                  out->cluster_size, out->block_threads, out->smem_bytes);
    dev.max_cluster_size = out->cluster_size / 2;
  }
  if (out->partial_rows > out->num_clusters && env_int("DSMEM_HIST_HELPER", 1) == 0)
    set_partial_rows(out, false);
  if (trace_enabled())
    fprintf(stderr,
            "[dsmem_hist] bins=%d n=%lld -> kernel=%s P=%d S=%d passes=%d threads=%d C=%d "
            "smem=%d agg=%d kpt=%d nq=%d ctas/SM=%d max_active_clusters=%d scratch=%lld B\n",
            num_bins, static_cast<long long>(n),
            out->kernel == DSMEM_HIST_KERNEL_SHIP ? "ship" : "direct", out->cluster_size,
            out->bins_per_cta, out->passes, out->block_threads, out->num_clusters,
            out->smem_bytes, out->aggregate, out->keys_per_thread, out->sub_vectors,
            out->ctas_per_sm, out->max_active_clusters,
            static_cast<long long>(out->workspace_bytes));
  return DSMEM_HIST_OK;
}

int check_args(const void* keys, int64_t n, int32_t num_bins, const void* bins) {
  if (n < 0) return fail(DSMEM_HIST_EINVAL, "n must be >= 0 (got %lld)", static_cast<long long>(n));
  if (num_bins < 1) return fail(DSMEM_HIST_EINVAL, "num_bins must be >= 1 (got %d)", num_bins);
  if (!bins) return fail(DSMEM_HIST_EINVAL, "bins is NULL");
  if (n > 0 && !keys) return fail(DSMEM_HIST_EINVAL, "keys is NULL with n > 0");
  if ((reinterpret_cast<uintptr_t>(keys) & 3u) || (reinterpret_cast<uintptr_t>(bins) & 3u))
    return fail(DSMEM_HIST_EINVAL, "keys and bins must be 4-byte aligned");
  return DSMEM_HIST_OK;
}

uint32_t head_keys(const int32_t* keys, int64_t n) {
  const uint32_t h = static_cast<uint32_t>(((16u - (reinterpret_cast<uintptr_t>(keys) & 15u)) & 15u) / 4u);
  return n < h ? static_cast<uint32_t>(n) : h;
}

ClusterHistArgs make_args(const dsmem_hist_plan_t& plan, const int32_t* keys, int64_t n,
                          int32_t num_bins, uint32_t* partials, int accumulate) {
  ClusterHistArgs a;
  a.keys = keys;
  a.n = n;
  a.partials = partials;
  a.num_bins = static_cast<uint32_t>(num_bins);
  a.S = static_cast<uint32_t>(plan.bins_per_cta);
  a.magic = owner_magic(a.S);
  a.passes = static_cast<uint32_t>(plan.passes);
  a.stride = static_cast<uint64_t>(plan.partial_stride);
  a.head = head_keys(keys, n);
  a.accumulate = static_cast<uint32_t>(accumulate);
  a.sub_vectors = static_cast<uint32_t>(plan.sub_vectors);
  a.status = nullptr;
  a.wait_cycles = wait_cycles_setting();
  a.withhold_last = env_flag("DSMEM_HIST_TEST_WITHHOLD_LAST_ROUND") ? 1u : 0u;
  a.hot_bin = plan.kernel == DSMEM_HIST_KERNEL_SHIP && plan.hot_bin >= 0
                  ? static_cast<uint32_t>(plan.hot_bin) : 0xFFFFFFFFu;
  a.cluster_tiles = 0xFFFFFFFFu;  // launch_plan sets the helper's split
  a.helper_tiles = 0;
  a.queue = nullptr;
  a.helper_report = nullptr;
  a.helper_seq = 0;
  return a;
}

int run_device(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
               const dsmem_hist_request_t* req, cudaStream_t stream) {
  int rc = check_args(keys, n, num_bins, bins);
  if (rc) return rc;
  dsmem_hist_plan_t plan;
  DeviceState* st = nullptr;
  SlotRef sr;
  HotReport hot_report;
  {
    std::lock_guard<std::mutex> g(g_mutex);
    if ((rc = device_state(&st))) return rc;
    if ((rc = stream_slot(st, stream, true, &sr))) return rc;
    if ((rc = take_pending_timeout(sr.h_status))) return rc;
    if ((rc = plan_locked(st, num_bins, n, req, &plan))) return rc;
    if ((rc = ensure_pool(st))) return rc;
    // The hot-bin kernel: on the caller's request, or (unless the caller
    // turned it off) when the previous histogram on this stream had a hot bin.
    const int32_t chosen = choose_hot_bin(st, sr, n, num_bins, &hot_report);
    if (!req || req->hot_bin_valid == 0) use_hot_bin(&plan, chosen, sr);
  }
  cudaError_t e;
  if (n == 0) {
    e = cudaMemsetAsync(bins, 0, sizeof(uint32_t) * static_cast<size_t>(num_bins), stream);
    return e == cudaSuccess ? DSMEM_HIST_OK : fail_cuda(e, "cudaMemsetAsync");
  }
  if (injected_alloc_failure())
    return fail(DSMEM_HIST_ENOMEM, "scratch pool: %lld bytes: allocation failure injected by "
                "DSMEM_HIST_TEST_FAIL_ALLOC", static_cast<long long>(plan.workspace_bytes));
  void* scratch = nullptr;
  e = cudaMallocFromPoolAsync(&scratch, static_cast<size_t>(plan.workspace_bytes), st->pool, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DSMEM_HIST_ENOMEM, "scratch pool: %lld bytes: %s",
                static_cast<long long>(plan.workspace_bytes), cudaGetErrorString(e));
  }
  uint32_t* partials = static_cast<uint32_t*>(scratch);
  ClusterHistArgs args = make_args(plan, keys, n, num_bins, partials, 0);
  args.status = sr.d_status;
  e = launch_plan(plan, args, stream, st, &sr);
  if (e == cudaSuccess)
    e = launch_reduce_partials(partials, args.stride, static_cast<uint32_t>(plan.partial_rows),
                               args.num_bins, bins, stream, hot_report.min_count,
                               hot_report.word, hot_report.seq_word, hot_report.seq);
  const cudaError_t ef = cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return fail_cuda(e, "cluster histogram launch");
  if (ef != cudaSuccess) return fail_cuda(ef, "cudaFreeAsync");
  return DSMEM_HIST_OK;
}

// Consistency of a caller-supplied plan with num_bins and the device.
int check_plan(const DeviceState* st, const dsmem_hist_plan_t* p, int32_t num_bins) {
  if (!p) return fail(DSMEM_HIST_EINVAL, "plan is NULL");
  const int64_t P = p->cluster_size, S = p->bins_per_cta;
  if (P < 1 || P > 16 || P > st->dev.max_cluster_size)
    return fail(DSMEM_HIST_EINVAL, "plan: cluster_size %lld out of range", static_cast<long long>(P));
  if (p->kernel == DSMEM_HIST_KERNEL_SHIP) {
    const int nq = p->sub_vectors;
    if (P < 2 || p->block_threads != kShipThreads || (p->keys_per_thread != 4 && p->keys_per_thread != 8) ||
        nq < 1 || nq > 4096 || S + 32 >= 0xFFFF ||
        p->smem_bytes != 4 * S + static_cast<int64_t>(ship_staging_bytes(static_cast<int>(P), nq)))
      return fail(DSMEM_HIST_EINVAL, "plan: ship kernel fields inconsistent");
  } else if (p->kernel != DSMEM_HIST_KERNEL_DIRECT || p->smem_bytes != 4 * S) {
    return fail(DSMEM_HIST_EINVAL, "plan: kernel / smem_bytes inconsistent");
  }
  if (S < 4 || (S & 3) || S >= (int64_t{1} << 18) ||
      p->smem_bytes > st->dev.max_smem_per_block_optin)
    return fail(DSMEM_HIST_EINVAL, "plan: bins_per_cta / smem_bytes inconsistent");
  if (p->passes < 1 || static_cast<int64_t>(p->passes) * P * S < num_bins ||
      static_cast<int64_t>(p->passes - 1) * P * S >= num_bins)
    return fail(DSMEM_HIST_EINVAL, "plan: passes do not cover num_bins exactly");
  if (p->block_threads < 64 || p->block_threads > 1024 || (p->block_threads & 31))
    return fail(DSMEM_HIST_EINVAL, "plan: block_threads invalid");
  if (p->num_clusters < 1 || p->aggregate < 0 || p->aggregate > 1)
    return fail(DSMEM_HIST_EINVAL, "plan: num_clusters / aggregate invalid");
  if (p->partial_stride < num_bins || (p->partial_stride & 3))
    return fail(DSMEM_HIST_EINVAL, "plan: partial_stride must be >= num_bins and a multiple of 4");
  if (p->hot_bin < -1 || p->hot_bin >= num_bins ||
      (p->hot_bin >= 0 && p->kernel != DSMEM_HIST_KERNEL_SHIP))
    return fail(DSMEM_HIST_EINVAL, "plan: hot_bin must be -1 or a bin of a ship-kernel plan");
  if (p->partial_rows != p->num_clusters &&
      !(p->partial_rows == p->num_clusters + 1 && p->kernel == DSMEM_HIST_KERNEL_SHIP && p->passes == 1))
    return fail(DSMEM_HIST_EINVAL, "plan: partial_rows must be num_clusters, or num_clusters + 1 "
                "(the helper's row) for a single-pass ship plan");
  return DSMEM_HIST_OK;
}

int run_partials(const int32_t* keys, int64_t n, int32_t num_bins, const dsmem_hist_plan_t* plan,
                 uint32_t* partials, int32_t accumulate, cudaStream_t stream) {
  int rc = check_args(keys, n, num_bins, partials);
  if (rc) return rc;
  if (reinterpret_cast<uintptr_t>(partials) & 15u)
    return fail(DSMEM_HIST_EINVAL, "partials must be 16-byte aligned");
  if (accumulate != 0 && accumulate != 1) return fail(DSMEM_HIST_EINVAL, "accumulate must be 0 or 1");
  SlotRef sr;
  DeviceState* st = nullptr;
  {
    std::lock_guard<std::mutex> g(g_mutex);
    if ((rc = device_state(&st))) return rc;
    if ((rc = check_plan(st, plan, num_bins))) return rc;
    if (plan->kernel == DSMEM_HIST_KERNEL_SHIP && n >= kShipMaxKeys)
      return fail(DSMEM_HIST_EINVAL, "the ship kernel takes fewer than 2^38 keys per call");
    if ((rc = stream_slot(st, stream, true, &sr))) return rc;
    if ((rc = take_pending_timeout(sr.h_status))) return rc;
    if ((rc = prepare_locked(st, *plan))) return rc;
  }
  // The caller's plan decides the kernel (its hot_bin included): no automatic choice.
  ClusterHistArgs args = make_args(*plan, keys, n, num_bins, partials, accumulate);
  args.status = sr.d_status;
  const cudaError_t e = launch_plan(*plan, args, stream, st, &sr);
  return e == cudaSuccess ? DSMEM_HIST_OK : fail_cuda(e, "cluster histogram launch");
}

int run_reduce(const uint32_t* partials, int32_t num_rows, int64_t stride, int32_t num_bins,
               uint32_t* bins, cudaStream_t stream) {
  if (num_bins < 1) return fail(DSMEM_HIST_EINVAL, "num_bins must be >= 1");
  if (!partials || !bins) return fail(DSMEM_HIST_EINVAL, "partials and bins must not be NULL");
  if (num_rows < 1) return fail(DSMEM_HIST_EINVAL, "num_rows must be >= 1");
  if (stride < num_bins || (stride & 3))
    return fail(DSMEM_HIST_EINVAL, "partial_stride must be >= num_bins and a multiple of 4");
  if ((reinterpret_cast<uintptr_t>(partials) & 15u) || (reinterpret_cast<uintptr_t>(bins) & 3u))
    return fail(DSMEM_HIST_EINVAL, "partials must be 16-byte and bins 4-byte aligned");
  const cudaError_t e = launch_reduce_partials(partials, static_cast<uint64_t>(stride),
                                               static_cast<uint32_t>(num_rows),
                                               static_cast<uint32_t>(num_bins), bins, stream);
  return e == cudaSuccess ? DSMEM_HIST_OK : fail_cuda(e, "reduce launch");
}

constexpr int64_t kHostChunkKeys = int64_t{1} << 24;  // 64 MiB of keys per staged chunk

int run_host(const int32_t* h_keys, int64_t n, int32_t num_bins, uint32_t* h_bins,
             cudaStream_t stream) {
  int rc = check_args(h_keys, n, num_bins, h_bins);
  if (rc) return rc;
  DeviceState* st = nullptr;
  dsmem_hist_plan_t plan;
  const int64_t chunk = n < kHostChunkKeys ? n : kHostChunkKeys;
  SlotRef sr;
  HotReport hot_report;
  {
    std::lock_guard<std::mutex> g(g_mutex);
    if ((rc = device_state(&st))) return rc;
    if ((rc = stream_slot(st, stream, true, &sr))) return rc;
    if ((rc = take_pending_timeout(sr.h_status))) return rc;
    if ((rc = plan_locked(st, num_bins, chunk, nullptr, &plan))) return rc;
    if ((rc = ensure_pool(st))) return rc;
    const int32_t chosen = choose_hot_bin(st, sr, n, num_bins, &hot_report);
    use_hot_bin(&plan, chosen, sr);
    cudaError_t e;
    if (!st->copy_stream) {
      if ((e = cudaStreamCreateWithFlags(&st->copy_stream, cudaStreamNonBlocking)) != cudaSuccess)
        return fail_cuda(e, "cudaStreamCreateWithFlags");
      for (int i = 0; i < 2; ++i) {
        if ((e = cudaEventCreateWithFlags(&st->ev_copied[i], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&st->ev_consumed[i], cudaEventDisableTiming)) != cudaSuccess)
          return fail_cuda(e, "cudaEventCreateWithFlags");
      }
    }
  }
  std::lock_guard<std::mutex> serial(st->host_call);
  cudaError_t e;
  const size_t bins_bytes = sizeof(uint32_t) * static_cast<size_t>(num_bins);
  const size_t bins_alloc = (bins_bytes + 255) & ~size_t{255};
  const size_t chunk_bytes = ((sizeof(int32_t) * static_cast<size_t>(chunk)) + 255) & ~size_t{255};
  const size_t total = bins_alloc + static_cast<size_t>(plan.workspace_bytes) + 2 * chunk_bytes;
  void* scratch = nullptr;
  if (injected_alloc_failure())
    return fail(DSMEM_HIST_ENOMEM, "scratch pool: %zu bytes: allocation failure injected by "
                "DSMEM_HIST_TEST_FAIL_ALLOC", total);
  if ((e = cudaMallocFromPoolAsync(&scratch, total, st->pool, stream)) != cudaSuccess) {
    cudaGetLastError();
    return fail(DSMEM_HIST_ENOMEM, "scratch pool: %zu bytes: %s", total, cudaGetErrorString(e));
  }
  char* base = static_cast<char*>(scratch);
  uint32_t* d_bins = reinterpret_cast<uint32_t*>(base);
  uint32_t* partials = reinterpret_cast<uint32_t*>(base + bins_alloc);
  int32_t* stage[2] = {
      reinterpret_cast<int32_t*>(base + bins_alloc + plan.workspace_bytes),
      reinterpret_cast<int32_t*>(base + bins_alloc + plan.workspace_bytes + chunk_bytes)};

  // Order the copy stream after the allocation made on `stream`.
  rc = DSMEM_HIST_OK;
  if ((e = cudaEventRecord(st->ev_consumed[0], stream)) != cudaSuccess ||
      (e = cudaEventRecord(st->ev_consumed[1], stream)) != cudaSuccess)
    rc = fail_cuda(e, "cudaEventRecord");
  if (n == 0 && rc == DSMEM_HIST_OK) {
    if ((e = cudaMemsetAsync(d_bins, 0, bins_bytes, stream)) != cudaSuccess)
      rc = fail_cuda(e, "cudaMemsetAsync");
  }
  for (int64_t off = 0, j = 0; rc == DSMEM_HIST_OK && off < n; off += chunk, ++j) {
    const int b = static_cast<int>(j & 1);
    const int64_t cnt = (n - off) < chunk ? (n - off) : chunk;
    if ((e = cudaStreamWaitEvent(st->copy_stream, st->ev_consumed[b], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(stage[b], h_keys + off, sizeof(int32_t) * cnt,
                             cudaMemcpyHostToDevice, st->copy_stream)) != cudaSuccess ||
        (e = cudaEventRecord(st->ev_copied[b], st->copy_stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, st->ev_copied[b], 0)) != cudaSuccess) {
      rc = fail_cuda(e, "staging copy");
      break;
    }
    ClusterHistArgs args = make_args(plan, stage[b], cnt, num_bins, partials, j > 0);
    args.status = sr.d_status;
    if ((e = launch_plan(plan, args, stream, st, &sr)) != cudaSuccess ||
        (e = cudaEventRecord(st->ev_consumed[b], stream)) != cudaSuccess) {
      rc = fail_cuda(e, "cluster histogram launch");
      break;
    }
  }
  if (rc == DSMEM_HIST_OK && n > 0) {
    if ((e = launch_reduce_partials(partials, static_cast<uint64_t>(plan.partial_stride),
                                    static_cast<uint32_t>(plan.partial_rows),
                                    static_cast<uint32_t>(num_bins), d_bins, stream,
                                    hot_report.min_count, hot_report.word,
                                    hot_report.seq_word, hot_report.seq)) != cudaSuccess)
      rc = fail_cuda(e, "reduce launch");
  }
  if (rc == DSMEM_HIST_OK) {
    if ((e = cudaMemcpyAsync(h_bins, d_bins, bins_bytes, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
      rc = fail_cuda(e, "result copy");
  }
  // The copy stream's last use of the staging buffers is ordered before the
  // kernels on `stream`, so freeing on `stream` is safe.
  cudaFreeAsync(scratch, stream);
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess && rc == DSMEM_HIST_OK)
    rc = fail_cuda(e, "cudaStreamSynchronize");
  return rc;
}

}  // namespace

// For the entry point with caller-free scratch (static_scratch.cu): the same
// argument checks, plan and launches as dsmem_hist, with the partial rows in
// memory the caller of this function supplies, at most `max_rows_bytes`.
int run_with_fixed_scratch(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
                           uint32_t* scratch, int64_t max_rows_bytes, cudaStream_t stream) {
  int rc = check_args(keys, n, num_bins, bins);
  if (rc) return rc;
  const int64_t row_bytes = 4 * ((static_cast<int64_t>(num_bins) + 3) & ~int64_t{3});
  if (row_bytes > max_rows_bytes)
    return fail(DSMEM_HIST_EINVAL,
                "num_bins %d needs %lld bytes of static scratch per cluster; the static scratch "
                "holds %lld bytes (at most %lld bins)",
                num_bins, static_cast<long long>(row_bytes), static_cast<long long>(max_rows_bytes),
                static_cast<long long>(max_rows_bytes / 4));
  dsmem_hist_plan_t plan;
  SlotRef sr;
  HotReport hot_report;
  {
    std::lock_guard<std::mutex> g(g_mutex);
    DeviceState* st = nullptr;
    if ((rc = device_state(&st))) return rc;
    // Stream words only if an earlier call already allocated them: this path
    // allocates nothing.
    if ((rc = stream_slot(st, stream, false, &sr))) return rc;
    if ((rc = take_pending_timeout(sr.h_status))) return rc;
    if ((rc = plan_locked(st, num_bins, n, nullptr, &plan))) return rc;
    // No helper kernel here: it would need a stream of its own.
    set_partial_rows(&plan, false);
    if (plan.workspace_bytes > max_rows_bytes) {
      // Fewer clusters, so their partial rows fit the static scratch.  The
      // forced count is below the automatic one (whose rows did not fit), so
      // it never exceeds the clusters that can be resident or the rows the
      // scratch holds.
      const int32_t auto_clusters = plan.num_clusters;
      dsmem_hist_request_t req = {0, 0, static_cast<int32_t>(max_rows_bytes / row_bytes), -1, 0, -1, 0, 0};
      if (req.num_clusters >= auto_clusters || req.num_clusters < 1)
        return fail(DSMEM_HIST_EINVAL, "static scratch: %d rows of %lld bytes do not fit below the "
                    "automatic %d clusters", req.num_clusters, static_cast<long long>(row_bytes),
                    auto_clusters);
      if ((rc = plan_locked(st, num_bins, n, &req, &plan))) return rc;
      set_partial_rows(&plan, false);
      if (plan.num_clusters > req.num_clusters || plan.workspace_bytes > max_rows_bytes)
        return fail(DSMEM_HIST_EINVAL, "static scratch: forced plan exceeds the scratch");
    }
    const int32_t chosen = choose_hot_bin(st, sr, n, num_bins, &hot_report);
    use_hot_bin(&plan, chosen, sr);
  }
  cudaError_t e;
  if (n == 0) {
    e = cudaMemsetAsync(bins, 0, sizeof(uint32_t) * static_cast<size_t>(num_bins), stream);
    return e == cudaSuccess ? DSMEM_HIST_OK : fail_cuda(e, "cudaMemsetAsync");
  }
  ClusterHistArgs args = make_args(plan, keys, n, num_bins, scratch, 0);
  args.status = sr.d_status;
  e = launch_plan(plan, args, stream);
  if (e == cudaSuccess)
    e = launch_reduce_partials(scratch, args.stride, static_cast<uint32_t>(plan.num_clusters),
                               args.num_bins, bins, stream, hot_report.min_count,
                               hot_report.word, hot_report.seq_word, hot_report.seq);
  return e == cudaSuccess ? DSMEM_HIST_OK : fail_cuda(e, "cluster histogram launch");
}

int record_error(int code, const char* what) { return fail(code, "%s", what); }

namespace {

// Median of the elapsed times of `reps` launches of `fn`, each bracketed by
// its own pair of events on `stream`.
template <class Fn>
int time_median(Fn fn, cudaStream_t stream, int reps, float* out) {
  cudaEvent_t a = nullptr, b = nullptr;
  cudaError_t e;
  if ((e = cudaEventCreate(&a)) != cudaSuccess || (e = cudaEventCreate(&b)) != cudaSuccess) {
    if (a) cudaEventDestroy(a);
    return fail_cuda(e, "cudaEventCreate");
  }
  float t[16];
  int rc = DSMEM_HIST_OK;
  if ((rc = fn()) != DSMEM_HIST_OK) goto done;  // warm-up
  for (int i = 0; i < reps && i < 16; ++i) {
    cudaEventRecord(a, stream);
    if ((rc = fn()) != DSMEM_HIST_OK) goto done;
    cudaEventRecord(b, stream);
    if ((e = cudaEventSynchronize(b)) != cudaSuccess) {
      rc = fail_cuda(e, "cudaEventSynchronize");
      goto done;
    }
    cudaEventElapsedTime(&t[i], a, b);
  }
  for (int i = 1; i < reps; ++i)
    for (int j = i; j > 0 && t[j] < t[j - 1]; --j) std::swap(t[j], t[j - 1]);
  *out = t[reps / 2];
done:
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  return rc;
}

}  // namespace

int run_tune(const int32_t* keys, int64_t n, int32_t num_bins, int64_t sample_keys,
             int32_t max_results, dsmem_hist_tune_result_t* results, int32_t* num_results,
             cudaStream_t stream) {
  int rc = check_args(keys, n, num_bins, keys);
  if (rc) return rc;
  if (!results || !num_results || max_results < 1)
    return fail(DSMEM_HIST_EINVAL, "results, num_results and max_results >= 1 are required");
  const int64_t m = std::min<int64_t>(n, sample_keys > 0 ? sample_keys : (int64_t{1} << 24));
  DeviceState* st = nullptr;
  {
    std::lock_guard<std::mutex> g(g_mutex);
    if ((rc = device_state(&st))) return rc;
    if ((rc = ensure_pool(st))) return rc;
  }
  // Candidates: every cluster size with each kernel, duplicates of one shape
  // removed, then the global-atomics kernel.
  std::vector<dsmem_hist_tune_result_t> cand;
  const int sizes[] = {1, 2, 4, 8, 16};
  for (int P : sizes) {
    for (int k = DSMEM_HIST_KERNEL_DIRECT; k <= DSMEM_HIST_KERNEL_SHIP; ++k) {
      dsmem_hist_request_t req = {P, 0, 0, 0, 0, k, 0, 0};
      dsmem_hist_plan_t plan;
      {
        std::lock_guard<std::mutex> g(g_mutex);
        if (plan_locked(st, num_bins, m, &req, &plan) != DSMEM_HIST_OK) continue;
      }
      bool dup = false;
      for (const auto& c : cand)
        dup |= c.plan.cluster_size == plan.cluster_size && c.plan.kernel == plan.kernel;
      if (dup) continue;
      dsmem_hist_tune_result_t r = {};
      r.plan = plan;
      cand.push_back(r);
    }
  }
  dsmem_hist_tune_result_t ga = {};
  ga.global_atomic = 1;
  cand.push_back(ga);
  g_last_error.clear();

  int64_t ws = 0;
  for (const auto& c : cand) ws = std::max(ws, c.plan.workspace_bytes);
  const size_t bins_bytes = (4 * static_cast<size_t>(num_bins) + 255) & ~size_t{255};
  void* scratch = nullptr;
  if (injected_alloc_failure())
    return fail(DSMEM_HIST_ENOMEM, "tune scratch: allocation failure injected by "
                "DSMEM_HIST_TEST_FAIL_ALLOC");
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, bins_bytes + static_cast<size_t>(ws) + 256,
                                          st->pool, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DSMEM_HIST_ENOMEM, "tune scratch: %s", cudaGetErrorString(e));
  }
  uint32_t* d_bins = static_cast<uint32_t*>(scratch);
  uint32_t* partials = reinterpret_cast<uint32_t*>(static_cast<char*>(scratch) + bins_bytes);
  uint32_t* sink = reinterpret_cast<uint32_t*>(static_cast<char*>(scratch) + bins_bytes + ws);
  for (auto& c : cand) {
    if (c.global_atomic) {
      rc = time_median([&] {
        const cudaError_t le = launch_global_atomic(keys, m, static_cast<uint32_t>(num_bins), d_bins, stream);
        return le == cudaSuccess ? DSMEM_HIST_OK : fail_cuda(le, "global-atomic launch");
      }, stream, 5, &c.ms);
      if (rc) break;
      continue;
    }
    const dsmem_hist_plan_t plan = c.plan;
    rc = time_median([&] {
      const ClusterHistArgs args = make_args(plan, keys, m, num_bins, partials, 0);
      cudaError_t le = launch_plan(plan, args, stream);
      if (le == cudaSuccess)
        le = launch_reduce_partials(partials, args.stride, static_cast<uint32_t>(plan.num_clusters),
                                    args.num_bins, d_bins, stream);
      return le == cudaSuccess ? DSMEM_HIST_OK : fail_cuda(le, "tune launch");
    }, stream, 5, &c.ms);
    if (rc) break;
    rc = time_median([&] {
      const cudaError_t le = launch_cluster_control(plan, sink, stream);
      return le == cudaSuccess ? DSMEM_HIST_OK : fail_cuda(le, "control launch");
    }, stream, 5, &c.control_ms);
    if (rc) break;
  }
  cudaFreeAsync(scratch, stream);
  cudaStreamSynchronize(stream);
  if (rc) return rc;
  std::sort(cand.begin(), cand.end(),
            [](const dsmem_hist_tune_result_t& x, const dsmem_hist_tune_result_t& y) { return x.ms < y.ms; });
  const int32_t k = std::min<int32_t>(max_results, static_cast<int32_t>(cand.size()));
  for (int32_t i = 0; i < k; ++i) results[i] = cand[i];
  *num_results = k;
  return DSMEM_HIST_OK;
}

}  // namespace dsmh

using namespace dsmh;

extern "C" {

int dsmem_hist(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
               cudaStream_t stream) {
  return run_device(keys, n, num_bins, bins, nullptr, stream);
}

int dsmem_hist_ex(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
                  const dsmem_hist_request_t* request, cudaStream_t stream) {
  return run_device(keys, n, num_bins, bins, request, stream);
}

int dsmem_hist_global_atomic(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
                             cudaStream_t stream) {
  int rc = check_args(keys, n, num_bins, bins);
  if (rc) return rc;
  const cudaError_t e = launch_global_atomic(keys, n, static_cast<uint32_t>(num_bins), bins, stream);
  return e == cudaSuccess ? DSMEM_HIST_OK : fail_cuda(e, "global-atomic histogram launch");
}

int dsmem_hist_host(const int32_t* h_keys, int64_t n, int32_t num_bins, uint32_t* h_bins,
                    cudaStream_t stream) {
  return run_host(h_keys, n, num_bins, h_bins, stream);
}

int dsmem_hist_tune(const int32_t* keys, int64_t n, int32_t num_bins, int64_t sample_keys,
                    int32_t max_results, dsmem_hist_tune_result_t* results, int32_t* num_results,
                    cudaStream_t stream) {
  return run_tune(keys, n, num_bins, sample_keys, max_results, results, num_results, stream);
}

int dsmem_hist_partials(const int32_t* keys, int64_t n, int32_t num_bins,
                        const dsmem_hist_plan_t* plan, uint32_t* partials, int32_t accumulate,
                        cudaStream_t stream) {
  return run_partials(keys, n, num_bins, plan, partials, accumulate, stream);
}

int dsmem_hist_reduce(const uint32_t* partials, int32_t num_rows, int64_t partial_stride,
                      int32_t num_bins, uint32_t* bins, cudaStream_t stream) {
  return run_reduce(partials, num_rows, partial_stride, num_bins, bins, stream);
}

int dsmem_hist_plan_ex(int32_t num_bins, int64_t n, const dsmem_hist_request_t* request,
                       dsmem_hist_plan_t* out) {
  if (!out) return fail(DSMEM_HIST_EINVAL, "out is NULL");
  if (n < 0) return fail(DSMEM_HIST_EINVAL, "n must be >= 0 (got %lld)", static_cast<long long>(n));
  std::lock_guard<std::mutex> g(g_mutex);
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  return plan_locked(st, num_bins, n, request, out);
}

int dsmem_hist_plan(int32_t num_bins, int64_t n, dsmem_hist_plan_t* out) {
  return dsmem_hist_plan_ex(num_bins, n, nullptr, out);
}

int dsmem_hist_plan_for_device(const dsmem_hist_device_t* device, int32_t num_bins, int64_t n,
                               const dsmem_hist_request_t* request, int32_t max_active_clusters,
                               dsmem_hist_plan_t* out) {
  const char* why = "";
  const int rc = plan_shape(device, num_bins, n, request, max_active_clusters, out, &why);
  return rc == DSMEM_HIST_OK ? rc : fail(rc, "plan: %s", why);
}

const char* dsmem_hist_strerror(int code) {
  switch (code) {
    case DSMEM_HIST_OK: return "DSMEM_HIST_OK";
    case DSMEM_HIST_EINVAL: return "DSMEM_HIST_EINVAL: invalid argument";
    case DSMEM_HIST_EUNSUPPORTED: return "DSMEM_HIST_EUNSUPPORTED: unsupported device or shape";
    case DSMEM_HIST_ECUDA: return "DSMEM_HIST_ECUDA: CUDA runtime error";
    case DSMEM_HIST_ETIMEOUT: return "DSMEM_HIST_ETIMEOUT: device-side wait timed out";
    case DSMEM_HIST_ENOMEM: return "DSMEM_HIST_ENOMEM: scratch allocation failed";
    default: return "DSMEM_HIST: unknown error code";
  }
}

const char* dsmem_hist_last_error(void) { return g_last_error.c_str(); }

void dsmem_hist_release(void) {
  std::lock_guard<std::mutex> g(g_mutex);
  int cur = 0;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (auto& kv : g_devices) {
    DeviceState* st = kv.second;
    if (!st) continue;
    if (cudaSetDevice(kv.first) != cudaSuccess) continue;
    if (st->pool) {
      cudaDeviceSynchronize();
      cudaMemPoolDestroy(st->pool);
      st->pool = nullptr;
    }
    if (st->h_status) {
      cudaDeviceSynchronize();
      cudaFreeHost(st->h_status);
      st->h_status = st->d_status = nullptr;
      st->status_slot.clear();
      for (int i = 0; i < kStatusSlots; ++i)
        st->slot_seq[i] = st->slot_bins_since[i] = 0, st->slot_bins[i] = 0;
    }
    for (auto& hs : st->helper_streams) {
      if (!hs.stream) continue;
      cudaStreamSynchronize(hs.stream);
      cudaStreamSynchronize(hs.cluster_stream);
      cudaStreamDestroy(hs.stream);
      cudaStreamDestroy(hs.cluster_stream);
      cudaEventDestroy(hs.fork);
      cudaEventDestroy(hs.clusters_done);
      cudaEventDestroy(hs.join);
      hs = DeviceState::HelperStream{};
    }
    if (st->copy_stream) {
      cudaStreamDestroy(st->copy_stream);
      st->copy_stream = nullptr;
      for (int i = 0; i < 2; ++i) {
        cudaEventDestroy(st->ev_copied[i]);
        cudaEventDestroy(st->ev_consumed[i]);
        st->ev_copied[i] = st->ev_consumed[i] = nullptr;
      }
    }
  }
  if (have_cur) cudaSetDevice(cur);
}

int dsmem_hist_device_status(uint32_t* status) {
  uint32_t word = 0;
  const cudaError_t e = read_and_clear_ship_status(&word);
  if (status) *status = word;
  if (e != cudaSuccess) return fail(DSMEM_HIST_ECUDA, "device_status: %s", cudaGetErrorString(e));
  if (word) return fail(DSMEM_HIST_ETIMEOUT, "device_status: a bounded inbox wait gave up (word 0x%x)", word);
  return DSMEM_HIST_OK;
}

int dsmem_hist_version(void) { return 100; }

}  // extern "C"
