/*
 * dsmem_hist -- thread-block-cluster histogram for NVIDIA GB300 (sm_103a).
 *
 * The operation ("Distributed Shared Memory", section "The cluster
 * histogram"): a bin array too large for one CTA's shared memory is split
 * into equal slices of S counters, one slice in the shared memory of each of
 * the P CTAs of a thread-block cluster (owner = bin / S).  Every thread
 * increments the owning CTA's counter through distributed shared memory,
 * cluster barriers bracket that phase, and the per-cluster slices are then
 * reduced into global memory.  The result is the plain histogram:
 *
 *     bins[b] = #{ i in [0, n) : keys[i] == b }  (mod 2^32),  0 <= b < num_bins
 *
 * Conventions for every entry point:
 *   - Return value: 0 (DSMEM_HIST_OK) or one of the negative codes below;
 *     dsmem_hist_strerror() names a code and dsmem_hist_last_error() gives
 *     the calling thread's most recent detailed message (CUDA error text
 *     included).
 *   - Keys are int32; keys outside [0, num_bins) -- negatives included --
 *     are not counted.  `bins` is OVERWRITTEN (not accumulated into).
 *   - Counters are uint32 and wrap modulo 2^32.
 *   - Device pointers belong to the caller and must be valid on the current
 *     CUDA device; `keys` must be 4-byte aligned (any 16-byte misalignment is
 *     handled), `bins` 4-byte aligned.
 *   - Device entry points are asynchronous on `stream` (0 = legacy default
 *     stream): they return after enqueueing, results are valid once the
 *     stream has reached that point.  Scratch memory (per-cluster partial
 *     histograms) comes from a library-owned, stream-ordered CUDA memory pool
 *     and is returned to the pool on the same stream, so calls on different
 *     streams never share scratch.
 *   - Thread-safe: the per-device state is guarded by a mutex.
 *   - Device-side failures (no counterpart in the pages' design, which waits
 *     only on cluster barriers): the key-shipping kernel waits for its peers'
 *     inbox bytes with bounded waits (about 50 ms each).  A wait that gives
 *     up skips that inbox (the launch's histogram is then wrong) and records
 *     the failure in two places: a word for the call's stream in pinned,
 *     host-mapped memory, and the device-wide status word.  The first
 *     histogram call on the same stream that starts after the failing launch
 *     has finished returns DSMEM_HIST_ETIMEOUT and enqueues nothing (call it
 *     again); dsmem_hist_device_status() reads and clears the device-wide
 *     word.  The host-mapped words (64 streams per device; later streams
 *     share the last word) are allocated by the first dsmem_hist,
 *     dsmem_hist_ex, dsmem_hist_host or dsmem_hist_partials call on a device;
 *     dsmem_hist_static, which allocates nothing, uses them only if they
 *     exist already and otherwise reports through the device-wide word alone.
 *   - Test hooks, read from the environment at every call (for tests of the
 *     failure paths above; leave them unset otherwise):
 *       DSMEM_HIST_TEST_WAIT_CYCLES=c           bound one inbox wait to c clock
 *                                               cycles (1000 .. 1e8)
 *       DSMEM_HIST_TEST_WITHHOLD_LAST_ROUND=1   the key-shipping kernel's senders
 *                                               skip their last round's arrival
 *                                               and stores, so owners' last waits
 *                                               run out with nothing in flight
 *       DSMEM_HIST_TEST_FAIL_ALLOC=1            scratch allocations of dsmem_hist,
 *                                               dsmem_hist_ex, dsmem_hist_host and
 *                                               dsmem_hist_tune fail with
 *                                               DSMEM_HIST_ENOMEM
 */
#ifndef DSMEM_HIST_H
#define DSMEM_HIST_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define DSMEM_HIST_API __attribute__((visibility("default")))
#else
#define DSMEM_HIST_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum {
  DSMEM_HIST_OK = 0,
  DSMEM_HIST_EINVAL = -1,       /* bad argument (null pointer with n > 0, n < 0, num_bins < 1, misaligned) */
  DSMEM_HIST_EUNSUPPORTED = -2, /* device below compute capability 9.0, or no legal cluster shape */
  DSMEM_HIST_ECUDA = -3,        /* a CUDA runtime call or kernel launch failed */
  DSMEM_HIST_ETIMEOUT = -4,     /* a bounded device-side wait of an earlier launch gave up (see below) */
  DSMEM_HIST_ENOMEM = -5        /* the scratch pool could not supply the partial histograms */
};

/* How increments reach a remote owner's slice.
 *   DIRECT: one `red.shared::cluster` per key (the page's kernel, optionally
 *           with __match_any_sync warp aggregation).
 *   SHIP:   keys travel to their owner as 16-bit local indices in coalesced
 *           16-byte DSMEM stores and the owner applies local shared-memory
 *           atomics (DSMEM_HIST_SHIP_THREADS threads per CTA; P >= 2). */
enum { DSMEM_HIST_KERNEL_DIRECT = 0, DSMEM_HIST_KERNEL_SHIP = 1 };

/* Threads per CTA of the ship kernel (fixed at build time). */
#define DSMEM_HIST_SHIP_THREADS 896

/* Launch shape chosen by the planner (all fields filled by dsmem_hist_plan*). */
typedef struct dsmem_hist_plan {
  int32_t cluster_size;        /* P: CTAs per cluster, 1..16 (16 is non-portable) */
  int32_t bins_per_cta;        /* S: counters in each CTA's shared-memory slice (multiple of 4) */
  int32_t passes;              /* bin ranges of P*S bins streamed one after the other (1 unless
                                  num_bins exceeds what one cluster holds) */
  int32_t block_threads;       /* threads per CTA */
  int32_t num_clusters;        /* C: clusters launched (persistent grid of C*P CTAs) */
  int32_t smem_bytes;          /* dynamic shared memory per CTA: 4*S (+ staging for SHIP) */
  int32_t aggregate;           /* 1: warp pre-aggregation of equal keys (__match_any_sync + popc) */
  int32_t ctas_per_sm;         /* resident CTAs per SM the shape allows */
  int32_t max_active_clusters; /* occupancy answer for this shape (0 when not queried) */
  int32_t kernel;              /* DSMEM_HIST_KERNEL_DIRECT or DSMEM_HIST_KERNEL_SHIP */
  int32_t keys_per_thread;     /* ship kernel: keys each thread partitions per round (4 or 8) */
  int32_t sub_vectors;         /* ship kernel: rows of each owner's staging block (each row:
                                  32 columns of 16-bit entries) */
  int32_t hot_bin;             /* ship kernel: a bin expected to hold a large share of the keys;
                                  its keys are counted in registers instead of staged (see
                                  dsmem_hist_request_t.hot_bin).  -1: none.  The planner sets it
                                  only on request; dsmem_hist_partials uses it as given */
  int32_t partial_rows;        /* partial rows the reduction sums: num_clusters, plus one when a
                                  helper kernel runs beside a single-pass ship launch of at least
                                  2^24 keys, on the SMs its clusters leave idle (see
                                  dsmem_hist_partials) */
  int64_t partial_stride;      /* u32 elements between two partial rows (num_bins rounded up to 4) */
  int64_t workspace_bytes;     /* scratch: partial_rows * partial_stride * 4, plus 32 bytes of
                                  tile counter and timing with the helper */
} dsmem_hist_plan_t;

/* Planner overrides; a zero field (or -1 for `aggregate` and `kernel`) means "choose". */
typedef struct dsmem_hist_request {
  int32_t cluster_size;    /* force P (1..16) */
  int32_t block_threads;   /* force threads per CTA (multiple of 32, 64..1024) */
  int32_t num_clusters;    /* force C */
  int32_t aggregate;       /* -1 choose, 0 off, 1 on */
  int32_t max_slice_bytes; /* cap on 4*S (default 128 KiB) */
  int32_t kernel;          /* -1 choose, else DSMEM_HIST_KERNEL_* */
  int32_t hot_bin_valid;   /* 0: automatic (see below); 1: hot_bin below is a hint; -1: never
                              use the hot-bin kernel */
  int32_t hot_bin;         /* with hot_bin_valid == 1: a bin in [0, num_bins) expected to take a
                              large share of the keys (a sixth or more).  The ship kernel then
                              counts that bin's keys in registers instead of staging them; one
                              bin with a quarter of the keys otherwise overflows its owner's
                              staging columns every round and sends each overflowing key as a
                              remote atomic.  The comparison costs about 9% more instructions on
                              keys without such a bin.  Exact either way; ignored by the direct
                              kernel.
                              Automatic: dsmem_hist, dsmem_hist_ex (hot_bin_valid == 0),
                              dsmem_hist_host and dsmem_hist_static use the hot-bin kernel when
                              the latest histogram on the same stream whose reduction has run
                              had the same num_bins and one bin holding a sixth or more of its
                              keys, as that reduction reported it through pinned, host-mapped
                              memory (no device synchronisation).  In a loop of calls that is a
                              histogram a few calls back; one without such a bin turns the
                              choice off again.  dsmem_hist_static takes part only on streams
                              whose words an allocating call has set up. */
} dsmem_hist_request_t;

/* The device facts the planner uses; filled from cudaGetDeviceProperties by
 * dsmem_hist_plan, or by hand to plan for a described device. */
typedef struct dsmem_hist_device {
  int32_t cc_major, cc_minor;
  int32_t sm_count;
  int32_t max_smem_per_block_optin; /* bytes a CTA may opt in to */
  int32_t max_smem_per_sm;          /* bytes per SM */
  int32_t max_threads_per_sm;
  int32_t max_cluster_size;         /* 8 portable, 16 where non-portable sizes are allowed */
} dsmem_hist_device_t;

/* Histogram of n int32 keys into num_bins uint32 counters on the GPU, through
 * the cluster/DSMEM path with the planner's shape ("Distributed Shared
 * Memory", section "The cluster histogram").
 *   keys     device, n int32 keys (read only)
 *   n        >= 0; n == 0 zeroes `bins`
 *   num_bins >= 1; more bins than one cluster holds are streamed in passes
 *   bins     device, num_bins uint32 (overwritten)
 *   stream   CUDA stream the work is enqueued on
 * Errors: EINVAL for bad arguments (nothing enqueued), EUNSUPPORTED, ECUDA,
 * ENOMEM (the scratch pool could not supply the partial rows; nothing
 * enqueued), ETIMEOUT (an earlier launch on this stream had a wait give up;
 * nothing enqueued). */
DSMEM_HIST_API int dsmem_hist(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
               cudaStream_t stream);

/* Same as dsmem_hist with planner overrides (NULL = none).  Used to force a
 * cluster size, block size, grid or aggregation mode; the forced shape must
 * be legal on the device or EUNSUPPORTED is returned. */
DSMEM_HIST_API int dsmem_hist_ex(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
                  const dsmem_hist_request_t* request, cudaStream_t stream);

/* Comparison point ("Distributed Shared Memory", section "When it beats global
 * atomics"): zero `bins`, then one global atomic add per in-range key,
 * contended grid-wide.  Same arguments, semantics and errors as dsmem_hist;
 * uses no scratch. */
DSMEM_HIST_API int dsmem_hist_global_atomic(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
                             cudaStream_t stream);

/* Histogram of HOST keys into HOST bins: the keys are copied to the device in
 * chunks on an internal copy stream, overlapped with the cluster kernel on
 * `stream`, and the bins copied back.  Pinned host memory gives full copy
 * speed; pageable memory works but copies slower.  SYNCHRONOUS: returns after
 * `h_bins` holds the result.  Device scratch (two chunk buffers, partial
 * histograms, the device bins) comes from the library's stream-ordered pool. */
DSMEM_HIST_API int dsmem_hist_host(const int32_t* h_keys, int64_t n, int32_t num_bins, uint32_t* h_bins,
                    cudaStream_t stream);

/* Stage 1 of dsmem_hist, with caller-owned scratch: the plan's kernels write
 * (accumulate == 0) or add into (accumulate == 1) the partial rows
 *     partials[r * plan->partial_stride + b],  r < plan->partial_rows,
 * which, summed over r, are the histogram of these keys ("Distributed Shared
 * Memory", section "The cluster histogram": zero, barrier, DSMEM increments,
 * barrier, flush).  Row c < num_clusters is cluster c's.  With a helper row
 * (partial_rows == num_clusters + 1: a single-pass ship plan of at least
 * 2^24 keys that leaves SMs idle) a global-atomic
 * helper kernel runs beside the clusters on the idle SMs, on a second
 * stream of the library forked from and joined back into `stream`: the
 * clusters' rounds take the first tiles of the keys, the helper the rest
 * ("When it beats global atomics": one global atomic per key, into the last
 * row), and a small mop-up kernel after the cluster kernel takes the
 * helper's tiles it has not claimed yet.  The helper's share of the tiles
 * starts from the idle SMs' expected pace and then follows what earlier
 * launches on the same stream report: the mop-up kernel's first CTA computes,
 * from the GPU's global timer, the share at which both sides would have
 * finished together.  DSMEM_HIST_HELPER=0 in the environment makes the planner leave
 * the helper out.
 *   plan      from dsmem_hist_plan for the same num_bins (checked for
 *             consistency; EINVAL otherwise)
 *   partials  device, 16-byte aligned, plan->workspace_bytes bytes: the
 *             partial rows, then (helper) a tile counter and timing words
 *             the call zeroes;
 *             with accumulate == 1 the rows must hold those of an earlier
 *             call with the same plan (used to fold key chunks into one
 *             histogram)
 * Asynchronous on `stream`. */
DSMEM_HIST_API int dsmem_hist_partials(const int32_t* keys, int64_t n, int32_t num_bins,
                                       const dsmem_hist_plan_t* plan, uint32_t* partials,
                                       int32_t accumulate, cudaStream_t stream);

/* Stage 2 of dsmem_hist: bins[b] = sum over r < num_rows of
 * partials[r * partial_stride + b] (mod 2^32), b < num_bins.
 *   partials  device, 16-byte aligned; partial_stride a multiple of 4 and
 *             >= num_bins
 *   num_rows  rows to sum: the plan's partial_rows after dsmem_hist_partials
 *   bins      device, num_bins uint32 (overwritten)
 * Asynchronous on `stream`. */
DSMEM_HIST_API int dsmem_hist_reduce(const uint32_t* partials, int32_t num_rows,
                                     int64_t partial_stride, int32_t num_bins, uint32_t* bins,
                                     cudaStream_t stream);

/* Same result as dsmem_hist, but the library allocates nothing.  The pages
 * have no counterpart: this is for callers that cannot let a library
 * allocate device memory -- code running while a stream is captured into a
 * CUDA graph, applications that own all device memory through their own
 * arena or budget, and latency-critical paths that must not enter the
 * allocator (which can synchronise or block).
 *   keys, n, bins, stream   as for dsmem_hist (device pointers, asynchronous)
 *   num_bins                1 .. 8,388,608; larger values return EINVAL
 * The per-cluster partial histograms live in a fixed 32 MiB
 * `static __device__` array inside the library, held by every GPU that loads
 * the library until the process exits; fewer clusters are launched when
 * their rows would not fit.  The first call on a device looks up that
 * array's device address and prepares the kernels and the plan cache; make
 * that first call before any stream capture.  The array is overwritten by
 * every call (nothing in it needs clearing), and all calls share it: calls
 * that may overlap on the GPU (different streams without ordering, or
 * different host threads) race on it and must be serialised by the caller. */
DSMEM_HIST_API int dsmem_hist_static(const int32_t* keys, int64_t n, int32_t num_bins,
                                     uint32_t* bins, cudaStream_t stream);

/* One candidate timed by dsmem_hist_tune. */
typedef struct dsmem_hist_tune_result {
  dsmem_hist_plan_t plan;  /* the shape (meaningless when global_atomic == 1) */
  int32_t global_atomic;   /* 1: the global-atomics kernel, no cluster */
  float ms;                /* median time of the whole histogram (cluster kernel + reduction) */
  float control_ms;        /* median time of the work-free control launch of this shape */
} dsmem_hist_tune_result_t;

/* Cluster-shape screen ("CREDIT", sections on the profitability model and
 * the matched control kernel): times every legal shape for this num_bins --
 * cluster sizes 1, 2, 4, 8, 16 with the direct and the ship kernel -- and
 * the global-atomics kernel on the first min(n, sample_keys) keys
 * (sample_keys <= 0: 16,777,216), each as the median of 5 timed runs after a
 * warm-up, together with a work-free control launch of the same grid,
 * cluster and shared memory.  Writes up to max_results results sorted by
 * `ms` (fastest first) and their count; the fastest plan can be passed back
 * through dsmem_hist_ex (cluster_size, block_threads, kernel, aggregate).
 * SYNCHRONOUS on `stream`; uses scratch from the library's pool and writes
 * nothing the caller owns. */
DSMEM_HIST_API int dsmem_hist_tune(const int32_t* keys, int64_t n, int32_t num_bins,
                                   int64_t sample_keys, int32_t max_results,
                                   dsmem_hist_tune_result_t* results, int32_t* num_results,
                                   cudaStream_t stream);

/* DSMEM primitive microbenchmarks (kinds for dsmem_hist_microbench). */
enum {
  DSMEM_HIST_MB_LOCAL_RED = 0,             /* red.shared.add.u32, random counter of own slice */
  DSMEM_HIST_MB_REMOTE_RED = 1,            /* red.shared::cluster.add.u32 into a peer's slice */
  DSMEM_HIST_MB_REMOTE_ST16_SCATTERED = 2, /* st.shared::cluster.v4, random peer and address */
  DSMEM_HIST_MB_REMOTE_ST16_COALESCED = 3, /* st.shared::cluster.v4, 512 contiguous bytes per warp */
  DSMEM_HIST_MB_CLUSTER_BARRIER = 4,       /* barrier.cluster arrive + wait */
  DSMEM_HIST_MB_DSMEM_PINGPONG = 5,        /* one-way latency of a flag in a peer CTA's shared memory */
  DSMEM_HIST_MB_GMEM_PINGPONG = 6,         /* one-way latency of a flag in global memory */
  DSMEM_HIST_MB_TILE_EXCHANGE_DSMEM = 7,   /* 16 KB tile pulled from the pair CTA's shared memory */
  DSMEM_HIST_MB_TILE_EXCHANGE_GMEM = 8     /* 16 KB tile exchanged through a global scratch + fence */
};

/* One microbenchmark's answer. */
typedef struct dsmem_hist_microbench_result {
  double value;          /* rate kinds (0..3): operations per clock per SM (bytes per clock
                            per SM for the two store kinds); barrier kind: clock cycles per
                            barrier; ping-pong kinds: clock cycles per one-way hop (half a
                            round trip); tile-exchange kinds: milliseconds for all iterations */
  double ms;             /* CUDA-event time of the timed launch */
  double bytes_per_s;    /* tile-exchange kinds: tile bytes landed per second, counted once
                            (every CTA receives one 16 KiB tile per iteration); 0 otherwise */
  uint64_t ops_expected; /* the work the probe issues by construction (see below) */
  uint64_t ops_counted;  /* the same work as counted on the device after the closing barrier */
  int32_t ctas;          /* CTAs launched (tile-exchange kinds; 0 otherwise) */
  int32_t reserved;      /* zero */
} dsmem_hist_microbench_result_t;

/* Measures one DSMEM primitive on the current GPU ("Hopper DSMEM vs HBM",
 * the ping-pong test and the 16 KB tile-exchange test; "CREDIT",
 * microbenchmark section).  One warm-up launch, then the timed launch.
 *   Rate kinds (0..4): 1024 threads per CTA, 128 KiB of shared memory per
 *     CTA, every resident cluster of `cluster_size` CTAs, `iters` operations
 *     per thread, timed with clock64 per CTA.  With cluster_size 1 the
 *     "remote" kinds address this CTA itself.
 *   Ping-pong kinds (5, 6): one cluster of `cluster_size` >= 2 CTAs; one
 *     thread of CTA 0 and one of CTA 1 pass a counter back and forth `iters`
 *     times through a flag in the receiver's shared memory (written with a
 *     release store to shared::cluster, read with acquire loads) or in global
 *     memory (release/acquire at GPU scope).  Every wait for the peer is
 *     bounded (2^20 polls); a wait that gives up ends the test with
 *     DSMEM_HIST_ETIMEOUT.
 *   Tile-exchange kinds (7, 8): every resident cluster of an even
 *     `cluster_size` (the page uses 2), 128 threads per CTA, one CTA per SM.
 *     CTAs 2j and 2j+1 of a cluster each own a 16 KiB tile of 4096 32-bit
 *     words in shared memory, and every iteration lands the other's tile in
 *     its own shared memory: kind 7 pulls it through the cluster address of
 *     the peer's tile and meets one cluster barrier; kind 8 writes its tile
 *     to a global scratch, fences, meets the barrier, reads the peer's slot
 *     from L2 and meets the barrier again.
 * Counted work (ops_expected against ops_counted, equal when the probe did
 * what it claims): the two reduction kinds count the increments that landed
 * in the slices; the store and barrier kinds the operations every thread
 * issued; the ping-pong kinds the completed round trips; the tile-exchange
 * kinds the sum of every word pulled from the peer over all iterations.
 * Synchronous; allocates and frees its own small device buffers. */
DSMEM_HIST_API int dsmem_hist_microbench(int32_t kind, int32_t cluster_size, int32_t iters,
                                         dsmem_hist_microbench_result_t* out);

/* The launch shape dsmem_hist would use on the current device for num_bins
 * bins and n keys: cluster size P, counters per CTA S, passes, threads per
 * CTA, clusters C, dynamic shared memory per CTA and the partial-row scratch.
 *
 * Where the rules come from:
 *   - "Distributed Shared Memory", section "The cluster histogram": the bins
 *     are split into P equal slices of S counters, one per CTA of a cluster,
 *     and the page's kernel needs P * S to cover every bin (a smaller total
 *     reaches past the cluster, a larger one drops bins).  Here S =
 *     ceil(num_bins / (P * passes)) rounded up to a multiple of 4, so no bin
 *     is dropped; the last CTA's few extra counters are never hit.
 *   - CUDA Handbook, chapter 7, "Thread Block Clusters and Distributed Shared
 *     Memory": up to 8 CTAs form a cluster portably and 16 as a non-portable
 *     opt-in; the largest usable size for a kernel is what
 *     cudaOccupancyMaxPotentialClusterSize reports; the shape is set at
 *     launch through cudaLaunchKernelEx with a
 *     cudaLaunchAttributeClusterDimension attribute.  The planner takes P
 *     from 2..16 (16 after setting the non-portable attribute) and confirms
 *     it, and the number of resident clusters, with
 *     cudaOccupancyMaxPotentialClusterSize and cudaOccupancyMaxActiveClusters.
 *   - "@dynshared", section "What it changes": static shared memory stops at
 *     48 KB per CTA, and more comes only as dynamic shared memory requested at
 *     launch.  A slice of 4*S bytes (128 KiB at the published shapes) is
 *     therefore dynamic shared memory, opted in with
 *     cudaFuncAttributeMaxDynamicSharedMemorySize up to the device's
 *     per-block limit.
 *   num_bins  >= 1
 *   n         >= 0 (sizes C: small inputs get fewer clusters)
 *   out       host pointer, filled on success
 * Errors: EINVAL (bad argument or NULL `out`), EUNSUPPORTED (no cluster shape
 * can be resident), ECUDA.  Enqueues nothing. */
DSMEM_HIST_API int dsmem_hist_plan(int32_t num_bins, int64_t n, dsmem_hist_plan_t* out);

/* dsmem_hist_plan with planner overrides (`request` may be NULL), as
 * dsmem_hist_ex takes them.  The pages have no counterpart: it exists so that
 * tests and the bench can ask for the exact shape they then force.
 *
 * Every entry point that plans on the current device (dsmem_hist,
 * dsmem_hist_ex, dsmem_hist_host, dsmem_hist_static, dsmem_hist_plan,
 * dsmem_hist_plan_ex) reads these environment variables for the request
 * fields the caller left to the planner: DSMEM_HIST_CLUSTER (cluster_size),
 * DSMEM_HIST_BLOCK (block_threads), DSMEM_HIST_GRID (num_clusters),
 * DSMEM_HIST_AGGREGATE (aggregate) and DSMEM_HIST_KERNEL (kernel).
 * DSMEM_HIST_TRACE=1 prints each plan to stderr.  A shape whose clusters
 * cannot be resident falls back from the ship kernel to the direct one, then
 * (unless the cluster size was forced) to smaller clusters. */
DSMEM_HIST_API int dsmem_hist_plan_ex(int32_t num_bins, int64_t n, const dsmem_hist_request_t* request,
                                      dsmem_hist_plan_t* out);

/* Plan for a described device without touching CUDA (host logic only).
 * `max_active_clusters` is the occupancy answer to use for the chosen shape;
 * pass 0 to estimate it as floor(sm_count * ctas_per_sm / P). */
DSMEM_HIST_API int dsmem_hist_plan_for_device(const dsmem_hist_device_t* device, int32_t num_bins, int64_t n,
                               const dsmem_hist_request_t* request, int32_t max_active_clusters,
                               dsmem_hist_plan_t* out);

/* Name of an error code (static string). */
DSMEM_HIST_API const char* dsmem_hist_strerror(int code);

/* The calling thread's most recent error message ("" if none). */
DSMEM_HIST_API const char* dsmem_hist_last_error(void);

/* Frees the library's cached device resources (memory pools, copy streams,
 * events) on every device it touched.  Call only when no dsmem_hist work is
 * in flight; later calls recreate what they need. */
DSMEM_HIST_API void dsmem_hist_release(void);

/* Reads and clears the current device's status word of the key-shipping
 * kernel (DSMEM_HIST_KERNEL_SHIP).  That kernel waits for its peers' inbox
 * bytes with bounded waits (about 50 ms each); a wait that gives up sets bit 0
 * of the word (and of the calling stream's host-mapped word, see the
 * conventions at the top) and skips that inbox, so the histogram of that
 * launch is wrong.  *status (may be NULL) receives the word.  Reads with
 * cudaMemcpyFromSymbol, which is ordered with the legacy default stream only:
 * synchronise the streams of interest first.  Returns DSMEM_HIST_OK if the
 * word was 0, DSMEM_HIST_ETIMEOUT if a wait gave up since the last call,
 * DSMEM_HIST_ECUDA on a CUDA error.  No counterpart in the pages' design,
 * which waits only on cluster barriers. */
DSMEM_HIST_API int dsmem_hist_device_status(uint32_t* status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
DSMEM_HIST_API int dsmem_hist_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSMEM_HIST_H */
