// DSMEM primitive microbenchmarks on the current GPU: the rates that decide
// how a cluster histogram should move increments between CTAs.  They
// re-measure on this hardware what "Hopper DSMEM vs HBM" (tile exchange and
// ping-pong sections) and "CREDIT" (microbenchmark section: remote versus
// local access) measured on Hopper.
//
// Every rate kernel runs 1024 threads per CTA with 128 KiB of dynamic shared
// memory (one CTA per SM), as many clusters as can be resident, and times
// its loop with clock64 per CTA.  Addresses stay inside the 32768-counter
// slice; every thread reaches the closing cluster barrier, so no CTA exits
// while a peer may still touch its shared memory.  The ping-pong kernels run
// one cluster and time one thread's round trips.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsmem_hist.h"
#include "internal.h"
#include "ptx.cuh"

namespace dsmh {
namespace {

using namespace ptx;

constexpr uint32_t kSlice = 32768;  // counters (128 KiB)

template <int kKind>
__global__ void __launch_bounds__(1024, 1) probe_kernel(int iters, unsigned long long* cycles,
                                                         uint32_t* sink) {
  extern __shared__ __align__(16) uint32_t slice[];
  const uint32_t P = cluster_nctarank(), rank = cluster_ctarank();
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  for (uint32_t i = threadIdx.x; i < kSlice; i += blockDim.x) slice[i] = 0;
  cluster_barrier();
  const uint32_t base = smem_u32(slice);
  uint32_t x = (blockIdx.x * 1024u + threadIdx.x) * 2654435761u + 12345u;  // LCG state
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    x = x * 1664525u + 1013904223u;
    const uint32_t local = (x >> 14) & (kSlice - 1u);
    // a peer other than this CTA (this CTA itself when P == 1)
    const uint32_t peer = P > 1 ? (rank + 1u + (x >> 29) % (P - 1u)) % P : rank;
    if (kKind == DSMEM_HIST_MB_LOCAL_RED) {
      red_add_local(base + 4u * local, 1u);
    } else if (kKind == DSMEM_HIST_MB_REMOTE_RED) {
      red_add_cluster(map_rank(base + 4u * local, peer), 1u);
    } else if (kKind == DSMEM_HIST_MB_REMOTE_ST16_SCATTERED) {
      st_cluster_v4(map_rank(base + 4u * (local & ~3u), peer), make_uint4(x, x, x, x));
    } else if (kKind == DSMEM_HIST_MB_REMOTE_ST16_COALESCED) {
      // each warp writes 512 contiguous bytes of one peer's slice
      const uint32_t p2 = P > 1 ? (rank + 1u + static_cast<uint32_t>(it + warp) % (P - 1u)) % P : rank;
      const uint32_t off = ((warp * 512u + static_cast<uint32_t>(it) * 16384u) & (4u * kSlice - 1u)) + 16u * lane;
      st_cluster_v4(map_rank(base + off, p2), make_uint4(x, x, x, x));
    } else {  // DSMEM_HIST_MB_CLUSTER_BARRIER
      cluster_barrier();
    }
  }
  const long long t1 = clock64();
  cluster_barrier();
  if (threadIdx.x == 0) cycles[blockIdx.x] = static_cast<unsigned long long>(t1 - t0);
  if (slice[threadIdx.x & (kSlice - 1u)] == 0xFFFFFFFFu) sink[0] = x;
}

// Ping-pong between thread 0 of CTA 0 and thread 0 of CTA 1 of one
// cluster: round k, CTA 0 stores k into CTA 1's flag and waits for CTA 1 to
// store k into its own.  Flags live in the receiver's shared memory
// (kGlobal = false) or in `gflags` (kGlobal = true).  Every poll loop is
// bounded; a loop that gives up sets sink[1] and ends the test on both sides
// (the peer then gives up too, after at most its own bound).
template <bool kGlobal>
__global__ void pingpong_kernel(int iters, unsigned long long* cycles, uint32_t* sink,
                                uint32_t* gflags) {
  __shared__ uint32_t flag;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) flag = 0;
  cluster_barrier();
  constexpr uint32_t kPolls = 1u << 20;
  if (threadIdx.x == 0 && rank < 2) {
    const uint32_t peer = rank ^ 1u;
    const uint32_t mine = smem_u32(&flag);
    const uint32_t theirs = map_rank(mine, peer);
    uint32_t* gmine = gflags + rank;
    uint32_t* gtheirs = gflags + peer;
    bool ok = true;
    const long long t0 = clock64();
    for (uint32_t k = 1; ok && k <= static_cast<uint32_t>(iters); ++k) {
      if (rank == 0) {
        if (kGlobal) st_release_gpu(gtheirs, k);
        else st_release_cluster(theirs, k);
      }
      uint32_t polls = 0, seen = 0;
      do {
        seen = kGlobal ? ld_acquire_gpu(gmine) : ld_acquire_cluster(mine);
      } while (seen < k && ++polls < kPolls);
      if (seen < k) {
        ok = false;
        atomicOr(sink + 1, 1u);
        break;
      }
      if (rank == 1) {
        if (kGlobal) st_release_gpu(gtheirs, k);
        else st_release_cluster(theirs, k);
      }
    }
    const long long t1 = clock64();
    if (rank == 0) cycles[0] = static_cast<unsigned long long>(t1 - t0);
  }
  cluster_barrier();  // no CTA exits while its peer may still store into it
}

template <bool kGlobal>
cudaError_t run_pingpong(int cluster_size, int iters, double* hop_cycles, double* ms, bool* timed_out) {
  auto fn = pingpong_kernel<kGlobal>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(32);
  cfg.gridDim = dim3(cluster_size);
  unsigned long long* cycles = nullptr;
  uint32_t* buf = nullptr;  // sink[2], then the two global flags
  if ((e = cudaMalloc(&cycles, sizeof(unsigned long long))) != cudaSuccess) return e;
  if ((e = cudaMalloc(&buf, 4 * sizeof(uint32_t))) != cudaSuccess) {
    cudaFree(cycles);
    return e;
  }
  cudaEvent_t a = nullptr, b = nullptr;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  uint32_t host[2] = {0, 0};
  for (int run = 0; run < 2 && e == cudaSuccess; ++run) {  // warm-up, then the timed run
    if ((e = cudaMemset(buf, 0, 4 * sizeof(uint32_t))) != cudaSuccess) break;
    cudaEventRecord(a);
    e = cudaLaunchKernelEx(&cfg, fn, iters, cycles, buf, buf + 2);
    cudaEventRecord(b);
    if (e == cudaSuccess) e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaMemcpy(host, buf, 2 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && host[1]) break;
  }
  if (e == cudaSuccess) {
    float t = 0;
    cudaEventElapsedTime(&t, a, b);
    *ms = t;
    unsigned long long c = 0;
    e = cudaMemcpy(&c, cycles, sizeof(c), cudaMemcpyDeviceToHost);
    *hop_cycles = static_cast<double>(c) / (2.0 * iters);
    *timed_out = host[1] != 0;
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  cudaFree(cycles);
  cudaFree(buf);
  return e;
}

template <int kKind>
cudaError_t run_probe(int cluster_size, int iters, double* per_clk, double* ms) {
  const int threads = 1024, smem = 4 * kSlice;
  auto fn = probe_kernel<kKind>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.gridDim = dim3(cluster_size);
  int clusters = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg)) != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const int grid = clusters * cluster_size;
  cfg.gridDim = dim3(grid);
  unsigned long long* cycles = nullptr;
  uint32_t* sink = nullptr;
  if ((e = cudaMalloc(&cycles, sizeof(unsigned long long) * grid)) != cudaSuccess) return e;
  if ((e = cudaMalloc(&sink, sizeof(uint32_t))) != cudaSuccess) {
    cudaFree(cycles);
    return e;
  }
  cudaEvent_t a = nullptr, b = nullptr;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  e = cudaLaunchKernelEx(&cfg, fn, iters, cycles, sink);  // warm-up
  if (e == cudaSuccess) {
    cudaEventRecord(a);
    e = cudaLaunchKernelEx(&cfg, fn, iters, cycles, sink);
    cudaEventRecord(b);
  }
  if (e == cudaSuccess) e = cudaEventSynchronize(b);
  if (e == cudaSuccess) {
    float t = 0;
    cudaEventElapsedTime(&t, a, b);
    *ms = t;
    unsigned long long* h = new unsigned long long[grid];
    e = cudaMemcpy(h, cycles, sizeof(unsigned long long) * grid, cudaMemcpyDeviceToHost);
    double sum = 0;
    for (int i = 0; i < grid; ++i) sum += static_cast<double>(h[i]);
    delete[] h;
    const double mean_cycles = sum / grid;
    const double units = kKind == DSMEM_HIST_MB_CLUSTER_BARRIER ? iters
                         : kKind == DSMEM_HIST_MB_REMOTE_ST16_SCATTERED ||
                                 kKind == DSMEM_HIST_MB_REMOTE_ST16_COALESCED
                             ? 16.0 * threads * iters
                             : 1.0 * threads * iters;
    // barriers: cycles per barrier; the others: units per clock per SM
    *per_clk = kKind == DSMEM_HIST_MB_CLUSTER_BARRIER ? mean_cycles / units : units / mean_cycles;
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  cudaFree(cycles);
  cudaFree(sink);
  return e;
}

}  // namespace
}  // namespace dsmh

extern "C" int dsmem_hist_microbench(int32_t kind, int32_t cluster_size, int32_t iters,
                                     double* value, double* ms) {
  if (!value || !ms || iters < 1 || iters > (1 << 24) || cluster_size < 1 || cluster_size > 16)
    return dsmh::record_error(DSMEM_HIST_EINVAL, "microbench: bad arguments");
  cudaError_t e;
  switch (kind) {
    case DSMEM_HIST_MB_LOCAL_RED:
      e = dsmh::run_probe<DSMEM_HIST_MB_LOCAL_RED>(cluster_size, iters, value, ms);
      break;
    case DSMEM_HIST_MB_REMOTE_RED:
      e = dsmh::run_probe<DSMEM_HIST_MB_REMOTE_RED>(cluster_size, iters, value, ms);
      break;
    case DSMEM_HIST_MB_REMOTE_ST16_SCATTERED:
      e = dsmh::run_probe<DSMEM_HIST_MB_REMOTE_ST16_SCATTERED>(cluster_size, iters, value, ms);
      break;
    case DSMEM_HIST_MB_REMOTE_ST16_COALESCED:
      e = dsmh::run_probe<DSMEM_HIST_MB_REMOTE_ST16_COALESCED>(cluster_size, iters, value, ms);
      break;
    case DSMEM_HIST_MB_CLUSTER_BARRIER:
      e = dsmh::run_probe<DSMEM_HIST_MB_CLUSTER_BARRIER>(cluster_size, iters, value, ms);
      break;
    case DSMEM_HIST_MB_DSMEM_PINGPONG:
    case DSMEM_HIST_MB_GMEM_PINGPONG: {
      if (cluster_size < 2 || iters > (1 << 20))
        return dsmh::record_error(DSMEM_HIST_EINVAL, "microbench: ping-pong needs cluster_size >= 2, iters <= 2^20");
      bool timed_out = false;
      e = kind == DSMEM_HIST_MB_DSMEM_PINGPONG
              ? dsmh::run_pingpong<false>(cluster_size, iters, value, ms, &timed_out)
              : dsmh::run_pingpong<true>(cluster_size, iters, value, ms, &timed_out);
      if (e == cudaSuccess && timed_out)
        return dsmh::record_error(DSMEM_HIST_ETIMEOUT, "microbench: ping-pong peer did not answer");
      break;
    }
    default:
      return dsmh::record_error(DSMEM_HIST_EINVAL, "microbench: unknown kind");
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return dsmh::record_error(e == cudaErrorInvalidConfiguration ? DSMEM_HIST_EUNSUPPORTED
                                                                 : DSMEM_HIST_ECUDA,
                              cudaGetErrorString(e));
  }
  return DSMEM_HIST_OK;
}
