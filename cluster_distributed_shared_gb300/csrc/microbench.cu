// DSMEM primitive microbenchmarks on the current GPU: the rates that decide
// how a cluster histogram should move increments between CTAs.  They
// re-measure on this hardware what "Hopper DSMEM vs HBM" (ping-pong test and
// the 16 KB tile-exchange test) and "CREDIT" (microbenchmark section: remote
// versus local access) measured on Hopper.
//
// Every rate kernel runs 1024 threads per CTA with 128 KiB of dynamic shared
// memory (one CTA per SM), as many clusters as can be resident, and times
// its loop with clock64 per CTA.  Addresses stay inside the 32768-counter
// slice; every thread reaches the closing cluster barrier, so no CTA exits
// while a peer may still touch its shared memory.  The ping-pong kernels run
// one cluster and time one thread's round trips.  The tile-exchange kernels
// run every resident cluster with 128 threads per CTA and are timed with CUDA
// events.
//
// Every probe also counts its work on the device after its closing barrier,
// into a 64-bit counter the host compares with the operations the probe
// issues by construction: the reductions by summing the counters they
// landed in (every increment must have arrived), the stores and barriers by
// each thread's count of operations issued, the ping-pong by the rounds that
// completed, and the tile exchanges by the sum of every word pulled from the
// peer (which must equal the peer's tile, summed over every iteration).
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
                                                         uint32_t* sink, unsigned long long* counted) {
  extern __shared__ __align__(16) uint32_t slice[];
  const uint32_t P = cluster_nctarank(), rank = cluster_ctarank();
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  for (uint32_t i = threadIdx.x; i < kSlice; i += blockDim.x) slice[i] = 0;
  cluster_barrier();
  const uint32_t base = smem_u32(slice);
  uint32_t x = (blockIdx.x * 1024u + threadIdx.x) * 2654435761u + 12345u;  // LCG state
  uint32_t issued = 0;
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
      ++issued;
    } else if (kKind == DSMEM_HIST_MB_REMOTE_ST16_COALESCED) {
      // each warp writes 512 contiguous bytes of one peer's slice
      const uint32_t p2 = P > 1 ? (rank + 1u + static_cast<uint32_t>(it + warp) % (P - 1u)) % P : rank;
      const uint32_t off = ((warp * 512u + static_cast<uint32_t>(it) * 16384u) & (4u * kSlice - 1u)) + 16u * lane;
      st_cluster_v4(map_rank(base + off, p2), make_uint4(x, x, x, x));
      ++issued;
    } else {  // DSMEM_HIST_MB_CLUSTER_BARRIER
      cluster_barrier();
      ++issued;
    }
  }
  const long long t1 = clock64();
  cluster_barrier();  // every remote operation has landed
  if (threadIdx.x == 0) cycles[blockIdx.x] = static_cast<unsigned long long>(t1 - t0);
  if (kKind == DSMEM_HIST_MB_LOCAL_RED || kKind == DSMEM_HIST_MB_REMOTE_RED) {
    // The increments that landed in this CTA's slice.
    unsigned long long s = 0;
    for (uint32_t i = threadIdx.x; i < kSlice; i += blockDim.x) s += slice[i];
    atomicAdd(counted, s);
  } else {
    atomicAdd(counted, static_cast<unsigned long long>(issued));
    if (slice[threadIdx.x & (kSlice - 1u)] == 0xFFFFFFFFu) sink[0] = x;
  }
}

// Ping-pong between thread 0 of CTA 0 and thread 0 of CTA 1 of one
// cluster: round k, CTA 0 stores k into CTA 1's flag and waits for CTA 1 to
// store k into its own.  Flags live in the receiver's shared memory
// (kGlobal = false) or in `gflags` (kGlobal = true).  Every poll loop is
// bounded; a loop that gives up sets sink[1] and ends the test on both sides
// (the peer then gives up too, after at most its own bound).  CTA 0 counts
// the rounds that completed.
template <bool kGlobal>
__global__ void pingpong_kernel(int iters, unsigned long long* cycles, uint32_t* sink,
                                uint32_t* gflags, unsigned long long* counted) {
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
    uint32_t rounds = 0;
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
      ++rounds;
    }
    const long long t1 = clock64();
    if (rank == 0) {
      cycles[0] = static_cast<unsigned long long>(t1 - t0);
      *counted = rounds;
    }
  }
  cluster_barrier();  // no CTA exits while its peer may still store into it
}

// The 16 KB tile exchange between the two CTAs of a pair (ranks 2j and
// 2j + 1 of a cluster): every CTA owns a tile of 4096 32-bit words, word i of
// CTA b (global index) holding b * 4096 + i, and each iteration lands the
// peer's whole tile in this CTA's shared memory.
//   kGlobal = false: pulled straight from the peer's shared memory through
//     the cluster address of the same offset (ld.shared::cluster), then one
//     cluster barrier, so the peer's tile is not reused before everyone has
//     read it.
//   kGlobal = true: this CTA writes its tile to its slot of a global scratch,
//     fences, meets the cluster barrier, reads the peer's slot (at L2, not
//     from a stale L1 line), and meets the barrier again before the slot is
//     rewritten.
// Every pulled word is added into a per-thread sum; the sums reach `counted`
// after the closing barrier, where the host compares them with
// iters * (sum of every peer tile).
constexpr uint32_t kTileWords = 4096;
constexpr uint32_t kTileThreads = 128;

__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t cluster_addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(cluster_addr));
  return v;
}
__device__ __forceinline__ uint4 ld_global_cg_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

template <bool kGlobal>
__global__ void __launch_bounds__(kTileThreads) tile_exchange_kernel(int iters, uint4* scratch,
                                                                    unsigned long long* counted) {
  __shared__ __align__(16) uint32_t src[kTileWords];
  __shared__ __align__(16) uint32_t dst[kTileWords];
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const uint32_t me = blockIdx.x, them = blockIdx.x ^ 1u;  // pairs stay inside a cluster (P even)
  for (uint32_t i = threadIdx.x; i < kTileWords; i += kTileThreads) src[i] = me * kTileWords + i;
  cluster_barrier();
  constexpr uint32_t kVecs = kTileWords / 4;  // 16-byte vectors per tile
  const uint32_t src_peer = map_rank(smem_u32(src), peer);
  uint4* dst4 = reinterpret_cast<uint4*>(dst);
  const uint4* src4 = reinterpret_cast<const uint4*>(src);
  uint4* mine = scratch + static_cast<size_t>(me) * kVecs;
  const uint4* theirs = scratch + static_cast<size_t>(them) * kVecs;
  unsigned long long sum = 0;
  for (int it = 0; it < iters; ++it) {
    if (kGlobal) {
      for (uint32_t v = threadIdx.x; v < kVecs; v += kTileThreads) mine[v] = src4[v];
      __threadfence();
      cluster_barrier();
      for (uint32_t v = threadIdx.x; v < kVecs; v += kTileThreads) {
        const uint4 w = ld_global_cg_v4(theirs + v);
        dst4[v] = w;
        sum += static_cast<unsigned long long>(w.x) + w.y + w.z + w.w;
      }
      cluster_barrier();
    } else {
      for (uint32_t v = threadIdx.x; v < kVecs; v += kTileThreads) {
        const uint4 w = ld_cluster_v4(src_peer + 16u * v);
        dst4[v] = w;
        sum += static_cast<unsigned long long>(w.x) + w.y + w.z + w.w;
      }
      cluster_barrier();
    }
  }
  atomicAdd(counted, sum);
  cluster_barrier();  // no CTA exits while its pair may still read its tile
}

cudaLaunchConfig_t cluster_config(int cluster_size, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Small device buffers of one probe, freed by the destructor.
struct ProbeBuffers {
  unsigned long long* cycles = nullptr;
  uint32_t* words = nullptr;
  unsigned long long* counted = nullptr;
  ~ProbeBuffers() {
    cudaFree(cycles);
    cudaFree(words);
    cudaFree(counted);
  }
  cudaError_t alloc(size_t n_cycles, size_t n_words) {
    cudaError_t e;
    if ((e = cudaMalloc(&cycles, sizeof(unsigned long long) * n_cycles)) != cudaSuccess) return e;
    if ((e = cudaMalloc(&words, sizeof(uint32_t) * n_words)) != cudaSuccess) return e;
    return cudaMalloc(&counted, sizeof(unsigned long long));
  }
};

// Times launches: one warm-up, then the timed one; `counted` is zeroed before
// each, so it holds the timed launch's count afterwards.
template <class Launch>
cudaError_t timed_launch(Launch launch, unsigned long long* counted, float* ms) {
  cudaEvent_t a = nullptr, b = nullptr;
  cudaError_t e = cudaEventCreate(&a);
  if (e == cudaSuccess) e = cudaEventCreate(&b);
  for (int run = 0; run < 2 && e == cudaSuccess; ++run) {
    if ((e = cudaMemset(counted, 0, sizeof(unsigned long long))) != cudaSuccess) break;
    if (run == 1) cudaEventRecord(a);
    e = launch();
    if (run == 1) cudaEventRecord(b);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
  }
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, a, b);
  if (a) cudaEventDestroy(a);
  if (b) cudaEventDestroy(b);
  return e;
}

template <bool kGlobal>
cudaError_t run_pingpong(int cluster_size, int iters, dsmem_hist_microbench_result_t* out,
                         bool* timed_out) {
  auto fn = pingpong_kernel<kGlobal>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(cluster_size, attr);
  cfg.blockDim = dim3(32);
  cfg.gridDim = dim3(cluster_size);
  ProbeBuffers buf;  // words: sink[2], then the two global flags
  if ((e = buf.alloc(1, 4)) != cudaSuccess) return e;
  uint32_t host[2] = {0, 0};
  float ms = 0;
  e = timed_launch([&] {
    cudaError_t le = cudaMemset(buf.words, 0, 4 * sizeof(uint32_t));
    return le != cudaSuccess ? le : cudaLaunchKernelEx(&cfg, fn, iters, buf.cycles, buf.words,
                                                        buf.words + 2, buf.counted);
  }, buf.counted, &ms);
  unsigned long long c = 0, counted = 0;
  if (e == cudaSuccess) e = cudaMemcpy(host, buf.words, 2 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&c, buf.cycles, sizeof(c), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&counted, buf.counted, sizeof(counted), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) {
    out->ms = ms;
    out->value = static_cast<double>(c) / (2.0 * iters);
    out->ops_expected = static_cast<uint64_t>(iters);
    out->ops_counted = counted;
    *timed_out = host[1] != 0;
  }
  return e;
}

template <int kKind>
cudaError_t run_probe(int cluster_size, int iters, dsmem_hist_microbench_result_t* out) {
  const int threads = 1024, smem = 4 * kSlice;
  auto fn = probe_kernel<kKind>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(cluster_size, attr);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.gridDim = dim3(cluster_size);
  int clusters = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg)) != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const int grid = clusters * cluster_size;
  cfg.gridDim = dim3(grid);
  ProbeBuffers buf;
  if ((e = buf.alloc(grid, 1)) != cudaSuccess) return e;
  float ms = 0;
  e = timed_launch([&] { return cudaLaunchKernelEx(&cfg, fn, iters, buf.cycles, buf.words, buf.counted); },
                   buf.counted, &ms);
  unsigned long long counted = 0;
  unsigned long long* h = nullptr;
  if (e == cudaSuccess) e = cudaMemcpy(&counted, buf.counted, sizeof(counted), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) {
    h = new unsigned long long[grid];
    e = cudaMemcpy(h, buf.cycles, sizeof(unsigned long long) * grid, cudaMemcpyDeviceToHost);
  }
  if (e == cudaSuccess) {
    double sum = 0;
    for (int i = 0; i < grid; ++i) sum += static_cast<double>(h[i]);
    const double mean_cycles = sum / grid;
    const double units = kKind == DSMEM_HIST_MB_CLUSTER_BARRIER ? iters
                         : kKind == DSMEM_HIST_MB_REMOTE_ST16_SCATTERED ||
                                 kKind == DSMEM_HIST_MB_REMOTE_ST16_COALESCED
                             ? 16.0 * threads * iters
                             : 1.0 * threads * iters;
    // barriers: cycles per barrier; the others: units per clock per SM
    out->value = kKind == DSMEM_HIST_MB_CLUSTER_BARRIER ? mean_cycles / units : units / mean_cycles;
    out->ms = ms;
    out->ops_expected = static_cast<uint64_t>(grid) * threads * static_cast<uint64_t>(iters);
    out->ops_counted = counted;
  }
  delete[] h;
  return e;
}

template <bool kGlobal>
cudaError_t run_tile_exchange(int cluster_size, int iters, dsmem_hist_microbench_result_t* out) {
  auto fn = tile_exchange_kernel<kGlobal>;
  // One CTA per SM, as in the page's test (every SM runs one CTA of a
  // pair): unused dynamic shared memory keeps a second CTA off each SM.
  const int pad_smem = 100 * 1024;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, pad_smem)) != cudaSuccess)
    return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(cluster_size, attr);
  cfg.blockDim = dim3(kTileThreads);
  cfg.dynamicSmemBytes = pad_smem;
  cfg.gridDim = dim3(cluster_size);
  int clusters = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg)) != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const int grid = clusters * cluster_size;
  cfg.gridDim = dim3(grid);
  ProbeBuffers buf;
  void* scratch = nullptr;
  if ((e = buf.alloc(1, 1)) != cudaSuccess) return e;
  if (kGlobal && (e = cudaMalloc(&scratch, static_cast<size_t>(grid) * kTileWords * 4)) != cudaSuccess)
    return e;
  float ms = 0;
  e = timed_launch([&] {
    return cudaLaunchKernelEx(&cfg, fn, iters, static_cast<uint4*>(scratch), buf.counted);
  }, buf.counted, &ms);
  unsigned long long counted = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&counted, buf.counted, sizeof(counted), cudaMemcpyDeviceToHost);
  if (scratch) cudaFree(scratch);
  if (e == cudaSuccess) {
    // Expected: every CTA b pulls the tile of b ^ 1 once per iteration;
    // sum_i ((b ^ 1) * 4096 + i) = 4096 * 4096 * (b ^ 1) + 4096 * 4095 / 2.
    unsigned long long per_iter = 0;
    for (int b = 0; b < grid; ++b)
      per_iter += 4096ull * 4096ull * static_cast<unsigned long long>(b ^ 1) + 4096ull * 4095ull / 2ull;
    out->value = ms;
    out->ms = ms;
    out->bytes_per_s = static_cast<double>(grid) * kTileWords * 4.0 * iters / (ms * 1e-3);
    out->ops_expected = per_iter * static_cast<unsigned long long>(iters);
    out->ops_counted = counted;
    out->ctas = grid;
  }
  return e;
}

}  // namespace
}  // namespace dsmh

extern "C" int dsmem_hist_microbench(int32_t kind, int32_t cluster_size, int32_t iters,
                                     dsmem_hist_microbench_result_t* out) {
  if (!out || iters < 1 || iters > (1 << 24) || cluster_size < 1 || cluster_size > 16)
    return dsmh::record_error(DSMEM_HIST_EINVAL, "microbench: bad arguments");
  *out = dsmem_hist_microbench_result_t{};
  cudaError_t e;
  switch (kind) {
    case DSMEM_HIST_MB_LOCAL_RED:
      e = dsmh::run_probe<DSMEM_HIST_MB_LOCAL_RED>(cluster_size, iters, out);
      break;
    case DSMEM_HIST_MB_REMOTE_RED:
      e = dsmh::run_probe<DSMEM_HIST_MB_REMOTE_RED>(cluster_size, iters, out);
      break;
    case DSMEM_HIST_MB_REMOTE_ST16_SCATTERED:
      e = dsmh::run_probe<DSMEM_HIST_MB_REMOTE_ST16_SCATTERED>(cluster_size, iters, out);
      break;
    case DSMEM_HIST_MB_REMOTE_ST16_COALESCED:
      e = dsmh::run_probe<DSMEM_HIST_MB_REMOTE_ST16_COALESCED>(cluster_size, iters, out);
      break;
    case DSMEM_HIST_MB_CLUSTER_BARRIER:
      e = dsmh::run_probe<DSMEM_HIST_MB_CLUSTER_BARRIER>(cluster_size, iters, out);
      break;
    case DSMEM_HIST_MB_DSMEM_PINGPONG:
    case DSMEM_HIST_MB_GMEM_PINGPONG: {
      if (cluster_size < 2 || iters > (1 << 20))
        return dsmh::record_error(DSMEM_HIST_EINVAL, "microbench: ping-pong needs cluster_size >= 2, iters <= 2^20");
      bool timed_out = false;
      e = kind == DSMEM_HIST_MB_DSMEM_PINGPONG
              ? dsmh::run_pingpong<false>(cluster_size, iters, out, &timed_out)
              : dsmh::run_pingpong<true>(cluster_size, iters, out, &timed_out);
      if (e == cudaSuccess && timed_out)
        return dsmh::record_error(DSMEM_HIST_ETIMEOUT, "microbench: ping-pong peer did not answer");
      break;
    }
    case DSMEM_HIST_MB_TILE_EXCHANGE_DSMEM:
    case DSMEM_HIST_MB_TILE_EXCHANGE_GMEM:
      if (cluster_size < 2 || (cluster_size & 1) || iters > (1 << 20))
        return dsmh::record_error(DSMEM_HIST_EINVAL,
                                  "microbench: tile exchange needs an even cluster_size, iters <= 2^20");
      e = kind == DSMEM_HIST_MB_TILE_EXCHANGE_DSMEM ? dsmh::run_tile_exchange<false>(cluster_size, iters, out)
                                                    : dsmh::run_tile_exchange<true>(cluster_size, iters, out);
      break;
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
