// Kernels of the thread-block-cluster histogram, written for sm_103a.
//
// Method ("Distributed Shared Memory", section "The cluster histogram"): the
// bins are split into equal slices of S counters, one slice in the dynamic
// shared memory of each of the P CTAs of a cluster; a key's owner is
// rel / S and its counter rel mod S in the owner's slice.  Every CTA zeroes
// its slice, the cluster synchronises, every thread increments the owner's
// counter through distributed shared memory, the cluster synchronises again,
// and the slices leave the chip.
//
// GB300 design (what differs from the page's Hopper listing):
//   - cluster shape chosen at launch (cudaLaunchKernelEx) by the planner;
//   - a persistent grid of C clusters; the keys are streamed with 16-byte
//     read-only loads, four vectors in flight per thread, one warp covering
//     512 contiguous bytes per load;
//   - optional warp pre-aggregation: lanes holding equal keys are found with
//     __match_any_sync, and their lowest lane adds the popcount once;
//   - remote increments are `mapa` + `red.shared::cluster.add.u32` (no
//     return value), bracketed by `barrier.cluster` arrive.release /
//     wait.acquire;
//   - each cluster writes its slices as one partial row with 16-byte
//     coalesced stores (no per-bin global atomics), and a second kernel sums
//     the rows into `bins`;
//   - bin counts beyond one cluster's capacity are handled by passes over
//     bin ranges inside the same launch.
// Exit rule ("Hopper DSMEM vs HBM", section on the SMEM lifecycle trap):
// no CTA touches a peer's shared memory after the closing cluster barrier,
// and every thread of every CTA reaches every cluster barrier.

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace dsmh {
namespace {

using namespace ptx;

struct SliceMap {
  uint32_t base;        // first bin of the current pass
  uint32_t range;       // bins in this pass (<= P*S, <= num_bins - base)
  uint32_t S;
  uint64_t magic;
  uint32_t slice_addr;  // shared::cta address of this CTA's slice
};

// One key, warp-converged.  `rel < range` also rejects negative keys:
// base + range <= num_bins < 2^31, so a negative key viewed as unsigned
// gives rel >= 2^31 - base > range.
template <bool kAggregate>
__device__ __forceinline__ void count_key(int32_t key, const SliceMap& m, uint32_t lane) {
  const uint32_t rel = static_cast<uint32_t>(key) - m.base;
  uint32_t add = 1;
  bool issue = rel < m.range;
  if (kAggregate) {
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    issue = issue && (static_cast<uint32_t>(__ffs(peers) - 1) == lane);
    add = static_cast<uint32_t>(__popc(peers));
  }
  if (issue) {
    const uint32_t owner = static_cast<uint32_t>((static_cast<uint64_t>(rel) * m.magic) >> 40);
    const uint32_t local = rel - owner * m.S;
    red_add_cluster(map_rank(m.slice_addr + 4u * local, owner), add);
  }
}

template <bool kAggregate>
__device__ __forceinline__ void count_vec(const int4& v, const SliceMap& m, uint32_t lane) {
  count_key<kAggregate>(v.x, m, lane);
  count_key<kAggregate>(v.y, m, lane);
  count_key<kAggregate>(v.z, m, lane);
  count_key<kAggregate>(v.w, m, lane);
}

// Streams every key of the input once and counts those of the current pass.
// Warp-tiles of 32 vectors (512 B) are dealt round-robin over all warps of
// the grid; the ragged leftovers (unaligned head, a partial tile, the last
// 1-3 keys) are swept by the grid's last warp, 32 at a time, with
// out-of-range sentinels filling idle lanes so the warp stays converged.
template <bool kAggregate>
__device__ __forceinline__ void stream_keys(const ClusterHistArgs& a, const SliceMap& m) {
  const uint32_t lane = threadIdx.x & 31u;
  const int64_t warps_per_cta = blockDim.x >> 5;
  const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * warps_per_cta;

  const int64_t rest = a.n - a.head;
  const int64_t nvec = rest >> 2;
  const int64_t ntiles = nvec >> 5;
  const int4* vec = reinterpret_cast<const int4*>(a.keys + a.head) + lane;

  int64_t t = gwarp;
  for (; t + (kVecPerThread - 1) * nwarps < ntiles; t += kVecPerThread * nwarps) {
    int4 v[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) v[u] = ld_stream_v4(vec + ((t + u * nwarps) << 5));
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) count_vec<kAggregate>(v[u], m, lane);
  }
  for (; t < ntiles; t += nwarps) count_vec<kAggregate>(ld_stream_v4(vec + (t << 5)), m, lane);

  if (gwarp == nwarps - 1) {
    // Leftover index j < head maps to keys[j]; j >= head maps to the keys
    // after the last full tile, which run contiguously up to n.
    const int64_t after = a.head + (ntiles << 7);
    const int64_t leftover = static_cast<int64_t>(a.head) + (a.n - after);
    for (int64_t j0 = 0; j0 < leftover; j0 += 32) {
      const int64_t j = j0 + lane;
      int32_t key = -1;
      if (j < leftover) key = a.keys[j < a.head ? j : after + (j - a.head)];
      count_key<kAggregate>(key, m, lane);
    }
  }
}

template <bool kAggregate>
__global__ void __launch_bounds__(1024, 1) cluster_hist_kernel(const ClusterHistArgs a) {
  extern __shared__ __align__(16) uint32_t slice[];
  const uint32_t P = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const uint32_t cid = cluster_id_x();
  const uint32_t S = a.S;

  SliceMap m;
  m.S = S;
  m.magic = a.magic;
  m.slice_addr = smem_u32(slice);

  for (uint32_t pass = 0; pass < a.passes; ++pass) {
    m.base = pass * P * S;
    const uint32_t left = a.num_bins - m.base;
    m.range = left < P * S ? left : P * S;

    // 1. zero this CTA's slice; the barrier publishes every slice's zeros
    //    to the whole cluster before any remote increment.
    uint4* s4 = reinterpret_cast<uint4*>(slice);
    for (uint32_t i = threadIdx.x; i < S / 4; i += blockDim.x) s4[i] = make_uint4(0, 0, 0, 0);
    cluster_barrier();

    // 2. stream the keys, increments to the owners' slices.
    stream_keys<kAggregate>(a, m);

    // 3. every remote increment has landed once all CTAs pass this barrier;
    //    after it, each CTA touches only its own shared memory.
    cluster_barrier();

    // 4. flush this CTA's slice into the cluster's partial row.
    const uint32_t first = m.base + rank * S;
    if (m.range > rank * S) {
      const uint32_t cnt = m.range - rank * S < S ? m.range - rank * S : S;
      uint4* dst = reinterpret_cast<uint4*>(a.partials + static_cast<size_t>(cid) * a.stride + first);
      const uint32_t nv = (cnt + 3) / 4;  // row padding absorbs the last partial vector
      for (uint32_t i = threadIdx.x; i < nv; i += blockDim.x) {
        uint4 v = s4[i];
        if (a.accumulate) {
          const uint4 o = dst[i];
          v.x += o.x;
          v.y += o.y;
          v.z += o.z;
          v.w += o.w;
        }
        dst[i] = v;
      }
    }
    if (pass + 1 < a.passes) __syncthreads();  // flush reads finish before re-zeroing
  }
}

// bins[i] = sum over clusters c of partials[c][i] (mod 2^32).  A CTA owns
// 256 / G columns of 16-byte vectors; its G row groups each sum every G-th
// partial row of those columns with four loads in flight, so a thread waits
// on about ceil(C / 4G) loads in turn instead of ceil(C / 4), and the groups'
// sums meet in shared memory.
// With hot_word non-null the kernel also reports hot bins, for the library to
// pick the hot-bin kernel on later calls on the same stream (both words are
// pinned, host-mapped):
//   - the first thread stamps *seq_word with this call's sequence number;
//   - a thread whose bin holds at least hot_min keys writes (seq << 32) | bin
//     to *hot_word.  At most n / hot_min bins can qualify; any one will do.
template <int G>
__global__ void __launch_bounds__(256) reduce_partials_kernel(const uint32_t* __restrict__ partials,
                                                              uint64_t stride, uint32_t num_clusters,
                                                              uint32_t num_bins,
                                                              uint32_t* __restrict__ bins,
                                                              int bins_vec_ok, uint32_t hot_min,
                                                              unsigned long long* hot_word,
                                                              uint32_t* seq_word, uint32_t seq) {
  if (hot_word && blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<volatile uint32_t*>(seq_word) = seq;
  constexpr uint32_t kCols = 256 / G;
  __shared__ uint4 part[G][kCols];
  const uint32_t col = threadIdx.x % kCols, g = threadIdx.x / kCols;
  const uint32_t nv = (num_bins + 3) / 4;
  const size_t row4 = stride / 4;
  for (uint32_t tile = blockIdx.x * kCols; tile < nv; tile += gridDim.x * kCols) {
    const uint32_t i = tile + col;
    uint4 s = make_uint4(0, 0, 0, 0);
    if (i < nv) {
      const uint4* p = reinterpret_cast<const uint4*>(partials) + i;
      uint32_t c = g;
      for (; c + 3 * G < num_clusters; c += 4 * G) {
        const uint4 a0 = __ldcs(p + (c + 0 * G) * row4);
        const uint4 a1 = __ldcs(p + (c + 1 * G) * row4);
        const uint4 a2 = __ldcs(p + (c + 2 * G) * row4);
        const uint4 a3 = __ldcs(p + (c + 3 * G) * row4);
        s.x += a0.x + a1.x + a2.x + a3.x;
        s.y += a0.y + a1.y + a2.y + a3.y;
        s.z += a0.z + a1.z + a2.z + a3.z;
        s.w += a0.w + a1.w + a2.w + a3.w;
      }
      for (; c < num_clusters; c += G) {
        const uint4 a0 = __ldcs(p + c * row4);
        s.x += a0.x;
        s.y += a0.y;
        s.z += a0.z;
        s.w += a0.w;
      }
    }
    if (G > 1) {
      part[g][col] = s;
      __syncthreads();
      if (g == 0) {
#pragma unroll
        for (int h = 1; h < G; ++h) {
          const uint4 o = part[h][col];
          s.x += o.x;
          s.y += o.y;
          s.z += o.z;
          s.w += o.w;
        }
      }
      __syncthreads();  // part is rewritten by the next tile
    }
    if (g == 0 && i < nv) {
      const uint32_t b = 4 * i;
      if (bins_vec_ok && b + 3 < num_bins) {
        reinterpret_cast<uint4*>(bins)[i] = s;
      } else {
        if (b + 0 < num_bins) bins[b + 0] = s.x;
        if (b + 1 < num_bins) bins[b + 1] = s.y;
        if (b + 2 < num_bins) bins[b + 2] = s.z;
        if (b + 3 < num_bins) bins[b + 3] = s.w;
      }
      if (hot_word) {
        // Bins past num_bins are row padding (always zero) and never qualify.
        const uint32_t c4[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c4[q] >= hot_min && b + q < num_bins)
            *reinterpret_cast<volatile unsigned long long*>(hot_word) =
                (static_cast<unsigned long long>(seq) << 32) | (b + q);
      }
    }
  }
}

// Comparison point ("Distributed Shared Memory", section "When it beats
// global atomics"): one global atomic per in-range key.
__global__ void __launch_bounds__(512) global_atomic_hist_kernel(const int32_t* __restrict__ keys,
                                                                 int64_t n, uint32_t head,
                                                                 uint32_t num_bins,
                                                                 uint32_t* __restrict__ bins) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t nvec = (n - head) >> 2;
  const int4* vec = reinterpret_cast<const int4*>(keys + head);
  for (int64_t i = tid; i < nvec; i += nthreads) {
    const int4 v = ld_stream_v4(vec + i);
    if (static_cast<uint32_t>(v.x) < num_bins) atomicAdd(bins + v.x, 1u);
    if (static_cast<uint32_t>(v.y) < num_bins) atomicAdd(bins + v.y, 1u);
    if (static_cast<uint32_t>(v.z) < num_bins) atomicAdd(bins + v.z, 1u);
    if (static_cast<uint32_t>(v.w) < num_bins) atomicAdd(bins + v.w, 1u);
  }
  // head keys [0, head) and tail keys [head + 4*nvec, n)
  const int64_t tail0 = head + 4 * nvec;
  const int64_t leftover = static_cast<int64_t>(head) + (n - tail0);
  if (tid < leftover) {
    const int32_t k = keys[tid < head ? tid : tail0 + (tid - head)];
    if (static_cast<uint32_t>(k) < num_bins) atomicAdd(bins + k, 1u);
  }
}

// Work-free control ("CREDIT", section on the profitability model): the same
// grid, cluster shape and dynamic shared memory as a cluster histogram
// launch, zeroing its slice and passing the two cluster barriers, but
// streaming no keys.  Its time is the launch, residency and synchronisation
// cost a cluster shape pays before doing any work.
__global__ void __launch_bounds__(1024, 1) cluster_control_kernel(uint32_t S, uint32_t* sink) {
  extern __shared__ __align__(16) uint32_t slice[];
  for (uint32_t i = threadIdx.x; i < S; i += blockDim.x) slice[i] = 0;
  cluster_barrier();
  cluster_barrier();
  if (threadIdx.x == 0 && slice[0] != 0) sink[0] = slice[0];
}

template <bool kAggregate>
void* cluster_kernel_ptr() {
  return reinterpret_cast<void*>(&cluster_hist_kernel<kAggregate>);
}

void* cluster_kernel(int aggregate) {
  return aggregate ? cluster_kernel_ptr<true>() : cluster_kernel_ptr<false>();
}

}  // namespace

cudaError_t prepare_cluster_kernel(int aggregate, int smem_bytes) {
  const void* fn = cluster_kernel(aggregate);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

cudaError_t launch_cluster_control(const dsmem_hist_plan_t& plan, uint32_t* sink,
                                   cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(&cluster_control_kernel);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       plan.smem_bytes);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.num_clusters) * plan.cluster_size, 1, 1);
  cfg.blockDim = dim3(plan.block_threads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cluster_control_kernel, static_cast<uint32_t>(plan.bins_per_cta),
                            sink);
}

cudaError_t query_max_active_clusters(int aggregate, int cluster_size, int block_threads,
                                      int smem_bytes, int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster_size, 1, 1);
  cfg.blockDim = dim3(block_threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, cluster_kernel(aggregate), &cfg);
}

// Largest cluster that can be co-scheduled for the direct kernel with this
// block size and dynamic shared memory (non-portable sizes allowed).
cudaError_t query_max_potential_cluster_size(int aggregate, int block_threads, int smem_bytes,
                                             int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16, 1, 1);
  cfg.blockDim = dim3(block_threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  return cudaOccupancyMaxPotentialClusterSize(out, cluster_kernel(aggregate), &cfg);
}

cudaError_t launch_cluster_hist(const dsmem_hist_plan_t& plan, const ClusterHistArgs& args,
                                cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.num_clusters) * plan.cluster_size, 1, 1);
  cfg.blockDim = dim3(plan.block_threads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (plan.aggregate) return cudaLaunchKernelEx(&cfg, cluster_hist_kernel<true>, args);
  return cudaLaunchKernelEx(&cfg, cluster_hist_kernel<false>, args);
}

cudaError_t launch_reduce_partials(const uint32_t* partials, uint64_t stride,
                                   uint32_t num_clusters, uint32_t num_bins, uint32_t* bins,
                                   cudaStream_t stream, uint32_t hot_min,
                                   unsigned long long* hot_word, uint32_t* seq_word, uint32_t seq) {
  if (hot_min == 0 || !seq_word) hot_word = nullptr;
  const uint32_t nv = (num_bins + 3) / 4;
  const int vec_ok = (reinterpret_cast<uintptr_t>(bins) & 15u) == 0;
  // Row groups: the largest power of two <= min(16, C / 2), so each group
  // sums at least two rows with both loads in flight (16 rows in 16 groups
  // took 2.4 us longer than in 8).
  int G = 1;
  while (G < 16 && static_cast<uint32_t>(4 * G) <= num_clusters) G *= 2;
  uint32_t blocks = (nv + (256 / G) - 1) / (256 / G);
  if (blocks > 8192) blocks = 8192;
  switch (G) {
    case 16:
      reduce_partials_kernel<16><<<blocks, 256, 0, stream>>>(partials, stride, num_clusters, num_bins, bins, vec_ok, hot_min, hot_word, seq_word, seq);
      break;
    case 8:
      reduce_partials_kernel<8><<<blocks, 256, 0, stream>>>(partials, stride, num_clusters, num_bins, bins, vec_ok, hot_min, hot_word, seq_word, seq);
      break;
    case 4:
      reduce_partials_kernel<4><<<blocks, 256, 0, stream>>>(partials, stride, num_clusters, num_bins, bins, vec_ok, hot_min, hot_word, seq_word, seq);
      break;
    case 2:
      reduce_partials_kernel<2><<<blocks, 256, 0, stream>>>(partials, stride, num_clusters, num_bins, bins, vec_ok, hot_min, hot_word, seq_word, seq);
      break;
    default:
      reduce_partials_kernel<1><<<blocks, 256, 0, stream>>>(partials, stride, num_clusters, num_bins, bins, vec_ok, hot_min, hot_word, seq_word, seq);
  }
  return cudaGetLastError();
}

cudaError_t launch_global_atomic(const int32_t* keys, int64_t n, uint32_t num_bins,
                                 uint32_t* bins, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(bins, 0, sizeof(uint32_t) * num_bins, stream);
  if (e != cudaSuccess || n == 0) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const uint32_t head_align =
      static_cast<uint32_t>(((16u - (reinterpret_cast<uintptr_t>(keys) & 15u)) & 15u) / 4u);
  const uint32_t head = n < head_align ? static_cast<uint32_t>(n) : head_align;
  const int64_t nvec = (n - head) / 4;
  int64_t blocks = (nvec + 511) / 512;
  const int64_t cap = static_cast<int64_t>(sms) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  global_atomic_hist_kernel<<<static_cast<unsigned>(blocks), 512, 0, stream>>>(keys, n, head,
                                                                                num_bins, bins);
  return cudaGetLastError();
}

}  // namespace dsmh
