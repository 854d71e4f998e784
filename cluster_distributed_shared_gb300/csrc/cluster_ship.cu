// Cluster histogram with owner-routed key shipping, written for sm_103a.
//
// Same result and the same ownership as the page's cluster histogram
// ("Distributed Shared Memory", section "The cluster histogram"): bin
// `base + o*S + l` is counter `l` of CTA `o` of the cluster, every key
// becomes exactly one increment of its owner's shared-memory counter, and
// cluster barriers bracket the phase in which CTAs write each other's shared
// memory.  What changes is how an increment reaches its owner.  On GB300 a
// remote `red.shared::cluster` sustains ~0.33 operations per clock per SM
// while a local shared-memory atomic sustains ~12, and coalesced 16-byte
// remote stores move ~19 bytes per clock per SM.  So each key travels as a
// 16-bit local index inside 16-byte vectors, and its owner applies a local
// `red.shared` (the "push compact data to its owner, combine locally" idea of
// "CREDIT", section on the clustered reduction-reuse schedule).
//
// Per CTA (1024 threads, 32 warps), keys are processed in rounds of
// 1024 * kKpt keys.
//   A  partition (all warps): sub-bucket (owner o, lane L) is a contiguous
//      run of qs 16-bit entries; consecutive sub-buckets are 2*qs + 4 bytes
//      apart, a 4-byte skew that puts lane L's next entry in bank
//      (L + fill/2) mod 32, so a warp's 32 stores spread over the banks.  Its
//      cursor holds the shared-memory byte address of its next entry, so one
//      local `atom.add 2` both reserves the slot and yields the store address;
//      the 32 lanes of a warp touch 32 different cursors (one bank each).  A
//      key whose sub-bucket is full goes to its owner with a remote red
//      (exact, slow, only on skewed rounds).  A warp tile of 128 equal keys
//      is counted with one red of 128 (pre-aggregation of runs).
//   After a CTA barrier:
//   B  `ns` shipper warps per owner close its 32 sub-buckets (lane = sub-
//      bucket): pad the last vector with the index of one of 32 dummy
//      counters after the slice, scan the vector counts, and copy every
//      vector (four 32-bit shared loads, one st.shared::cluster.v4) into the
//      owner's inbox slot for this sender, plus one vector count; the CTA's
//      own keys go to its own inbox the same way.
//   D  the other warps apply the previous round's inbox (complete since the
//      last cluster barrier wait) with one local red per entry.
//   After a CTA barrier, receivers arrive on the cluster barrier (relaxed:
//   they published no remote writes), every warp partitions the next round,
//   shippers arrive (release: their inbox stores), and all wait.
// Inboxes are double-buffered: a sender writes round r into buffer r%2 only
// after waiting on the barrier of round r-1, which every owner arrives on
// only after it has applied round r-2 from that buffer.

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace dsmh {
namespace {

using namespace ptx;

struct Ctx {
  uint32_t base, range;   // current pass: first bin, bins in the pass
  uint32_t S, lgS, P, lane;
  uint32_t owner_bytes;   // bytes between sub-buckets (o, L) and (o + 1, L): 32*(2*qs + 4)
  uint64_t magic;
  uint32_t slice;         // shared::cta address of u32[S + 32]
  uint32_t cursor_lane;   // &cursor[0*32 + lane]
  uint32_t limit_lane;    // end of sub-bucket (0, lane)
};

__device__ __forceinline__ void owner_local(uint32_t rel, const Ctx& c, uint32_t& o,
                                            uint32_t& loc, bool pow2) {
  if (pow2) {
    o = rel >> c.lgS;
    loc = rel & (c.S - 1u);
  } else {
    o = static_cast<uint32_t>((static_cast<uint64_t>(rel) * c.magic) >> 40);
    loc = rel - o * c.S;
  }
}

// One key of A, fused into one predicated PTX block: if `rel < range`,
// reserve the next slot of sub-bucket (owner, lane) (`atom.add` on its
// cursor returns the slot's byte address) and, if that address is below the
// sub-bucket's end, store the 16-bit local index there.  Returns 1 when the key is valid
// but its sub-bucket is full (the caller increments the owner directly).
__device__ __forceinline__ uint32_t place_key(uint32_t rel, uint32_t range, uint32_t cursor_addr,
                                              uint32_t stride, uint32_t limit, uint32_t loc,
                                              uint32_t& ea) {
  uint32_t spill;
  asm volatile(
      "{\n\t.reg .pred pv, pf, ps;\n\t"
      "setp.lt.u32 pv, %2, %3;\n\t"
      "mov.u32 %0, 0;\n\t"
      "@pv atom.shared.add.u32 %0, [%4], %5;\n\t"
      "setp.lt.and.u32 pf, %0, %6, pv;\n\t"
      "setp.ge.and.u32 ps, %0, %6, pv;\n\t"
      "@pf st.shared.u16 [%0], %7;\n\t"
      "selp.u32 %1, 1, 0, ps;\n\t}"
      : "=&r"(ea), "=r"(spill)
      : "r"(rel), "r"(range), "r"(cursor_addr), "r"(stride), "r"(limit), "h"(static_cast<uint16_t>(loc)));
  return spill;
}

// A: partition one warp tile (four keys per lane).
template <bool kPow2>
__device__ __forceinline__ void partition_vec(const int4& v, const Ctx& c) {
  const bool eq4 = (v.x == v.y) & (v.y == v.z) & (v.z == v.w);
  const int32_t k0 = __shfl_sync(0xffffffffu, v.x, 0);
  if (__all_sync(0xffffffffu, eq4 & (v.x == k0))) {
    const uint32_t rel = static_cast<uint32_t>(k0) - c.base;
    if (c.lane == 0 && rel < c.range) {
      uint32_t o, loc;
      owner_local(rel, c, o, loc, kPow2);
      red_add_cluster(map_rank(c.slice + 4u * loc, o), 128u);
    }
    return;
  }
  const int32_t keys[4] = {v.x, v.y, v.z, v.w};
  uint32_t rel[4], own[4], loc[4], ea[4], spill = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    rel[k] = static_cast<uint32_t>(keys[k]) - c.base;
    owner_local(rel[k], c, own[k], loc[k], kPow2);
    spill |= place_key(rel[k], c.range, c.cursor_lane + 128u * own[k], 2u,
                       c.limit_lane + c.owner_bytes * own[k], loc[k], ea[k]) << k;
  }
  if (__any_sync(0xffffffffu, spill != 0)) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (spill & (1u << k)) red_add_cluster(map_rank(c.slice + 4u * loc[k], own[k]), 1u);
  }
}

// Applies the 8 entries of one received vector (16-bit local indices; padding
// entries index the dummy counters after the slice).
__device__ __forceinline__ void apply_vector(uint32_t slice, const uint4& x) {
  red_add_local(slice + 4u * (x.x & 0xFFFFu), 1u);
  red_add_local(slice + 4u * (x.x >> 16), 1u);
  red_add_local(slice + 4u * (x.y & 0xFFFFu), 1u);
  red_add_local(slice + 4u * (x.y >> 16), 1u);
  red_add_local(slice + 4u * (x.z & 0xFFFFu), 1u);
  red_add_local(slice + 4u * (x.z >> 16), 1u);
  red_add_local(slice + 4u * (x.w & 0xFFFFu), 1u);
  red_add_local(slice + 4u * (x.w >> 16), 1u);
}

template <int kKpt>
__device__ __forceinline__ void load_round(int4 (&v)[kKpt / 4], const int4* vec, int64_t ntiles,
                                           int64_t t0, int64_t nwarps) {
#pragma unroll
  for (int u = 0; u < kKpt / 4; ++u) {
    const int64_t t = t0 + u * nwarps;
    v[u] = t < ntiles ? ld_stream_v4(vec + (t << 5)) : make_int4(-1, -1, -1, -1);
  }
}

template <int kKpt, bool kPow2>
__global__ void __launch_bounds__(1024, 1) cluster_ship_kernel(const ClusterHistArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  Ctx c;
  c.P = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  c.lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  c.S = a.S;
  c.lgS = 31u - __clz(a.S);
  c.magic = a.magic;
  const uint32_t P = c.P;
  const uint32_t qs = 8u * a.sub_vectors;   // entries per sub-bucket
  const uint32_t sb = 2u * qs + 4u;         // bytes per sub-bucket (4-byte skew)
  const uint32_t cap_vecs = 4u * qs;        // inbox vectors per sender slot
  c.owner_bytes = 32u * sb;
  const uint32_t cid = cluster_id_x();

  // Layout (must match ship_staging_bytes): slice u32[S + 32], cursors
  // u32[P*32], headers u32[2][16], sub-buckets [P][32] of sb bytes (16-byte
  // padded in total), inboxes uint4[2][P][4*qs].
  const uint32_t sbase = smem_u32(smem);
  c.slice = sbase;
  const uint32_t cursor0 = sbase + 4u * (a.S + 32u);
  const uint32_t header0 = cursor0 + 4u * 32u * P;
  const uint32_t rows0 = header0 + 4u * 32u;
  const uint32_t inbox0 = rows0 + ((P * c.owner_bytes + 15u) & ~15u);
  c.cursor_lane = cursor0 + 4u * c.lane;
  c.limit_lane = rows0 + c.lane * sb + 2u * qs;
  uint32_t* cursor = reinterpret_cast<uint32_t*>(smem + (cursor0 - sbase));
  const uint32_t* header = reinterpret_cast<const uint32_t*>(smem + (header0 - sbase));

  // Key stream: warp tiles of 32 vectors, kKpt/4 tiles per warp per round.
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * 32;
  const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * 32 + warp;
  const int64_t ntiles = ((a.n - a.head) >> 2) >> 5;
  const int4* vec = reinterpret_cast<const int4*>(a.keys + a.head) + c.lane;
  constexpr int kTiles = kKpt / 4;
  const int64_t per_round = nwarps * kTiles;
  const uint32_t rounds = static_cast<uint32_t>((ntiles + per_round - 1) / per_round);

  // Roles: ns shipper warps per owner, the rest receive.
  const uint32_t ns = P >= 16 ? 1u : 16u / P;
  const bool shipper = warp < ns * P;
  const uint32_t so = shipper ? warp / ns : 0u;      // owner shipped by this warp
  const uint32_t sh = shipper ? warp % ns : 0u;      // vector phase
  const uint32_t nrecv = 32u - ns * P;
  const uint32_t rw = shipper ? 0u : warp - ns * P;
  const uint32_t dslot = rw % P;                     // sender slot applied by this warp
  const uint32_t dq = rw / P;
  const uint32_t dnw = shipper ? 1u : (nrecv - 1u - dslot) / P + 1u;

  for (uint32_t pass = 0; pass < a.passes; ++pass) {
    c.base = pass * P * c.S;
    const uint32_t left = a.num_bins - c.base;
    c.range = left < P * c.S ? left : P * c.S;

    uint4* s4 = reinterpret_cast<uint4*>(smem);
    for (uint32_t i = threadIdx.x; i < (c.S + 32u) / 4; i += blockDim.x) s4[i] = make_uint4(0, 0, 0, 0);
    for (uint32_t i = threadIdx.x; i < 32u * P; i += blockDim.x) cursor[i] = rows0 + i * sb;
    cluster_barrier();  // every slice zeroed before any increment

    int4 cur[kTiles];
    if (rounds > 0) {
      load_round<kKpt>(cur, vec, ntiles, gwarp, nwarps);
#pragma unroll
      for (int u = 0; u < kTiles; ++u) partition_vec<kPow2>(cur[u], c);
    }
    for (uint32_t r = 0; r < rounds; ++r) {
      const bool more = r + 1 < rounds;
      if (more) load_round<kKpt>(cur, vec, ntiles, gwarp + static_cast<int64_t>(r + 1) * per_round, nwarps);
      __syncthreads();  // partition of round r complete
      const uint32_t buf = r & 1u;
      if (shipper) {
        // B: close owner so's sub-bucket `lane`, ship vectors j = sh (mod ns).
        const uint32_t sub = so * 32u + c.lane;
        const uint32_t col = rows0 + sub * sb;
        const uint32_t fill = (cursor[sub] - col) >> 1;
        const uint32_t cnt = fill < qs ? fill : qs;
        const uint32_t nv = (cnt + 7u) >> 3;
        if (sh == 0)  // pad the last vector with this lane's dummy counter
          for (uint32_t p = cnt; p < 8u * nv; ++p)
            st_shared_u16(col + 2u * p, static_cast<uint16_t>(c.S + c.lane));
        if (ns > 1) named_barrier(1, 32u * ns * P);  // cursors read, padding written
        if (sh == 0) cursor[sub] = col;
        uint32_t incl = nv;
#pragma unroll
        for (uint32_t d = 1; d < 32; d <<= 1) {
          const uint32_t t = __shfl_up_sync(0xffffffffu, incl, d);
          if (c.lane >= d) incl += t;
        }
        const uint32_t dst = inbox0 + 16u * ((buf * P + rank) * cap_vecs + incl - nv);
        for (uint32_t j = sh; j < nv; j += ns) {
          const uint32_t a4 = col + 16u * j;  // 4-byte aligned
          uint4 x;
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x.x) : "r"(a4));
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x.y) : "r"(a4 + 4u));
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x.z) : "r"(a4 + 8u));
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x.w) : "r"(a4 + 12u));
          st_cluster_v4(map_rank(dst + 16u * j, so), x);
        }
        if (sh == 0 && c.lane == 31)
          st_cluster_u32(map_rank(header0 + 4u * (buf * 16u + rank), so), incl);
      } else if (r > 0) {
        // D: apply the previous round's inbox from sender slot `dslot`.
        const uint32_t pb = buf ^ 1u;
        const uint32_t nvec = header[pb * 16u + dslot];
        const uint32_t src0 = inbox0 + 16u * ((pb * P + dslot) * cap_vecs);
        for (uint32_t v = dq * 32u + c.lane; v < nvec; v += dnw * 32u)
          apply_vector(c.slice, ld_shared_v4(src0 + 16u * v));
      }
      __syncthreads();  // rows read and cursors reset before the next partition
      if (!shipper) cluster_arrive_relaxed();
      if (more) {
#pragma unroll
        for (int u = 0; u < kTiles; ++u) partition_vec<kPow2>(cur[u], c);
      }
      if (shipper) cluster_arrive();
      cluster_wait();  // round r's inboxes complete everywhere
    }
    if (rounds > 0 && !shipper) {
      const uint32_t pb = (rounds - 1u) & 1u;
      const uint32_t nvec = header[pb * 16u + dslot];
      const uint32_t src0 = inbox0 + 16u * ((pb * P + dslot) * cap_vecs);
      for (uint32_t v = dq * 32u + c.lane; v < nvec; v += dnw * 32u)
        apply_vector(c.slice, ld_shared_v4(src0 + 16u * v));
    }

    // Ragged keys (unaligned head, partial tile, tail): the grid's last warp,
    // straight to the owners.
    if (gwarp == nwarps - 1) {
      const int64_t after = a.head + (ntiles << 7);
      const int64_t leftover = static_cast<int64_t>(a.head) + (a.n - after);
      for (int64_t j = c.lane; j < leftover; j += 32) {
        const int32_t key = a.keys[j < a.head ? j : after + (j - a.head)];
        const uint32_t rel = static_cast<uint32_t>(key) - c.base;
        if (rel < c.range) {
          uint32_t o, loc;
          owner_local(rel, c, o, loc, kPow2);
          red_add_cluster(map_rank(c.slice + 4u * loc, o), 1u);
        }
      }
    }

    cluster_barrier();  // every increment has landed; only own memory after this

    const uint32_t first = c.base + rank * c.S;
    if (c.range > rank * c.S) {
      const uint32_t cnt = c.range - rank * c.S < c.S ? c.range - rank * c.S : c.S;
      uint4* dst = reinterpret_cast<uint4*>(a.partials + static_cast<size_t>(cid) * a.stride + first);
      const uint32_t nv = (cnt + 3) / 4;
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
    if (pass + 1 < a.passes) __syncthreads();
  }
}

template <int kKpt, bool kPow2>
void* kernel_ptr_t() {
  return reinterpret_cast<void*>(&cluster_ship_kernel<kKpt, kPow2>);
}

void* ship_kernel_ptr(int kpt, bool pow2) {
  if (kpt == 8) return pow2 ? kernel_ptr_t<8, true>() : kernel_ptr_t<8, false>();
  return pow2 ? kernel_ptr_t<4, true>() : kernel_ptr_t<4, false>();
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

}  // namespace

cudaError_t prepare_ship_kernel(int kpt, int smem_bytes) {
  for (int p2 = 0; p2 < 2; ++p2) {
    const void* fn = ship_kernel_ptr(kpt, p2 != 0);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t query_ship_active_clusters(int kpt, int cluster_size, int smem_bytes, int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster_size, 1, 1);
  cfg.blockDim = dim3(1024, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, ship_kernel_ptr(kpt, true), &cfg);
}

cudaError_t launch_cluster_ship(const dsmem_hist_plan_t& plan, const ClusterHistArgs& args,
                                cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.num_clusters) * plan.cluster_size, 1, 1);
  cfg.blockDim = dim3(1024, 1, 1);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool p2 = is_pow2(plan.bins_per_cta);
  if (plan.keys_per_thread == 8)
    return p2 ? cudaLaunchKernelEx(&cfg, cluster_ship_kernel<8, true>, args)
              : cudaLaunchKernelEx(&cfg, cluster_ship_kernel<8, false>, args);
  return p2 ? cudaLaunchKernelEx(&cfg, cluster_ship_kernel<4, true>, args)
            : cudaLaunchKernelEx(&cfg, cluster_ship_kernel<4, false>, args);
}

}  // namespace dsmh
