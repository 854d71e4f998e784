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
// 16-bit local index inside contiguous 16-byte vectors, and its owner applies
// a local `red.shared` (the "push compact data to its owner, combine locally"
// idea of "CREDIT", section on the clustered reduction-reuse schedule).
//
// Per CTA (kShipThreads threads), keys are processed in rounds of
// kShipThreads * kKpt keys.  Round r stages into staging buffer r % 2 with
// cursor set r % 3 and travels in inbox buffer r % 2.
//   Partition.  Owner o's staging block is column-major: rows of 64 bytes,
//     column L (0..31) holding the keys that lane L of any warp routed to o.
//     Cursor (o, L) is the byte address of the column's next free entry, so
//     one local `atom.add 64` both reserves the entry and yields the store
//     address.  The 32 lanes of a warp touch 32 cursors in 32 banks, and
//     their 16-bit stores fall at most two to a bank.  A key whose column is
//     full goes to its owner with a remote red (exact, slow, only on skewed
//     rounds); a key outside the pass's bins meets a cursor row that is
//     always full and is dropped on the same path.  A warp tile of 128 equal
//     keys becomes one remote red of 128, and a warp's two consecutive tiles
//     of one key one red of 256 (pre-aggregation of runs).
//   Ship.  Warps serve owner w mod P: the block's row count is the fullest
//     column's fill, and its rows go out as contiguous 16-byte `st.async`
//     stores into the owner's inbox slot for this sender, then are
//     overwritten with padding entries (column c pads with index S + c, one
//     of 32 never-read counters after the slice).  The row count goes to the
//     owner's header the same way.  Each store's bytes are counted on the
//     owner's mbarrier for that inbox buffer, on which every sender arrives
//     once per round with its byte count (`mbarrier.arrive.expect_tx`).
//   Apply.  Warps wait (bounded) for a round's mbarrier phase, then apply
//     that round's inbox block from sender w mod P: one `dp2a` turns a
//     16-bit entry into its counter's address, one local red increments it.
// In round r every warp applies round r-1, waits (bounded) on the CTA's
// `staged` mbarrier until every warp has partitioned round r, resets the
// cursor set of round r+2, arrives on the cluster barrier, ships round r,
// partitions round r+1 into the other staging buffer, loads the keys of round
// r+2, arrives on `staged`, and waits on the cluster barrier.  No CTA barrier
// ends the round: a warp that has partitioned goes on to apply the next
// round while others still partition, and it only waits for them where it
// reads what they staged.  Since the mbarriers publish the inbox data, the
// cluster barrier is relaxed: it only tells senders that the inbox they are
// about to overwrite has been read, so no warp waits for its remote stores to
// be acknowledged.  A sender writes round r into inbox buffer r%2 only after
// the barrier of round r-1, which every owner arrives on only after it has
// applied round r-2 from that buffer.

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace dsmh {
namespace {

using namespace ptx;

constexpr uint32_t kFullMask = 0xffffffffu;
// Cursor value of the row that collects keys outside the pass's bins: at or
// above every block's end for any number of increments in one round.
constexpr uint32_t kAlwaysFull = 0xFFFF0000u;

struct Ctx {
  uint32_t base, range;   // current pass: first bin, bins in the pass
  uint32_t S, lgS, P, PS; // PS = P * S
  uint32_t lane;
  uint64_t magic;
  uint32_t slice;         // shared::cta address of u32[S + 32]
  uint32_t cur_lane;      // this round's cursor set + 4 * lane
  uint32_t lim0;          // end of owner 0's staging block
  uint32_t blk;           // bytes per owner block: 64 * rows
  uint32_t sink;          // 16-bit store target of keys that are not staged
  uint32_t hot_rel;       // kSkew: in-pass offset of the caller's hot bin (kNoHot: none in this pass)
};

// kSkew instantiation (the caller named a hot bin, see the plan's hot_bin):
// keys of the hot bin are counted per thread in the partition instead of
// being staged, and each warp sends its total to the owner once, at the end
// of the pass.  One bin holding a quarter of the keys otherwise overflows its
// owner's staging columns on every round, and every overflowing key costs a
// remote red (about 0.33 per clock per SM).  The comparison costs about 9%
// more instructions, so the planner leaves it off unless asked.
constexpr uint32_t kNoHot = 0xFFFFFFFFu;

// Owner and local counter of an in-pass offset `rel` < P*S.
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

// Stores a 16-bit entry at `ea` if `ea` is below its block's end `lim`,
// else counts a spill; predicated, without a branch.
__device__ __forceinline__ void stage_entry(uint32_t ea, uint32_t lim, uint32_t loc, uint32_t& spill) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.lt.u32 p, %1, %2;\n\t"
      "@p st.shared.u16 [%1], %3;\n\t"
      "@!p add.u32 %0, %0, 1;\n\t}"
      : "+r"(spill)
      : "r"(ea), "r"(lim), "h"(static_cast<uint16_t>(loc)));
}

// Partition one warp tile (four keys per lane).  All four reservations are
// issued before the first store so their latencies overlap.  kBase0: the
// pass starts at bin 0, so a key is its own in-pass offset.  kRunTest: test
// first whether the tile holds one key (off when the caller already has).
template <bool kPow2, bool kBase0, bool kRunTest, bool kSkew>
__device__ __forceinline__ void partition_tile(const int4& v, const Ctx& c, uint32_t& hot_keys) {
  if (kRunTest && __all_sync(kFullMask, v.x == v.w)) {  // rare on most inputs: then test the whole tile
    const int32_t k0 = __shfl_sync(kFullMask, v.x, 0);
    const bool eq4 = (v.x == v.y) & (v.y == v.z) & (v.z == v.w);
    if (__all_sync(kFullMask, eq4 & (v.x == k0))) {
      const uint32_t rel = static_cast<uint32_t>(k0) - (kBase0 ? 0u : c.base);
      if (c.lane == 0 && rel < c.range) {
        uint32_t o, loc;
        owner_local(rel, c, o, loc, kPow2);
        red_add_cluster(map_rank(c.slice + 4u * loc, o), 128u);
      }
      return;
    }
  }
  const int32_t keys[4] = {v.x, v.y, v.z, v.w};
  uint32_t own[4], loc[4], ea[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    // Offsets at or past P*S clamp to owner P, the always-full cursor row.
    if constexpr (kSkew) {
      // Compare the clamped offset: it is at most P*S, while hot_rel is either
      // below the pass's range or kNoHot, so no key of a pass without the hot
      // bin can match (the unclamped offset of key base - 1 equals kNoHot).
      const uint32_t rel = min(static_cast<uint32_t>(keys[k]) - (kBase0 ? 0u : c.base), c.PS);
      const bool hot = rel == c.hot_rel;
      hot_keys += hot ? 1u : 0u;
      owner_local(rel, c, own[k], loc[k], kPow2);
      // A hot key reserves nothing; its 16-bit store goes to this lane's sink.
      ea[k] = hot ? c.sink : atom_add_local(c.cur_lane + (own[k] << 7), 64u);
    } else {
      const uint32_t rel = min(static_cast<uint32_t>(keys[k]) - (kBase0 ? 0u : c.base), c.PS);
      owner_local(rel, c, own[k], loc[k], kPow2);
      ea[k] = atom_add_local(c.cur_lane + (own[k] << 7), 64u);
    }
  }
  uint32_t spill = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) stage_entry(ea[k], c.lim0 + own[k] * c.blk, loc[k], spill);
  if (__any_sync(kFullMask, spill != 0)) {
    // Rare: redo the test per key and send each spilled in-range key to its owner.
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t rel = static_cast<uint32_t>(keys[k]) - (kBase0 ? 0u : c.base);
      if (ea[k] >= c.lim0 + own[k] * c.blk && rel < c.range)
        red_add_cluster(map_rank(c.slice + 4u * loc[k], own[k]), 1u);
    }
  }
}

template <int kTiles, bool kPow2, bool kSkew>
__device__ __forceinline__ void partition_round(const int4 (&v)[kTiles], const Ctx& c,
                                                uint32_t& hot_keys) {
  static_assert(kTiles == 1 || kTiles == 2, "one or two tiles per warp and round");
  // The warp's tiles are consecutive in the input.  The first tile's run test
  // runs here: a run tile followed by a run tile of the same key (a run of
  // 256) becomes one remote red, a lone run tile one red of 128.
  if (__all_sync(kFullMask, v[0].x == v[0].w)) {  // rare on most inputs
    const int32_t k0 = __shfl_sync(kFullMask, v[0].x, 0);
    const bool eq0 = (v[0].x == v[0].y) & (v[0].y == v[0].z) & (v[0].z == v[0].w) & (v[0].x == k0);
    if (__all_sync(kFullMask, eq0)) {
      const int4& w = v[kTiles - 1];
      const bool eq1 = (w.x == k0) & (w.y == k0) & (w.z == k0) & (w.w == k0);
      const bool both = kTiles == 2 && __all_sync(kFullMask, eq1);
      const uint32_t rel = static_cast<uint32_t>(k0) - c.base;
      if (c.lane == 0 && rel < c.range) {
        uint32_t o, loc;
        owner_local(rel, c, o, loc, kPow2);
        red_add_cluster(map_rank(c.slice + 4u * loc, o), both ? 256u : 128u);
      }
      if (kTiles == 1 || both) return;
      if (c.base == 0)
        partition_tile<kPow2, true, true, kSkew>(w, c, hot_keys);
      else
        partition_tile<kPow2, false, true, kSkew>(w, c, hot_keys);
      return;
    }
  }
  // Past here the first tile is known not to be a run.
  if (c.base == 0) {
    partition_tile<kPow2, true, false, kSkew>(v[0], c, hot_keys);
#pragma unroll
    for (int u = 1; u < kTiles; ++u) partition_tile<kPow2, true, true, kSkew>(v[u], c, hot_keys);
  } else {
    partition_tile<kPow2, false, false, kSkew>(v[0], c, hot_keys);
#pragma unroll
    for (int u = 1; u < kTiles; ++u) partition_tile<kPow2, false, true, kSkew>(v[u], c, hot_keys);
  }
}

// Applies the 8 entries of one received vector.  dp2a.lo with b = 4 gives
// slice + 4 * low half, with b = 0x400 slice + 4 * high half.
__device__ __forceinline__ void apply_vector(uint32_t slice, const uint4& x) {
  red_add_local(__dp2a_lo(x.x, 4u, slice), 1u);
  red_add_local(__dp2a_lo(x.x, 0x400u, slice), 1u);
  red_add_local(__dp2a_lo(x.y, 4u, slice), 1u);
  red_add_local(__dp2a_lo(x.y, 0x400u, slice), 1u);
  red_add_local(__dp2a_lo(x.z, 4u, slice), 1u);
  red_add_local(__dp2a_lo(x.z, 0x400u, slice), 1u);
  red_add_local(__dp2a_lo(x.w, 4u, slice), 1u);
  red_add_local(__dp2a_lo(x.w, 0x400u, slice), 1u);
}

__device__ uint32_t g_ship_status;  // bit 0: a bounded wait gave up (until read and cleared)

// Waits for phase `parity` of an mbarrier (an inbox buffer's, or the CTA's
// `staged` one), at most `limit` cycles (by default ~1e8, about 50 ms).  On a
// timeout the device status word and the call's host-mapped word (if any)
// record it, this CTA's shared flag at `gave_up` is set, and the caller skips
// the inbox buffer (or goes on without the other warps); once a wait of this
// CTA has timed out, its later waits in the same launch give up after one
// probe.  Later launches start with the flag clear.
__device__ __forceinline__ bool wait_mbar(uint32_t mbar, uint32_t parity, uint32_t gave_up,
                                           long long limit, uint32_t* status) {
  if (mbar_try_wait(mbar, parity)) return true;
  if (ld_shared_u32(gave_up) != 0u) return false;
  const long long deadline = clock64() + limit;
  while (clock64() < deadline)
    if (mbar_try_wait(mbar, parity)) return true;
  st_shared_u32(gave_up, 1u);
  atomicOr(&g_ship_status, 1u);
  if (status) st_volatile_u32(status, 1u);
  return false;
}

__device__ __forceinline__ uint4 pad_vector(uint32_t pad0) {
  return make_uint4(pad0, pad0 + 0x00020002u, pad0 + 0x00040004u, pad0 + 0x00060006u);
}

// Reports, from the mop-up kernel's first CTA (which starts when the cluster
// kernel has finished), the helper's share of the tiles at which the helper
// and the clusters would have finished together.  rho is how far the
// helper's pace carried it through its range by now: the ratio of the times
// since the helper started when it has finished already, else the fraction
// of its tiles claimed.  With helper share f the target is
// rho f / (rho f + 1 - f).  (Scalars by
// value: a reference to the kernel's arguments would move them to local
// memory.)
__device__ __forceinline__ void report_helper_share(const uint32_t* queue, uint32_t helper_tiles,
                                                 uint32_t cluster_tiles, unsigned long long* report,
                                                 uint32_t seq, uint32_t claimed) {
  const unsigned long long* times = reinterpret_cast<const unsigned long long*>(queue + 2);
  const unsigned long long now = global_timer_ns();
  const unsigned long long t0 = ld_volatile_u64(times), th = ld_volatile_u64(times + 1);
  if (helper_tiles == 0 || cluster_tiles == 0 || t0 == 0 || now <= t0) return;
  const float H = static_cast<float>(helper_tiles), C = static_cast<float>(cluster_tiles);
  const float rho = th > t0 && th <= now ? static_cast<float>(now - t0) / static_cast<float>(th - t0)
                                         : fminf(static_cast<float>(claimed), H) / H;
  const float f = H / (H + C);
  const float target = rho * f / (rho * f + 1.0f - f);
  st_volatile_u64(report, (static_cast<unsigned long long>(seq) << 32) | __float_as_uint(target));
}

// Loads a warp's consecutive tiles t0, t0 + 1, ... of a round; tiles past
// the end read as keys -1 (outside every pass).  Only the last round can
// reach past the end.
template <int kKpt>
__device__ __forceinline__ void load_round(int4 (&v)[kKpt / 4], const int4* vec, uint32_t ntiles,
                                           uint32_t t0, bool last) {
  if (!last) {
#pragma unroll
    for (int u = 0; u < kKpt / 4; ++u) v[u] = ld_stream_v4(vec + static_cast<size_t>(t0 + u) * 32u);
    return;
  }
#pragma unroll
  for (int u = 0; u < kKpt / 4; ++u) {
    const uint32_t t = t0 + u;
    v[u] = t < ntiles ? ld_stream_v4(vec + static_cast<size_t>(t) * 32u) : make_int4(-1, -1, -1, -1);
  }
}

template <int kKpt, bool kPow2, bool kSkew>
__global__ void __launch_bounds__(kShipThreads, 1) cluster_ship_kernel(const ClusterHistArgs a) {
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
  c.PS = P * a.S;
  const uint32_t qs = a.sub_vectors;  // rows of an owner block
  c.blk = 64u * qs;
  const uint32_t cid = cluster_id_x();

  // Layout (must match ship_staging_bytes): slice u32[S + 32], cursors
  // u32[3][P + 1][32], headers u32[2][16], sink u16[32], two inbox
  // mbarriers, a timeout flag and the `staged` mbarrier (256 bytes with
  // padding), staging u16[2][P][qs][32], inboxes
  // u16[2][P][qs][32].  Round r partitions into staging buffer r % 2 with
  // cursor set r % 3, and its blocks travel in inbox buffer r % 2.
  const uint32_t sbase = smem_u32(smem);
  c.slice = sbase;
  const uint32_t set_words = 32u * (P + 1u);
  const uint32_t set_bytes = 4u * set_words;
  const uint32_t cur0 = sbase + 4u * (a.S + 32u);
  const uint32_t header0 = cur0 + 3u * set_bytes;
  c.sink = header0 + 128u + 2u * c.lane;
  const uint32_t full0 = header0 + 192u;  // mbarriers full[2]: inbox buffer complete
  // A bounded wait of this CTA timed out in this launch (cleared below, before
  // the first cluster barrier, so before any wait).
  const uint32_t gave_up = header0 + 208u;
  const uint32_t staged = header0 + 216u;  // mbarrier: every warp partitioned the next round
  uint32_t hot_keys = 0;  // kSkew: keys of the hot bin this thread counted in this pass
  const uint32_t stage0 = header0 + 256u;
  const uint32_t buf_bytes = P * c.blk;   // one staging or inbox buffer
  const uint32_t inbox0 = stage0 + 2u * buf_bytes;

  // Key stream: warp tiles of 32 vectors (tile t = vectors 32t .. 32t+31),
  // kKpt/4 consecutive tiles per warp per round; tile indices fit 32 bits with room for
  // three rounds on top (the library keeps n below 2^38 for this kernel).
  constexpr uint32_t kWarps = kShipThreads / 32;
  const uint32_t nwarps = gridDim.x * kWarps;
  const uint32_t gwarp = blockIdx.x * kWarps + warp;
  const uint32_t ntiles = static_cast<uint32_t>(((a.n - a.head) >> 2) >> 5);
  const int4* vec = reinterpret_cast<const int4*>(a.keys + a.head) + c.lane;
  constexpr int kTiles = kKpt / 4;
  const uint32_t per_round = nwarps * kTiles;
  const uint32_t wtile0 = gwarp * kTiles;  // this warp's first tile of round 0
  const uint32_t rounds = static_cast<uint32_t>((static_cast<uint64_t>(ntiles) + per_round - 1) / per_round);

  // Ship and apply: warp w serves owner (and sender) w mod P, as member sg of
  // the sng warps that do; lane l of member sg starts at vector 32*sg + l of
  // a block and steps by 32*sng vectors.  Addresses below are for buffer 0;
  // buffer 1 adds buf_bytes.
  const uint32_t so = warp % P;
  const uint32_t sg = warp / P;
  const uint32_t sng = (kWarps - 1u - so) / P + 1u;
  const uint32_t step = 512u * sng;                          // bytes between a lane's vectors
  const uint32_t vofs = 16u * (32u * sg + c.lane);           // this lane's first vector
  const uint32_t top0 = stage0 + so * c.blk;                 // owner so's staging block
  const uint32_t fill_rd = cur0 + 4u * (32u * so + c.lane);  // cursor (so, lane) of set 0
  const uint32_t hdr_out = map_rank(header0 + 4u * rank, so);
  const uint32_t dst0 = map_rank(inbox0 + rank * c.blk, so) + vofs;
  const uint32_t src0 = inbox0 + so * c.blk + vofs;
  const uint32_t hdr_in = header0 + 4u * so;
  const uint32_t full_out = map_rank(full0, so);
  const uint32_t cur_lane0 = cur0 + 4u * c.lane;
  // Cursor reset: thread i < set_words owns word i of a set.
  const uint32_t rs_row = threadIdx.x >> 5;
  const uint32_t rs_addr = cur0 + 4u * threadIdx.x;
  const bool resets = threadIdx.x < set_words;
  const uint32_t rs_val0 = rs_row < P ? stage0 + rs_row * c.blk + 2u * c.lane : kAlwaysFull;
  const uint32_t rs_val1 = rs_row < P ? rs_val0 + buf_bytes : kAlwaysFull;

  // Padding of this lane: it only ever touches vectors v with v mod 4 ==
  // lane mod 4, i.e. columns 8*(lane mod 4) .. +7.
  const uint32_t d0 = a.S + 8u * (c.lane & 3u);
  const uint32_t pad0 = d0 | ((d0 + 1u) << 16);
  const uint4 pad = pad_vector(pad0);

  for (uint32_t pass = 0; pass < a.passes; ++pass) {
    c.base = pass * P * c.S;
    const uint32_t left = a.num_bins - c.base;
    c.range = left < P * c.S ? left : P * c.S;
    c.hot_rel = a.hot_bin - c.base;
    if (!kSkew || a.hot_bin == kNoHot || c.hot_rel >= c.range) c.hot_rel = kNoHot;

    uint4* s4 = reinterpret_cast<uint4*>(smem);
    for (uint32_t i = threadIdx.x; i < (c.S + 32u) / 4; i += blockDim.x) s4[i] = make_uint4(0, 0, 0, 0);
    for (uint32_t v = threadIdx.x; v < 8u * qs * P; v += blockDim.x) st_shared_v4(stage0 + 16u * v, pad);
    if (resets) {
      st_shared_u32(rs_addr, rs_val0);              // set 0: round 0, buffer 0
      st_shared_u32(rs_addr + set_bytes, rs_val1);  // set 1: round 1, buffer 1
    }
    if (threadIdx.x < 32u) st_shared_u32(header0 + 4u * threadIdx.x, 0u);
    if (threadIdx.x == 0) st_shared_u32(gave_up, 0u);
    if (threadIdx.x == 0) {
      // One arrival per other sender and round; their bytes complete it.
      mbar_init(full0, P - 1u);
      mbar_init(full0 + 8u, P - 1u);
      mbar_init(staged, kWarps);
      fence_mbar_init();
    }
    cluster_barrier();  // slices zeroed and mbarriers initialised cluster-wide

    int4 cur[kTiles];
    if (rounds > 0) {
      load_round<kKpt>(cur, vec, ntiles, wtile0, rounds == 1);
      c.cur_lane = cur_lane0;
      c.lim0 = stage0 + c.blk;
      partition_round<kTiles, kPow2, kSkew>(cur, c, hot_keys);
      if (rounds > 1) load_round<kKpt>(cur, vec, ntiles, wtile0 + per_round, rounds == 2);
    }
    __syncthreads();  // round 0 staged
    uint32_t k = 0;  // r % 3
    for (uint32_t r = 0; r < rounds; ++r) {
      const uint32_t b = r & 1u;
      if (r > 0 && so != rank) {
        // Apply sender so's block of round r - 1, once every sender has
        // arrived and every byte has landed (this CTA's own block was
        // applied straight from staging when it was shipped).
        const uint32_t pb = b ^ 1u;
        if (wait_mbar(full0 + 8u * pb, ((r - 1u) >> 1) & 1u, gave_up, a.wait_cycles, a.status)) {
          const uint32_t src = src0 + pb * buf_bytes;
          const uint32_t end = src - vofs + 64u * min(ld_shared_u32(hdr_in + 64u * pb), qs);
          for (uint32_t at = src; at < end; at += step) apply_vector(c.slice, ld_shared_v4(at));
        }
      }
      // Round r is staged once every warp has arrived after partitioning it
      // (in round r - 1, after its ship of round r - 1).  On a timeout the
      // warp goes on: the launch is already reported, and every access below
      // stays inside its buffers whatever the cursors hold.
      if (r > 0) wait_mbar(staged, (r - 1u) & 1u, gave_up, a.wait_cycles, a.status);
      // Relaxed: inbox data is published through the mbarriers; this
      // barrier only tells senders that round r-1's inbox has been read
      // (every load of it has returned: its values fed the reds above).
      cluster_arrive_relaxed();
      // Set (r + 2) % 3 was last read by round r - 1's ship, which every warp
      // finished before the wait above; round r + 2 partitions with it into
      // buffer b, after the wait of round r + 1.
      const uint32_t k2 = k == 0 ? 2u : k - 1u;
      if (resets) st_shared_u32(rs_addr + k2 * set_bytes, b ? rs_val1 : rs_val0);
      {
        // Ship owner so's block of round r: rows = its fullest column.
        const uint32_t top = top0 + b * buf_bytes;
        const uint32_t fill = (ld_shared_u32(fill_rd + k * set_bytes) - (top + 2u * c.lane)) >> 6;
        const uint32_t rows = __reduce_max_sync(kFullMask, min(fill, qs));
        const uint32_t end = top + 64u * rows;
        if (so == rank) {
          // This CTA's own block: apply it here instead of shipping it.
          for (uint32_t at = top + vofs; at < end; at += step) {
            apply_vector(c.slice, ld_shared_v4(at));
            st_shared_v4(at, pad);
          }
        } else if (!(a.withhold_last && r + 1u == rounds)) {
          const uint32_t mbar = full_out + 8u * b;
          if (sg == 0 && c.lane == 0) {
            mbar_arrive_expect_tx_remote(mbar, 64u * rows + 4u);
            st_async_u32(hdr_out + 64u * b, rows, mbar);
          }
          for (uint32_t at = top + vofs, dt = dst0 + b * buf_bytes; at < end; at += step, dt += step) {
            st_async_v4(dt, ld_shared_v4(at), mbar);
            st_shared_v4(at, pad);
          }
        }
      }
      const uint32_t k1 = k == 2 ? 0u : k + 1u;
      if (r + 1 < rounds) {
        // Partition round r + 1 into the other buffer while other warps
        // still ship and apply round r; then load round r + 2.
        c.cur_lane = cur_lane0 + k1 * set_bytes;
        c.lim0 = stage0 + (b ^ 1u) * buf_bytes + c.blk;
        partition_round<kTiles, kPow2, kSkew>(cur, c, hot_keys);
        if (r + 2 < rounds)
          load_round<kKpt>(cur, vec, ntiles, wtile0 + (r + 2) * per_round, r + 3 == rounds);
        __syncwarp();  // the warp's staging stores and cursor updates precede the arrival
        if (c.lane == 0) mbar_arrive_local(staged);
      }
      cluster_wait();   // round r's inboxes complete everywhere
      k = k1;
    }
    if (rounds > 0 && so != rank) {
      const uint32_t pb = (rounds - 1u) & 1u;
      if (wait_mbar(full0 + 8u * pb, ((rounds - 1u) >> 1) & 1u, gave_up, a.wait_cycles, a.status)) {
        const uint32_t src = src0 + pb * buf_bytes;
        const uint32_t end = src - vofs + 64u * min(ld_shared_u32(hdr_in + 64u * pb), qs);
        for (uint32_t at = src; at < end; at += step) apply_vector(c.slice, ld_shared_v4(at));
      }
    }

    // Ragged keys (unaligned head, partial tile, tail): the grid's last warp,
    // straight to the owners.
    if (gwarp == nwarps - 1) {
      const int64_t after = a.head + (static_cast<int64_t>(ntiles) << 7);
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

    if constexpr (kSkew) {
      // The hot bin's keys of this pass, one remote increment per warp.
      const uint32_t t = __reduce_add_sync(kFullMask, hot_keys);
      if (c.lane == 0 && t != 0u && c.hot_rel < c.range) {
        uint32_t o, loc;
        owner_local(c.hot_rel, c, o, loc, kPow2);
        red_add_cluster(map_rank(c.slice + 4u * loc, o), t);
      }
      hot_keys = 0;
    }

    cluster_barrier();  // every increment has landed; only own memory after this
    if (ld_shared_u32(gave_up) != 0u) {
      // A wait of this CTA gave up, so an inbox phase may be incomplete.
      // Every sender has issued all its stores (it reached the barrier
      // above), but only the mbarrier tracks their delivery: give bytes still
      // in flight a bounded grace period (DSMEM delivery takes about a
      // microsecond) before the mbarriers are invalidated and the CTA leaves.
      const long long grace = a.wait_cycles < (1ll << 22) ? a.wait_cycles : (1ll << 22);
      const long long until = clock64() + grace;
      while (clock64() < until) {
      }
    }
    if (threadIdx.x == 0) {
      mbar_inval(full0);
      mbar_inval(full0 + 8u);
      mbar_inval(staged);
    }

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

// The helper beside a single-pass ship launch, on the SMs its clusters
// leave idle (clusters of 8 fit only 15 times into this GPU's 152 SMs).  Its
// warps claim kHelperTiles tiles at a time of the tiles after the clusters'
// rounds, [cluster_tiles, cluster_tiles + helper_tiles), from the counter
// the mop-up kernel claims from (the next claim in flight while the
// current one is counted, kHelperBatch tiles loaded at a time), and count
// each in-range key into the helper's
// partial row: with a global atomic, the comparison kernel's method
// ("Distributed Shared Memory", section "When it beats global atomics"),
// unless the key owns its slot of a direct-mapped cache in shared memory
// (kHelperSlots slots of a key and a count; a slot belongs to the first key
// that reaches it).  Frequent keys take their slots early, so a bin holding
// a large share of the keys is counted in shared memory instead of
// serialising the L2 on one address; the cache is added to the row at the
// end.  A tile of 128 equal keys (runs) is one atomic of 128.  Exact: every
// key is counted once, in its slot or in the row.
__device__ __forceinline__ void helper_count(int32_t key, uint32_t num_bins, uint32_t* tags,
                                             uint32_t* cnts, uint32_t* row) {
  const uint32_t k = static_cast<uint32_t>(key);
  if (k >= num_bins) return;
  const uint32_t s = (k * 0x9E3779B1u) >> (32 - kHelperSlotsLog2);
  uint32_t t = *reinterpret_cast<volatile uint32_t*>(tags + s);
  if (t == kNoKey) {
    const uint32_t o = atomicCAS(tags + s, kNoKey, k);
    t = o == kNoKey ? k : o;
  }
  if (t == k)
    atomicAdd(cnts + s, 1u);
  else
    red_add_global(row + k, 1u);
}

__global__ void __launch_bounds__(kHelperThreads, 1) ship_helper_kernel(const ClusterHistArgs a,
                                                                      uint32_t* row) {
  extern __shared__ __align__(16) uint32_t hc[];
  uint32_t* tags = hc;                  // key owning each slot (kNoKey: free)
  uint32_t* cnts = hc + kHelperSlots;   // its count
  if (threadIdx.x == 0)  // the first CTA to start stamps the time (for the report)
    atomicCAS(reinterpret_cast<unsigned long long*>(a.queue + 2), 0ull, global_timer_ns());
  for (uint32_t i = threadIdx.x; i < kHelperSlots; i += kHelperThreads) {
    tags[i] = kNoKey;
    cnts[i] = 0u;
  }
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31u;
  const int4* hvec = reinterpret_cast<const int4*>(a.keys + a.head) + lane +
                     static_cast<size_t>(a.cluster_tiles) * 32u;
  uint32_t mine = 0;
  if (lane == 0) mine = atomicAdd(a.queue, kHelperTiles);
  uint32_t t0 = __shfl_sync(kFullMask, mine, 0);
  while (t0 < a.helper_tiles) {
    if (lane == 0) mine = atomicAdd(a.queue, kHelperTiles);  // the next claim
    for (uint32_t bt = t0; bt < t0 + kHelperTiles; bt += kHelperBatch) {
      int4 v[kHelperBatch];
#pragma unroll
      for (uint32_t u = 0; u < kHelperBatch; ++u)
        v[u] = bt + u < a.helper_tiles ? ld_stream_v4(hvec + static_cast<size_t>(bt + u) * 32u)
                                       : make_int4(-1, -1, -1, -1);
#pragma unroll
      for (uint32_t u = 0; u < kHelperBatch; ++u) {
        // A tile of 128 equal keys (runs) is one atomic of 128.
        const int32_t k0 = __shfl_sync(kFullMask, v[u].x, 0);
        const bool eq = (v[u].x == k0) & (v[u].y == k0) & (v[u].z == k0) & (v[u].w == k0);
        if (__all_sync(kFullMask, eq)) {
          if (lane == 0 && static_cast<uint32_t>(k0) < a.num_bins) red_add_global(row + k0, 128u);
          continue;
        }
        helper_count(v[u].x, a.num_bins, tags, cnts, row);
        helper_count(v[u].y, a.num_bins, tags, cnts, row);
        helper_count(v[u].z, a.num_bins, tags, cnts, row);
        helper_count(v[u].w, a.num_bins, tags, cnts, row);
      }
    }
    t0 = __shfl_sync(kFullMask, mine, 0);
  }
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < kHelperSlots; i += kHelperThreads) {
    const uint32_t n = cnts[i];
    if (n != 0u) red_add_global(row + tags[i], n);
  }
  // The last CTA to finish stamps the time (for the report of the mop-up
  // kernel).
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(a.queue + 6, 1u) == gridDim.x - 1u)
    atomicExch(reinterpret_cast<unsigned long long*>(a.queue + 4), global_timer_ns());
}

// The mop-up, on the caller's stream right after the cluster kernel (whose
// launch covered only its own tiles), beside the helper that may still run:
// its first CTA reports how the split went, CTA 0 counts the ragged tail
// after the last full tile, and every CTA claims kMopTiles tiles at a time
// of the helper's range from the helper's counter (the next claim in flight
// while its warps count the current one) and counts them into the helper's
// row with global atomics.  When the helper has kept pace, each CTA's first
// claim finds the range spent.  The cluster kernel itself carries none of
// this: code after its rounds made the rounds compile 3-4% slower.
__global__ void __launch_bounds__(kMopThreads) ship_mop_up_kernel(const ClusterHistArgs a,
                                                                  uint32_t* row) {
  __shared__ uint32_t s_claim[2];
  constexpr uint32_t kMopWarps = kMopThreads / 32;
  if (threadIdx.x == 0) {
    if (a.helper_report != nullptr && atomicCAS(a.queue + 1, 0u, 1u) == 0u)
      report_helper_share(a.queue, a.helper_tiles, a.cluster_tiles, a.helper_report, a.helper_seq,
                          *reinterpret_cast<volatile uint32_t*>(a.queue));
    s_claim[0] = atomicAdd(a.queue, kMopTiles);
  }
  const uint32_t ntiles = static_cast<uint32_t>(((a.n - a.head) >> 2) >> 5);
  if (blockIdx.x == 0) {
    const int64_t after = a.head + (static_cast<int64_t>(ntiles) << 7);
    for (int64_t j = after + threadIdx.x; j < a.n; j += kMopThreads) {
      const int32_t key = a.keys[j];
      if (static_cast<uint32_t>(key) < a.num_bins) red_add_global(row + key, 1u);
    }
  }
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const int4* hvec = reinterpret_cast<const int4*>(a.keys + a.head) + lane +
                     static_cast<size_t>(a.cluster_tiles) * 32u;
  uint32_t t0 = s_claim[0];
  for (uint32_t j = 1; t0 < a.helper_tiles; ++j) {
    // Slot j % 2 was last read after the barrier of iteration j - 2.
    uint32_t next = 0;
    if (threadIdx.x == 0) next = atomicAdd(a.queue, kMopTiles);
    const uint32_t t1 = min(t0 + kMopTiles, a.helper_tiles);
    for (uint32_t t = t0 + warp; t < t1; t += kMopWarps) {
      const int4 v = ld_stream_v4(hvec + static_cast<size_t>(t) * 32u);
      if (static_cast<uint32_t>(v.x) < a.num_bins) red_add_global(row + v.x, 1u);
      if (static_cast<uint32_t>(v.y) < a.num_bins) red_add_global(row + v.y, 1u);
      if (static_cast<uint32_t>(v.z) < a.num_bins) red_add_global(row + v.z, 1u);
      if (static_cast<uint32_t>(v.w) < a.num_bins) red_add_global(row + v.w, 1u);
    }
    if (threadIdx.x == 0) s_claim[j & 1u] = next;
    __syncthreads();
    t0 = s_claim[j & 1u];
  }
}

template <int kKpt, bool kPow2, bool kSkew>
void* kernel_ptr_t() {
  return reinterpret_cast<void*>(&cluster_ship_kernel<kKpt, kPow2, kSkew>);
}

void* ship_kernel_ptr(int kpt, bool pow2, bool skew) {
  if (skew) {
    if (kpt == 8) return pow2 ? kernel_ptr_t<8, true, true>() : kernel_ptr_t<8, false, true>();
    return pow2 ? kernel_ptr_t<4, true, true>() : kernel_ptr_t<4, false, true>();
  }
  if (kpt == 8) return pow2 ? kernel_ptr_t<8, true, false>() : kernel_ptr_t<8, false, false>();
  return pow2 ? kernel_ptr_t<4, true, false>() : kernel_ptr_t<4, false, false>();
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

}  // namespace

cudaError_t read_and_clear_ship_status(uint32_t* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_ship_status, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  return *out ? cudaMemcpyToSymbol(g_ship_status, &zero, sizeof(uint32_t)) : cudaSuccess;
}

cudaError_t prepare_ship_kernel(int kpt, int smem_bytes) {
  for (int v = 0; v < 4; ++v) {
    const void* fn = ship_kernel_ptr(kpt, (v & 1) != 0, (v & 2) != 0);
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
  cfg.blockDim = dim3(kShipThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, ship_kernel_ptr(kpt, true, false), &cfg);
}

// Largest cluster that can be co-scheduled for this kernel with `smem_bytes`
// of dynamic shared memory per CTA (non-portable sizes allowed).
cudaError_t query_ship_potential_cluster_size(int kpt, int smem_bytes, int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16, 1, 1);
  cfg.blockDim = dim3(kShipThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  return cudaOccupancyMaxPotentialClusterSize(out, ship_kernel_ptr(kpt, true, false), &cfg);
}

cudaError_t launch_cluster_ship(const dsmem_hist_plan_t& plan, const ClusterHistArgs& args,
                                cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.num_clusters) * plan.cluster_size, 1, 1);
  cfg.blockDim = dim3(kShipThreads, 1, 1);
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
  if (args.hot_bin != kNoHot) {
    if (plan.keys_per_thread == 8)
      return p2 ? cudaLaunchKernelEx(&cfg, cluster_ship_kernel<8, true, true>, args)
                : cudaLaunchKernelEx(&cfg, cluster_ship_kernel<8, false, true>, args);
    return p2 ? cudaLaunchKernelEx(&cfg, cluster_ship_kernel<4, true, true>, args)
              : cudaLaunchKernelEx(&cfg, cluster_ship_kernel<4, false, true>, args);
  }
  if (plan.keys_per_thread == 8)
    return p2 ? cudaLaunchKernelEx(&cfg, cluster_ship_kernel<8, true, false>, args)
              : cudaLaunchKernelEx(&cfg, cluster_ship_kernel<8, false, false>, args);
  return p2 ? cudaLaunchKernelEx(&cfg, cluster_ship_kernel<4, true, false>, args)
            : cudaLaunchKernelEx(&cfg, cluster_ship_kernel<4, false, false>, args);
}

cudaError_t prepare_ship_helper() {
  return cudaFuncSetAttribute(ship_helper_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kHelperSmemBytes);
}

cudaError_t launch_ship_mop_up(const ClusterHistArgs& args, uint32_t* row, int ctas,
                               cudaStream_t stream) {
  ship_mop_up_kernel<<<static_cast<unsigned>(ctas), kMopThreads, 0, stream>>>(args, row);
  return cudaGetLastError();
}

cudaError_t launch_ship_helper(const ClusterHistArgs& args, uint32_t* row, int ctas,
                               cudaStream_t stream) {
  ship_helper_kernel<<<static_cast<unsigned>(ctas), kHelperThreads, kHelperSmemBytes, stream>>>(args, row);
  return cudaGetLastError();
}

}  // namespace dsmh
