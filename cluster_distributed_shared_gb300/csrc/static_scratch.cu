// dsmem_hist_static: the histogram without any allocation by the library.
//
// Some callers cannot let a library allocate device memory:
//   - code that runs while a CUDA stream is being captured into a graph,
//     where cudaMalloc is not allowed and a stream-ordered allocation would
//     become part of the graph;
//   - applications that own all device memory through their own arena or
//     pool, or that run under a memory budget the library must not grow;
//   - latency-sensitive paths that must not call into the allocator, which
//     can synchronise the device or block on the driver.
// For them this entry point keeps the per-cluster partial histograms in a
// file-scope `static __device__` array of fixed size, which every GPU that
// loads the library holds for the life of the process.  The caller still
// passes the keys and the bins.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "dsmem_hist.h"
#include "internal.h"

namespace dsmh {
namespace {

// 32 MiB of partial rows: one row of num_bins counters (rounded up to a
// multiple of 4) per cluster, so up to 8,388,608 bins, and as many clusters
// as fit for smaller bin counts (15 rows of 262,144 bins need 15 MiB).
constexpr int64_t kStaticScratchBytes = int64_t{32} << 20;
static __device__ __align__(256) uint32_t g_static_partials[kStaticScratchBytes / 4];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
uint32_t* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_partials on the current device, looked up once
// per device (the host-side name of the array is only a stand-in).
int static_scratch(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_error(DSMEM_HIST_ECUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return record_error(DSMEM_HIST_EUNSUPPORTED, "device ordinal beyond the static scratch table");
  std::lock_guard<std::mutex> g(g_static_mutex);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_partials);
    if (e != cudaSuccess || !p)
      return record_error(DSMEM_HIST_ECUDA, "cudaGetSymbolAddress of the static scratch failed");
    g_static_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_static_ptr[dev];
  return DSMEM_HIST_OK;
}

}  // namespace
}  // namespace dsmh

extern "C" int dsmem_hist_static(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins,
                                 cudaStream_t stream) {
  uint32_t* scratch = nullptr;
  // Reject sizes the static scratch cannot hold before touching the device.
  const int64_t row_bytes = 4 * ((static_cast<int64_t>(num_bins) + 3) & ~int64_t{3});
  if (num_bins >= 1 && row_bytes > dsmh::kStaticScratchBytes)
    return dsmh::record_error(DSMEM_HIST_EINVAL,
                              "num_bins exceeds the static scratch (at most 8388608 bins)");
  const int rc = dsmh::static_scratch(&scratch);
  if (rc) return rc;
  return dsmh::run_with_fixed_scratch(keys, n, num_bins, bins, scratch, dsmh::kStaticScratchBytes,
                                      stream);
}
