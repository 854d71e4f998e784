/*
 * CPU ORACLE for the thread-block-cluster histogram.  TEST INFRASTRUCTURE
 * ONLY: the tests, the package smoke check and the benchmark's CPU-baseline
 * leg call it; the CUDA library never does, and it shares no code, header or
 * table with the library.
 *
 * What the method computes ("Distributed Shared Memory", section "The cluster
 * histogram"): the bins are split into equal slices owned by the cluster's
 * blocks; every key increments the counter of bin `key` in the slice of the
 * block that owns it; after the second cluster barrier every block adds its
 * slice into the final bin array.  Integer addition is associative and
 * commutative, so however the keys are split over threads, blocks, clusters
 * and passes, the final array is the plain count of each bin.  The oracle is
 * that definition written out:
 *
 *     bins[b] = #{ i in [0, n) : keys[i] == b }   (mod 2^32),  0 <= b < num_bins
 *
 * Readings of points the page leaves open (each also listed in the design
 * notes):
 *   - keys outside [0, num_bins), negative ones included, are not counted
 *     (the page's kernel assumes every key is a valid bin);
 *   - `bins` is overwritten, not accumulated into (the page adds into an
 *     array whose zeroing it does not show);
 *   - counters are 32-bit unsigned and wrap modulo 2^32.
 *
 * Single-threaded, no blocking, no vectorisation hints.
 */
#include <stdint.h>

void oracle_histogram(const int32_t* keys, int64_t n, int32_t num_bins, uint32_t* bins) {
  for (int32_t b = 0; b < num_bins; ++b) bins[b] = 0u;
  for (int64_t i = 0; i < n; ++i) {
    int32_t k = keys[i];
    if (k >= 0 && k < num_bins) bins[k] += 1u;
  }
}
