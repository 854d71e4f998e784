/*
 * Seeded synthetic key generators for the cluster-histogram workloads.
 *
 * These produce INPUTS only.  Nothing here counts keys, owns bins or knows
 * about clusters: the histogram arithmetic lives in oracle/ (CPU reference)
 * and in the CUDA library, and both receive the keys written here.
 *
 * Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014), used in its
 * counter form: draw number i of a stream with seed s is
 *     mix64(s + (i + 1) * 0x9E3779B97F4A7C15)
 * so any index range can be generated independently of the others (the
 * Python side splits large arrays across threads and gets the same bytes).
 *
 * Workloads (the key distributions of the five synthetic configurations):
 *   uniform   keys uniform on [0, B)
 *   zipf      truncated Zipf(s) over ranks 1..B, ranks mapped to bin ids by a
 *             seeded Fisher-Yates permutation of [0, B)
 *   runs      first half uniform on [0, B); second half consecutive runs of
 *             run_len identical keys, each run's value uniform on [0, B)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Draw number i (0-based) of the SplitMix64 stream with this seed. */
uint64_t gen_splitmix64_draw(uint64_t seed, uint64_t i) {
  return mix64(seed + (i + 1) * GOLDEN_GAMMA);
}

static int log2_exact(uint32_t b) { /* -1 if b is not a power of two */
  if (b == 0 || (b & (b - 1)) != 0) return -1;
  int l = 0;
  while ((1u << l) != b) ++l;
  return l;
}

/* Map a 64-bit draw to [0, b): the top log2(b) bits when b is a power of two
 * (exactly uniform), else Lemire's multiply-shift on the top 32 bits. */
static uint32_t to_range(uint64_t u, uint32_t b, int lg) {
  if (lg == 0) return 0;
  if (lg > 0) return (uint32_t)(u >> (64 - lg));
  return (uint32_t)(((u >> 32) * (uint64_t)b) >> 32);
}

/* out[j] = uniform key for global index (offset + j), j < count. */
void gen_uniform(int32_t* out, int64_t offset, int64_t count, uint32_t num_bins,
                 uint64_t seed) {
  int lg = log2_exact(num_bins);
  for (int64_t j = 0; j < count; ++j)
    out[j] = (int32_t)to_range(gen_splitmix64_draw(seed, (uint64_t)(offset + j)),
                               num_bins, lg);
}

/* Half uniform, half runs.  Indices [0, n/2) are uniform with stream `seed`;
 * index i >= n/2 belongs to run (i - n/2) / run_len, whose value is draw
 * number `run` of the stream seed ^ GOLDEN_GAMMA. */
void gen_runs(int32_t* out, int64_t offset, int64_t count, int64_t n,
              uint32_t num_bins, uint32_t run_len, uint64_t seed) {
  int lg = log2_exact(num_bins);
  int64_t half = n / 2;
  uint64_t seed_runs = seed ^ GOLDEN_GAMMA;
  if (run_len == 0) run_len = 1;
  for (int64_t j = 0; j < count; ++j) {
    int64_t i = offset + j;
    uint64_t u = (i < half) ? gen_splitmix64_draw(seed, (uint64_t)i)
                            : gen_splitmix64_draw(seed_runs, (uint64_t)((i - half) / run_len));
    out[j] = (int32_t)to_range(u, num_bins, lg);
  }
}

/* One hot bin plus uniform keys.  The hot bin is draw 0 of the stream
 * seed ^ GOLDEN_GAMMA mapped to [0, num_bins).  Key i takes the hot bin when
 * the low 32 bits of draw i of stream `seed` fall below hot_share (a fraction
 * of 2^32), and otherwise the uniform value of that draw's top bits. */
uint32_t gen_hot_bin(uint32_t num_bins, uint64_t seed) {
  return to_range(gen_splitmix64_draw(seed ^ GOLDEN_GAMMA, 0), num_bins, log2_exact(num_bins));
}

void gen_hot(int32_t* out, int64_t offset, int64_t count, uint32_t num_bins, uint32_t hot_share,
             uint64_t seed) {
  int lg = log2_exact(num_bins);
  uint32_t hot = gen_hot_bin(num_bins, seed);
  for (int64_t j = 0; j < count; ++j) {
    uint64_t u = gen_splitmix64_draw(seed, (uint64_t)(offset + j));
    out[j] = (int32_t)((uint32_t)u < hot_share ? hot : to_range(u, num_bins, lg));
  }
}

/* Zipf tables: cdf over ranks, a guide table for O(1) expected search
 * (Chen and Asau's indexed search), and the rank -> bin permutation. */
typedef struct {
  uint32_t b;
  double* cdf;     /* cdf[r] = P(rank <= r + 1), r in [0, b) */
  uint32_t* guide; /* guide[g] = first r with cdf[r] > g / b */
  uint32_t* perm;  /* perm[r] = bin id of rank r + 1 */
} zipf_tables;

static void zipf_free(zipf_tables* t) {
  free(t->cdf);
  free(t->guide);
  free(t->perm);
}

static int zipf_build(zipf_tables* t, uint32_t b, double s, uint64_t seed) {
  t->b = b;
  t->cdf = (double*)malloc(sizeof(double) * b);
  t->guide = (uint32_t*)malloc(sizeof(uint32_t) * b);
  t->perm = (uint32_t*)malloc(sizeof(uint32_t) * b);
  if (!t->cdf || !t->guide || !t->perm) {
    zipf_free(t);
    return -1;
  }
  /* Normaliser summed smallest-first for accuracy. */
  double h = 0.0;
  for (uint32_t r = b; r >= 1; --r) h += pow((double)r, -s);
  double acc = 0.0;
  for (uint32_t r = 0; r < b; ++r) {
    acc += pow((double)(r + 1), -s);
    t->cdf[r] = acc / h;
  }
  t->cdf[b - 1] = 1.0;
  uint32_t r = 0;
  for (uint32_t g = 0; g < b; ++g) {
    double x = (double)g / (double)b;
    while (r < b - 1 && t->cdf[r] <= x) ++r;
    t->guide[g] = r;
  }
  /* Fisher-Yates with the stream seed ^ GOLDEN_GAMMA: swap step k uses draw k. */
  uint64_t seed_perm = seed ^ GOLDEN_GAMMA;
  for (uint32_t i = 0; i < b; ++i) t->perm[i] = i;
  for (uint32_t i = b - 1, k = 0; i >= 1; --i, ++k) {
    uint64_t u = gen_splitmix64_draw(seed_perm, k);
    uint32_t j = (uint32_t)(((u >> 32) * (uint64_t)(i + 1)) >> 32);
    uint32_t tmp = t->perm[i];
    t->perm[i] = t->perm[j];
    t->perm[j] = tmp;
  }
  return 0;
}

static uint32_t zipf_rank(const zipf_tables* t, uint64_t draw) {
  double u = (double)(draw >> 11) * (1.0 / 9007199254740992.0); /* [0, 1) */
  uint32_t g = (uint32_t)(u * (double)t->b);
  if (g >= t->b) g = t->b - 1;
  uint32_t r = t->guide[g];
  while (r < t->b - 1 && t->cdf[r] <= u) ++r;
  return r; /* 0-based rank */
}

/* out[j] = bin id of the Zipf draw for global index (offset + j).
 * Returns 0, or -1 when the tables cannot be allocated. */
int gen_zipf(int32_t* out, int64_t offset, int64_t count, uint32_t num_bins, double s,
             uint64_t seed) {
  zipf_tables t;
  if (num_bins == 0 || zipf_build(&t, num_bins, s, seed) != 0) return -1;
  for (int64_t j = 0; j < count; ++j)
    out[j] = (int32_t)t.perm[zipf_rank(&t, gen_splitmix64_draw(seed, (uint64_t)(offset + j)))];
  zipf_free(&t);
  return 0;
}

/* The rank -> bin permutation and CDF used by gen_zipf, exposed so tests can
 * check the generator's shape (rank-1 share, top-k mass) in closed form. */
int gen_zipf_tables(uint32_t num_bins, double s, uint64_t seed, double* cdf_out,
                    uint32_t* perm_out) {
  zipf_tables t;
  if (num_bins == 0 || zipf_build(&t, num_bins, s, seed) != 0) return -1;
  memcpy(cdf_out, t.cdf, sizeof(double) * num_bins);
  memcpy(perm_out, t.perm, sizeof(uint32_t) * num_bins);
  zipf_free(&t);
  return 0;
}
