/*
 * Seeded synthetic input generator, shared by the tests, the benchmark and the
 * oracle's callers.  It holds none of the attention / selection arithmetic: it
 * only produces bf16 bit patterns for queries, keys and values, heavy-hitter
 * position sets and ragged lengths.
 *
 * Every value is a pure function of (seed, stream, index): any slice of any
 * tensor can be regenerated on its own, on any machine, bit for bit.  The
 * arithmetic is integer except for one float multiply and one float add per
 * element (this file is compiled with -ffp-contract=off so no FMA is formed),
 * and double-precision normalisation of the direction vector u.  Both are
 * plain IEEE operations, so x86-64 and aarch64 produce identical bits.
 *
 * Counter hash: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; constants as published by
 * S. Vigna for splitmix64).
 *
 * Normal deviates: Irwin-Hall sum of twelve 16-bit uniforms minus 6 (mean 0,
 * variance 1 - 2^-32, support [-6, 6]).  Each sum is an integer over 2^16, so
 * the value is exact in fp32 before the final round-to-nearest-even to bf16.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

static inline uint64_t smix(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

/* Key of one independent stream: (seed, stream id). */
static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return smix(smix(seed) ^ (stream * 0xD1B54A32D192ED03ull));
}

/* Standard-normal approximation for element `idx` of a stream, exact in fp32. */
static inline float normal_at(uint64_t key, uint64_t idx) {
  uint32_t s = 0;
  for (int j = 0; j < 3; ++j) {
    uint64_t h = smix(key + 3ull * idx + (uint64_t)j);
    s += (uint32_t)(h & 0xFFFF) + (uint32_t)((h >> 16) & 0xFFFF) +
         (uint32_t)((h >> 32) & 0xFFFF) + (uint32_t)(h >> 48);
  }
  /* sum of u_i = (s + 6) / 2^16 with u_i = (x_i + 1/2) / 2^16; subtract 6. */
  int32_t num = (int32_t)(s + 6u) - 6 * 65536;
  return (float)num * (1.0f / 65536.0f);
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs only). */
static inline uint16_t bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* i.i.d. N(0,1) bf16 values for indices [start, start+count) of a stream. */
void vgs_fill_normal(uint64_t seed, uint64_t stream, uint64_t start, int64_t count, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static) if (count > 65536)
  for (int64_t i = 0; i < count; ++i) out[i] = bf16_rne(normal_at(key, start + (uint64_t)i));
}

/* Unit direction in R^d: a normal draw normalised in double, rounded to fp32. */
void vgs_unit_vector(uint64_t seed, uint64_t stream, int d, float* out) {
  uint64_t key = stream_key(seed, stream);
  double ss = 0.0;
  for (int e = 0; e < d; ++e) {
    double z = (double)normal_at(key, (uint64_t)e);
    ss += z * z;
  }
  double nrm = sqrt(ss);
  for (int e = 0; e < d; ++e) out[e] = (float)((double)normal_at(key, (uint64_t)e) / nrm);
}

/*
 * Keys (or values) for `npos` consecutive positions of one sequence, all
 * heads: out[p][h][e], element index ((start_pos + p) * H + h) * d + e.
 * kind[p] (may be NULL = all 0): 0 -> N(0,1); 1 -> heavy hitter 3u + N(0,1)/2;
 * 2 -> sink 4u.  u (length d) is needed only when some kind is non-zero.
 */
void vgs_fill_keys(uint64_t seed, uint64_t stream, int64_t start_pos, int64_t npos, int H, int d,
                   const uint8_t* kind, const float* u, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
  const int64_t row = (int64_t)H * d;
#pragma omp parallel for schedule(static) if (npos * row > 65536)
  for (int64_t p = 0; p < npos; ++p) {
    const uint8_t k = kind ? kind[p] : 0;
    uint16_t* o = out + p * row;
    const uint64_t base = (uint64_t)(start_pos + p) * (uint64_t)row;
    for (int64_t j = 0; j < row; ++j) {
      const int e = (int)(j % d);
      if (k == 0) {
        o[j] = bf16_rne(normal_at(key, base + (uint64_t)j));
      } else if (k == 1) {
        float a = 3.0f * u[e];
        float b = 0.5f * normal_at(key, base + (uint64_t)j);
        o[j] = bf16_rne(a + b);
      } else {
        o[j] = bf16_rne(4.0f * u[e]);
      }
    }
  }
}

/* Queries N(0,1) + u (u may be NULL for plain N(0,1)): element i of a stream
 * whose innermost axis has length d. */
void vgs_fill_query(uint64_t seed, uint64_t stream, uint64_t start, int64_t count, int d, const float* u,
                    uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static) if (count > 65536)
  for (int64_t i = 0; i < count; ++i) {
    const uint64_t idx = start + (uint64_t)i;
    float z = normal_at(key, idx);
    out[i] = u ? bf16_rne(z + u[idx % (uint64_t)d]) : bf16_rne(z);
  }
}

typedef struct {
  uint64_t h;
  int64_t p;
} hp_t;

static int hp_cmp(const void* a, const void* b) {
  const hp_t* x = (const hp_t*)a;
  const hp_t* y = (const hp_t*)b;
  if (x->h != y->h) return x->h < y->h ? -1 : 1;
  return x->p < y->p ? -1 : (x->p > y->p);
}

/* Mark exactly m distinct positions of [lo, hi) with `value` in flags[]
 * (indexed by absolute position): the m smallest hashes, a uniform choice
 * without replacement.  Returns 0, or -1 on bad arguments / no memory. */
int vgs_choose(uint64_t seed, uint64_t stream, int64_t lo, int64_t hi, int64_t m, uint8_t value, uint8_t* flags) {
  if (hi < lo || m < 0 || m > hi - lo) return -1;
  int64_t n = hi - lo;
  if (n == 0 || m == 0) return 0;
  hp_t* a = (hp_t*)malloc(sizeof(hp_t) * (size_t)n);
  if (!a) return -1;
  uint64_t key = stream_key(seed, stream);
  for (int64_t i = 0; i < n; ++i) {
    a[i].h = smix(key + (uint64_t)(lo + i));
    a[i].p = lo + i;
  }
  qsort(a, (size_t)n, sizeof(hp_t), hp_cmp);
  for (int64_t i = 0; i < m; ++i) flags[a[i].p] = value;
  free(a);
  return 0;
}

/* Uniform integer in [lo, hi] for element idx of a stream. */
int64_t vgs_uniform_int(uint64_t seed, uint64_t stream, uint64_t idx, int64_t lo, int64_t hi) {
  uint64_t span = (uint64_t)(hi - lo) + 1ull;
  return lo + (int64_t)(smix(stream_key(seed, stream) + idx) % span);
}
