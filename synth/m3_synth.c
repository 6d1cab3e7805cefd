/*
 * Seeded synthetic input generator for the Mamba-3 scan workloads.
 *
 * This module holds no arithmetic of the scan itself: it only draws the
 * random tensors (x, B, C, dt, lam, theta, A, D, initial states, carries,
 * sequence lengths) with the distributions of the synthetic workloads, and
 * rounds them to the storage type.  Both the CPU oracle and the GPU tests
 * and benchmark consume its output, so every element is a pure function of
 * (seed, stream, flat index): the same call always yields the same bits,
 * whatever the thread count.
 *
 * Random numbers: a counter-based generator built on the SplitMix64 output
 * function (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014).  Word i of stream s under seed k is
 *     mix64(key(k, s) + (i + 1) * 0x9E3779B97F4A7C15)
 * with key(k, s) = mix64(k ^ mix64(s + 0x632BE59BD9B4E019)).
 * Uniforms take the top 53 bits.  Normals use the Box-Muller transform on
 * words 2i and 2i+1 (one normal per index, the cosine branch).
 *
 * Rounding: values are produced in double, rounded to float (round to
 * nearest even, the C cast), and for bf16 rounded again from the float
 * bits with round-to-nearest-even.  NaN never occurs for these draws.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYN_OUT_F32 0
#define SYN_OUT_BF16 1
#define SYN_OUT_F64 2

enum {
  SYN_NORMAL = 0,          /* mean p0, standard deviation p1           */
  SYN_NORMAL_RMS = 1,      /* N(0,1) rows of row_len, then x/sqrt(mean(x^2)+p0) */
  SYN_SOFTPLUS_NORMAL = 2, /* softplus(N(0,1) + p0)                    */
  SYN_NEG_EXP_NORMAL = 3,  /* -exp(N(0, p1))                           */
  SYN_UNIFORM = 4,         /* U(p0, p1)                                */
  SYN_SIGMOID_NORMAL = 5   /* sigmoid(N(0,1))                          */
};

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed ^ mix64(stream + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t word(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1ULL) * 0x9E3779B97F4A7C15ULL);
}

/* uniform in [0, 1) */
static inline double u01(uint64_t w) { return (double)(w >> 11) * 0x1.0p-53; }

static inline double std_normal(uint64_t key, uint64_t i) {
  double u1 = ((double)(word(key, 2 * i) >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
  double u2 = u01(word(key, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t rounding = 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)((u + rounding) >> 16);
}

static inline void store(void* out, int64_t i, double v, int out_dtype) {
  if (out_dtype == SYN_OUT_F64) {
    ((double*)out)[i] = v;
  } else if (out_dtype == SYN_OUT_F32) {
    ((float*)out)[i] = (float)v;
  } else {
    ((uint16_t*)out)[i] = f32_to_bf16_rne((float)v);
  }
}

static double draw(int kind, uint64_t key, uint64_t idx, double p0, double p1) {
  switch (kind) {
    case SYN_NORMAL:
      return p0 + p1 * std_normal(key, idx);
    case SYN_SOFTPLUS_NORMAL: {
      double z = std_normal(key, idx) + p0;
      return z > 30.0 ? z : log1p(exp(z));
    }
    case SYN_NEG_EXP_NORMAL:
      return -exp(p1 * std_normal(key, idx));
    case SYN_UNIFORM:
      return p0 + (p1 - p0) * u01(word(key, idx));
    case SYN_SIGMOID_NORMAL:
      return 1.0 / (1.0 + exp(-std_normal(key, idx)));
    default:
      return 0.0;
  }
}

/*
 * Fill out[0 .. count) with elements offset .. offset+count of the tensor
 * (seed, stream).  For SYN_NORMAL_RMS, count and offset must be multiples
 * of row_len.  Returns 0 on success, -1 on a bad argument.
 */
int synth_fill(uint64_t seed, uint64_t stream, int kind, double p0, double p1,
               int64_t offset, int64_t count, int64_t row_len, int out_dtype,
               void* out) {
  if (count < 0 || offset < 0 || !out) return -1;
  if (out_dtype != SYN_OUT_F32 && out_dtype != SYN_OUT_BF16 && out_dtype != SYN_OUT_F64)
    return -1;
  uint64_t key = stream_key(seed, stream);
  if (kind == SYN_NORMAL_RMS) {
    if (row_len <= 0 || count % row_len || offset % row_len) return -1;
    int64_t rows = count / row_len;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      double ss = 0.0;
      for (int64_t j = 0; j < row_len; ++j) {
        double v = std_normal(key, (uint64_t)(offset + r * row_len + j));
        ss += v * v;
      }
      double inv = 1.0 / sqrt(ss / (double)row_len + p0);
      for (int64_t j = 0; j < row_len; ++j) {
        double v = std_normal(key, (uint64_t)(offset + r * row_len + j));
        store(out, r * row_len + j, v * inv, out_dtype);
      }
    }
    return 0;
  }
  if (kind < SYN_NORMAL || kind > SYN_SIGMOID_NORMAL) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i)
    store(out, i, draw(kind, key, (uint64_t)(offset + i), p0, p1), out_dtype);
  return 0;
}

/* Integer lengths uniform on [lo, hi] (inclusive), one per index. */
int synth_lengths(uint64_t seed, uint64_t stream, int64_t lo, int64_t hi, int64_t count,
                  int32_t* out) {
  if (count < 0 || hi < lo || !out) return -1;
  uint64_t key = stream_key(seed, stream);
  for (int64_t i = 0; i < count; ++i) {
    double u = u01(word(key, (uint64_t)i));
    int64_t v = lo + (int64_t)floor(u * (double)(hi - lo + 1));
    if (v > hi) v = hi;
    out[i] = (int32_t)v;
  }
  return 0;
}
