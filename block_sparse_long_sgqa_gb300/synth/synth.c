/*
 * Seeded synthetic inputs for the block-wise Sparse GQA prefill path.
 *
 * This file draws random numbers and lays them out; it computes nothing of
 * the method itself (no block merge, no scores, no selection, no attention).
 * Both the CUDA path and the CPU oracle consume what it writes, so it is the
 * one piece of code the two share.
 *
 * Every value is a pure function of (seed, stream, flat index): SplitMix64
 * (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014; the finaliser constants are Vigna's published ones) turns the
 * counter into 53 random bits, and the Box-Muller transform (1958) turns two
 * uniforms into one standard normal.  The AR(1) noise is the one sequential
 * exception: lane l at step t depends on lane l at step t-1.
 *
 * Built with -ffp-contract=off so that the same source gives the same bits on
 * x86-64 and AArch64 hosts (up to the host libm's log/cos/sqrt).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_base(uint64_t seed, uint64_t stream) {
  return splitmix64(splitmix64(seed) ^ (stream * 0xD1B54A32D192ED03ull));
}

/* uniform in [0, 1) with 53 random bits */
static inline double u01(uint64_t base, uint64_t idx) {
  return (double)(splitmix64(base + idx) >> 11) * (1.0 / 9007199254740992.0);
}

/* standard normal number idx of the stream (Box-Muller, cosine branch) */
static inline double normal_at(uint64_t base, uint64_t idx) {
  double u1 = u01(base, 2 * idx);
  double u2 = u01(base, 2 * idx + 1);
  double r = sqrt(-2.0 * log(1.0 - u1)); /* 1-u1 is in (0, 1] */
  return r * cos(6.283185307179586 * u2);
}

void synth_fill_normal(uint64_t seed, uint64_t stream, int64_t n, float* out) {
  uint64_t base = stream_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)normal_at(base, (uint64_t)i);
}

void synth_fill_uniform(uint64_t seed, uint64_t stream, int64_t n, double* out) {
  uint64_t base = stream_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = u01(base, (uint64_t)i);
}

/* n unit vectors of length d (normalised Gaussian draws), row-major [n][d] */
void synth_unit_dirs(uint64_t seed, uint64_t stream, int64_t n, int d, float* out) {
  uint64_t base = stream_base(seed, stream);
  for (int64_t r = 0; r < n; ++r) {
    double tmp[1024];
    double ss = 0.0;
    for (int i = 0; i < d; ++i) {
      tmp[i] = normal_at(base, (uint64_t)(r * d + i));
      ss += tmp[i] * tmp[i];
    }
    double inv = 1.0 / sqrt(ss);
    for (int i = 0; i < d; ++i) out[r * d + i] = (float)(tmp[i] * inv);
  }
}

/* Topic label per position: runs of geometric length (mean mean_len, at least
 * 1), each run's topic uniform in [0, n_topics). */
void synth_topic_runs(uint64_t seed, uint64_t stream, int64_t n, double mean_len,
                      int n_topics, int32_t* out) {
  uint64_t base = stream_base(seed, stream);
  double p = 1.0 / mean_len;
  double lq = log(1.0 - p);
  int64_t pos = 0;
  uint64_t k = 0;
  while (pos < n) {
    double u = u01(base, 2 * k);
    int64_t len = 1 + (int64_t)floor(log(1.0 - u) / lq);
    int32_t topic = (int32_t)(u01(base, 2 * k + 1) * n_topics);
    if (topic >= n_topics) topic = n_topics - 1;
    for (int64_t i = 0; i < len && pos < n; ++i) out[pos++] = topic;
    ++k;
  }
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void synth_to_bf16(const float* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

/*
 * Clustered rows: X[r][h][i] = amp * dirs[h / hpg][topic[pos0 + r]][i]
 *                             + add_scale * add[(r / add_div)][h / hpg][i]   (if add)
 *                             + noise[r][h][i]
 * noise is i.i.d. N(0,1) (rho == 0) or, per lane (h, i), a stationary AR(1)
 * process along r with N(0,1) marginals: e_0 = z_0, e_r = rho e_{r-1} +
 * sqrt(1 - rho^2) z_r.  Output is fp32 (out_bf16 == 0) or bf16 bits.
 * topic may be NULL (no topic term); add may be NULL.
 */
void synth_clustered(uint64_t seed, uint64_t stream, int64_t P, int H, int hpg, int d,
                     int64_t pos0, const int32_t* topic, const float* dirs, int n_topics,
                     float amp, double rho, const float* add, int64_t add_div, float add_scale,
                     int out_bf16, void* out) {
  enum { LB = 64 }; /* lanes per work item: contiguous output runs */
  uint64_t base = stream_base(seed, stream);
  const int64_t lanes = (int64_t)H * d;
  const int G = H / hpg; /* number of groups */
  const double s = sqrt(1.0 - rho * rho);
  const int64_t nlb = (lanes + LB - 1) / LB;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nlb; ++b) {
    double e[LB];
    const int64_t l0 = b * LB;
    const int64_t l1 = (l0 + LB < lanes) ? l0 + LB : lanes;
    for (int64_t r = 0; r < P; ++r) {
      for (int64_t l = l0; l < l1; ++l) {
        const int h = (int)(l / d), i = (int)(l % d), g = h / hpg;
        double z = normal_at(base, (uint64_t)(r * lanes + l));
        double ev = (r == 0 || rho == 0.0) ? z : rho * e[l - l0] + s * z;
        e[l - l0] = ev;
        double v = ev;
        if (topic) v += (double)amp * dirs[((int64_t)g * n_topics + topic[pos0 + r]) * d + i];
        if (add) v += (double)add_scale * add[((r / add_div) * G + g) * (int64_t)d + i];
        float fv = (float)v;
        if (out_bf16)
          ((uint16_t*)out)[r * lanes + l] = f32_to_bf16_rne(fv);
        else
          ((float*)out)[r * lanes + l] = fv;
      }
    }
  }
}
