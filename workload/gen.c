/*
 * Seeded, counter-based input generators for the Beam MoE block workloads.
 *
 * This file holds no arithmetic of the MoE block itself: it only draws the
 * synthetic inputs (activations, router weight, expert weights, routing
 * indices for stage tests) and converts checkpoint formats (bf16 -> NVFP4).
 * Both the CUDA path's tests/bench and the CPU oracle consume its output.
 *
 * Random stream: SplitMix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used counter-style: draw i of
 * stream (seed, tensor_id) is mix64(key + (i + 1) * gamma), so any index range
 * of any tensor can be generated independently and in parallel.
 * Normal deviates: Box-Muller (Box & Muller 1958) on two uniform draws.
 *
 * The NVFP4 layout follows the format named for the NVFP4 workload: e2m1
 * values in 16-element blocks along K, one e4m3 scale per block and one fp32
 * scale per tensor (release article, section "Mixture of Experts", on the
 * NVFP4 checkpoint storing most parameters in 4-bit precision).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
  return mix64(mix64(seed + GOLDEN) ^ (tensor_id * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* i-th standard normal deviate of a stream (pairs share one Box-Muller draw). */
static inline double normal_at(uint64_t key, uint64_t i) {
  const uint64_t p = i >> 1;
  const uint64_t a = draw(key, 2 * p), b = draw(key, 2 * p + 1);
  const double u1 = ((double)(a >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
  const double u2 = (double)(b >> 11) * 0x1.0p-53;         /* [0, 1) */
  const double r = sqrt(-2.0 * log(u1));
  const double th = 6.283185307179586476925 * u2;
  return (i & 1) ? r * sin(th) : r * cos(th);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* out[i] = bf16(float(mean[col] + std * N_i)) for i in [start, start+count).
 * mean may be NULL (zero mean); otherwise column col = i % ncols. */
void gen_normal_bf16(uint64_t seed, uint64_t tensor_id, int64_t start, int64_t count,
                     double std, const double* mean, int64_t ncols, uint16_t* out) {
  const uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    const uint64_t g = (uint64_t)(start + i);
    double v = std * normal_at(key, g);
    if (mean) v += mean[(int64_t)(g % (uint64_t)ncols)];
    out[i] = f32_to_bf16_rne((float)v);
  }
}

/* out[i] = float(std * N_i) */
void gen_normal_f32(uint64_t seed, uint64_t tensor_id, int64_t start, int64_t count, double std,
                    float* out) {
  const uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) out[i] = (float)(std * normal_at(key, (uint64_t)(start + i)));
}

/* out[i] = std * N_i in double (no rounding) */
void gen_normal_f64(uint64_t seed, uint64_t tensor_id, int64_t start, int64_t count, double std,
                    double* out) {
  const uint64_t key = stream_key(seed, tensor_id);
  for (int64_t i = 0; i < count; ++i) out[i] = std * normal_at(key, (uint64_t)(start + i));
}

/* out[i] = uniform draw in [0, 1) */
void gen_uniform_f64(uint64_t seed, uint64_t tensor_id, int64_t start, int64_t count,
                     double* out) {
  const uint64_t key = stream_key(seed, tensor_id);
  for (int64_t i = 0; i < count; ++i)
    out[i] = (double)(draw(key, (uint64_t)(start + i)) >> 11) * 0x1.0p-53;
}

/* Random routing for stage tests: per token, K distinct experts out of E,
 * drawn by a partial Fisher-Yates shuffle on counter-based draws. When
 * hot_count > 0, experts [0, hot_count) are drawn first with probability
 * hot_prob per slot, which skews the per-expert load. */
void gen_random_topk(uint64_t seed, uint64_t tensor_id, int T, int E, int K, int hot_count,
                     double hot_prob, int32_t* idx) {
  const uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    int perm[1024];
    for (int e = 0; e < E; ++e) perm[e] = e;
    uint64_t c = (uint64_t)t * 4096u;
    for (int k = 0; k < K; ++k) {
      int lo = k, hi = E; /* choose from perm[lo..hi) */
      if (hot_count > 0) {
        const double u = (double)(draw(key, c++) >> 11) * 0x1.0p-53;
        if (u < hot_prob) {
          /* restrict to the hot experts still unpicked: they sit in perm[k..E) */
          int n_hot = 0;
          for (int j = k; j < E; ++j)
            if (perm[j] < hot_count) ++n_hot;
          if (n_hot > 0) {
            int pick = (int)(draw(key, c++) % (uint64_t)n_hot);
            for (int j = k; j < E; ++j)
              if (perm[j] < hot_count && pick-- == 0) {
                int tmp = perm[k]; perm[k] = perm[j]; perm[j] = tmp;
                break;
              }
            idx[(int64_t)t * K + k] = perm[k];
            continue;
          }
        }
      }
      const int j = lo + (int)(draw(key, c++) % (uint64_t)(hi - lo));
      int tmp = perm[k]; perm[k] = perm[j]; perm[j] = tmp;
      idx[(int64_t)t * K + k] = perm[k];
    }
  }
}

/* ---------------- NVFP4 checkpoint conversion (input preparation) ---------------- */

/* e2m1 magnitudes by 3-bit code (exponent bias 1, one mantissa bit). */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Nearest e2m1 code of |v| (v >= 0), ties to the even code (mantissa bit 0). */
static inline uint8_t e2m1_code_rne(double v) {
  if (v >= 6.0) return 7;
  int best = 0;
  double bd = v;
  for (int c = 1; c < 8; ++c) {
    const double d = fabs(v - kE2M1[c]);
    if (d < bd || (d == bd && (c & 1) == 0)) { bd = d; best = c; }
  }
  return (uint8_t)best;
}

/* e4m3 (bias 7, no infinities, max 448) value of a code. */
static inline double e4m3_value(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Nearest non-negative e4m3 code of v >= 0, ties to even mantissa, saturating
 * at 448 (code 0x7E; 0x7F is NaN in this format). */
static inline uint8_t e4m3_code_rne(double v) {
  if (!(v > 0.0)) return 0;
  if (v >= 448.0) return 0x7E;
  if (v < 0x1.0p-6) { /* subnormal range: multiples of 2^-9 */
    const double m = nearbyint(v * 512.0); /* 0..8; 8 is the smallest normal */
    return (uint8_t)m;
  }
  int x;
  const double f = frexp(v, &x); /* v = f * 2^x, f in [0.5, 1) */
  int ex = x - 1;                 /* v = (2f) * 2^ex, 2f in [1, 2) */
  double m = nearbyint((2.0 * f - 1.0) * 8.0);
  if (m >= 8.0) { m = 0.0; ++ex; }
  const int code = ((ex + 7) << 3) | (int)m;
  return (uint8_t)(code > 0x7E ? 0x7E : code);
}

static inline double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Quantise one [N][K] bf16 matrix to FP8 with 128 x 128 block scales (the
 * layout of DeepSeek-V3's FP8 checkpoints; the article's router follows that
 * model and names FP8 checkpoints for Hopper-class GPUs):
 *   block scale  s = amax_block / 448   (fp32; 0 for an all-zero block)
 *   value        q = e4m3(w / s)        (round to nearest even, saturating)
 * codes[n][k]: e4m3 byte (bit 7 = sign). scales[n/128][k/128]: fp32.
 * N and K must be multiples of 128. */
void gen_quantize_fp8(const uint16_t* w, int64_t N, int64_t K, uint8_t* codes, float* scales) {
  const int64_t nbn = N / 128, nbk = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t bn = 0; bn < nbn; ++bn)
    for (int64_t bk = 0; bk < nbk; ++bk) {
      double amax = 0.0;
      for (int64_t n = bn * 128; n < bn * 128 + 128; ++n)
        for (int64_t k = bk * 128; k < bk * 128 + 128; ++k) {
          const double a = fabs(bf16_to_f64(w[n * K + k]));
          if (a > amax) amax = a;
        }
      const float sc = (float)(amax / 448.0);
      scales[bn * nbk + bk] = sc;
      for (int64_t n = bn * 128; n < bn * 128 + 128; ++n)
        for (int64_t k = bk * 128; k < bk * 128 + 128; ++k) {
          const double v = bf16_to_f64(w[n * K + k]);
          uint8_t code = 0;
          if (sc > 0.0f) code = e4m3_code_rne(fabs(v) / (double)sc);
          codes[n * K + k] = (uint8_t)(code | ((v < 0.0 && code != 0) ? 0x80 : 0));
        }
    }
}

/* Quantise one [N][K] bf16 matrix to NVFP4:
 *   tensor scale  s_t = amax / (6 * 448)
 *   block scale   s_b = e4m3(amax_block / (6 * s_t))       (16 values along K)
 *   value         q   = e2m1(w / (s_b * s_t)), clamped to +-6
 * packed[n][k/2]: low nibble = even k; nibble bit 3 = sign.
 * scales[n][k/16]: e4m3 code. Returns s_t. K must be a multiple of 16. */
float gen_quantize_nvfp4(const uint16_t* w, int64_t N, int64_t K, uint8_t* packed,
                         uint8_t* scales) {
  double amax = 0.0;
  for (int64_t i = 0; i < N * K; ++i) {
    const double a = fabs(bf16_to_f64(w[i]));
    if (a > amax) amax = a;
  }
  const float st = (float)(amax / (6.0 * 448.0));
  const int64_t nb = K / 16;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint16_t* blk = w + n * K + b * 16;
      double bmax = 0.0;
      for (int j = 0; j < 16; ++j) {
        const double a = fabs(bf16_to_f64(blk[j]));
        if (a > bmax) bmax = a;
      }
      const uint8_t sc = (st > 0.0f) ? e4m3_code_rne(bmax / (6.0 * (double)st)) : 0;
      scales[n * nb + b] = sc;
      const double denom = e4m3_value(sc) * (double)st;
      for (int j = 0; j < 16; j += 2) {
        uint8_t nib[2];
        for (int h = 0; h < 2; ++h) {
          const double v = bf16_to_f64(blk[j + h]);
          uint8_t code = 0;
          if (denom > 0.0) code = e2m1_code_rne(fabs(v) / denom);
          nib[h] = (uint8_t)(code | ((v < 0.0 && code != 0) ? 8 : 0));
        }
        packed[n * (K / 2) + (b * 16 + j) / 2] = (uint8_t)(nib[0] | (nib[1] << 4));
      }
    }
  }
  return st;
}
