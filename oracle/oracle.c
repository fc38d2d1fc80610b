/*
 * CPU oracle for one Beam MoE block forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow, obviously-correct
 * restatement of what the block computes, used to check the CUDA path. Only
 * the test suite, the package smoke check and the benchmark's CPU-baseline leg
 * may load it; the product path never calls it and has no CPU fallback.
 * It shares no code with the CUDA library.
 *
 * What it restates (Reflection "Beam 1.0" release article):
 *  - section "Mixture of Experts": 256 experts per MoE layer, each a SwiGLU
 *    MLP with intermediate size 2,560; a DeepSeek-V3-style group-limited
 *    router that scores all experts with a sigmoid, splits them into 8 groups
 *    of 32, keeps the 4 groups with the best sum of their two top scores and
 *    picks the top 8 experts inside those groups; no shared expert; expert
 *    outputs combined with router weights normalised to sum 1, times 2.5.
 *  - section "Residual stream", last paragraph: the router and the SwiGLU
 *    product are computed in FP32.
 *  - section "Key specifications": 8 experts routed per token.
 *
 * Readings where the article is silent (each one is listed in the design
 * notes): ties go to the lower group / expert index; the router logits have no
 * bias term (the optional selection bias of load balancing is separate);
 * the normalisation has no epsilon; h = silu(g) * u is formed in FP32 and
 * rounded to bf16 before the down projection (the down GEMM takes bf16 input);
 * the block output is returned unrounded (double).
 *
 * All sums accumulate in double, in index order. FP32 appears only where the
 * article fixes it (logits, scores, group scores, SwiGLU product).
 *
 * Weight storage (shared with the CUDA library's ABI, K-contiguous):
 *   gate, up: [E][I][d]   (row i of expert e holds the i-th column of W_gate)
 *   down:     [E][d][I]   (row n holds the n-th column of W_down)
 *   router:   [d][E] fp32 (logits = x . W_r)
 * NVFP4 weights: packed e2m1 [E][N][K/2] (low nibble = even k), e4m3 block
 * scales [E][N][K/16], one fp32 tensor scale per expert and matrix.
 * FP8 weights: e4m3 codes [E][N][K], one fp32 scale per 128 x 128 block
 * [E][N/128][K/128] (DeepSeek-V3's block-scaled layout).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------- scalar formats ---------------- */

static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* float -> bf16, round to nearest even */
static uint16_t bf16_round(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return 0x7FC0;
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* e2m1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
 * subnormal (m * 0.5). */
double oracle_e2m1_value(int code) {
  const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* e4m3 (OCP FP8 E4M3FN): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities. */
double oracle_e4m3_value(int code) {
  const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* ---------------- weights ---------------- */

enum { WFMT_BF16 = 0, WFMT_NVFP4 = 1, WFMT_FP8 = 2 };

typedef struct {
  int fmt;
  const uint16_t* bf16;  /* [E][N][K] */
  const uint8_t* packed; /* NVFP4 [E][N][K/2]; FP8 [E][N][K] e4m3 codes */
  const uint8_t* sf;     /* NVFP4 [E][N][K/16] e4m3; FP8: fp32 [E][N/128][K/128] */
  const float* ts;       /* [E] (NVFP4) */
  int64_t N, K;
} wmat;

/* Value of element (n, k) of expert e's matrix, dequantised exactly. */
static double wmat_at(const wmat* w, int e, int64_t n, int64_t k) {
  const int64_t row = (int64_t)e * w->N + n;
  if (w->fmt == WFMT_BF16) return bf16_value(w->bf16[row * w->K + k]);
  if (w->fmt == WFMT_FP8) {
    /* e4m3 code times the fp32 scale of its 128 x 128 block (DeepSeek-V3's FP8 layout) */
    const float* bs = (const float*)w->sf;
    const int64_t nbn = w->N / 128, nbk = w->K / 128;
    return oracle_e4m3_value(w->packed[row * w->K + k]) *
           (double)bs[((int64_t)e * nbn + n / 128) * nbk + k / 128];
  }
  const uint8_t byte = w->packed[row * (w->K / 2) + k / 2];
  const int nib = (k & 1) ? (byte >> 4) : (byte & 15);
  return oracle_e2m1_value(nib) * oracle_e4m3_value(w->sf[row * (w->K / 16) + k / 16]) *
         (double)w->ts[e];
}

/* ---------------- router: article section "Mixture of Experts" ---------------- */

/* Logits in FP32 from exact bf16 x and fp32 W_r (sum in double, rounded once),
 * then the sigmoid score of every expert, rounded to FP32. */
void oracle_router_scores(int T, int d, int E, const uint16_t* x, const float* wr, float* logits,
                          float* scores) {
#pragma omp parallel
  {
    double* acc = (double*)malloc(sizeof(double) * (size_t)E);
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      for (int e = 0; e < E; ++e) acc[e] = 0.0;
      for (int j = 0; j < d; ++j) {
        const double xj = bf16_value(x[(int64_t)t * d + j]);
        const float* wrow = wr + (int64_t)j * E;
        for (int e = 0; e < E; ++e) acc[e] += xj * (double)wrow[e];
      }
      for (int e = 0; e < E; ++e) {
        const float l = (float)acc[e];
        if (logits) logits[(int64_t)t * E + e] = l;
        scores[(int64_t)t * E + e] = (float)(1.0 / (1.0 + exp(-(double)l)));
      }
    }
    free(acc);
  }
}

/* Group-limited top-k selection for one token.
 *   selection score = s, or s + bias[e] (FP32 add) with a per-expert bias:
 *                  the balancing bias of DeepSeek-V3's router, which the
 *                  article's router follows; it steers the choice only
 *   group score  = sum of the two largest selection scores in the group (FP32 add)
 *   kept groups  = the topk_groups best group scores
 *   chosen       = the top_k best selection scores among experts of kept groups
 *   weight       = routed_scale * s / (sum of chosen s)   (unbiased scores)
 * Ties: lower index first. Slots are in descending selection-score order.
 * margin_group  = (worst kept group score) - (best dropped group score)
 * margin_expert = (worst chosen selection score) - (best unchosen candidate's)
 * (+INFINITY when nothing was dropped). Returns 0, or 1 if the score sum is 0. */
static int select_one(int E, int G, int Gk, int K, double scale, const float* s, const float* bias,
                      int32_t* idx, double* w, float* gs, double* mg, double* me) {
  const int gsz = E / G;
  float sel[1024];
  for (int e = 0; e < E; ++e) sel[e] = bias ? s[e] + bias[e] : s[e];
  for (int g = 0; g < G; ++g) {
    int b1 = -1, b2 = -1;
    for (int e = g * gsz; e < (g + 1) * gsz; ++e) {
      if (b1 < 0 || sel[e] > sel[b1]) { b2 = b1; b1 = e; }
      else if (b2 < 0 || sel[e] > sel[b2]) { b2 = e; }
    }
    gs[g] = (gsz >= 2) ? (sel[b1] + sel[b2]) : sel[b1];
  }
  char kept[64] = {0};
  int last_kept = -1;
  for (int r = 0; r < Gk; ++r) {
    int best = -1;
    for (int g = 0; g < G; ++g)
      if (!kept[g] && (best < 0 || gs[g] > gs[best])) best = g;
    kept[best] = 1;
    last_kept = best;
  }
  int best_dropped = -1;
  for (int g = 0; g < G; ++g)
    if (!kept[g] && (best_dropped < 0 || gs[g] > gs[best_dropped])) best_dropped = g;
  *mg = (best_dropped < 0) ? INFINITY : (double)gs[last_kept] - (double)gs[best_dropped];

  char taken[1024] = {0};
  double sum = 0.0;
  for (int k = 0; k < K; ++k) {
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (kept[e / gsz] && !taken[e] && (best < 0 || sel[e] > sel[best])) best = e;
    taken[best] = 1;
    idx[k] = best;
    sum += (double)s[best];
  }
  int best_left = -1;
  for (int e = 0; e < E; ++e)
    if (kept[e / gsz] && !taken[e] && (best_left < 0 || sel[e] > sel[best_left])) best_left = e;
  *me = (best_left < 0) ? INFINITY : (double)sel[idx[K - 1]] - (double)sel[best_left];
  if (sum == 0.0) {
    for (int k = 0; k < K; ++k) w[k] = 0.0;
    return 1;
  }
  for (int k = 0; k < K; ++k) w[k] = scale * (double)s[idx[k]] / sum;
  return 0;
}

/* Selection for T tokens from their FP32 scores and an optional per-expert
 * selection bias [E] (NULL: none). Output arrays are [T][K] (idx, w), [T][G]
 * (gscores, nullable), [T] (margins, nullable). Returns the number of tokens
 * whose chosen scores summed to zero. */
int oracle_select_biased(int T, int E, int G, int Gk, int K, double scale, const float* scores,
                         const float* bias, int32_t* idx, double* w, float* gscores, double* margin_group,
                         double* margin_expert) {
  if (E <= 0 || G <= 0 || E % G || G > 64 || E > 1024 || Gk < 1 || Gk > G || K < 1 ||
      K > Gk * (E / G))
    return -1;
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : bad)
  for (int t = 0; t < T; ++t) {
    float gs[64];
    double mg, me;
    bad += select_one(E, G, Gk, K, scale, scores + (int64_t)t * E, bias, idx + (int64_t)t * K,
                      w + (int64_t)t * K, gs, &mg, &me);
    if (gscores)
      for (int g = 0; g < G; ++g) gscores[(int64_t)t * G + g] = gs[g];
    if (margin_group) margin_group[t] = mg;
    if (margin_expert) margin_expert[t] = me;
  }
  return bad;
}

int oracle_select(int T, int E, int G, int Gk, int K, double scale, const float* scores,
                  int32_t* idx, double* w, float* gscores, double* margin_group,
                  double* margin_expert) {
  return oracle_select_biased(T, E, G, Gk, K, scale, scores, NULL, idx, w, gscores, margin_group,
                              margin_expert);
}

/* ---------------- permutation (grouping of token slots by expert) ---------------- */

/* Rows sorted by (expert, token): row r of expert e holds the r-th smallest
 * token that chose e. counts[E], offsets[E+1], row_token[T*K],
 * inv_row[T*K] (inv_row[t*K+k] = row of token t's slot k). */
void oracle_permute(int T, int E, int K, const int32_t* idx, int32_t* counts, int32_t* offsets,
                    int32_t* row_token, int32_t* inv_row) {
  int32_t r = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = r;
    for (int t = 0; t < T; ++t)
      for (int k = 0; k < K; ++k)
        if (idx[(int64_t)t * K + k] == e) {
          row_token[r] = t;
          inv_row[(int64_t)t * K + k] = r;
          ++r;
        }
    counts[e] = r - offsets[e];
  }
  offsets[E] = r;
}

/* ---------------- expert SwiGLU MLP: article section "Mixture of Experts" ---------------- */

/* One row through expert e: g = x.Wg, u = x.Wu (double sums of exact
 * operands), h = silu(g) * u formed in FP32 and rounded to bf16, y = h.Wd in
 * double. h_out (bf16 bits, [I]) is optional. */
static void ffn_row(int d, int I, int e, const uint16_t* xr, const wmat* gate, const wmat* up,
                    const wmat* down, uint16_t* h_out, double* y, double* xbuf, double* hbuf) {
  for (int j = 0; j < d; ++j) xbuf[j] = bf16_value(xr[j]);
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int j = 0; j < d; ++j) {
      g += xbuf[j] * wmat_at(gate, e, i, j);
      u += xbuf[j] * wmat_at(up, e, i, j);
    }
    const float gf = (float)g, uf = (float)u;
    const float silu = (float)((double)gf / (1.0 + exp(-(double)gf)));
    const uint16_t hb = bf16_round(silu * uf);
    if (h_out) h_out[i] = hb;
    hbuf[i] = bf16_value(hb);
  }
  for (int n = 0; n < d; ++n) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += hbuf[i] * wmat_at(down, e, n, i);
    y[n] = acc;
  }
}

static void make_wmats(int d, int I, int wfmt, const void* gate, const void* up, const void* down,
                       const uint8_t* gate_sf, const uint8_t* up_sf, const uint8_t* down_sf,
                       const float* gate_ts, const float* up_ts, const float* down_ts, wmat* G,
                       wmat* U, wmat* D) {
  const wmat g = {wfmt, (const uint16_t*)gate, (const uint8_t*)gate, gate_sf, gate_ts, I, d};
  const wmat u = {wfmt, (const uint16_t*)up, (const uint8_t*)up, up_sf, up_ts, I, d};
  const wmat dn = {wfmt, (const uint16_t*)down, (const uint8_t*)down, down_sf, down_ts, d, I};
  *G = g;
  *U = u;
  *D = dn;
}

/* Expert FFN over n independent rows: row r goes through expert row_expert[r].
 * xrows [n][d] bf16; h_out [n][I] bf16 (nullable); y_out [n][d] double. */
void oracle_ffn_rows(int n, int d, int I, int wfmt, const int32_t* row_expert,
                     const uint16_t* xrows, const void* gate, const void* up, const void* down,
                     const uint8_t* gate_sf, const uint8_t* up_sf, const uint8_t* down_sf,
                     const float* gate_ts, const float* up_ts, const float* down_ts,
                     uint16_t* h_out, double* y_out) {
  wmat G, U, D;
  make_wmats(d, I, wfmt, gate, up, down, gate_sf, up_sf, down_sf, gate_ts, up_ts, down_ts, &G, &U,
             &D);
#pragma omp parallel
  {
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)d);
    double* hbuf = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r)
      ffn_row(d, I, row_expert[r], xrows + (int64_t)r * d, &G, &U, &D,
              h_out ? h_out + (int64_t)r * I : NULL, y_out + (int64_t)r * d, xbuf, hbuf);
    free(xbuf);
    free(hbuf);
  }
}

/* ---------------- combine: article section "Mixture of Experts" ---------------- */

/* out[t] = sum_k w[t][k] * y[inv_row[t*K+k]] in double, slot order. The
 * routed scale (2.5) is already inside w. y rows are fp32 [R][d]. */
void oracle_combine(int T, int K, int d, const float* y, const int32_t* inv_row, const double* w,
                    double* out) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k)
        acc += w[(int64_t)t * K + k] * (double)y[(int64_t)inv_row[(int64_t)t * K + k] * d + c];
      out[(int64_t)t * d + c] = acc;
    }
}

/* ---------------- block forward for a subset of tokens ---------------- */

/* out[i] = sum_k w[t][k] * SwiGLU_{idx[t][k]}(x[t]) for t = tokens[i], using
 * the given routing (idx, w are [T][K]); out is [n_sel][d] double. */
void oracle_forward_tokens(int d, int I, int K, int wfmt, const uint16_t* x, const int32_t* idx,
                           const double* w, int n_sel, const int32_t* tokens, const void* gate,
                           const void* up, const void* down, const uint8_t* gate_sf,
                           const uint8_t* up_sf, const uint8_t* down_sf, const float* gate_ts,
                           const float* up_ts, const float* down_ts, double* out) {
  wmat G, U, D;
  make_wmats(d, I, wfmt, gate, up, down, gate_sf, up_sf, down_sf, gate_ts, up_ts, down_ts, &G, &U,
             &D);
  double* y = (double*)malloc(sizeof(double) * (size_t)n_sel * K * d);
#pragma omp parallel
  {
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)d);
    double* hbuf = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
    for (int p = 0; p < n_sel * K; ++p) {
      const int i = p / K, k = p % K, t = tokens[i];
      ffn_row(d, I, idx[(int64_t)t * K + k], x + (int64_t)t * d, &G, &U, &D, NULL,
              y + (int64_t)p * d, xbuf, hbuf);
    }
    free(xbuf);
    free(hbuf);
  }
  for (int i = 0; i < n_sel; ++i) {
    const int t = tokens[i];
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += w[(int64_t)t * K + k] * y[((int64_t)i * K + k) * d + c];
      out[(int64_t)i * d + c] = acc;
    }
  }
  free(y);
}

/* ---------------- residual update: article section "Residual stream" ---------------- */

/* Post-norm and depth-scaled residual addition of one sublayer output, per
 * token row t (the article: every sublayer is normalised before and after; at
 * step k the sublayer output is added with weight 1/sqrt(k) and the existing
 * stream kept with weight sqrt((k-1)/k); the norms are computed in FP32 --
 * here in double, the exact value):
 *   r       = sqrt(mean_c(out[t][c]^2) + eps)
 *   normed  = out[t][c] / r * gamma[c]                    (RMSNorm)
 *   h_new   = sqrt((k-1)/k) * h_old[t][c] + (1/sqrt(k)) * normed
 * out [T][d] double (the sublayer output), h_old [T][d] bf16 bits, gamma [d]
 * bf16 bits, h_new [T][d] double. k >= 1 (k = 1 keeps nothing of h_old). */
void oracle_residual_update(int T, int d, const double* out, const uint16_t* h_old, const uint16_t* gamma,
                            double eps, int k, double* h_new) {
  const double keep = sqrt((double)(k - 1) / (double)k), add = 1.0 / sqrt((double)k);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const double* o = out + (int64_t)t * d;
    double ss = 0.0;
    for (int c = 0; c < d; ++c) ss += o[c] * o[c];
    const double r = sqrt(ss / d + eps);
    for (int c = 0; c < d; ++c)
      h_new[(int64_t)t * d + c] =
          keep * bf16_value(h_old[(int64_t)t * d + c]) + add * (o[c] / r * bf16_value(gamma[c]));
  }
}

/* Pre-norm of the sublayer input, per token row t (the article: every sublayer
 * is normalised before and after, the norms in FP32): the exact RMSNorm value
 * is rounded to FP32, then to bf16, the dtype the block takes as x:
 *   r       = sqrt(mean_c(h[t][c]^2) + eps)
 *   x[t][c] = bf16( fp32( h[t][c] / r * gamma[c] ) )
 * h [T][d] bf16 bits (the residual stream), gamma [d] bf16 bits, x [T][d] bf16
 * bits. */
void oracle_pre_norm(int T, int d, const uint16_t* h, const uint16_t* gamma, double eps, uint16_t* x) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const uint16_t* row = h + (int64_t)t * d;
    double ss = 0.0;
    for (int c = 0; c < d; ++c) ss += bf16_value(row[c]) * bf16_value(row[c]);
    const double r = sqrt(ss / d + eps);
    for (int c = 0; c < d; ++c)
      x[(int64_t)t * d + c] = bf16_round((float)(bf16_value(row[c]) / r * bf16_value(gamma[c])));
  }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
