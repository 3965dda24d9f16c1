/*
 * Plain CPU oracle for decode-phase sparse attention over a hierarchically
 * paged KV cache (LServe-style unified sparse attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library) shares no code, header, table or helper with it.
 *
 * The oracle works on LOGICAL token positions only: the caller hands it the
 * key/value rows of one kv head as a dense [L][d] array of the exact 16-bit
 * values (fp16 or bf16 bit patterns), so the physical page layout never
 * enters it.  Every function is a direct transcription of a definition:
 *
 *   - page min/max metadata   "LServe long-sequence LLM serving system",
 *                             section 2.1 (dynamic sparsity: min-max pooling
 *                             of each text block during prefill) and 2.2
 *                             (logical pages of 16-64 tokens).
 *   - page score              section 2.1 (query similarity to the pooled
 *                             features); the formula sum_d max(q_d*kmax_d,
 *                             q_d*kmin_d) is the query-aware block estimate
 *                             listed as "Quest" in the sparse-attention
 *                             table of "Long-context inference optimization
 *                             for LLMs", section 2.2.
 *   - budget / top-k          LServe write-up, section 2.1 (fixed KV token
 *                             budget, default 4096) and section 3.2
 *                             (dynamic budget min(4096, length/32)).
 *   - attended token sets     LServe write-up, section 2.1 (streaming heads:
 *                             local context) and the StreamingLLM row
 *                             (attention sink + local window) of the
 *                             sparse-attention table, survey section 2.2.
 *   - attention               softmax(q k^T / sqrt(d)) v restricted to the
 *                             attended set; scale as in the GQA example of
 *                             the survey, section 2.3.  Two passes, no
 *                             online rescaling, fp64 accumulation.
 *
 * Precision: attention is computed in fp64.  Page scores decide an integer
 * result (which pages are kept), so they are computed in fp32, the precision
 * the GPU path takes that decision in, summing channels in increasing order.
 * An fp64 twin of the score exists for the upper-bound pin.
 *
 * Compile with -ffp-contract=off so that results do not depend on whether
 * the host compiler fuses multiply-adds.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F16 0
#define ORC_BF16 1
#define ORC_E4M3 2 /* fp8 KV storage: the low byte holds an e4m3 code */

/* ---- exact decoding of the 16-bit storage formats --------------------- */

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double orc_f16_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25); /* (1.m) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
static double orc_bf16_value(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int m = b & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)m, -133); /* subnormal: m * 2^-126 * 2^-7 */
  else if (e == 255)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x80), e - 134); /* (1.m) * 2^(e-127) */
  return sign ? -v : v;
}

/* OCP fp8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 fraction bits; no
 * infinities, exponent 15 with fraction 7 is NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_value(unsigned code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xf;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp((double)(m | 8), e - 10); /* (1.m) * 2^(e-7) */
  return sign ? -v : v;
}

double orc_value(uint16_t bits, int dtype) {
  if (dtype == ORC_E4M3) return orc_e4m3_value(bits & 0xffu);
  return dtype == ORC_BF16 ? orc_bf16_value(bits) : orc_f16_value(bits);
}

/*
 * fp32 -> e4m3 code: round to nearest, ties to even fraction, saturating:
 * magnitudes that round beyond 448 (and infinities) become 448; NaN becomes
 * the NaN code.  Written from the format: for |x| below the smallest normal
 * 2^-6 the code counts multiples of 2^-9; above, (exponent + 7, fraction
 * rounded to 3 bits), a fraction that rounds up to 8 carrying into the
 * exponent.
 */
unsigned orc_e4m3_from_float(float x) {
  unsigned sign = signbit(x) ? 0x80u : 0u;
  double a = fabs((double)x);
  if (isnan(x)) return sign | 0x7fu;
  if (a >= 448.0) return sign | 0x7eu;
  if (a < ldexp(1.0, -6)) {
    double m = rint(a * 512.0); /* exact scaling; rint: ties to even */
    return sign | (unsigned)m;  /* m = 8 is the smallest normal's code */
  }
  int e = ilogb(a);                      /* 2^e <= a < 2^(e+1), e in [-6, 8] */
  double f = rint((ldexp(a, -e) - 1.0) * 8.0);  /* fraction, 0..8 */
  if (f == 8.0) {
    f = 0.0;
    e += 1;
  }
  unsigned code = (unsigned)((e + 7) << 3) | (unsigned)f;
  return sign | (code > 0x7eu ? 0x7eu : code);
}

/*
 * fp8 KV quantisation of n 16-bit values x (dtype) with a positive scale:
 * code_i = e4m3(fl32(x_i / scale)), the division rounded once to fp32, so
 * that the stored value is code * scale.  Codes go to the low byte of
 * codes[i].
 */
void orc_quantize_e4m3(const uint16_t *x, int dtype, long n, float scale, uint16_t *codes) {
  for (long i = 0; i < n; ++i) {
    float xv = (float)orc_value(x[i], dtype); /* exact: 16-bit values fit in fp32 */
    volatile float t = xv / scale;            /* one fp32 division */
    codes[i] = (uint16_t)orc_e4m3_from_float(t);
  }
}

void orc_decode(const uint16_t *in, int dtype, long n, double *out) {
  for (long i = 0; i < n; ++i) out[i] = orc_value(in[i], dtype);
}

/* ---- (metadata) per logical page, per channel min and max of the keys --- */

/*
 * K is [L][d] (one kv head, logical positions).  For logical pages
 * j in [j0, j1) the page holds tokens [j*ell, min((j+1)*ell, L)); only those
 * valid tokens are reduced (a partially filled last page reduces over what
 * it holds).  Outputs are the original 16-bit patterns of the minimum and
 * maximum element, rows [j - j0] of kmin/kmax ([j1-j0][d]).  Among equal
 * values the first token wins, so +0/-0 ties keep the earlier token's bits.
 * Returns 0, or -1 on a bad argument.
 */
int orc_page_minmax(const uint16_t *K, int dtype, int L, int d, int ell, int j0,
                    int j1, uint16_t *kmin, uint16_t *kmax) {
  if (L <= 0 || d <= 0 || ell <= 0 || j0 < 0 || j1 < j0) return -1;
  if ((long)j1 * ell >= (long)L + ell) return -1; /* page j1-1 must hold a token */
  for (int j = j0; j < j1; ++j) {
    int t0 = j * ell;
    int t1 = t0 + ell < L ? t0 + ell : L;
    for (int c = 0; c < d; ++c) {
      uint16_t bmin = K[(long)t0 * d + c], bmax = bmin;
      double vmin = orc_value(bmin, dtype), vmax = vmin;
      for (int t = t0 + 1; t < t1; ++t) {
        uint16_t b = K[(long)t * d + c];
        double v = orc_value(b, dtype);
        if (v < vmin) { vmin = v; bmin = b; }
        if (v > vmax) { vmax = v; bmax = b; }
      }
      kmin[(long)(j - j0) * d + c] = bmin;
      kmax[(long)(j - j0) * d + c] = bmax;
    }
  }
  return 0;
}

/* ---- (score) query-aware page score ------------------------------------ */

/*
 * q is [G][d]: the G query heads that share this kv head.  kmin/kmax are
 * [nL][d], stored as kv_dtype codes of value / kscale (kscale = 1 for 16-bit
 * keys; fp8 keys carry their kv head's scale).  For each page j and head h
 *     s_h(j) = sum_{c=0}^{d-1} max(q_h[c]*kmax_j[c], q_h[c]*kmin_j[c])
 * summed in increasing c, in fp32; the kv-head score is the maximum over
 * the group, S(j) = max_h s_h(j).  Scores are not scaled by 1/sqrt(d): a
 * positive scale does not change the ranking.
 */
void orc_page_scores_f32_kv(const uint16_t *q, int q_dtype, const uint16_t *kmin,
                            const uint16_t *kmax, int kv_dtype, double kscale, int nL, int G,
                            int d, float *S) {
  for (int j = 0; j < nL; ++j) {
    float best = -INFINITY;
    for (int h = 0; h < G; ++h) {
      float acc = 0.0f;
      for (int c = 0; c < d; ++c) {
        float qv = (float)orc_value(q[(long)h * d + c], q_dtype);
        float a = qv * (float)(kscale * orc_value(kmax[(long)j * d + c], kv_dtype));
        float b = qv * (float)(kscale * orc_value(kmin[(long)j * d + c], kv_dtype));
        acc = acc + (a > b ? a : b);
      }
      if (acc > best || h == 0) best = acc;
    }
    S[j] = best;
  }
}

/* q and the keys in one 16-bit dtype, no scale. */
void orc_page_scores_f32(const uint16_t *q, const uint16_t *kmin,
                         const uint16_t *kmax, int dtype, int nL, int G, int d,
                         float *S) {
  orc_page_scores_f32_kv(q, dtype, kmin, kmax, dtype, 1.0, nL, G, d, S);
}

/* The same score in fp64 (per head, not reduced over the group): [G][nL]. */
void orc_page_scores_f64_kv(const uint16_t *q, int q_dtype, const uint16_t *kmin,
                            const uint16_t *kmax, int kv_dtype, double kscale, int nL, int G,
                            int d, double *s) {
  for (int h = 0; h < G; ++h)
    for (int j = 0; j < nL; ++j) {
      double acc = 0.0;
      for (int c = 0; c < d; ++c) {
        double qv = orc_value(q[(long)h * d + c], q_dtype);
        double a = qv * (kscale * orc_value(kmax[(long)j * d + c], kv_dtype));
        double b = qv * (kscale * orc_value(kmin[(long)j * d + c], kv_dtype));
        acc += a > b ? a : b;
      }
      s[(long)h * nL + j] = acc;
    }
}

void orc_page_scores_f64(const uint16_t *q, const uint16_t *kmin,
                         const uint16_t *kmax, int dtype, int nL, int G, int d,
                         double *s) {
  orc_page_scores_f64_kv(q, dtype, kmin, kmax, dtype, 1.0, nL, G, d, s);
}

/* ---- (budget, top-k) --------------------------------------------------- */

/*
 * Pages kept per dynamic head.  budget = token_budget if positive, else
 * min(4096, floor(L/32)) tokens; K_sel = max(1, floor(budget/ell)).
 */
int orc_budget_pages(long L, int token_budget, int ell) {
  long budget = token_budget > 0 ? token_budget : (L / 32 < 4096 ? L / 32 : 4096);
  long k = budget / ell;
  return k < 1 ? 1 : (int)k;
}

typedef struct {
  float s;
  int j;
} orc_scored;

/* Order: higher score first; equal scores -> lower page index first.  A NaN
 * score counts as lower than every number. */
static int orc_cmp_scored(const void *pa, const void *pb) {
  const orc_scored *a = (const orc_scored *)pa, *b = (const orc_scored *)pb;
  int an = isnan(a->s), bn = isnan(b->s);
  if (an != bn) return an ? 1 : -1;
  if (!an && a->s != b->s) return a->s > b->s ? -1 : 1;
  return a->j < b->j ? -1 : (a->j > b->j ? 1 : 0);
}

static int orc_cmp_int(const void *pa, const void *pb) {
  int a = *(const int *)pa, b = *(const int *)pb;
  return a < b ? -1 : (a > b ? 1 : 0);
}

/*
 * Selection over nL logical pages with scores S[nL] (S[nL-1] is not read).
 * If nL <= K_sel every page is kept.  Otherwise the page holding the newest
 * token, nL-1, is always kept and counts against K_sel, and the other
 * K_sel-1 are the best of pages [0, nL-1) by (score desc, index asc).
 * Output sel[] ascending.  Returns the count, or -1 on a bad argument.
 */
int orc_select(const float *S, int nL, int K_sel, int *sel) {
  if (nL <= 0 || K_sel < 1) return -1;
  if (nL <= K_sel) {
    for (int j = 0; j < nL; ++j) sel[j] = j;
    return nL;
  }
  int n = nL - 1;
  orc_scored *cand = (orc_scored *)malloc(sizeof(orc_scored) * (size_t)n);
  if (!cand) return -1;
  for (int j = 0; j < n; ++j) {
    cand[j].s = S[j];
    cand[j].j = j;
  }
  qsort(cand, (size_t)n, sizeof(orc_scored), orc_cmp_scored);
  for (int i = 0; i < K_sel - 1; ++i) sel[i] = cand[i].j;
  sel[K_sel - 1] = nL - 1;
  free(cand);
  qsort(sel, (size_t)K_sel, sizeof(int), orc_cmp_int);
  return K_sel;
}

/* ---- attended token sets ----------------------------------------------- */

/*
 * Dynamic head: the union of the selected pages and the pages that came
 * into existence since the selection was taken, [nL0-1, nL) with
 * nL = ceil(L/ell); every token t < L of those pages, ascending.
 * Returns the count (out must hold L entries), or -1 on a bad argument.
 */
int orc_dynamic_tokens(const int *sel, int count, int nL0, long L, int ell,
                       int *out) {
  if (L <= 0 || ell <= 0 || nL0 < 1) return -1;
  long nL = (L + ell - 1) / ell;
  unsigned char *keep = (unsigned char *)calloc((size_t)nL, 1);
  if (!keep) return -1;
  for (int i = 0; i < count; ++i) {
    if (sel[i] < 0 || sel[i] >= nL) {
      free(keep);
      return -1;
    }
    keep[sel[i]] = 1;
  }
  for (long j = nL0 - 1; j < nL; ++j) keep[j] = 1;
  int n = 0;
  for (long t = 0; t < L; ++t)
    if (keep[t / ell]) out[n++] = (int)t;
  free(keep);
  return n;
}

/*
 * Streaming head: sink tokens t < S and the local window t >= L-W (the
 * window includes the newest token), each position once.  Returns count.
 */
int orc_streaming_tokens(long L, int S, int W, int *out) {
  int n = 0;
  for (long t = 0; t < L; ++t)
    if (t < S || t >= L - W) out[n++] = (int)t;
  return n;
}

/* ---- attention ---------------------------------------------------------- */

/*
 * q [G][d] (q_dtype), K and V [L][d] of one kv head as kv_dtype codes whose
 * values are code * kscale (keys) and code * vscale (values) -- 1 for 16-bit
 * storage; tokens[n] are positions into K/V.
 * For each head g:  z_i = (q_g . k_{t_i}) / sqrt(d);  m = max_i z_i;
 *   out_g = sum_i exp(z_i - m) v_{t_i} / sum_i exp(z_i - m)   (fp64).
 * Returns 0, or -1 if n <= 0 or scratch cannot be allocated.
 */
int orc_attention_kv(const uint16_t *q, int q_dtype, const uint16_t *K, const uint16_t *V,
                     int kv_dtype, double kscale, double vscale, int G, int d,
                     const int *tokens, int n, double *out) {
  if (n <= 0) return -1;
  double *z = (double *)malloc(sizeof(double) * (size_t)n);
  double *qd = (double *)malloc(sizeof(double) * (size_t)d);
  if (!z || !qd) {
    free(z);
    free(qd);
    return -1;
  }
  double scale = 1.0 / sqrt((double)d);
  for (int g = 0; g < G; ++g) {
    for (int c = 0; c < d; ++c) qd[c] = orc_value(q[(long)g * d + c], q_dtype);
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) {
      const uint16_t *k = K + (long)tokens[i] * d;
      double dot = 0.0;
      for (int c = 0; c < d; ++c) dot += qd[c] * (kscale * orc_value(k[c], kv_dtype));
      z[i] = dot * scale;
      if (z[i] > m) m = z[i];
    }
    double den = 0.0;
    for (int i = 0; i < n; ++i) {
      z[i] = exp(z[i] - m);
      den += z[i];
    }
    double *o = out + (long)g * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int i = 0; i < n; ++i) {
      const uint16_t *v = V + (long)tokens[i] * d;
      for (int c = 0; c < d; ++c) o[c] += z[i] * (vscale * orc_value(v[c], kv_dtype));
    }
    for (int c = 0; c < d; ++c) o[c] /= den;
  }
  free(z);
  free(qd);
  return 0;
}

int orc_attention(const uint16_t *q, const uint16_t *K, const uint16_t *V,
                  int dtype, int G, int d, const int *tokens, int n,
                  double *out) {
  return orc_attention_kv(q, dtype, K, V, dtype, 1.0, 1.0, G, d, tokens, n, out);
}

/*
 * Softmax statistics a split FlashAttention exports alongside its partial
 * output (the row max and row sum; Novita KV-sparsity article, "attention
 * mechanism modifications"), over the same logits as orc_attention:
 *   z_i = q_g . k_{t_i} / sqrt(d),  row_max_g = max_i z_i,
 *   row_sum_g = sum_i exp(z_i - row_max_g)          (fp64).
 * Returns 0, or -1 if n <= 0.
 */
int orc_softmax_stats_kv(const uint16_t *q, int q_dtype, const uint16_t *K, int kv_dtype,
                         double kscale, int G, int d, const int *tokens, int n,
                         double *row_max, double *row_sum) {
  if (n <= 0) return -1;
  double scale = 1.0 / sqrt((double)d);
  for (int g = 0; g < G; ++g) {
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) {
      const uint16_t *k = K + (long)tokens[i] * d;
      double dot = 0.0;
      for (int c = 0; c < d; ++c)
        dot += orc_value(q[(long)g * d + c], q_dtype) * (kscale * orc_value(k[c], kv_dtype));
      if (dot * scale > m) m = dot * scale;
    }
    double sum = 0.0;
    for (int i = 0; i < n; ++i) {
      const uint16_t *k = K + (long)tokens[i] * d;
      double dot = 0.0;
      for (int c = 0; c < d; ++c)
        dot += orc_value(q[(long)g * d + c], q_dtype) * (kscale * orc_value(k[c], kv_dtype));
      sum += exp(dot * scale - m);
    }
    row_max[g] = m;
    row_sum[g] = sum;
  }
  return 0;
}

int orc_softmax_stats(const uint16_t *q, const uint16_t *K, int dtype, int G, int d,
                      const int *tokens, int n, double *row_max, double *row_sum) {
  return orc_softmax_stats_kv(q, dtype, K, dtype, 1.0, G, d, tokens, n, row_max, row_sum);
}


/*
 * Per-page attention mass (the third statistic of the same export: how much
 * of each head's softmax weight falls on each attended logical page -- the
 * eviction-style importance a modified FlashAttention can report; Novita
 * KV-sparsity article, "attention mechanism modifications").  Same logits as
 * orc_attention:
 *   z_i = q_g . k_{t_i} / sqrt(d),  w_i = exp(z_i - max z) / sum exp(z - max z),
 *   mass[g][k] = sum of w_i over the tokens t_i of logical page pages[k]
 *                (t_i / ell == pages[k]).
 * A token on a page missing from `pages` counts in no entry.  fp64, two
 * passes.  Returns 0, or -1 if n <= 0 or out of memory.
 */
int orc_page_mass_kv(const uint16_t *q, int q_dtype, const uint16_t *K, int kv_dtype,
                     double kscale, int G, int d, const int *tokens, int n, int ell,
                     const int *pages, int n_pages, double *mass) {
  if (n <= 0) return -1;
  double *w = (double *)malloc(sizeof(double) * (size_t)n);
  if (!w) return -1;
  const double scale = 1.0 / sqrt((double)d);
  for (int g = 0; g < G; ++g) {
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) {
      const uint16_t *k = K + (long)tokens[i] * d;
      double dot = 0.0;
      for (int c = 0; c < d; ++c)
        dot += orc_value(q[(long)g * d + c], q_dtype) * (kscale * orc_value(k[c], kv_dtype));
      w[i] = dot * scale;
      if (w[i] > m) m = w[i];
    }
    double den = 0.0;
    for (int i = 0; i < n; ++i) {
      w[i] = exp(w[i] - m);
      den += w[i];
    }
    for (int k = 0; k < n_pages; ++k) {
      double acc = 0.0;
      for (int i = 0; i < n; ++i)
        if (tokens[i] / ell == pages[k]) acc += w[i];
      mass[(long)g * n_pages + k] = acc / den;
    }
  }
  free(w);
  return 0;
}

int orc_page_mass(const uint16_t *q, const uint16_t *K, int dtype, int G, int d,
                  const int *tokens, int n, int ell, const int *pages, int n_pages,
                  double *mass) {
  return orc_page_mass_kv(q, dtype, K, dtype, 1.0, G, d, tokens, n, ell, pages, n_pages, mass);
}

/* ---- (prefill) low-rank block importance ------------------------------- */

/*
 * Block importance for prefill ("LServe long-sequence LLM serving system",
 * section 3.1): Score(Q, K_i) ~ (Q W_q)(K_i W_k)^T / sqrt(d), with low-rank
 * projections W_q, W_k of d x r (r = d/8), estimated for every (query
 * block b, key block i) before exact attention runs on the chosen blocks.
 * Reading: the score of a block pair is the mean of the approximate logits
 * over its token pairs, and a kv head's score the maximum over its G query
 * heads.  The mean of a bilinear form over all pairs (t in b, u in i) is the
 * form of the two means, so the score is computed as
 *   s_g(b, i) = (mean_{t in b} q_{g,t} W_q) . (mean_{u in i} k_u W_k) / sqrt(d)
 * (the test-suite checks it against the pairwise mean on small inputs).
 * Q [G][L][d] (q_dtype), K [L][d] (kv_dtype codes, value = code * kscale),
 * W_q, W_k [d][r] fp32 row-major; blocks of `blk` tokens (the last may be
 * shorter).  Output S [nb][nb] (nb = ceil(L / blk)), S[b][i] for i <= b,
 * -inf above the diagonal (causal: a query block sees earlier blocks only).
 * fp64.  Returns 0, or -1 on a bad argument or out of memory.
 */
int orc_prefill_block_scores(const uint16_t *Q, int q_dtype, const uint16_t *K, int kv_dtype,
                             double kscale, const float *Wq, const float *Wk, int G, int d,
                             int r, int L, int blk, double *S) {
  if (L <= 0 || d <= 0 || r <= 0 || blk <= 0 || G <= 0) return -1;
  int nb = (L + blk - 1) / blk;
  double *qbar = (double *)calloc((size_t)G * nb * r, sizeof(double)); /* [G][nb][r] */
  double *kbar = (double *)calloc((size_t)nb * r, sizeof(double));     /* [nb][r] */
  if (!qbar || !kbar) {
    free(qbar);
    free(kbar);
    return -1;
  }
  for (int b = 0; b < nb; ++b) {
    int t0 = b * blk, t1 = t0 + blk < L ? t0 + blk : L;
    for (int t = t0; t < t1; ++t)
      for (int j = 0; j < r; ++j) {
        double kp = 0.0;
        for (int c = 0; c < d; ++c)
          kp += kscale * orc_value(K[(long)t * d + c], kv_dtype) * (double)Wk[(long)c * r + j];
        kbar[(long)b * r + j] += kp / (t1 - t0);
        for (int g = 0; g < G; ++g) {
          double qp = 0.0;
          for (int c = 0; c < d; ++c)
            qp += orc_value(Q[((long)g * L + t) * d + c], q_dtype) * (double)Wq[(long)c * r + j];
          qbar[((long)g * nb + b) * r + j] += qp / (t1 - t0);
        }
      }
  }
  double scale = 1.0 / sqrt((double)d);
  for (int b = 0; b < nb; ++b)
    for (int i = 0; i < nb; ++i) {
      double best = -INFINITY;
      if (i <= b)
        for (int g = 0; g < G; ++g) {
          double acc = 0.0;
          for (int j = 0; j < r; ++j) acc += qbar[((long)g * nb + b) * r + j] * kbar[(long)i * r + j];
          acc *= scale;
          if (acc > best) best = acc;
        }
      S[(long)b * nb + i] = best;
    }
  free(qbar);
  free(kbar);
  return 0;
}

/*
 * Block-sparse causal attention of a prompt for one kv head (LServe write-up,
 * section 3.1): query token t of each of the G heads attends the keys u <= t
 * of the key blocks chosen for its query block t / blk, blocks[offsets[b] ..
 * offsets[b+1]).  Per query token the two-pass fp64 softmax of
 * orc_attention_kv (same products, same order).  Q [G][L][d] (q_dtype), K
 * and V [L][d] (kv_dtype codes, values code * kscale / code * vscale), out
 * [G][L][d].  Returns 0, or -1 on a bad argument or out of memory.
 */
int orc_prefill_attention(const uint16_t *Q, int q_dtype, const uint16_t *K, const uint16_t *V,
                          int kv_dtype, double kscale, double vscale, int G, int d, int L,
                          int blk, const int *blocks, const int *offsets, double *out) {
  if (L <= 0 || d <= 0 || G <= 0 || blk <= 0) return -1;
  int nb = (L + blk - 1) / blk;
  double *kd = (double *)malloc(sizeof(double) * (size_t)L * d);
  double *vd = (double *)malloc(sizeof(double) * (size_t)L * d);
  double *qd = (double *)malloc(sizeof(double) * (size_t)d);
  double *z = (double *)malloc(sizeof(double) * (size_t)L);
  int *keys = (int *)malloc(sizeof(int) * (size_t)L);
  if (!kd || !vd || !qd || !z || !keys) {
    free(kd); free(vd); free(qd); free(z); free(keys);
    return -1;
  }
  for (long x = 0; x < (long)L * d; ++x) {
    kd[x] = kscale * orc_value(K[x], kv_dtype);
    vd[x] = vscale * orc_value(V[x], kv_dtype);
  }
  double scale = 1.0 / sqrt((double)d);
  for (int b = 0; b < nb; ++b) {
    for (int t = b * blk; t < L && t < (b + 1) * blk; ++t) {
      int n = 0;
      for (int e = offsets[b]; e < offsets[b + 1]; ++e) {
        int i = blocks[e];
        if (i < 0 || i >= nb) {
          free(kd); free(vd); free(qd); free(z); free(keys);
          return -1;
        }
        for (int u = i * blk; u < L && u < (i + 1) * blk && u <= t; ++u) keys[n++] = u;
      }
      for (int g = 0; g < G; ++g) {
        double *o = out + ((long)g * L + t) * d;
        for (int c = 0; c < d; ++c) qd[c] = orc_value(Q[((long)g * L + t) * d + c], q_dtype);
        double m = -INFINITY;
        for (int j = 0; j < n; ++j) {
          const double *k = kd + (long)keys[j] * d;
          double dot = 0.0;
          for (int c = 0; c < d; ++c) dot += qd[c] * k[c];
          z[j] = dot * scale;
          if (z[j] > m) m = z[j];
        }
        double den = 0.0;
        for (int j = 0; j < n; ++j) {
          z[j] = exp(z[j] - m);
          den += z[j];
        }
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int j = 0; j < n; ++j) {
          const double *v = vd + (long)keys[j] * d;
          for (int c = 0; c < d; ++c) o[c] += z[j] * v[c];
        }
        for (int c = 0; c < d; ++c) o[c] = n > 0 ? o[c] / den : 0.0;
      }
    }
  }
  free(kd); free(vd); free(qd); free(z); free(keys);
  return 0;
}
