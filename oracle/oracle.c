/*
 * oracle.c -- the plain CPU oracle of content-routed sparse attention.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA path never
 * calls it, shares no code with it and does not fall back to it.
 *
 * What it computes (double accumulation throughout, inputs widened exactly
 * from fp32 / bf16 / fp16):
 *
 *   The method is the one the superlinear release post describes under its
 *   key-idea section: the context is cut into O(L^0.5) spans, each query
 *   scores the candidate spans, keeps the top k and then runs token-level
 *   attention inside the chosen spans; the SubQ / SSA pages call the last
 *   step exact attention over a content-selected token subset.  The pages
 *   leave the router open ("learned routing"); this oracle uses the fixed
 *   router of the specification: a span's summary is the mean of its keys,
 *   its score is q . summary, and equal scores go to the lower span index.
 *
 *   1. spans: span j covers tokens [jS, min((j+1)S, L)).
 *   2. summary_j = mean of K over span j's valid tokens.
 *   3. a query at position t with head h has local span l = floor(t/S); its
 *      candidates are the complete spans 0 .. l-1.
 *   4. score_j = q . summary_j (no scale), in double.
 *   5. candidates are ordered by (score descending, j ascending); the first
 *      min(k, l) are kept and reported in ascending j, padded with -1.
 *   6. attended tokens T = union of the kept spans and [lS, t].
 *   7. x = scale * q . K_tau; w = exp(x - max x) / sum; O = sum w V_tau;
 *      lse = max x + ln sum exp(x - max x).
 *
 * Every function is a direct loop over that definition; there is no tiling,
 * no online softmax and no reordering beyond what the definition states.
 * The candidate sort is the C library's qsort.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2, ORACLE_F64 = 3 };

/* Exact widening of one stored element to double. */
static double load_f64(int dtype, const void* base, int64_t i) {
  if (dtype == ORACLE_F64) return ((const double*)base)[i];
  if (dtype == ORACLE_F32) return (double)((const float*)base)[i];
  uint16_t h = ((const uint16_t*)base)[i];
  if (dtype == ORACLE_BF16) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
  }
  /* IEEE binary16 */
  int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m + 1024), e - 25);
  return sign ? -v : v;
}

void oracle_set_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
}

int oracle_max_threads(void) { return omp_get_max_threads(); }

/*
 * Step 2 for spans [j0, j1) of every (b, kv-head).
 *   K    [B, Hkv, L_cap, d] (dtype), tokens 0 .. L-1 valid
 *   summ [B, Hkv, ns_cap, d] double; spans with no valid token are left alone
 */
void oracle_summaries(int dtype, const void* K, int B, int Hkv, int64_t L_cap, int64_t L, int d,
                      int S, int64_t j0, int64_t j1, double* summ, int64_t ns_cap) {
  int64_t nbh = (int64_t)B * Hkv;
  int64_t nj = j1 - j0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t w = 0; w < nbh * nj; ++w) {
    int64_t bh = w / nj, j = j0 + w % nj;
    int64_t t0 = j * S, t1 = t0 + S < L ? t0 + S : L;
    if (t1 <= t0) continue;
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int64_t t = t0; t < t1; ++t) acc += load_f64(dtype, K, (bh * L_cap + t) * d + c);
      summ[(bh * ns_cap + j) * d + c] = acc / (double)(t1 - t0);
    }
  }
}

typedef struct {
  double score;
  int32_t j;
} cand_t;

/* Step 5's order: score descending, then span index ascending. */
static int cand_order(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->j > y->j) - (x->j < y->j);
}

static int int_ascending(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* Decompose a row index of [B, Hq, n_q] into (b, h, i). */
static void row_coords(int64_t r, int Hq, int64_t n_q, int64_t* b, int64_t* h, int64_t* i) {
  *i = r % n_q;
  *h = (r / n_q) % Hq;
  *b = r / (n_q * Hq);
}

/*
 * Steps 3-5 for the rows of Q [B, Hq, n_q, d] (query i at q_pos0 + i).
 * rows == NULL: every row, outputs in row order; otherwise outputs are
 * compact in the order of rows[0 .. n_rows).
 *   sel    [n, topk] int32, ascending, -1 padded
 *   margin [n] double, nullable: score of the k-th minus the (k+1)-th kept
 *          candidate in step 5's order (+inf when l <= k)
 *   sel_score [n, topk] double, nullable: scores of the kept spans (NaN pad)
 * Returns 0, or -1 when a candidate span has no summary slot.
 */
int oracle_route(int dtype, const void* Q, int B, int Hq, int Hkv, int64_t n_q, int64_t q_pos0,
                 int d, int S, int topk, const double* summ, int64_t ns_cap, const int64_t* rows,
                 int64_t n_rows, int32_t* sel, double* margin, double* sel_score) {
  int g = Hq / Hkv;
  int64_t n = rows ? n_rows : (int64_t)B * Hq * n_q;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t o = 0; o < n; ++o) {
    int64_t r = rows ? rows[o] : o;
    int64_t b, h, i;
    row_coords(r, Hq, n_q, &b, &h, &i);
    int64_t t = q_pos0 + i;
    int64_t l = t / S;
    if (l > ns_cap) {
      bad = 1;
      continue;
    }
    int64_t kvh = b * Hkv + h / g;
    const int64_t qoff = r * d;
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(l > 0 ? l : 1));
    for (int64_t j = 0; j < l; ++j) {
      double acc = 0.0;
      for (int x = 0; x < d; ++x) acc += load_f64(dtype, Q, qoff + x) * summ[(kvh * ns_cap + j) * d + x];
      c[j].score = acc;
      c[j].j = (int32_t)j;
    }
    qsort(c, (size_t)l, sizeof(cand_t), cand_order);
    int64_t nsel = l < topk ? l : topk;
    int32_t* out = sel + o * topk;
    for (int64_t s = 0; s < nsel; ++s) out[s] = c[s].j;
    qsort(out, (size_t)nsel, sizeof(int32_t), int_ascending);
    for (int64_t s = nsel; s < topk; ++s) out[s] = -1;
    if (sel_score) {
      for (int64_t s = 0; s < topk; ++s) {
        double v = NAN;
        for (int64_t u = 0; u < nsel; ++u)
          if (c[u].j == out[s]) v = c[u].score;
        sel_score[o * topk + s] = v;
      }
    }
    if (margin) margin[o] = l > topk ? c[topk - 1].score - c[topk].score : INFINITY;
    free(c);
  }
  return bad ? -1 : 0;
}

/*
 * Group-shared selection (GQA): one selection per (b, kv-head, query), which
 * every query head of the group then uses.  The pages leave the router open;
 * this variant scores span j by the sum of the group's query heads' scores,
 *   score_j = sum over the g heads hh of kv-head h / g of q_hh . summary_j,
 * and keeps the top k under the same order (score desc, j asc) over the
 * same candidates as oracle_route.  Row convention and outputs as for
 * oracle_route: every head row of a group gets the group's selection.
 */
int oracle_route_group(int dtype, const void* Q, int B, int Hq, int Hkv, int64_t n_q, int64_t q_pos0,
                       int d, int S, int topk, const double* summ, int64_t ns_cap, const int64_t* rows,
                       int64_t n_rows, int32_t* sel, double* margin, double* sel_score) {
  int g = Hq / Hkv;
  int64_t n = rows ? n_rows : (int64_t)B * Hq * n_q;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t o = 0; o < n; ++o) {
    int64_t r = rows ? rows[o] : o;
    int64_t b, h, i;
    row_coords(r, Hq, n_q, &b, &h, &i);
    int64_t t = q_pos0 + i;
    int64_t l = t / S;
    if (l > ns_cap) {
      bad = 1;
      continue;
    }
    int64_t grp = h / g;
    int64_t kvh = b * Hkv + grp;
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(l > 0 ? l : 1));
    for (int64_t span = 0; span < l; ++span) {
      double sum = 0.0;  /* over the group's heads and the dimensions */
      for (int64_t hh = grp * g; hh < grp * g + g; ++hh) {
        const int64_t qoff = ((b * Hq + hh) * n_q + i) * d;
        for (int x = 0; x < d; ++x) sum += load_f64(dtype, Q, qoff + x) * summ[(kvh * ns_cap + span) * d + x];
      }
      c[span].score = sum;
      c[span].j = (int32_t)span;
    }
    qsort(c, (size_t)l, sizeof(cand_t), cand_order);
    int64_t nsel = l < topk ? l : topk;
    int32_t* out = sel + o * topk;
    for (int64_t s = 0; s < nsel; ++s) out[s] = c[s].j;
    qsort(out, (size_t)nsel, sizeof(int32_t), int_ascending);
    for (int64_t s = nsel; s < topk; ++s) out[s] = -1;
    if (sel_score) {
      for (int64_t s = 0; s < topk; ++s) {
        double v = NAN;
        for (int64_t u = 0; u < nsel; ++u)
          if (c[u].j == out[s]) v = c[u].score;
        sel_score[o * topk + s] = v;
      }
    }
    if (margin) margin[o] = l > topk ? c[topk - 1].score - c[topk].score : INFINITY;
    free(c);
  }
  return bad ? -1 : 0;
}

/*
 * Steps 6-7 for the rows of Q (same row convention as oracle_route).
 *   K, V [B, Hkv, L_cap, d]; sel [n, topk] as produced by step 5
 *   O    [n, d] double; lse [n] double; wsum [n] double (nullable): the sum
 *        of the softmax weights, which the definition makes 1
 * Returns 0, or -1 on a selected span that is not a complete span before
 * the query's local span.
 */
int oracle_attend(int dtype, const void* Q, const void* K, const void* V, int B, int Hq, int Hkv,
                  int64_t n_q, int64_t q_pos0, int64_t L_cap, int d, int S, int topk, double scale,
                  const int32_t* sel, const int64_t* rows, int64_t n_rows, double* O, double* lse,
                  double* wsum) {
  int g = Hq / Hkv;
  int64_t n = rows ? n_rows : (int64_t)B * Hq * n_q;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t o = 0; o < n; ++o) {
    int64_t r = rows ? rows[o] : o;
    int64_t b, h, i;
    row_coords(r, Hq, n_q, &b, &h, &i);
    int64_t t = q_pos0 + i;
    int64_t l = t / S;
    int64_t kvh = b * Hkv + h / g;
    const int32_t* js = sel + o * topk;
    /* step 6: the attended token positions */
    int64_t cap = (int64_t)topk * S + S;
    int64_t* tok = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
    int64_t nt = 0;
    for (int s = 0; s < topk; ++s) {
      int64_t j = js[s];
      if (j < 0) continue;
      if (j >= l) {
        bad = 1;
        continue;
      }
      for (int64_t tau = j * S; tau < (j + 1) * S; ++tau) tok[nt++] = tau;
    }
    for (int64_t tau = l * S; tau <= t; ++tau) tok[nt++] = tau;
    /* step 7 */
    double* x = (double*)malloc(sizeof(double) * (size_t)nt);
    double mx = -INFINITY;
    for (int64_t u = 0; u < nt; ++u) {
      double acc = 0.0;
      for (int c = 0; c < d; ++c)
        acc += load_f64(dtype, Q, r * d + c) * load_f64(dtype, K, (kvh * L_cap + tok[u]) * d + c);
      x[u] = scale * acc;
      if (x[u] > mx) mx = x[u];
    }
    double denom = 0.0;
    for (int64_t u = 0; u < nt; ++u) denom += exp(x[u] - mx);
    double ws = 0.0;
    for (int c = 0; c < d; ++c) O[o * d + c] = 0.0;
    for (int64_t u = 0; u < nt; ++u) {
      double wgt = exp(x[u] - mx) / denom;
      ws += wgt;
      for (int c = 0; c < d; ++c) O[o * d + c] += wgt * load_f64(dtype, V, (kvh * L_cap + tok[u]) * d + c);
    }
    lse[o] = mx + log(denom);
    if (wsum) wsum[o] = ws;
    free(x);
    free(tok);
  }
  return bad ? -1 : 0;
}

/*
 * 8-bit cache rows (the SubQ release post's quantisation plan: 8-bit / 4-bit
 * K / V so that a 1M-token cache fits a 24 GB card; the summaries stay fp32).
 * The pages fix no scheme; the plainest one is used: symmetric, one fp32
 * scale per (b, kv-head, token) row, round to nearest even.  For each of the
 * `rows` rows of d elements of X (dtype, widened exactly to fp32):
 *   amax = max |x_i|,  s = amax / 127 (fp32 division)
 *   q_i  = 0 if s == 0, else clamp(rint(x_i / s), -127, 127) (fp32 division)
 * The row's dequantised value is q_i * s.  Every step is fp32, as the
 * quantised code is an integer decided in floating point.
 */
void oracle_quantize_rows(int dtype, const void* X, int64_t rows, int d, int8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    float amax = 0.f;
    for (int c = 0; c < d; ++c) {
      const float x = (float)load_f64(dtype, X, r * d + c);
      const float a = fabsf(x);
      if (a > amax) amax = a;
    }
    const float s = amax / 127.0f;
    scale[r] = s;
    for (int c = 0; c < d; ++c) {
      int v = 0;
      if (s != 0.f) {
        const float x = (float)load_f64(dtype, X, r * d + c);
        float t = rintf(x / s);
        if (t > 127.f) t = 127.f;
        if (t < -127.f) t = -127.f;
        v = (int)t;
      }
      q[r * d + c] = (int8_t)v;
    }
  }
}

/*
 * 4-bit cache rows (the same quantisation plan of the SubQ release post, its
 * 4-bit half).  The same scheme with 15 levels: symmetric, one fp32 scale
 * per row, round to nearest even.  For each of the `rows` rows of d
 * elements of X:
 *   amax = max |x_i|,  s = amax / 7 (fp32 division)
 *   q_i  = 0 if s == 0, else clamp(rint(x_i / s), -7, 7) (fp32 division)
 * The row's dequantised value is q_i * s.
 */
void oracle_quantize_rows4(int dtype, const void* X, int64_t rows, int d, int8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    float amax4 = 0.f;
    for (int c = 0; c < d; ++c) {
      const float x = (float)load_f64(dtype, X, r * d + c);
      const float a = fabsf(x);
      if (a > amax4) amax4 = a;
    }
    const float s4 = amax4 / 7.0f;
    scale[r] = s4;
    for (int c = 0; c < d; ++c) {
      int v = 0;
      if (s4 != 0.f) {
        const float x = (float)load_f64(dtype, X, r * d + c);
        float t4 = rintf(x / s4);
        if (t4 > 7.f) t4 = 7.f;
        if (t4 < -7.f) t4 = -7.f;
        v = (int)t4;
      }
      q[r * d + c] = (int8_t)v;
    }
  }
}
