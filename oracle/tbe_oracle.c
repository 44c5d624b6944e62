/*
 * tbe_oracle.c -- the oracle for table-batched embedding bags (TBE).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously correct
 * CPU statement of what the operator computes.  Only the tests, the smoke
 * check and the CPU-baseline leg of the benchmark load it; the CUDA library
 * never links, calls or includes anything from here, and this file includes
 * nothing from the library.
 *
 * Source of every definition: the page "FBTriton table-batched embeddings:
 * the backward win is a threshold moved from 32 to 256" (cited below as
 * [FBT] plus the section title).
 *
 *   - Jagged feature-major layout, bag (t,b) = indices[offsets[t*B+b] :
 *     offsets[t*B+b+1]], all tables in one buffer, output [B, sum D] with
 *     each feature at its own column offset, empty bag stays zero, a
 *     repeated id is added twice:  [FBT] "A lookup table that is most of
 *     the model".
 *   - Sum pooling, optional per-sample weights, FP32 accumulation on the
 *     device (the oracle accumulates in FP64): [FBT] "The forward: a general
 *     gather and one clever special case".
 *   - Histogram form: a pooled sum is a count-weighted sum of table rows:
 *     [FBT] "The forward: a general gather and one clever special case".
 *   - Backward: each row read by the batch gets the sum of the output
 *     gradients of every bag that read it; lookups are inverted by the key
 *     hash_size_cumsum[t] + row, sorted and run-length encoded:
 *     [FBT] "Why the backward is the hard half".
 *   - Weighted backward pairs each lookup with its own weight through a
 *     stable ordering: [FBT] "Using it, and the import that stops you".
 *   - Exact optimizers (SGD, row-wise Adagrad) applied once per distinct
 *     row to its finished gradient: [FBT] "Why the backward is the hard
 *     half".
 *
 * Readings where the page is silent (each is stated beside its use):
 *   ids are table-local; an id outside [0, rows_t) is reported and contributes
 *   nothing; offsets must start at 0, never decrease and end at N; sums are
 *   rounded once, round-to-nearest-even, to the output dtype.
 *
 * Arithmetic: every sum is accumulated in IEEE double.  For unweighted fp16
 * tables this is exact: an fp16 value is an integer multiple of 2^-24 of
 * magnitude below 2^16, so a sum of at most 2^13 of them is an integer
 * multiple of 2^-24 below 2^53 * 2^-24, which double holds exactly whatever
 * the order.  Elsewhere the double rounding error (about n * 2^-53 * sum|terms|)
 * is far below every tolerance the tests use.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes of the packed-table format (a data convention) */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };
/* status bits */
enum { ORC_BAD_INDEX = 1, ORC_BAD_OFFSETS = 2, ORC_BAD_ARG = 4 };

/* ------------------------------------------------------------------------- */
/* scalar formats                                                             */
/* ------------------------------------------------------------------------- */

/* IEEE binary16: value = (-1)^s * 2^(e-15) * 1.m, subnormal 2^-14 * 0.m */
double orc_decode_f16(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25);
  return s ? -v : v;
}

/* bfloat16 = the upper 16 bits of binary32: 8 exponent bits, 7 mantissa bits */
double orc_decode_bf16(uint16_t h) {
  int s = h >> 15, e = (h >> 7) & 0xff, m = h & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)m, -133);
  else if (e == 255)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x80), e - 134);
  return s ? -v : v;
}

/* Round a double once to binary16, to nearest with ties to even.  The
 * significand is scaled to an integer range and rounded with rint(), which
 * follows the default (nearest-even) rounding mode. */
uint16_t orc_encode_f16(double x) {
  if (isnan(x)) return 0x7e00;
  uint16_t s = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isinf(a)) return s | 0x7c00;
  if (a < ldexp(1.0, -14)) { /* subnormal range: multiples of 2^-24 */
    double q = rint(ldexp(a, 24)); /* <= 1024; 1024 is the smallest normal */
    return s | (uint16_t)q;
  }
  int e;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  double q = rint(ldexp(a, 11 - e)); /* in [1024, 2048] */
  int E = e - 1 + 15;
  if (q == 2048.0) { q = 1024.0; E += 1; }
  if (E >= 31) return s | 0x7c00;
  return s | (uint16_t)(E << 10) | (uint16_t)((int)q - 1024);
}

uint16_t orc_encode_bf16(double x) {
  if (isnan(x)) return 0x7fc0;
  uint16_t s = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isinf(a)) return s | 0x7f80;
  if (a < ldexp(1.0, -126)) { /* subnormal range: multiples of 2^-133 */
    double q = rint(ldexp(a, 133));
    return s | (uint16_t)q;
  }
  int e;
  frexp(a, &e);
  double q = rint(ldexp(a, 8 - e)); /* in [128, 256] */
  int E = e - 1 + 127;
  if (q == 256.0) { q = 128.0; E += 1; }
  if (E >= 255) return s | 0x7f80;
  return s | (uint16_t)(E << 7) | (uint16_t)((int)q - 128);
}

static int elem_bytes(int32_t dt) { return dt == ORC_F32 ? 4 : 2; }

/* element c of row r of table t, as an exact double */
static double table_elem(const uint8_t* weights, int64_t w_off, int32_t dt, int32_t D,
                         int64_t r, int32_t c) {
  const uint8_t* p = weights + w_off + (r * (int64_t)D + c) * elem_bytes(dt);
  if (dt == ORC_F32) {
    float f;
    memcpy(&f, p, 4);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, p, 2);
  return dt == ORC_F16 ? orc_decode_f16(h) : orc_decode_bf16(h);
}

/* Round n doubles to the output dtype (0: float bits, 1/2: 16-bit codes). */
void orc_round(const double* in, int64_t n, int32_t dt, void* out) {
  for (int64_t i = 0; i < n; ++i) {
    if (dt == ORC_F32)
      ((float*)out)[i] = (float)in[i]; /* C conversion: nearest-even */
    else if (dt == ORC_F16)
      ((uint16_t*)out)[i] = orc_encode_f16(in[i]);
    else
      ((uint16_t*)out)[i] = orc_encode_bf16(in[i]);
  }
}

/* ------------------------------------------------------------------------- */
/* layout checks                                                              */
/* ------------------------------------------------------------------------- */

/* Offsets must start at 0, never decrease and end at N (reading of the
 * jagged layout in [FBT] "A lookup table that is most of the model"). */
int orc_check_offsets(int32_t T, int32_t B, const int64_t* offsets, int64_t N) {
  int64_t nb = (int64_t)T * B;
  if (offsets[0] != 0 || offsets[nb] != N) return ORC_BAD_OFFSETS;
  for (int64_t g = 0; g < nb; ++g)
    if (offsets[g + 1] < offsets[g]) return ORC_BAD_OFFSETS;
  return 0;
}

/* ------------------------------------------------------------------------- */
/* forward: out[b, D_offsets[t] + c] = sum_{i in bag(t,b)} w_i * W_t[id_i, c] */
/* ------------------------------------------------------------------------- */

/* Computes the pooled sums of the listed bags.  Bag k of the list is
 * g = bags[k] (t = g / B, b = g % B); its D_t sums go to
 * out_sum[out_pos[k] + c] and the matching sum of |terms| to out_abs.
 * Listing every bag in (b, t) order with out_pos = b*sumD + D_offsets[t]
 * fills the whole [B, sum D] output.  Returns status bits. */
int orc_forward(int32_t T, int32_t B, const int64_t* table_row_base, const int32_t* D_offsets,
                const int64_t* weights_offsets, const int32_t* weights_dtype,
                const uint8_t* table_weighted, const uint8_t* weights, const int64_t* indices,
                int64_t N, const int64_t* offsets, const float* per_sample_weights,
                const int64_t* bags, int64_t n_bags, const int64_t* out_pos, double* out_sum,
                double* out_abs, int32_t nthreads) {
  int st = orc_check_offsets(T, B, offsets, N);
  if (st) return st;
  int bad_index = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64) reduction(| : bad_index)
#endif
  for (int64_t k = 0; k < n_bags; ++k) {
    int64_t g = bags[k];
    int32_t t = (int32_t)(g / B);
    int32_t D = D_offsets[t + 1] - D_offsets[t];
    int64_t rows = table_row_base[t + 1] - table_row_base[t];
    int weighted = per_sample_weights != NULL && (table_weighted == NULL || table_weighted[t]);
    double* s = out_sum + out_pos[k];
    double* a = out_abs + out_pos[k];
    for (int32_t c = 0; c < D; ++c) s[c] = a[c] = 0.0; /* an empty bag stays zero */
    for (int64_t i = offsets[g]; i < offsets[g + 1]; ++i) {
      int64_t id = indices[i];
      if (id < 0 || id >= rows) { /* reported, contributes nothing */
        bad_index = 1;
        continue;
      }
      double w = weighted ? (double)per_sample_weights[i] : 1.0;
      for (int32_t c = 0; c < D; ++c) {
        double term = w * table_elem(weights, weights_offsets[t], weights_dtype[t], D, id, c);
        s[c] += term; /* a repeated id is simply added again */
        a[c] += fabs(term);
      }
    }
  }
  return bad_index ? ORC_BAD_INDEX : 0;
}

/* Histogram form of one unweighted table: cnt[b][r] = #{i in bag(t,b) : id_i = r}
 * ([FBT] "The forward: a general gather and one clever special case"). */
int orc_histogram_counts(int32_t T, int32_t B, int32_t t, int64_t rows_t, const int64_t* indices,
                         int64_t N, const int64_t* offsets, int32_t* counts /* [B, rows_t] */) {
  int st = orc_check_offsets(T, B, offsets, N);
  if (st) return st;
  int bad_index = 0;
  memset(counts, 0, sizeof(int32_t) * (size_t)B * (size_t)rows_t);
  for (int32_t b = 0; b < B; ++b) {
    int64_t g = (int64_t)t * B + b;
    for (int64_t i = offsets[g]; i < offsets[g + 1]; ++i) {
      int64_t id = indices[i];
      if (id < 0 || id >= rows_t) { bad_index = 1; continue; }
      counts[(int64_t)b * rows_t + id] += 1;
    }
  }
  return bad_index ? ORC_BAD_INDEX : 0;
}

/* Mean pooling (reading: the page pools "usually by summing"; the other
 * pooling mode, the mean, is the sum divided by the bag's number of lookups,
 * L_{t,b} = offsets[t*B+b+1] - offsets[t*B+b]): divides each bag's block of
 * a [B, sum D] array -- a pooled output, its absolute-term sums, or the
 * output gradient before the backward -- by L_{t,b}.  An empty bag's block
 * is left as it is (it holds zeros, and no lookup reads its gradient).  The
 * backward of the mean is the backward of the sum on the scaled gradient:
 * each lookup of bag (t,b) receives (w_i / L_{t,b}) * grad_out[b]. */
void orc_scale_by_bag_length(int32_t T, int32_t B, const int32_t* D_offsets, const int64_t* offsets,
                             double* values /* [B, sum D] */) {
  const int32_t sumD = D_offsets[T];
  for (int32_t t = 0; t < T; ++t)
    for (int32_t b = 0; b < B; ++b) {
      const int64_t g = (int64_t)t * B + b;
      const int64_t len = offsets[g + 1] - offsets[g];
      if (len <= 0) continue;
      for (int32_t c = D_offsets[t]; c < D_offsets[t + 1]; ++c) values[(int64_t)b * sumD + c] /= (double)len;
    }
}

/* out[b, c] = sum_r cnt[b][r] * W_t[r, c]  (counts times table) */
void orc_counts_times_table(int32_t B, int64_t rows_t, int32_t D, const int32_t* counts,
                            const uint8_t* weights, int64_t w_off, int32_t dt, double* out) {
  for (int32_t b = 0; b < B; ++b)
    for (int32_t c = 0; c < D; ++c) {
      double s = 0.0;
      for (int64_t r = 0; r < rows_t; ++r)
        s += (double)counts[(int64_t)b * rows_t + r] * table_elem(weights, w_off, dt, D, r, c);
      out[(int64_t)b * D + c] = s;
    }
}

/* ------------------------------------------------------------------------- */
/* backward indexing: key = table_row_base[t] + id, stable sort, runs         */
/* ------------------------------------------------------------------------- */

typedef struct {
  int64_t key;
  int64_t pos;
} orc_pair;

static int cmp_pair(const void* x, const void* y) {
  const orc_pair* a = (const orc_pair*)x;
  const orc_pair* b = (const orc_pair*)y;
  if (a->key != b->key) return a->key < b->key ? -1 : 1;
  if (a->pos != b->pos) return a->pos < b->pos ? -1 : 1;
  return 0;
}

/* Inverts the batch ([FBT] "Why the backward is the hard half"): every
 * lookup i of bag (t, b) gets the key table_row_base[t] + id_i, so rows of
 * different tables never collide.  Ordering by (key, position) is the stable
 * sort by key, so inside one row the lookups keep their position order.
 * A lookup with an id outside its table gets the key total_rows (sorts last,
 * belongs to no run).
 *
 * Outputs: sorted_pos[N]; unique_rows[U] (ascending global rows);
 * run_starts[U+1] with run_starts[U] = number of valid lookups;
 * unique_count[T+1] with unique_count[t] = #unique rows below
 * table_row_base[t]; *n_unique = U. */
int orc_backward_indexing(int32_t T, int32_t B, const int64_t* table_row_base,
                          const int64_t* indices, int64_t N, const int64_t* offsets,
                          int32_t* sorted_pos, int64_t* unique_rows, int32_t* run_starts,
                          int64_t* unique_count, int64_t* n_unique) {
  int st = orc_check_offsets(T, B, offsets, N);
  if (st) return st;
  int bad_index = 0;
  int64_t total_rows = table_row_base[T];
  orc_pair* p = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)(N > 0 ? N : 1));
  if (!p) return ORC_BAD_ARG;
  for (int32_t t = 0; t < T; ++t) {
    int64_t rows = table_row_base[t + 1] - table_row_base[t];
    for (int32_t b = 0; b < B; ++b) {
      int64_t g = (int64_t)t * B + b;
      for (int64_t i = offsets[g]; i < offsets[g + 1]; ++i) {
        int64_t id = indices[i];
        int ok = id >= 0 && id < rows;
        if (!ok) bad_index = 1;
        p[i].key = ok ? table_row_base[t] + id : total_rows;
        p[i].pos = i;
      }
    }
  }
  qsort(p, (size_t)N, sizeof(orc_pair), cmp_pair);
  int64_t U = 0, n_valid = 0;
  for (int64_t j = 0; j < N; ++j) {
    sorted_pos[j] = (int32_t)p[j].pos;
    if (p[j].key >= total_rows) continue;
    n_valid = j + 1;
    if (j == 0 || p[j].key != p[j - 1].key) {
      unique_rows[U] = p[j].key;
      run_starts[U] = (int32_t)j;
      ++U;
    }
  }
  run_starts[U] = (int32_t)n_valid;
  *n_unique = U;
  for (int32_t t = 0; t <= T; ++t) {
    int64_t c = 0;
    while (c < U && unique_rows[c] < table_row_base[t]) ++c;
    unique_count[t] = c;
  }
  free(p);
  return bad_index ? ORC_BAD_INDEX : 0;
}

/* ------------------------------------------------------------------------- */
/* backward values: row_grad[u, c] = sum_{i in run u} w_i * G[b_i, D_off[t]+c] */
/* ------------------------------------------------------------------------- */

/* For each listed run u (runs[k]) writes the D_t sums of its row gradient to
 * rg_sum[rg_pos[k] + c] and the sums of |terms| to rg_abs.  The bag of each
 * sorted position comes from a plain walk over the offsets. */
int orc_backward_values(int32_t T, int32_t B, const int64_t* table_row_base,
                        const int32_t* D_offsets, const uint8_t* table_weighted,
                        const int64_t* offsets, int64_t N, const float* per_sample_weights,
                        const double* grad_out, const int64_t* unique_rows,
                        const int32_t* run_starts, const int32_t* sorted_pos, const int64_t* runs,
                        int64_t n_runs, const int64_t* rg_pos, double* rg_sum, double* rg_abs,
                        int32_t nthreads) {
  int st = orc_check_offsets(T, B, offsets, N);
  if (st) return st;
  int64_t nb = (int64_t)T * B;
  int32_t sumD = D_offsets[T];
  int32_t* bag_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
  if (!bag_of) return ORC_BAD_ARG;
  for (int64_t g = 0; g < nb; ++g)
    for (int64_t i = offsets[g]; i < offsets[g + 1]; ++i) bag_of[i] = (int32_t)g;
  int bad = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
#endif
  for (int64_t k = 0; k < n_runs; ++k) {
    int64_t u = runs[k];
    int64_t row = unique_rows[u];
    int32_t t = 0;
    while (t < T && table_row_base[t + 1] <= row) ++t;
    int32_t D = D_offsets[t + 1] - D_offsets[t];
    int weighted = per_sample_weights != NULL && (table_weighted == NULL || table_weighted[t]);
    double* s = rg_sum + rg_pos[k];
    double* a = rg_abs + rg_pos[k];
    for (int32_t c = 0; c < D; ++c) s[c] = a[c] = 0.0;
    for (int64_t j = run_starts[u]; j < run_starts[u + 1]; ++j) {
      int32_t pos = sorted_pos[j];
      int64_t g = bag_of[pos];
      if (g / B != t) { bad = 1; continue; } /* would mean an inconsistent key */
      int64_t b = g % B;
      double w = weighted ? (double)per_sample_weights[pos] : 1.0;
      const double* grow = grad_out + b * sumD + D_offsets[t];
      for (int32_t c = 0; c < D; ++c) {
        double term = w * (double)grow[c];
        s[c] += term;
        a[c] += fabs(term);
      }
    }
  }
  free(bag_of);
  return bad ? ORC_BAD_ARG : 0;
}

/* ------------------------------------------------------------------------- */
/* exact optimizer step on finished row gradients                             */
/* ------------------------------------------------------------------------- */

/* [FBT] "Why the backward is the hard half": the optimizer runs inside the
 * backward, once per distinct row, on that row's finished gradient g (the
 * sum over its run), never once per lookup.  Two kinds:
 *   kind 0, exact SGD (the plain reading: the step is lr times g):
 *       W[r] <- W[r] - lr * g
 *   kind 1, exact row-wise Adagrad (one momentum scalar per row, fed by the
 *   mean of the squared gradient over the row's D_t columns):
 *       m[r] <- m[r] + (sum_c g_c^2) / D_t
 *       W[r] <- W[r] - lr / (sqrt(m[r]) + eps) * g
 * For each listed row k (global row rows[k], gradient values
 * grads[g_pos[k] + c], c < D_t) the updated weights are written in double,
 * unrounded, to w_new[g_pos[k] + c]: the caller rounds to the table dtype
 * where it needs to.  For Adagrad, momentum[] is the state before the step
 * (fp32, indexed by global row) and the new value goes to m_new[k].
 * Returns ORC_BAD_INDEX if a listed row lies outside every table,
 * ORC_BAD_ARG for an unknown kind. */
int orc_exact_update(int32_t T, const int64_t* table_row_base, const int32_t* D_offsets,
                     const int64_t* weights_offsets, const int32_t* weights_dtype,
                     const uint8_t* weights, int32_t kind, double lr, double eps,
                     const float* momentum, int64_t n_rows, const int64_t* rows,
                     const double* grads, const int64_t* g_pos, double* w_new, double* m_new) {
  if (kind != 0 && kind != 1) return ORC_BAD_ARG;
  for (int64_t k = 0; k < n_rows; ++k) {
    int64_t row = rows[k];
    if (row < 0 || row >= table_row_base[T]) return ORC_BAD_INDEX;
    int32_t t = 0;
    while (table_row_base[t + 1] <= row) ++t;
    int32_t D = D_offsets[t + 1] - D_offsets[t];
    int64_t id = row - table_row_base[t];
    const double* g = grads + g_pos[k];
    double step = lr;
    if (kind == 1) {
      double sq = 0.0;
      for (int32_t c = 0; c < D; ++c) sq += g[c] * g[c];
      double m = (double)momentum[row] + sq / (double)D;
      m_new[k] = m;
      step = lr / (sqrt(m) + eps);
    }
    for (int32_t c = 0; c < D; ++c)
      w_new[g_pos[k] + c] =
          table_elem(weights, weights_offsets[t], weights_dtype[t], D, id, c) - step * g[c];
  }
  return 0;
}
