/*
 * oracle.c -- plain, slow, CPU reference of the CTR sparse-embedding path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load or call this code.  The
 * product path (libctr, the CUDA library) shares no source with it and never
 * calls it.
 *
 * Every floating-point result is accumulated in fp64 from the exact input
 * values and rounded once to the output type (fp32: C's double->float
 * conversion, round to nearest even; bf16: round to nearest even from the
 * double, see round_bf16).  Loops follow the definitions in the order the pages
 * state them; there is no blocking or reordering.
 *
 * Functions and the passages they follow:
 *   oracle_dedup                 "How TensorNet Supercharges Sparse Feature
 *                                Training on TensorFlow", Core Optimizations,
 *                                embedding_lookup (collect the batch IDs, sort
 *                                them, give each a continuous index, build a
 *                                batch-sized matrix).
 *   oracle_embedding_bag_fwd     "DHEN" notes, section 2.1 (one trainable
 *                                d-vector per categorical term) and Solution 2
 *                                of section 3.1 (sum of the active embeddings);
 *                                "Meta DLRM", section 02 (categorical features
 *                                go through embeddings).
 *   oracle_dot_interaction       "Meta DLRM", section 02 (dot product between
 *                                all pairs of embedding vectors and the
 *                                processed dense features, cross terms only);
 *                                "DHEN" notes, section 3.1, Eq. (3) (pairwise
 *                                inner products concatenated with the dense
 *                                features).
 *   oracle_dot_interaction_bwd   derivative of the interaction above (not on
 *                                the pages; follows from the definition).
 *   oracle_dot_interaction_mode  the interaction's variants: mode 0 as above;
 *                                mode 1 all <x_i, x_j> for i >= j ("DHEN"
 *                                notes, section 3.1: inner products for
 *                                i <= j); mode 2 the full Gram matrix X X^T
 *                                ("DHEN" notes, section 3.3, Eq. (7), the
 *                                input of the cross network).
 *   oracle_dot_interaction_bwd_mode
 *                                their derivatives, accumulated entry by
 *                                entry: dZ_ij adds dZ_ij x_j to dX_i and
 *                                dZ_ij x_i to dX_j.
 *   oracle_embedding_bag_bwd_update
 *                                TensorNet, Synchronous Architecture (only the
 *                                sparse features present in the batch are
 *                                synchronised): the table gradient of the
 *                                pooled output restricted to the batch's rows,
 *                                applied as plain SGD (rule not on the pages).
 *   oracle_bag_fm                the factorization-machine second-order term
 *                                of each bag's active embeddings, summed over
 *                                pairs of positions ("DHEN" notes, section
 *                                3.1, Solution 2; each occurrence is one
 *                                active feature).
 *   oracle_optimizer_step        the row update of the listed rows under SGD,
 *                                Adagrad (state: sum of squared gradients),
 *                                row-wise Adagrad (one state per row: sum of
 *                                the mean squared gradient) or Adam (Kingma
 *                                and Ba 2015, with bias correction), moments
 *                                kept only for the rows the batch touches
 *                                (the pages name no rule; the Baidu page's
 *                                k-step Adam merge is multi-worker).
 *   oracle_bf16_stochastic_round the stochastic rounding of updated bf16 rows
 *                                ("DHEN" notes, section 6.4: low-precision
 *                                embeddings with stochastic rounding), its
 *                                random bits drawn from splitmix64.
 *   oracle_table_rows            the counter-based table generator
 *                                (splitmix64, Steele/Lea/Flood 2014); input
 *                                generation, not the method.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_OK = 0, OR_ERR_ARG = -1, OR_ERR_INDEX = -4 };
enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_SUM = 0, OR_MEAN = 1 };
enum { OR_GEN_UNIFORM = 0, OR_GEN_NORMAL4 = 1 };

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------------- */
/* scalar conversions                                                      */
/* ---------------------------------------------------------------------- */
static double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits), ties to even.
 * Values below the smallest normal bf16 use the subnormal spacing 2^-133. */
static uint16_t round_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  double y;
  if (fabs(x) < 0x1p-126) {
    y = nearbyint(x * 0x1p133) * 0x1p-133;
  } else {
    int e;
    double m = frexp(x, &e); /* x = m * 2^e, 0.5 <= |m| < 1 */
    y = ldexp(nearbyint(m * 256.0), e - 8);
  }
  float f = (float)y; /* exact: y has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

static void store_value(void* out, int dtype, int64_t i, double v) {
  if (dtype == OR_F32) ((float*)out)[i] = (float)v;
  else ((uint16_t*)out)[i] = round_bf16(v);
}

static double load_value(const void* p, int dtype, int64_t i) {
  if (dtype == OR_F32) return (double)((const float*)p)[i];
  return bf16_to_f64(((const uint16_t*)p)[i]);
}

/* ---------------------------------------------------------------------- */
/* counter-based table generator (input generation, not the method)        */
/* ---------------------------------------------------------------------- */
uint64_t oracle_splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Value of global table element idx, returned as the stored type's bits. */
static float gen_uniform(uint64_t seed, float scale, uint64_t idx) {
  uint64_t h = oracle_splitmix64(seed ^ idx);
  int32_t c = (int32_t)(h >> 40) - (1 << 23);
  float cf = (float)c; /* exact, |c| <= 2^23 */
  volatile float v = cf * scale; /* one fp32 rounding */
  return v;
}

static uint16_t gen_normal4_bf16(uint64_t seed, float scale, uint64_t idx) {
  const uint64_t m22 = (1ull << 22) - 1;
  uint64_t h1 = oracle_splitmix64(seed ^ (2 * idx));
  uint64_t h2 = oracle_splitmix64(seed ^ (2 * idx + 1));
  uint64_t s = (h1 >> 42) + ((h1 >> 20) & m22) + (h2 >> 42) + ((h2 >> 20) & m22);
  int32_t c = (int32_t)s - ((1 << 23) - 2);
  float cf = (float)c; /* exact, |c| < 2^24 */
  volatile float v = cf * scale;
  float vf = v;
  uint32_t u;
  memcpy(&u, &vf, 4);
  uint32_t r = ((u >> 16) & 1u) + 0x7FFFu; /* fp32 -> bf16, ties to even */
  return (uint16_t)((u + r) >> 16);
}

/* Fill out[n_rows][d] with the generated values of the listed global rows.
 * kind OR_GEN_UNIFORM writes fp32, OR_GEN_NORMAL4 writes bf16 bits. */
void oracle_table_rows(int kind, uint64_t seed, float scale, int32_t d, const int64_t* rows, int64_t n_rows,
                       void* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n_rows; ++r) {
    for (int32_t c = 0; c < d; ++c) {
      uint64_t idx = (uint64_t)rows[r] * (uint64_t)d + (uint64_t)c;
      if (kind == OR_GEN_UNIFORM) ((float*)out)[r * d + c] = gen_uniform(seed, scale, idx);
      else ((uint16_t*)out)[r * d + c] = gen_normal4_bf16(seed, scale, idx);
    }
  }
}

/* A table is either a host array (table != NULL) or the generator. */
typedef struct {
  const void* table;
  int dtype;
  int gen_kind;
  uint64_t gen_seed;
  float gen_scale;
  int32_t d;
} table_src;

static double table_value(const table_src* t, int64_t row, int32_t c) {
  if (t->table) return load_value(t->table, t->dtype, row * t->d + c);
  uint64_t idx = (uint64_t)row * (uint64_t)t->d + (uint64_t)c;
  if (t->gen_kind == OR_GEN_UNIFORM) return (double)gen_uniform(t->gen_seed, t->gen_scale, idx);
  return bf16_to_f64(gen_normal4_bf16(t->gen_seed, t->gen_scale, idx));
}

/* ---------------------------------------------------------------------- */
/* bag bookkeeping shared by the oracle functions                          */
/* ---------------------------------------------------------------------- */
static int check_bags(const int64_t* offsets, int32_t F, int32_t B) {
  if (!offsets || F < 0 || B < 0) return OR_ERR_ARG;
  if (offsets[0] != 0) return OR_ERR_ARG;
  for (int64_t b = 0; b < (int64_t)F * B; ++b)
    if (offsets[b + 1] < offsets[b]) return OR_ERR_ARG;
  return OR_OK;
}

/* Global row of occurrence i of bag (f, b): row_base[table(f)] + id. */
static int key_of(const int64_t* ids, int64_t i, int32_t f, const int32_t* bag_to_table, const int64_t* row_base,
                  int32_t T, int64_t* key) {
  int32_t t = bag_to_table[f];
  if (t < 0 || t >= T) return OR_ERR_ARG;
  int64_t id = ids[i];
  if (id < 0 || id >= row_base[t + 1] - row_base[t]) return OR_ERR_INDEX;
  *key = row_base[t] + id;
  return OR_OK;
}

/* ---------------------------------------------------------------------- */
/* dedup                                                                   */
/* ---------------------------------------------------------------------- */
typedef struct {
  int64_t key;
  int64_t pos;
} key_pos;

static int cmp_key_pos(const void* a, const void* b) {
  const key_pos* x = (const key_pos*)a;
  const key_pos* y = (const key_pos*)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  return (x->pos > y->pos) - (x->pos < y->pos);
}

/* TensorNet's embedding_lookup, steps 2-3: collect the batch's IDs (as global
 * rows, so equal IDs of different tables stay apart), sort them, and give each
 * distinct one a continuous index (0-based rank in ascending order).
 * Sorting the (key, position) pairs lexicographically is the stable sort by
 * key.  Outputs (any of the int32 arrays may be NULL):
 *   unique_rows[n_unique]   distinct keys, ascending
 *   inverse[i]              rank of key i            (the virtual sparse feature)
 *   sorted_pos[s]           position of the s-th key in sorted order
 *   sorted_bag[s]           bag (f*B + b) of that position
 *   run_offsets[u]          first sorted slot of unique u; run_offsets[n_unique] = n_ids
 *   unique_offsets[t]       number of unique keys below row_base[t], t = 0..T
 */
int oracle_dedup(const int64_t* ids, const int64_t* offsets, int32_t F, int32_t B, const int32_t* bag_to_table,
                 const int64_t* row_base, int32_t T, int64_t* unique_rows, int64_t* n_unique, int32_t* inverse,
                 int32_t* sorted_pos, int32_t* sorted_bag, int32_t* run_offsets, int64_t* unique_offsets) {
  int st = check_bags(offsets, F, B);
  if (st) return st;
  int64_t n = offsets[(int64_t)F * B];
  key_pos* kp = (key_pos*)malloc(sizeof(key_pos) * (size_t)(n > 0 ? n : 1));
  int32_t* bag_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  if (!kp || !bag_of) {
    free(kp);
    free(bag_of);
    return OR_ERR_ARG;
  }
  /* step 2: collect the IDs of the batch */
  for (int32_t f = 0; f < F; ++f) {
    for (int32_t b = 0; b < B; ++b) {
      int64_t bag = (int64_t)f * B + b;
      for (int64_t i = offsets[bag]; i < offsets[bag + 1]; ++i) {
        int64_t key;
        st = key_of(ids, i, f, bag_to_table, row_base, T, &key);
        if (st) {
          free(kp);
          free(bag_of);
          return st;
        }
        kp[i].key = key;
        kp[i].pos = i;
        bag_of[i] = (int32_t)bag;
      }
    }
  }
  /* step 3: sort, then number the distinct keys 0, 1, 2, ... */
  qsort(kp, (size_t)n, sizeof(key_pos), cmp_key_pos);
  int64_t u = -1;
  for (int64_t s = 0; s < n; ++s) {
    if (s == 0 || kp[s].key != kp[s - 1].key) {
      ++u;
      unique_rows[u] = kp[s].key;
      if (run_offsets) run_offsets[u] = (int32_t)s;
    }
    if (inverse) inverse[kp[s].pos] = (int32_t)u;
    if (sorted_pos) sorted_pos[s] = (int32_t)kp[s].pos;
    if (sorted_bag) sorted_bag[s] = bag_of[kp[s].pos];
  }
  int64_t nu = u + 1;
  *n_unique = nu;
  if (run_offsets) run_offsets[nu] = (int32_t)n;
  if (unique_offsets) {
    for (int32_t t = 0; t <= T; ++t) {
      int64_t cnt = 0;
      while (cnt < nu && unique_rows[cnt] < row_base[t]) ++cnt;
      unique_offsets[t] = cnt;
    }
  }
  free(kp);
  free(bag_of);
  return OR_OK;
}

/* ---------------------------------------------------------------------- */
/* pooled embedding-bag forward                                            */
/* ---------------------------------------------------------------------- */
/* out(b, f) = sum over the bag's IDs (each occurrence counts) of the table row,
 * divided by the bag length for MEAN (an empty bag gives 0).  The sum runs in
 * the bag's index order in fp64.  If bag_list is NULL every bag is computed and
 * out(b, f) sits at out + b*out_stride_b + f*out_stride_f; otherwise only the
 * listed bags (f*B + b) are computed into a compact out[n_list][d].  mag_out,
 * if given, receives the sum of |row values| (scaled like the output) in the
 * same layout as a double array. */
int oracle_embedding_bag_fwd(const void* table, int dtype, int gen_kind, uint64_t gen_seed, float gen_scale,
                             int32_t d, const int64_t* ids, const int64_t* offsets, int32_t F, int32_t B,
                             const int32_t* bag_to_table, const int64_t* row_base, int32_t T, int pool,
                             const int64_t* bag_list, int64_t n_list, void* out, int out_dtype, int64_t out_stride_b,
                             int64_t out_stride_f, double* mag_out) {
  if (!ids || !out || d <= 0) return OR_ERR_ARG;
  int st = check_bags(offsets, F, B);
  if (st) return st;
  table_src src = {table, dtype, gen_kind, gen_seed, gen_scale, d};
  int64_t nb = bag_list ? n_list : (int64_t)F * B;
  int err = OR_OK;
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t k = 0; k < nb; ++k) {
    int64_t bag = bag_list ? bag_list[k] : k;
    int32_t f = (int32_t)(bag / B), b = (int32_t)(bag % B);
    int64_t base = bag_list ? k * d : (int64_t)b * out_stride_b + (int64_t)f * out_stride_f;
    int64_t len = offsets[bag + 1] - offsets[bag];
    for (int32_t c = 0; c < d; ++c) {
      double acc = 0.0, mag = 0.0;
      for (int64_t i = offsets[bag]; i < offsets[bag + 1]; ++i) {
        int64_t key;
        if (key_of(ids, i, f, bag_to_table, row_base, T, &key)) {
          err = OR_ERR_INDEX;
          continue;
        }
        double v = table_value(&src, key, c);
        acc += v;
        mag += fabs(v);
      }
      if (pool == OR_MEAN) {
        acc = len > 0 ? acc / (double)len : 0.0;
        mag = len > 0 ? mag / (double)len : 0.0;
      }
      store_value(out, out_dtype, base + c, acc);
      if (mag_out) mag_out[base + c] = mag;
    }
  }
  return err;
}

/* FM second-order term of each bag: fm = sum over pairs of positions i < j
 * of the bag of <v_i, v_j>, v the table rows of the bag's IDs (a repeated ID
 * is a repeated feature), independent of the pooling mode.  fp64, rounded
 * once to fp32.  bag_list (or NULL for all F*B bags, bag-major) selects bags;
 * out is compact over the list.  mag_out (may be NULL) gets the sum over the
 * same pairs of sum_c |v_i[c] v_j[c]|. */
int oracle_bag_fm(const void* table, int dtype, int gen_kind, uint64_t gen_seed, float gen_scale, int32_t d,
                  const int64_t* ids, const int64_t* offsets, int32_t F, int32_t B, const int32_t* bag_to_table,
                  const int64_t* row_base, int32_t T, const int64_t* bag_list, int64_t n_list, float* out,
                  double* mag_out) {
  if (!ids || !out || d <= 0) return OR_ERR_ARG;
  int st = check_bags(offsets, F, B);
  if (st) return st;
  table_src src = {table, dtype, gen_kind, gen_seed, gen_scale, d};
  int64_t nb = bag_list ? n_list : (int64_t)F * B;
  int err = OR_OK;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t k = 0; k < nb; ++k) {
    int64_t bag = bag_list ? bag_list[k] : k;
    int32_t f = (int32_t)(bag / B);
    double acc = 0.0, mag = 0.0;
    for (int64_t i = offsets[bag]; i < offsets[bag + 1]; ++i) {
      for (int64_t j = i + 1; j < offsets[bag + 1]; ++j) {
        int64_t ki, kj;
        if (key_of(ids, i, f, bag_to_table, row_base, T, &ki) || key_of(ids, j, f, bag_to_table, row_base, T, &kj)) {
          err = OR_ERR_INDEX;
          continue;
        }
        for (int32_t c = 0; c < d; ++c) {
          double p = table_value(&src, ki, c) * table_value(&src, kj, c);
          acc += p;
          mag += fabs(p);
        }
      }
    }
    out[k] = (float)acc;
    if (mag_out) mag_out[k] = mag;
  }
  return err;
}

/* One optimizer step on n rows of d values.  w_old and g in fp64 (the row's
 * value and its exact gradient); state in fp32, updated into s0_out/s1_out:
 *   opt 0 SGD:               w -= lr g
 *   opt 1 Adagrad:           s += g^2 (per value);          w -= lr g / (sqrt(s) + eps)
 *   opt 2 row-wise Adagrad:  s += mean over the row of g^2;  w -= lr g / (sqrt(s) + eps)
 *   opt 3 Adam (step t >= 1): m = b1 m + (1 - b1) g;  v = b2 v + (1 - b2) g^2;
 *                            w -= lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
 * s0 is the Adagrad state or Adam's m ([n][d]; [n] for row-wise), s1 Adam's v.
 * New values are computed in fp64 and rounded once (w to the table dtype,
 * state to fp32); x_out (may be NULL) receives the unrounded new values, for
 * stochastic rounding. */
int oracle_optimizer_step(int opt, double lr, double eps, double beta1, double beta2, int64_t step, int32_t d,
                          int64_t n, const double* w_old, const double* g, const float* s0_in, const float* s1_in,
                          void* w_new, int dtype, float* s0_out, float* s1_out, double* x_out) {
  if (opt < 0 || opt > 3 || d <= 0 || n < 0 || !w_old || !g || !w_new) return OR_ERR_ARG;
  if (opt != 0 && (!s0_in || !s0_out)) return OR_ERR_ARG;
  if (opt == 3 && (!s1_in || !s1_out || step < 1)) return OR_ERR_ARG;
  double bc1 = 1.0, bc2 = 1.0;
  if (opt == 3) {
    bc1 = 1.0 - pow(beta1, (double)step);
    bc2 = 1.0 - pow(beta2, (double)step);
  }
  for (int64_t r = 0; r < n; ++r) {
    double srow = 0.0;
    if (opt == 2) {
      double msq = 0.0;
      for (int32_t c = 0; c < d; ++c) msq += g[r * d + c] * g[r * d + c];
      srow = (double)s0_in[r] + msq / (double)d;
      s0_out[r] = (float)srow;
    }
    for (int32_t c = 0; c < d; ++c) {
      int64_t e = r * d + c;
      double gv = g[e], upd;
      if (opt == 0) {
        upd = lr * gv;
      } else if (opt == 1) {
        double sv = (double)s0_in[e] + gv * gv;
        s0_out[e] = (float)sv;
        upd = lr * gv / (sqrt(sv) + eps);
      } else if (opt == 2) {
        upd = lr * gv / (sqrt(srow) + eps);
      } else {
        double m = beta1 * (double)s0_in[e] + (1.0 - beta1) * gv;
        double v = beta2 * (double)s1_in[e] + (1.0 - beta2) * gv * gv;
        s0_out[e] = (float)m;
        s1_out[e] = (float)v;
        upd = lr * (m / bc1) / (sqrt(v / bc2) + eps);
      }
      store_value(w_new, dtype, e, w_old[e] - upd);
      if (x_out) x_out[e] = w_old[e] - upd;
    }
  }
  return OR_OK;
}

/* Stochastic rounding of values x (fp64) at elements (rows[r], c) of a table
 * with d columns to bf16.  With lo and hi the bf16 neighbours of x below and
 * above in magnitude (lo = x when x is a bf16 value) and f = (|x| - |lo|) /
 * (|hi| - |lo|) in [0, 1), x rounds to hi when f + u / 2^16 >= 1, u the 16
 * random bits of the element: the 4 values of column chunk q = c / 4 of a row
 * take bits 16 j .. 16 j + 15 (j = c mod 4) of splitmix64(seed ^ (row d / 4 +
 * q)); d must be a multiple of 4.  So P(hi) = f: the rounding is unbiased.
 * Values outside the finite bf16 range round to nearest (not exercised).
 * out: uint16 bf16 bits [n][d]. */
int oracle_bf16_stochastic_round(const double* x, const int64_t* rows, int64_t n, int32_t d, uint64_t seed,
                                 uint16_t* out) {
  if (!x || !rows || !out || d <= 0 || d % 4 != 0) return OR_ERR_ARG;
  for (int64_t r = 0; r < n; ++r) {
    for (int32_t c = 0; c < d; ++c) {
      double v = x[r * d + c];
      uint64_t h = oracle_splitmix64(seed ^ (uint64_t)(rows[r] * (d / 4) + c / 4));
      uint32_t u = (uint32_t)((h >> (16 * (c % 4))) & 0xFFFFu);
      double a = fabs(v);
      if (!(a < 0x1.fep127) || a == 0.0) {  /* zero, huge, inf, nan: nearest */
        out[r * d + c] = round_bf16(v);
        continue;
      }
      /* lo: |v| with its fp32 mantissa cut to bf16's 7 bits (toward zero) */
      int e;
      double m = frexp(a, &e);                    /* a = m 2^e, 0.5 <= m < 1 */
      double lo, ulp;
      if (e - 1 < -126) {                         /* below the normal range: spacing 2^-133 */
        ulp = 0x1p-133;
        lo = floor(a / ulp) * ulp;
      } else {
        ulp = ldexp(1.0, e - 8);                  /* bf16 keeps 8 significant bits */
        lo = floor(m * 256.0) / 256.0 * ldexp(1.0, e);
      }
      double f = (a - lo) / ulp;                  /* exact: a - lo < ulp */
      double mag = (f + (double)u / 65536.0 >= 1.0) ? lo + ulp : lo;
      out[r * d + c] = round_bf16(v < 0 ? -mag : mag);
    }
  }
  return OR_OK;
}

/* ---------------------------------------------------------------------- */
/* dot interaction                                                         */
/* ---------------------------------------------------------------------- */
/* For each sample b with vectors x_0 (dense) .. x_{n-1} (pooled), each of
 * length d: out[b] = [ x_0 | Z ] where Z lists <x_i, x_j> for 1 <= i < n,
 * 0 <= j < i, row by row: Z index i(i-1)/2 + j.  Output dtype = input dtype.
 * sample_list (or NULL for all) selects samples; out is compact over the list.
 * mag_out (double, same layout, may be NULL) gets sum_c |x_i[c] x_j[c]| for
 * the pair columns and |x_0[c]| for the dense columns. */
int oracle_dot_interaction(const void* X, int dtype, int32_t B, int32_t n, int32_t d, const int64_t* sample_list,
                           int64_t n_list, void* out, double* mag_out) {
  if (!X || !out || n < 1 || d < 1) return OR_ERR_ARG;
  int64_t width = d + (int64_t)n * (n - 1) / 2;
  int64_t ns = sample_list ? n_list : B;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < ns; ++k) {
    int64_t b = sample_list ? sample_list[k] : k;
    int64_t xb = b * (int64_t)n * d;
    int64_t ob = k * width;
    for (int32_t c = 0; c < d; ++c) {
      double v = load_value(X, dtype, xb + c);
      store_value(out, dtype, ob + c, v);
      if (mag_out) mag_out[ob + c] = fabs(v);
    }
    for (int32_t i = 1; i < n; ++i) {
      for (int32_t j = 0; j < i; ++j) {
        double acc = 0.0, mag = 0.0;
        for (int32_t c = 0; c < d; ++c) {
          double p = load_value(X, dtype, xb + (int64_t)i * d + c) * load_value(X, dtype, xb + (int64_t)j * d + c);
          acc += p;
          mag += fabs(p);
        }
        int64_t o = ob + d + (int64_t)i * (i - 1) / 2 + j;
        store_value(out, dtype, o, acc);
        if (mag_out) mag_out[o] = mag;
      }
    }
  }
  return OR_OK;
}

/* Derivative of the interaction: with dZ(i,j) the upstream gradient of pair
 * (max(i,j), min(i,j)),  dX_i = sum_{j != i} dZ(i,j) x_j, plus the dense
 * pass-through dout[b][0:d] added to dX_0.  fp32 in and out. */
int oracle_dot_interaction_bwd(const float* dout, const float* X, int32_t B, int32_t n, int32_t d,
                               const int64_t* sample_list, int64_t n_list, float* dX, double* mag_out) {
  if (!dout || !X || !dX || n < 1 || d < 1) return OR_ERR_ARG;
  int64_t width = d + (int64_t)n * (n - 1) / 2;
  int64_t ns = sample_list ? n_list : B;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < ns; ++k) {
    int64_t b = sample_list ? sample_list[k] : k;
    const float* xb = X + b * (int64_t)n * d;
    const float* gb = dout + b * width;
    for (int32_t i = 0; i < n; ++i) {
      for (int32_t c = 0; c < d; ++c) {
        double acc = 0.0, mag = 0.0;
        if (i == 0) {
          acc = gb[c];
          mag = fabs((double)gb[c]);
        }
        for (int32_t j = 0; j < n; ++j) {
          if (j == i) continue;
          int32_t hi = i > j ? i : j, lo = i > j ? j : i;
          double g = gb[d + (int64_t)hi * (hi - 1) / 2 + lo];
          double p = g * (double)xb[(int64_t)j * d + c];
          acc += p;
          mag += fabs(p);
        }
        int64_t o = k * (int64_t)n * d + (int64_t)i * d + c;
        dX[o] = (float)acc;
        if (mag_out) mag_out[o] = mag;
      }
    }
  }
  return OR_OK;
}

/* Interaction variants.  Output row of a sample:
 *   mode 0  [dense (d) | <x_i, x_j>, i > j, at i(i-1)/2 + j]      width d + n(n-1)/2
 *   mode 1  [dense (d) | <x_i, x_j>, i >= j, at i(i+1)/2 + j]     width d + n(n+1)/2
 *   mode 2  [<x_i, x_j> for all i, j, at i n + j]                  width n n
 * (the order of the pairs and whether the dense vector leads are layout
 * choices: the pages fix which products appear, not where). */
static int64_t mode_width(int mode, int32_t n, int32_t d) {
  if (mode == 0) return d + (int64_t)n * (n - 1) / 2;
  if (mode == 1) return d + (int64_t)n * (n + 1) / 2;
  return (int64_t)n * n;
}

/* Output slot of product (i, j) under `mode`, or -1 if the mode omits it. */
static int64_t mode_slot(int mode, int32_t n, int32_t d, int32_t i, int32_t j) {
  if (mode == 0) return i > j ? d + (int64_t)i * (i - 1) / 2 + j : -1;
  if (mode == 1) return i >= j ? d + (int64_t)i * (i + 1) / 2 + j : -1;
  return (int64_t)i * n + j;
}

int oracle_dot_interaction_mode(const void* X, int dtype, int32_t B, int32_t n, int32_t d, int mode,
                                const int64_t* sample_list, int64_t n_list, void* out, double* mag_out) {
  if (!X || !out || n < 1 || d < 1 || mode < 0 || mode > 2) return OR_ERR_ARG;
  int64_t width = mode_width(mode, n, d);
  int64_t ns = sample_list ? n_list : B;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < ns; ++k) {
    int64_t b = sample_list ? sample_list[k] : k;
    int64_t xb = b * (int64_t)n * d;
    int64_t ob = k * width;
    if (mode != 2) {
      for (int32_t c = 0; c < d; ++c) {
        double v = load_value(X, dtype, xb + c);
        store_value(out, dtype, ob + c, v);
        if (mag_out) mag_out[ob + c] = fabs(v);
      }
    }
    for (int32_t i = 0; i < n; ++i) {
      for (int32_t j = 0; j < n; ++j) {
        int64_t slot = mode_slot(mode, n, d, i, j);
        if (slot < 0) continue;
        double acc = 0.0, mag = 0.0;
        for (int32_t c = 0; c < d; ++c) {
          double p = load_value(X, dtype, xb + (int64_t)i * d + c) * load_value(X, dtype, xb + (int64_t)j * d + c);
          acc += p;
          mag += fabs(p);
        }
        store_value(out, dtype, ob + slot, acc);
        if (mag_out) mag_out[ob + slot] = mag;
      }
    }
  }
  return OR_OK;
}

/* Derivative of a mode's output: every emitted product Z_ij = <x_i, x_j>
 * with upstream gradient g adds g x_j to dX_i and g x_i to dX_j (so a
 * diagonal entry adds 2 g x_i); modes 0 and 1 also pass dout[b][0:d] to
 * dX_0.  fp64 accumulation, fp32 out. */
int oracle_dot_interaction_bwd_mode(const float* dout, const float* X, int32_t B, int32_t n, int32_t d, int mode,
                                    const int64_t* sample_list, int64_t n_list, float* dX, double* mag_out) {
  if (!dout || !X || !dX || n < 1 || d < 1 || mode < 0 || mode > 2) return OR_ERR_ARG;
  int64_t width = mode_width(mode, n, d);
  int64_t ns = sample_list ? n_list : B;
  int64_t nd = (int64_t)n * d;
#pragma omp parallel
  {
    double* acc = (double*)malloc((size_t)nd * sizeof(double));
    double* mag = (double*)malloc((size_t)nd * sizeof(double));
#pragma omp for schedule(static)
    for (int64_t k = 0; k < ns; ++k) {
      if (!acc || !mag) continue;
      int64_t b = sample_list ? sample_list[k] : k;
      const float* xb = X + b * nd;
      const float* gb = dout + b * width;
      for (int64_t e = 0; e < nd; ++e) acc[e] = mag[e] = 0.0;
      if (mode != 2)
        for (int32_t c = 0; c < d; ++c) {
          acc[c] += (double)gb[c];
          mag[c] += fabs((double)gb[c]);
        }
      for (int32_t i = 0; i < n; ++i)
        for (int32_t j = 0; j < n; ++j) {
          int64_t slot = mode_slot(mode, n, d, i, j);
          if (slot < 0) continue;
          double g = gb[slot];
          for (int32_t c = 0; c < d; ++c) {
            double pi = g * (double)xb[(int64_t)j * d + c];  /* into dX_i */
            double pj = g * (double)xb[(int64_t)i * d + c];  /* into dX_j */
            acc[(int64_t)i * d + c] += pi;
            mag[(int64_t)i * d + c] += fabs(pi);
            acc[(int64_t)j * d + c] += pj;
            mag[(int64_t)j * d + c] += fabs(pj);
          }
        }
      for (int64_t e = 0; e < nd; ++e) {
        dX[k * nd + e] = (float)acc[e];
        if (mag_out) mag_out[k * nd + e] = mag[e];
      }
    }
    free(acc);
    free(mag);
  }
  return OR_OK;
}

/* ---------------------------------------------------------------------- */
/* sparse backward + SGD row update                                        */
/* ---------------------------------------------------------------------- */
static int64_t find_row(const int64_t* rows, int64_t n, int64_t key) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    int64_t mid = lo + (hi - lo) / 2;
    if (rows[mid] < key) lo = mid + 1;
    else hi = mid;
  }
  return (lo < n && rows[lo] == key) ? lo : -1;
}

/* The gradient of the pooled outputs with respect to the table, kept only for
 * the rows the batch touches: g[row] = sum over every occurrence i with key
 * row of scale(bag_i) * G(bag_i), where scale is 1 (SUM) or 1/len (MEAN) and
 * G(bag) = G[b*g_stride_b + f*g_stride_f + 0..d).  Then the SGD update
 * w_new = w - lr * g, evaluated in fp64 and rounded once to the table type.
 * target_rows (ascending global rows, n_targets of them) lists the rows to
 * report; their old values come from `table` or the generator.  Outputs:
 * new_rows[n_targets][d] (table dtype), grad_out and mag_out (double, may be
 * NULL; mag = sum of |scale * G| per component). */
int oracle_embedding_bag_bwd_update(const float* G, int64_t g_stride_b, int64_t g_stride_f, const int64_t* ids,
                                    const int64_t* offsets, int32_t F, int32_t B, const int32_t* bag_to_table,
                                    const int64_t* row_base, int32_t T, int pool, float lr, int32_t d,
                                    const int64_t* target_rows, int64_t n_targets, const void* table, int dtype,
                                    int gen_kind, uint64_t gen_seed, float gen_scale, void* new_rows,
                                    double* grad_out, double* mag_out) {
  if (!G || !ids || !target_rows || !new_rows || d <= 0) return OR_ERR_ARG;
  int st = check_bags(offsets, F, B);
  if (st) return st;
  double* g = (double*)calloc((size_t)(n_targets > 0 ? n_targets : 1) * (size_t)d, sizeof(double));
  double* m = (double*)calloc((size_t)(n_targets > 0 ? n_targets : 1) * (size_t)d, sizeof(double));
  if (!g || !m) {
    free(g);
    free(m);
    return OR_ERR_ARG;
  }
  for (int32_t f = 0; f < F; ++f) {
    for (int32_t b = 0; b < B; ++b) {
      int64_t bag = (int64_t)f * B + b;
      int64_t len = offsets[bag + 1] - offsets[bag];
      double scale = pool == OR_MEAN ? 1.0 / (double)len : 1.0;
      const float* gb = G + (int64_t)b * g_stride_b + (int64_t)f * g_stride_f;
      for (int64_t i = offsets[bag]; i < offsets[bag + 1]; ++i) {
        int64_t key;
        st = key_of(ids, i, f, bag_to_table, row_base, T, &key);
        if (st) {
          free(g);
          free(m);
          return st;
        }
        int64_t r = find_row(target_rows, n_targets, key);
        if (r < 0) continue;
        for (int32_t c = 0; c < d; ++c) {
          double t = scale * (double)gb[c];
          g[r * d + c] += t;
          m[r * d + c] += fabs(t);
        }
      }
    }
  }
  table_src src = {table, dtype, gen_kind, gen_seed, gen_scale, d};
  for (int64_t r = 0; r < n_targets; ++r) {
    for (int32_t c = 0; c < d; ++c) {
      double w = table_value(&src, target_rows[r], c);
      store_value(new_rows, dtype, r * d + c, w - (double)lr * g[r * d + c]);
      if (grad_out) grad_out[r * d + c] = g[r * d + c];
      if (mag_out) mag_out[r * d + c] = m[r * d + c];
    }
  }
  free(g);
  free(m);
  return OR_OK;
}
