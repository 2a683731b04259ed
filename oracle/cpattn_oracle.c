/*
 * cpattn_oracle.c -- plain fp64 CPU oracle for the context-parallel attention
 * hot path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU
 * baseline leg of the benchmark load it; the library never does.  It shares no
 * code, header or constant with the CUDA path.
 *
 * Everything here is written for a reader to check against the sources by
 * eye: no blocking, no fusion, no reordering beyond what each definition says.
 * All arithmetic is IEEE double (compile without -ffast-math).  Inputs are
 * contiguous row-major double arrays: q [NBH, S_q, D], k and v [NBH, S_kv, D],
 * where NBH = batch * heads.  Outputs: out [NBH, S_q, D], lse [NBH, S_q].
 *
 * Sources (page title, section):
 *   [CP]   Diffusers "Context parallelism" guide: the variants table,
 *          "Ring Attention", "Ulysses Attention", "Ring Anything Attention",
 *          "Ulysses Anything Attention".
 *   [API]  Diffusers "Parallelism" API page: ContextParallelConfig parameters
 *          ring_degree, ulysses_degree, convert_to_fp32, ring_anything,
 *          ulysses_anything.
 *   [PARA] ParaAttention README, "Run Unified Attention ... with
 *          torch.compile": the sharded result must equal the matching slice of
 *          F.scaled_dot_product_attention (no mask, no dropout, not causal).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CPO_OK 0
#define CPO_ERR_DIVISIBILITY 1
#define CPO_ERR_SHAPE 2
#define CPO_ERR_ALLOC 3

/* ---------------------------------------------------------------------------
 * 1. Full softmax attention -- the definition the method reaches exactly.
 *    [PARA] compares against scaled_dot_product_attention, whose value for
 *    query row i is  out_i = sum_j softmax_j(scale * q_i . k_j) v_j.
 *    lse_i = log sum_j exp(scale * q_i . k_j)   (natural log), written as
 *    M + log(sum_j exp(s_j - M)) with M = max_j s_j so exp never overflows.
 *    row_ids: flat indices into [NBH * S_q]; NULL means every row.
 *    causal != 0: scaled_dot_product_attention's is_causal, i.e. query i
 *    attends keys j <= i only; a row with no such key gives (0, -inf).
 * ------------------------------------------------------------------------- */
int cpo_attention_rows(const double* q, const double* k, const double* v,
                       int64_t nbh, int64_t s_q, int64_t s_kv, int64_t d,
                       double scale, const int64_t* row_ids, int64_t n_rows,
                       double* out, double* lse, int causal) {
  if (s_kv < 1) return CPO_ERR_SHAPE;
  if (row_ids == NULL) n_rows = nbh * s_q;
  int failed = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc((size_t)s_kv * sizeof(double));
    if (s == NULL) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
      if (s == NULL) continue;
      int64_t row = row_ids ? row_ids[r] : r;
      int64_t bh = row / s_q;
      int64_t i = row % s_q;
      const double* qi = q + row * d;
      const double* kb = k + bh * s_kv * d;
      const double* vb = v + bh * s_kv * d;
      /* the keys this row attends: all, or j <= i when causal */
      int64_t n_keys = s_kv;
      if (causal && i + 1 < s_kv) n_keys = i + 1;
      double* oi = out + r * d;
      for (int64_t e = 0; e < d; ++e) oi[e] = 0.0;
      if (n_keys == 0) {
        lse[r] = -INFINITY;
        continue;
      }
      /* scores s_j = scale * <q_i, k_j> */
      for (int64_t j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (int64_t e = 0; e < d; ++e) dot += qi[e] * kb[j * d + e];
        s[j] = scale * dot;
      }
      double m = s[0];
      for (int64_t j = 1; j < n_keys; ++j)
        if (s[j] > m) m = s[j];
      double z = 0.0;
      for (int64_t j = 0; j < n_keys; ++j) z += exp(s[j] - m);
      for (int64_t j = 0; j < n_keys; ++j) {
        double w = exp(s[j] - m) / z;
        for (int64_t e = 0; e < d; ++e) oi[e] += w * vb[j * d + e];
      }
      lse[r] = m + log(z);
    }
    free(s);
  }
  return failed ? CPO_ERR_ALLOC : CPO_OK;
}

/* ---------------------------------------------------------------------------
 * 2. One ring step: attention of query rows against the key range [k0, k1)
 *    only, emitting the partial output and its fp32-able LSE ([API]
 *    convert_to_fp32: "output and LSE").  Deliberately a separate routine from
 *    (1): two passes over the keys, scores recomputed in the second pass, the
 *    normalisation applied once at the end.  causal != 0: only keys
 *    j <= i of the range count; a row left with none gives the empty partial
 *    (0, -inf), which the merge below treats as its identity.
 * ------------------------------------------------------------------------- */
int cpo_partial_rows(const double* q, const double* k, const double* v,
                     int64_t nbh, int64_t s_q, int64_t s_kv, int64_t d,
                     double scale, int64_t k0, int64_t k1,
                     const int64_t* row_ids, int64_t n_rows,
                     double* out, double* lse, int causal) {
  if (k0 < 0 || k1 > s_kv || k1 <= k0) return CPO_ERR_SHAPE;
  if (row_ids == NULL) n_rows = nbh * s_q;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t row = row_ids ? row_ids[r] : r;
    int64_t bh = row / s_q;
    int64_t i = row % s_q;
    const double* qi = q + row * d;
    const double* kb = k + bh * s_kv * d;
    const double* vb = v + bh * s_kv * d;
    int64_t hi_key = k1;
    if (causal && i + 1 < k1) hi_key = i + 1;
    double* oi = out + r * d;
    if (hi_key <= k0) {
      for (int64_t e = 0; e < d; ++e) oi[e] = 0.0;
      lse[r] = -INFINITY;
      continue;
    }
    /* pass 1: the largest score in the range */
    double m = -INFINITY;
    for (int64_t j = k0; j < hi_key; ++j) {
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e) dot += qi[e] * kb[j * d + e];
      if (scale * dot > m) m = scale * dot;
    }
    /* pass 2: unnormalised weights, their sum and the weighted V rows */
    for (int64_t e = 0; e < d; ++e) oi[e] = 0.0;
    double z = 0.0;
    for (int64_t j = k0; j < hi_key; ++j) {
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e) dot += qi[e] * kb[j * d + e];
      double p = exp(scale * dot - m);
      z += p;
      for (int64_t e = 0; e < d; ++e) oi[e] += p * vb[j * d + e];
    }
    for (int64_t e = 0; e < d; ++e) oi[e] /= z;
    lse[r] = m + log(z);
  }
  return CPO_OK;
}

/* ---------------------------------------------------------------------------
 * 3. LSE merge of two partials over disjoint key sets ([API]
 *    convert_to_fp32: the ring steps' outputs and LSEs are combined in fp32
 *    for stability).  The pages print no formula; it follows from the
 *    definition of LSE:
 *      lse = log(e^a + e^b) = max(a,b) + log1p(exp(min(a,b) - max(a,b)))
 *      o   = e^(a - lse) o_a + e^(b - lse) o_b
 *    lse = -inf marks an empty partial (the identity); two empty partials
 *    merge to (0, -inf).  In place: the result overwrites (o_a, lse_a).
 * ------------------------------------------------------------------------- */
void cpo_merge(double* o_a, double* lse_a, const double* o_b,
               const double* lse_b, int64_t n_rows, int64_t d) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n_rows; ++r) {
    double a = lse_a[r], b = lse_b[r];
    double* oa = o_a + r * d;
    const double* ob = o_b + r * d;
    if (a == -INFINITY && b == -INFINITY) {
      for (int64_t e = 0; e < d; ++e) oa[e] = 0.0;
      lse_a[r] = -INFINITY;
      continue;
    }
    double hi = a > b ? a : b;
    double lo = a > b ? b : a;
    double l = hi + log1p(exp(lo - hi));
    double wa = exp(a - l), wb = exp(b - l);
    for (int64_t e = 0; e < d; ++e) oa[e] = wa * oa[e] + wb * ob[e];
    lse_a[r] = l;
  }
}

/* ---------------------------------------------------------------------------
 * 4. Chunk partition of the key sequence across a ring of R ranks.
 *    [CP] variants table: plain ring needs S divisible by ring_degree, every
 *    rank holds S/R tokens.  [CP] "Ring Anything Attention": any S; each rank's
 *    block is sliced back to its true length.  Reading for the uneven split:
 *    the first (S mod R) blocks hold one extra token (1537/1536/1536 for
 *    S = 4609, R = 3).  An empty block is not allowed (R > S is an error).
 *    bounds has R + 1 entries: chunk c is [bounds[c], bounds[c+1]).
 * ------------------------------------------------------------------------- */
int cpo_chunk_bounds(int64_t s_kv, int64_t ring_degree, int ring_anything,
                     int64_t* bounds) {
  if (ring_degree < 1 || s_kv < 1) return CPO_ERR_SHAPE;
  if (!ring_anything && s_kv % ring_degree != 0) return CPO_ERR_DIVISIBILITY;
  if (ring_anything && ring_degree > s_kv) return CPO_ERR_SHAPE;
  int64_t base = s_kv / ring_degree, extra = s_kv % ring_degree;
  bounds[0] = 0;
  for (int64_t c = 0; c < ring_degree; ++c)
    bounds[c + 1] = bounds[c] + base + (c < extra ? 1 : 0);
  return CPO_OK;
}

/* ---------------------------------------------------------------------------
 * 5. The ring schedule ([CP] "Ring Attention"): each query row meets every
 *    K/V chunk once; each meeting emits a partial (2) and the partials are
 *    folded with the merge (3) in chunk order 0 .. R-1.
 * ------------------------------------------------------------------------- */
int cpo_ring_rows(const double* q, const double* k, const double* v,
                  int64_t nbh, int64_t s_q, int64_t s_kv, int64_t d,
                  double scale, int64_t ring_degree, int ring_anything,
                  const int64_t* row_ids, int64_t n_rows,
                  double* out, double* lse, int causal) {
  if (ring_degree < 1) return CPO_ERR_SHAPE;
  int64_t* bounds = (int64_t*)malloc((size_t)(ring_degree + 1) * sizeof(int64_t));
  if (bounds == NULL) return CPO_ERR_ALLOC;
  int rc = cpo_chunk_bounds(s_kv, ring_degree, ring_anything, bounds);
  if (rc != CPO_OK) {
    free(bounds);
    return rc;
  }
  if (row_ids == NULL) n_rows = nbh * s_q;
  double* o_c = (double*)malloc((size_t)n_rows * (size_t)d * sizeof(double));
  double* l_c = (double*)malloc((size_t)n_rows * sizeof(double));
  if (o_c == NULL || l_c == NULL) {
    free(bounds); free(o_c); free(l_c);
    return CPO_ERR_ALLOC;
  }
  rc = cpo_partial_rows(q, k, v, nbh, s_q, s_kv, d, scale, bounds[0], bounds[1],
                        row_ids, n_rows, out, lse, causal);
  for (int64_t c = 1; c < ring_degree && rc == CPO_OK; ++c) {
    rc = cpo_partial_rows(q, k, v, nbh, s_q, s_kv, d, scale, bounds[c],
                          bounds[c + 1], row_ids, n_rows, o_c, l_c, causal);
    if (rc == CPO_OK) cpo_merge(out, lse, o_c, l_c, n_rows, d);
  }
  free(bounds); free(o_c); free(l_c);
  return rc;
}

/* ---------------------------------------------------------------------------
 * 6. Ulysses head regroup ([CP] "Ulysses Attention"): the all-to-all leaves
 *    each of the G ranks every token for H/G of the heads.  On one device this
 *    is a layout permute of x [B, S, H, D]:
 *      forward (dir = +1): y[g, b, s, hh, :] = x[b, s, g*(H/G) + hh, :]
 *      inverse (dir = -1): y[b, s, g*(H/G) + hh, :] = x[g, b, s, hh, :]
 *    A byte copy of elem_bytes-sized elements; H must be divisible by G.
 * ------------------------------------------------------------------------- */
int cpo_ulysses_permute(const void* x, void* y, int64_t b, int64_t s,
                        int64_t h, int64_t d, int64_t g, int dir,
                        int64_t elem_bytes) {
  if (g < 1 || h % g != 0 || (dir != 1 && dir != -1)) return CPO_ERR_SHAPE;
  int64_t hg = h / g;
  const unsigned char* src = (const unsigned char*)x;
  unsigned char* dst = (unsigned char*)y;
  for (int64_t gi = 0; gi < g; ++gi)
    for (int64_t bi = 0; bi < b; ++bi)
      for (int64_t si = 0; si < s; ++si)
        for (int64_t hh = 0; hh < hg; ++hh)
          for (int64_t e = 0; e < d; ++e) {
            int64_t bshd = ((bi * s + si) * h + gi * hg + hh) * d + e;
            int64_t grouped = (((gi * b + bi) * s + si) * hg + hh) * d + e;
            int64_t from = dir == 1 ? bshd : grouped;
            int64_t to = dir == 1 ? grouped : bshd;
            memcpy(dst + to * elem_bytes, src + from * elem_bytes,
                   (size_t)elem_bytes);
          }
  return CPO_OK;
}

/* ---------------------------------------------------------------------------
 * 7. Ulysses Anything ([CP] "Ulysses Anything Attention"; [API]
 *    ulysses_anything): Ulysses without the requirement that H and S divide
 *    by G (ring_degree stays 1).  The pages do not say how uneven heads are
 *    dealt out; the reading taken is torch.tensor_split's: G consecutive
 *    groups, the first H mod G of them one head longer.  On one device the
 *    whole sequence lands in every group, so S needs no rule.
 *
 *    cpo_ulysses_anything_heads: start[0 .. G] with group g holding heads
 *    [start[g], start[g+1]).
 * ------------------------------------------------------------------------- */
int cpo_ulysses_anything_heads(int64_t h, int64_t g, int64_t* start) {
  if (g < 1 || h < 0) return CPO_ERR_SHAPE;
  int64_t base = h / g, longer = h % g;
  start[0] = 0;
  for (int64_t i = 0; i < g; ++i)
    start[i + 1] = start[i] + base + (i < longer ? 1 : 0);
  return CPO_OK;
}

/*    cpo_ulysses_anything_permute: the regroup with every group padded to
 *    hm = ceil(H/G) head slots (a reading: the exchange buffer must give all
 *    groups one shape), group g filling slots 0 .. h_g - 1:
 *      forward (dir = +1): y[g, b, s, j, :] = x[b, s, start[g] + j, :]
 *                          for j < h_g; slots j >= h_g are not written.
 *      inverse (dir = -1): y[b, s, start[g] + j, :] = x[g, b, s, j, :]
 *                          for j < h_g; slots j >= h_g are not read.       */
int cpo_ulysses_anything_permute(const void* x, void* y, int64_t b, int64_t s,
                                 int64_t h, int64_t d, int64_t g, int dir,
                                 int64_t elem_bytes) {
  if (g < 1 || h < 1 || (dir != 1 && dir != -1)) return CPO_ERR_SHAPE;
  int64_t hm = (h + g - 1) / g;
  int64_t* start = (int64_t*)malloc((size_t)(g + 1) * sizeof(int64_t));
  if (!start) return CPO_ERR_ALLOC;
  cpo_ulysses_anything_heads(h, g, start);
  const unsigned char* src = (const unsigned char*)x;
  unsigned char* dst = (unsigned char*)y;
  for (int64_t gi = 0; gi < g; ++gi) {
    int64_t hg = start[gi + 1] - start[gi];
    for (int64_t bi = 0; bi < b; ++bi)
      for (int64_t si = 0; si < s; ++si)
        for (int64_t j = 0; j < hg; ++j)
          for (int64_t e = 0; e < d; ++e) {
            int64_t bshd = ((bi * s + si) * h + start[gi] + j) * d + e;
            int64_t grouped = (((gi * b + bi) * s + si) * hm + j) * d + e;
            int64_t from = dir == 1 ? bshd : grouped;
            int64_t to = dir == 1 ? grouped : bshd;
            memcpy(dst + to * elem_bytes, src + from * elem_bytes,
                   (size_t)elem_bytes);
          }
  }
  free(start);
  return CPO_OK;
}

/* Threads OpenMP uses for the parallel loops above (1 without OpenMP). */
int cpo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
