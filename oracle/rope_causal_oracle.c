/*
 * Reference oracle for causal softmax attention with Rotary Position Embedding (RoPE).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct definition that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark may build, load or call it; the library's product path never does.  It shares no
 * code, header, table or constant with the CUDA sources.
 *
 * What it computes (all arithmetic in IEEE double, no blocking, no fusion, no reordering):
 *
 *   RoPE, half-split pairing.  "AttnFuse Makes RoPE a First-Class Attention Compilation Operation"
 *   (2026-09-13 AI papers report), paragraph 1, and the AttnFuse abstract (arxivdaily 2609.13612):
 *   RoPE is a transformation applied to Q and K *before* the QK^T product.  The pages name RoPE
 *   but print no formula; this library fixes the common half-split convention:
 *       theta_k = base^(-2k/d),                 k = 0 .. d/2-1
 *       x'[k]       = x[k]       cos(p theta_k) - x[k+d/2] sin(p theta_k)
 *       x'[k+d/2]   = x[k+d/2]   cos(p theta_k) + x[k]     sin(p theta_k)
 *   with p the token index.  V is not rotated.
 *
 *   Variants (the "_ex" entry points): a rotary dimension r <= d rotates only the first r entries
 *   of each head vector, with theta_k = base^(-2k/r), k = 0 .. r/2-1, and leaves entries r .. d-1
 *   unchanged; the interleaved form pairs (2k, 2k+1) instead of (k, k+r/2):
 *       x'[2k]   = x[2k]   cos(p theta_k) - x[2k+1] sin(p theta_k)
 *       x'[2k+1] = x[2k+1] cos(p theta_k) + x[2k]   sin(p theta_k)
 *   Both are the same plane rotations as the half-split form on a permuted set of planes.
 *
 *   Causal softmax attention.  Same report, paragraph 2 (causality and softmax building blocks):
 *       s_ij = (q'_i . k'_j) / sqrt(d)      for j <= i   (keys j > i are excluded)
 *       o_i  = sum_j softmax_j(s_ij) v_j
 *       lse_i = max_j s_ij + ln sum_j exp(s_ij - max_j s_ij)     (natural log)
 *   GQA: query head h reads key/value head floor(h / (Hq/Hkv)).
 *
 *   Key length and positions (the "_kv" entry point).  The pages fix neither; this library takes
 *   the plainest general reading of "causal" when there are Nk >= Nq keys (a prefill that extends
 *   a cache of Nk - Nq earlier tokens): the Nq queries are the last Nq of the Nk tokens, so query i
 *   sees keys j <= (Nk - Nq) + i.  The rotation position of query i is (Nk - Nq) + i and that of key
 *   j is j, unless explicit per-token positions are given (any integers, one per query and one per
 *   key); positions change only the angles, never the mask.  Nk == Nq with default positions is the
 *   definition above.
 *
 * Layouts (row-major, contiguous): q, out [B, N, Hq, d]; k, v [B, N, Hkv, d]; lse [B, Hq, N]
 * (with the "_kv" entry: q, out [B, Nq, Hq, d]; k, v [B, Nk, Hkv, d]; lse [B, Hq, Nq]).
 * Inputs may be raw bf16 or fp16 bit patterns (decoded exactly to double here) or doubles.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F64 = 0, ORC_BF16 = 1, ORC_F16 = 2 };

/* bf16 is the upper half of an IEEE binary32: widen and reinterpret (exact). */
static double decode_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits (exact). */
static double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-14 / 2^10 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25); /* (1024 + m) * 2^(e - 15 - 10) */
  return sign ? -v : v;
}

static double load_elem(const void *p, int dtype, size_t idx) {
  if (dtype == ORC_F64) return ((const double *)p)[idx];
  uint16_t h = ((const uint16_t *)p)[idx];
  return dtype == ORC_BF16 ? decode_bf16(h) : decode_f16(h);
}

/* Which entries of a head vector are rotated, and how they are paired. */
typedef struct {
  int d;           /* head dimension */
  int r;           /* rotary dimension: entries [0, r) are rotated, [r, d) copied; even, 2 <= r <= d */
  int interleaved; /* 0: pairs (k, k + r/2); 1: pairs (2k, 2k + 1) */
} rope_form_t;

/* theta_k = base^(-2k/r) for k in [0, r/2). */
static void rope_frequencies(int r, double base, double *theta) {
  for (int k = 0; k < r / 2; ++k) theta[k] = pow(base, -2.0 * (double)k / (double)r);
}

/* Rotate one head vector x[0..d) that sits at position pos. */
static void rope_rotate_vec(const double *x, double *y, rope_form_t f, double pos, const double *theta) {
  int half = f.r / 2;
  for (int k = 0; k < half; ++k) {
    double angle = pos * theta[k];
    double c = cos(angle), s = sin(angle);
    int ia = f.interleaved ? 2 * k : k;
    int ib = f.interleaved ? 2 * k + 1 : k + half;
    double a = x[ia], b = x[ib];
    y[ia] = a * c - b * s;
    y[ib] = b * c + a * s;
  }
  for (int e = f.r; e < f.d; ++e) y[e] = x[e];
}

static int form_ok(rope_form_t f) {
  return f.d >= 2 && f.r >= 2 && f.r <= f.d && (f.r % 2) == 0 && (f.interleaved == 0 || f.interleaved == 1);
}

/* ------------------------------------------------------------------------------------------- */
/* A tiny work queue over pthreads: items [0, n_items) are claimed one at a time.               */

typedef struct {
  void (*fn)(void *ctx, int64_t item, double *scratch);
  void *ctx;
  int64_t n_items;
  int64_t next; /* claimed with an atomic fetch-add */
  size_t scratch_doubles;
  int failed;
} orc_pool_t;

static void *orc_worker(void *arg) {
  orc_pool_t *pool = (orc_pool_t *)arg;
  double *scratch = (double *)malloc(sizeof(double) * (pool->scratch_doubles ? pool->scratch_doubles : 1));
  if (!scratch) {
    __atomic_store_n(&pool->failed, 1, __ATOMIC_SEQ_CST);
    return NULL;
  }
  for (;;) {
    int64_t item = __atomic_fetch_add(&pool->next, 1, __ATOMIC_SEQ_CST);
    if (item >= pool->n_items) break;
    pool->fn(pool->ctx, item, scratch);
  }
  free(scratch);
  return NULL;
}

static int orc_run(orc_pool_t *pool, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  pool->next = 0;
  pool->failed = 0;
  pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!tids) return -1;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, orc_worker, pool) != 0) break;
    ++started;
  }
  if (started == 0) orc_worker(pool); /* no thread could start: do the work here */
  for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
  free(tids);
  return pool->failed ? -1 : 0;
}

/* ------------------------------------------------------------------------------------------- */
/* Public entry 1: rotate x[rows, H, d] where row r sits at position positions[r].              */

typedef struct {
  const void *x;
  int dtype;
  int H;
  rope_form_t form;
  const double *positions;
  const double *theta;
  double *out;
} rot_ctx_t;

static void rot_item(void *vctx, int64_t r, double *scratch) {
  rot_ctx_t *c = (rot_ctx_t *)vctx;
  int d = c->form.d;
  for (int h = 0; h < c->H; ++h) {
    size_t base = ((size_t)r * c->H + h) * d;
    for (int e = 0; e < d; ++e) scratch[e] = load_elem(c->x, c->dtype, base + e);
    rope_rotate_vec(scratch, c->out + base, c->form, c->positions[r], c->theta);
  }
}

int orc_rope_rotate_ex(const void *x, int dtype, int64_t rows, int H, int d, int rotary_dim, int interleaved,
                       const double *positions, double base, double *out, int nthreads) {
  rope_form_t f = {d, rotary_dim, interleaved};
  if (!x || !positions || !out || rows < 0 || H < 1 || !form_ok(f)) return -1;
  double *theta = (double *)malloc(sizeof(double) * (size_t)(f.r / 2));
  if (!theta) return -1;
  rope_frequencies(f.r, base, theta);
  rot_ctx_t ctx = {x, dtype, H, f, positions, theta, out};
  orc_pool_t pool = {rot_item, &ctx, rows, 0, (size_t)d, 0};
  int rc = orc_run(&pool, nthreads);
  free(theta);
  return rc;
}

int orc_rope_rotate(const void *x, int dtype, int64_t rows, int H, int d, const double *positions, double base,
                    double *out, int nthreads) {
  if (d < 2 || (d % 2) != 0) return -1;
  return orc_rope_rotate_ex(x, dtype, rows, H, d, d, 0, positions, base, out, nthreads);
}

/* ------------------------------------------------------------------------------------------- */
/* Public entry 2: causal attention with RoPE on Q and K.                                        */
/*   sel_rows: the query positions to evaluate (NULL = all N, in order), n_sel of them.          */
/*   out: [B, n_sel, Hq, d] doubles;  lse: [B, Hq, n_sel] doubles (may be NULL).                 */

typedef struct {
  const void *q, *v;
  int dtype;
  int B, Hq, Hkv, Nq, Nk, d;
  rope_form_t form;
  const double *theta;
  const double *qpos; /* [B, Nq] rotation positions of the queries, or NULL: (Nk - Nq) + i */
  const double *krot; /* [B, Nk, Hkv, d] rotated keys */
  const int64_t *sel;
  int64_t n_sel;
  double *out, *lse;
} attn_ctx_t;

typedef struct {
  const void *k;
  int dtype;
  int Hkv;
  rope_form_t form;
  int Nk;
  const double *theta;
  const double *kpos; /* [B, Nk] rotation positions of the keys, or NULL: j */
  double *krot;
} krot_ctx_t;

/* One item = one key token (b, j): rotate its Hkv head vectors. */
static void krot_item(void *vctx, int64_t bj, double *scratch) {
  krot_ctx_t *c = (krot_ctx_t *)vctx;
  int j = (int)(bj % c->Nk);
  double pos = c->kpos ? c->kpos[bj] : (double)j;
  int d = c->form.d;
  for (int h = 0; h < c->Hkv; ++h) {
    size_t base = ((size_t)bj * c->Hkv + h) * d;
    for (int e = 0; e < d; ++e) scratch[e] = load_elem(c->k, c->dtype, base + e);
    rope_rotate_vec(scratch, c->krot + base, c->form, pos, c->theta);
  }
}

/* One item = one (b, h, selected query row i). scratch holds: raw q (d), rotated q (d), scores (Nk).
 * Query i sees keys j <= last = (Nk - Nq) + i. */
static void attn_item(void *vctx, int64_t item, double *scratch) {
  attn_ctx_t *c = (attn_ctx_t *)vctx;
  int64_t s = item % c->n_sel;
  int h = (int)((item / c->n_sel) % c->Hq);
  int b = (int)(item / (c->n_sel * c->Hq));
  int64_t i = c->sel ? c->sel[s] : s;
  int g = c->Hq / c->Hkv;
  int hk = h / g; /* GQA: consecutive query heads share one key/value head */
  int d = c->d;
  double *qraw = scratch, *qrot = scratch + d, *score = scratch + 2 * d;

  int64_t last = (int64_t)(c->Nk - c->Nq) + i;
  size_t qbase = (((size_t)b * c->Nq + (size_t)i) * c->Hq + h) * d;
  for (int e = 0; e < d; ++e) qraw[e] = load_elem(c->q, c->dtype, qbase + e);
  double qp = c->qpos ? c->qpos[(size_t)b * c->Nq + (size_t)i] : (double)last;
  rope_rotate_vec(qraw, qrot, c->form, qp, c->theta);

  double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int64_t j = 0; j <= last; ++j) { /* causal: keys j <= last only */
    const double *kr = c->krot + (((size_t)b * c->Nk + (size_t)j) * c->Hkv + hk) * d;
    double dot = 0.0;
    for (int e = 0; e < d; ++e) dot += qrot[e] * kr[e];
    score[j] = dot * scale;
    if (score[j] > mx) mx = score[j];
  }
  double denom = 0.0;
  for (int64_t j = 0; j <= last; ++j) {
    score[j] = exp(score[j] - mx);
    denom += score[j];
  }
  double *o = c->out + (((size_t)b * c->n_sel + (size_t)s) * c->Hq + h) * d;
  for (int e = 0; e < d; ++e) o[e] = 0.0;
  for (int64_t j = 0; j <= last; ++j) {
    double p = score[j] / denom;
    size_t vbase = (((size_t)b * c->Nk + (size_t)j) * c->Hkv + hk) * d;
    for (int e = 0; e < d; ++e) o[e] += p * load_elem(c->v, c->dtype, vbase + e);
  }
  if (c->lse) c->lse[((size_t)b * c->Hq + h) * c->n_sel + (size_t)s] = mx + log(denom);
}

/* Public entry 3: the general form.  Nq queries, the last Nq of Nk >= Nq tokens; q_pos [B, Nq]
 * and k_pos [B, Nk] are the rotation positions (either may be NULL for the defaults). */
int orc_rope_causal_kv(const void *q, const void *k, const void *v, int dtype, int B, int Hq, int Hkv, int Nq, int Nk,
                       int d, int rotary_dim, int interleaved, double base, const double *q_pos, const double *k_pos,
                       const int64_t *sel_rows, int64_t n_sel, double *out, double *lse, int nthreads) {
  rope_form_t f = {d, rotary_dim, interleaved};
  if (!q || !k || !v || !out || B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < Nq || !form_ok(f) || (Hq % Hkv) != 0)
    return -1;
  if (!sel_rows) n_sel = Nq;
  if (n_sel < 0) return -1;
  if (sel_rows)
    for (int64_t s = 0; s < n_sel; ++s)
      if (sel_rows[s] < 0 || sel_rows[s] >= Nq) return -1;

  double *theta = (double *)malloc(sizeof(double) * (size_t)(f.r / 2));
  double *krot = (double *)malloc(sizeof(double) * (size_t)B * (size_t)Nk * (size_t)Hkv * (size_t)d);
  if (!theta || !krot) {
    free(theta);
    free(krot);
    return -1;
  }
  rope_frequencies(f.r, base, theta);

  krot_ctx_t kctx = {k, dtype, Hkv, f, Nk, theta, k_pos, krot};
  orc_pool_t kpool = {krot_item, &kctx, (int64_t)B * Nk, 0, (size_t)d, 0};
  int rc = orc_run(&kpool, nthreads);

  if (rc == 0) {
    attn_ctx_t actx = {q, v, dtype, B, Hq, Hkv, Nq, Nk, d, f, theta, q_pos, krot, sel_rows, n_sel, out, lse};
    orc_pool_t apool = {attn_item, &actx, (int64_t)B * Hq * n_sel, 0, (size_t)(2 * d + Nk), 0};
    rc = orc_run(&apool, nthreads);
  }
  free(theta);
  free(krot);
  return rc;
}

int orc_rope_causal_ex(const void *q, const void *k, const void *v, int dtype, int B, int Hq, int Hkv, int N, int d,
                       int rotary_dim, int interleaved, double base, const int64_t *sel_rows, int64_t n_sel,
                       double *out, double *lse, int nthreads) {
  return orc_rope_causal_kv(q, k, v, dtype, B, Hq, Hkv, N, N, d, rotary_dim, interleaved, base, NULL, NULL, sel_rows,
                            n_sel, out, lse, nthreads);
}

int orc_rope_causal(const void *q, const void *k, const void *v, int dtype, int B, int Hq, int Hkv, int N, int d,
                    double base, const int64_t *sel_rows, int64_t n_sel, double *out, double *lse, int nthreads) {
  if (d < 2 || (d % 2) != 0) return -1;
  return orc_rope_causal_ex(q, k, v, dtype, B, Hq, Hkv, N, d, d, 0, base, sel_rows, n_sel, out, lse, nthreads);
}

/* ------------------------------------------------------------------------------------------- */
/* Public entry 4: the backward pass of entry 3 (Nq queries, the last Nq of Nk >= Nq tokens;   */
/* query i sees keys j <= (Nk - Nq) + i; positions (Nk - Nq) + i and j unless given).           */
/*                                                                                               */
/* Given dO = dL/dO for the loss L, with P_ij = softmax_j(s_ij) over visible j, s_ij = q'_i.k'_j/ */
/* sqrt(d), q' = R(i) q_i, k' = R(j) k_j (R(p) the RoPE rotation at position p), the chain rule  */
/* through o_i = sum_j P_ij v_j gives                                                            */
/*   dv_j   = sum_{h in the group of j's head} sum_{i that see j} P_ij dO_i                      */
/*   dP_ij  = dO_i . v_j                                                                          */
/*   dS_ij  = P_ij (dP_ij - sum_k P_ik dP_ik)            (softmax Jacobian)                       */
/*   dq'_i  = sum_j dS_ij k'_j / sqrt(d),   dk'_j = sum_{h, i that see j} dS_ij q'_i / sqrt(d)     */
/*   dq_i   = R(i)^T dq'_i,                 dk_j  = R(j)^T dk'_j    (R^T = rotation by -p)        */
/* The loss has no lse term (dL/dlse = 0).  Pass 1 (per query row) computes dq and keeps the row  */
/* max m_i, denominator l_i and D_i = sum_k P_ik dP_ik; pass 2 (per key row) recomputes P_ij from  */
/* them and accumulates dk and dv.  Outputs: dq [B, nq, Hq, d], dk and dv [B, nk, Hkv, d] for the  */
/* selected query rows (q_rows, NULL = all) and key rows (k_rows, NULL = all), in doubles.        */

typedef struct {
  const void *v, *dout;
  int dtype;
  int B, Hq, Hkv, Nq, Nk, d;
  rope_form_t form;
  const double *theta;
  const double *qrot, *krot; /* [B, Nq, Hq, d], [B, Nk, Hkv, d] */
  const double *qpos;        /* [B, Nq] rotation positions of the queries, or NULL: (Nk - Nq) + i */
  const int64_t *qslot;      /* [Nq]: output slot of query row i, or -1 if its dq is not reported */
  int64_t nq;                /* reported query rows per batch entry */
  double *dq;                /* [B, nq, Hq, d] */
  double *m, *l, *D;         /* [B, Hq, Nq] row statistics */
} bwd_q_ctx_t;

static double dot_d(const double *a, const double *b, int d) {
  double s = 0.0;
  for (int e = 0; e < d; ++e) s += a[e] * b[e];
  return s;
}

/* One item = one (b, h, i).  Query i sees keys j <= last = (Nk - Nq) + i.
 * scratch: dO_i (d), dq' (d), scores (Nk), dP (Nk). */
static void bwd_q_item(void *vctx, int64_t item, double *scratch) {
  bwd_q_ctx_t *c = (bwd_q_ctx_t *)vctx;
  int Nq = c->Nq, Nk = c->Nk, d = c->d;
  int64_t i = item % Nq;
  int h = (int)((item / Nq) % c->Hq);
  int b = (int)(item / ((int64_t)Nq * c->Hq));
  int hk = h / (c->Hq / c->Hkv);
  int64_t last = (int64_t)(Nk - Nq) + i;
  double *dOi = scratch, *dqr = scratch + d, *s = scratch + 2 * d, *dP = s + Nk;
  const double *qi = c->qrot + (((size_t)b * Nq + (size_t)i) * c->Hq + h) * d;
  size_t obase = (((size_t)b * Nq + (size_t)i) * c->Hq + h) * d;
  for (int e = 0; e < d; ++e) dOi[e] = load_elem(c->dout, c->dtype, obase + e);
  double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int64_t j = 0; j <= last; ++j) {
    const double *kj = c->krot + (((size_t)b * Nk + (size_t)j) * c->Hkv + hk) * d;
    s[j] = dot_d(qi, kj, d) * scale;
    if (s[j] > mx) mx = s[j];
    double dp = 0.0;
    size_t vbase = (((size_t)b * Nk + (size_t)j) * c->Hkv + hk) * d;
    for (int e = 0; e < d; ++e) dp += dOi[e] * load_elem(c->v, c->dtype, vbase + e);
    dP[j] = dp;
  }
  double den = 0.0;
  for (int64_t j = 0; j <= last; ++j) den += exp(s[j] - mx);
  double Dsum = 0.0;
  for (int64_t j = 0; j <= last; ++j) Dsum += exp(s[j] - mx) / den * dP[j];
  size_t st = ((size_t)b * c->Hq + h) * Nq + (size_t)i;
  c->m[st] = mx;
  c->l[st] = den;
  c->D[st] = Dsum;
  int64_t slot = c->qslot[i];
  if (slot < 0) return;
  for (int e = 0; e < d; ++e) dqr[e] = 0.0;
  for (int64_t j = 0; j <= last; ++j) {
    double dS = exp(s[j] - mx) / den * (dP[j] - Dsum);
    const double *kj = c->krot + (((size_t)b * Nk + (size_t)j) * c->Hkv + hk) * d;
    for (int e = 0; e < d; ++e) dqr[e] += dS * kj[e] * scale;
  }
  double *out = c->dq + (((size_t)b * (size_t)c->nq + (size_t)slot) * c->Hq + h) * d;
  double qp = c->qpos ? c->qpos[(size_t)b * Nq + (size_t)i] : (double)last;
  rope_rotate_vec(dqr, out, c->form, -qp, c->theta); /* R(p_i)^T */
}

typedef struct {
  const void *v, *dout;
  int dtype;
  int B, Hq, Hkv, Nq, Nk, d;
  rope_form_t form;
  const double *theta;
  const double *qrot, *krot;
  const double *kpos;        /* [B, Nk] rotation positions of the keys, or NULL: j */
  const int64_t *ksel;
  int64_t nk;
  const double *m, *l, *D;
  double *dk, *dv; /* [B, nk, Hkv, d] */
} bwd_k_ctx_t;

/* One item = one (b, hk, selected key row j).  Key j is seen by query rows i >= j - (Nk - Nq).
 * scratch: v_j (d), dk' (d), dv (d), dO_i (d). */
static void bwd_k_item(void *vctx, int64_t item, double *scratch) {
  bwd_k_ctx_t *c = (bwd_k_ctx_t *)vctx;
  int Nq = c->Nq, Nk = c->Nk, d = c->d;
  int64_t sl = item % c->nk;
  int hk = (int)((item / c->nk) % c->Hkv);
  int b = (int)(item / (c->nk * c->Hkv));
  int64_t j = c->ksel ? c->ksel[sl] : sl;
  int64_t first = j - (int64_t)(Nk - Nq);
  if (first < 0) first = 0;
  int g = c->Hq / c->Hkv;
  double *vj = scratch, *dkr = scratch + d, *dvj = scratch + 2 * d, *dOi = scratch + 3 * d;
  size_t vbase = (((size_t)b * Nk + (size_t)j) * c->Hkv + hk) * d;
  for (int e = 0; e < d; ++e) {
    vj[e] = load_elem(c->v, c->dtype, vbase + e);
    dkr[e] = 0.0;
    dvj[e] = 0.0;
  }
  const double *kj = c->krot + vbase;
  double scale = 1.0 / sqrt((double)d);
  for (int h = hk * g; h < (hk + 1) * g; ++h) {
    for (int64_t i = first; i < Nq; ++i) { /* causal: query rows that see key j */
      const double *qi = c->qrot + (((size_t)b * Nq + (size_t)i) * c->Hq + h) * d;
      size_t st = ((size_t)b * c->Hq + h) * Nq + (size_t)i;
      double p = exp(dot_d(qi, kj, d) * scale - c->m[st]) / c->l[st];
      size_t obase = (((size_t)b * Nq + (size_t)i) * c->Hq + h) * d;
      for (int e = 0; e < d; ++e) dOi[e] = load_elem(c->dout, c->dtype, obase + e);
      double dP = dot_d(dOi, vj, d);
      double dS = p * (dP - c->D[st]);
      for (int e = 0; e < d; ++e) {
        dvj[e] += p * dOi[e];
        dkr[e] += dS * qi[e] * scale;
      }
    }
  }
  size_t obase = (((size_t)b * c->nk + (size_t)sl) * c->Hkv + hk) * d;
  double kp = c->kpos ? c->kpos[(size_t)b * Nk + (size_t)j] : (double)j;
  rope_rotate_vec(dkr, c->dk + obase, c->form, -kp, c->theta); /* R(p_j)^T */
  for (int e = 0; e < d; ++e) c->dv[obase + e] = dvj[e];
}

typedef struct {
  const void *x;
  int dtype;
  int H, N;
  rope_form_t form;
  const double *theta;
  const double *pos; /* [B, N] positions, or NULL: pos_off + n */
  int pos_off;
  double *out;
} rot_all_ctx_t;

/* One item = one token (b, n): rotate its H head vectors at its position. */
static void rot_all_item(void *vctx, int64_t bn, double *scratch) {
  rot_all_ctx_t *c = (rot_all_ctx_t *)vctx;
  int d = c->form.d;
  double pos = c->pos ? c->pos[bn] : (double)(c->pos_off + bn % c->N);
  for (int h = 0; h < c->H; ++h) {
    size_t base = ((size_t)bn * c->H + h) * d;
    for (int e = 0; e < d; ++e) scratch[e] = load_elem(c->x, c->dtype, base + e);
    rope_rotate_vec(scratch, c->out + base, c->form, pos, c->theta);
  }
}

/* q_pos [B, Nq], k_pos [B, Nk]: rotation positions (NULL: the defaults), as for entry 3. */
int orc_rope_causal_bwd_kv(const void *q, const void *k, const void *v, const void *dout, int dtype, int B, int Hq,
                           int Hkv, int Nq, int Nk, int d, int rotary_dim, int interleaved, double base,
                           const double *q_pos, const double *k_pos, const int64_t *q_rows, int64_t nq,
                           const int64_t *k_rows, int64_t nk, double *dq, double *dk, double *dv, int nthreads) {
  rope_form_t f = {d, rotary_dim, interleaved};
  if (!q || !k || !v || !dout || !dq || !dk || !dv || B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < Nq ||
      !form_ok(f) || (Hq % Hkv) != 0)
    return -1;
  if (!q_rows) nq = Nq;
  if (!k_rows) nk = Nk;
  if (nq < 0 || nk < 0) return -1;
  for (int64_t s = 0; q_rows && s < nq; ++s)
    if (q_rows[s] < 0 || q_rows[s] >= Nq) return -1;
  for (int64_t s = 0; k_rows && s < nk; ++s)
    if (k_rows[s] < 0 || k_rows[s] >= Nk) return -1;

  size_t nst = (size_t)B * Hq * Nq;
  double *theta = (double *)malloc(sizeof(double) * (size_t)(f.r / 2));
  double *qrot = (double *)malloc(sizeof(double) * (size_t)B * Nq * Hq * d);
  double *krot = (double *)malloc(sizeof(double) * (size_t)B * Nk * Hkv * d);
  double *stats = (double *)malloc(sizeof(double) * 3 * nst);
  int64_t *qslot = (int64_t *)malloc(sizeof(int64_t) * (size_t)Nq);
  int rc = -1;
  if (theta && qrot && krot && stats && qslot) {
    rope_frequencies(f.r, base, theta);
    for (int64_t i = 0; i < Nq; ++i) qslot[i] = q_rows ? -1 : i;
    for (int64_t s = 0; q_rows && s < nq; ++s) qslot[q_rows[s]] = s;
    rot_all_ctx_t rq = {q, dtype, Hq, Nq, f, theta, q_pos, Nk - Nq, qrot};
    orc_pool_t p1 = {rot_all_item, &rq, (int64_t)B * Nq, 0, (size_t)d, 0};
    rot_all_ctx_t rk = {k, dtype, Hkv, Nk, f, theta, k_pos, 0, krot};
    orc_pool_t p2 = {rot_all_item, &rk, (int64_t)B * Nk, 0, (size_t)d, 0};
    rc = orc_run(&p1, nthreads);
    if (rc == 0) rc = orc_run(&p2, nthreads);
    if (rc == 0) {
      bwd_q_ctx_t qc = {v, dout, dtype, B, Hq, Hkv, Nq, Nk, d, f, theta, qrot, krot, q_pos, qslot, nq, dq,
                        stats, stats + nst, stats + 2 * nst};
      orc_pool_t p3 = {bwd_q_item, &qc, (int64_t)B * Hq * Nq, 0, (size_t)(2 * d + 2 * Nk), 0};
      rc = orc_run(&p3, nthreads);
    }
    if (rc == 0 && nk > 0) {
      bwd_k_ctx_t kc = {v, dout, dtype, B, Hq, Hkv, Nq, Nk, d, f, theta, qrot, krot, k_pos, k_rows, nk,
                        stats, stats + nst, stats + 2 * nst, dk, dv};
      orc_pool_t p4 = {bwd_k_item, &kc, (int64_t)B * Hkv * nk, 0, (size_t)(4 * d), 0};
      rc = orc_run(&p4, nthreads);
    }
  }
  free(theta);
  free(qrot);
  free(krot);
  free(stats);
  free(qslot);
  return rc;
}

int orc_rope_causal_bwd_ex(const void *q, const void *k, const void *v, const void *dout, int dtype, int B, int Hq,
                           int Hkv, int N, int d, int rotary_dim, int interleaved, double base, const double *q_pos,
                           const double *k_pos, const int64_t *q_rows, int64_t nq, const int64_t *k_rows, int64_t nk,
                           double *dq, double *dk, double *dv, int nthreads) {
  return orc_rope_causal_bwd_kv(q, k, v, dout, dtype, B, Hq, Hkv, N, N, d, rotary_dim, interleaved, base, q_pos, k_pos,
                                q_rows, nq, k_rows, nk, dq, dk, dv, nthreads);
}

int orc_rope_causal_bwd(const void *q, const void *k, const void *v, const void *dout, int dtype, int B, int Hq,
                        int Hkv, int N, int d, int rotary_dim, int interleaved, double base, const int64_t *q_rows,
                        int64_t nq, const int64_t *k_rows, int64_t nk, double *dq, double *dk, double *dv,
                        int nthreads) {
  return orc_rope_causal_bwd_ex(q, k, v, dout, dtype, B, Hq, Hkv, N, d, rotary_dim, interleaved, base, NULL, NULL,
                                q_rows, nq, k_rows, nk, dq, dk, dv, nthreads);
}
