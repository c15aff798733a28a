/*
 * rec_attn_oracle.c -- plain fp64 CPU oracle for masked time-RoPE softmax attention
 * over a packed, jagged, request-centric token sequence.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package smoke
 * check and the benchmark's CPU-baseline leg may load this library.  It shares no
 * code, header, table or constant with the CUDA path and must never serve as a
 * fallback for it.
 *
 * Everything here is the definition written out, in fp64, one row at a time:
 *
 *   - Softmax attention with an additive -inf mask, Softmax(QK^T/sqrt(d) + M) V:
 *     TM20K review page, section 2.1 (full-attention equation); LazFormer review
 *     page, section 2.3, Eq. 19-21 (SparseAttn).
 *   - Time-RoPE angle alpha_i(t) = t * phi_min / dt_max * base^(2i/d), applied to
 *     adjacent component pairs of Q and K: CADET review page, section on time
 *     encoding and self-gating.  The angle is formed from the absolute timestamp
 *     exactly as printed; fp64 keeps it accurate to ~1e-12 rad at Unix scale.
 *   - Mask predicate vis(i, j) (see orc_visible): CADET delay rule
 *     M_ij = -inf if t_j > t_i - delta (section "why mask the last hour");
 *     candidate isolation (section "scoring hundreds of candidates in 50 ms");
 *     SORT U2U / C2U / C2C regions (section 3.1) and local attention (3.2.1);
 *     LazFormer Eq. 19-21 (causal window + global history, target -> history,
 *     target self only); MTGR hybrid dynamic mask (static part fully visible,
 *     real-time block causal, targets see real-time events before them).
 *   - Fused prologue / epilogue steps (orc_attention_fused): QK-RMSNorm, the
 *     normalisation of each query and key head vector before the scores are formed
 *     (SORT review page, section 3.3.2 "Attention Gate & QK Norm"; TM20K review
 *     page, the QK Norm added after the query/key projections); the sigmoid gates
 *     on the projected Q and K (CADET review page, section on time encoding and
 *     self-gating: a per-dimension coefficient in (0, 1) multiplied back onto the
 *     vector); and the attention output gate, an elementwise sigmoid gate on the
 *     attention output (SORT section 3.3.2).  Order: norm, then gate, then RoPE.
 *   - Backward pass (orc_attention_bwd): the gradients of the attention above
 *     with respect to Q, K and V, written out by the chain rule on the materialised
 *     probabilities (dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dO * O)),
 *     dQ~ = scale dS K~, dK~ = scale dS^T Q~, then the inverse rotation).  The pages
 *     train these models (TM20K section 2.1, LazFormer's FlexAttention training)
 *     but print no backward formula; this is the derivative of the definition.
 *   - History compression (orc_compress): the history is merged by summing groups
 *     of consecutive tokens, the group size set per recency segment.  LazFormer
 *     review page, Eq. 16-18 (keep the most recent l tokens, sum the rest in groups
 *     of g, the last group partial) and its Table 6 configurations; TM20K review
 *     page, PATM (position segments with merge factors, zero-padded sums) and LPTM
 *     (sum of adjacent history pairs, targets never merged).
 *   - Query pruning (orc_kept_rows, orc_query_keep): only some queries are
 *     computed; every key stays.  SORT review page, section 3.2.2 (queries are
 *     pruned on the user side only, history and profile; candidates are never
 *     dropped); LazFormer review page, Eq. 22 (layer l keeps the most recent N_l
 *     history tokens and every target, N_l falling linearly from the history length
 *     to N_min) and the target-attention (TA) variant of the TM20K review page, in
 *     which only targets query the history (N_l = 0).
 *   - The tile classification (orc_tile_classes) is NOT a definition from the
 *     pages: it is the bounding-box interval rule this project uses to skip fully
 *     masked 128x128 tiles (the pages' "mask preload check" of SORT section 4.1 and
 *     the block skipping of the CADET serving kernel).  It is written here
 *     independently so the GPU planner can be checked bit-exactly against it; the
 *     tests check its soundness against the brute-force mask.
 *
 * Token types: 0 GLOBAL (special / profile / global summary), 1 HIST (history),
 * 2 RT (real-time block), 3 CAND (candidate / target).  Positions are local to a
 * request.  Tokens of different requests never see each other.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "rec_attn_oracle.h"

enum { TY_GLOBAL = 0, TY_HIST = 1, TY_RT = 2, TY_CAND = 3 };

/* ------------------------------------------------------------------------- */
/* Mask predicate                                                             */
/* ------------------------------------------------------------------------- */

/* Delay clause t_j <= t_i - delta, evaluated exactly in 128-bit integers. */
static int delay_clause(int64_t ti, int64_t tj, int64_t delta) {
  return (__int128)tj <= (__int128)ti - (__int128)delta;
}

static int is_user(int ty) { return ty == TY_GLOBAL || ty == TY_HIST; }

int orc_visible(const orc_params* p, int64_t pi, int64_t ti, int ty_i,
                int64_t pj, int64_t tj, int ty_j) {
  int vis;
  if (ty_i < 0 || ty_i > 3 || ty_j < 0 || ty_j > 3) return 0;
  if (is_user(ty_i) && is_user(ty_j)) {
    if (p->hist_bidirectional) {
      vis = 1; /* MTGR: profile + history fully mutually visible */
    } else {
      vis = (pj <= pi); /* causal user sequence (SORT U2U, LazFormer row 1) */
      if (vis && p->window > 0 && ty_i != TY_GLOBAL && ty_j != TY_GLOBAL)
        vis = (pi - pj) < p->window; /* local window; GLOBAL tokens exempt */
    }
  } else if (is_user(ty_i)) {
    vis = 0; /* the user side reads neither real-time events nor candidates */
  } else if (ty_i == TY_RT) {
    if (is_user(ty_j)) vis = 1;            /* real-time block reads the static part */
    else if (ty_j == TY_RT) vis = pj <= pi; /* and is causal inside itself */
    else vis = 0;                           /* and never reads candidates */
  } else { /* candidate query */
    if (is_user(ty_j)) vis = 1;            /* C2U full */
    else if (ty_j == TY_RT) vis = tj < ti;  /* real-time events strictly before it */
    else vis = (pi == pj);                  /* C2C: itself only */
  }
  if (p->use_delay) {
    int cand_self = (ty_i == TY_CAND && ty_j == TY_CAND && pi == pj);
    if (!cand_self) vis = vis && delay_clause(ti, tj, p->delay_s);
  }
  return vis;
}

void orc_mask(const orc_params* p, int64_t L, const int64_t* t, const int8_t* ty,
              uint8_t* out) {
  for (int64_t i = 0; i < L; ++i)
    for (int64_t j = 0; j < L; ++j)
      out[i * L + j] = (uint8_t)orc_visible(p, i, t[i], ty[i], j, t[j], ty[j]);
}

/* The block [i0, i0 + ni) x [j0, j0 + nj) of orc_mask, with 0 for an index past the
 * request end (no such token). */
void orc_mask_block(const orc_params* p, int64_t L, const int64_t* t, const int8_t* ty,
                    int64_t i0, int64_t ni, int64_t j0, int64_t nj, uint8_t* out) {
  for (int64_t a = 0; a < ni; ++a)
    for (int64_t c = 0; c < nj; ++c) {
      const int64_t i = i0 + a, j = j0 + c;
      out[a * nj + c] = (i < L && j < L) ? (uint8_t)orc_visible(p, i, t[i], ty[i], j, t[j], ty[j]) : 0;
    }
}

uint64_t orc_visible_pairs(const orc_params* p, int32_t B, const int64_t* offsets,
                           const int64_t* t, const int8_t* ty) {
  uint64_t n = 0;
  for (int32_t b = 0; b < B; ++b) {
    int64_t s = offsets[b], L = offsets[b + 1] - offsets[b];
    for (int64_t i = 0; i < L; ++i)
      for (int64_t j = 0; j < L; ++j)
        n += (uint64_t)orc_visible(p, i, t[s + i], ty[s + i], j, t[s + j], ty[s + j]);
  }
  return n;
}

/* ------------------------------------------------------------------------- */
/* Time-RoPE                                                                  */
/* ------------------------------------------------------------------------- */

void orc_rope(const orc_params* p, int64_t t, const double* x, double* y) {
  const int d = p->head_dim;
  for (int i = 0; i < d / 2; ++i) {
    double omega = p->phi_min / p->dt_max_s * pow(p->rope_base, 2.0 * i / d);
    double a = (double)t * omega;
    double c = cos(a), s = sin(a);
    y[2 * i] = x[2 * i] * c - x[2 * i + 1] * s;
    y[2 * i + 1] = x[2 * i] * s + x[2 * i + 1] * c;
  }
}

/* ------------------------------------------------------------------------- */
/* QK-RMSNorm and sigmoid gates                                               */
/* ------------------------------------------------------------------------- */

/* y = x / sqrt(mean(x^2) + eps) * w, over one head vector of length d. */
void orc_rmsnorm(const double* x, const double* w, int d, double eps, double* y) {
  double ss = 0.0;
  for (int e = 0; e < d; ++e) ss += x[e] * x[e];
  const double r = 1.0 / sqrt(ss / d + eps);
  for (int e = 0; e < d; ++e) y[e] = x[e] * r * w[e];
}

/* The logistic function 1 / (1 + e^-x). */
double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------------- */
/* Attention                                                                  */
/* ------------------------------------------------------------------------- */

static double load_elem(int dtype, const void* base, int64_t idx) {
  if (dtype == ORC_BF16) {
    uint16_t h = ((const uint16_t*)base)[idx];
    uint32_t bits = (uint32_t)h << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float*)base)[idx];
}

typedef struct {
  const orc_params* p;
  int32_t B;
  const int64_t* offsets;
  const int64_t* t;
  const int8_t* ty;
  int dtype;
  const void *q, *k, *v;
  /* selected rows: sorted global token indices; row_lo[b]..row_hi[b] index rows[] */
  const int64_t* rows;
  const int64_t* row_lo;
  const int64_t* row_hi;
  double* out; /* [n_rows][H][d] */
  double* lse; /* [n_rows][H] or NULL */
  const orc_fused* f; /* NULL: plain attention */
  int64_t n_units;
  int64_t next_unit; /* atomic work counter over (request, head) */
} attn_job;

/* One query (is_q) or key head vector of global token g: loaded, then QK-RMSNorm,
 * then the sigmoid gate, then the time-RoPE, in that order.  tmp holds d doubles. */
static void prep_row(const attn_job* J, int is_q, int64_t g, int32_t h, double* tmp, double* y) {
  const orc_params* p = J->p;
  const int H = p->num_heads, d = p->head_dim;
  const int64_t base = (g * H + h) * (int64_t)d;
  for (int e = 0; e < d; ++e) tmp[e] = load_elem(J->dtype, is_q ? J->q : J->k, base + e);
  if (J->f) {
    const double* w = is_q ? J->f->q_norm_w : J->f->k_norm_w;
    const void* gate = is_q ? J->f->q_gate : J->f->k_gate;
    if (w) {
      orc_rmsnorm(tmp, w + (int64_t)h * d, d, J->f->norm_eps, y);
      memcpy(tmp, y, sizeof(double) * d);
    }
    if (gate)
      for (int e = 0; e < d; ++e) tmp[e] *= orc_sigmoid(load_elem(J->dtype, gate, base + e));
  }
  if (p->use_rope) orc_rope(p, J->t[g], tmp, y);
  else memcpy(y, tmp, sizeof(double) * d);
}

static void attn_unit(attn_job* J, int32_t b, int32_t h, double* krot, double* vrow,
                      double* qin, double* qrot, double* s, uint8_t* vis) {
  const orc_params* p = J->p;
  const int H = p->num_heads, d = p->head_dim;
  const int64_t base = J->offsets[b], L = J->offsets[b + 1] - base;
  const double scale = p->softmax_scale > 0 ? p->softmax_scale : 1.0 / sqrt((double)d);
  (void)vrow;
  /* rotated keys of this request and head */
  for (int64_t j = 0; j < L; ++j) prep_row(J, 0, base + j, h, qin, krot + j * d);
  for (int64_t r = J->row_lo[b]; r < J->row_hi[b]; ++r) {
    const int64_t gi = J->rows[r], i = gi - base;
    prep_row(J, 1, gi, h, qin, qrot);
    /* one row of the mask and of the scores */
    double m = -INFINITY;
    int any = 0;
    for (int64_t j = 0; j < L; ++j) {
      vis[j] = (uint8_t)orc_visible(p, i, J->t[gi], J->ty[gi], j, J->t[base + j], J->ty[base + j]);
      if (!vis[j]) continue;
      double acc = 0.0;
      for (int e = 0; e < d; ++e) acc += qrot[e] * krot[j * d + e];
      s[j] = scale * acc;
      if (s[j] > m) m = s[j];
      any = 1;
    }
    double* o = J->out + (r * H + h) * (int64_t)d;
    for (int e = 0; e < d; ++e) o[e] = 0.0;
    if (!any) { /* no visible key: defined zero output, lse = -inf */
      if (J->lse) J->lse[r * H + h] = -INFINITY;
      continue;
    }
    double den = 0.0;
    for (int64_t j = 0; j < L; ++j)
      if (vis[j]) den += exp(s[j] - m);
    for (int64_t j = 0; j < L; ++j) {
      if (!vis[j]) continue;
      double w = exp(s[j] - m) / den;
      for (int e = 0; e < d; ++e)
        o[e] += w * load_elem(J->dtype, J->v, ((base + j) * H + h) * (int64_t)d + e);
    }
    if (J->f && J->f->out_gate) /* attention output gate */
      for (int e = 0; e < d; ++e)
        o[e] *= orc_sigmoid(load_elem(J->dtype, J->f->out_gate, (gi * H + h) * (int64_t)d + e));
    if (J->lse) J->lse[r * H + h] = m + log(den);
  }
}

static void* attn_worker(void* arg) {
  attn_job* J = (attn_job*)arg;
  const int d = J->p->head_dim;
  int64_t Lmax = 0;
  for (int32_t b = 0; b < J->B; ++b) {
    int64_t L = J->offsets[b + 1] - J->offsets[b];
    if (L > Lmax) Lmax = L;
  }
  double* krot = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1) * d);
  double* s = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
  uint8_t* vis = (uint8_t*)malloc((size_t)(Lmax > 0 ? Lmax : 1));
  double* qin = (double*)malloc(sizeof(double) * d);
  double* qrot = (double*)malloc(sizeof(double) * d);
  for (;;) {
    int64_t u = __atomic_fetch_add(&J->next_unit, 1, __ATOMIC_RELAXED);
    if (u >= J->n_units) break;
    int32_t b = (int32_t)(u / J->p->num_heads), h = (int32_t)(u % J->p->num_heads);
    if (J->row_hi[b] > J->row_lo[b]) attn_unit(J, b, h, krot, NULL, qin, qrot, s, vis);
  }
  free(krot); free(s); free(vis); free(qin); free(qrot);
  return NULL;
}

int orc_attention(const orc_params* p, int32_t B, const int64_t* offsets,
                  const int64_t* t, const int8_t* ty, int32_t dtype,
                  const void* q, const void* k, const void* v,
                  int64_t n_rows, const int64_t* rows, double* out, double* lse,
                  int32_t n_threads) {
  return orc_attention_fused(p, B, offsets, t, ty, dtype, q, k, v, NULL, n_rows, rows, out, lse,
                             n_threads);
}

int orc_attention_fused(const orc_params* p, int32_t B, const int64_t* offsets,
                        const int64_t* t, const int8_t* ty, int32_t dtype,
                        const void* q, const void* k, const void* v, const orc_fused* f,
                        int64_t n_rows, const int64_t* rows, double* out, double* lse,
                        int32_t n_threads) {
  if (f && !(f->norm_eps >= 0.0)) return -1;
  if (!p || B < 0 || !offsets || p->num_heads <= 0 || p->head_dim <= 0 || (p->head_dim & 1))
    return -1;
  if (dtype != ORC_BF16 && dtype != ORC_FP32) return -1;
  for (int32_t b = 0; b < B; ++b)
    if (offsets[b + 1] < offsets[b]) return -1;
  const int64_t T = offsets[B] - offsets[0];
  int64_t* all_rows = NULL;
  if (!rows) { /* every token of the batch */
    n_rows = T;
    all_rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T > 0 ? T : 1));
    for (int64_t r = 0; r < T; ++r) all_rows[r] = offsets[0] + r;
    rows = all_rows;
  }
  for (int64_t r = 0; r < n_rows; ++r) {
    if (rows[r] < offsets[0] || rows[r] >= offsets[B]) { free(all_rows); return -2; }
    if (r > 0 && rows[r] <= rows[r - 1]) { free(all_rows); return -2; } /* must be sorted */
  }
  int64_t* lo = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  int64_t* hi = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  int64_t r = 0;
  for (int32_t b = 0; b < B; ++b) {
    while (r < n_rows && rows[r] < offsets[b]) ++r;
    lo[b] = r;
    while (r < n_rows && rows[r] < offsets[b + 1]) ++r;
    hi[b] = r;
  }
  attn_job J = {p, B, offsets, t, ty, dtype, q, k, v, rows, lo, hi, out, lse, f,
                (int64_t)B * p->num_heads, 0};
  if (n_threads < 1) n_threads = 1;
  if (n_threads == 1) {
    attn_worker(&J);
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, attn_worker, &J);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
    free(th);
  }
  free(lo); free(hi); free(all_rows);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Backward pass                                                              */
/* ------------------------------------------------------------------------- */

/* y = R(t)^T x: the inverse of orc_rope (rotation by the negative angle). */
static void rope_inverse(const orc_params* p, int64_t t, const double* x, double* y) {
  const int d = p->head_dim;
  for (int i = 0; i < d / 2; ++i) {
    double omega = p->phi_min / p->dt_max_s * pow(p->rope_base, 2.0 * i / d);
    double a = (double)t * omega;
    double c = cos(a), s = sin(a);
    y[2 * i] = x[2 * i] * c + x[2 * i + 1] * s;
    y[2 * i + 1] = -x[2 * i] * s + x[2 * i + 1] * c;
  }
}

typedef struct {
  const orc_params* p;
  int32_t B;
  const int64_t *offsets, *t;
  const int8_t* ty;
  int dtype;
  const void *q, *k, *v, *dout;
  double *dq, *dk, *dv; /* [T][H][d] */
  int64_t n_units, next_unit;
} bwd_job;

static void bwd_unit(bwd_job* J, int32_t b, int32_t h) {
  const orc_params* p = J->p;
  const int H = p->num_heads, d = p->head_dim;
  const int64_t base = J->offsets[b], L = J->offsets[b + 1] - base;
  if (L <= 0) return;
  const double scale = p->softmax_scale > 0 ? p->softmax_scale : 1.0 / sqrt((double)d);
  double* qr = (double*)malloc(sizeof(double) * (size_t)L * d);  /* rotated queries */
  double* kr = (double*)malloc(sizeof(double) * (size_t)L * d);  /* rotated keys */
  double* vv = (double*)malloc(sizeof(double) * (size_t)L * d);
  double* go = (double*)malloc(sizeof(double) * (size_t)L * d);  /* dO */
  double* P = (double*)calloc((size_t)L * L, sizeof(double));    /* probabilities, 0 where masked */
  double* gq = (double*)calloc((size_t)L * d, sizeof(double));   /* dQ~ */
  double* gk = (double*)calloc((size_t)L * d, sizeof(double));   /* dK~ */
  double* tmp = (double*)malloc(sizeof(double) * d);
  for (int64_t i = 0; i < L; ++i) {
    const int64_t off = ((base + i) * H + h) * (int64_t)d;
    for (int e = 0; e < d; ++e) {
      tmp[e] = load_elem(J->dtype, J->q, off + e);
      vv[i * d + e] = load_elem(J->dtype, J->v, off + e);
      go[i * d + e] = load_elem(J->dtype, J->dout, off + e);
    }
    if (p->use_rope) orc_rope(p, J->t[base + i], tmp, qr + i * d);
    else memcpy(qr + i * d, tmp, sizeof(double) * d);
    for (int e = 0; e < d; ++e) tmp[e] = load_elem(J->dtype, J->k, off + e);
    if (p->use_rope) orc_rope(p, J->t[base + i], tmp, kr + i * d);
    else memcpy(kr + i * d, tmp, sizeof(double) * d);
  }
  /* forward probabilities row by row */
  for (int64_t i = 0; i < L; ++i) {
    double m = -INFINITY;
    double* Pi = P + i * L;
    for (int64_t j = 0; j < L; ++j) {
      if (!orc_visible(p, i, J->t[base + i], J->ty[base + i], j, J->t[base + j], J->ty[base + j])) {
        Pi[j] = -INFINITY;
        continue;
      }
      double acc = 0.0;
      for (int e = 0; e < d; ++e) acc += qr[i * d + e] * kr[j * d + e];
      Pi[j] = scale * acc;
      if (Pi[j] > m) m = Pi[j];
    }
    if (m == -INFINITY) { /* no visible key: O = 0, no gradient flows */
      for (int64_t j = 0; j < L; ++j) Pi[j] = 0.0;
      continue;
    }
    double den = 0.0;
    for (int64_t j = 0; j < L; ++j) den += (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - m);
    for (int64_t j = 0; j < L; ++j) Pi[j] = (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - m) / den;
  }
  /* dV = P^T dO; D_i = sum_j P_ij dP_ij; dS = P (dP - D); dQ~ = scale dS K~; dK~ = scale dS^T Q~ */
  for (int64_t i = 0; i < L; ++i) {
    const double* Pi = P + i * L;
    double Di = 0.0;
    for (int64_t j = 0; j < L; ++j) {
      if (Pi[j] == 0.0) continue;
      double dp = 0.0;
      for (int e = 0; e < d; ++e) dp += go[i * d + e] * vv[j * d + e];
      Di += Pi[j] * dp;
    }
    for (int64_t j = 0; j < L; ++j) {
      if (Pi[j] == 0.0) continue;
      double dp = 0.0;
      for (int e = 0; e < d; ++e) dp += go[i * d + e] * vv[j * d + e];
      const double ds = Pi[j] * (dp - Di);
      for (int e = 0; e < d; ++e) {
        J->dv[((base + j) * H + h) * (int64_t)d + e] += Pi[j] * go[i * d + e];
        gq[i * d + e] += scale * ds * kr[j * d + e];
        gk[j * d + e] += scale * ds * qr[i * d + e];
      }
    }
  }
  /* back through the rotation */
  for (int64_t i = 0; i < L; ++i) {
    double* dqo = J->dq + ((base + i) * H + h) * (int64_t)d;
    double* dko = J->dk + ((base + i) * H + h) * (int64_t)d;
    if (p->use_rope) {
      rope_inverse(p, J->t[base + i], gq + i * d, dqo);
      rope_inverse(p, J->t[base + i], gk + i * d, dko);
    } else {
      memcpy(dqo, gq + i * d, sizeof(double) * d);
      memcpy(dko, gk + i * d, sizeof(double) * d);
    }
  }
  free(qr); free(kr); free(vv); free(go); free(P); free(gq); free(gk); free(tmp);
}

static void* bwd_worker(void* arg) {
  bwd_job* J = (bwd_job*)arg;
  for (;;) {
    int64_t u = __atomic_fetch_add(&J->next_unit, 1, __ATOMIC_RELAXED);
    if (u >= J->n_units) break;
    bwd_unit(J, (int32_t)(u / J->p->num_heads), (int32_t)(u % J->p->num_heads));
  }
  return NULL;
}

int orc_attention_bwd(const orc_params* p, int32_t B, const int64_t* offsets, const int64_t* t,
                      const int8_t* ty, int32_t dtype, const void* q, const void* k, const void* v,
                      const void* dout, double* dq, double* dk, double* dv, int32_t n_threads) {
  if (!p || B < 0 || !offsets || p->num_heads <= 0 || p->head_dim <= 0 || (p->head_dim & 1)) return -1;
  if (dtype != ORC_BF16 && dtype != ORC_FP32) return -1;
  for (int32_t b = 0; b < B; ++b)
    if (offsets[b + 1] < offsets[b]) return -1;
  const int64_t n = (offsets[B] - offsets[0]) * p->num_heads * (int64_t)p->head_dim;
  memset(dq, 0, sizeof(double) * (size_t)n);
  memset(dk, 0, sizeof(double) * (size_t)n);
  memset(dv, 0, sizeof(double) * (size_t)n);
  bwd_job J = {p, B, offsets, t, ty, dtype, q, k, v, dout, dq, dk, dv, (int64_t)B * p->num_heads, 0};
  if (n_threads < 1) n_threads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, bwd_worker, &J);
  for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  free(th);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Backward pass through the fused steps                                      */
/* ------------------------------------------------------------------------- */

/* The chain rule through the steps orc_attention_fused applies, in reverse order:
 *   forward, per query / key head vector a:  n = a / r * w  (r = sqrt(mean(a^2) + eps),
 *   when a norm gain is given), g = n * sigmoid(c) (when a gate is given), x = R(t) g;
 *   the attention on the x's gives A; the output is O = A * sigmoid(c_o).
 *   backward:  dA = dO * sigmoid(c_o),  dc_o = dO * A * sigmoid'(c_o);
 *   the attention backward (bwd_unit's formulas) with dA gives dx_q, dx_k and dV;
 *   dg = R(t)^T dx;  dc = dg * n * sigmoid'(c),  dn = dg * sigmoid(c);
 *   da = (w * dn) / r - a * sum_e(dn_e w_e a_e) / (d r^3),  dw += dn * a / r.
 * sigmoid'(c) = sigmoid(c) (1 - sigmoid(c)).  Every quantity is fp64. */
typedef struct {
  const orc_params* p;
  int32_t B;
  const int64_t *offsets, *t;
  const int8_t* ty;
  int dtype;
  const void *q, *k, *v, *dout;
  const orc_fused* f;
  double *dq, *dk, *dv, *dqg, *dkg, *dog; /* [T][H][d] */
  double *dqw, *dkw;                      /* [B][H][d]: per-request parts of the gain gradients */
  int64_t n_units, next_unit;
} fbwd_job;

/* The forward steps of one head vector: a (input), n (normalised), sg (the gate's
 * sigmoid, 1 without a gate), r (the norm's root mean square, 1 without a norm) and
 * the rotated x. */
static void fbwd_prep(const fbwd_job* J, int is_q, int64_t g, int32_t h, double* a, double* n, double* sg,
                      double* r, double* x) {
  const orc_params* p = J->p;
  const int H = p->num_heads, d = p->head_dim;
  const int64_t base = (g * H + h) * (int64_t)d;
  const double* w = is_q ? J->f->q_norm_w : J->f->k_norm_w;
  const void* gate = is_q ? J->f->q_gate : J->f->k_gate;
  for (int e = 0; e < d; ++e) a[e] = load_elem(J->dtype, is_q ? J->q : J->k, base + e);
  *r = 1.0;
  if (w) {
    double ss = 0.0;
    for (int e = 0; e < d; ++e) ss += a[e] * a[e];
    *r = sqrt(ss / d + J->f->norm_eps);
    for (int e = 0; e < d; ++e) n[e] = a[e] / *r * w[(int64_t)h * d + e];
  } else {
    memcpy(n, a, sizeof(double) * d);
  }
  double* gv = x; /* the gated vector, rotated in place below */
  for (int e = 0; e < d; ++e) {
    sg[e] = gate ? orc_sigmoid(load_elem(J->dtype, gate, base + e)) : 1.0;
    gv[e] = n[e] * sg[e];
  }
  if (p->use_rope) {
    double* tmp = (double*)malloc(sizeof(double) * d);
    orc_rope(p, J->t[g], gv, tmp);
    memcpy(x, tmp, sizeof(double) * d);
    free(tmp);
  }
}

/* dg -> da (and the gate and gain gradients) for one head vector. */
static void fbwd_back(const fbwd_job* J, int is_q, int32_t b, int64_t g, int32_t h, const double* dg,
                      const double* a, const double* n, const double* sg, double r) {
  const orc_params* p = J->p;
  const int H = p->num_heads, d = p->head_dim;
  const int64_t base = (g * H + h) * (int64_t)d;
  const double* w = is_q ? J->f->q_norm_w : J->f->k_norm_w;
  const void* gate = is_q ? J->f->q_gate : J->f->k_gate;
  double* da = (is_q ? J->dq : J->dk) + base;
  double* dc = (is_q ? J->dqg : J->dkg) + base;
  double* dw = (is_q ? J->dqw : J->dkw) + ((int64_t)b * H + h) * d;
  double dot = 0.0;
  for (int e = 0; e < d; ++e) {
    const double dn = dg[e] * sg[e];
    dc[e] = gate ? dg[e] * n[e] * sg[e] * (1.0 - sg[e]) : 0.0;
    if (w) {
      dot += dn * w[(int64_t)h * d + e] * a[e];
      dw[e] += dn * a[e] / r;
    }
  }
  for (int e = 0; e < d; ++e) {
    const double dn = dg[e] * sg[e];
    da[e] = w ? w[(int64_t)h * d + e] * dn / r - a[e] * dot / (d * r * r * r) : dn;
  }
}

static void fbwd_unit(fbwd_job* J, int32_t b, int32_t h) {
  const orc_params* p = J->p;
  const int H = p->num_heads, d = p->head_dim;
  const int64_t base = J->offsets[b], L = J->offsets[b + 1] - base;
  if (L <= 0) return;
  const double scale = p->softmax_scale > 0 ? p->softmax_scale : 1.0 / sqrt((double)d);
  const size_t Ld = (size_t)L * d;
  double *qa = malloc(sizeof(double) * Ld), *qn = malloc(sizeof(double) * Ld), *qs = malloc(sizeof(double) * Ld);
  double *ka = malloc(sizeof(double) * Ld), *kn = malloc(sizeof(double) * Ld), *ks = malloc(sizeof(double) * Ld);
  double *qx = malloc(sizeof(double) * Ld), *kx = malloc(sizeof(double) * Ld);
  double *qr = malloc(sizeof(double) * L), *kr = malloc(sizeof(double) * L);
  double *vv = malloc(sizeof(double) * Ld), *dA = malloc(sizeof(double) * Ld);
  double* P = calloc((size_t)L * L, sizeof(double));
  double *gq = calloc(Ld, sizeof(double)), *gk = calloc(Ld, sizeof(double));
  double* tmp = malloc(sizeof(double) * d);
  for (int64_t i = 0; i < L; ++i) {
    fbwd_prep(J, 1, base + i, h, qa + i * d, qn + i * d, qs + i * d, qr + i, qx + i * d);
    fbwd_prep(J, 0, base + i, h, ka + i * d, kn + i * d, ks + i * d, kr + i, kx + i * d);
    for (int e = 0; e < d; ++e) vv[i * d + e] = load_elem(J->dtype, J->v, ((base + i) * H + h) * (int64_t)d + e);
  }
  /* probabilities (0 where masked or for a row that sees nothing) */
  for (int64_t i = 0; i < L; ++i) {
    double m = -INFINITY;
    double* Pi = P + i * L;
    for (int64_t j = 0; j < L; ++j) {
      if (!orc_visible(p, i, J->t[base + i], J->ty[base + i], j, J->t[base + j], J->ty[base + j])) {
        Pi[j] = -INFINITY;
        continue;
      }
      double acc = 0.0;
      for (int e = 0; e < d; ++e) acc += qx[i * d + e] * kx[j * d + e];
      Pi[j] = scale * acc;
      if (Pi[j] > m) m = Pi[j];
    }
    if (m == -INFINITY) {
      for (int64_t j = 0; j < L; ++j) Pi[j] = 0.0;
      continue;
    }
    double den = 0.0;
    for (int64_t j = 0; j < L; ++j) den += (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - m);
    for (int64_t j = 0; j < L; ++j) Pi[j] = (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - m) / den;
  }
  /* the output gate: dA = dO * sigmoid(c_o), dc_o = dO * A * sigmoid'(c_o) */
  for (int64_t i = 0; i < L; ++i) {
    const int64_t off = ((base + i) * H + h) * (int64_t)d;
    for (int e = 0; e < d; ++e) {
      double A = 0.0;
      for (int64_t j = 0; j < L; ++j) A += P[i * L + j] * vv[j * d + e];
      const double go = load_elem(J->dtype, J->dout, off + e);
      const double so = J->f->out_gate ? orc_sigmoid(load_elem(J->dtype, J->f->out_gate, off + e)) : 1.0;
      dA[i * d + e] = go * so;
      J->dog[off + e] = J->f->out_gate ? go * A * so * (1.0 - so) : 0.0;
    }
  }
  /* the attention backward with dA */
  for (int64_t i = 0; i < L; ++i) {
    const double* Pi = P + i * L;
    double Di = 0.0;
    for (int64_t j = 0; j < L; ++j) {
      if (Pi[j] == 0.0) continue;
      double dp = 0.0;
      for (int e = 0; e < d; ++e) dp += dA[i * d + e] * vv[j * d + e];
      Di += Pi[j] * dp;
    }
    for (int64_t j = 0; j < L; ++j) {
      if (Pi[j] == 0.0) continue;
      double dp = 0.0;
      for (int e = 0; e < d; ++e) dp += dA[i * d + e] * vv[j * d + e];
      const double ds = Pi[j] * (dp - Di);
      for (int e = 0; e < d; ++e) {
        J->dv[((base + j) * H + h) * (int64_t)d + e] += Pi[j] * dA[i * d + e];
        gq[i * d + e] += scale * ds * kx[j * d + e];
        gk[j * d + e] += scale * ds * qx[i * d + e];
      }
    }
  }
  /* back through the rotation, the gates and the norms */
  for (int64_t i = 0; i < L; ++i) {
    if (p->use_rope) rope_inverse(p, J->t[base + i], gq + i * d, tmp);
    else memcpy(tmp, gq + i * d, sizeof(double) * d);
    fbwd_back(J, 1, b, base + i, h, tmp, qa + i * d, qn + i * d, qs + i * d, qr[i]);
    if (p->use_rope) rope_inverse(p, J->t[base + i], gk + i * d, tmp);
    else memcpy(tmp, gk + i * d, sizeof(double) * d);
    fbwd_back(J, 0, b, base + i, h, tmp, ka + i * d, kn + i * d, ks + i * d, kr[i]);
  }
  free(qa); free(qn); free(qs); free(ka); free(kn); free(ks); free(qx); free(kx); free(qr); free(kr);
  free(vv); free(dA); free(P); free(gq); free(gk); free(tmp);
}

static void* fbwd_worker(void* arg) {
  fbwd_job* J = (fbwd_job*)arg;
  for (;;) {
    int64_t u = __atomic_fetch_add(&J->next_unit, 1, __ATOMIC_RELAXED);
    if (u >= J->n_units) break;
    fbwd_unit(J, (int32_t)(u / J->p->num_heads), (int32_t)(u % J->p->num_heads));
  }
  return NULL;
}

int orc_attention_bwd_fused(const orc_params* p, int32_t B, const int64_t* offsets, const int64_t* t,
                            const int8_t* ty, int32_t dtype, const void* q, const void* k, const void* v,
                            const orc_fused* f, const void* dout, double* dq, double* dk, double* dv,
                            double* dq_gate, double* dk_gate, double* dout_gate, double* dq_norm_w,
                            double* dk_norm_w, int32_t n_threads) {
  if (!p || !f || B < 0 || !offsets || p->num_heads <= 0 || p->head_dim <= 0 || (p->head_dim & 1)) return -1;
  if (dtype != ORC_BF16 && dtype != ORC_FP32) return -1;
  if (!(f->norm_eps >= 0.0) || offsets[0] != 0) return -1;
  for (int32_t b = 0; b < B; ++b)
    if (offsets[b + 1] < offsets[b]) return -1;
  const int H = p->num_heads, d = p->head_dim;
  const int64_t n = offsets[B] * H * (int64_t)d;
  double* outs[6] = {dq, dk, dv, dq_gate, dk_gate, dout_gate};
  for (int i = 0; i < 6; ++i) memset(outs[i], 0, sizeof(double) * (size_t)n);
  const size_t nw = (size_t)(B > 0 ? B : 1) * H * d;
  double* pq = calloc(nw, sizeof(double));
  double* pk = calloc(nw, sizeof(double));
  fbwd_job J = {p, B, offsets, t, ty, dtype, q, k, v, dout, f, dq, dk, dv, dq_gate, dk_gate, dout_gate,
                pq, pk, (int64_t)B * H, 0};
  if (n_threads < 1) n_threads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, fbwd_worker, &J);
  for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  free(th);
  /* the gains' gradients: the requests' parts summed in request order */
  for (int64_t e = 0; e < (int64_t)H * d; ++e) {
    double sq = 0.0, sk = 0.0;
    for (int32_t b = 0; b < B; ++b) {
      sq += pq[(int64_t)b * H * d + e];
      sk += pk[(int64_t)b * H * d + e];
    }
    if (dq_norm_w) dq_norm_w[e] = sq;
    if (dk_norm_w) dk_norm_w[e] = sk;
  }
  free(pq); free(pk);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* History compression                                                        */
/* ------------------------------------------------------------------------- */

/* Groups of one request's history of Lh tokens under the segment spec: segment i
 * (i = 0 the most recent) covers the next seg_len[i] tokens going back in time
 * (seg_len < 0: all the rest) and merges them in groups of seg_group[i], the oldest
 * group of a segment being the partial one.  Writes the groups oldest first as
 * [first, last) history indices (0 = oldest) and returns their count; lo/hi may be
 * NULL to count. */
static int64_t history_groups(int64_t Lh, int32_t n_seg, const int64_t* seg_len, const int32_t* seg_group,
                              int64_t* lo, int64_t* hi) {
  int64_t n = 0, rank = 0; /* rank: tokens already covered, counted from the newest */
  /* segments are laid out from the newest; the output wants the oldest first, so
   * collect per segment and emit in reverse at the end */
  int64_t nseg_groups[64];
  int64_t seg_start[64], seg_m[64];
  int32_t used = 0;
  for (int32_t i = 0; i < n_seg && rank < Lh && i < 64; ++i) {
    const int64_t room = Lh - rank;
    const int64_t m = (seg_len[i] < 0 || seg_len[i] > room) ? room : seg_len[i];
    const int64_t g = seg_group[i];
    seg_start[used] = rank;
    seg_m[used] = m;
    nseg_groups[used] = (m + g - 1) / g;
    ++used;
    rank += m;
  }
  if (rank < Lh) return -1; /* the spec does not cover the whole history */
  for (int32_t u = used - 1; u >= 0; --u) {
    const int32_t g = seg_group[u];
    for (int64_t q = nseg_groups[u] - 1; q >= 0; --q) { /* q = 0 is the newest group */
      const int64_t r0 = seg_start[u] + q * g;                        /* newest rank in it */
      const int64_t r1 = seg_start[u] + ((q + 1) * g < seg_m[u] ? (q + 1) * g : seg_m[u]); /* past oldest */
      if (lo) { lo[n] = Lh - r1; hi[n] = Lh - r0; }
      ++n;
    }
  }
  return n;
}

int64_t orc_compress(int32_t B, const int64_t* offsets, const int64_t* hist_begin, const int64_t* hist_len,
                     int32_t n_seg, const int64_t* seg_len, const int32_t* seg_group, int32_t dtype, int64_t width,
                     const void* x, const int64_t* t, const int8_t* ty, int64_t* out_offsets, double* out_x,
                     int64_t* out_t, int8_t* out_ty) {
  if (B < 0 || !offsets || n_seg < 1 || n_seg > 64 || width < 1) return -1;
  for (int32_t i = 0; i < n_seg; ++i)
    if (seg_group[i] < 1) return -1;
  int64_t n_out = 0;
  if (out_offsets) out_offsets[0] = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t s = offsets[b], L = offsets[b + 1] - s, hb = hist_begin[b], Lh = hist_len[b];
    if (L < 0 || hb < 0 || Lh < 0 || hb + Lh > L) return -1;
    const int64_t G = history_groups(Lh, n_seg, seg_len, seg_group, NULL, NULL);
    if (G < 0) return -1;
    int64_t* glo = (int64_t*)malloc(sizeof(int64_t) * (size_t)(G > 0 ? G : 1));
    int64_t* ghi = (int64_t*)malloc(sizeof(int64_t) * (size_t)(G > 0 ? G : 1));
    history_groups(Lh, n_seg, seg_len, seg_group, glo, ghi);
    const int64_t Lo = L - Lh + G;
    if (out_x) {
      int64_t o = n_out;
      for (int64_t p = 0; p < hb; ++p, ++o) { /* tokens before the history */
        for (int64_t e = 0; e < width; ++e) out_x[o * width + e] = load_elem(dtype, x, (s + p) * width + e);
        out_t[o] = t[s + p]; out_ty[o] = ty[s + p];
      }
      for (int64_t gi = 0; gi < G; ++gi, ++o) { /* merged groups: sums, latest time */
        int64_t tmax = INT64_MIN;
        for (int64_t e = 0; e < width; ++e) out_x[o * width + e] = 0.0;
        for (int64_t j = glo[gi]; j < ghi[gi]; ++j) {
          const int64_t g = s + hb + j;
          for (int64_t e = 0; e < width; ++e) out_x[o * width + e] += load_elem(dtype, x, g * width + e);
          if (t[g] > tmax) tmax = t[g];
        }
        out_t[o] = tmax; out_ty[o] = TY_HIST;
      }
      for (int64_t p = hb + Lh; p < L; ++p, ++o) { /* tokens after the history */
        for (int64_t e = 0; e < width; ++e) out_x[o * width + e] = load_elem(dtype, x, (s + p) * width + e);
        out_t[o] = t[s + p]; out_ty[o] = ty[s + p];
      }
    }
    free(glo); free(ghi);
    n_out += Lo;
    if (out_offsets) out_offsets[b + 1] = n_out;
  }
  return n_out;
}

/* ------------------------------------------------------------------------- */
/* Query pruning                                                              */
/* ------------------------------------------------------------------------- */

/* LazFormer Eq. 22: N_l = min(Lh, max(N_min, Round[Lh - (l-1)/(L-1) (Lh - N_min)]))
 * for layer l of L (1-based); Round is round-half-away-from-zero.  A single layer
 * keeps the whole history. */
int64_t orc_query_keep(int64_t hist_len, int64_t n_min, int32_t layer, int32_t n_layers) {
  if (hist_len < 0 || n_min < 0 || n_layers < 1 || layer < 1 || layer > n_layers) return -1;
  if (n_layers == 1) return hist_len;
  const double x = (double)hist_len - (double)(layer - 1) / (double)(n_layers - 1) * (double)(hist_len - n_min);
  int64_t r = (int64_t)floor(fabs(x) + 0.5);
  if (x < 0) r = -r;
  if (r < n_min) r = n_min;
  if (r > hist_len) r = hist_len;
  return r;
}

/* Rows a pruned layer computes, as sorted global token indices: in each request,
 * every token that is not a user token (real-time events, candidates) and the last
 * `keep` user tokens (GLOBAL or HIST) by position; keep < 0 keeps every token.
 * Returns the number of rows (rows may be NULL to count). */
int64_t orc_kept_rows(int32_t B, const int64_t* offsets, const int8_t* ty, int64_t keep, int64_t* rows) {
  int64_t n = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t s = offsets[b], e = offsets[b + 1];
    int64_t seen = 0; /* user tokens at or after the current position */
    int64_t first_kept = s; /* the first kept user token's global index */
    if (keep >= 0) {
      first_kept = e;
      for (int64_t g = e - 1; g >= s; --g)
        if (is_user(ty[g])) {
          if (seen == keep) break;
          ++seen;
          first_kept = g;
        }
    }
    for (int64_t g = s; g < e; ++g)
      if (!is_user(ty[g]) || g >= first_kept) {
        if (rows) rows[n] = g;
        ++n;
      }
  }
  return n;
}

/* ------------------------------------------------------------------------- */
/* Tile classification (bounding-box interval rule)                           */
/* ------------------------------------------------------------------------- */

/* Three-valued clause outcome; with NONE < SOME < ALL a conjunction is the
 * minimum and a disjunction the maximum. */
enum { TV_NONE = 0, TV_SOME = 1, TV_ALL = 2 };

typedef struct { int64_t cnt, pmin, pmax, tmin, tmax; } orc_box;

static int tv_min(int a, int b) { return a < b ? a : b; }

static int tv_causal(const orc_box* q, const orc_box* k) { /* p_j <= p_i */
  if (k->pmax <= q->pmin) return TV_ALL;
  if (k->pmin > q->pmax) return TV_NONE;
  return TV_SOME;
}
static int tv_window(const orc_box* q, const orc_box* k, int64_t W) { /* p_i - p_j < W */
  if (q->pmax - k->pmin < W) return TV_ALL;
  if (q->pmin - k->pmax >= W) return TV_NONE;
  return TV_SOME;
}
static int tv_delay(const orc_box* q, const orc_box* k, int64_t delta) { /* t_j <= t_i - delta */
  if ((__int128)k->tmax <= (__int128)q->tmin - delta) return TV_ALL;
  if ((__int128)k->tmin > (__int128)q->tmax - delta) return TV_NONE;
  return TV_SOME;
}
static int tv_before(const orc_box* q, const orc_box* k) { /* t_j < t_i */
  if (k->tmax < q->tmin) return TV_ALL;
  if (k->tmin >= q->tmax) return TV_NONE;
  return TV_SOME;
}
static int tv_diag(const orc_box* q, const orc_box* k) { /* i == j; never ALL */
  if (k->pmax < q->pmin || k->pmin > q->pmax) return TV_NONE;
  return TV_SOME;
}

static int tv_pair(const orc_params* p, int tq, int tk, const orc_box* q, const orc_box* k) {
  int v;
  if (is_user(tq) && is_user(tk)) {
    if (p->hist_bidirectional) v = TV_ALL;
    else {
      v = tv_causal(q, k);
      if (p->window > 0 && tq != TY_GLOBAL && tk != TY_GLOBAL) v = tv_min(v, tv_window(q, k, p->window));
    }
  } else if (is_user(tq)) v = TV_NONE;
  else if (tq == TY_RT) v = is_user(tk) ? TV_ALL : (tk == TY_RT ? tv_causal(q, k) : TV_NONE);
  else v = is_user(tk) ? TV_ALL : (tk == TY_RT ? tv_before(q, k) : tv_diag(q, k));
  /* candidate -> candidate is its own diagonal, exempt from the delay */
  if (p->use_delay && !(tq == TY_CAND && tk == TY_CAND)) v = tv_min(v, tv_delay(q, k, p->delay_s));
  return v;
}

static void tile_boxes(int64_t base, int64_t L, int64_t tile, const int64_t* t,
                       const int8_t* ty, orc_box box[4]) {
  for (int c = 0; c < 4; ++c) {
    box[c].cnt = 0; box[c].pmin = INT64_MAX; box[c].pmax = INT64_MIN;
    box[c].tmin = INT64_MAX; box[c].tmax = INT64_MIN;
  }
  for (int64_t i = tile * ORC_TILE; i < L && i < (tile + 1) * ORC_TILE; ++i) {
    int c = ty[base + i];
    if (c < 0 || c > 3) continue;
    int64_t tt = t[base + i];
    box[c].cnt++;
    if (i < box[c].pmin) box[c].pmin = i;
    if (i > box[c].pmax) box[c].pmax = i;
    if (tt < box[c].tmin) box[c].tmin = tt;
    if (tt > box[c].tmax) box[c].tmax = tt;
  }
}

int64_t orc_tile_classes(const orc_params* p, int32_t B, const int64_t* offsets,
                         const int64_t* t, const int8_t* ty, uint8_t* cls) {
  int64_t n = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t base = offsets[b], L = offsets[b + 1] - base;
    const int64_t nt = (L + ORC_TILE - 1) / ORC_TILE;
    for (int64_t qt = 0; qt < nt; ++qt) {
      orc_box qb[4];
      tile_boxes(base, L, qt, t, ty, qb);
      for (int64_t kt = 0; kt < nt; ++kt) {
        orc_box kb[4];
        tile_boxes(base, L, kt, t, ty, kb);
        int lo = TV_ALL, hi = TV_NONE;
        for (int a = 0; a < 4; ++a) {
          if (!qb[a].cnt) continue;
          for (int c = 0; c < 4; ++c) {
            if (!kb[c].cnt) continue;
            int v = tv_pair(p, a, c, &qb[a], &kb[c]);
            if (v < lo) lo = v;
            if (v > hi) hi = v;
          }
        }
        const int k_full = (kt + 1) * ORC_TILE <= L;
        uint8_t c;
        if (hi == TV_NONE) c = ORC_SKIP;            /* every present type pair sees nothing */
        else if (lo == TV_ALL && k_full) c = ORC_FULL; /* every pair visible, no ragged keys */
        else c = ORC_PARTIAL;
        if (cls) cls[n] = c;
        ++n;
      }
    }
  }
  return n;
}
