/*
 * oracle.c -- the plain, slow, obviously-correct CPU definition of what the
 * GPU path computes.  TEST INFRASTRUCTURE ONLY: nothing in the product
 * library links, includes or calls this file.  Only tests/, the smoke check
 * and the bench's CPU-baseline leg use it.
 *
 * Everything is computed in IEEE double (fp64).  Inputs may be given as
 * fp64, fp32 or bf16 (raw uint16 bit patterns); they are widened exactly to
 * double before any arithmetic.  No blocking, fusion or reordering beyond the
 * plain definitions below: each function names the passage it follows.
 *
 * Sources (web pages on online softmax):
 *   [OS-RM]  "Online Softmax -- the mathematical heart of FlashAttention"
 *            (inference-engineering roadmap page), sections 1-7.
 *   [OS-RH]  "Online Softmax" (research-hub concept page), "Key math".
 *   [OS-PT]  "Online softmax in attention -- why and how".
 *   [OS-IL]  "Online Softmax & FlashAttention -- AI infra interview lesson",
 *            Step 1 (online stats and merge) and Step 2 (FlashAttention V1).
 *
 * Conventions fixed where the pages leave a point open (each is listed in
 * the design notes of the repository):
 *   - a score or input element equal to -inf contributes exactly zero;
 *   - a row whose elements are all -inf (fully masked) has output +0.0 and
 *     log-sum-exp -inf, never NaN ([OS-RM] s.7 "fully-masked rows";
 *     [OS-IL] Step 1, both-sides -inf special case);
 *   - causal visibility: query t1 sees keys t2 = 0..t1 ([OS-PT] "Why this
 *     matters for attention specifically"), positions counted along the
 *     sequence.  With Nq queries and Nk keys the queries are the sequence's
 *     last Nq positions (new tokens after a cache of Nk - Nq keys), so key j
 *     is visible to query i iff j <= i + (Nk - Nq); for Nq == Nk that is
 *     j <= i.  A query with no visible key (Nq > Nk, i < Nq - Nk) has output
 *     +0.0 and log-sum-exp -inf;
 *   - the log-sum-exp is natural-log, over the scaled scores.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC -pthread.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F64 0
#define ORACLE_F32 1
#define ORACLE_BF16 2

/* Exact widening of one element of an input buffer to double. */
static double widen(const void* p, int dtype, int64_t idx) {
  if (dtype == ORACLE_F64) return ((const double*)p)[idx];
  if (dtype == ORACLE_F32) return (double)((const float*)p)[idx];
  /* bf16: the 16 stored bits are the top half of an fp32 bit pattern */
  uint32_t bits = (uint32_t)((const uint16_t*)p)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------------ */
/* Simple static partition of [0, n) over worker threads.              */
/* ------------------------------------------------------------------ */
typedef void (*range_fn)(void* ctx, int64_t begin, int64_t end, double* scratch);

typedef struct {
  range_fn fn;
  void* ctx;
  int64_t begin, end;
  int64_t scratch_len;
  int failed;
} worker_arg;

static void* worker_main(void* p) {
  worker_arg* a = (worker_arg*)p;
  double* scratch = NULL;
  if (a->scratch_len > 0) {
    scratch = (double*)malloc((size_t)a->scratch_len * sizeof(double));
    if (!scratch) {
      a->failed = 1;
      return NULL;
    }
  }
  a->fn(a->ctx, a->begin, a->end, scratch);
  free(scratch);
  return NULL;
}

/* Runs fn over [0, n) split into nthreads contiguous pieces.  Returns 0 on
 * success, -1 if a thread or its scratch could not be created. */
static int parallel_for(int64_t n, int nthreads, int64_t scratch_len, range_fn fn, void* ctx) {
  if (n <= 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n) nthreads = (int)n;
  pthread_t tid[256];
  worker_arg args[256];
  int started[256];
  int rc = 0;
  for (int t = 0; t < nthreads; ++t) {
    args[t].fn = fn;
    args[t].ctx = ctx;
    args[t].begin = n * t / nthreads;
    args[t].end = n * (t + 1) / nthreads;
    args[t].scratch_len = scratch_len;
    args[t].failed = 0;
    started[t] = (pthread_create(&tid[t], NULL, worker_main, &args[t]) == 0);
    if (!started[t]) {
      worker_main(&args[t]); /* run inline rather than fail */
    }
  }
  for (int t = 0; t < nthreads; ++t) {
    if (started[t]) pthread_join(tid[t], NULL);
    if (args[t].failed) rc = -1;
  }
  return rc;
}

/* ------------------------------------------------------------------ */
/* Row softmax with log-sum-exp: the three-pass safe softmax.          */
/* [OS-RM] s.1 "Standard (offline) softmax -- 3 passes";               */
/* [OS-PT] "The textbook softmax: stable, but two passes".             */
/* ------------------------------------------------------------------ */
typedef struct {
  const void* x;
  int dtype;
  int64_t cols, ld_x, ld_y;
  double* y;
  double* lse;
} softmax_ctx;

static void softmax_range(void* p, int64_t r0, int64_t r1, double* scratch) {
  (void)scratch;
  const softmax_ctx* c = (const softmax_ctx*)p;
  for (int64_t r = r0; r < r1; ++r) {
    const int64_t base = r * c->ld_x;
    /* pass 1: m = max_j x_j */
    double m = -INFINITY;
    for (int64_t j = 0; j < c->cols; ++j) {
      double xj = widen(c->x, c->dtype, base + j);
      if (xj > m) m = xj;
    }
    if (m == -INFINITY) { /* fully -inf row: y = 0, lse = -inf */
      if (c->y)
        for (int64_t j = 0; j < c->cols; ++j) c->y[r * c->ld_y + j] = 0.0;
      if (c->lse) c->lse[r] = -INFINITY;
      continue;
    }
    /* pass 2: d = sum_j exp(x_j - m) */
    double d = 0.0;
    for (int64_t j = 0; j < c->cols; ++j) d += exp(widen(c->x, c->dtype, base + j) - m);
    /* pass 3: y_j = exp(x_j - m) / d */
    if (c->y)
      for (int64_t j = 0; j < c->cols; ++j)
        c->y[r * c->ld_y + j] = exp(widen(c->x, c->dtype, base + j) - m) / d;
    if (c->lse) c->lse[r] = m + log(d);
  }
}

/* x: rows x cols, row stride ld_x elements; y: rows x cols (row stride ld_y)
 * or NULL; lse: rows or NULL.  Returns 0, or -1 on a bad argument. */
int oracle_softmax_rows(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld_x,
                        double* y, int64_t ld_y, double* lse, int nthreads) {
  if (!x || rows < 0 || cols < 0 || ld_x < cols || (y && ld_y < cols)) return -1;
  softmax_ctx c = {x, dtype, cols, ld_x, ld_y, y, lse};
  return parallel_for(rows, nthreads, 0, softmax_range, &c);
}

/* ------------------------------------------------------------------ */
/* Attention: materialise one full score row, safe softmax, weighted    */
/* sum of value rows.                                                   */
/* [OS-RM] s.5: A_i = sum_j softmax(Q K^T)_ij V_j;                      */
/* [OS-PT]: s_t2 = (q_t1 . k_t2) / sqrt(hd), causal t2 <= t1 (query i   */
/* at position i + Nk - Nq of the sequence, see the conventions above); */
/* [OS-IL] Step 2: S = q K^T * scale.                                   */
/* Layout: q [B,H,Nq,d], k and v [B,Hkv,Nk,d], row-major contiguous;  */
/* query head h reads key/value head h / (H / Hkv) (grouped heads;      */
/* Hkv == H is one key/value head per query head).                      */
/* ------------------------------------------------------------------ */
typedef struct {
  const void *q, *k, *v;
  int dtype;
  int64_t B, H, Hkv, Nq, Nk, d;
  int causal;
  double scale;
  const int32_t* kv_len;
  const int64_t* rows; /* flattened (b*H + h)*Nq + i, or NULL for all */
  double* o;
  double* lse;
} attn_ctx;

static void attn_range(void* p, int64_t t0, int64_t t1, double* s) {
  const attn_ctx* c = (const attn_ctx*)p;
  const int64_t d = c->d;
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t row = c->rows ? c->rows[t] : t;
    const int64_t bh = row / c->Nq, i = row % c->Nq, b = bh / c->H;
    int64_t kvl = c->Nk;
    if (c->kv_len) {
      kvl = c->kv_len[b];
      if (kvl > c->Nk) kvl = c->Nk;
      if (kvl < 0) kvl = 0;
    }
    const int64_t h = bh % c->H, kvh = b * c->Hkv + h / (c->H / c->Hkv);
    const int64_t qbase = row * d, kvbase = kvh * c->Nk * d;
    const int64_t last = i + (c->Nk - c->Nq); /* causal: last visible key */
    /* full score row, -inf where masked */
    for (int64_t j = 0; j < c->Nk; ++j) {
      int visible = (j < kvl) && (!c->causal || j <= last);
      if (!visible) {
        s[j] = -INFINITY;
        continue;
      }
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e)
        dot += widen(c->q, c->dtype, qbase + e) * widen(c->k, c->dtype, kvbase + j * d + e);
      s[j] = c->scale * dot;
    }
    double* o = c->o ? c->o + t * d : NULL;
    if (o)
      for (int64_t e = 0; e < d; ++e) o[e] = 0.0;
    /* three-pass safe softmax over the row */
    double m = -INFINITY;
    for (int64_t j = 0; j < c->Nk; ++j)
      if (s[j] > m) m = s[j];
    if (m == -INFINITY) {
      if (c->lse) c->lse[t] = -INFINITY;
      continue; /* o stays +0.0 */
    }
    double l = 0.0;
    for (int64_t j = 0; j < c->Nk; ++j) l += exp(s[j] - m);
    if (o)
      for (int64_t j = 0; j < c->Nk; ++j) {
        if (s[j] == -INFINITY) continue; /* weight exactly zero */
        double y = exp(s[j] - m) / l;
        for (int64_t e = 0; e < d; ++e) o[e] += y * widen(c->v, c->dtype, kvbase + j * d + e);
      }
    if (c->lse) c->lse[t] = m + log(l);
  }
}

/* Computes output rows of softmax(Q K^T * scale) V and their log-sum-exp.
 * rows == NULL: all B*H*Nq rows, o is [B*H*Nq, d]; else only the nrows
 * listed flattened rows, o is [nrows, d], lse is [nrows].  kv_len (NULL or
 * int32[B]) hides keys j >= kv_len[b].  Returns 0, or -1 on bad arguments. */
int oracle_attn(const void* q, const void* k, const void* v, int dtype, int64_t B, int64_t H,
                int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int causal, double scale,
                const int32_t* kv_len, const int64_t* rows, int64_t nrows, double* o, double* lse,
                int nthreads) {
  if (!q || !k || !v || B < 0 || H < 0 || Nq < 0 || Nk < 0 || d < 0) return -1;
  if (Hkv < 1 || H % Hkv != 0) return -1;
  attn_ctx c = {q, k, v, dtype, B, H, Hkv, Nq, Nk, d, causal, scale, kv_len, rows, o, lse};
  int64_t n = rows ? nrows : B * H * Nq;
  if (rows)
    for (int64_t t = 0; t < nrows; ++t)
      if (rows[t] < 0 || rows[t] >= B * H * Nq) return -1;
  return parallel_for(n, nthreads, Nk > 0 ? Nk : 1, attn_range, &c);
}

/* ------------------------------------------------------------------ */
/* Attention backward: the gradients of O = softmax(scale Q K^T) V      */
/* (the forward definition above) given dO, for one (b, h) at a time.   */
/* [OS-PT] "Where this is heading: FA2": the backward recomputes the    */
/* scores instead of reading a stored [T, T] attention matrix; here the */
/* definition is written out with P materialised in fp64:               */
/*   P = softmax_row(scale Q K^T) (masked keys 0),  O = P V,            */
/*   dV = P^T dO,   dP = dO V^T,   D_i = sum_e dO_ie O_ie,              */
/*   dS = P o (dP - D 1^T),   dQ = scale dS K,   dK = scale dS^T Q.     */
/* (the softmax Jacobian row i is diag(P_i) - P_i P_i^T, and            */
/*  P_i . dP_i = dO_i . O_i = D_i).  A row with no visible key has      */
/* P = 0 and contributes nothing.  Layout: q, dout [B,H,Nq,d]; k, v     */
/* [B,Hkv,Nk,d] (query head h reads key/value head h / (H / Hkv)); dq   */
/* [B,H,Nq,d], dk and dv [B,Hkv,Nk,d], all fp64 out.  A key/value head  */
/* used by several query heads receives the sum of their dK, dV (each   */
/* use is a separate term of the loss).                                 */
/* ------------------------------------------------------------------ */
typedef struct {
  const void *q, *k, *v, *dout;
  int dtype;
  int64_t H, Hkv, Nq, Nk, d;
  int causal;
  double scale;
  double *dq, *dk, *dv;
} bwd_ctx;

static void bwd_range(void* p, int64_t t0, int64_t t1, double* scratch) {
  const bwd_ctx* c = (const bwd_ctx*)p;
  const int64_t Nq = c->Nq, Nk = c->Nk, d = c->d;
  double* P = scratch;            /* [Nq][Nk] */
  double* dS = P + Nq * Nk;       /* [Nq][Nk] */
  double* O = dS + Nq * Nk;       /* [Nq][d]  */
  const int64_t g = c->H / c->Hkv;
  /* one key/value plane per item; its query heads in turn, summing into its dK, dV */
  for (int64_t kvp = t0; kvp < t1; ++kvp)
  for (int64_t t = 0; t < g; ++t) {
    const int64_t bh = kvp * g + t; /* query plane: (b, h) with h = (kvp % Hkv) g + t */
    const int64_t qb = bh * Nq * d, kb = kvp * Nk * d;
    /* P, row by row (safe softmax of the visible scaled scores) */
    for (int64_t i = 0; i < Nq; ++i) {
      double m = -INFINITY;
      for (int64_t j = 0; j < Nk; ++j) {
        double s = -INFINITY;
        if (!c->causal || j <= i + (Nk - Nq)) {
          double dot = 0.0;
          for (int64_t e = 0; e < d; ++e)
            dot += widen(c->q, c->dtype, qb + i * d + e) * widen(c->k, c->dtype, kb + j * d + e);
          s = c->scale * dot;
        }
        P[i * Nk + j] = s;
        if (s > m) m = s;
      }
      double l = 0.0;
      for (int64_t j = 0; j < Nk; ++j) {
        double w = (m == -INFINITY || P[i * Nk + j] == -INFINITY) ? 0.0 : exp(P[i * Nk + j] - m);
        P[i * Nk + j] = w;
        l += w;
      }
      for (int64_t j = 0; j < Nk; ++j) P[i * Nk + j] = (l > 0.0) ? P[i * Nk + j] / l : 0.0;
    }
    /* O = P V; dS = P o (dO V^T - D) */
    for (int64_t i = 0; i < Nq; ++i) {
      for (int64_t e = 0; e < d; ++e) {
        double acc = 0.0;
        for (int64_t j = 0; j < Nk; ++j) acc += P[i * Nk + j] * widen(c->v, c->dtype, kb + j * d + e);
        O[i * d + e] = acc;
      }
      double D = 0.0;
      for (int64_t e = 0; e < d; ++e) D += widen(c->dout, c->dtype, qb + i * d + e) * O[i * d + e];
      for (int64_t j = 0; j < Nk; ++j) {
        double dp = 0.0;
        for (int64_t e = 0; e < d; ++e)
          dp += widen(c->dout, c->dtype, qb + i * d + e) * widen(c->v, c->dtype, kb + j * d + e);
        dS[i * Nk + j] = P[i * Nk + j] * (dp - D);
      }
    }
    /* dQ = scale dS K */
    for (int64_t i = 0; i < Nq; ++i)
      for (int64_t e = 0; e < d; ++e) {
        double acc = 0.0;
        for (int64_t j = 0; j < Nk; ++j) acc += dS[i * Nk + j] * widen(c->k, c->dtype, kb + j * d + e);
        c->dq[qb + i * d + e] = c->scale * acc;
      }
    /* dK = scale dS^T Q,  dV = P^T dO */
    for (int64_t j = 0; j < Nk; ++j)
      for (int64_t e = 0; e < d; ++e) {
        double ak = 0.0, av = 0.0;
        for (int64_t i = 0; i < Nq; ++i) {
          ak += dS[i * Nk + j] * widen(c->q, c->dtype, qb + i * d + e);
          av += P[i * Nk + j] * widen(c->dout, c->dtype, qb + i * d + e);
        }
        if (t == 0) {
          c->dk[kb + j * d + e] = 0.0;
          c->dv[kb + j * d + e] = 0.0;
        }
        c->dk[kb + j * d + e] += c->scale * ak;
        c->dv[kb + j * d + e] += av;
      }
  }
}

/* Gradients of attention for B*H independent heads (see above).  Returns 0,
 * or -1 on bad arguments. */
int oracle_attn_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype, int64_t B,
                    int64_t H, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int causal, double scale, double* dq,
                    double* dk, double* dv, int nthreads) {
  if (!q || !k || !v || !dout || !dq || !dk || !dv || B < 0 || H < 0 || Nq < 0 || Nk < 0 || d < 0) return -1;
  if (Hkv < 1 || H % Hkv != 0) return -1;
  bwd_ctx c = {q, k, v, dout, dtype, H, Hkv, Nq, Nk, d, causal, scale, dq, dk, dv};
  const int64_t scratch = 2 * Nq * Nk + Nq * d + 1;
  return parallel_for(B * Hkv, nthreads, scratch, bwd_range, &c);
}

/* ------------------------------------------------------------------ */
/* The same gradients for one head at chosen rows only: dQ at query     */
/* rows qi[], dK and dV at key rows kj[] (so that a large problem can   */
/* be checked without the [Nq, Nk] matrices).  The formulas are those   */
/* of oracle_attn_bwd; P_ij = exp(s_ij - m_i) / l_i from each query     */
/* row's max m_i and sum l_i, which phase A takes over all query rows   */
/* together with O_i and D_i = dO_i . O_i.                              */
/* ------------------------------------------------------------------ */
typedef struct {
  const void *q, *k, *v, *dout;
  int dtype;
  int64_t Nq, Nk, d;
  int causal;
  double scale;
  double *m, *l, *D;
  const int64_t *qi, *kj;
  double *dq, *dk, *dv;
} bwds_ctx;

static double bwds_score(const bwds_ctx* c, int64_t i, int64_t j) {
  if (c->causal && j > i + (c->Nk - c->Nq)) return -INFINITY;
  double dot = 0.0;
  for (int64_t e = 0; e < c->d; ++e) dot += widen(c->q, c->dtype, i * c->d + e) * widen(c->k, c->dtype, j * c->d + e);
  return c->scale * dot;
}

static double bwds_prob(const bwds_ctx* c, int64_t i, int64_t j) {
  double s = bwds_score(c, i, j);
  if (s == -INFINITY || c->l[i] == 0.0) return 0.0;
  return exp(s - c->m[i]) / c->l[i];
}

static double bwds_dp(const bwds_ctx* c, int64_t i, int64_t j) {
  double dp = 0.0;
  for (int64_t e = 0; e < c->d; ++e)
    dp += widen(c->dout, c->dtype, i * c->d + e) * widen(c->v, c->dtype, j * c->d + e);
  return dp;
}

/* phase A: m_i, l_i, O_i (scratch) and D_i for query rows [t0, t1) */
static void bwds_rows(void* p, int64_t t0, int64_t t1, double* scratch) {
  const bwds_ctx* c = (const bwds_ctx*)p;
  double* S = scratch;        /* [Nk] */
  double* O = scratch + c->Nk; /* [d] */
  for (int64_t i = t0; i < t1; ++i) {
    double m = -INFINITY;
    for (int64_t j = 0; j < c->Nk; ++j) {
      S[j] = bwds_score(c, i, j);
      if (S[j] > m) m = S[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < c->Nk; ++j) {
      S[j] = (m == -INFINITY || S[j] == -INFINITY) ? 0.0 : exp(S[j] - m);
      l += S[j];
    }
    double D = 0.0;
    for (int64_t e = 0; e < c->d; ++e) {
      double acc = 0.0;
      for (int64_t j = 0; j < c->Nk; ++j) acc += S[j] * widen(c->v, c->dtype, j * c->d + e);
      O[e] = l > 0.0 ? acc / l : 0.0;
      D += widen(c->dout, c->dtype, i * c->d + e) * O[e];
    }
    c->m[i] = m;
    c->l[i] = l;
    c->D[i] = D;
  }
}

/* phase B: dQ_i = scale sum_j dS_ij K_j at sampled query rows [t0, t1) */
static void bwds_dq(void* p, int64_t t0, int64_t t1, double* scratch) {
  const bwds_ctx* c = (const bwds_ctx*)p;
  double* dS = scratch; /* [Nk] */
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t i = c->qi[t];
    for (int64_t j = 0; j < c->Nk; ++j) {
      double P = bwds_prob(c, i, j);
      dS[j] = P == 0.0 ? 0.0 : P * (bwds_dp(c, i, j) - c->D[i]);
    }
    for (int64_t e = 0; e < c->d; ++e) {
      double acc = 0.0;
      for (int64_t j = 0; j < c->Nk; ++j) acc += dS[j] * widen(c->k, c->dtype, j * c->d + e);
      c->dq[t * c->d + e] = c->scale * acc;
    }
  }
}

/* phase C: dV_j = sum_i P_ij dO_i and dK_j = scale sum_i dS_ij Q_i at sampled key rows [t0, t1) */
static void bwds_dkv(void* p, int64_t t0, int64_t t1, double* scratch) {
  const bwds_ctx* c = (const bwds_ctx*)p;
  (void)scratch;
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t j = c->kj[t];
    for (int64_t e = 0; e < c->d; ++e) {
      c->dk[t * c->d + e] = 0.0;
      c->dv[t * c->d + e] = 0.0;
    }
    for (int64_t i = 0; i < c->Nq; ++i) {
      double P = bwds_prob(c, i, j);
      if (P == 0.0) continue;
      double dS = P * (bwds_dp(c, i, j) - c->D[i]);
      for (int64_t e = 0; e < c->d; ++e) {
        c->dk[t * c->d + e] += c->scale * dS * widen(c->q, c->dtype, i * c->d + e);
        c->dv[t * c->d + e] += P * widen(c->dout, c->dtype, i * c->d + e);
      }
    }
  }
}

/* One head: q, dout [Nq, d], k, v [Nk, d]; dq [nq, d] at rows qi, dk and
 * dv [nk, d] at rows kj.  Returns 0, or -1 on bad arguments. */
int oracle_attn_bwd_sampled(const void* q, const void* k, const void* v, const void* dout, int dtype, int64_t Nq,
                            int64_t Nk, int64_t d, int causal, double scale, const int64_t* qi, int64_t nq,
                            const int64_t* kj, int64_t nk, double* dq, double* dk, double* dv, int nthreads) {
  if (!q || !k || !v || !dout || Nq < 0 || Nk < 0 || d < 0 || nq < 0 || nk < 0) return -1;
  if ((nq > 0 && (!qi || !dq)) || (nk > 0 && (!kj || !dk || !dv))) return -1;
  for (int64_t t = 0; t < nq; ++t)
    if (qi[t] < 0 || qi[t] >= Nq) return -1;
  for (int64_t t = 0; t < nk; ++t)
    if (kj[t] < 0 || kj[t] >= Nk) return -1;
  double* stats = (double*)malloc(sizeof(double) * (size_t)(3 * Nq + 1));
  if (!stats) return -1;
  bwds_ctx c = {q, k, v, dout, dtype, Nq, Nk, d, causal, scale, stats, stats + Nq, stats + 2 * Nq, qi, kj, dq, dk, dv};
  int rc = parallel_for(Nq, nthreads, Nk + d + 1, bwds_rows, &c);
  if (rc == 0) rc = parallel_for(nq, nthreads, Nk + 1, bwds_dq, &c);
  if (rc == 0) rc = parallel_for(nk, nthreads, 1, bwds_dkv, &c);
  free(stats);
  return rc;
}

/* ------------------------------------------------------------------ */
/* Merge of split partials: each partial c of row r holds the output   */
/* normalised over its own keys, o_c, and its log-sum-exp lse_c.  The   */
/* merged row is the softmax over the union of the keys:                */
/*   lse = log sum_c exp(lse_c),  o = sum_c exp(lse_c - lse) o_c.       */
/* A partial with lse_c = -inf (no visible key) has weight zero; if all */
/* are -inf, o = 0 and lse = -inf.                                      */
/* [OS-IL] Step 1 (merge of (m, l), direct logsumexp) and Step 2        */
/* (O_new = (l_old e^(m_old-m_new) O_old + ...)/l_new).                 */
/* part_o [S, R, d] (may be NULL when d == 0), part_lse [S, R].         */
/* ------------------------------------------------------------------ */
int oracle_lse_merge(const double* part_o, const double* part_lse, int64_t S, int64_t R,
                     int64_t d, double* o, double* lse) {
  if (!part_lse || S < 0 || R < 0 || d < 0 || (d > 0 && (!part_o || !o))) return -1;
  for (int64_t r = 0; r < R; ++r) {
    double L = -INFINITY;
    for (int64_t c = 0; c < S; ++c)
      if (part_lse[c * R + r] > L) L = part_lse[c * R + r];
    for (int64_t e = 0; e < d; ++e) o[r * d + e] = 0.0;
    if (L == -INFINITY) {
      if (lse) lse[r] = -INFINITY;
      continue;
    }
    double W = 0.0;
    for (int64_t c = 0; c < S; ++c) W += exp(part_lse[c * R + r] - L);
    double total = L + log(W);
    for (int64_t c = 0; c < S; ++c) {
      double lc = part_lse[c * R + r];
      if (lc == -INFINITY) continue;
      double w = exp(lc - total);
      for (int64_t e = 0; e < d; ++e) o[r * d + e] += w * part_o[(c * R + r) * d + e];
    }
    if (lse) lse[r] = total;
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* The algorithmic forms, kept only so the tests can show that they     */
/* reach the definitions above.  They follow the pages' steps in order.  */
/* ------------------------------------------------------------------ */

/* Single pass over x: running max m and running sum l, referred to m.
 * [OS-RM] s.2 recurrence; [OS-IL] Step 1 "a single-pass scan merges in
 * each element as (x_i, 1)", skipping elements while nothing finite has
 * been seen (avoids -inf - -inf). */
void oracle_online_stats(const double* x, int64_t n, double* m_out, double* l_out) {
  double m = -INFINITY, l = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double m_new = x[i] > m ? x[i] : m;
    if (m_new == -INFINITY) continue;
    l = l * exp(m - m_new) + exp(x[i] - m_new);
    m = m_new;
  }
  *m_out = m;
  *l_out = l;
}

/* Online stats that also records (m_k, d_k) after every element, for the
 * step-by-step worked example ([OS-RM] s.3).  m_steps and l_steps hold n. */
void oracle_online_stats_trace(const double* x, int64_t n, double* m_steps, double* l_steps) {
  double m = -INFINITY, l = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double m_new = x[i] > m ? x[i] : m;
    if (m_new != -INFINITY) {
      l = l * exp(m - m_new) + exp(x[i] - m_new);
      m = m_new;
    }
    m_steps[i] = m;
    l_steps[i] = l;
  }
}

/* Merge of two segment statistics ([OS-IL] Step 1):
 *   m = max(m1, m2),  l = exp(m1 - m) l1 + exp(m2 - m) l2,
 * with 0 used as the reference when both sides are -inf. */
void oracle_merge_ml(double m1, double l1, double m2, double l2, double* m_out, double* l_out) {
  double m = m1 > m2 ? m1 : m2;
  double safe = (m == -INFINITY) ? 0.0 : m;
  *m_out = m;
  *l_out = l1 * exp(m1 - safe) + l2 * exp(m2 - safe);
}

/* FlashAttention V1 for one head, non-causal ([OS-IL] Step 2): KV blocks
 * of Bc rows outside, Q blocks of Br rows inside; O, m, l kept normalised
 * and merged per block.  q [N,d], k and v [Nk,d] fp64; o [N,d].  Needs
 * scratch for O/m/l only.  Returns 0, or -1 on bad arguments. */
int oracle_attn_fa1(const double* q, const double* k, const double* v, int64_t N, int64_t Nk,
                    int64_t d, int64_t Br, int64_t Bc, double scale, double* o) {
  if (!q || !k || !v || !o || N < 0 || Nk < 0 || d < 0 || Br < 1 || Bc < 1) return -1;
  double* m = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
  double* l = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
  double* S = (double*)malloc((size_t)(Br * Bc) * sizeof(double));
  double* PV = (double*)malloc((size_t)(d > 0 ? d : 1) * sizeof(double));
  if (!m || !l || !S || !PV) {
    free(m), free(l), free(S), free(PV);
    return -1;
  }
  for (int64_t i = 0; i < N; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.0;
    for (int64_t e = 0; e < d; ++e) o[i * d + e] = 0.0;
  }
  for (int64_t j0 = 0; j0 < Nk; j0 += Bc) {
    int64_t bc = (Nk - j0 < Bc) ? Nk - j0 : Bc;
    for (int64_t i0 = 0; i0 < N; i0 += Br) {
      int64_t br = (N - i0 < Br) ? N - i0 : Br;
      for (int64_t a = 0; a < br; ++a) {
        const int64_t i = i0 + a;
        /* S = q K^T * scale for this block row, and its block-local max */
        double m_ij = -INFINITY;
        for (int64_t b = 0; b < bc; ++b) {
          double dot = 0.0;
          for (int64_t e = 0; e < d; ++e) dot += q[i * d + e] * k[(j0 + b) * d + e];
          S[a * Bc + b] = dot * scale;
          if (S[a * Bc + b] > m_ij) m_ij = S[a * Bc + b];
        }
        /* P = exp(S - m_ij), l_ij = sum P, PV = P V_j */
        double l_ij = 0.0;
        for (int64_t e = 0; e < d; ++e) PV[e] = 0.0;
        for (int64_t b = 0; b < bc; ++b) {
          double p = exp(S[a * Bc + b] - m_ij);
          l_ij += p;
          for (int64_t e = 0; e < d; ++e) PV[e] += p * v[(j0 + b) * d + e];
        }
        double m_new, l_new;
        oracle_merge_ml(m[i], l[i], m_ij, l_ij, &m_new, &l_new);
        double w_old = l[i] * exp(m[i] - m_new); /* 0 on the first block */
        double w_new = exp(m_ij - m_new);
        for (int64_t e = 0; e < d; ++e) o[i * d + e] = (w_old * o[i * d + e] + w_new * PV[e]) / l_new;
        m[i] = m_new;
        l[i] = l_new;
      }
    }
  }
  free(m), free(l), free(S), free(PV);
  return 0;
}
