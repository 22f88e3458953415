/*
 * fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the attention path computes.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark load it; the product
 * library never does, and the two share no code, headers or tables.
 *
 * What it follows (FlashAttention: Fast and Memory-Efficient Exact Attention
 * with IO-Awareness, hackmd summary, "Standard Attention Implementation"):
 *   S = Q K^T,  P = softmax(S) taken row by row,  O = P V,
 * with Q, K, V in R^{N x d} per (batch, head).  The score scale and the masks
 * are the plainest reading of the text, which names masking only:
 *   s_ij = scale * <q_i, k_j>                    if (i, j) is allowed
 *        = -inf                                  otherwise
 *   allowed(i, j) = (!causal || j <= i) && (!mask || mask[i/T][j/T] != 0)
 * (T = tile edge of the block mask; "Block-sparse FlashAttention" in the same
 * summary, section "Introduction").  The stored statistic is the natural-log
 * logsumexp lse_i = m_i + ln(sum_j exp(s_ij - m_i)), which carries the two
 * running statistics m and l that the "Recomputation" section says are kept
 * for the backward pass.
 *
 * Gradients: the pages only state that the backward recomputes S and P from
 * the stored statistics ("Recomputation").  The oracle writes out the chain
 * rule of the definition above:
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,
 *   dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
 *
 * A row with no allowed key has O_i = 0, lse_i = -inf and contributes nothing
 * to any gradient (reading taken where the pages are silent).
 *
 * Grouped key/value heads (the multi-head-attention variants the summary's
 * "Future Directions" section lists): with Hkv key/value heads and H query
 * heads, query head h reads key/value head h / (H / Hkv).  A shared key or
 * value row gets the sum of the gradients of every query head that reads it
 * (chain rule over the shared parameter).  Hkv = H is ordinary attention.
 *
 * Dropout on P (the summary fuses dropout into the kernel, "Kernel Fusion",
 * and benchmarks with it, section 4.4; it names no generator and no
 * scaling).  Reading taken: inverted dropout of the attention weights,
 *   P~_ij = z_ij * P_ij / (1 - p'),   O = P~ V,
 * with lse still the statistic of the undropped row.  The keep indicator
 * z_ij comes from a counter-based generator, Philox4x32-10 (Salmon, Moraes,
 * Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
 *   counter = (j / 16, i, b * H + h, offset),  key = (seed mod 2^32, seed / 2^32)
 *   byte    = byte (j mod 4) of output word ((j / 4) mod 4), little-endian
 *   z_ij    = byte >= t,   t = rint(256 * p) with p taken in float32
 * so the effective drop probability is p' = t / 256 and kept weights are
 * scaled by 1 / (1 - p') = 256 / (256 - t).  i and j are row indices within
 * the sequence and b the batch (sequence) index.  The chain rule then gives
 *   dV = P~^T dO,  dP_ij = z_ij <dO_i, v_j> / (1 - p'),
 *   D_i = sum_j P_ij dP_ij,  dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
 *
 * Every loop is a straight restatement of a sum in the definition, in fp64,
 * summed in index order.  Work is split over independent (head, row-block)
 * units with POSIX threads; that changes nothing in any sum.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  const double *q, *k, *v, *dO; /* q, dO: [B,H,N,d];  k, v: [B,Hkv,N,d] */
  long B, H, N, d;
  double scale;
  int causal;
  const unsigned char *mask; /* [mask_heads, nT, nT] or NULL */
  long mask_heads, tile, nT;
  long Hkv;
  /* dropout: t = 0 means none */
  unsigned t;
  double keep_scale; /* 256 / (256 - t) */
  uint64_t seed;
  uint32_t offset;
  long batch0; /* batch index of b = 0 in the dropout counter */
} problem_t;

/* ---------------------------------------------------------------------- */
/* Philox4x32-10: ten rounds of the Philox S-box on a 128-bit counter; round
 * r uses the key plus r times the Weyl increments.                        */
static void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint64_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    uint64_t p0 = M0 * (uint64_t)c0; /* hi:lo of M0 * c0 */
    uint64_t p1 = M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += W0;
    k1 += W1;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* random byte of element (bhc, i, j) of the dropout stream */
static unsigned keep_byte(uint64_t seed, uint32_t offset, uint64_t bhc, uint64_t i, uint64_t j) {
  uint32_t ctr[4] = {(uint32_t)(j >> 4), (uint32_t)i, (uint32_t)bhc, offset};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t r[4];
  philox4x32_10(ctr, key, r);
  return (r[(j >> 2) & 3] >> (8 * (j & 3))) & 0xFFu;
}

/* dropout factor z_ij / (1 - p') of query slice bh, or 1 without dropout */
static double drop_factor(const problem_t *p, long bh, long i, long j) {
  if (p->t == 0) return 1.0;
  long b = bh / p->H, h = bh % p->H;
  uint64_t bhc = (uint64_t)((p->batch0 + b) * p->H + h);
  return keep_byte(p->seed, p->offset, bhc, (uint64_t)i, (uint64_t)j) >= p->t ? p->keep_scale
                                                                               : 0.0;
}

/* (batch, key/value head) slice that query slice bh reads */
static long kv_slice(const problem_t *p, long bh) {
  long b = bh / p->H, h = bh % p->H;
  return b * p->Hkv + h / (p->H / p->Hkv);
}

static int allowed(const problem_t *p, long h, long i, long j) {
  if (j < 0 || j >= p->N || i < 0 || i >= p->N) return 0;
  if (p->causal && j > i) return 0;
  if (p->mask) {
    long hm = (p->mask_heads == 1) ? 0 : h;
    unsigned char m = p->mask[(hm * p->nT + i / p->tile) * p->nT + j / p->tile];
    if (m == 0) return 0;
  }
  return 1;
}

static double dot(const double *a, const double *b, long d) {
  double s = 0.0;
  for (long c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

/* ---------------------------------------------------------------------- */
/* a tiny thread pool: parallel-for over independent units                 */
typedef void (*unit_fn)(void *ctx, long unit);
typedef struct {
  unit_fn fn;
  void *ctx;
  long n;
  atomic_long next;
} pool_t;

static void *pool_worker(void *arg) {
  pool_t *pl = (pool_t *)arg;
  for (;;) {
    long u = atomic_fetch_add(&pl->next, 1);
    if (u >= pl->n) break;
    pl->fn(pl->ctx, u);
  }
  return NULL;
}

static void parallel_for(long n, unit_fn fn, void *ctx, int nthreads) {
  pool_t pl;
  pl.fn = fn;
  pl.ctx = ctx;
  pl.n = n;
  atomic_init(&pl.next, 0);
  if (nthreads <= 1 || n <= 1) {
    pool_worker(&pl);
    return;
  }
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, pool_worker, &pl) != 0) break;
    ++started;
  }
  if (started == 0) pool_worker(&pl);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------------- */
/* Row statistics and output of one query row: the definition, written out. */
/* Returns lse_i; fills o_row (d values) when it is not NULL.                */
static double row_forward(const problem_t *p, long bh, long i, double *o_row) {
  long h = bh % p->H;
  const double *qi = p->q + (bh * p->N + i) * p->d;
  const double *K = p->k + kv_slice(p, bh) * p->N * p->d;
  const double *V = p->v + kv_slice(p, bh) * p->N * p->d;
  /* m_i = max over allowed j of s_ij */
  double m = -INFINITY;
  long cnt = 0;
  for (long j = 0; j < p->N; ++j) {
    if (!allowed(p, h, i, j)) continue;
    double s = p->scale * dot(qi, K + j * p->d, p->d);
    if (s > m) m = s;
    ++cnt;
  }
  if (o_row) memset(o_row, 0, sizeof(double) * p->d);
  if (cnt == 0) return -INFINITY;
  /* l_i = sum_j exp(s_ij - m_i);  lse_i = m_i + ln l_i */
  double l = 0.0;
  for (long j = 0; j < p->N; ++j) {
    if (!allowed(p, h, i, j)) continue;
    double s = p->scale * dot(qi, K + j * p->d, p->d);
    l += exp(s - m);
  }
  double lse = m + log(l);
  /* O_i = sum_j P_ij v_j with P_ij = exp(s_ij - lse_i) */
  if (o_row) {
    for (long j = 0; j < p->N; ++j) {
      if (!allowed(p, h, i, j)) continue;
      double s = p->scale * dot(qi, K + j * p->d, p->d);
      double pij = exp(s - lse) * drop_factor(p, bh, i, j);
      const double *vj = V + j * p->d;
      for (long c = 0; c < p->d; ++c) o_row[c] += pij * vj[c];
    }
  }
  return lse;
}

/* D_i = sum_j P_ij dP_ij with dP_ij = z_ij <dO_i, v_j> / (1 - p'). */
static double row_delta(const problem_t *p, long bh, long i, double lse) {
  if (lse == -INFINITY) return 0.0;
  long h = bh % p->H;
  const double *qi = p->q + (bh * p->N + i) * p->d;
  const double *doi = p->dO + (bh * p->N + i) * p->d;
  const double *K = p->k + kv_slice(p, bh) * p->N * p->d;
  const double *V = p->v + kv_slice(p, bh) * p->N * p->d;
  double D = 0.0;
  for (long j = 0; j < p->N; ++j) {
    if (!allowed(p, h, i, j)) continue;
    double pij = exp(p->scale * dot(qi, K + j * p->d, p->d) - lse);
    D += pij * drop_factor(p, bh, i, j) * dot(doi, V + j * p->d, p->d);
  }
  return D;
}

/* ---------------------------------------------------------------------- */
/* forward                                                                 */
typedef struct {
  const problem_t *p;
  const long *rows; /* NULL: all rows */
  long nrows, rows_per_unit, units_per_head;
  double *o, *lse;
} fwd_ctx_t;

static void fwd_unit(void *vctx, long unit) {
  fwd_ctx_t *c = (fwd_ctx_t *)vctx;
  const problem_t *p = c->p;
  long bh = unit / c->units_per_head;
  long r0 = (unit % c->units_per_head) * c->rows_per_unit;
  long r1 = r0 + c->rows_per_unit;
  if (r1 > c->nrows) r1 = c->nrows;
  for (long r = r0; r < r1; ++r) {
    long i = c->rows ? c->rows[r] : r;
    double *orow = c->o ? c->o + (bh * c->nrows + r) * p->d : NULL;
    double lse = row_forward(p, bh, i, orow);
    if (c->lse) c->lse[bh * c->nrows + r] = lse;
  }
}

/* t = rint(256 p) for p in [0, 1); t = 256 (everything dropped) is refused */
static int set_dropout(problem_t *p, float p_drop) {
  if (!(p_drop >= 0.0f && p_drop < 1.0f)) return 1;
  double t = nearbyint(256.0 * (double)p_drop);
  if (t >= 256.0) return 1;
  p->t = (unsigned)t;
  p->keep_scale = 256.0 / (256.0 - t);
  return 0;
}

static int check_problem(const problem_t *p) {
  if (p->B < 1 || p->H < 1 || p->N < 1 || p->d < 1) return 1;
  if (p->Hkv < 1 || p->H % p->Hkv != 0) return 1;
  if (!isfinite(p->scale)) return 1;
  if (p->mask && (p->tile < 1 || (p->mask_heads != 1 && p->mask_heads != p->H))) return 1;
  return 0;
}

/* Forward over all rows (rows == NULL, nrows ignored) or the listed rows of
 * every head.  o: [B,H,nrows,d], lse: [B,H,nrows]. */
int fao_forward(const double *q, const double *k, const double *v, long B, long H, long Hkv,
                long N, long d, double scale, int causal, const unsigned char *mask,
                long mask_heads, long tile, const long *rows, long nrows, double *o, double *lse,
                float p_drop, uint64_t seed, uint32_t offset, long batch0, int nthreads) {
  problem_t p = {q, k, v, NULL, B, H, N, d, scale, causal, mask, mask_heads, tile, 0, Hkv,
                 0, 1.0, seed, offset, batch0};
  if (mask) p.nT = (N + tile - 1) / tile;
  if (set_dropout(&p, p_drop)) return 1;
  if (check_problem(&p)) return 1;
  if (!rows) nrows = N;
  for (long r = 0; rows && r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return 1;
  fwd_ctx_t c = {&p, rows, nrows, 64, 0, o, lse};
  c.units_per_head = (nrows + c.rows_per_unit - 1) / c.rows_per_unit;
  if (c.units_per_head == 0) return 0;
  parallel_for(B * H * c.units_per_head, fwd_unit, &c, nthreads);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* backward                                                                */
typedef struct {
  const problem_t *p;
  const unsigned char *need; /* [B*H*N] rows whose lse and D are needed */
  double *lse_all, *D_all;   /* [B*H*N] */
  const long *qrows, *krows;
  long nq, nk, rows_per_unit, upH_stats, upH_q, upH_k;
  double *dq, *dk, *dv;
} bwd_ctx_t;

static void bwd_stats_unit(void *vctx, long unit) {
  bwd_ctx_t *c = (bwd_ctx_t *)vctx;
  const problem_t *p = c->p;
  long bh = unit / c->upH_stats;
  long i0 = (unit % c->upH_stats) * c->rows_per_unit;
  long i1 = i0 + c->rows_per_unit;
  if (i1 > p->N) i1 = p->N;
  for (long i = i0; i < i1; ++i) {
    if (!c->need[bh * p->N + i]) continue;
    double lse = row_forward(p, bh, i, NULL);
    c->lse_all[bh * p->N + i] = lse;
    c->D_all[bh * p->N + i] = row_delta(p, bh, i, lse);
  }
}

/* dQ_i = scale * sum_j dS_ij k_j,  dS_ij = P_ij (dP_ij - D_i) */
static void bwd_dq_unit(void *vctx, long unit) {
  bwd_ctx_t *c = (bwd_ctx_t *)vctx;
  const problem_t *p = c->p;
  long bh = unit / c->upH_q, h = bh % p->H;
  long r0 = (unit % c->upH_q) * c->rows_per_unit;
  long r1 = r0 + c->rows_per_unit;
  if (r1 > c->nq) r1 = c->nq;
  const double *K = p->k + kv_slice(p, bh) * p->N * p->d;
  const double *V = p->v + kv_slice(p, bh) * p->N * p->d;
  for (long r = r0; r < r1; ++r) {
    long i = c->qrows ? c->qrows[r] : r;
    double *dqi = c->dq + (bh * c->nq + r) * p->d;
    memset(dqi, 0, sizeof(double) * p->d);
    double lse = c->lse_all[bh * p->N + i], D = c->D_all[bh * p->N + i];
    if (lse == -INFINITY) continue;
    const double *qi = p->q + (bh * p->N + i) * p->d;
    const double *doi = p->dO + (bh * p->N + i) * p->d;
    for (long j = 0; j < p->N; ++j) {
      if (!allowed(p, h, i, j)) continue;
      double pij = exp(p->scale * dot(qi, K + j * p->d, p->d) - lse);
      double dpij = drop_factor(p, bh, i, j) * dot(doi, V + j * p->d, p->d);
      double dsij = pij * (dpij - D);
      for (long cc = 0; cc < p->d; ++cc) dqi[cc] += p->scale * dsij * K[j * p->d + cc];
    }
  }
}

/* dK_j = scale * sum_i dS_ij q_i,  dV_j = sum_i P~_ij dO_i, summed over every
 * query head that reads key/value head j belongs to */
static void bwd_dkdv_unit(void *vctx, long unit) {
  bwd_ctx_t *c = (bwd_ctx_t *)vctx;
  const problem_t *p = c->p;
  long bkv = unit / c->upH_k;             /* b * Hkv + kv head */
  long b = bkv / p->Hkv, kvh = bkv % p->Hkv, G = p->H / p->Hkv;
  long r0 = (unit % c->upH_k) * c->rows_per_unit;
  long r1 = r0 + c->rows_per_unit;
  if (r1 > c->nk) r1 = c->nk;
  for (long r = r0; r < r1; ++r) {
    long j = c->krows ? c->krows[r] : r;
    double *dkj = c->dk + (bkv * c->nk + r) * p->d;
    double *dvj = c->dv + (bkv * c->nk + r) * p->d;
    memset(dkj, 0, sizeof(double) * p->d);
    memset(dvj, 0, sizeof(double) * p->d);
    const double *kj = p->k + (bkv * p->N + j) * p->d;
    const double *vj = p->v + (bkv * p->N + j) * p->d;
    for (long g = 0; g < G; ++g) {
      long h = kvh * G + g, bh = b * p->H + h;
      const double *Q = p->q + bh * p->N * p->d;
      const double *dO = p->dO + bh * p->N * p->d;
      for (long i = 0; i < p->N; ++i) {
        if (!allowed(p, h, i, j)) continue;
        double lse = c->lse_all[bh * p->N + i], D = c->D_all[bh * p->N + i];
        double pij = exp(p->scale * dot(Q + i * p->d, kj, p->d) - lse);
        double zf = drop_factor(p, bh, i, j);
        double dpij = zf * dot(dO + i * p->d, vj, p->d);
        double dsij = pij * (dpij - D);
        for (long cc = 0; cc < p->d; ++cc) {
          dkj[cc] += p->scale * dsij * Q[i * p->d + cc];
          dvj[cc] += pij * zf * dO[i * p->d + cc];
        }
      }
    }
  }
}

/* Backward for the listed query rows (dq: [B,H,nq,d]) and key rows
 * (dk, dv: [B,Hkv,nk,d]); a NULL row list means every row (nq / nk ignored).
 * Only the rows whose statistics a requested gradient needs are evaluated. */
int fao_backward(const double *q, const double *k, const double *v, const double *dO, long B,
                 long H, long Hkv, long N, long d, double scale, int causal,
                 const unsigned char *mask, long mask_heads, long tile, const long *qrows, long nq,
                 const long *krows, long nk, double *dq, double *dk, double *dv, float p_drop,
                 uint64_t seed, uint32_t offset, long batch0, int nthreads) {
  problem_t p = {q, k, v, dO, B, H, N, d, scale, causal, mask, mask_heads, tile, 0, Hkv,
                 0, 1.0, seed, offset, batch0};
  if (mask) p.nT = (N + tile - 1) / tile;
  if (set_dropout(&p, p_drop)) return 1;
  if (check_problem(&p)) return 1;
  if (!qrows) nq = N;
  if (!krows) nk = N;
  for (long r = 0; qrows && r < nq; ++r)
    if (qrows[r] < 0 || qrows[r] >= N) return 1;
  for (long r = 0; krows && r < nk; ++r)
    if (krows[r] < 0 || krows[r] >= N) return 1;
  long BHN = B * H * N;
  unsigned char *need = (unsigned char *)calloc((size_t)BHN, 1);
  double *lse_all = (double *)calloc((size_t)BHN, sizeof(double));
  double *D_all = (double *)calloc((size_t)BHN, sizeof(double));
  if (!need || !lse_all || !D_all) {
    free(need); free(lse_all); free(D_all);
    return 2;
  }
  /* rows needed: every requested query row, and every query row that can
   * reach a requested key row */
  for (long bh = 0; bh < B * H; ++bh) {
    long h = bh % H;
    for (long r = 0; r < nq; ++r) need[bh * N + (qrows ? qrows[r] : r)] = 1;
    for (long r = 0; r < nk; ++r) {
      long j = krows ? krows[r] : r;
      for (long i = 0; i < N; ++i)
        if (!need[bh * N + i] && allowed(&p, h, i, j)) need[bh * N + i] = 1;
    }
  }
  bwd_ctx_t c;
  memset(&c, 0, sizeof(c));
  c.p = &p;
  c.need = need;
  c.lse_all = lse_all;
  c.D_all = D_all;
  c.qrows = qrows;
  c.krows = krows;
  c.nq = nq;
  c.nk = nk;
  c.rows_per_unit = 32;
  c.upH_stats = (N + c.rows_per_unit - 1) / c.rows_per_unit;
  c.upH_q = (nq + c.rows_per_unit - 1) / c.rows_per_unit;
  c.upH_k = (nk + c.rows_per_unit - 1) / c.rows_per_unit;
  c.dq = dq;
  c.dk = dk;
  c.dv = dv;
  parallel_for(B * H * c.upH_stats, bwd_stats_unit, &c, nthreads);
  if (dq && c.upH_q) parallel_for(B * H * c.upH_q, bwd_dq_unit, &c, nthreads);
  if (dk && dv && c.upH_k) parallel_for(B * Hkv * c.upH_k, bwd_dkdv_unit, &c, nthreads);
  free(need);
  free(lse_all);
  free(D_all);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* integer work: block mask -> tile lists, and tile counts                 */

/* CSR by query tile (ascending key tiles) and CSC by key tile (ascending
 * query tiles) of a [mask_heads, nT, nT] block mask, nonzero = keep.
 * row_ptr: [mask_heads, nT+1] (offsets local to the head), col_idx:
 * [mask_heads, nT*nT] (entries of head h start at h*nT*nT); same for CSC. */
int fao_mask_lists(const unsigned char *mask, long mask_heads, long nT, int *row_ptr,
                   int *col_idx, int *col_ptr, int *row_idx) {
  if (!mask || mask_heads < 1 || nT < 1) return 1;
  for (long h = 0; h < mask_heads; ++h) {
    const unsigned char *m = mask + h * nT * nT;
    int *rp = row_ptr + h * (nT + 1), *ci = col_idx + h * nT * nT;
    int *cp = col_ptr + h * (nT + 1), *ri = row_idx + h * nT * nT;
    int n = 0;
    for (long i = 0; i < nT; ++i) {
      rp[i] = n;
      for (long j = 0; j < nT; ++j)
        if (m[i * nT + j]) ci[n++] = (int)j;
    }
    rp[nT] = n;
    n = 0;
    for (long j = 0; j < nT; ++j) {
      cp[j] = n;
      for (long i = 0; i < nT; ++i)
        if (m[i * nT + j]) ri[n++] = (int)i;
    }
    cp[nT] = n;
  }
  return 0;
}

/* For every query tile of every mask head (or the single dense head when
 * mask is NULL): the number of key tiles that hold at least one allowed
 * (query, key) element.  Brute force over elements.  counts: [heads, nT]. */
int fao_tile_counts(long N, long tile, int causal, const unsigned char *mask, long mask_heads,
                    long *counts) {
  if (N < 1 || tile < 1) return 1;
  long nT = (N + tile - 1) / tile;
  long heads = mask ? mask_heads : 1;
  problem_t p;
  memset(&p, 0, sizeof(p));
  p.N = N;
  p.H = heads;
  p.causal = causal;
  p.mask = mask;
  p.mask_heads = mask_heads;
  p.tile = tile;
  p.nT = nT;
  for (long h = 0; h < heads; ++h) {
    for (long a = 0; a < nT; ++a) {
      long cnt = 0;
      for (long b = 0; b < nT; ++b) {
        int any = 0;
        for (long i = a * tile; i < (a + 1) * tile && i < N && !any; ++i)
          for (long j = b * tile; j < (b + 1) * tile && j < N && !any; ++j)
            any = allowed(&p, h, i, j);
        cnt += any;
      }
      counts[h * nT + a] = cnt;
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* the dropout generator, exported for its known-answer pins               */
void fao_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  philox4x32_10(ctr, key, out);
}

/* random bytes of elements (bhc, i, j0 + n), n < count */
void fao_dropout_bytes(uint64_t seed, uint32_t offset, uint64_t bhc, uint64_t i, uint64_t j0,
                       long count, unsigned char *out) {
  for (long n = 0; n < count; ++n) out[n] = (unsigned char)keep_byte(seed, offset, bhc, i, j0 + n);
}
