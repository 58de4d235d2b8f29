/*
 * ulysses_oracle.c -- plain fp64 CPU oracle for the Ulysses attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  The CUDA library never links, includes or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark load it (through oracle/__init__.py).  It shares no code,
 * header, table or constant with the GPU path.
 *
 * Sources, cited by page title and section:
 *   [SP2] "Sequence Parallelism II: DeepSpeed Ulysses and All-to-All Attention"
 *   [CMP] "Comparing Ulysses and Megatron Sequence Parallelism"
 *
 * Everything is computed in double precision with plain loops, in the order
 * the pages describe the method.  Each virtual rank owns its own buffer (an
 * array of P pointers), and the All-to-All is an explicit double loop over
 * (destination, source) pairs that counts the bytes that cross ranks.
 *
 * Per-rank layouts (row-major, innermost last):
 *   sequence-sharded  X_r[b][t][head][e],  t < Sl = S/P    [CMP] "DeepSpeed Attention"
 *   head-sharded      Y_r[b][p][j][e],     p < S, j < heads/P
 *   log-sum-exp       L_r[b][j][p]
 *
 * Readings where the pages are silent (the plainest one that the rest of the
 * pages support):
 *   - rank r owns tokens [r*Sl, (r+1)*Sl) and, inside attention, the heads
 *     [r*hp, (r+1)*hp); received pieces are stored in source-rank order
 *     ([SP2] §1: rank 0 goes from S0H0,S0H1,S0H2,S0H3 to S0H0,S1H0,S2H0,S3H0);
 *   - softmax scale defaults to 1/sqrt(D) (the pages call plain scaled dot
 *     product attention, [CMP] "A simple attention skeleton");
 *   - causal mask: key position k attends for query position i iff k <= i;
 *   - grouped K/V heads: q-head g reads kv-head floor(g / (n_head/n_kv_head));
 *   - RoPE: rotate-half form, theta_i = base^(-2i/D) for i < D/2, applied to
 *     q and k with the token's global position before the transpose
 *     ([CMP] skeleton applies rope, then transposes).
 *
 * Parity: every function here is pinned by CPU tests against a pure-Python
 * brute force, closed forms, invariants, the pages' ownership example and
 * the pages' volume formula; see tests/test_oracle_pins.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

/* ------------------------------------------------------------------------ */
/* A tiny thread pool: items [0, n) are handed out by an atomic counter.     */
/* ------------------------------------------------------------------------ */
typedef void (*item_fn)(void *ctx, long item, double *scratch);

typedef struct {
  item_fn fn;
  void *ctx;
  long n_items;
  long next;
  long scratch_len;
} pool_job;

static void *pool_worker(void *arg) {
  pool_job *job = (pool_job *)arg;
  double *scratch = (double *)malloc(sizeof(double) * (size_t)(job->scratch_len > 0 ? job->scratch_len : 1));
  for (;;) {
    long it = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
    if (it >= job->n_items) break;
    job->fn(job->ctx, it, scratch);
  }
  free(scratch);
  return NULL;
}

static double wall_seconds(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return (double)ts.tv_sec + 1e-9 * (double)ts.tv_nsec;
}

static void run_items(item_fn fn, void *ctx, long n_items, long scratch_len, int nthreads) {
  pool_job job = {fn, ctx, n_items, 0, scratch_len};
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads == 1 || n_items <= 1) {
    pool_worker(&job);
    return;
  }
  pthread_t tid[256];
  int started = 0;
  for (int i = 0; i < nthreads; ++i)
    if (pthread_create(&tid[i], NULL, pool_worker, &job) == 0) ++started;
  if (started == 0) pool_worker(&job);
  for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
}

/* ------------------------------------------------------------------------ */
/* All-to-All, sequence shards -> head shards.                               */
/* [SP2] §3: every rank splits its local tensor into P pieces, keeps the     */
/* piece addressed to itself and sends the others; afterwards each rank has  */
/* one piece from every rank.  [CMP] "DeepSpeed Attention": the per-rank     */
/* tensor goes from [B, S/P, heads, D] to [B, S, heads/P, D].                */
/* The piece that rank `src` addresses to rank `dst` is its head slice       */
/* [dst*hp, (dst+1)*hp); rank `dst` stores it at sequence block `src`.       */
/* sent[r]/recv[r] accumulate the bytes of pieces with src != dst, counted   */
/* at `elem_bytes` per element ([CMP] "DeepSpeed Attention costs").          */
/* skip_src/skip_dst (>= 0) leave one piece undelivered: a test hook that    */
/* models a lost message.                                                     */
/* Returns 0, or -1 if heads is not a multiple of P.                          */
/* ------------------------------------------------------------------------ */
int oracle_a2a_seq_to_head(int P, int B, int Sl, int heads, int D, int elem_bytes,
                           const double *const *x_seq, double *const *y_head,
                           long long *sent, long long *recv, int skip_src, int skip_dst) {
  if (P <= 0 || heads % P != 0) return -1;
  const int hp = heads / P;
  const long S = (long)Sl * P;
  for (int dst = 0; dst < P; ++dst) {
    for (int src = 0; src < P; ++src) {
      if (src == skip_src && dst == skip_dst) continue;
      const double *x = x_seq[src];
      double *y = y_head[dst];
      for (int b = 0; b < B; ++b)
        for (int t = 0; t < Sl; ++t)
          for (int j = 0; j < hp; ++j) {
            const double *from = x + (((long)b * Sl + t) * heads + ((long)dst * hp + j)) * D;
            double *to = y + (((long)b * S + ((long)src * Sl + t)) * hp + j) * D;
            for (int e = 0; e < D; ++e) to[e] = from[e];
          }
      if (src != dst) {
        long long piece = (long long)B * Sl * hp * D * elem_bytes;
        if (sent) sent[src] += piece;
        if (recv) recv[dst] += piece;
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* All-to-All, head shards -> sequence shards (the inverse).                 */
/* [SP2] §2 fifth step and [CMP] "DeepSpeed Attention": [B, S, heads/P, D]   */
/* becomes [B, S/P, heads, D], equivalently [B, S/P, heads*D] with feature   */
/* index head*D + e.  Rank `src` (holding heads [src*hp, ...)) sends its     */
/* sequence block `dst` to rank `dst`.                                        */
/* ------------------------------------------------------------------------ */
int oracle_a2a_head_to_seq(int P, int B, int Sl, int heads, int D, int elem_bytes,
                           const double *const *y_head, double *const *x_seq,
                           long long *sent, long long *recv, int skip_src, int skip_dst) {
  if (P <= 0 || heads % P != 0) return -1;
  const int hp = heads / P;
  const long S = (long)Sl * P;
  for (int dst = 0; dst < P; ++dst) {
    for (int src = 0; src < P; ++src) {
      if (src == skip_src && dst == skip_dst) continue;
      const double *y = y_head[src];
      double *x = x_seq[dst];
      for (int b = 0; b < B; ++b)
        for (int t = 0; t < Sl; ++t)
          for (int j = 0; j < hp; ++j) {
            const double *from = y + (((long)b * S + ((long)dst * Sl + t)) * hp + j) * D;
            double *to = x + (((long)b * Sl + t) * heads + ((long)src * hp + j)) * D;
            for (int e = 0; e < D; ++e) to[e] = from[e];
          }
      if (src != dst) {
        long long piece = (long long)B * Sl * hp * D * elem_bytes;
        if (sent) sent[src] += piece;
        if (recv) recv[dst] += piece;
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* RoPE on sequence-sharded buffers, in place.                               */
/* [CMP] "A simple attention skeleton" applies rope to q and k right after   */
/* the projections, before the transpose; the formula itself is not on the  */
/* pages.  Rotate-half form: for i < D/2, angle a = p * base^(-2i/D),        */
/*   x'_i       = x_i cos a - x_{i+D/2} sin a                                */
/*   x'_{i+D/2} = x_{i+D/2} cos a + x_i sin a                                */
/* with p = r*Sl + t the token's global position.  direction = -1 applies    */
/* the inverse rotation (angle -a), which is the chain rule of RoPE for the  */
/* gradients of q and k.                                                      */
/* ------------------------------------------------------------------------ */
void oracle_rope_seq(int P, int B, int Sl, int heads, int D, double base, int direction,
                     double *const *x_seq) {
  const int half = D / 2;
  double *c = (double *)malloc(sizeof(double) * (size_t)(half > 0 ? half : 1));
  double *s = (double *)malloc(sizeof(double) * (size_t)(half > 0 ? half : 1));
  for (int r = 0; r < P; ++r)
    for (int t = 0; t < Sl; ++t) {
      const double p = (double)r * Sl + t;
      for (int i = 0; i < half; ++i) {
        double theta = pow(base, -2.0 * i / D);
        double a = direction * p * theta;
        c[i] = cos(a);
        s[i] = sin(a);
      }
      for (int b = 0; b < B; ++b)
        for (int h = 0; h < heads; ++h) {
          double *v = x_seq[r] + (((long)b * Sl + t) * heads + h) * D;
          for (int i = 0; i < half; ++i) {
            double x1 = v[i], x2 = v[i + half];
            v[i] = x1 * c[i] - x2 * s[i];
            v[i + half] = x2 * c[i] + x1 * s[i];
          }
        }
    }
  free(c);
  free(s);
}

/* ------------------------------------------------------------------------ */
/* Softmax attention for one query row of one head.                          */
/* [SP2] §2 fourth step: the rank has the full sequence for its heads, so    */
/* the attention for those heads is ordinary local attention.                */
/*   s_k = scale * <q, k_k>,  k < n_keys                                     */
/*   o   = sum_k exp(s_k - m) v_k / sum_k exp(s_k - m),  m = max_k s_k       */
/*   lse = m + log(sum_k exp(s_k - m))                                       */
/* k_k lives at kb + k*ks, v_k at vb + k*vs.  w is scratch of n_keys.        */
/* ------------------------------------------------------------------------ */
static void attend_row(int D, long n_keys, const double *q, const double *kb, long ks,
                       const double *vb, long vs, double scale, double *o, double *lse, double *w) {
  double m = -INFINITY;
  for (long k = 0; k < n_keys; ++k) {
    const double *kk = kb + k * ks;
    double dot = 0.0;
    for (int e = 0; e < D; ++e) dot += q[e] * kk[e];
    w[k] = scale * dot;
    if (w[k] > m) m = w[k];
  }
  double l = 0.0;
  for (long k = 0; k < n_keys; ++k) {
    w[k] = exp(w[k] - m);
    l += w[k];
  }
  for (int e = 0; e < D; ++e) o[e] = 0.0;
  for (long k = 0; k < n_keys; ++k) {
    const double *vv = vb + k * vs;
    for (int e = 0; e < D; ++e) o[e] += w[k] * vv[e];
  }
  for (int e = 0; e < D; ++e) o[e] /= l;
  *lse = m + log(l);
}

typedef struct {
  int P, B, S, n_head, n_kv_head, D, causal;
  double scale;
} oracle_shape;

/* Query-head g (global) -> kv-head (global), contiguous groups. */
static int kv_head_of(const oracle_shape *sh, int g) { return g / (sh->n_head / sh->n_kv_head); }

/* KV-head replication (n_kv_head < P, P a multiple of n_kv_head): the q-heads
   of rank r all read kv-head r / R (R = P / n_kv_head), so the seq -> head
   All-to-All hands that kv-head to each of its R ranks and every rank holds
   one kv-head in head layout.  Otherwise a rank holds n_kv_head / P kv-heads
   starting at r * n_kv_head / P. */
static int kv_per_rank(const oracle_shape *sh) {
  return sh->n_kv_head >= sh->P ? sh->n_kv_head / sh->P : 1;
}
static int rank_kv_base(const oracle_shape *sh, int r) {
  return sh->n_kv_head >= sh->P ? r * (sh->n_kv_head / sh->P) : r / (sh->P / sh->n_kv_head);
}
/* The head counts the method defines: P divides n_head, n_kv_head divides
   n_head, and P and n_kv_head divide one another. */
static int heads_ok(const oracle_shape *sh) {
  if (sh->P <= 0 || sh->n_kv_head <= 0 || sh->n_head % sh->P || sh->n_head % sh->n_kv_head) return 0;
  return sh->n_kv_head % sh->P == 0 || sh->P % sh->n_kv_head == 0;
}

typedef struct {
  const oracle_shape *sh;
  const double *const *q, *const *k, *const *v;
  double *const *o;
  double *const *lse;
  const int *rows;
  long n_rows;
  long chunk;
} fwd_ctx;

/* One work item = (rank, batch, local head, chunk of query rows). */
static void fwd_item(void *vctx, long item, double *w) {
  fwd_ctx *c = (fwd_ctx *)vctx;
  const oracle_shape *sh = c->sh;
  const int hp = sh->n_head / sh->P, kvp = kv_per_rank(sh), D = sh->D;
  const long S = sh->S;
  long n_chunks = (c->n_rows + c->chunk - 1) / c->chunk;
  long ch = item % n_chunks;
  long rest = item / n_chunks;
  int j = (int)(rest % hp);
  rest /= hp;
  int b = (int)(rest % sh->B);
  int r = (int)(rest / sh->B);
  int g = r * hp + j;
  int kl = kv_head_of(sh, g) - rank_kv_base(sh, r); /* local kv index on rank r */
  const double *K = c->k[r] + ((long)b * S * kvp + kl) * D;
  const double *V = c->v[r] + ((long)b * S * kvp + kl) * D;
  for (long ii = ch * c->chunk; ii < c->n_rows && ii < (ch + 1) * c->chunk; ++ii) {
    long i = c->rows ? c->rows[ii] : ii;
    const double *qi = c->q[r] + (((long)b * S + i) * hp + j) * D;
    double *oi = c->o[r] + (((long)b * S + i) * hp + j) * D;
    long n_keys = sh->causal ? i + 1 : S;
    attend_row(D, n_keys, qi, K, (long)kvp * D, V, (long)kvp * D, sh->scale, oi,
               c->lse[r] + ((long)b * hp + j) * S + i, w);
  }
}

/* ------------------------------------------------------------------------ */
/* Attention on head-sharded buffers: for every rank r, batch b and local    */
/* head j, attention of q-head g = r*hp + j over the full sequence.          */
/* rows = NULL computes every query row; otherwise only the listed global    */
/* positions (each row is exact over its full key range).                    */
/* Returns 0, or -1 on a shape the method does not define.                   */
/* ------------------------------------------------------------------------ */
int oracle_attention_fwd(const oracle_shape *sh, const double *const *q_head,
                         const double *const *k_head, const double *const *v_head,
                         double *const *o_head, double *const *lse, const int *rows, long n_rows,
                         int nthreads) {
  if (!heads_ok(sh)) return -1;
  fwd_ctx c = {sh, q_head, k_head, v_head, o_head, lse, rows, rows ? n_rows : sh->S, 64};
  long n_chunks = (c.n_rows + c.chunk - 1) / c.chunk;
  long items = (long)sh->P * sh->B * (sh->n_head / sh->P) * n_chunks;
  run_items(fwd_item, &c, items, sh->S, nthreads);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Unsharded attention on global tensors q[B][S][n_head][D], k/v[B][S][n_kv] */
/* [D]; o[B][S][n_head][D], lse[B][n_head][S].  The pages' claim that the    */
/* Ulysses transposes are only a permutation of ownership ([SP2] §1, §3) is  */
/* tested by comparing this with the sharded pipeline.                       */
/* ------------------------------------------------------------------------ */
typedef struct {
  const oracle_shape *sh;
  const double *q, *k, *v;
  double *o, *lse;
} glob_ctx;

static void glob_item(void *vctx, long item, double *w) {
  glob_ctx *c = (glob_ctx *)vctx;
  const oracle_shape *sh = c->sh;
  const int H = sh->n_head, KV = sh->n_kv_head, D = sh->D;
  const long S = sh->S;
  int g = (int)(item % H);
  int b = (int)(item / H);
  int kvh = kv_head_of(sh, g);
  const double *K = c->k + ((long)b * S * KV + kvh) * D;
  const double *V = c->v + ((long)b * S * KV + kvh) * D;
  for (long i = 0; i < S; ++i) {
    long n_keys = sh->causal ? i + 1 : S;
    attend_row(D, n_keys, c->q + (((long)b * S + i) * H + g) * D, K, (long)KV * D, V,
               (long)KV * D, sh->scale, c->o + (((long)b * S + i) * H + g) * D,
               c->lse + ((long)b * H + g) * S + i, w);
  }
}

int oracle_attention_unsharded(const oracle_shape *sh, const double *q, const double *k,
                               const double *v, double *o, double *lse, int nthreads) {
  if (sh->n_kv_head <= 0 || sh->n_head % sh->n_kv_head) return -1;
  glob_ctx c = {sh, q, k, v, o, lse};
  run_items(glob_item, &c, (long)sh->B * sh->n_head, sh->S, nthreads);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward of the per-head attention, head-sharded buffers.                 */
/* [SP2] §6: the output gradient arrives in head layout; Q, K, V gradients   */
/* are produced per head and sent back.  The gradient formulas are those of  */
/* softmax(scale * q k^T) v, written out (the pages do not print them):      */
/*   P_ik  = exp(s_ik - lse_i)            dP_ik = <dO_i, v_k>                */
/*   D_i   = <dO_i, o_i>                  dS_ik = P_ik (dP_ik - D_i)         */
/*   dq_i  = scale * sum_k dS_ik k_k                                          */
/*   dk_k  = scale * sum_{g in group} sum_i dS_ik q_i                         */
/*   dv_k  = sum_{g in group} sum_i P_ik dO_i                                 */
/* where the group of a kv-head is the q-heads that read it.                 */
/* One call handles one (rank, batch, local kv-head) group.  It recomputes   */
/* o_i and lse_i for all rows of the group's q-heads first.  dq is written   */
/* for the rows in q_rows (NULL = all), dk/dv for the key rows in kv_rows    */
/* (NULL = all); other rows are left untouched.  phase_seconds (NULL: not    */
/* wanted) receives the wall time of the three phases (statistics, dq,       */
/* dk/dv): instrumentation for the benchmark's CPU baseline, no arithmetic.  */
/* ------------------------------------------------------------------------ */
typedef struct {
  const oracle_shape *sh;
  int r, b, kl, G;
  const double *const *q, *const *k, *const *v, *const *dout;
  double *const *dq, *const *dk, *const *dv;
  const int *q_rows, *kv_rows;
  long n_q_rows, n_kv_rows;
  double *lse;   /* [G][S] */
  double *delta; /* [G][S] */
  int phase;
} bwd_ctx;

static const double *row_ptr(const double *base, long S, int width, int b, long i, int j, int D) {
  return base + (((long)b * S + i) * width + j) * D;
}

static void bwd_item(void *vctx, long item, double *w) {
  bwd_ctx *c = (bwd_ctx *)vctx;
  const oracle_shape *sh = c->sh;
  const int hp = sh->n_head / sh->P, kvp = kv_per_rank(sh), D = sh->D;
  const long S = sh->S;
  const int r = c->r, b = c->b, kl = c->kl;
  const double *K = row_ptr(c->k[r], S, kvp, b, 0, kl, D);
  const double *V = row_ptr(c->v[r], S, kvp, b, 0, kl, D);
  const long kvs = (long)kvp * D;
  if (c->phase == 0) {
    /* forward statistics for row i of group head gi: lse_i and D_i. */
    int gi = (int)(item / S);
    long i = item % S;
    int j = kl * c->G + gi; /* local q-head on rank r */
    const double *qi = row_ptr(c->q[r], S, hp, b, i, j, D);
    const double *doi = row_ptr(c->dout[r], S, hp, b, i, j, D);
    double *o = w + S;
    double lse;
    attend_row(D, sh->causal ? i + 1 : S, qi, K, kvs, V, kvs, sh->scale, o, &lse, w);
    double dd = 0.0;
    for (int e = 0; e < D; ++e) dd += doi[e] * o[e];
    c->lse[(long)gi * S + i] = lse;
    c->delta[(long)gi * S + i] = dd;
  } else if (c->phase == 1) {
    /* dq for one query row of one group head. */
    int gi = (int)(item / c->n_q_rows);
    long ii = item % c->n_q_rows;
    long i = c->q_rows ? c->q_rows[ii] : ii;
    int j = kl * c->G + gi;
    const double *qi = row_ptr(c->q[r], S, hp, b, i, j, D);
    const double *doi = row_ptr(c->dout[r], S, hp, b, i, j, D);
    double *dqi = (double *)row_ptr(c->dq[r], S, hp, b, i, j, D);
    const double lse = c->lse[(long)gi * S + i], dd = c->delta[(long)gi * S + i];
    for (int e = 0; e < D; ++e) dqi[e] = 0.0;
    long n_keys = sh->causal ? i + 1 : S;
    for (long kk = 0; kk < n_keys; ++kk) {
      const double *kr = K + kk * kvs, *vr = V + kk * kvs;
      double s = 0.0, dp = 0.0;
      for (int e = 0; e < D; ++e) s += qi[e] * kr[e];
      for (int e = 0; e < D; ++e) dp += doi[e] * vr[e];
      double p = exp(sh->scale * s - lse);
      double ds = p * (dp - dd);
      for (int e = 0; e < D; ++e) dqi[e] += sh->scale * ds * kr[e];
    }
  } else {
    /* dk, dv for one key row, summed over the group's q-heads. */
    long kk = c->kv_rows ? c->kv_rows[item] : item;
    const double *kr = K + kk * kvs, *vr = V + kk * kvs;
    double *dkr = (double *)row_ptr(c->dk[r], S, kvp, b, kk, kl, D);
    double *dvr = (double *)row_ptr(c->dv[r], S, kvp, b, kk, kl, D);
    for (int e = 0; e < D; ++e) dkr[e] = dvr[e] = 0.0;
    for (int gi = 0; gi < c->G; ++gi) {
      int j = kl * c->G + gi;
      for (long i = sh->causal ? kk : 0; i < S; ++i) {
        const double *qi = row_ptr(c->q[r], S, hp, b, i, j, D);
        const double *doi = row_ptr(c->dout[r], S, hp, b, i, j, D);
        double s = 0.0, dp = 0.0;
        for (int e = 0; e < D; ++e) s += qi[e] * kr[e];
        for (int e = 0; e < D; ++e) dp += doi[e] * vr[e];
        double p = exp(sh->scale * s - c->lse[(long)gi * S + i]);
        double ds = p * (dp - c->delta[(long)gi * S + i]);
        for (int e = 0; e < D; ++e) {
          dvr[e] += p * doi[e];
          dkr[e] += sh->scale * ds * qi[e];
        }
      }
    }
  }
}

int oracle_attention_bwd_group(const oracle_shape *sh, int r, int b, int kl,
                               const double *const *q_head, const double *const *k_head,
                               const double *const *v_head, const double *const *do_head,
                               double *const *dq_head, double *const *dk_head,
                               double *const *dv_head, const int *q_rows, long n_q_rows,
                               const int *kv_rows, long n_kv_rows, int nthreads,
                               double *phase_seconds) {
  if (!heads_ok(sh)) return -1;
  const long S = sh->S;
  bwd_ctx c;
  memset(&c, 0, sizeof c);
  c.sh = sh;
  c.r = r;
  c.b = b;
  c.kl = kl;
  /* q-heads of rank r that read local kv-head kl: the whole group, or with
     replicated kv-heads the rank's own hp (its share of the group; the other
     replicas hold the rest and their dk, dv are summed afterwards). */
  c.G = (sh->n_head / sh->P) / kv_per_rank(sh);
  c.q = q_head;
  c.k = k_head;
  c.v = v_head;
  c.dout = do_head;
  c.dq = dq_head;
  c.dk = dk_head;
  c.dv = dv_head;
  c.q_rows = q_rows;
  c.kv_rows = kv_rows;
  c.n_q_rows = q_rows ? n_q_rows : S;
  c.n_kv_rows = kv_rows ? n_kv_rows : S;
  c.lse = (double *)malloc(sizeof(double) * (size_t)c.G * S);
  c.delta = (double *)malloc(sizeof(double) * (size_t)c.G * S);
  if (!c.lse || !c.delta) {
    free(c.lse);
    free(c.delta);
    return -2;
  }
  double t[4] = {0.0, 0.0, 0.0, 0.0};
  t[0] = wall_seconds();
  c.phase = 0;
  run_items(bwd_item, &c, (long)c.G * S, S + sh->D, nthreads);
  t[1] = wall_seconds();
  if (dq_head) {
    c.phase = 1;
    run_items(bwd_item, &c, (long)c.G * c.n_q_rows, 1, nthreads);
  }
  t[2] = wall_seconds();
  if (dk_head && dv_head) {
    c.phase = 2;
    run_items(bwd_item, &c, c.n_kv_rows, 1, nthreads);
  }
  t[3] = wall_seconds();
  if (phase_seconds)
    for (int i = 0; i < 3; ++i) phase_seconds[i] = t[i + 1] - t[i];
  free(c.lse);
  free(c.delta);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* KV-head replication, seq -> head: the All-to-All for K and V when        */
/* n_kv_head = heads < P.  Destination rank dst needs the kv-head its        */
/* q-heads read, kv = dst / R (R = P / heads), over the full sequence; every */
/* source rank sends it its Sl tokens of that head:                          */
/*   y_dst[b][src*Sl + t][0][e] = x_src[b][t][dst/R][e]                       */
/* Bytes of pieces with src != dst are counted as in oracle_a2a_seq_to_head. */
/* Returns 0, or -1 unless heads divides P.                                  */
/* ------------------------------------------------------------------------ */
int oracle_a2a_seq_to_head_rep(int P, int B, int Sl, int heads, int D, int elem_bytes,
                               const double *const *x_seq, double *const *y_head,
                               long long *sent, long long *recv) {
  if (P <= 0 || heads <= 0 || P % heads != 0) return -1;
  const int R = P / heads;
  const long S = (long)Sl * P;
  for (int dst = 0; dst < P; ++dst) {
    const int kv = dst / R;
    for (int src = 0; src < P; ++src) {
      const double *x = x_seq[src];
      double *y = y_head[dst];
      for (int b = 0; b < B; ++b)
        for (int t = 0; t < Sl; ++t) {
          const double *from = x + (((long)b * Sl + t) * heads + kv) * D;
          double *to = y + ((long)b * S + ((long)src * Sl + t)) * D;
          for (int e = 0; e < D; ++e) to[e] = from[e];
        }
      if (src != dst) {
        const long long piece = (long long)B * Sl * D * elem_bytes;
        if (sent) sent[src] += piece;
        if (recv) recv[dst] += piece;
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* KV-head replication, head -> seq for the gradients of K and V.  The       */
/* forward copied kv-head kv to the R ranks kv*R .. kv*R+R-1, so its         */
/* gradient is the sum of what those ranks computed (the chain rule of a     */
/* copy), added in rank order:                                               */
/*   x_dst[b][t][kv][e] = sum_{j<R} y_{kv*R+j}[b][dst*Sl + t][0][e]           */
/* Every replica sends its Sl rows for dst to dst; bytes of pieces with      */
/* src != dst are counted.  Returns 0, or -1 unless heads divides P.         */
/* ------------------------------------------------------------------------ */
int oracle_reduce_head_to_seq_rep(int P, int B, int Sl, int heads, int D, int elem_bytes,
                                  const double *const *y_head, double *const *x_seq,
                                  long long *sent, long long *recv) {
  if (P <= 0 || heads <= 0 || P % heads != 0) return -1;
  const int R = P / heads;
  const long S = (long)Sl * P;
  for (int dst = 0; dst < P; ++dst) {
    double *x = x_seq[dst];
    for (int b = 0; b < B; ++b)
      for (int t = 0; t < Sl; ++t)
        for (int kv = 0; kv < heads; ++kv) {
          double *to = x + (((long)b * Sl + t) * heads + kv) * D;
          for (int e = 0; e < D; ++e) to[e] = 0.0;
          for (int j = 0; j < R; ++j) {
            const double *from = y_head[kv * R + j] + ((long)b * S + ((long)dst * Sl + t)) * D;
            for (int e = 0; e < D; ++e) to[e] += from[e];
          }
        }
    for (int src = 0; src < P; ++src)
      if (src != dst) {
        const long long piece = (long long)B * Sl * D * elem_bytes;
        if (sent) sent[src] += piece;
        if (recv) recv[dst] += piece;
      }
  }
  return 0;
}
