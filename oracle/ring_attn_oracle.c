/*
 * ring_attn_oracle.c -- plain fp64 CPU oracle for blockwise Ring Self-Attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or constant with
 * the CUDA library.
 *
 * What it computes (all arithmetic in double precision on the bf16 input
 * values, which the caller passes already widened to double):
 *
 *   Self-attention as two matrix products, softmax(Q K^T / sqrt(d)) V
 *   ("Sequence parallelism" series, section 2.3 Ring Self-Attention: the
 *   computation is Q*K^T followed by AttentionScore*V).  For batch b, query
 *   head h and query row i, with kv head g = floor(h / (Hq/Hkv)) (grouped
 *   query attention with consecutive grouping) and scale = 1/sqrt(d):
 *
 *     s_ij  = scale * sum_c q[b,h,i,c] * k[b,g,j,c]     for j in V(i)
 *     V(i)  = {0..L-1} (encoder, no mask)  or  {0..i} (causal decoder)
 *     lse_i = log sum_{j in V(i)} exp(s_ij)   (natural log, max-subtracted)
 *     P_ij  = exp(s_ij - lse_i)
 *     o_i   = sum_j P_ij v[b,g,j,:]
 *
 *   Backward of the loss l = sum(dO * O), derived by hand (the pages only
 *   say that the backward pass recomputes the attention; Ring Attention
 *   section 6.2 and the BPT section 4.3 use activation recomputation):
 *
 *     D_i   = sum_c dO_ic * o_ic          (o from this oracle, in fp64)
 *     dP_ij = dO_i . v_j
 *     dS_ij = P_ij * (dP_ij - D_i)
 *     dq_i  = scale * sum_j dS_ij k_j
 *     dk_j  = scale * sum_{h in group(g)} sum_i dS_ij q_i
 *     dv_j  =         sum_{h in group(g)} sum_i P_ij dO_i
 *
 *   Ring form (Ring Self-Attention, section 2.3; Ring Attention, section
 *   6.2): the sequence is cut into N chunks, rank r owns chunk r (encoder)
 *   or the folded pair of sub-chunks {r, 2N-1-r} of length L/(2N) (causal,
 *   the fold of the USP section 8.2).  At ring step s = 0..N-1 rank r holds
 *   the keys/values of rank (r - s) mod N, computes the partial result of
 *   that block (o_s, lse_s) and merges it into its running result with the
 *   log-sum-exp rule (the online-softmax correction of section 6.2).  With
 *   the striped assignment (a causal schedule variant the pages compare
 *   with the fold: rank r owns positions r, r+N, r+2N, ...), every rank's
 *   chunk spreads over the whole sequence instead; with contiguous causal
 *   chunks, either the plain ring or DistFlashAttention's balanced schedule
 *   (section 7.2: a worker that would wait takes over a later worker's
 *   block; see dfa_pair) orders the blocks.  The merge:
 *
 *     lse <- log(exp(lse) + exp(lse_s)),
 *     o   <- exp(lse_old - lse) * o + exp(lse_s - lse) * o_s.
 *
 *   Blockwise feed-forward of the BPT layer (section 4.2: per query block,
 *   attention, then the FFN and the residual; section 8: two linear layers
 *   around a 4x up-projection).  Per row x_m (rows are independent, so the
 *   blockwise order does not change the result):
 *
 *     y_m = x_m + W2^T gelu(W1^T x_m + b1) + b2,  gelu(t) = t Phi(t),
 *     Phi(t) = erfc(-t / sqrt 2) / 2  (the standard normal CDF)
 *
 *   and its backward for the loss sum(dy * y) by the chain rule, with the
 *   hidden activation recomputed (oracle_ffn_bwd).  Pinned by torch's fp64
 *   autograd, central differences, closed forms (W2 = 0) and a 40-digit
 *   evaluation of the GELU tail.
 *
 * Layout: q, o, dO, dq are [B][Hq][L][d]; k, v, dk, dv are [B][Hkv][L][d];
 * lse and D are [B][Hq][L]; all contiguous, row-major.  FFN: x, y, dy, dx
 * [M][D], W1 [D][F], W2 [F][D].
 *
 * Parallelism: plain pthreads over independent rows; no blocking, fusion
 * or reordering of the arithmetic of one row.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
  const double *q, *k, *v, *dO;
  int B, Hq, Hkv, L, d, causal;
  double scale;
} problem_t;

static const double *q_row(const problem_t *P, int b, int h, int i) {
  return P->q + (((size_t)b * P->Hq + h) * P->L + i) * (size_t)P->d;
}
static const double *do_row(const problem_t *P, int b, int h, int i) {
  return P->dO + (((size_t)b * P->Hq + h) * P->L + i) * (size_t)P->d;
}
static const double *k_row(const problem_t *P, int b, int g, int j) {
  return P->k + (((size_t)b * P->Hkv + g) * P->L + j) * (size_t)P->d;
}
static const double *v_row(const problem_t *P, int b, int g, int j) {
  return P->v + (((size_t)b * P->Hkv + g) * P->L + j) * (size_t)P->d;
}
static double dot(const double *a, const double *b, int n) {
  double s = 0.0;
  for (int c = 0; c < n; ++c) s += a[c] * b[c];
  return s;
}
/* Number of keys row i may attend to: j in [0, n_visible). */
static int n_visible(const problem_t *P, int i) { return P->causal ? i + 1 : P->L; }

/* ---------------------------------------------------------------- forward */

/* One query row of the plain definition.  s is scratch of length L. */
static void fwd_row(const problem_t *P, int b, int h, int i, double *s, double *o, double *lse_out) {
  const int g = h / (P->Hq / P->Hkv);
  const double *qi = q_row(P, b, h, i);
  const int n = n_visible(P, i);
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    s[j] = P->scale * dot(qi, k_row(P, b, g, j), P->d);
    if (s[j] > m) m = s[j];
  }
  double sum = 0.0;
  for (int j = 0; j < n; ++j) sum += exp(s[j] - m);
  const double lse = m + log(sum);
  for (int c = 0; c < P->d; ++c) o[c] = 0.0;
  for (int j = 0; j < n; ++j) {
    const double p = exp(s[j] - lse);
    const double *vj = v_row(P, b, g, j);
    for (int c = 0; c < P->d; ++c) o[c] += p * vj[c];
  }
  *lse_out = lse;
}

/* ------------------------------------------------------------ thread pool */

typedef struct task_s task_t;
typedef void (*task_fn)(task_t *t, long item, double *scratch);
struct task_s {
  const problem_t *P;
  long n_items;
  long next; /* atomic work counter */
  task_fn fn;
  size_t scratch_len;
  /* per-task arguments */
  const int *rows; int n_rows;
  double *o, *lse, *D, *dq, *dk, *dv;
  int n_chunks;
  int rank, src;      /* ring step mode: query rank and key/value source rank */
  int schedule;       /* ring forms: chunk map and step order (SCHED_*) */
  const int *stat_lo; /* per (b,h): first query row whose stats exist (rows mode) */
};

static void *worker(void *arg) {
  task_t *t = (task_t *)arg;
  double *scratch = (double *)malloc(sizeof(double) * (t->scratch_len ? t->scratch_len : 1));
  for (;;) {
    long it = __atomic_fetch_add(&t->next, 1, __ATOMIC_RELAXED);
    if (it >= t->n_items) break;
    t->fn(t, it, scratch);
  }
  free(scratch);
  return NULL;
}

static int run_parallel(task_t *t, int n_threads) {
  if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if ((long)n_threads > t->n_items) n_threads = (int)(t->n_items > 0 ? t->n_items : 1);
  t->next = 0;
  pthread_t th[256];
  int started = 0;
  for (int i = 1; i < n_threads; ++i)
    if (pthread_create(&th[i], NULL, worker, t) == 0) started = i; else break;
  worker(t);
  for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
  return n_threads;
}

static problem_t make_problem(const double *q, const double *k, const double *v, const double *dO,
                              int B, int Hq, int Hkv, int L, int d, int causal) {
  problem_t P;
  P.q = q; P.k = k; P.v = v; P.dO = dO;
  P.B = B; P.Hq = Hq; P.Hkv = Hkv; P.L = L; P.d = d; P.causal = causal;
  P.scale = 1.0 / sqrt((double)d);
  return P;
}

static int bad_shape(int B, int Hq, int Hkv, int L, int d) {
  return B < 0 || Hq <= 0 || Hkv <= 0 || L < 0 || d <= 0 || Hq % Hkv != 0;
}

/* Full forward: every row of every (b, h). */
static void fwd_full_item(task_t *t, long item, double *s) {
  const problem_t *P = t->P;
  const int i = (int)(item % P->L);
  const long bh = item / P->L;
  const int h = (int)(bh % P->Hq), b = (int)(bh / P->Hq);
  const size_t r = (size_t)bh * P->L + i;
  fwd_row(P, b, h, i, s, t->o + r * P->d, t->lse + r);
}

int oracle_fwd(const double *q, const double *k, const double *v, int B, int Hq, int Hkv, int L, int d,
               int causal, double *o, double *lse, int n_threads) {
  if (bad_shape(B, Hq, Hkv, L, d)) return -1;
  problem_t P = make_problem(q, k, v, NULL, B, Hq, Hkv, L, d, causal);
  task_t t; memset(&t, 0, sizeof t);
  t.P = &P; t.n_items = (long)B * Hq * L; t.fn = fwd_full_item; t.scratch_len = (size_t)L;
  t.o = o; t.lse = lse;
  return run_parallel(&t, n_threads);
}

/* Forward on a list of query rows, the same list for every (b, h).
 * o_rows is [B][Hq][n_rows][d], lse_rows is [B][Hq][n_rows]. */
static void fwd_rows_item(task_t *t, long item, double *s) {
  const problem_t *P = t->P;
  const int ri = (int)(item % t->n_rows);
  const long bh = item / t->n_rows;
  const int h = (int)(bh % P->Hq), b = (int)(bh / P->Hq);
  const size_t r = (size_t)bh * t->n_rows + ri;
  fwd_row(P, b, h, t->rows[ri], s, t->o + r * P->d, t->lse + r);
}

int oracle_fwd_rows(const double *q, const double *k, const double *v, int B, int Hq, int Hkv, int L, int d,
                    int causal, const int *rows, int n_rows, double *o_rows, double *lse_rows,
                    int n_threads) {
  if (bad_shape(B, Hq, Hkv, L, d) || n_rows < 0) return -1;
  for (int i = 0; i < n_rows; ++i) if (rows[i] < 0 || rows[i] >= L) return -1;
  problem_t P = make_problem(q, k, v, NULL, B, Hq, Hkv, L, d, causal);
  task_t t; memset(&t, 0, sizeof t);
  t.P = &P; t.n_items = (long)B * Hq * n_rows; t.fn = fwd_rows_item; t.scratch_len = (size_t)L;
  t.rows = rows; t.n_rows = n_rows; t.o = o_rows; t.lse = lse_rows;
  return run_parallel(&t, n_threads);
}

/* --------------------------------------------------------------- backward */

/* Statistics of one query row needed by the backward: lse_i and D_i. */
static void stats_row(const problem_t *P, int b, int h, int i, double *s, double *lse, double *D) {
  double *o = s + P->L; /* scratch holds L + d doubles */
  fwd_row(P, b, h, i, s, o, lse);
  *D = dot(do_row(P, b, h, i), o, P->d);
}

/* dq for one query row, given its lse and D. */
static void dq_row(const problem_t *P, int b, int h, int i, double lse, double D, double *dq) {
  const int g = h / (P->Hq / P->Hkv);
  const double *qi = q_row(P, b, h, i), *doi = do_row(P, b, h, i);
  for (int c = 0; c < P->d; ++c) dq[c] = 0.0;
  const int n = n_visible(P, i);
  for (int j = 0; j < n; ++j) {
    const double sij = P->scale * dot(qi, k_row(P, b, g, j), P->d);
    const double pij = exp(sij - lse);
    const double dpij = dot(doi, v_row(P, b, g, j), P->d);
    const double dsij = pij * (dpij - D);
    const double *kj = k_row(P, b, g, j);
    for (int c = 0; c < P->d; ++c) dq[c] += P->scale * dsij * kj[c];
  }
}

/* dk and dv for one key row j of kv head g.  lse and D are indexed
 * [(b*Hq + h)*L + i] and must be valid for every query row that sees j. */
static void dkdv_row(const problem_t *P, int b, int g, int j, const double *lse, const double *D,
                     double *dk, double *dv) {
  const int G = P->Hq / P->Hkv;
  const double *kj = k_row(P, b, g, j), *vj = v_row(P, b, g, j);
  for (int c = 0; c < P->d; ++c) { dk[c] = 0.0; dv[c] = 0.0; }
  for (int h = g * G; h < (g + 1) * G; ++h) {
    const size_t base = ((size_t)b * P->Hq + h) * P->L;
    for (int i = P->causal ? j : 0; i < P->L; ++i) {
      const double *qi = q_row(P, b, h, i), *doi = do_row(P, b, h, i);
      const double sij = P->scale * dot(qi, kj, P->d);
      const double pij = exp(sij - lse[base + i]);
      const double dpij = dot(doi, vj, P->d);
      const double dsij = pij * (dpij - D[base + i]);
      for (int c = 0; c < P->d; ++c) {
        dv[c] += pij * doi[c];
        dk[c] += P->scale * dsij * qi[c];
      }
    }
  }
}

static void stats_item(task_t *t, long item, double *s) {
  const problem_t *P = t->P;
  const long bh = item / P->L;
  const int i = (int)(item % P->L);
  const int h = (int)(bh % P->Hq), b = (int)(bh / P->Hq);
  if (t->stat_lo && i < t->stat_lo[bh]) return;
  const size_t r = (size_t)bh * P->L + i;
  stats_row(P, b, h, i, s, t->lse + r, t->D + r);
}
static void dq_full_item(task_t *t, long item, double *s) {
  (void)s;
  const problem_t *P = t->P;
  const long bh = item / P->L;
  const int i = (int)(item % P->L);
  const int h = (int)(bh % P->Hq), b = (int)(bh / P->Hq);
  const size_t r = (size_t)bh * P->L + i;
  dq_row(P, b, h, i, t->lse[r], t->D[r], t->dq + r * P->d);
}
static void dkdv_full_item(task_t *t, long item, double *s) {
  (void)s;
  const problem_t *P = t->P;
  const long bg = item / P->L;
  const int j = (int)(item % P->L);
  const int g = (int)(bg % P->Hkv), b = (int)(bg / P->Hkv);
  const size_t r = (size_t)bg * P->L + j;
  dkdv_row(P, b, g, j, t->lse, t->D, t->dk + r * P->d, t->dv + r * P->d);
}

/* Full backward.  Also returns the oracle's own lse and D ([B][Hq][L]). */
int oracle_bwd(const double *q, const double *k, const double *v, const double *dO, int B, int Hq,
               int Hkv, int L, int d, int causal, double *dq, double *dk, double *dv, double *lse,
               double *D, int n_threads) {
  if (bad_shape(B, Hq, Hkv, L, d)) return -1;
  problem_t P = make_problem(q, k, v, dO, B, Hq, Hkv, L, d, causal);
  task_t t; memset(&t, 0, sizeof t);
  t.P = &P; t.lse = lse; t.D = D; t.dq = dq; t.dk = dk; t.dv = dv;
  t.scratch_len = (size_t)L + d;
  t.n_items = (long)B * Hq * L; t.fn = stats_item; run_parallel(&t, n_threads);
  t.n_items = (long)B * Hq * L; t.fn = dq_full_item; run_parallel(&t, n_threads);
  t.n_items = (long)B * Hkv * L; t.fn = dkdv_full_item;
  return run_parallel(&t, n_threads);
}

/* Sampled backward: dq on query rows q_rows (same list for every (b, h)),
 * dk/dv on key rows k_rows (same list for every (b, g)).  The statistics
 * are computed for every query row that can see one of the sampled keys
 * (for causal: rows >= min(k_rows); otherwise all rows) and for q_rows.
 * Outputs: dq_rows [B][Hq][n_q][d], dk_rows/dv_rows [B][Hkv][n_k][d]. */
static void dq_rows_item(task_t *t, long item, double *s) {
  const problem_t *P = t->P;
  const int ri = (int)(item % t->n_rows);
  const long bh = item / t->n_rows;
  const int h = (int)(bh % P->Hq), b = (int)(bh / P->Hq);
  double lse, D;
  stats_row(P, b, h, t->rows[ri], s, &lse, &D);
  dq_row(P, b, h, t->rows[ri], lse, D, t->dq + ((size_t)bh * t->n_rows + ri) * P->d);
}
static void dkdv_rows_item(task_t *t, long item, double *s) {
  (void)s;
  const problem_t *P = t->P;
  const int ri = (int)(item % t->n_rows);
  const long bg = item / t->n_rows;
  const int g = (int)(bg % P->Hkv), b = (int)(bg / P->Hkv);
  const size_t r = (size_t)bg * t->n_rows + ri;
  dkdv_row(P, b, g, t->rows[ri], t->lse, t->D, t->dk + r * P->d, t->dv + r * P->d);
}

int oracle_bwd_rows(const double *q, const double *k, const double *v, const double *dO, int B, int Hq,
                    int Hkv, int L, int d, int causal, const int *q_rows, int n_q, const int *k_rows,
                    int n_k, double *dq_rows, double *dk_rows, double *dv_rows, int n_threads) {
  if (bad_shape(B, Hq, Hkv, L, d) || n_q < 0 || n_k < 0) return -1;
  for (int i = 0; i < n_q; ++i) if (q_rows[i] < 0 || q_rows[i] >= L) return -1;
  int kmin = L;
  for (int i = 0; i < n_k; ++i) {
    if (k_rows[i] < 0 || k_rows[i] >= L) return -1;
    if (k_rows[i] < kmin) kmin = k_rows[i];
  }
  problem_t P = make_problem(q, k, v, dO, B, Hq, Hkv, L, d, causal);
  task_t t; memset(&t, 0, sizeof t);
  t.P = &P; t.scratch_len = (size_t)L + d;
  int nt = 1;
  if (n_q > 0) {
    t.rows = q_rows; t.n_rows = n_q; t.dq = dq_rows;
    t.n_items = (long)B * Hq * n_q; t.fn = dq_rows_item;
    nt = run_parallel(&t, n_threads);
  }
  if (n_k > 0) {
    const size_t nrow = (size_t)B * Hq * L;
    double *lse = (double *)malloc(sizeof(double) * nrow);
    double *D = (double *)malloc(sizeof(double) * nrow);
    int *lo = (int *)malloc(sizeof(int) * (size_t)B * Hq);
    if (!lse || !D || !lo) { free(lse); free(D); free(lo); return -2; }
    for (size_t r = 0; r < nrow; ++r) { lse[r] = NAN; D[r] = NAN; }
    for (long bh = 0; bh < (long)B * Hq; ++bh) lo[bh] = causal ? kmin : 0;
    t.lse = lse; t.D = D; t.stat_lo = lo;
    t.n_items = (long)B * Hq * L; t.fn = stats_item; run_parallel(&t, n_threads);
    t.stat_lo = NULL;
    t.rows = k_rows; t.n_rows = n_k; t.dk = dk_rows; t.dv = dv_rows;
    t.n_items = (long)B * Hkv * n_k; t.fn = dkdv_rows_item;
    nt = run_parallel(&t, n_threads);
    free(lse); free(D); free(lo);
  }
  return nt;
}

/* --------------------------------------------------------------- ring form */

/* Ring schedules: which rows each rank owns, and which key/value chunk it
 * works on at each step.
 *   SCHED_FOLD     contiguous chunks (encoder) or, causal, the fold of the
 *                  USP section 8.2; N ring steps, step s pairs rank r with
 *                  the keys of rank (r - s) mod N.
 *   SCHED_STRIPED  rank r owns positions r, r+N, r+2N, ...; ring steps.
 *   SCHED_CONTIG   causal, contiguous chunks, ring steps: the unbalanced
 *                  ring of the DistFlashAttention section 7.2 (rank r has
 *                  work only at steps s <= r).
 *   SCHED_DFA      causal, contiguous chunks, DistFlashAttention's balanced
 *                  schedule (section 7.2: a worker that would wait takes
 *                  over work of a later worker): see dfa_pair. */
enum { SCHED_FOLD = 0, SCHED_STRIPED = 1, SCHED_CONTIG = 2, SCHED_DFA = 3 };

/* Rank that owns sequence position p under the schedule's chunk map. */
static int owner_rank(int L, int N, int causal, int schedule, int p) {
  if (schedule == SCHED_STRIPED) return p % N;
  if (!causal || schedule != SCHED_FOLD) return p / (L / N);
  const int sub = p / (L / (2 * N));
  return sub < N ? sub : 2 * N - 1 - sub;
}

/* Chunk map valid for this length: L % 2N == 0 for the fold, L % N == 0
 * otherwise; the contiguous causal schedules need causal. */
static int bad_chunking(int L, int n_chunks, int causal, int schedule) {
  if (n_chunks <= 0 || schedule < SCHED_FOLD || schedule > SCHED_DFA) return 1;
  if (schedule >= SCHED_CONTIG && !causal) return 1;
  return L % ((causal && schedule == SCHED_FOLD) ? 2 * n_chunks : n_chunks) != 0;
}

/* DistFlashAttention's balanced schedule for N workers (section 7.2).  In
 * the plain causal ring, worker w (query chunk w) has work at step s only if
 * s <= w (keys of chunk w - s); the others wait.  Here, at launch t = 0, 1,
 * ..., N/2 (rounded down), worker w >= t computes its own block (query chunk
 * w, keys of chunk w - t), and a worker w < t, which would wait, computes a
 * block of the step N - t instead: query chunk N - t + w against its own
 * keys, chunk w (the block worker N - t + w would meet at step N - t).  The
 * step N - t is then never run on its own.  When N is even the middle launch
 * t = N/2 has no such block (step N - t is that launch itself), and its
 * workers w < N/2 stay idle.  Returns 0 for an idle worker. */
static int dfa_pair(int N, int t, int w, int *q_chunk, int *kv_chunk) {
  if (w >= t) {
    *q_chunk = w;
    *kv_chunk = w - t;
    return 1;
  }
  if (t < N - t) {
    *q_chunk = N - t + w;
    *kv_chunk = w;
    return 1;
  }
  return 0;
}

/* Partial attention of query row i against the keys of rank src that i may
 * see.  Returns 0 if there is none; otherwise writes (o_s, lse_s). */
static int ring_block(const problem_t *P, int N, int b, int h, int i, int src, double *s, double *o_s,
                      double *lse_s, int schedule) {
  const int g = h / (P->Hq / P->Hkv);
  const double *qi = q_row(P, b, h, i);
  double m = -INFINITY;
  int cnt = 0;
  for (int j = 0; j < P->L; ++j) {
    s[j] = -INFINITY;
    if (owner_rank(P->L, N, P->causal, schedule, j) != src) continue;
    if (P->causal && j > i) continue;
    s[j] = P->scale * dot(qi, k_row(P, b, g, j), P->d);
    if (s[j] > m) m = s[j];
    ++cnt;
  }
  if (cnt == 0) return 0;
  double sum = 0.0;
  for (int j = 0; j < P->L; ++j) if (s[j] != -INFINITY) sum += exp(s[j] - m);
  *lse_s = m + log(sum);
  for (int c = 0; c < P->d; ++c) o_s[c] = 0.0;
  for (int j = 0; j < P->L; ++j) {
    if (s[j] == -INFINITY) continue;
    const double p = exp(s[j] - *lse_s);
    const double *vj = v_row(P, b, g, j);
    for (int c = 0; c < P->d; ++c) o_s[c] += p * vj[c];
  }
  return 1;
}

/* Merge the partial result of row i against the keys of rank src into the
 * running (o, lse) by the log-sum-exp rule; nothing if i sees none of them. */
static void ring_merge_block(const problem_t *P, int N, int b, int h, int i, int src, double *s, double *o_s,
                             int schedule, double *o, double *lse) {
  double lse_s;
  if (!ring_block(P, N, b, h, i, src, s, o_s, &lse_s, schedule)) return;
  const double hi = *lse > lse_s ? *lse : lse_s;
  const double merged = hi + log(exp(*lse - hi) + exp(lse_s - hi));
  const double a = exp(*lse - merged), w = exp(lse_s - merged);
  for (int c = 0; c < P->d; ++c) o[c] = a * o[c] + w * o_s[c];
  *lse = merged;
}

static void ring_item(task_t *t, long item, double *s) {
  const problem_t *P = t->P;
  const int N = t->n_chunks;
  const int i = (int)(item % P->L);
  const long bh = item / P->L;
  const int h = (int)(bh % P->Hq), b = (int)(bh / P->Hq);
  const int r = owner_rank(P->L, N, P->causal, t->schedule, i);
  double *o_s = s + P->L;
  double *o = t->o + ((size_t)bh * P->L + i) * P->d;
  double lse = -INFINITY;
  for (int c = 0; c < P->d; ++c) o[c] = 0.0;
  if (t->schedule == SCHED_DFA) {
    /* every block of each launch whose query chunk is r, in worker order */
    for (int launch = 0; launch <= N / 2; ++launch)
      for (int w = 0; w < N; ++w) {
        int qc, kc;
        if (dfa_pair(N, launch, w, &qc, &kc) && qc == r) ring_merge_block(P, N, b, h, i, kc, s, o_s, t->schedule, o, &lse);
      }
  } else {
    /* ring step s brings the keys of rank (r - s) mod N */
    for (int step = 0; step < N; ++step)
      ring_merge_block(P, N, b, h, i, ((r - step) % N + N) % N, s, o_s, t->schedule, o, &lse);
  }
  t->lse[(size_t)bh * P->L + i] = lse;
}

/* Ring form of the forward with n_chunks ranks.  Requires L % n_chunks == 0
 * (encoder) or L % (2 n_chunks) == 0 (causal, folded sub-chunks). */
int oracle_ring_fwd(const double *q, const double *k, const double *v, int B, int Hq, int Hkv, int L,
                    int d, int causal, int n_chunks, int schedule, double *o, double *lse, int n_threads) {
  if (bad_shape(B, Hq, Hkv, L, d) || bad_chunking(L, n_chunks, causal, schedule)) return -1;
  problem_t P = make_problem(q, k, v, NULL, B, Hq, Hkv, L, d, causal);
  task_t t; memset(&t, 0, sizeof t);
  t.P = &P; t.n_items = (long)B * Hq * L; t.fn = ring_item; t.scratch_len = (size_t)L + d;
  t.o = o; t.lse = lse; t.n_chunks = n_chunks; t.schedule = schedule;
  return run_parallel(&t, n_threads);
}

/* One ring step in isolation: rank `rank`'s query rows against the keys and
 * values rank `src` holds (at step s = (rank - src) mod N of its ring).  For
 * every row i owned by `rank`, (o_s, lse_s) of that block; a row that sees
 * none of src's keys (causal) gets lse_s = -inf and o_s = 0, the neutral
 * element of the merge.  Rows of other ranks are left untouched. */
static void step_item(task_t *t, long item, double *s) {
  const problem_t *P = t->P;
  const int i = (int)(item % P->L);
  const long bh = item / P->L;
  const int h = (int)(bh % P->Hq), b = (int)(bh / P->Hq);
  if (owner_rank(P->L, t->n_chunks, P->causal, t->schedule, i) != t->rank) return;
  double *o_s = t->o + ((size_t)bh * P->L + i) * P->d;
  double lse_s;
  if (!ring_block(P, t->n_chunks, b, h, i, t->src, s, o_s, &lse_s, t->schedule)) {
    for (int c = 0; c < P->d; ++c) o_s[c] = 0.0;
    lse_s = -INFINITY;
  }
  t->lse[(size_t)bh * P->L + i] = lse_s;
}

int oracle_ring_step(const double *q, const double *k, const double *v, int B, int Hq, int Hkv, int L, int d,
                     int causal, int n_chunks, int rank, int src, int schedule, double *o_s, double *lse_s,
                     int n_threads) {
  if (bad_shape(B, Hq, Hkv, L, d) || bad_chunking(L, n_chunks, causal, schedule)) return -1;
  if (rank < 0 || rank >= n_chunks || src < 0 || src >= n_chunks) return -1;
  problem_t P = make_problem(q, k, v, NULL, B, Hq, Hkv, L, d, causal);
  task_t t; memset(&t, 0, sizeof t);
  t.P = &P; t.n_items = (long)B * Hq * L; t.fn = step_item; t.scratch_len = (size_t)L;
  t.o = o_s; t.lse = lse_s; t.n_chunks = n_chunks; t.rank = rank; t.src = src; t.schedule = schedule;
  return run_parallel(&t, n_threads);
}

/* One ring block of the backward (Ring Attention, section 6.2: each block
 * is recomputed in the backward pass; the key/value gradients travel with
 * their block).  For the rows i of rank `rank` and the keys j of rank `src`
 * that i may see, with the full statistics lse_i and D_i of the plain
 * definition:
 *   P_ij = exp(s_ij - lse_i),  dS_ij = P_ij (dO_i . v_j - D_i)
 *   dq_i += scale sum_j dS_ij k_j                (rows of rank)
 *   dk_j += scale sum_{h in group} sum_i dS_ij q_i,
 *   dv_j +=       sum_{h in group} sum_i P_ij dO_i  (rows of src)
 * Outputs are in global row order (full [B][H][L][d] arrays), zero outside
 * those rows.  Summed over every (rank, src) block they give the plain
 * backward. */
static int block_visible(const problem_t *P, const task_t *t, int i, int j) {
  return owner_rank(P->L, t->n_chunks, P->causal, t->schedule, i) == t->rank &&
         owner_rank(P->L, t->n_chunks, P->causal, t->schedule, j) == t->src && (!P->causal || j <= i);
}
static void block_dq_item(task_t *t, long item, double *s) {
  (void)s;
  const problem_t *P = t->P;
  const int i = (int)(item % P->L);
  const long bh = item / P->L;
  const int h = (int)(bh % P->Hq), b = (int)(bh / P->Hq);
  const int g = h / (P->Hq / P->Hkv);
  double *dq = t->dq + ((size_t)bh * P->L + i) * P->d;
  for (int c = 0; c < P->d; ++c) dq[c] = 0.0;
  if (owner_rank(P->L, t->n_chunks, P->causal, t->schedule, i) != t->rank) return;
  const double *qi = q_row(P, b, h, i), *doi = do_row(P, b, h, i);
  const double lse = t->lse[(size_t)bh * P->L + i], D = t->D[(size_t)bh * P->L + i];
  for (int j = 0; j < P->L; ++j) {
    if (!block_visible(P, t, i, j)) continue;
    const double pij = exp(P->scale * dot(qi, k_row(P, b, g, j), P->d) - lse);
    const double dsij = pij * (dot(doi, v_row(P, b, g, j), P->d) - D);
    const double *kj = k_row(P, b, g, j);
    for (int c = 0; c < P->d; ++c) dq[c] += P->scale * dsij * kj[c];
  }
}
static void block_dkdv_item(task_t *t, long item, double *s) {
  (void)s;
  const problem_t *P = t->P;
  const int j = (int)(item % P->L);
  const long bg = item / P->L;
  const int g = (int)(bg % P->Hkv), b = (int)(bg / P->Hkv);
  const int G = P->Hq / P->Hkv;
  double *dk = t->dk + ((size_t)bg * P->L + j) * P->d, *dv = t->dv + ((size_t)bg * P->L + j) * P->d;
  for (int c = 0; c < P->d; ++c) { dk[c] = 0.0; dv[c] = 0.0; }
  if (owner_rank(P->L, t->n_chunks, P->causal, t->schedule, j) != t->src) return;
  const double *kj = k_row(P, b, g, j), *vj = v_row(P, b, g, j);
  for (int h = g * G; h < (g + 1) * G; ++h) {
    const size_t base = ((size_t)b * P->Hq + h) * P->L;
    for (int i = 0; i < P->L; ++i) {
      if (!block_visible(P, t, i, j)) continue;
      const double *qi = q_row(P, b, h, i), *doi = do_row(P, b, h, i);
      const double pij = exp(P->scale * dot(qi, kj, P->d) - t->lse[base + i]);
      const double dsij = pij * (dot(doi, vj, P->d) - t->D[base + i]);
      for (int c = 0; c < P->d; ++c) {
        dv[c] += pij * doi[c];
        dk[c] += P->scale * dsij * qi[c];
      }
    }
  }
}

int oracle_ring_step_bwd(const double *q, const double *k, const double *v, const double *dO, const double *lse,
                         const double *D, int B, int Hq, int Hkv, int L, int d, int causal, int n_chunks, int rank,
                         int src, int schedule, double *dq, double *dk, double *dv, int n_threads) {
  if (bad_shape(B, Hq, Hkv, L, d) || bad_chunking(L, n_chunks, causal, schedule)) return -1;
  if (rank < 0 || rank >= n_chunks || src < 0 || src >= n_chunks) return -1;
  problem_t P = make_problem(q, k, v, dO, B, Hq, Hkv, L, d, causal);
  task_t t; memset(&t, 0, sizeof t);
  t.P = &P; t.n_chunks = n_chunks; t.rank = rank; t.src = src; t.schedule = schedule;
  t.lse = (double *)lse; t.D = (double *)D; t.dq = dq; t.dk = dk; t.dv = dv;
  t.n_items = (long)B * Hq * L; t.fn = block_dq_item; run_parallel(&t, n_threads);
  t.n_items = (long)B * Hkv * L; t.fn = block_dkdv_item;
  return run_parallel(&t, n_threads);
}

/* The merge of two partial results of the same query rows (the log-sum-exp
 * rule above), written out on its own: for each of n_rows rows of width d,
 *   lse = log(exp(lse_a) + exp(lse_b)),
 *   o   = exp(lse_a - lse) o_a + exp(lse_b - lse) o_b,
 * into (o_a, lse_a).  A side with lse = -inf contributes nothing (both
 * -inf: (o_a, lse_a) stay as they are). */
void oracle_merge(double *o_a, double *lse_a, const double *o_b, const double *lse_b, long n_rows, int d) {
  for (long r = 0; r < n_rows; ++r) {
    double *oa = o_a + (size_t)r * d;
    const double *ob = o_b + (size_t)r * d;
    const double la = lse_a[r], lb = lse_b[r];
    if (lb == -INFINITY) continue;
    if (la == -INFINITY) {
      for (int c = 0; c < d; ++c) oa[c] = ob[c];
      lse_a[r] = lb;
      continue;
    }
    const double hi = la > lb ? la : lb;
    const double merged = hi + log(exp(la - hi) + exp(lb - hi));
    const double wa = exp(la - merged), wb = exp(lb - merged);
    for (int c = 0; c < d; ++c) oa[c] = wa * oa[c] + wb * ob[c];
    lse_a[r] = merged;
  }
}

/* ------------------------------------------------------ blockwise FFN */

/* The standard normal CDF, Phi(x) = (1 + erf(x / sqrt 2)) / 2, written with
 * erfc so that the tail x << 0 keeps its relative accuracy (1 + erf cancels
 * to exactly 0 below x = -8.3 in double precision). */
static double normal_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

/* GELU in its exact form, x * Phi(x) with the standard normal CDF Phi. */
static double gelu(double x) { return x * normal_cdf(x); }

/* The feed-forward block the BPT section of the pages fuses after attention
 * for each query block ("Large-scale distributed AI model training series:
 * sequence parallelism", section 4.2: for the current query block, attention,
 * then the FFN and the residual connection), with the two linear layers and
 * the 4x up-projection of the GPT-style FFN the pages assume (section 8):
 *   y_m = x_m + W2^T gelu(W1^T x_m + b1) + b2
 * for rows m of x [M][D]; W1 [D][F], W2 [F][D], b1 [F], b2 [D].  Rows are
 * independent, so the blockwise order changes nothing: plain row loop. */
typedef struct { const double *x, *w1, *b1, *w2, *b2; double *y, *h_out; int D, F; } ffn_t;

/* One row.  Each sum runs in ascending order of its index (k for the first
 * layer, j for the second) starting from the bias; the loops walk the
 * weights row by row so that they stream through memory. */
static void ffn_row(const ffn_t *f, long m, double *h, double *acc) {
  const double *x = f->x + (size_t)m * f->D;
  for (int j = 0; j < f->F; ++j) h[j] = f->b1[j];
  for (int k = 0; k < f->D; ++k) {
    const double *w = f->w1 + (size_t)k * f->F;
    for (int j = 0; j < f->F; ++j) h[j] += x[k] * w[j];
  }
  for (int j = 0; j < f->F; ++j) h[j] = gelu(h[j]);
  if (f->h_out) memcpy(f->h_out + (size_t)m * f->F, h, sizeof(double) * (size_t)f->F);
  for (int c = 0; c < f->D; ++c) acc[c] = f->b2[c];
  for (int j = 0; j < f->F; ++j) {
    const double *w = f->w2 + (size_t)j * f->D;
    for (int c = 0; c < f->D; ++c) acc[c] += h[j] * w[c];
  }
  double *y = f->y + (size_t)m * f->D;
  for (int c = 0; c < f->D; ++c) y[c] = x[c] + acc[c];
}

typedef struct { const ffn_t *f; long n, next; } ffn_task_t;

static void *ffn_worker(void *arg) {
  ffn_task_t *t = (ffn_task_t *)arg;
  double *h = (double *)malloc(sizeof(double) * ((size_t)t->f->F + (size_t)t->f->D));
  for (;;) {
    long i = __atomic_fetch_add(&t->next, 1, __ATOMIC_RELAXED);
    if (i >= t->n) break;
    ffn_row(t->f, i, h, h + t->f->F);
  }
  free(h);
  return NULL;
}

/* y [M][D] and, if h_out is not NULL, the hidden activation
 * gelu(W1^T x_m + b1) of every row into h_out [M][F]. */
int oracle_ffn(const double *x, const double *w1, const double *b1, const double *w2, const double *b2, long M,
               int D, int F, double *y, double *h_out, int n_threads) {
  if (M < 0 || D <= 0 || F <= 0) return -1;
  ffn_t f = {x, w1, b1, w2, b2, y, h_out, D, F};
  ffn_task_t t = {&f, M, 0};
  if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, ffn_worker, &t);
  for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  return n_threads;
}

/* ------------------------------------------------ blockwise FFN backward */

/* Derivative of the exact GELU: d/dx [x Phi(x)] = Phi(x) + x phi(x). */
static double gelu_grad(double x) {
  const double Phi = normal_cdf(x);
  const double phi = exp(-0.5 * x * x) / sqrt(2.0 * acos(-1.0));  /* standard normal density */
  return Phi + x * phi;
}

/* Gradients of the loss sum(dy * y) for the FFN block above, by the chain
 * rule, with a and h recomputed from x (the BPT section's recomputation of
 * the block's activations in the backward pass):
 *   dh_f  = sum_d dy_d W2[f][d]
 *   da_f  = dh_f gelu'(a_f)
 *   dx_d  = dy_d + sum_f da_f W1[d][f]
 *   dW2[f][d] = sum_m h_mf dy_md     db2_d = sum_m dy_md
 *   dW1[d][f] = sum_m x_md da_mf     db1_f = sum_m da_mf
 * Sums over rows run in ascending row order. */
typedef struct {
  const double *x, *w1, *b1, *w2, *dy;
  double *dx, *h, *da, *dw1, *db1, *dw2, *db2;
  long M;
  int D, F;
} ffn_bwd_t;

typedef struct { const ffn_bwd_t *f; int phase; long n, next; } ffn_bwd_task_t;

static void ffn_bwd_row(const ffn_bwd_t *f, long m) {
  const double *x = f->x + (size_t)m * f->D, *dy = f->dy + (size_t)m * f->D;
  double *h = f->h + (size_t)m * f->F, *da = f->da + (size_t)m * f->F;
  /* a (kept in da until it is replaced), then h */
  for (int j = 0; j < f->F; ++j) da[j] = f->b1[j];
  for (int k = 0; k < f->D; ++k) {
    const double *w = f->w1 + (size_t)k * f->F;
    for (int j = 0; j < f->F; ++j) da[j] += x[k] * w[j];
  }
  for (int j = 0; j < f->F; ++j) {
    const double a = da[j];
    h[j] = gelu(a);
    double dh = 0.0;
    const double *w = f->w2 + (size_t)j * f->D;
    for (int c = 0; c < f->D; ++c) dh += dy[c] * w[c];
    da[j] = dh * gelu_grad(a);
  }
  double *dx = f->dx + (size_t)m * f->D;
  for (int c = 0; c < f->D; ++c) dx[c] = dy[c];
  for (int j = 0; j < f->F; ++j) {
    const double *w = f->w1;
    for (int c = 0; c < f->D; ++c) dx[c] += da[j] * w[(size_t)c * f->F + j];
  }
}

/* weight and bias gradients of hidden unit j (row j of dW2, column j of dW1) */
static void ffn_bwd_unit(const ffn_bwd_t *f, long j) {
  double *dw2 = f->dw2 + (size_t)j * f->D;
  for (int c = 0; c < f->D; ++c) dw2[c] = 0.0;
  double db1 = 0.0;
  for (int c = 0; c < f->D; ++c) f->dw1[(size_t)c * f->F + j] = 0.0;
  for (long m = 0; m < f->M; ++m) {
    const double hm = f->h[(size_t)m * f->F + j], dam = f->da[(size_t)m * f->F + j];
    const double *dy = f->dy + (size_t)m * f->D, *x = f->x + (size_t)m * f->D;
    for (int c = 0; c < f->D; ++c) dw2[c] += hm * dy[c];
    for (int c = 0; c < f->D; ++c) f->dw1[(size_t)c * f->F + j] += x[c] * dam;
    db1 += dam;
  }
  f->db1[j] = db1;
}

static void *ffn_bwd_worker(void *arg) {
  ffn_bwd_task_t *t = (ffn_bwd_task_t *)arg;
  for (;;) {
    long i = __atomic_fetch_add(&t->next, 1, __ATOMIC_RELAXED);
    if (i >= t->n) break;
    if (t->phase == 0)
      ffn_bwd_row(t->f, i);
    else
      ffn_bwd_unit(t->f, i);
  }
  return NULL;
}

/* x [M][D], W1 [D][F], b1 [F], W2 [F][D], dy [M][D] -> dx [M][D],
 * dW1 [D][F], db1 [F], dW2 [F][D], db2 [D] (b2 does not enter); h_out and
 * da_out [M][F], if not NULL, receive h and da. */
int oracle_ffn_bwd(const double *x, const double *w1, const double *b1, const double *w2, const double *dy, long M,
                   int D, int F, double *dx, double *dw1, double *db1, double *dw2, double *db2, double *h_out,
                   double *da_out, int n_threads) {
  if (M < 0 || D <= 0 || F <= 0) return -1;
  double *h = h_out ? h_out : (double *)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1) * F);
  double *da = da_out ? da_out : (double *)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1) * F);
  if (!h || !da) {
    if (!h_out) free(h);
    if (!da_out) free(da);
    return -2;
  }
  ffn_bwd_t f = {x, w1, b1, w2, dy, dx, h, da, dw1, db1, dw2, db2, M, D, F};
  if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  for (int phase = 0; phase < 2; ++phase) {
    ffn_bwd_task_t t = {&f, phase, phase == 0 ? M : (long)F, 0};
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, ffn_bwd_worker, &t);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  }
  for (int c = 0; c < D; ++c) {
    double s = 0.0;
    for (long m = 0; m < M; ++m) s += dy[(size_t)m * D + c];
    db2[c] = s;
  }
  if (!h_out) free(h);
  if (!da_out) free(da);
  return n_threads;
}

int oracle_owner_rank(int L, int n_chunks, int causal, int schedule, int p) {
  if (p < 0 || p >= L || bad_chunking(L, n_chunks, causal, schedule)) return -1;
  return owner_rank(L, n_chunks, causal, schedule, p);
}
