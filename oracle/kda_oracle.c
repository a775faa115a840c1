/*
 * kda_oracle.c -- plain, slow, fp64 CPU oracle for the Kimi Delta Attention
 * (KDA) forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness yardstick for the
 * CUDA path in chunked_gated_delta_11_gb300/.  Only tests/, the smoke() check
 * in __graft_entry__.py and the cpu_baseline / reference legs of bench.py may
 * load it.  It shares no code, header, table or helper with the CUDA path, and
 * the CUDA path never calls it.
 *
 * Sources (cited by page title and section):
 *   [DW]  "You Could Have Come Up with Kimi Delta Attention" (Doubleword blog)
 *         sec. 4 (boxed KDA recurrence), sec. 6.1-6.5 (chunkwise form),
 *         sec. 2.1 (read-back and locality), sec. 3 (Gated DeltaNet).
 *   [FK]  "FlashKDA Delta Attention Algorithm" (instagit explainer), "Core
 *         Architecture": sigmoid gates, L2 norm of q and k, decay
 *         A = exp(g_c * lower_bound).
 *   [API] FlashKDA repository summary, "flash_kda.fwd API reference":
 *         [T_total, H, D] packing, cu_seqlens, state layout [N, H, V, K].
 *
 * Everything is double precision.  No blocking, fusion or reordering beyond
 * what the cited definitions state.  Readings where the pages are silent:
 *   - L2 norm: x / sqrt(sum x^2 + eps), eps passed in (1e-6 by default); the
 *     pages give no epsilon.
 *   - log alpha = lower_bound * sigmoid(g_raw) per key channel; beta =
 *     sigmoid(beta_raw) per token and head.
 *   - state S is V x K (maps keys to values); final_state[n][h][v][k] = S[v][k].
 *
 * Parity pins for every exported function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Input transforms ([FK] "Core Architecture"; [DW] sec. 4 uses unit keys).  */
/* ------------------------------------------------------------------------ */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* q_hat, k_hat: per (token, head) L2-normalised rows of length K.
 * log_alpha[t][h][d] = lower_bound * sigmoid(g_raw[t][h][d]).
 * beta[t][h] = sigmoid(beta_raw[t][h]).  Any output pointer may be NULL. */
void kda_oracle_prepare(const double *q_raw, const double *k_raw,
                        const double *g_raw, const double *beta_raw,
                        int64_t T, int H, int K, double lower_bound, double eps,
                        double *q_hat, double *k_hat, double *log_alpha,
                        double *beta) {
  for (int64_t t = 0; t < T; ++t) {
    for (int h = 0; h < H; ++h) {
      const int64_t row = (t * H + h) * (int64_t)K;
      if (q_hat) {
        double ss = 0.0;
        for (int d = 0; d < K; ++d) ss += q_raw[row + d] * q_raw[row + d];
        const double inv = 1.0 / sqrt(ss + eps);
        for (int d = 0; d < K; ++d) q_hat[row + d] = q_raw[row + d] * inv;
      }
      if (k_hat) {
        double ss = 0.0;
        for (int d = 0; d < K; ++d) ss += k_raw[row + d] * k_raw[row + d];
        const double inv = 1.0 / sqrt(ss + eps);
        for (int d = 0; d < K; ++d) k_hat[row + d] = k_raw[row + d] * inv;
      }
      if (log_alpha)
        for (int d = 0; d < K; ++d)
          log_alpha[row + d] = lower_bound * sigmoid(g_raw[row + d]);
      if (beta) beta[t * H + h] = sigmoid(beta_raw[t * H + h]);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Sequence boundaries ([API]: cu_seqlens, or N equal sequences).           */
/* ------------------------------------------------------------------------ */

static void seq_bounds(const int32_t *cu_seqlens, int64_t T_total, int N, int n,
                       int64_t *bos, int64_t *eos) {
  if (cu_seqlens) {
    *bos = cu_seqlens[n];
    *eos = cu_seqlens[n + 1];
  } else {
    const int64_t L = T_total / N;
    *bos = (int64_t)n * L;
    *eos = *bos + L;
  }
}

/* ------------------------------------------------------------------------ */
/* Token-by-token recurrence: the boxed KDA update of [DW] sec. 4.          */
/*   forget  S~ = S Diag(alpha_t)          (column d scaled by alpha_t[d])   */
/*   predict vhat = S~ k_t                                                    */
/*   correct e = beta_t (v_t - vhat)                                          */
/*   write   S = S~ + e k_t^T                                                 */
/*   read    o_t = S (scale q_t)                                              */
/* ------------------------------------------------------------------------ */

typedef struct {
  const double *q, *k, *v, *la, *beta, *init;
  const int32_t *cu;
  int64_t T_total;
  int H, N, K, V, chunk;
  double scale;
  double *out, *final_state;
} fwd_args;

static void recur_unit(const fwd_args *a, int n, int h, double *S,
                       double *work) {
  const int H = a->H, K = a->K, V = a->V;
  int64_t bos, eos;
  seq_bounds(a->cu, a->T_total, a->N, n, &bos, &eos);
  double *pred = work;     /* V */
  double *e = work + V;    /* V */
  double *alpha = work + 2 * V;  /* K */
  for (int64_t t = bos; t < eos; ++t) {
    const double *qt = a->q + (t * H + h) * (int64_t)K;
    const double *kt = a->k + (t * H + h) * (int64_t)K;
    const double *vt = a->v + (t * H + h) * (int64_t)V;
    const double *lat = a->la + (t * H + h) * (int64_t)K;
    const double bt = a->beta[t * H + h];
    /* forget: every key channel (column) d decays by alpha_t[d] */
    for (int d = 0; d < K; ++d) alpha[d] = exp(lat[d]);
    for (int vi = 0; vi < V; ++vi)
      for (int d = 0; d < K; ++d) S[vi * K + d] *= alpha[d];
    /* predict */
    for (int vi = 0; vi < V; ++vi) {
      double acc = 0.0;
      for (int d = 0; d < K; ++d) acc += S[vi * K + d] * kt[d];
      pred[vi] = acc;
    }
    /* correct */
    for (int vi = 0; vi < V; ++vi) e[vi] = bt * (vt[vi] - pred[vi]);
    /* write */
    for (int vi = 0; vi < V; ++vi)
      for (int d = 0; d < K; ++d) S[vi * K + d] += e[vi] * kt[d];
    /* read (after the write: o_t sees its own token) */
    double *ot = a->out + (t * H + h) * (int64_t)V;
    for (int vi = 0; vi < V; ++vi) {
      double acc = 0.0;
      for (int d = 0; d < K; ++d) acc += S[vi * K + d] * (a->scale * qt[d]);
      ot[vi] = acc;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Chunkwise form of the same recurrence, [DW] sec. 6.1-6.5, chunk size C.  */
/* Decay products D_{j+1:i} are formed from differences of per-chunk prefix */
/* sums of log alpha ([DW] sec. 6.6: "differences between two prefix sums"),*/
/* never as products of exp(+G) and exp(-G), so any lower_bound is valid.   */
/* ------------------------------------------------------------------------ */

static void chunk_unit(const fwd_args *a, int n, int h, double *S,
                       double *work) {
  const int H = a->H, K = a->K, V = a->V, C = a->chunk;
  int64_t bos, eos;
  seq_bounds(a->cu, a->T_total, a->N, n, &bos, &eos);
  double *G = work;                     /* C x K  prefix sums of log alpha */
  double *ebar = G + (int64_t)C * K;    /* C x V  provisional errors        */
  double *e = ebar + (int64_t)C * V;    /* C x V  corrected errors          */
  double *rho = e + (int64_t)C * V;     /* C x C                            */
  double *chi = rho + (int64_t)C * C;   /* C x C                            */
  double *o = chi + (int64_t)C * C;     /* C x V                            */
  for (int64_t c0 = bos; c0 < eos; c0 += C) {
    const int nc = (int)((eos - c0) < C ? (eos - c0) : C);
#define Q(i) (a->q + ((c0 + (i)) * H + h) * (int64_t)K)
#define KK(i) (a->k + ((c0 + (i)) * H + h) * (int64_t)K)
#define VV(i) (a->v + ((c0 + (i)) * H + h) * (int64_t)V)
#define LA(i) (a->la + ((c0 + (i)) * H + h) * (int64_t)K)
#define BETA(i) (a->beta[(c0 + (i)) * H + h])
    /* sec. 6.1: G_i = log of D_{0:i} = sum_{m<=i} log alpha_m */
    for (int i = 0; i < nc; ++i)
      for (int d = 0; d < K; ++d)
        G[i * K + d] = (i ? G[(i - 1) * K + d] : 0.0) + LA(i)[d];
    /* sec. 6.2: provisional errors ebar_i = beta_i (v_i - S_c D_{0:i} k_i) */
    for (int i = 0; i < nc; ++i)
      for (int vi = 0; vi < V; ++vi) {
        double acc = 0.0;
        for (int d = 0; d < K; ++d)
          acc += S[vi * K + d] * exp(G[i * K + d]) * KK(i)[d];
        ebar[i * V + vi] = BETA(i) * (VV(i)[vi] - acc);
      }
    /* sec. 6.3: rho_ij = beta_i <k_j| D_{j+1:i} |k_i>, j < i */
    for (int i = 0; i < nc; ++i)
      for (int j = 0; j < nc; ++j) {
        double acc = 0.0;
        if (j < i)
          for (int d = 0; d < K; ++d)
            acc += KK(j)[d] * exp(G[i * K + d] - G[j * K + d]) * KK(i)[d];
        rho[i * C + j] = (j < i) ? BETA(i) * acc : 0.0;
      }
    /* sec. 6.3: causal triangular solve e_i = ebar_i - sum_{j<i} rho_ij e_j */
    for (int i = 0; i < nc; ++i)
      for (int vi = 0; vi < V; ++vi) {
        double acc = ebar[i * V + vi];
        for (int j = 0; j < i; ++j) acc -= rho[i * C + j] * e[j * V + vi];
        e[i * V + vi] = acc;
      }
    /* sec. 6.5: chi_ij = s <k_j| D_{j+1:i} |q_i>, j <= i (diagonal kept) */
    for (int i = 0; i < nc; ++i)
      for (int j = 0; j < nc; ++j) {
        double acc = 0.0;
        if (j <= i)
          for (int d = 0; d < K; ++d)
            acc += KK(j)[d] * exp(G[i * K + d] - G[j * K + d]) * Q(i)[d];
        chi[i * C + j] = (j <= i) ? a->scale * acc : 0.0;
      }
    /* sec. 6.5: o_i = s S_c D_{0:i} q_i + sum_{j<=i} chi_ij e_j (old S_c) */
    for (int i = 0; i < nc; ++i)
      for (int vi = 0; vi < V; ++vi) {
        double acc = 0.0;
        for (int d = 0; d < K; ++d)
          acc += S[vi * K + d] * exp(G[i * K + d]) * Q(i)[d];
        acc *= a->scale;
        for (int j = 0; j <= i; ++j) acc += chi[i * C + j] * e[j * V + vi];
        o[i * V + vi] = acc;
      }
    /* sec. 6.4: S_{c+1} = S_c D_{0:C-1} + sum_j e_j (k_j D_{j+1:C-1})^T */
    const int L = nc - 1;
    for (int vi = 0; vi < V; ++vi)
      for (int d = 0; d < K; ++d) {
        double acc = S[vi * K + d] * exp(G[L * K + d]);
        for (int j = 0; j < nc; ++j)
          acc += e[j * V + vi] * KK(j)[d] * exp(G[L * K + d] - G[j * K + d]);
        S[vi * K + d] = acc;
      }
    for (int i = 0; i < nc; ++i)
      memcpy(a->out + ((c0 + i) * H + h) * (int64_t)V, o + (int64_t)i * V,
             sizeof(double) * V);
#undef Q
#undef KK
#undef VV
#undef LA
#undef BETA
  }
}

/* ------------------------------------------------------------------------ */
/* Thread pool over independent (sequence, head) units.                     */
/* ------------------------------------------------------------------------ */

typedef struct {
  const fwd_args *a;
  int tid, nthreads;
  int rc;
} worker_arg;

static void *worker(void *p) {
  worker_arg *w = (worker_arg *)p;
  const fwd_args *a = w->a;
  const int K = a->K, V = a->V, C = a->chunk > 0 ? a->chunk : 1;
  const size_t wsz = (size_t)C * K + 3 * (size_t)C * V + 2 * (size_t)C * C +
                     2 * (size_t)V + (size_t)K;
  double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
  double *work = (double *)malloc(sizeof(double) * wsz);
  if (!S || !work) {
    free(S);
    free(work);
    w->rc = -1;
    return NULL;
  }
  const int units = a->N * a->H;
  for (int u = w->tid; u < units; u += w->nthreads) {
    const int n = u / a->H, h = u % a->H;
    if (a->init)
      memcpy(S, a->init + (int64_t)u * V * K, sizeof(double) * (size_t)V * K);
    else
      memset(S, 0, sizeof(double) * (size_t)V * K);
    if (a->chunk > 0)
      chunk_unit(a, n, h, S, work);
    else
      recur_unit(a, n, h, S, work);
    if (a->final_state)
      memcpy(a->final_state + (int64_t)u * V * K, S,
             sizeof(double) * (size_t)V * K);
  }
  free(S);
  free(work);
  w->rc = 0;
  return NULL;
}

/* Forward pass over already-transformed inputs.
 *   q, k       [T_total, H, K]  (normalised by the caller, see prepare)
 *   v          [T_total, H, V]
 *   log_alpha  [T_total, H, K]  natural-log retention, <= 0
 *   beta       [T_total, H]
 *   init_state [N, H, V, K] or NULL (zeros)
 *   cu_seqlens [N + 1] or NULL (N equal sequences of T_total / N)
 *   chunk      0 = token-by-token ([DW] sec. 4); C > 0 = chunkwise ([DW] sec. 6)
 *   out        [T_total, H, V];  final_state [N, H, V, K] or NULL
 * Returns 0, or -1 on a bad argument or allocation failure. */
int kda_oracle_fwd(const double *q, const double *k, const double *v,
                   const double *log_alpha, const double *beta,
                   const double *init_state, const int32_t *cu_seqlens,
                   int64_t T_total, int H, int N, int K, int V, double scale,
                   int chunk, int nthreads, double *out, double *final_state) {
  if (H <= 0 || N <= 0 || K <= 0 || V <= 0 || T_total < 0 || chunk < 0)
    return -1;
  if (!cu_seqlens && (T_total % N) != 0) return -1;
  if (nthreads <= 0) nthreads = 1;
  fwd_args a = {q, k, v, log_alpha, beta, init_state, cu_seqlens, T_total,
                H, N, K, V, chunk, scale, out, final_state};
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  worker_arg *wa = (worker_arg *)calloc((size_t)nthreads, sizeof(worker_arg));
  if (!th || !wa) {
    free(th);
    free(wa);
    return -1;
  }
  int rc = 0, started = 0;
  for (int i = 0; i < nthreads; ++i) {
    wa[i].a = &a;
    wa[i].tid = i;
    wa[i].nthreads = nthreads;
    wa[i].rc = -1;
    if (pthread_create(&th[i], NULL, worker, &wa[i]) != 0) {
      rc = -1;
      break;
    }
    ++started;
  }
  for (int i = 0; i < started; ++i) {
    pthread_join(th[i], NULL);
    if (wa[i].rc != 0) rc = -1;
  }
  free(th);
  free(wa);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Per-chunk factors of the chunkwise form ([DW] sec. 6.1-6.6), used to     */
/* check a chunk kernel's intermediates.  For chunk c of head h, with       */
/* G_i = sum_{m<=i} log alpha_m (natural log) and n_c tokens:               */
/*   Akk  = (I + R)^-1, R_ij = rho_ij (sec. 6.3), by forward substitution   */
/*   Aqk  = chi (sec. 6.5), lower triangle including the diagonal           */
/*   Qdec_i = s q_i * exp(G_i)            (query decayed to the boundary)   */
/*   Kdec_i = k_i * exp(G_i)                                                */
/*   Kend_j = k_j * exp(G_last - G_j)     (K^end of sec. 6.4)               */
/*   W = Akk diag(beta) Kdec,  U = Akk diag(beta) V   (WY factors: the      */
/*        corrected errors of sec. 6.3 are E^T = U - W S_c^T)               */
/*   dlast = exp(G_last)                  (diagonal of D_{0:C-1})           */
/* Rows past n_c are zero.  Chunks are numbered sequence by sequence, each  */
/* sequence restarting at its first token; record index = chunk * H + h.   */
/* Array shapes per record: Akk, Aqk C x C; W, Qdec, Kend C x K; U C x V;   */
/* dlast K.  Returns the number of chunks, or -1 on a bad argument.        */
/* ------------------------------------------------------------------------ */

int64_t kda_oracle_num_chunks(const int32_t *cu_seqlens, int64_t T_total, int N,
                              int C) {
  if (N <= 0 || C <= 0 || T_total < 0) return -1;
  if (!cu_seqlens && (T_total % N) != 0) return -1;
  int64_t total = 0;
  for (int n = 0; n < N; ++n) {
    int64_t bos, eos;
    seq_bounds(cu_seqlens, T_total, N, n, &bos, &eos);
    total += (eos - bos + C - 1) / C;
  }
  return total;
}

int64_t kda_oracle_chunk_factors(const double *q, const double *k,
                                 const double *v, const double *log_alpha,
                                 const double *beta, const int32_t *cu_seqlens,
                                 int64_t T_total, int H, int N, int K, int V,
                                 double scale, int C, double *Akk, double *Aqk,
                                 double *W, double *U, double *Qdec,
                                 double *Kend, double *dlast) {
  const int64_t nchunks = kda_oracle_num_chunks(cu_seqlens, T_total, N, C);
  if (nchunks < 0 || H <= 0 || K <= 0 || V <= 0) return -1;
  double *G = (double *)malloc(sizeof(double) * (size_t)C * K);
  double *R = (double *)malloc(sizeof(double) * (size_t)C * C);
  double *A = (double *)malloc(sizeof(double) * (size_t)C * C);
  double *Kdec = (double *)malloc(sizeof(double) * (size_t)C * K);
  if (!G || !R || !A || !Kdec) {
    free(G); free(R); free(A); free(Kdec);
    return -1;
  }
  int64_t chunk = 0;
  for (int n = 0; n < N; ++n) {
    int64_t bos, eos;
    seq_bounds(cu_seqlens, T_total, N, n, &bos, &eos);
    for (int64_t c0 = bos; c0 < eos; c0 += C, ++chunk) {
      const int nc = (int)((eos - c0) < C ? (eos - c0) : C);
      for (int h = 0; h < H; ++h) {
        const int64_t rec = chunk * H + h;
        double *akk = Akk + rec * C * C, *aqk = Aqk + rec * C * C;
        double *w = W + rec * C * K, *u = U + rec * C * V;
        double *qd = Qdec + rec * C * K, *ke = Kend + rec * C * K;
        double *dl = dlast + rec * K;
        memset(akk, 0, sizeof(double) * (size_t)C * C);
        memset(aqk, 0, sizeof(double) * (size_t)C * C);
        memset(w, 0, sizeof(double) * (size_t)C * K);
        memset(u, 0, sizeof(double) * (size_t)C * V);
        memset(qd, 0, sizeof(double) * (size_t)C * K);
        memset(ke, 0, sizeof(double) * (size_t)C * K);
#define Q(i) (q + ((c0 + (i)) * H + h) * (int64_t)K)
#define KK(i) (k + ((c0 + (i)) * H + h) * (int64_t)K)
#define VV(i) (v + ((c0 + (i)) * H + h) * (int64_t)V)
#define LA(i) (log_alpha + ((c0 + (i)) * H + h) * (int64_t)K)
#define BETA(i) (beta[(c0 + (i)) * H + h])
        for (int i = 0; i < nc; ++i)
          for (int d = 0; d < K; ++d)
            G[i * K + d] = (i ? G[(i - 1) * K + d] : 0.0) + LA(i)[d];
        const int L = nc - 1;
        for (int d = 0; d < K; ++d) dl[d] = exp(G[L * K + d]);
        for (int i = 0; i < nc; ++i)
          for (int d = 0; d < K; ++d) {
            qd[i * K + d] = scale * Q(i)[d] * exp(G[i * K + d]);
            Kdec[i * K + d] = KK(i)[d] * exp(G[i * K + d]);
            ke[i * K + d] = KK(i)[d] * exp(G[L * K + d] - G[i * K + d]);
          }
        /* R (strictly lower) and chi (lower incl. diagonal) */
        for (int i = 0; i < C; ++i)
          for (int j = 0; j < C; ++j) R[i * C + j] = 0.0;
        for (int i = 0; i < nc; ++i)
          for (int j = 0; j <= i; ++j) {
            double rk = 0.0, rq = 0.0;
            for (int d = 0; d < K; ++d) {
              const double dec = exp(G[i * K + d] - G[j * K + d]);
              rk += KK(j)[d] * dec * KK(i)[d];
              rq += KK(j)[d] * dec * Q(i)[d];
            }
            if (j < i) R[i * C + j] = BETA(i) * rk;
            aqk[i * C + j] = scale * rq;
          }
        /* (I + R)^-1 by forward substitution: rows of A satisfy
           A_i = e_i - sum_{j<i} R_ij A_j (unit lower triangular system) */
        for (int i = 0; i < C; ++i)
          for (int m = 0; m < C; ++m) {
            double acc = (i == m) ? 1.0 : 0.0;
            for (int j = 0; j < i; ++j) acc -= R[i * C + j] * A[j * C + m];
            A[i * C + m] = acc;
          }
        for (int i = 0; i < nc; ++i)
          for (int m = 0; m < nc; ++m) akk[i * C + m] = A[i * C + m];
        /* WY factors */
        for (int i = 0; i < nc; ++i) {
          for (int d = 0; d < K; ++d) {
            double acc = 0.0;
            for (int j = 0; j <= i; ++j)
              acc += A[i * C + j] * BETA(j) * Kdec[j * K + d];
            w[i * K + d] = acc;
          }
          for (int vi = 0; vi < V; ++vi) {
            double acc = 0.0;
            for (int j = 0; j <= i; ++j)
              acc += A[i * C + j] * BETA(j) * VV(j)[vi];
            u[i * V + vi] = acc;
          }
        }
#undef Q
#undef KK
#undef VV
#undef LA
#undef BETA
      }
    }
  }
  free(G); free(R); free(A); free(Kdec);
  return nchunks;
}

/* ------------------------------------------------------------------------ */
/* Three ways to invert a unit lower-triangular I + R (R strictly lower,    */
/* n x n, row-major), used to pin one another ([DW] sec. 6.3; the Neumann   */
/* series is exact because R is nilpotent: R^n = 0).                        */
/* ------------------------------------------------------------------------ */

static void matmul_sq(const double *A, const double *B, double *Cm, int n) {
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      double acc = 0.0;
      for (int m = 0; m < n; ++m) acc += A[i * n + m] * B[m * n + j];
      Cm[i * n + j] = acc;
    }
}

/* sum_{m=0}^{n-1} (-R)^m, term by term. */
int kda_oracle_neumann_inverse(const double *R, int n, double *out) {
  if (n <= 0) return -1;
  double *term = (double *)malloc(sizeof(double) * (size_t)n * n);
  double *tmp = (double *)malloc(sizeof(double) * (size_t)n * n);
  if (!term || !tmp) { free(term); free(tmp); return -1; }
  for (int i = 0; i < n * n; ++i) term[i] = (i / n == i % n) ? 1.0 : 0.0;
  memcpy(out, term, sizeof(double) * (size_t)n * n);
  for (int p = 1; p < n; ++p) {
    matmul_sq(term, R, tmp, n);
    for (int i = 0; i < n * n; ++i) {
      term[i] = -tmp[i];
      out[i] += term[i];
    }
  }
  free(term); free(tmp);
  return 0;
}

/* (I - R)(I + R^2)(I + R^4)...(I + R^(2^(m-1))) with 2^m >= n: the same
 * finite series grouped by powers of two. */
int kda_oracle_product_inverse(const double *R, int n, double *out) {
  if (n <= 0) return -1;
  double *P = (double *)malloc(sizeof(double) * (size_t)n * n);
  double *F = (double *)malloc(sizeof(double) * (size_t)n * n);
  double *T = (double *)malloc(sizeof(double) * (size_t)n * n);
  if (!P || !F || !T) { free(P); free(F); free(T); return -1; }
  for (int i = 0; i < n * n; ++i) {
    const double I = (i / n == i % n) ? 1.0 : 0.0;
    out[i] = I - R[i];       /* running product, starts at I - R */
    P[i] = R[i];             /* current power R^(2^p)            */
  }
  for (int span = 2; span < n; span *= 2) {
    matmul_sq(P, P, T, n);   /* P becomes R^span */
    memcpy(P, T, sizeof(double) * (size_t)n * n);
    for (int i = 0; i < n * n; ++i) F[i] = ((i / n == i % n) ? 1.0 : 0.0) + P[i];
    matmul_sq(out, F, T, n);
    memcpy(out, T, sizeof(double) * (size_t)n * n);
  }
  free(P); free(F); free(T);
  return 0;
}

/* Forward substitution on (I + R) X = I. */
int kda_oracle_trisolve_inverse(const double *R, int n, double *out) {
  if (n <= 0) return -1;
  for (int i = 0; i < n; ++i)
    for (int m = 0; m < n; ++m) {
      double acc = (i == m) ? 1.0 : 0.0;
      for (int j = 0; j < i; ++j) acc -= R[i * n + j] * out[j * n + m];
      out[i * n + m] = acc;
    }
  return 0;
}
