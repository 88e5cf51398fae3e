/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the causal linear-attention
 * recurrence.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may call it; the product path never does.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (web pages; cited by title and section/equation):
 *   [NB]  "History Replays Itself: Unleashing Long-Context Capability in
 *         Linear Attention" (NoteBank full text), Sec. 2, Eq. (1):
 *             S_t = S_{t-1} A_t + beta_t v_t k_t^T ,   o_t = S_t q_t ,
 *         S_t in R^{d_v x d_k}; A_t = I, beta_t = 1 is additive linear
 *         attention; input scaling is absorbed, output gates and
 *         normalisation are omitted.
 *   [NB-C6] same page, App. C.6, Eq. (11): the recurrent cost
 *         J(7 d_k d_v + d_k + 2 d_v) counts one state decay, the key and
 *         query readouts, one rank-one update and vector scalings -- the
 *         structure of the gated delta rule
 *             A_t = alpha_t (I - beta_t k_t k_t^T)
 *         used by the Gated DeltaNet backbone that the page wraps.
 *   [NB-G] same page, Sec. 2: besides the delta rule it names the "gated"
 *         family, whose retention is a scalar decay of the whole state:
 *             A_t = alpha_t I   (alpha = beta = 1: additive linear attention)
 *   [BN]  "BASED：简单线性注意力如何平衡召回能力与生成吞吐" (reading notes of
 *         "Simple linear attention language models balance the
 *         recall-throughput tradeoff"), Sec. 2.2 (the paper's Eqs. (1)-(3)):
 *             y_i = s_i^T phi(q_i) / z_i^T phi(q_i),
 *             s_i = s_{i-1} + phi(k_i) v_i^T,  z_i = z_{i-1} + phi(k_i),
 *             s_0 = 0, z_0 = 0;
 *         Sec. 2.3 (the paper's Eq. (4)): the 2nd-order Taylor map
 *             phi(x) = [1, x, vec(x x^T)/sqrt(2)],  D = 1 + d' + d'^2.
 *   [BN-D] same page, the paragraph on decay after Table 7: the 10B-token
 *         runs use a fixed decay rate per head (the 30B/50B runs none).
 *
 * Readings taken where the pages leave a step open:
 *   - o_t / y_i are read AFTER token t's write (inclusive prefix, Eq. (1)
 *     writes S_t then reads S_t q_t; BN sums over j <= i).
 *   - vec(x x^T) is row-major: feature index 1 + d' + a*d' + b holds
 *     x_a x_b / sqrt(2).  The Taylor state s is stored D x d_v.
 *   - No 1/sqrt(d_k) on q (input scaling absorbed); a q_scale factor is
 *     exposed and defaults to 1 at every call site.
 *   - The Taylor denominator gets + eps (0 by default); the pages state it
 *     is positive for a non-empty prefix and that implementations add eps.
 *   - The initial state is zero unless one is passed in.
 *   - [BN-D] gives no formula for the per-head decay; the plain reading is
 *     a constant scalar retention of the whole state before each write,
 *         s_i = lambda_h s_{i-1} + phi(k_i) v_i^T,
 *         z_i = lambda_h z_{i-1} + phi(k_i),
 *     the A_t = lambda I member of the [NB-G] family; lambda = 1 (the
 *     default) is the undecayed recurrence above.
 *
 * Everything is computed token by token in double precision, exactly as
 * the definitions above read; the only parallelism is over independent
 * (batch, head) pairs, one pthread per slice of pairs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_IN_F32 0
#define ORACLE_IN_BF16 1

/* Read element i of an input array given as float32 or as raw bf16 bits
 * (bf16 is the upper half of an IEEE float32). */
static double in_at(int kind, const void* base, int64_t i) {
  if (kind == ORACLE_IN_F32) return (double)((const float*)base)[i];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

int64_t oracle_taylor_dim(int64_t dfeat) { return 1 + dfeat + dfeat * dfeat; }

/* phi(x) = [1, x, vec(x x^T)/sqrt(2)]   ([BN] Sec. 2.3, paper Eq. (4)). */
void oracle_taylor_feature(const double* x, int64_t dfeat, double* phi) {
  const double inv_sqrt2 = 1.0 / sqrt(2.0);
  phi[0] = 1.0;
  for (int64_t a = 0; a < dfeat; ++a) phi[1 + a] = x[a];
  for (int64_t a = 0; a < dfeat; ++a)
    for (int64_t b = 0; b < dfeat; ++b)
      phi[1 + dfeat + a * dfeat + b] = x[a] * x[b] * inv_sqrt2;
}

/* ------------------------------------------------------------------------ */
/* Worker plumbing: each worker takes (b,h) pairs w, w+nthreads, ...          */

typedef struct {
  int64_t B, H, N, dk, dv;
  int in_kind;
  const void *q, *k, *v;
  const float *alpha, *beta;
  double q_scale, eps;
  const double *s_in, *z_in;
  const double* decay; /* Taylor: per-head lambda [H], or NULL (no decay) */
  const int64_t* t_samples;
  int64_t n_samples;
  double *out, *den, *s_out, *z_out;
  int worker, nthreads;
} job_t;

static int64_t n_out_rows(const job_t* j) {
  return j->t_samples ? j->n_samples : j->N;
}

/* ---------------------------------------------------------------------- */
/* Taylor / BASED recurrence with normaliser ([BN] Sec. 2.2).              */

static void* taylor_worker(void* arg) {
  const job_t* j = (const job_t*)arg;
  const int64_t df = j->dk, dv = j->dv, N = j->N;
  const int64_t D = oracle_taylor_dim(df);
  double* s = (double*)malloc(sizeof(double) * D * dv);
  double* z = (double*)malloc(sizeof(double) * D);
  double* xk = (double*)malloc(sizeof(double) * df);
  double* xq = (double*)malloc(sizeof(double) * df);
  double* phk = (double*)malloc(sizeof(double) * D);
  double* phq = (double*)malloc(sizeof(double) * D);
  double* vt = (double*)malloc(sizeof(double) * dv);
  const int64_t rows = n_out_rows(j);
  for (int64_t bh = j->worker; bh < j->B * j->H; bh += j->nthreads) {
    /* s_0, z_0: given state or zero; lambda: this head's decay ([BN-D]). */
    const double lam = j->decay ? j->decay[bh % j->H] : 1.0;
    for (int64_t i = 0; i < D * dv; ++i) s[i] = j->s_in ? j->s_in[bh * D * dv + i] : 0.0;
    for (int64_t i = 0; i < D; ++i) z[i] = j->z_in ? j->z_in[bh * D + i] : 0.0;
    int64_t next = 0; /* next sample slot */
    for (int64_t t = 0; t < N; ++t) {
      const int64_t qk_off = (bh * N + t) * df, v_off = (bh * N + t) * dv;
      for (int64_t a = 0; a < df; ++a) {
        xk[a] = in_at(j->in_kind, j->k, qk_off + a);
        xq[a] = in_at(j->in_kind, j->q, qk_off + a);
      }
      for (int64_t c = 0; c < dv; ++c) vt[c] = in_at(j->in_kind, j->v, v_off + c);
      /* s_t = lambda s_{t-1} + phi(k_t) v_t^T ;  z_t = lambda z_{t-1} + phi(k_t) */
      oracle_taylor_feature(xk, df, phk);
      for (int64_t r = 0; r < D; ++r) {
        for (int64_t c = 0; c < dv; ++c) s[r * dv + c] = lam * s[r * dv + c] + phk[r] * vt[c];
        z[r] = lam * z[r] + phk[r];
      }
      int record = j->t_samples ? (next < j->n_samples && j->t_samples[next] == t) : 1;
      if (!record) continue;
      /* y_t = s_t^T phi(q_t) / (z_t^T phi(q_t) + eps) */
      oracle_taylor_feature(xq, df, phq);
      double dn = 0.0;
      for (int64_t r = 0; r < D; ++r) dn += z[r] * phq[r];
      const int64_t slot = j->t_samples ? next : t;
      double* y = j->out + (bh * rows + slot) * dv;
      for (int64_t c = 0; c < dv; ++c) {
        double nm = 0.0;
        for (int64_t r = 0; r < D; ++r) nm += s[r * dv + c] * phq[r];
        y[c] = nm / (dn + j->eps);
      }
      if (j->den) j->den[bh * rows + slot] = dn;
      if (j->t_samples) ++next;
    }
    if (j->s_out) memcpy(j->s_out + bh * D * dv, s, sizeof(double) * D * dv);
    if (j->z_out) memcpy(j->z_out + bh * D, z, sizeof(double) * D);
  }
  free(s); free(z); free(xk); free(xq); free(phk); free(phq); free(vt);
  return NULL;
}

/* ---------------------------------------------------------------------- */
/* Gated delta rule ([NB] Sec. 2 Eq. (1), A_t = alpha_t (I - beta_t k k^T)) */

static void* gdn_worker(void* arg) {
  const job_t* j = (const job_t*)arg;
  const int64_t dk = j->dk, dv = j->dv, N = j->N;
  double* S = (double*)malloc(sizeof(double) * dv * dk);
  double* Sk = (double*)malloc(sizeof(double) * dv);
  double* kt = (double*)malloc(sizeof(double) * dk);
  double* qt = (double*)malloc(sizeof(double) * dk);
  double* vt = (double*)malloc(sizeof(double) * dv);
  const int64_t rows = n_out_rows(j);
  for (int64_t bh = j->worker; bh < j->B * j->H; bh += j->nthreads) {
    for (int64_t i = 0; i < dv * dk; ++i) S[i] = j->s_in ? j->s_in[bh * dv * dk + i] : 0.0;
    int64_t next = 0;
    for (int64_t t = 0; t < N; ++t) {
      const int64_t qk_off = (bh * N + t) * dk, v_off = (bh * N + t) * dv;
      for (int64_t a = 0; a < dk; ++a) {
        kt[a] = in_at(j->in_kind, j->k, qk_off + a);
        qt[a] = j->q_scale * in_at(j->in_kind, j->q, qk_off + a);
      }
      for (int64_t c = 0; c < dv; ++c) vt[c] = in_at(j->in_kind, j->v, v_off + c);
      const double al = (double)j->alpha[bh * N + t];
      const double be = (double)j->beta[bh * N + t];
      /* S_{t-1} A_t = alpha (S_{t-1} - beta (S_{t-1} k) k^T) */
      for (int64_t i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int64_t a = 0; a < dk; ++a) acc += S[i * dk + a] * kt[a];
        Sk[i] = acc;
      }
      for (int64_t i = 0; i < dv; ++i)
        for (int64_t a = 0; a < dk; ++a)
          S[i * dk + a] = al * (S[i * dk + a] - be * Sk[i] * kt[a]) + be * vt[i] * kt[a];
      int record = j->t_samples ? (next < j->n_samples && j->t_samples[next] == t) : 1;
      if (!record) continue;
      /* o_t = S_t q_t */
      const int64_t slot = j->t_samples ? next : t;
      double* o = j->out + (bh * rows + slot) * dv;
      for (int64_t i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int64_t a = 0; a < dk; ++a) acc += S[i * dk + a] * qt[a];
        o[i] = acc;
      }
      if (j->t_samples) ++next;
    }
    if (j->s_out) memcpy(j->s_out + bh * dv * dk, S, sizeof(double) * dv * dk);
  }
  free(S); free(Sk); free(kt); free(qt); free(vt);
  return NULL;
}

/* ---------------------------------------------------------------------- */
/* Scalar gate ([NB-G]: Eq. (1) with A_t = alpha_t I)                      */

static void* gated_worker(void* arg) {
  const job_t* j = (const job_t*)arg;
  const int64_t dk = j->dk, dv = j->dv, N = j->N;
  double* S = (double*)malloc(sizeof(double) * dv * dk);
  double* kt = (double*)malloc(sizeof(double) * dk);
  double* qt = (double*)malloc(sizeof(double) * dk);
  double* vt = (double*)malloc(sizeof(double) * dv);
  const int64_t rows = n_out_rows(j);
  for (int64_t bh = j->worker; bh < j->B * j->H; bh += j->nthreads) {
    for (int64_t i = 0; i < dv * dk; ++i) S[i] = j->s_in ? j->s_in[bh * dv * dk + i] : 0.0;
    int64_t next = 0;
    for (int64_t t = 0; t < N; ++t) {
      const int64_t qk_off = (bh * N + t) * dk, v_off = (bh * N + t) * dv;
      for (int64_t a = 0; a < dk; ++a) {
        kt[a] = in_at(j->in_kind, j->k, qk_off + a);
        qt[a] = j->q_scale * in_at(j->in_kind, j->q, qk_off + a);
      }
      for (int64_t c = 0; c < dv; ++c) vt[c] = in_at(j->in_kind, j->v, v_off + c);
      const double al = (double)j->alpha[bh * N + t];
      const double be = (double)j->beta[bh * N + t];
      /* S_t = S_{t-1} (alpha I) + beta v k^T */
      for (int64_t i = 0; i < dv; ++i)
        for (int64_t a = 0; a < dk; ++a) S[i * dk + a] = al * S[i * dk + a] + be * vt[i] * kt[a];
      int record = j->t_samples ? (next < j->n_samples && j->t_samples[next] == t) : 1;
      if (!record) continue;
      /* o_t = S_t q_t */
      const int64_t slot = j->t_samples ? next : t;
      double* o = j->out + (bh * rows + slot) * dv;
      for (int64_t i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int64_t a = 0; a < dk; ++a) acc += S[i * dk + a] * qt[a];
        o[i] = acc;
      }
      if (j->t_samples) ++next;
    }
    if (j->s_out) memcpy(j->s_out + bh * dv * dk, S, sizeof(double) * dv * dk);
  }
  free(S); free(kt); free(qt); free(vt);
  return NULL;
}

static int run_jobs(const job_t* proto, void* (*fn)(void*), int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > proto->B * proto->H) nthreads = (int)(proto->B * proto->H);
  if (nthreads < 1) nthreads = 1;
  job_t* jobs = (job_t*)malloc(sizeof(job_t) * nthreads);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
  int rc = 0;
  for (int w = 0; w < nthreads; ++w) {
    jobs[w] = *proto;
    jobs[w].worker = w;
    jobs[w].nthreads = nthreads;
  }
  int started = 0;
  for (int w = 1; w < nthreads; ++w) {
    if (pthread_create(&th[w], NULL, fn, &jobs[w]) != 0) { rc = -2; break; }
    started = w;
  }
  if (rc == 0) fn(&jobs[0]);
  for (int w = 1; w <= started; ++w) pthread_join(th[w], NULL);
  free(jobs);
  free(th);
  return rc;
}

static int check_samples(const int64_t* t, int64_t n, int64_t N) {
  for (int64_t i = 0; i < n; ++i) {
    if (t[i] < 0 || t[i] >= N) return -1;
    if (i > 0 && t[i] <= t[i - 1]) return -1;
  }
  return 0;
}

/* Taylor linear attention, token by token.
 * q, k: [B,H,N,dfeat]; v: [B,H,N,dv]; contiguous; float32 or bf16 bits.
 * s_in/z_in: [B,H,D,dv] / [B,H,D] or NULL (zero state).
 * decay: per-head lambda [H] or NULL (no decay).
 * t_samples: NULL (every token) or n_samples strictly increasing indices.
 * y: [B,H,rows,dv]; den (nullable): [B,H,rows] = z_t^T phi(q_t) (no eps);
 * s_out/z_out: final state (nullable).  Returns 0, or -1 on bad arguments. */
int oracle_taylor(int64_t B, int64_t H, int64_t N, int64_t dfeat, int64_t dv,
                  int in_kind, const void* q, const void* k, const void* v,
                  const double* s_in, const double* z_in, double eps, const double* decay,
                  const int64_t* t_samples, int64_t n_samples,
                  double* y, double* den, double* s_out, double* z_out,
                  int nthreads) {
  if (B < 0 || H < 0 || N < 0 || dfeat < 1 || dv < 1) return -1;
  if (in_kind != ORACLE_IN_F32 && in_kind != ORACLE_IN_BF16) return -1;
  if (t_samples && check_samples(t_samples, n_samples, N)) return -1;
  job_t j;
  memset(&j, 0, sizeof j);
  j.B = B; j.H = H; j.N = N; j.dk = dfeat; j.dv = dv; j.in_kind = in_kind;
  j.q = q; j.k = k; j.v = v; j.eps = eps; j.s_in = s_in; j.z_in = z_in; j.decay = decay;
  j.t_samples = t_samples; j.n_samples = n_samples;
  j.out = y; j.den = den; j.s_out = s_out; j.z_out = z_out;
  if (B * H == 0) return 0;
  return run_jobs(&j, taylor_worker, nthreads);
}

/* Gated delta rule, token by token.
 * q, k: [B,H,N,dk]; v: [B,H,N,dv]; alpha, beta: [B,H,N] float32.
 * S_in: [B,H,dv,dk] or NULL (zero).  o: [B,H,rows,dv]; S_out nullable. */
int oracle_gdn(int64_t B, int64_t H, int64_t N, int64_t dk, int64_t dv,
               int in_kind, const void* q, const void* k, const void* v,
               const float* alpha, const float* beta, double q_scale,
               const double* S_in, const int64_t* t_samples, int64_t n_samples,
               double* o, double* S_out, int nthreads) {
  if (B < 0 || H < 0 || N < 0 || dk < 1 || dv < 1) return -1;
  if (in_kind != ORACLE_IN_F32 && in_kind != ORACLE_IN_BF16) return -1;
  if (t_samples && check_samples(t_samples, n_samples, N)) return -1;
  job_t j;
  memset(&j, 0, sizeof j);
  j.B = B; j.H = H; j.N = N; j.dk = dk; j.dv = dv; j.in_kind = in_kind;
  j.q = q; j.k = k; j.v = v; j.alpha = alpha; j.beta = beta;
  j.q_scale = q_scale; j.s_in = S_in;
  j.t_samples = t_samples; j.n_samples = n_samples;
  j.out = o; j.s_out = S_out;
  if (B * H == 0) return 0;
  return run_jobs(&j, gdn_worker, nthreads);
}

/* Scalar gate, token by token; arguments as oracle_gdn. */
int oracle_gated(int64_t B, int64_t H, int64_t N, int64_t dk, int64_t dv,
                 int in_kind, const void* q, const void* k, const void* v,
                 const float* alpha, const float* beta, double q_scale,
                 const double* S_in, const int64_t* t_samples, int64_t n_samples,
                 double* o, double* S_out, int nthreads) {
  if (B < 0 || H < 0 || N < 0 || dk < 1 || dv < 1) return -1;
  if (in_kind != ORACLE_IN_F32 && in_kind != ORACLE_IN_BF16) return -1;
  if (t_samples && check_samples(t_samples, n_samples, N)) return -1;
  job_t j;
  memset(&j, 0, sizeof j);
  j.B = B; j.H = H; j.N = N; j.dk = dk; j.dv = dv; j.in_kind = in_kind;
  j.q = q; j.k = k; j.v = v; j.alpha = alpha; j.beta = beta;
  j.q_scale = q_scale; j.s_in = S_in;
  j.t_samples = t_samples; j.n_samples = n_samples;
  j.out = o; j.s_out = S_out;
  if (B * H == 0) return 0;
  return run_jobs(&j, gated_worker, nthreads);
}
