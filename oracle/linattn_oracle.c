/*
 * Plain fp64 CPU oracle for kernelized linear attention with phi(x) = elu(x) + 1.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's compute path may link,
 * load or call this file; only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Everything here is the plain token-by-token definition, written out with no
 * blocking, chunking or reordering:
 *
 *   phi(x)  = x + 1      for x > 0
 *           = exp(x)     for x <= 0          (elu with alpha = 1, plus 1)
 *     -- "Linear Attention Mechanisms" (dileepadev.github.io), section
 *        "Choosing the Feature Map", ELU-based features; and
 *        "Attention-Free / Sub-Quadratic Architectures", "Feature maps".
 *
 *   causal, for each head: S_0 = 0 (D x Dv), z_0 = 0 (D), and for i = 0..N-1
 *     S_i = gamma * S_{i-1} + phi(k_i) v_i^T
 *     z_i = gamma * z_{i-1} + phi(k_i)
 *     o_i = (phi(q_i)^T S_i) / (phi(q_i) . z_i + eps)
 *     -- "Linear Attention Mechanisms" (dileepadev.github.io), section
 *        "Recurrent Reformulation" (the rank-1 state update, the normaliser
 *        update and the read-out, in that order); decay gamma from the same
 *        page's "Gating and Selective State Updates" (RetNet, gamma^(t-j)) and
 *        from "Attention-Free / Sub-Quadratic Architectures", "Evolution: add
 *        decay/gating" (S_i = gamma S_{i-1} + phi(k_i) v_i^T), applied to z as
 *        well; eps added to the denominator as in the NumPy listing of
 *        "Linear Attention Mechanisms" (sadullah.online), "The linear
 *        attention trick".
 *
 *   non-causal: S = sum_j phi(k_j) v_j^T, z = sum_j phi(k_j) over all j, then
 *     o_i = phi(q_i)^T S / (phi(q_i) . z + eps)
 *     -- "Linear Attention Mechanisms" (dileepadev.github.io), "The Kernel
 *        Trick for Attention" (S and z computed once, reused for every
 *        query); "Attention-Free / Sub-Quadratic Architectures", "Linear
 *        Attention (the core trick)".
 *
 *   decode step: one iteration of the causal loop on a caller-held (S, z):
 *     update first, then read out.
 *
 *   gated: the causal loop with a data-dependent gate in place of gamma,
 *     S_i = G_i (.) S_{i-1} + phi(k_i) v_i^T, G_i = a_i 1^T (a gate a_i[d] in
 *     [0, 1] per step and key feature, the same for every value column), and
 *     z_i[d] = a_i[d] z_{i-1}[d] + phi(k_i)[d]; the same read-out.
 *     -- "Linear Attention Mechanisms" (dileepadev.github.io), "Gating and
 *        Selective State Updates", Gated Linear Attention (G_t applied
 *        elementwise to the state; G_t = 1 is plain linear attention,
 *        G_t = 0 overwrites the state); "Attention-Free / Sub-Quadratic
 *        Architectures", "Evolution: add decay/gating".
 *
 * Inputs are fp32 arrays (bf16 inputs are widened exactly by the caller);
 * all arithmetic and all outputs are fp64.  Layouts: q, k [U][N][D],
 * v [U][N][Dv], o [U][N][Dv], S [U][D][Dv], z [U][D], gamma [U], gates
 * a [U][N][D], where U is
 * the number of independent (batch, head) units.  Units are spread over
 * POSIX threads; each unit is computed by one thread in the order above, so
 * results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

double oracle_phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* ------------------------------------------------------------------------ */
/* One unit of the causal recurrence.  S, z are the running state (in/out). */
static void causal_unit(const float *q, const float *k, const float *v,
                        double gamma, double eps, int64_t N, int D, int Dv,
                        double *S, double *z, double *o, double *fq,
                        double *fk) {
  for (int64_t i = 0; i < N; ++i) {
    const float *ki = k + i * D, *vi = v + i * Dv;
    for (int d = 0; d < D; ++d) fk[d] = oracle_phi((double)ki[d]);
    /* S_i = gamma S_{i-1} + phi(k_i) v_i^T ;  z_i = gamma z_{i-1} + phi(k_i) */
    for (int d = 0; d < D; ++d) {
      double *Sd = S + (int64_t)d * Dv;
      for (int e = 0; e < Dv; ++e) Sd[e] = gamma * Sd[e] + fk[d] * (double)vi[e];
      z[d] = gamma * z[d] + fk[d];
    }
    if (o) {
      /* o_i = phi(q_i)^T S_i / (phi(q_i) . z_i + eps) */
      const float *qi = q + i * D;
      for (int d = 0; d < D; ++d) fq[d] = oracle_phi((double)qi[d]);
      double den = 0.0;
      for (int d = 0; d < D; ++d) den += fq[d] * z[d];
      den += eps;
      double *oi = o + i * Dv;
      for (int e = 0; e < Dv; ++e) {
        double num = 0.0;
        for (int d = 0; d < D; ++d) num += fq[d] * S[(int64_t)d * Dv + e];
        oi[e] = num / den;
      }
    }
  }
}

/* One unit of the gated recurrence: a [N][D] gates, S, z running state. */
static void gated_unit(const float *q, const float *k, const float *v,
                       const float *a, double eps, int64_t N, int D, int Dv,
                       double *S, double *z, double *o, double *fq,
                       double *fk) {
  for (int64_t i = 0; i < N; ++i) {
    const float *ki = k + i * D, *vi = v + i * Dv, *ai = a + i * D;
    for (int d = 0; d < D; ++d) fk[d] = oracle_phi((double)ki[d]);
    /* S_i[d][:] = a_i[d] S_{i-1}[d][:] + phi(k_i)[d] v_i^T ;
       z_i[d] = a_i[d] z_{i-1}[d] + phi(k_i)[d] */
    for (int d = 0; d < D; ++d) {
      const double g = (double)ai[d];
      double *Sd = S + (int64_t)d * Dv;
      for (int e = 0; e < Dv; ++e) Sd[e] = g * Sd[e] + fk[d] * (double)vi[e];
      z[d] = g * z[d] + fk[d];
    }
    if (o) {
      const float *qi = q + i * D;
      for (int d = 0; d < D; ++d) fq[d] = oracle_phi((double)qi[d]);
      double den = 0.0;
      for (int d = 0; d < D; ++d) den += fq[d] * z[d];
      den += eps;
      double *oi = o + i * Dv;
      for (int e = 0; e < Dv; ++e) {
        double num = 0.0;
        for (int d = 0; d < D; ++d) num += fq[d] * S[(int64_t)d * Dv + e];
        oi[e] = num / den;
      }
    }
  }
}

/* One unit of the non-causal form. */
static void noncausal_unit(const float *q, const float *k, const float *v,
                           double eps, int64_t N, int D, int Dv, double *S,
                           double *z, double *o, double *fq, double *fk) {
  memset(S, 0, sizeof(double) * (size_t)D * Dv);
  memset(z, 0, sizeof(double) * (size_t)D);
  /* S = sum_j phi(k_j) v_j^T ;  z = sum_j phi(k_j) */
  for (int64_t j = 0; j < N; ++j) {
    const float *kj = k + j * D, *vj = v + j * Dv;
    for (int d = 0; d < D; ++d) fk[d] = oracle_phi((double)kj[d]);
    for (int d = 0; d < D; ++d) {
      double *Sd = S + (int64_t)d * Dv;
      for (int e = 0; e < Dv; ++e) Sd[e] += fk[d] * (double)vj[e];
      z[d] += fk[d];
    }
  }
  if (!o) return;
  /* o_i = phi(q_i)^T S / (phi(q_i) . z + eps), the same S and z for every i */
  for (int64_t i = 0; i < N; ++i) {
    const float *qi = q + i * D;
    for (int d = 0; d < D; ++d) fq[d] = oracle_phi((double)qi[d]);
    double den = 0.0;
    for (int d = 0; d < D; ++d) den += fq[d] * z[d];
    den += eps;
    double *oi = o + i * Dv;
    for (int e = 0; e < Dv; ++e) {
      double num = 0.0;
      for (int d = 0; d < D; ++d) num += fq[d] * S[(int64_t)d * Dv + e];
      oi[e] = num / den;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Thread pool over units.                                                  */
enum { MODE_CAUSAL = 0, MODE_NONCAUSAL = 1, MODE_DECODE = 2, MODE_GATED = 3 };

typedef struct {
  int mode, tid, nthreads, D, Dv;
  int64_t U, N;
  const float *q, *k, *v;
  const float *a; /* gated: [U][N][D] */
  const double *gamma;
  double eps;
  double *o, *S, *z; /* S, z: per-unit state out (or in/out for decode) */
  int have_state_in; /* causal: start from S, z instead of zero */
} job_t;

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int D = J->D, Dv = J->Dv;
  double *fq = (double *)malloc(sizeof(double) * (size_t)D);
  double *fk = (double *)malloc(sizeof(double) * (size_t)D);
  double *Sloc = NULL, *zloc = NULL;
  if (!J->S) Sloc = (double *)malloc(sizeof(double) * (size_t)D * Dv);
  if (!J->z) zloc = (double *)malloc(sizeof(double) * (size_t)D);
  for (int64_t u = J->tid; u < J->U; u += J->nthreads) {
    double *S = J->S ? J->S + u * (int64_t)D * Dv : Sloc;
    double *z = J->z ? J->z + u * (int64_t)D : zloc;
    const int64_t N = J->N;
    const double g = J->gamma ? J->gamma[u] : 1.0;
    if (J->mode == MODE_CAUSAL) {
      if (!J->have_state_in) {
        memset(S, 0, sizeof(double) * (size_t)D * Dv);
        memset(z, 0, sizeof(double) * (size_t)D);
      }
      causal_unit(J->q ? J->q + u * N * D : NULL, J->k + u * N * D,
                  J->v + u * N * Dv, g,
                  J->eps, N, D, Dv, S, z, J->o ? J->o + u * N * Dv : NULL, fq,
                  fk);
    } else if (J->mode == MODE_GATED) {
      memset(S, 0, sizeof(double) * (size_t)D * Dv);
      memset(z, 0, sizeof(double) * (size_t)D);
      gated_unit(J->q ? J->q + u * N * D : NULL, J->k + u * N * D, J->v + u * N * Dv,
                 J->a + u * N * D, J->eps, N, D, Dv, S, z,
                 J->o ? J->o + u * N * Dv : NULL, fq, fk);
    } else if (J->mode == MODE_NONCAUSAL) {
      noncausal_unit(J->q ? J->q + u * N * D : NULL, J->k + u * N * D,
                     J->v + u * N * Dv, J->eps, N, D, Dv, S, z,
                     J->o ? J->o + u * N * Dv : NULL, fq, fk);
    } else { /* decode: one causal step on the given state */
      causal_unit(J->q + u * D, J->k + u * D, J->v + u * Dv, g, J->eps, 1, D,
                  Dv, S, z, J->o + u * Dv, fq, fk);
    }
  }
  free(fq);
  free(fk);
  free(Sloc);
  free(zloc);
  return NULL;
}

static int run_jobs(job_t proto, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > proto.U) nthreads = proto.U > 0 ? (int)proto.U : 1;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)nthreads);
  int started = 0, rc = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].tid = t;
    jobs[t].nthreads = nthreads;
    if (t == nthreads - 1) {
      worker(&jobs[t]);
    } else if (pthread_create(&th[t], NULL, worker, &jobs[t]) == 0) {
      ++started;
    } else {
      rc = -1;
      break;
    }
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Exported entry points.  Return 0 on success, -1 on a bad argument.       */

/* Causal form.  o [U][N][Dv] may be NULL (state only, i.e. prefill).
 * S_state [U][D][Dv] and z_state [U][D] may be NULL; when given they receive
 * the state after token N-1.  If state_in is nonzero they also provide the
 * starting state (continuing a sequence). */
int oracle_causal(const float *q, const float *k, const float *v,
                  const double *gamma, double eps, int64_t U, int64_t N, int D,
                  int Dv, double *o, double *S_state, double *z_state,
                  int state_in, int nthreads) {
  if (U < 0 || N < 0 || D <= 0 || Dv <= 0 || !k || !v || (o && !q)) return -1;
  if (state_in && (!S_state || !z_state)) return -1;
  job_t J;
  memset(&J, 0, sizeof J);
  J.mode = MODE_CAUSAL;
  J.U = U; J.N = N; J.D = D; J.Dv = Dv;
  J.q = q; J.k = k; J.v = v; J.gamma = gamma; J.eps = eps;
  J.o = o; J.S = S_state; J.z = z_state; J.have_state_in = state_in;
  return run_jobs(J, nthreads);
}

/* Non-causal form.  o may be NULL (then q may be NULL); S_state, z_state may
 * be NULL. */
int oracle_noncausal(const float *q, const float *k, const float *v,
                     double eps, int64_t U, int64_t N, int D, int Dv,
                     double *o, double *S_state, double *z_state,
                     int nthreads) {
  if (U < 0 || N < 0 || D <= 0 || Dv <= 0 || !k || !v || (o && !q)) return -1;
  job_t J;
  memset(&J, 0, sizeof J);
  J.mode = MODE_NONCAUSAL;
  J.U = U; J.N = N; J.D = D; J.Dv = Dv;
  J.q = q; J.k = k; J.v = v; J.eps = eps;
  J.o = o; J.S = S_state; J.z = z_state;
  return run_jobs(J, nthreads);
}

/* One decode step on U units: q, k [U][D], v [U][Dv]; S [U][D][Dv] and
 * z [U][D] are updated in place (fp64); o [U][Dv] receives the read-out. */
int oracle_decode_step(const float *q, const float *k, const float *v,
                       const double *gamma, double eps, int64_t U, int D,
                       int Dv, double *S, double *z, double *o, int nthreads) {
  if (U < 0 || D <= 0 || Dv <= 0 || !q || !k || !v || !S || !z || !o) return -1;
  job_t J;
  memset(&J, 0, sizeof J);
  J.mode = MODE_DECODE;
  J.U = U; J.N = 1; J.D = D; J.Dv = Dv;
  J.q = q; J.k = k; J.v = v; J.gamma = gamma; J.eps = eps;
  J.o = o; J.S = S; J.z = z;
  return run_jobs(J, nthreads);
}

/* Gated form.  a [U][N][D] gates; o may be NULL (state only); S_state,
 * z_state may be NULL, else they receive the state after token N-1. */
int oracle_gated(const float *q, const float *k, const float *v, const float *a,
                 double eps, int64_t U, int64_t N, int D, int Dv, double *o,
                 double *S_state, double *z_state, int nthreads) {
  if (U < 0 || N < 0 || D <= 0 || Dv <= 0 || !k || !v || !a || (o && !q)) return -1;
  job_t J;
  memset(&J, 0, sizeof J);
  J.mode = MODE_GATED;
  J.U = U; J.N = N; J.D = D; J.Dv = Dv;
  J.q = q; J.k = k; J.v = v; J.a = a; J.eps = eps;
  J.o = o; J.S = S_state; J.z = z_state;
  return run_jobs(J, nthreads);
}
