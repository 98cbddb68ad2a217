/*
 * FP64 CPU oracle for triangular (pair-biased, slice-batched) attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: it exists so that tests, the smoke check and the
 * benchmark's CPU-baseline leg can compare the CUDA kernels against a plain,
 * slow, obviously correct statement of the mathematics.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Source of the definition: "TurboPairFormer: Fast and Stable Protein Folding
 * Model Training with an Optimized Triangle Attention Kernel"
 * (thelatestinai.com/papers/2610.05854):
 *   - Abstract and Figure 1(a): N_o slices share one pair bias; the backward
 *     has three reductions: dQ over keys, dK/dV over queries, dbias over the
 *     outer slices.  P and dS are the shared intermediates.
 *   - Table 1 (notation): Q, K, V, O are [B, N_o, H, N, D]; for one example,
 *     slice and head each is an N x D matrix.
 *   - Figure 6 (worked example): the score of query q and key k in slice o
 *     adds the bias of pair (q, k), and every slice uses that same bias.
 * The per-slice operation is exact softmax attention with an additive bias
 * and an additive key mask:
 *     S[q,k]  = (Q[q,:] . K[k,:]) / sqrt(D) + bias[b,h,q,k] + mask[b,o,k]
 *     P       = softmax_k(S),  lse[q] = log sum_k exp(S[q,k])
 *     O[q,:]  = sum_k P[q,k] V[k,:]
 * and its exact gradient for an incoming dO:
 *     dV[k,:] = sum_q P[q,k] dO[q,:]
 *     dP[q,k] = dO[q,:] . V[k,:]
 *     delta[q]= sum_d dO[q,d] O[q,d]            (O in full FP64 precision)
 *     dS      = P * (dP - delta)
 *     dQ[q,:] = sum_k dS[q,k] K[k,:] / sqrt(D)
 *     dK[k,:] = sum_q dS[q,k] Q[q,:] / sqrt(D)
 *     dbias[b,h,q,k] = sum_o dS_o[q,k]           (the cross-slice reduction)
 *
 * Readings taken where the pages are silent:
 *   - the 1/sqrt(D) scale multiplies Q.K only;
 *   - the mask is additive, per (b, o, key), broadcast over queries and heads,
 *     and carries no gradient;
 *   - a query row whose keys are all masked (every S = -inf) has P = 0,
 *     O = 0, lse = -inf and contributes zero to every gradient.
 *
 * Generality beyond the method: the query count Nq and the key count Nk may
 * differ (the method has Nq = Nk = N).  Restricting Q, bias and dO to a subset
 * of query rows therefore yields exactly those rows of O, lse, dQ and dbias,
 * which lets tests check sampled outputs of full-size problems.
 *
 * Layouts (all row-major, contiguous, FP64):
 *   q, o, dO, dq : [B, No, H, Nq, D]
 *   k, v, dk, dv : [B, No, H, Nk, D]
 *   bias, dbias  : [B, H, Nq, Nk]
 *   mask         : [B, No, Nk] or NULL (no mask)
 *   lse          : [B, No, H, Nq]   natural logarithm
 *
 * Parallelism: OpenMP over independent slices (b, o, h).  dbias is summed
 * per (b, h) over o by each thread into a private buffer, and the private
 * buffers are added in thread order afterwards.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int B, No, H, Nq, Nk, D;
} oracle_shape;

static size_t qoff(const oracle_shape* s, int b, int o, int h) {
  return ((((size_t)b * s->No + o) * s->H + h) * (size_t)s->Nq) * s->D;
}
static size_t koff(const oracle_shape* s, int b, int o, int h) {
  return ((((size_t)b * s->No + o) * s->H + h) * (size_t)s->Nk) * s->D;
}

/* One slice forward: fills P (Nq x Nk), O rows and lse.  Returns nothing;
 * P is left in the caller's scratch for the backward. */
static void slice_forward(const oracle_shape* s, const double* Q, const double* K,
                          const double* V, const double* bias_bh, const double* mask_bo,
                          double* P, double* O, double* lse) {
  const int Nq = s->Nq, Nk = s->Nk, D = s->D;
  const double scale = 1.0 / sqrt((double)D);
  for (int q = 0; q < Nq; ++q) {
    double* Srow = P + (size_t)q * Nk;
    double m = -INFINITY;
    for (int k = 0; k < Nk; ++k) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += Q[(size_t)q * D + d] * K[(size_t)k * D + d];
      double sc = dot * scale + bias_bh[(size_t)q * Nk + k];
      if (mask_bo) sc += mask_bo[k];
      Srow[k] = sc;
      if (sc > m) m = sc;
    }
    if (m == -INFINITY) {           /* every key masked: empty softmax */
      for (int k = 0; k < Nk; ++k) Srow[k] = 0.0;
      for (int d = 0; d < D; ++d) O[(size_t)q * D + d] = 0.0;
      lse[q] = -INFINITY;
      continue;
    }
    double l = 0.0;
    for (int k = 0; k < Nk; ++k) {
      double e = exp(Srow[k] - m);
      Srow[k] = e;
      l += e;
    }
    for (int k = 0; k < Nk; ++k) Srow[k] /= l;
    lse[q] = m + log(l);
    for (int d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int k = 0; k < Nk; ++k) acc += Srow[k] * V[(size_t)k * D + d];
      O[(size_t)q * D + d] = acc;
    }
  }
}

void oracle_fwd(const oracle_shape* s, const double* q, const double* k, const double* v,
                const double* bias, const double* mask, double* o, double* lse) {
  const long nslices = (long)s->B * s->No * s->H;
#pragma omp parallel
  {
    double* P = (double*)malloc(sizeof(double) * (size_t)s->Nq * s->Nk);
#pragma omp for schedule(static)
    for (long idx = 0; idx < nslices; ++idx) {
      int h = (int)(idx % s->H);
      int o_ = (int)((idx / s->H) % s->No);
      int b = (int)(idx / ((long)s->H * s->No));
      const double* bias_bh = bias + ((size_t)b * s->H + h) * (size_t)s->Nq * s->Nk;
      const double* mask_bo = mask ? mask + ((size_t)b * s->No + o_) * (size_t)s->Nk : NULL;
      size_t lo = (((size_t)b * s->No + o_) * s->H + h) * (size_t)s->Nq;
      slice_forward(s, q + qoff(s, b, o_, h), k + koff(s, b, o_, h), v + koff(s, b, o_, h),
                    bias_bh, mask_bo, P, o + qoff(s, b, o_, h), lse + lo);
    }
    free(P);
  }
}

void oracle_bwd(const oracle_shape* s, const double* q, const double* k, const double* v,
                const double* bias, const double* mask, const double* dO,
                double* dq, double* dk, double* dv, double* dbias) {
  const int Nq = s->Nq, Nk = s->Nk, D = s->D, H = s->H, No = s->No;
  const double scale = 1.0 / sqrt((double)D);
  const size_t nbias = (size_t)s->B * H * Nq * Nk;
  int nthreads = 1;
#ifdef _OPENMP
  nthreads = omp_get_max_threads();
#endif
  double* priv = (double*)calloc((size_t)nthreads * nbias, sizeof(double));
  const long nslices = (long)s->B * No * H;
#pragma omp parallel
  {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    double* mine = priv + (size_t)tid * nbias;
    double* P = (double*)malloc(sizeof(double) * (size_t)Nq * Nk);
    double* O = (double*)malloc(sizeof(double) * (size_t)Nq * D);
    double* lse = (double*)malloc(sizeof(double) * (size_t)Nq);
    double* delta = (double*)malloc(sizeof(double) * (size_t)Nq);
    double* dSrow = (double*)malloc(sizeof(double) * (size_t)Nk);
#pragma omp for schedule(static)
    for (long idx = 0; idx < nslices; ++idx) {
      int h = (int)(idx % H);
      int o_ = (int)((idx / H) % No);
      int b = (int)(idx / ((long)H * No));
      const double* Q = q + qoff(s, b, o_, h);
      const double* K = k + koff(s, b, o_, h);
      const double* V = v + koff(s, b, o_, h);
      const double* G = dO + qoff(s, b, o_, h);
      const double* bias_bh = bias + ((size_t)b * H + h) * (size_t)Nq * Nk;
      const double* mask_bo = mask ? mask + ((size_t)b * No + o_) * (size_t)Nk : NULL;
      double* dQ = dq + qoff(s, b, o_, h);
      double* dK = dk + koff(s, b, o_, h);
      double* dV = dv + koff(s, b, o_, h);
      double* dB = mine + ((size_t)b * H + h) * (size_t)Nq * Nk;
      slice_forward(s, Q, K, V, bias_bh, mask_bo, P, O, lse);
      for (int qq = 0; qq < Nq; ++qq) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += G[(size_t)qq * D + d] * O[(size_t)qq * D + d];
        delta[qq] = acc;
      }
      memset(dK, 0, sizeof(double) * (size_t)Nk * D);
      memset(dV, 0, sizeof(double) * (size_t)Nk * D);
      for (int qq = 0; qq < Nq; ++qq) {
        const double* Prow = P + (size_t)qq * Nk;
        for (int kk = 0; kk < Nk; ++kk) {
          double dp = 0.0;
          for (int d = 0; d < D; ++d) dp += G[(size_t)qq * D + d] * V[(size_t)kk * D + d];
          dSrow[kk] = Prow[kk] * (dp - delta[qq]);
        }
        for (int d = 0; d < D; ++d) {
          double acc = 0.0;
          for (int kk = 0; kk < Nk; ++kk) acc += dSrow[kk] * K[(size_t)kk * D + d];
          dQ[(size_t)qq * D + d] = acc * scale;
        }
        for (int kk = 0; kk < Nk; ++kk) {
          for (int d = 0; d < D; ++d) {
            dK[(size_t)kk * D + d] += dSrow[kk] * Q[(size_t)qq * D + d] * scale;
            dV[(size_t)kk * D + d] += Prow[kk] * G[(size_t)qq * D + d];
          }
          dB[(size_t)qq * Nk + kk] += dSrow[kk];
        }
      }
    }
    free(P); free(O); free(lse); free(delta); free(dSrow);
  }
  memset(dbias, 0, sizeof(double) * nbias);
  for (int t = 0; t < nthreads; ++t) {
    const double* src = priv + (size_t)t * nbias;
    for (size_t i = 0; i < nbias; ++i) dbias[i] += src[i];
  }
  free(priv);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
