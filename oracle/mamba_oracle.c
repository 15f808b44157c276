/*
 * Float64 CPU oracle for the Mamba-1 selective scan.
 *
 * TEST INFRASTRUCTURE ONLY.  The plain sequential definition that the CUDA
 * library's selective-scan kernels are checked against; nothing in the
 * product library links, includes or calls it.
 *
 * What it computes (the op of the "kernel_mamba_cpu.json" benchmark records:
 * Mamba selective scan, state 16, arguments x, delta [B,L,D], A [D,N],
 * B, C [B,L,N], D [D] -- the records' argument bytes fit exactly these):
 *
 *   per batch b and channel d, state h[n], n < N, h_{-1} = 0
 *     h_t[n] = exp(delta_t[d] A[d,n]) h_{t-1}[n] + delta_t[d] B_t[n] x_t[d]
 *     y_t[d] = sum_n C_t[n] h_t[n] + D[d] x_t[d]
 *
 * (zero-order hold for A, the delta-scaled B for the input, as in the Mamba
 * selective scan; delta is used as given).  The backward is the exact
 * adjoint of <dy, y>, with g_t = dL/dh_t:
 *
 *     g_t[n]   = C_t[n] dy_t + exp(delta_{t+1} A[n]) g_{t+1}[n]     (g_L = 0)
 *     dx_t     = sum_n g_t[n] delta_t B_t[n] + D dy_t
 *     ddelta_t = sum_n g_t[n] (A[n] exp(delta_t A[n]) h_{t-1}[n] + B_t[n] x_t)
 *     dA[d,n] += g_t[n] delta_t exp(delta_t A[n]) h_{t-1}[n]   (over b, t)
 *     dB_t[n] += g_t[n] delta_t x_t                            (over d)
 *     dC_t[n] += dy_t h_t[n]                                   (over d)
 *     dD[d]   += dy_t x_t                                      (over b, t)
 *
 * Everything is float64.  The states are recomputed from checkpoints every
 * CKPT steps in the reverse sweep (no decay is divided out).  Sums over d
 * (dB, dC) and over b (dA, dD) are formed per thread / per batch entry and
 * added in a fixed order.  D may be NULL (no skip term, dD not written).
 *
 * Layouts (row-major): x, delta, y, dy, dx, ddelta [B,L,D]; A, dA [D,N];
 * Bm, Cm, dB, dC [B,L,N]; Dk, dD [D].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 64

int mamba_oracle_fwd(const double *x, const double *dt, const double *A, const double *Bm,
                     const double *Cm, const double *Dk, double *y, int64_t B, int64_t L,
                     int64_t D, int64_t N) {
  if (B < 0 || L < 0 || D <= 0 || N <= 0) return 1;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t bd = 0; bd < B * D; ++bd) {
    const int64_t b = bd / D, d = bd % D;
    double *h = (double *)calloc((size_t)N, sizeof(double));
    if (!h) { err = 2; continue; }
    for (int64_t t = 0; t < L; ++t) {
      const int64_t i = (b * L + t) * D + d;
      const double xt = x[i], dtt = dt[i];
      const double *Bt = Bm + (b * L + t) * N, *Ct = Cm + (b * L + t) * N;
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        h[n] = exp(dtt * A[d * N + n]) * h[n] + dtt * Bt[n] * xt;
        acc += Ct[n] * h[n];
      }
      y[i] = acc + (Dk ? Dk[d] * xt : 0.0);
    }
    free(h);
  }
  return err;
}

int mamba_oracle_bwd(const double *x, const double *dt, const double *A, const double *Bm,
                     const double *Cm, const double *Dk, const double *dy, double *dx,
                     double *ddt, double *dA, double *dB, double *dC, double *dD, int64_t B,
                     int64_t L, int64_t D, int64_t N) {
  if (B < 0 || L < 0 || D <= 0 || N <= 0) return 1;
  int nthr = 1;
#ifdef _OPENMP
  nthr = omp_get_max_threads();
#endif
  const int64_t nck = (L + CKPT - 1) / CKPT;
  /* per-thread partial sums of dB and dC over the channels a thread handles,
   * per-(b, d) partials of dA and dD over time */
  double *pB = (double *)calloc((size_t)nthr * B * L * N + 1, sizeof(double));
  double *pC = (double *)calloc((size_t)nthr * B * L * N + 1, sizeof(double));
  double *pA = (double *)calloc((size_t)B * D * N + 1, sizeof(double));
  double *pD = (double *)calloc((size_t)B * D + 1, sizeof(double));
  if (!pB || !pC || !pA || !pD) { free(pB); free(pC); free(pA); free(pD); return 2; }
  int err = 0;
#pragma omp parallel
  {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    double *myB = pB + (size_t)tid * B * L * N, *myC = pC + (size_t)tid * B * L * N;
    double *ck = (double *)malloc(sizeof(double) * N * (nck > 0 ? nck : 1));
    double *seg = (double *)malloc(sizeof(double) * N * (CKPT + 1));
    double *g = (double *)malloc(sizeof(double) * N);
    const int ok = ck && seg && g;
    if (!ok) err = 2;
    {
#pragma omp for schedule(static)
      for (int64_t bd = 0; bd < B * D; ++bd) {
        if (!ok) continue;
        const int64_t b = bd / D, d = bd % D;
        const double *Ad = A + d * N;
        /* forward sweep: checkpoints ck[c] = h_{c*CKPT - 1} */
        double *h = seg;
        memset(h, 0, sizeof(double) * N);
        for (int64_t t = 0; t < L; ++t) {
          if (t % CKPT == 0) memcpy(ck + (t / CKPT) * N, h, sizeof(double) * N);
          const int64_t i = (b * L + t) * D + d;
          const double *Bt = Bm + (b * L + t) * N;
          for (int64_t n = 0; n < N; ++n) h[n] = exp(dt[i] * Ad[n]) * h[n] + dt[i] * Bt[n] * x[i];
        }
        memset(g, 0, sizeof(double) * N);
        double dDs = 0.0;
        for (int64_t c = nck - 1; c >= 0; --c) {
          const int64_t t0 = c * CKPT, t1 = t0 + CKPT < L ? t0 + CKPT : L;
          /* seg[j] = h_{t0 - 1 + j}, j = 0 .. t1 - t0 */
          memcpy(seg, ck + c * N, sizeof(double) * N);
          for (int64_t t = t0; t < t1; ++t) {
            const int64_t i = (b * L + t) * D + d;
            const double *Bt = Bm + (b * L + t) * N;
            const double *hp = seg + (t - t0) * N;
            double *hn = seg + (t - t0 + 1) * N;
            for (int64_t n = 0; n < N; ++n) hn[n] = exp(dt[i] * Ad[n]) * hp[n] + dt[i] * Bt[n] * x[i];
          }
          for (int64_t t = t1 - 1; t >= t0; --t) {
            const int64_t i = (b * L + t) * D + d;
            const double *Bt = Bm + (b * L + t) * N, *Ct = Cm + (b * L + t) * N;
            const double *hp = seg + (t - t0) * N;      /* h_{t-1} */
            const double *ht = seg + (t - t0 + 1) * N;  /* h_t */
            double sx = 0.0, sdt = 0.0;
            for (int64_t n = 0; n < N; ++n) {
              g[n] += Ct[n] * dy[i];
              const double a = exp(dt[i] * Ad[n]);
              sx += g[n] * dt[i] * Bt[n];
              sdt += g[n] * (Ad[n] * a * hp[n] + Bt[n] * x[i]);
              pA[bd * N + n] += g[n] * dt[i] * a * hp[n];
              myB[(b * L + t) * N + n] += g[n] * dt[i] * x[i];
              myC[(b * L + t) * N + n] += dy[i] * ht[n];
              g[n] *= a;
            }
            dx[i] = sx + (Dk ? Dk[d] * dy[i] : 0.0);
            ddt[i] = sdt;
            dDs += dy[i] * x[i];
          }
        }
        pD[bd] = dDs;
      }
    }
    free(ck); free(seg); free(g);
  }
  if (!err) {
    for (int64_t e = 0; e < B * L * N; ++e) {
      double sb = 0.0, sc = 0.0;
      for (int r = 0; r < nthr; ++r) { sb += pB[(size_t)r * B * L * N + e]; sc += pC[(size_t)r * B * L * N + e]; }
      dB[e] = sb;
      dC[e] = sc;
    }
    for (int64_t e = 0; e < D * N; ++e) {
      double s = 0.0;
      for (int64_t b = 0; b < B; ++b) s += pA[b * D * N + e];
      dA[e] = s;
    }
    if (dD)
      for (int64_t d = 0; d < D; ++d) {
        double s = 0.0;
        for (int64_t b = 0; b < B; ++b) s += pD[b * D + d];
        dD[d] = s;
      }
  }
  free(pB); free(pC); free(pA); free(pD);
  return err;
}
