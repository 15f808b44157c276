/*
 * Float64 CPU oracle for the gated linear-attention (SSD) scan.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, sequential
 * definition that the CUDA library is checked against.  Nothing in the
 * product library links, includes or calls it; only the tests, the smoke
 * check and the CPU-baseline leg of the benchmark load it.
 *
 * What it computes (the definition fixed for the chunked SSD benchmark
 * records "kernel_ssd_gpu.json" / "kernel_ssd_cpu.json", which time a
 * chunked implementation against a step-by-step "scan" of the same op):
 *
 *   per batch b and head h, with group g = h / (H / G)   (contiguous split)
 *     S_{-1} = h0[b,h]                                   (dk x dv)
 *     S_t    = exp(la[b,t,h]) * S_{t-1} + k[b,t,g] v[b,t,h]^T
 *     out[b,t,h,:] = S_t^T q[b,t,g]                      (inclusive state,
 *                                                          unscaled q)
 *
 * and, for a cotangent dout with loss <dout, out>, the exact adjoint:
 *
 *     G_t      = q_t dout_t^T + exp(la_{t+1}) G_{t+1}    (G_L = 0)
 *     dq_h[t]  = S_t dout_t,   dk_h[t] = G_t v_t,   dv[t] = G_t^T k_t
 *     dla[t]   = exp(la_t) <G_t, S_{t-1}>_F
 *     dh0      = exp(la_0) G_0
 *     dq[b,t,g] = sum over the heads h of group g of dq_h[t]  (dk likewise)
 *
 * Everything is float64.  The backward needs S_{t-1} in reverse order; it
 * stores S at every CKPT-th step on the forward sweep and recomputes the
 * states inside each checkpoint segment (never by dividing out a decay).
 * dla uses the direct adjoint above, not a cumulative-sum identity.
 *
 * Optionally the forward also returns the final state hT = S_{L-1} and the
 * backward takes its cotangent dhT (loss <dout, out> + <dhT, hT>): the
 * adjoint then starts from G_{L-1} = q_{L-1} dout_{L-1}^T + dhT.
 *
 * Layouts (row-major, the benchmark records' argument sizes):
 *   q, k [B,L,G,dk]   v, out [B,L,H,dv]   la [B,L,H]   h0, dh0, hT, dhT [B,H,dk,dv]
 * h0 and dhT may be NULL (zeros); dh0, hT, dq_heads, dk_heads may be NULL
 * (not wanted).
 * dq_heads / dk_heads [B,L,H,dk] receive the per-head, pre-group-sum
 * gradients when given.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 64

static inline int64_t grp(int64_t h, int64_t H, int64_t G) { return h / (H / G); }

/* S <- a * S + k v^T */
static void state_step(double *S, double a, const double *kt, const double *vt,
                       int64_t dk, int64_t dv) {
  for (int64_t i = 0; i < dk; ++i) {
    double ki = kt[i];
    double *row = S + i * dv;
    for (int64_t j = 0; j < dv; ++j) row[j] = a * row[j] + ki * vt[j];
  }
}

int ssd_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

int ssd_oracle_fwd(const double *q, const double *k, const double *v,
                   const double *la, const double *h0, double *out, double *hT,
                   int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk,
                   int64_t dv) {
  if (B < 0 || L < 0 || G <= 0 || H <= 0 || dk <= 0 || dv <= 0 || H % G)
    return 1;
  int64_t BH = B * H;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < BH; ++bh) {
    int64_t b = bh / H, h = bh % H, g = grp(h, H, G);
    double *S = (double *)malloc(sizeof(double) * dk * dv);
    if (!S) { err = 2; continue; }
    if (h0) memcpy(S, h0 + bh * dk * dv, sizeof(double) * dk * dv);
    else memset(S, 0, sizeof(double) * dk * dv);
    for (int64_t t = 0; t < L; ++t) {
      const double *qt = q + ((b * L + t) * G + g) * dk;
      const double *kt = k + ((b * L + t) * G + g) * dk;
      const double *vt = v + ((b * L + t) * H + h) * dv;
      double a = exp(la[(b * L + t) * H + h]);
      state_step(S, a, kt, vt, dk, dv);
      double *ot = out + ((b * L + t) * H + h) * dv;
      for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
      for (int64_t i = 0; i < dk; ++i) {
        double qi = qt[i];
        const double *row = S + i * dv;
        for (int64_t j = 0; j < dv; ++j) ot[j] += qi * row[j];
      }
    }
    if (hT) memcpy(hT + bh * dk * dv, S, sizeof(double) * dk * dv);
    free(S);
  }
  return err;
}

int ssd_oracle_bwd(const double *q, const double *k, const double *v,
                   const double *la, const double *h0, const double *dout,
                   const double *dhT,
                   double *dq, double *dk_out, double *dv_out, double *dla,
                   double *dh0, double *dq_heads, double *dk_heads,
                   int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk,
                   int64_t dv) {
  if (B < 0 || L < 0 || G <= 0 || H <= 0 || dk <= 0 || dv <= 0 || H % G)
    return 1;
  const int64_t BH = B * H, sz = dk * dv;
  const int64_t nck = (L + CKPT - 1) / CKPT;
  /* per-head dq/dk are accumulated into the group outputs after the loop,
   * in a fixed head order, so the result does not depend on threading */
  double *dqh = dq_heads ? dq_heads : (double *)malloc(sizeof(double) * B * L * H * dk);
  double *dkh = dk_heads ? dk_heads : (double *)malloc(sizeof(double) * B * L * H * dk);
  if (!dqh || !dkh) return 2;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < BH; ++bh) {
    int64_t b = bh / H, h = bh % H, g = grp(h, H, G);
    /* checkpoints: ck[c] = state entering step c*CKPT (i.e. S_{c*CKPT-1}) */
    double *ck = (double *)malloc(sizeof(double) * sz * (nck > 0 ? nck : 1));
    double *seg = (double *)malloc(sizeof(double) * sz * (CKPT + 1));
    double *Gs = (double *)calloc((size_t)sz, sizeof(double));
    if (!ck || !seg || !Gs) { err = 2; free(ck); free(seg); free(Gs); continue; }
    if (dhT) memcpy(Gs, dhT + bh * sz, sizeof(double) * sz);
    double *S = seg; /* scratch for the forward sweep */
    if (h0) memcpy(S, h0 + bh * sz, sizeof(double) * sz);
    else memset(S, 0, sizeof(double) * sz);
    for (int64_t t = 0; t < L; ++t) {
      if (t % CKPT == 0) memcpy(ck + (t / CKPT) * sz, S, sizeof(double) * sz);
      const double *kt = k + ((b * L + t) * G + g) * dk;
      const double *vt = v + ((b * L + t) * H + h) * dv;
      state_step(S, exp(la[(b * L + t) * H + h]), kt, vt, dk, dv);
    }
    for (int64_t c = nck - 1; c >= 0; --c) {
      int64_t t0 = c * CKPT, t1 = t0 + CKPT < L ? t0 + CKPT : L;
      /* seg[j] = S_{t0-1+j}, j = 0 .. t1-t0 */
      memcpy(seg, ck + c * sz, sizeof(double) * sz);
      for (int64_t t = t0; t < t1; ++t) {
        double *nxt = seg + (t - t0 + 1) * sz;
        memcpy(nxt, seg + (t - t0) * sz, sizeof(double) * sz);
        state_step(nxt, exp(la[(b * L + t) * H + h]),
                   k + ((b * L + t) * G + g) * dk, v + ((b * L + t) * H + h) * dv, dk, dv);
      }
      for (int64_t t = t1 - 1; t >= t0; --t) {
        const double *qt = q + ((b * L + t) * G + g) * dk;
        const double *kt = k + ((b * L + t) * G + g) * dk;
        const double *vt = v + ((b * L + t) * H + h) * dv;
        const double *dot = dout + ((b * L + t) * H + h) * dv;
        const double *St = seg + (t - t0 + 1) * sz;   /* S_t */
        const double *Sp = seg + (t - t0) * sz;       /* S_{t-1} */
        double a = exp(la[(b * L + t) * H + h]);
        /* G_t = q_t dout_t^T + (decayed G_{t+1}, already in Gs) */
        for (int64_t i = 0; i < dk; ++i)
          for (int64_t j = 0; j < dv; ++j) Gs[i * dv + j] += qt[i] * dot[j];
        double *dqt = dqh + ((b * L + t) * H + h) * dk;
        double *dkt = dkh + ((b * L + t) * H + h) * dk;
        double *dvt = dv_out + ((b * L + t) * H + h) * dv;
        for (int64_t j = 0; j < dv; ++j) dvt[j] = 0.0;
        double inner = 0.0;
        for (int64_t i = 0; i < dk; ++i) {
          double sq = 0.0, sk = 0.0;
          for (int64_t j = 0; j < dv; ++j) {
            sq += St[i * dv + j] * dot[j];
            sk += Gs[i * dv + j] * vt[j];
            dvt[j] += Gs[i * dv + j] * kt[i];
            inner += Gs[i * dv + j] * Sp[i * dv + j];
          }
          dqt[i] = sq;
          dkt[i] = sk;
        }
        dla[(b * L + t) * H + h] = a * inner;
        for (int64_t i = 0; i < sz; ++i) Gs[i] *= a;
      }
    }
    if (dh0) memcpy(dh0 + bh * sz, Gs, sizeof(double) * sz);
    free(ck); free(seg); free(Gs);
  }
  if (!err) {
    const int64_t hpg = H / G;
#pragma omp parallel for schedule(static)
    for (int64_t bt = 0; bt < B * L; ++bt) {
      for (int64_t g = 0; g < G; ++g) {
        double *dqo = dq + (bt * G + g) * dk;
        double *dko = dk_out + (bt * G + g) * dk;
        for (int64_t i = 0; i < dk; ++i) { dqo[i] = 0.0; dko[i] = 0.0; }
        for (int64_t hh = 0; hh < hpg; ++hh) {
          int64_t h = g * hpg + hh;
          const double *a = dqh + (bt * H + h) * dk;
          const double *c = dkh + (bt * H + h) * dk;
          for (int64_t i = 0; i < dk; ++i) { dqo[i] += a[i]; dko[i] += c[i]; }
        }
      }
    }
  }
  if (!dq_heads) free(dqh);
  if (!dk_heads) free(dkh);
  return err;
}
