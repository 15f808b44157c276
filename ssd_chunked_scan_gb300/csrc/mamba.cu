// Mamba-1 selective scan (state N <= 16), forward and backward, all fp32 on
// the CUDA cores.  The op of the "kernel_mamba_cpu.json" benchmark records:
//
//   h_t[d,n] = exp(delta_t[d] A[d,n]) h_{t-1}[d,n] + delta_t[d] B_t[n] x_t[d],  h_{-1} = 0
//   y_t[d]   = sum_n C_t[n] h_t[d,n] + D[d] x_t[d]
//
// There is no dense contraction here (each state element has its own decay),
// so the work is elementwise recurrences and short reductions; it is bound by
// the exponentials (one per (token, channel, state)) and by HBM traffic.
//
// Each (batch, channel) sequence is cut into nseg segments so that enough
// threads run at once.  The forward-type passes give one thread a whole
// channel segment with the channel's 16 states in registers (B_t and C_t
// rows are shared-memory broadcasts); the backward's main kernel gives one
// thread one state of a channel (the 16 lanes of a half-warp hold a channel,
// the reduction over n is four shuffles) so that 32 tokens of recomputed
// states fit in its registers.
//
//   k_mb_local<false>  each segment's final state from a zero state, and its
//                      delta sum, from which the segment's decay
//                      exp(A * sum delta) follows
//   k_mb_scan<false>   state entering every segment (sequential over segments)
//   k_mb_out           each segment again from its entering state, emitting y
//
// The backward uses u_t = exp(delta_t A) g_t, g_t = dL/dh_t, which satisfies
// g_t = C_t dy_t + u_{t+1} (u_L = 0):
//
//   k_mb_local<true>   each segment's u at its left end from u = 0 at its right
//   k_mb_scan<true>    u entering every segment from the right
//   k_mb_bwd           per segment: a forward pass that checkpoints h every 16
//                      tokens (shared memory), then the 16-token windows right
//                      to left: recompute h_t and the decays into registers,
//                      walk them backwards accumulating
//                        dx_t = sum_n g delta B + D dy     dA += g delta a h_{t-1}
//                        ddelta_t = sum_n g (A a h_{t-1} + B x)
//                        dB_t[n] += g delta x,  dC_t[n] += dy h_t   (over d)
//                      dB / dC / dA / dD are summed across CTAs with fp32
//                      atomic adds (caller buffers zero-filled first).
#include "common.cuh"
#include "mamba.h"

namespace ssd {
namespace mamba {

constexpr int NL = 16;           // lanes per channel (N <= 16)
constexpr int CH = 16;           // channels per CTA
constexpr int NT = CH * NL;      // 256 threads
constexpr int TB = 32;           // tokens per staged block
constexpr float LOG2E = 1.4426950408889634f;

struct MGeo {
  int64_t B, L, D, N;
  int64_t Ls;    // segment length (multiple of TB)
  int64_t nseg;
};

__device__ inline float half_sum(float v) {  // sum over the 16 lanes of a half-warp
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Token staging of one block: per-channel series ([TB][CH]) and per-token
// state-indexed rows ([TB][NL]).
struct Stage {
  float *xs, *ds, *ys;  // x, delta, dy    [TB][CH]
  float *bs, *cs;       // B, C            [TB][NL]
};

// Each thread loads all of its elements of the block (two of each series at
// 256 threads) before it stores any, so staging costs one memory round trip.
__device__ inline void stage_block(const Stage &st, const float *x, const float *dt,
                                   const float *dy, const float *Bm, const float *Cm,
                                   const MGeo &g, int64_t b, int64_t d0, int64_t t0, int len) {
  constexpr int PC = (TB * CH + NT - 1) / NT, PN = (TB * NL + NT - 1) / NT;
  float vx[PC], vd[PC], vy[PC], vb[PN], vc[PN];
#pragma unroll
  for (int u = 0; u < PC; ++u) {
    const int idx = threadIdx.x + u * NT, tt = idx / CH, c = idx - tt * CH;
    const bool ok = idx < TB * CH && tt < len && d0 + c < g.D;
    const int64_t o = (b * g.L + t0 + tt) * g.D + d0 + c;
    vx[u] = ok ? x[o] : 0.f;
    vd[u] = ok ? dt[o] : 0.f;
    vy[u] = (dy && ok) ? dy[o] : 0.f;
  }
#pragma unroll
  for (int u = 0; u < PN; ++u) {
    const int idx = threadIdx.x + u * NT, tt = idx / NL, n = idx - tt * NL;
    const bool ok = idx < TB * NL && tt < len && n < g.N;
    const int64_t o = (b * g.L + t0 + tt) * g.N + n;
    vb[u] = (Bm && ok) ? Bm[o] : 0.f;
    vc[u] = (Cm && ok) ? Cm[o] : 0.f;
  }
#pragma unroll
  for (int u = 0; u < PC; ++u) {
    const int idx = threadIdx.x + u * NT;
    if (idx < TB * CH) {
      st.xs[idx] = vx[u];
      st.ds[idx] = vd[u];
      if (dy) st.ys[idx] = vy[u];
    }
  }
#pragma unroll
  for (int u = 0; u < PN; ++u) {
    const int idx = threadIdx.x + u * NT;
    if (idx < TB * NL) {
      if (Bm) st.bs[idx] = vb[u];
      if (Cm) st.cs[idx] = vc[u];
    }
  }
}

// The channel kernels: one thread per (batch, channel, segment) holding the
// channel's NL states in registers; a CTA covers CCH consecutive channels.
constexpr int CCH = 128;

// Per-block staging of the channel kernels: per-channel series [TB][CCH] and
// the per-token rows of B and C [TB][NL] (read as float4 broadcasts).
// The channel kernels' staging issues the loads of SB rows of the block per
// thread before storing them, so a block costs TB / SB memory round trips.
constexpr int SB = 4;
__device__ inline void stage_channels(float *xs, float *ds, float *ys, float *bs, float *cs,
                                      const float *x, const float *dt, const float *dy,
                                      const float *Bm, const float *Cm, const MGeo &g, int64_t b,
                                      int64_t d0, int64_t t0, int len) {
  const int c = threadIdx.x;  // idx = tt * CCH + c: thread c stages channel c of every row
  const bool cok = d0 + c < g.D;
  for (int t0b = 0; t0b < TB; t0b += SB) {
    float vx[SB], vd[SB], vy[SB];
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      const int tt = t0b + u;
      const bool ok = tt < len && cok;
      const int64_t o = (b * g.L + t0 + tt) * g.D + d0 + c;
      vx[u] = (xs && ok) ? x[o] : 0.f;
      vd[u] = ok ? dt[o] : 0.f;
      vy[u] = (ys && ok) ? dy[o] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      const int idx = (t0b + u) * CCH + c;
      if (xs) xs[idx] = vx[u];
      ds[idx] = vd[u];
      if (ys) ys[idx] = vy[u];
    }
  }
  constexpr int PN = (TB * NL + CCH - 1) / CCH;
  float vb[PN], vc[PN];
#pragma unroll
  for (int u = 0; u < PN; ++u) {
    const int idx = threadIdx.x + u * CCH, tt = idx / NL, n = idx - tt * NL;
    const bool ok = idx < TB * NL && tt < len && n < g.N;
    const int64_t o = (b * g.L + t0 + tt) * g.N + n;
    vb[u] = (bs && ok) ? Bm[o] : 0.f;
    vc[u] = (cs && ok) ? Cm[o] : 0.f;
  }
#pragma unroll
  for (int u = 0; u < PN; ++u) {
    const int idx = threadIdx.x + u * CCH;
    if (idx < TB * NL) {
      if (bs) bs[idx] = vb[u];
      if (cs) cs[idx] = vc[u];
    }
  }
}

// Segment-local pass.  Forward: the state after the segment from h = 0, and
// the segment's delta sum (fp32 per 32-token block, fp64 across blocks).
// Reverse: u at the segment's left end from u = 0 at its right end.
// grid (ceil(D/CCH), nseg, B), CCH threads
template <bool REV>
__global__ void __launch_bounds__(CCH) k_mb_local(const float *__restrict__ x,
                                                  const float *__restrict__ dt,
                                                  const float *__restrict__ A,
                                                  const float *__restrict__ Bm,
                                                  const float *__restrict__ Cm,
                                                  const float *__restrict__ dy,
                                                  float *__restrict__ states,
                                                  float *__restrict__ dsum, MGeo g) {
  __shared__ float xs[TB * CCH], ds[TB * CCH];
  __shared__ __align__(16) float rs[TB * NL];  // B rows (forward) or C rows (reverse)
  const int c = threadIdx.x;
  const int64_t d0 = (int64_t)blockIdx.x * CCH, seg = blockIdx.y, b = blockIdx.z;
  const int64_t d = d0 + c;
  const bool ok = d < g.D;
  float A2[NL], h[NL];
#pragma unroll
  for (int n = 0; n < NL; ++n) {
    A2[n] = (ok && n < g.N) ? A[d * g.N + n] * LOG2E : 0.f;
    h[n] = 0.f;
  }
  const int64_t s0 = seg * g.Ls, s1 = s0 + g.Ls < g.L ? s0 + g.Ls : g.L;
  const int64_t nb = (s1 - s0 + TB - 1) / TB;
  double dsacc = 0.0;
  for (int64_t k = 0; k < nb; ++k) {
    const int64_t kb = REV ? nb - 1 - k : k;
    const int64_t t0 = s0 + kb * TB;
    const int len = (int)(s1 - t0 < TB ? s1 - t0 : TB);
    // reverse: xs holds dy
    stage_channels(REV ? nullptr : xs, ds, REV ? xs : nullptr, REV ? nullptr : rs,
                   REV ? rs : nullptr, x, dt, dy, Bm, Cm, g, b, d0, t0, len);
    __syncthreads();
    float bsum = 0.f;
    for (int j = 0; j < len; ++j) {
      const int i = REV ? len - 1 - j : j;
      const float de = ds[i * CCH + c], sv = xs[i * CCH + c];
      const float4 *r4 = reinterpret_cast<const float4 *>(rs + i * NL);
      float r[NL];
#pragma unroll
      for (int q = 0; q < NL / 4; ++q) {
        const float4 v = r4[q];
        r[4 * q] = v.x; r[4 * q + 1] = v.y; r[4 * q + 2] = v.z; r[4 * q + 3] = v.w;
      }
      if (!REV) {
        const float dx_ = de * sv;
#pragma unroll
        for (int n = 0; n < NL; ++n) h[n] = fmaf(exp2f(de * A2[n]), h[n], dx_ * r[n]);
        bsum += de;
      } else {
#pragma unroll
        for (int n = 0; n < NL; ++n) h[n] = exp2f(de * A2[n]) * fmaf(r[n], sv, h[n]);
      }
    }
    dsacc += (double)bsum;
    __syncthreads();
  }
  if (ok) {
    float *dst = states + ((b * g.nseg + seg) * g.D + d) * g.N;
#pragma unroll
    for (int n = 0; n < NL; ++n)
      if (n < g.N) dst[n] = h[n];
    if (!REV) dsum[(b * g.nseg + seg) * g.D + d] = (float)dsacc;
  }
}

// Across segments, in place: states[s] <- the state entering segment s from
// the left (forward) or the u entering it from the right (reverse).  The
// segments' values are loaded MS at a time ahead of the dependent chain.
// grid (ceil(B*D*N / 256))
constexpr int MS = 12;
template <bool REV>
__global__ void __launch_bounds__(256) k_mb_scan(float *__restrict__ states,
                                                 const float *__restrict__ dsum,
                                                 const float *__restrict__ A, MGeo g) {
  const int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (e >= g.B * g.D * g.N) return;
  const int64_t b = e / (g.D * g.N), dn = e - b * g.D * g.N, d = dn / g.N;
  const float A2 = A[dn] * LOG2E;
  float run = 0.f;
  for (int64_t k0 = 0; k0 < g.nseg; k0 += MS) {
    float xv[MS], dec[MS];
#pragma unroll
    for (int u = 0; u < MS; ++u) {
      const int64_t k = k0 + u;
      if (k < g.nseg) {
        const int64_t s = REV ? g.nseg - 1 - k : k;
        xv[u] = states[(b * g.nseg + s) * g.D * g.N + dn];
        dec[u] = exp2f(A2 * dsum[(b * g.nseg + s) * g.D + d]);
      }
    }
#pragma unroll
    for (int u = 0; u < MS; ++u) {
      const int64_t k = k0 + u;
      if (k < g.nseg) {
        const int64_t s = REV ? g.nseg - 1 - k : k;
        states[(b * g.nseg + s) * g.D * g.N + dn] = run;
        run = fmaf(dec[u], run, xv[u]);
      }
    }
  }
}

// y of every segment from its entering state.  grid (ceil(D/CCH), nseg, B),
// CCH threads
__global__ void __launch_bounds__(CCH) k_mb_out(const float *__restrict__ x,
                                                const float *__restrict__ dt,
                                                const float *__restrict__ A,
                                                const float *__restrict__ Bm,
                                                const float *__restrict__ Cm,
                                                const float *__restrict__ Dk,
                                                const float *__restrict__ hin,
                                                float *__restrict__ y, MGeo g) {
  __shared__ float xs[TB * CCH], ds[TB * CCH];
  __shared__ __align__(16) float bs[TB * NL], cs[TB * NL];
  const int c = threadIdx.x;
  const int64_t d0 = (int64_t)blockIdx.x * CCH, seg = blockIdx.y, b = blockIdx.z;
  const int64_t d = d0 + c;
  const bool ok = d < g.D;
  float A2[NL], h[NL];
  const float *hsrc = hin + ((b * g.nseg + seg) * g.D + d) * g.N;
#pragma unroll
  for (int n = 0; n < NL; ++n) {
    const bool on = ok && n < g.N;
    A2[n] = on ? A[d * g.N + n] * LOG2E : 0.f;
    h[n] = on ? hsrc[n] : 0.f;
  }
  const float Dd = (Dk && ok) ? Dk[d] : 0.f;
  const int64_t s0 = seg * g.Ls, s1 = s0 + g.Ls < g.L ? s0 + g.Ls : g.L;
  for (int64_t t0 = s0; t0 < s1; t0 += TB) {
    const int len = (int)(s1 - t0 < TB ? s1 - t0 : TB);
    stage_channels(xs, ds, nullptr, bs, cs, x, dt, nullptr, Bm, Cm, g, b, d0, t0, len);
    __syncthreads();
    for (int i = 0; i < len; ++i) {
      const float de = ds[i * CCH + c], xv = xs[i * CCH + c];
      const float4 *b4 = reinterpret_cast<const float4 *>(bs + i * NL);
      const float4 *c4 = reinterpret_cast<const float4 *>(cs + i * NL);
      const float dx_ = de * xv;
      float y0 = 0.f, y1 = 0.f;
#pragma unroll
      for (int q = 0; q < NL / 4; ++q) {
        const float4 bv = b4[q], cv = c4[q];
        h[4 * q + 0] = fmaf(exp2f(de * A2[4 * q + 0]), h[4 * q + 0], dx_ * bv.x);
        h[4 * q + 1] = fmaf(exp2f(de * A2[4 * q + 1]), h[4 * q + 1], dx_ * bv.y);
        h[4 * q + 2] = fmaf(exp2f(de * A2[4 * q + 2]), h[4 * q + 2], dx_ * bv.z);
        h[4 * q + 3] = fmaf(exp2f(de * A2[4 * q + 3]), h[4 * q + 3], dx_ * bv.w);
        y0 = fmaf(cv.x, h[4 * q + 0], y0);
        y1 = fmaf(cv.y, h[4 * q + 1], y1);
        y0 = fmaf(cv.z, h[4 * q + 2], y0);
        y1 = fmaf(cv.w, h[4 * q + 3], y1);
      }
      xs[i * CCH + c] = fmaf(Dd, xv, y0 + y1);  // y replaces x in place
    }
    __syncthreads();
    for (int idx = c; idx < len * CCH; idx += CCH) {
      const int tt = idx / CCH, cc = idx - tt * CCH;
      if (d0 + cc < g.D) y[(b * g.L + t0 + tt) * g.D + d0 + cc] = xs[idx];
    }
    __syncthreads();
  }
}

// Backward of every segment, in windows of WB tokens.  Dynamic shared memory:
// the h checkpoints [Ls/WB][NT], then the staging and reduction buffers.
// The per-token sums over n (dx, ddelta) are collected for a whole window in
// registers and reduce-scattered over the half-warp at its end (15 shuffles
// per window instead of 4 per token), lane n ending with token n's sums.
// grid (ceil(D/CH), nseg, B)
constexpr int WB = 16;
__global__ void __launch_bounds__(NT, 3) k_mb_bwd(
    const float *__restrict__ x, const float *__restrict__ dt, const float *__restrict__ A,
    const float *__restrict__ Bm, const float *__restrict__ Cm, const float *__restrict__ Dk,
    const float *__restrict__ dy, const float *__restrict__ hin, const float *__restrict__ uin,
    float *__restrict__ dx, float *__restrict__ ddt, float *__restrict__ dA,
    float *__restrict__ dB, float *__restrict__ dC, float *__restrict__ dD, MGeo g) {
  extern __shared__ float4 smem4[];
  float *sm = reinterpret_cast<float *>(smem4);
  const int nck = (int)(g.Ls / WB);
  float *ck = sm;                        // [nck][NT]
  float *xs = ck + nck * NT;             // [TB][CH]
  float *ds = xs + TB * CH;
  float *ys = ds + TB * CH;
  float *bs = ys + TB * CH;              // [TB][NL]
  float *cs = bs + TB * NL;
  float *rdx = cs + TB * NL;             // [WB][CH]
  float *rdt = rdx + TB * CH;
  float *rB = rdt + TB * CH;             // [WB][NT/32][NL]
  float *rC = rB + TB * (NT / 32) * NL;
  const Stage st{xs, ds, ys, bs, cs};
  const int tid = threadIdx.x, c = tid / NL, n = tid % NL, warp = tid >> 5;
  const int64_t d0 = (int64_t)blockIdx.x * CH, seg = blockIdx.y, b = blockIdx.z;
  const int64_t d = d0 + c;
  const bool ok = d < g.D && n < g.N;
  const float Av = ok ? A[d * g.N + n] : 0.f;
  const float A2 = Av * LOG2E;
  const float Dd = (Dk && d < g.D) ? Dk[d] : 0.f;
  const int64_t s0 = seg * g.Ls, s1 = s0 + g.Ls < g.L ? s0 + g.Ls : g.L;
  const int nb = (int)((s1 - s0 + WB - 1) / WB);

  // forward over the segment: checkpoint h before every window
  float h = ok ? hin[((b * g.nseg + seg) * g.D + d) * g.N + n] : 0.f;
  for (int k = 0; k < nb; ++k) {
    const int64_t t0 = s0 + (int64_t)k * WB;
    const int len = (int)(s1 - t0 < WB ? s1 - t0 : WB);
    ck[k * NT + tid] = h;
    stage_block(st, x, dt, nullptr, Bm, nullptr, g, b, d0, t0, len);
    __syncthreads();
    for (int i = 0; i < len; ++i) {
      const float de = ds[i * CH + c];
      h = fmaf(exp2f(de * A2), h, de * xs[i * CH + c] * bs[i * NL + n]);
    }
    __syncthreads();
  }

  // windows right to left
  float u = ok ? uin[((b * g.nseg + seg) * g.D + d) * g.N + n] : 0.f;
  float dA_acc = 0.f, dD_acc = 0.f;
  for (int k = nb - 1; k >= 0; --k) {
    const int64_t t0 = s0 + (int64_t)k * WB;
    const int len = (int)(s1 - t0 < WB ? s1 - t0 : WB);
    stage_block(st, x, dt, dy, Bm, Cm, g, b, d0, t0, len);
    __syncthreads();
    const float hstart = ck[k * NT + tid];
    float hs[WB], as[WB];
    {
      float hh = hstart;
#pragma unroll
      for (int i = 0; i < WB; ++i) {
        if (i < len) {
          const float de = ds[i * CH + c];
          as[i] = exp2f(de * A2);
          hh = fmaf(as[i], hh, de * xs[i * CH + c] * bs[i * NL + n]);
        } else {
          as[i] = 1.f;
        }
        hs[i] = hh;
      }
    }
    float vdt[WB], vdx[WB];
#pragma unroll
    for (int i = WB - 1; i >= 0; --i) {
      vdt[i] = 0.f;
      vdx[i] = 0.f;
      if (i < len) {
        const float de = ds[i * CH + c], xv = xs[i * CH + c], dyv = ys[i * CH + c];
        const float Bn = bs[i * NL + n];
        const float gg = ok ? fmaf(cs[i * NL + n], dyv, u) : 0.f;
        const float hp = i > 0 ? hs[i - 1] : hstart;
        const float ahp = as[i] * hp;
        const float gde = gg * de;
        dA_acc = fmaf(gde, ahp, dA_acc);
        vdt[i] = gg * fmaf(Av, ahp, Bn * xv);
        vdx[i] = gde * Bn;
        float pB = gde * xv;
        float pC = ok ? dyv * hs[i] : 0.f;
        pB += __shfl_xor_sync(0xffffffffu, pB, 16);  // the warp's two channels
        pC += __shfl_xor_sync(0xffffffffu, pC, 16);
        if ((tid & 31) < NL) {
          rB[(i * (NT / 32) + warp) * NL + n] = pB;
          rC[(i * (NT / 32) + warp) * NL + n] = pC;
        }
        u = as[i] * gg;
      }
    }
    // reduce-scatter over the half-warp: lane n ends with token n's sums
#pragma unroll
    for (int o = WB / 2; o >= 1; o >>= 1) {
      const bool up = (n & o) != 0;
#pragma unroll
      for (int j = 0; j < o; ++j) {
        const float sdt = up ? vdt[j] : vdt[j + o], kdt = up ? vdt[j + o] : vdt[j];
        const float sdx = up ? vdx[j] : vdx[j + o], kdx = up ? vdx[j + o] : vdx[j];
        vdt[j] = kdt + __shfl_xor_sync(0xffffffffu, sdt, o);
        vdx[j] = kdx + __shfl_xor_sync(0xffffffffu, sdx, o);
      }
    }
    if (n < len) {
      const float dyn = ys[n * CH + c];
      rdx[n * CH + c] = fmaf(Dd, dyn, vdx[0]);
      rdt[n * CH + c] = vdt[0];
      dD_acc = fmaf(dyn, xs[n * CH + c], dD_acc);
    }
    __syncthreads();
    for (int idx = tid; idx < len * CH; idx += NT) {
      const int tt = idx / CH, cc = idx - tt * CH;
      if (d0 + cc < g.D) {
        const int64_t o = (b * g.L + t0 + tt) * g.D + d0 + cc;
        dx[o] = rdx[idx];
        ddt[o] = rdt[idx];
      }
    }
    for (int idx = tid; idx < len * NL; idx += NT) {
      const int tt = idx / NL, nn = idx - tt * NL;
      if (nn < g.N) {
        float sb = 0.f, sc = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NT / 32; ++w2) {
          sb += rB[(tt * (NT / 32) + w2) * NL + nn];
          sc += rC[(tt * (NT / 32) + w2) * NL + nn];
        }
        const int64_t o = (b * g.L + t0 + tt) * g.N + nn;
        atomicAdd(dB + o, sb);
        atomicAdd(dC + o, sc);
      }
    }
    __syncthreads();
  }
  if (ok) atomicAdd(dA + d * g.N + n, dA_acc);
  dD_acc = half_sum(dD_acc);
  if (dD && n == 0 && d < g.D) atomicAdd(dD + d, dD_acc);
}

// ---------------------------------------------------------------------------

namespace {

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); dev = 0; }
  if (dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      v = 0;
    }
    cache[dev] = v > 0 ? v : 148;
  }
  return cache[dev];
}

// Segments: about 640 channel threads per SM in all (the channel kernels'
// CTAs then fit in one wave; measured 3.21 -> 3.11 ms per fwd+bwd step at
// d1024 L8192 against 1024), each segment a multiple of TB tokens and at
// most MAX_LS (the backward's checkpoints live in shared memory).
constexpr int64_t MAX_LS = 1024;

MGeo make_geo(int64_t B, int64_t L, int64_t D, int64_t N) {
  MGeo g;
  g.B = B; g.L = L; g.D = D; g.N = N;
  const int64_t base = B * D;
  const int64_t want = std::max<int64_t>(1, (640 * (int64_t)num_sms()) / base);
  int64_t ls = (L + want - 1) / want;
  ls = (ls + TB - 1) / TB * TB;
  if (ls > MAX_LS) ls = MAX_LS;
  if (ls < TB) ls = TB;
  g.Ls = ls;
  g.nseg = (L + ls - 1) / ls;
  return g;
}

size_t bwd_smem(const MGeo &g) {
  return sizeof(float) * ((size_t)(g.Ls / WB) * NT + 5 * TB * CH + 2 * TB * NL +
                          2 * (size_t)TB * (NT / 32) * NL);
}

}  // namespace

size_t fwd_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N) {
  const MGeo g = make_geo(B, L, D, N);
  return sizeof(float) * (size_t)(g.B * g.nseg * g.D * (g.N + 1));
}

size_t bwd_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N) {
  const MGeo g = make_geo(B, L, D, N);
  return sizeof(float) * (size_t)(g.B * g.nseg * g.D * (2 * g.N + 1));
}

cudaError_t fwd(const float *x, const float *dt, const float *A, const float *Bm, const float *Cm,
                const float *Dk, float *y, int64_t B, int64_t L, int64_t D, int64_t N, void *ws,
                cudaStream_t s) {
  const MGeo g = make_geo(B, L, D, N);
  float *hst = static_cast<float *>(ws);
  float *dsum = hst + g.B * g.nseg * g.D * g.N;
  const dim3 cgrid((unsigned)((D + CCH - 1) / CCH), (unsigned)g.nseg, (unsigned)B);
  {
    LaunchTrace lt("mamba.seg_state", s);
    k_mb_local<false><<<cgrid, CCH, 0, s>>>(x, dt, A, Bm, Cm, nullptr, hst, dsum, g);
  }
  {
    LaunchTrace lt("mamba.seg_scan", s);
    k_mb_scan<false><<<(unsigned)cdiv(B * D * N, 256), 256, 0, s>>>(hst, dsum, A, g);
  }
  {
    LaunchTrace lt("mamba.out", s);
    k_mb_out<<<cgrid, CCH, 0, s>>>(x, dt, A, Bm, Cm, Dk, hst, y, g);
  }
  return cudaGetLastError();
}

cudaError_t bwd(const float *x, const float *dt, const float *A, const float *Bm, const float *Cm,
                const float *Dk, const float *dy, float *dx, float *ddt, float *dA, float *dB,
                float *dC, float *dD, int64_t B, int64_t L, int64_t D, int64_t N, void *ws,
                cudaStream_t s) {
  const MGeo g = make_geo(B, L, D, N);
  const int64_t nst = g.B * g.nseg * g.D * g.N;
  float *hst = static_cast<float *>(ws);
  float *ust = hst + nst;
  float *dsum = ust + nst;
  cudaError_t e;
  if ((e = cudaMemsetAsync(dA, 0, sizeof(float) * D * N, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dB, 0, sizeof(float) * B * L * N, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dC, 0, sizeof(float) * B * L * N, s)) != cudaSuccess) return e;
  if (dD && (e = cudaMemsetAsync(dD, 0, sizeof(float) * D, s)) != cudaSuccess) return e;
  const dim3 grid((unsigned)((D + CH - 1) / CH), (unsigned)g.nseg, (unsigned)B);
  const dim3 cgrid((unsigned)((D + CCH - 1) / CCH), (unsigned)g.nseg, (unsigned)B);
  const unsigned sgrid = (unsigned)cdiv(B * D * N, 256);
  {
    LaunchTrace lt("mamba.seg_state", s);
    k_mb_local<false><<<cgrid, CCH, 0, s>>>(x, dt, A, Bm, Cm, nullptr, hst, dsum, g);
  }
  {
    LaunchTrace lt("mamba.seg_scan", s);
    k_mb_scan<false><<<sgrid, 256, 0, s>>>(hst, dsum, A, g);
  }
  {
    LaunchTrace lt("mamba.seg_grad_state", s);
    k_mb_local<true><<<cgrid, CCH, 0, s>>>(x, dt, A, Bm, Cm, dy, ust, nullptr, g);
  }
  {
    LaunchTrace lt("mamba.seg_scan", s);
    k_mb_scan<true><<<sgrid, 256, 0, s>>>(ust, dsum, A, g);
  }
  const size_t sm = bwd_smem(g);
  if ((e = cudaFuncSetAttribute(k_mb_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) !=
      cudaSuccess)
    return e;
  {
    LaunchTrace lt("mamba.bwd", s);
    k_mb_bwd<<<grid, NT, sm, s>>>(x, dt, A, Bm, Cm, Dk, dy, hst, ust, dx, ddt, dA, dB, dC, dD, g);
  }
  return cudaGetLastError();
}

}  // namespace mamba
}  // namespace ssd
