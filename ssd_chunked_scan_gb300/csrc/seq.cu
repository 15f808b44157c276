// Sequential (chunk = 1) evaluation of the SSD scan: the recurrence taken one
// token at a time, as the step-by-step "scan" implementation of the
// "kernel_ssd_gpu.json" benchmark page does it, with the state held in
// registers for the whole sequence.  All arithmetic is fp32.  It needs no
// workspace in the forward, which suits decoding (a few tokens with the
// state carried in h0 / hT), and it is an independent in-GPU cross-check of
// the chunked kernels.
//
// Every pass is one "sweep" over a dk x dv state X:
//   forward sweep   X_t = exp(la_t) X_{t-1} + u_t w_t^T                (X_{-1} = X0)
//   reverse sweep   X_t = exp(la_{t+1}) X_{t+1} + u_t w_t^T            (X_L = X0,
//                   la_L taken as 0), and finally X <- exp(la_0) X_0
// emitting, after each step, the column reductions z_t = X_t^T p_t
// ([dv], stored and/or dotted with c_t) and the row reductions y_t = X_t r_t
// ([dk], accumulated into a group-shared output with atomic adds).
//
//   fwd:      forward (u, w, p) = (k, v, q):  z = out, final X = hT
//   bwd:      forward (k, v; p = q, r = dout, c = dout): y = dq_h, z.c = out.dout
//             reverse (q, dout; p = k, r = v, c = v):    y = dk_h, z = dv,
//                                                        z.c = dv.v, final X = dh0
//             dla_t = sum_{t' >= t} (out.dout - dv.v)_{t'} + <dhT, hT>
// The last line is the per-head identity q.dq_h - k.dk_h = out.dout - v.dv
// (both sides equal <S_t, q_t dout_t^T> - <G_t, k_t v_t^T>) summed from the
// right, the same reverse cumulative sum the chunked paths use.
//
// Layout of the work: one CTA per (column block of 32 state columns, head,
// batch entry); warp w of the CTA owns state rows 32w .. 32w+31 and lane l
// column 32*blockIdx.x + l, so each thread keeps 32 state elements in
// registers.  Columns of the state never mix, so z needs only a sum over the
// CTA's warps and y a sum over the 32 lanes of a warp (a reduce-scatter by
// shuffles); the y of different column blocks and heads meet in the atomic
// adds.  Tokens are staged through shared memory 32 at a time.
#include <algorithm>

#include "common.cuh"
#include "seq.h"

namespace ssd {
namespace seq {

constexpr int TB = 32;  // tokens staged per block

struct Sweep {
  const float *X0;  // [B,H,dk,dv] initial state, or null (zeros)
  float *Xfin;      // [B,H,dk,dv] final state, or null
  const float *U;   // [B,L,G,dk] row factor of the update
  const float *P;   // [B,L,G,dk] column-reduction weights, or null (no z)
  const float *W;   // [B,L,H,dv] column factor of the update
  const float *R;   // [B,L,H,dv] row-reduction weights, or null (no y)
  const float *Cz;  // [B,L,H,dv] weights of the z dot product, or null
  const float *la;  // [B,L,H]
  float *Z;         // [B,L,H,dv] z, or null (not stored)
  float *Y;         // [B,L,G,dk] y, accumulated (caller zero-fills), or null
  float *E;         // [nblk][B*L*H] per-column-block sum_j z_j c_j, or null
};

__host__ __device__ inline int rup32(int64_t x) { return (int)((x + 31) / 32 * 32); }

size_t sweep_smem(const Geo &g) {
  const int dkp = rup32(g.dk), nw = dkp / 32;
  return sizeof(float) * ((size_t)3 * TB * dkp + 3 * TB * 32 + (size_t)nw * TB * 32 + TB);
}

// grid (ceil(dv/32), H, B), 32 * ceil(dk/32) threads
template <bool REV>
__global__ void __launch_bounds__(128) k_sweep(Sweep a, Geo g) {
  extern __shared__ float4 smem4[];
  float *sm = reinterpret_cast<float *>(smem4);
  const int dkp = rup32(g.dk), nw = dkp / 32;
  float *sU = sm;                  // [TB][dkp]
  float *sP = sU + TB * dkp;       // [TB][dkp]
  float *sY = sP + TB * dkp;       // [TB][dkp]
  float *sW = sY + TB * dkp;       // [TB][32]
  float *sR = sW + TB * 32;        // [TB][32]
  float *sC = sR + TB * 32;        // [TB][32]
  float *sZ = sC + TB * 32;        // [nw][TB][32]
  float *sA = sZ + nw * TB * 32;   // [TB] decay applied at each step
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nth = blockDim.x;
  const int64_t cb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t grp = h / g.hpg, bh = b * g.H + h;
  const int row0 = 32 * warp;
  const int64_t col = cb * 32 + lane;
  const bool colok = col < g.dv;
  const int64_t sz = g.dk * g.dv;
  const bool want_z = a.P != nullptr, want_y = a.R != nullptr;

  float X[32];
#pragma unroll
  for (int ii = 0; ii < 32; ++ii)
    X[ii] = (a.X0 && colok && row0 + ii < g.dk) ? a.X0[bh * sz + (int64_t)(row0 + ii) * g.dv + col]
                                                 : 0.f;

  const int64_t nblk_t = cdiv(g.L, TB);
  for (int64_t blk = 0; blk < nblk_t; ++blk) {
    const int64_t bi = REV ? nblk_t - 1 - blk : blk;
    const int64_t t0 = bi * TB;
    const int len = (int)(g.L - t0 < TB ? g.L - t0 : TB);
    for (int idx = tid; idx < TB * dkp; idx += nth) {
      const int tt = idx / dkp, i = idx - tt * dkp;
      const bool ok = tt < len && i < g.dk;
      const int64_t o = qk_off(g, b, t0 + tt, grp) + i;
      sU[idx] = ok ? a.U[o] : 0.f;
      if (want_z) sP[idx] = ok ? a.P[o] : 0.f;
    }
    for (int idx = tid; idx < TB * 32; idx += nth) {
      const int tt = idx >> 5, j = idx & 31;
      const int64_t c = cb * 32 + j;
      const bool ok = tt < len && c < g.dv;
      const int64_t o = v_off(g, b, t0 + tt, h) + c;
      sW[idx] = ok ? a.W[o] : 0.f;
      if (want_y) sR[idx] = ok ? a.R[o] : 0.f;
      if (a.Cz) sC[idx] = ok ? a.Cz[o] : 0.f;
    }
    for (int tt = tid; tt < TB; tt += nth) {
      float d = 1.f;
      if (tt < len) {
        const int64_t t = t0 + tt + (REV ? 1 : 0);
        if (t < g.L) d = expf(a.la[la_off(g, b, t, h)]);
      }
      sA[tt] = d;
    }
    __syncthreads();

    for (int s = 0; s < len; ++s) {
      const int tt = REV ? len - 1 - s : s;
      const float d = sA[tt];
      const float w = sW[tt * 32 + lane];
      const float4 *u4 = reinterpret_cast<const float4 *>(sU + tt * dkp + row0);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 u = u4[q4];
        X[4 * q4 + 0] = fmaf(d, X[4 * q4 + 0], u.x * w);
        X[4 * q4 + 1] = fmaf(d, X[4 * q4 + 1], u.y * w);
        X[4 * q4 + 2] = fmaf(d, X[4 * q4 + 2], u.z * w);
        X[4 * q4 + 3] = fmaf(d, X[4 * q4 + 3], u.w * w);
      }
      if (want_z) {
        const float4 *p4 = reinterpret_cast<const float4 *>(sP + tt * dkp + row0);
        float z0 = 0.f, z1 = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 p = p4[q4];
          z0 = fmaf(X[4 * q4 + 0], p.x, z0);
          z1 = fmaf(X[4 * q4 + 1], p.y, z1);
          z0 = fmaf(X[4 * q4 + 2], p.z, z0);
          z1 = fmaf(X[4 * q4 + 3], p.w, z1);
        }
        sZ[(warp * TB + tt) * 32 + lane] = z0 + z1;
      }
      if (want_y) {
        // y_i = sum over the warp's 32 columns of X[i][j] r_j: reduce-scatter
        // so that lane l ends with row row0 + l
        const float r = sR[tt * 32 + lane];
        float v[32];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) v[ii] = X[ii] * r;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int ii = 0; ii < o; ++ii) {
            const float send = up ? v[ii] : v[ii + o];
            const float keep = up ? v[ii + o] : v[ii];
            v[ii] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        sY[tt * dkp + row0 + lane] = v[0];
      }
    }
    __syncthreads();

    if (want_z) {
      for (int tt = warp; tt < len; tt += nw) {
        float z = 0.f;
        for (int w2 = 0; w2 < nw; ++w2) z += sZ[(w2 * TB + tt) * 32 + lane];
        if (a.Z && colok) a.Z[v_off(g, b, t0 + tt, h) + col] = z;
        if (a.E) {
          float e = colok ? z * sC[tt * 32 + lane] : 0.f;
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
          if (lane == 0) a.E[cb * (g.B * g.L * g.H) + la_off(g, b, t0 + tt, h)] = e;
        }
      }
    }
    if (want_y) {
      for (int idx = tid; idx < len * dkp; idx += nth) {
        const int tt = idx / dkp, i = idx - tt * dkp;
        if (i < g.dk) atomicAdd(a.Y + qk_off(g, b, t0 + tt, grp) + i, sY[idx]);
      }
    }
    __syncthreads();  // the staging buffers are refilled next
  }

  if (REV) {
    const float d0 = expf(a.la[la_off(g, b, 0, h)]);
#pragma unroll
    for (int ii = 0; ii < 32; ++ii) X[ii] *= d0;
  }
  if (a.Xfin && colok) {
#pragma unroll
    for (int ii = 0; ii < 32; ++ii)
      if (row0 + ii < g.dk) a.Xfin[bh * sz + (int64_t)(row0 + ii) * g.dv + col] = X[ii];
  }
}

// dla[t] = sum_{t' >= t} sum_cb (E1 - E2)[cb][t'] + <dhT, hT>, the reverse
// sum carried in fp64.  grid (B*H), 256 threads.
constexpr int DT = 256;
__global__ void __launch_bounds__(DT) k_seq_dla(const float *__restrict__ E1,
                                                const float *__restrict__ E2, int nblk,
                                                const float *__restrict__ dhT,
                                                const float *__restrict__ hT,
                                                float *__restrict__ dla, Geo g) {
  __shared__ double wred[DT / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bh = blockIdx.x, b = bh / g.H, h = bh % g.H;
  const int64_t BLH = g.B * g.L * g.H;
  double part = 0.0;
  if (dhT) {
    const int64_t sz = g.dk * g.dv;
    for (int64_t e = tid; e < sz; e += DT) part += (double)dhT[bh * sz + e] * (double)hT[bh * sz + e];
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) wred[warp] = part;
  __syncthreads();
  double carry = 0.0;
#pragma unroll
  for (int w2 = 0; w2 < DT / 32; ++w2) carry += wred[w2];
  __syncthreads();
  for (int64_t hi = g.L; hi > 0; hi -= DT) {
    const int64_t t = hi - DT + tid;
    const bool ok = t >= 0;
    const int64_t idx = la_off(g, b, ok ? t : 0, h);
    double x = 0.0;
    if (ok)
      for (int c = 0; c < nblk; ++c) x += (double)E1[c * BLH + idx] - (double)E2[c * BLH + idx];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {  // inclusive suffix sum within the warp
      const double y = __shfl_down_sync(0xffffffffu, x, o);
      if (lane + o < 32) x += y;
    }
    if (lane == 0) wred[warp] = x;
    __syncthreads();
    double after = carry;
#pragma unroll
    for (int w2 = 0; w2 < DT / 32; ++w2)
      if (w2 > warp) after += wred[w2];
    if (ok) dla[idx] = (float)(x + after);
#pragma unroll
    for (int w2 = 0; w2 < DT / 32; ++w2) carry += wred[w2];
    __syncthreads();
  }
}

namespace {

template <bool REV>
cudaError_t launch_sweep(const Sweep &a, const Geo &g, cudaStream_t s, const char *name) {
  const size_t sm = sweep_smem(g);
  cudaError_t e =
      cudaFuncSetAttribute(k_sweep<REV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)cdiv(g.dv, 32), (unsigned)g.H, (unsigned)g.B);
  LaunchTrace lt(name, s);
  k_sweep<REV><<<grid, rup32(g.dk), sm, s>>>(a, g);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_workspace_bytes(const Geo &) { return 0; }

// Per-column-block dot products of both sweeps, and the final state (used only
// when it has a cotangent).
size_t bwd_workspace_bytes(const Geo &g) {
  const int64_t nblk = cdiv(g.dv, 32);
  return sizeof(float) * (size_t)(2 * nblk * g.B * g.L * g.H + g.B * g.H * g.dk * g.dv);
}

cudaError_t fwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                float *out, float *hT, const Geo &g, cudaStream_t s) {
  Sweep a{h0, hT, k, q, v, nullptr, nullptr, la, out, nullptr, nullptr};
  return launch_sweep<false>(a, g, s, "seq.sweep_out");
}

cudaError_t bwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                const float *dout, const float *dhT, float *dq, float *dk, float *dv, float *dla,
                float *dh0, const Geo &g, void *ws, cudaStream_t s) {
  const int64_t nblk = cdiv(g.dv, 32), BLH = g.B * g.L * g.H;
  float *E1 = static_cast<float *>(ws);
  float *E2 = E1 + nblk * BLH;
  float *hT = dhT ? E2 + nblk * BLH : nullptr;
  cudaError_t e;
  const size_t qk_bytes = sizeof(float) * (size_t)(g.B * g.L * g.G * g.dk);
  if ((e = cudaMemsetAsync(dq, 0, qk_bytes, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dk, 0, qk_bytes, s)) != cudaSuccess) return e;
  Sweep f{h0, hT, k, q, v, dout, dout, la, nullptr, dq, E1};
  if ((e = launch_sweep<false>(f, g, s, "seq.sweep_dq")) != cudaSuccess) return e;
  Sweep r{dhT, dh0, q, k, dout, v, v, la, dv, dk, E2};
  if ((e = launch_sweep<true>(r, g, s, "seq.sweep_dkdv")) != cudaSuccess) return e;
  {
    LaunchTrace lt("seq.dla", s);
    k_seq_dla<<<(unsigned)(g.B * g.H), DT, 0, s>>>(E1, E2, (int)nblk, dhT, hT, dla, g);
  }
  return cudaGetLastError();
}

}  // namespace seq
}  // namespace ssd
