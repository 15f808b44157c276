// All-fp32 CUDA-core ("SIMT") path of the chunked SSD scan.
//
// Chunked evaluation of S_t = exp(la_t) S_{t-1} + k_t v_t^T, out_t = S_t^T q_t
// (the op of the "kernel_ssd_gpu.json" benchmark page, impl "chunked").  For a
// chunk c of tokens [t0, t0 + len) with in-chunk log-decay prefix cs_t and
// total A_c = cs_{last}:
//
//   chunk state   S_c     = sum_s exp(A_c - cs_s) k_s v_s^T
//   state passing H_c     = exp(A_c) H_{c-1} + S_c          (H_{-1} = h0)
//   output        out_t   = sum_{s<=t} exp(cs_t - cs_s) (q_t.k_s) v_s
//                           + exp(cs_t) H_{c-1}^T q_t
//
// and for the backward, with dX_c the gradient of the state at the end of
// chunk c (dX_{N-1} = 0, dX_{c-1} = exp(A_c) dX_c + sum_t exp(cs_t) q_t dout_t^T,
// dh0 = dX_{-1}):
//
//   dq_t = sum_{s<=t} D_ts (dout_t.v_s) k_s + exp(cs_t) H_{c-1} dout_t
//   dk_s = sum_{t>=s} D_ts (dout_t.v_s) q_t + exp(A_c - cs_s) dX_c v_s
//   dv_s = sum_{t>=s} D_ts (q_t.k_s) dout_t + exp(A_c - cs_s) dX_c^T k_s
//   dla_t = sum_{t'>=t} (q_t'.dq_t' - k_t'.dk_t')   (per head, before the
//                                                     sum over a group's heads)
//
// with D_ts = exp(cs_t - cs_s) for s <= t.  Every decay factor is formed as
// exp of a non-positive difference, so none overflows.
//
// Kernels use a 256-thread CTA whose threads form a 16 x 16 grid; thread
// (ty, tx) owns rows 64a + 4ty + r and columns 64b + 4tx + c of each output
// tile.  Operands are staged through shared memory in slices of KS reduction
// indices, "reduction-major" ([k][m]), so the inner loop is two float4
// shared-memory loads per 16..64 FFMAs.
#include "common.cuh"
#include "simt.h"

namespace ssd {
namespace simt {

constexpr int NT = 256;
constexpr int KS = 32;
constexpr int CMAX = 64;
constexpr int LDT = CMAX + 4;  // leading dimension of [*][token] tiles

__host__ __device__ constexpr int ldn(int nb) { return 64 * nb + 4; }

// Stage dst[kk * ld + m] = src(k0 + kk, m) * kscale[kk] * mscale[m] for
// kk < KS, m < ld, zero outside kk < kmax - k0, m < mmax.  src(k, m) =
// src[k * sk + m * sm]; avail: elements from src to the end of its buffer
// (debug-build index checks).  MCONTIG selects which index consecutive threads walk
// (the one that is contiguous in global memory).
// Each thread issues the global loads of U elements before it stores any of
// them, so a stage costs about one memory round trip per U elements (16 by
// default; 8 in the output kernel, which then keeps three CTAs per SM).
constexpr int SU_ST = 16;
template <bool MCONTIG, int U = SU_ST>
__device__ inline void stage(float *__restrict__ dst, int ld, const float *__restrict__ src,
                             int64_t avail, int64_t sk, int64_t sm, int k0, int kmax, int mmax,
                             const float *kscale, const float *mscale) {
  const int total = KS * ld;
  for (int base = threadIdx.x; base < total; base += U * NT) {
    float x[U];
    int kk[U], m[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * NT;
      if (MCONTIG) { kk[u] = idx / ld; m[u] = idx - kk[u] * ld; }
      else { m[u] = idx / KS; kk[u] = idx - m[u] * KS; }
      const int kg = k0 + kk[u];
      x[u] = (idx < total && kg < kmax && m[u] < mmax) ? LDC(src, (int64_t)kg * sk + (int64_t)m[u] * sm, avail) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * NT;
      if (idx < total) {
        const int kg = k0 + kk[u];
        float v = x[u];
        if (kg < kmax && m[u] < mmax) {
          if (kscale) v *= kscale[kg];
          if (mscale) v *= mscale[m[u]];
        }
        dst[kk[u] * ld + m[u]] = v;
      }
    }
  }
}

template <int MA, int NB>
__device__ inline void zero_acc(float (&acc)[4 * MA][4 * NB]) {
#pragma unroll
  for (int r = 0; r < 4 * MA; ++r)
#pragma unroll
    for (int c = 0; c < 4 * NB; ++c) acc[r][c] = 0.f;
}

// acc[m][n] += sum_{kk < kcnt} As[kk][m] * Bs[kk][n]
template <int MA, int NB>
__device__ inline void mma_slice(float (&acc)[4 * MA][4 * NB], const float *__restrict__ As, int lda,
                                 const float *__restrict__ Bs, int ldb, int kcnt) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
  for (int kk = 0; kk < kcnt; ++kk) {
    float a[4 * MA], b[4 * NB];
#pragma unroll
    for (int ma = 0; ma < MA; ++ma) {
      float4 x = *reinterpret_cast<const float4 *>(As + kk * lda + 64 * ma + 4 * ty);
      a[4 * ma + 0] = x.x; a[4 * ma + 1] = x.y; a[4 * ma + 2] = x.z; a[4 * ma + 3] = x.w;
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float4 x = *reinterpret_cast<const float4 *>(Bs + kk * ldb + 64 * nb + 4 * tx);
      b[4 * nb + 0] = x.x; b[4 * nb + 1] = x.y; b[4 * nb + 2] = x.z; b[4 * nb + 3] = x.w;
    }
#pragma unroll
    for (int r = 0; r < 4 * MA; ++r)
#pragma unroll
      for (int c = 0; c < 4 * NB; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}

__device__ inline int row_of(int r) { return 64 * (r >> 2) + 4 * (threadIdx.x >> 4) + (r & 3); }
__device__ inline int col_of(int c) { return 64 * (c >> 2) + 4 * (threadIdx.x & 15) + (c & 3); }

// ---------------------------------------------------------------------------
// Chunk-state contraction, two uses:
//   QUERY = false:  states[c] = sum_s k_s (exp(A_c - cs_s) v_s)^T , Adec[c] = A_c
//   QUERY = true :  states[c] = sum_t q_t (exp(cs_t) dout_t)^T
// grid (N, H, B)
template <int MA, int NB, bool QUERY>
__global__ void __launch_bounds__(NT) k_chunk_state(const float *__restrict__ X,
                                                    const float *__restrict__ Y,
                                                    const float *__restrict__ la,
                                                    float *__restrict__ states,
                                                    float *__restrict__ Adec, Geo g) {
  __shared__ float cs[CMAX], sc[CMAX];
  __shared__ __align__(16) float As[KS * ldn(MA)];
  __shared__ __align__(16) float Bs[KS * ldn(NB)];
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t grp = h / g.hpg, bh = b * g.H + h;
  const int64_t t0 = c * g.C;
  const int len = (int)(g.L - t0 < g.C ? g.L - t0 : g.C);
  chunk_cumsum64(la, n_la(g), la_off(g, b, t0, h), g.H, len, cs);
  const float A = cs[len - 1];
  if (threadIdx.x < len) sc[threadIdx.x] = QUERY ? expf(cs[threadIdx.x]) : expf(A - cs[threadIdx.x]);
  if (!QUERY && threadIdx.x == 0) STC(Adec, bh * g.N + c, g.B * g.H * g.N, A);
  __syncthreads();

  float acc[4 * MA][4 * NB];
  zero_acc<MA, NB>(acc);
  const float *xs = X + qk_off(g, b, t0, grp);
  const float *ys = Y + v_off(g, b, t0, h);
  const int64_t ax = n_qk(g) - qk_off(g, b, t0, grp), ay = n_v(g) - v_off(g, b, t0, h);
  for (int k0 = 0; k0 < len; k0 += KS) {
    stage<true>(As, ldn(MA), xs, ax, g.G * g.dk, 1, k0, len, (int)g.dk, nullptr, nullptr);
    stage<true>(Bs, ldn(NB), ys, ay, g.H * g.dv, 1, k0, len, (int)g.dv, sc, nullptr);
    __syncthreads();
    mma_slice<MA, NB>(acc, As, ldn(MA), Bs, ldn(NB), min(KS, len - k0));
    __syncthreads();
  }
  const int64_t dst = st_off(g, bh, c), nst = n_st(g);
#pragma unroll
  for (int r = 0; r < 4 * MA; ++r) {
    const int i = row_of(r);
    if (i >= g.dk) continue;
#pragma unroll
    for (int cc = 0; cc < 4 * NB; ++cc) {
      const int j = col_of(cc);
      if (j < g.dv) STC(states, dst + (int64_t)i * g.dv + j, nst, acc[r][cc]);
    }
  }
}

// ---------------------------------------------------------------------------
// State passing, in place.  Forward: states[c] <- H_{c-1} (the state entering
// chunk c), from contributions S_c; the state after the last chunk goes to fin
// when given.  Reverse: states[c] <- dX_c (gradient of the state leaving chunk
// c), from query contributions, starting from dX_{N-1} = dfin (the cotangent
// of the final state, zero when NULL); dh0 <- dX_{-1}.
// Each thread owns V consecutive state elements (V = 4: one float4, when
// dk*dv is a multiple of 4) and loads SCU chunks' values ahead of the
// dependent chain, so a pass costs about one memory round trip per SCU chunks.
// grid (B*H, ceil(dk*dv / (V*NT)))
constexpr int SCU = 8;

// (a: element offset into p's buffer of n elements, a multiple of V)
template <int V>
__device__ inline void ld_v(float (&x)[V], const float *p, int64_t a, int64_t n) {
  if constexpr (V == 4) {
    const float4 f = LDC(reinterpret_cast<const float4 *>(p), a / 4, n / 4);
    x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
  } else {
    x[0] = LDC(p, a, n);
  }
}
template <int V>
__device__ inline void st_v(float *p, int64_t a, int64_t n, const float (&x)[V]) {
  if constexpr (V == 4) STC(reinterpret_cast<float4 *>(p), a / 4, n / 4, make_float4(x[0], x[1], x[2], x[3]));
  else STC(p, a, n, x[0]);
}

template <int V, bool REV>
__global__ void __launch_bounds__(NT) k_scan(float *__restrict__ states,
                                             const float *__restrict__ Adec,
                                             const float *__restrict__ init,
                                             float *__restrict__ fin, Geo g) {
  const int64_t bh = blockIdx.x;
  const int64_t e0 = (int64_t)V * ((int64_t)blockIdx.y * NT + threadIdx.x);
  const int64_t sz = g.dk * g.dv;
  if (e0 >= sz) return;
  float run[V];
#pragma unroll
  for (int j = 0; j < V; ++j) run[j] = init ? LDC(init, bh * sz + e0 + j, n_h(g)) : 0.f;
  const int64_t p0 = st_off(g, bh, 0) + e0, nst = n_st(g);
  const float *a = Adec + bh * g.N;
  for (int64_t k0 = 0; k0 < g.N; k0 += SCU) {
    float x[SCU][V], d[SCU];
#pragma unroll
    for (int u = 0; u < SCU; ++u) {
      const int64_t k = k0 + u;
      if (k < g.N) {
        const int64_t c = REV ? g.N - 1 - k : k;
        ld_v<V>(x[u], states, p0 + c * sz, nst);
        d[u] = expf(LDC(a, c, g.N));
      }
    }
#pragma unroll
    for (int u = 0; u < SCU; ++u) {
      const int64_t k = k0 + u;
      if (k < g.N) {
        const int64_t c = REV ? g.N - 1 - k : k;
        st_v<V>(states, p0 + c * sz, nst, run);
#pragma unroll
        for (int j = 0; j < V; ++j) run[j] = fmaf(d[u], run[j], x[u][j]);
      }
    }
  }
  if (fin) {
#pragma unroll
    for (int j = 0; j < V; ++j) STC(fin, bh * sz + e0 + j, n_h(g), run[j]);
  }
}

template <bool REV>
static void launch_scan(float *st, const float *Adec, const float *init, float *fin,
                        const Geo &g, cudaStream_t s, const char *name) {
  const int64_t sz = g.dk * g.dv;
  LaunchTrace lt(name, s);
  if (sz % 4 == 0) {
    const dim3 grid((unsigned)(g.B * g.H), (unsigned)cdiv(sz, 4 * NT));
    k_scan<4, REV><<<grid, NT, 0, s>>>(st, Adec, init, fin, g);
  } else {
    const dim3 grid((unsigned)(g.B * g.H), (unsigned)cdiv(sz, NT));
    k_scan<1, REV><<<grid, NT, 0, s>>>(st, Adec, init, fin, g);
  }
}

// ---------------------------------------------------------------------------
// Raw q.k scores of one chunk into registers: acc[t][s] (rows t, cols s).
template <int U = SU_ST>
// (aqk: elements from qs, and from ks, to the ends of their buffers)
__device__ inline void chunk_scores(float (&acc)[4][4], const float *qs, const float *ks, int64_t aqk,
                                    float *As, float *Bs, const Geo &g, int len) {
  zero_acc<1, 1>(acc);
  for (int i0 = 0; i0 < g.dk; i0 += KS) {
    stage<false, U>(As, LDT, qs + i0, aqk - i0, 1, g.G * g.dk, 0, (int)g.dk - i0, len, nullptr, nullptr);
    stage<false, U>(Bs, LDT, ks + i0, aqk - i0, 1, g.G * g.dk, 0, (int)g.dk - i0, len, nullptr, nullptr);
    __syncthreads();
    mma_slice<1, 1>(acc, As, LDT, Bs, LDT, min(KS, (int)g.dk - i0));
    __syncthreads();
  }
}

// Output of one chunk for one head.  grid (N, H, B)
template <int NB>
__global__ void __launch_bounds__(NT) k_chunk_out(const float *__restrict__ q,
                                                  const float *__restrict__ k,
                                                  const float *__restrict__ v,
                                                  const float *__restrict__ la,
                                                  const float *__restrict__ states,
                                                  float *__restrict__ out, Geo g) {
  __shared__ float cs[CMAX], ecs[CMAX];
  __shared__ __align__(16) float Pt[CMAX * LDT];  // [s][t]
  __shared__ __align__(16) float As[KS * LDT];
  __shared__ __align__(16) float Bs[KS * ldn(NB)];
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t grp = h / g.hpg, bh = b * g.H + h;
  const int64_t t0 = c * g.C;
  const int len = (int)(g.L - t0 < g.C ? g.L - t0 : g.C);
  chunk_cumsum64(la, n_la(g), la_off(g, b, t0, h), g.H, len, cs);
  if (threadIdx.x < len) ecs[threadIdx.x] = expf(cs[threadIdx.x]);
  const float *qs = q + qk_off(g, b, t0, grp);
  const float *ks = k + qk_off(g, b, t0, grp);
  const int64_t aqk = n_qk(g) - qk_off(g, b, t0, grp), av = n_v(g) - v_off(g, b, t0, h);
  const int64_t ast = n_st(g) - st_off(g, bh, c);

  float sc[4][4];
  chunk_scores<8>(sc, qs, ks, aqk, As, Bs, g, len);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = row_of(r);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int s = col_of(cc);
      float p = 0.f;
      if (t < len && s <= t) p = expf(cs[t] - cs[s]) * sc[r][cc];
      Pt[s * LDT + t] = p;
    }
  }
  __syncthreads();

  float acc[4][4 * NB];
  zero_acc<1, NB>(acc);
  const float *vs = v + v_off(g, b, t0, h);
  for (int s0 = 0; s0 < len; s0 += KS) {
    stage<true, 8>(Bs, ldn(NB), vs, av, g.H * g.dv, 1, s0, len, (int)g.dv, nullptr, nullptr);
    __syncthreads();
    mma_slice<1, NB>(acc, Pt + s0 * LDT, LDT, Bs, ldn(NB), min(KS, len - s0));
    __syncthreads();
  }
  const float *Hs = states + st_off(g, bh, c);
  for (int i0 = 0; i0 < g.dk; i0 += KS) {
    stage<false, 8>(As, LDT, qs + i0, aqk - i0, 1, g.G * g.dk, 0, (int)g.dk - i0, len, nullptr, ecs);
    stage<true, 8>(Bs, ldn(NB), Hs + (int64_t)i0 * g.dv, ast - (int64_t)i0 * g.dv, g.dv, 1, 0, (int)g.dk - i0,
                   (int)g.dv, nullptr, nullptr);
    __syncthreads();
    mma_slice<1, NB>(acc, As, LDT, Bs, ldn(NB), min(KS, (int)g.dk - i0));
    __syncthreads();
  }
  const int64_t os = v_off(g, b, t0, h), nv = n_v(g);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = row_of(r);
    if (t >= len) continue;
#pragma unroll
    for (int cc = 0; cc < 4 * NB; ++cc) {
      const int j = col_of(cc);
      if (j < g.dv) STC(out, os + (int64_t)t * g.H * g.dv + j, nv, acc[r][cc]);
    }
  }
}

// Row dot products of a register tile with a global [row][col] matrix (ax
// elements from x to the end of its buffer), reduced over the 16 threads that
// share the rows; written to dst[row].
template <int NB>
__device__ inline void row_dots(const float (&acc)[4][4 * NB], const float *x, int64_t ax, int64_t ldx,
                                int len, int ncols, float *dst) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = row_of(r);
    float s = 0.f;
    if (t < len) {
#pragma unroll
      for (int cc = 0; cc < 4 * NB; ++cc) {
        const int i = col_of(cc);
        if (i < ncols) s = fmaf(LDC(x, (int64_t)t * ldx + i, ax), acc[r][cc], s);
      }
    }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 15) == 0 && t < len) dst[t] = s;
  }
}

// Store (first head of the group) or add (later heads) a register tile (ad
// elements from dst to the end of its buffer).
template <int NB>
__device__ inline void store_or_add(const float (&acc)[4][4 * NB], float *dst, int64_t ad, int64_t ldd,
                                    int len, int ncols, bool add) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = row_of(r);
    if (t >= len) continue;
#pragma unroll
    for (int cc = 0; cc < 4 * NB; ++cc) {
      const int i = col_of(cc);
      if (i < ncols) {
        const int64_t o = (int64_t)t * ldd + i;
        STC(dst, o, ad, add ? LDC(dst, o, ad) + acc[r][cc] : acc[r][cc]);
      }
    }
  }
}

// Gradients of one chunk for all heads of one group.  grid (N, G, B)
// Hst holds H_{c-1} per chunk, dXst holds dX_c per chunk.  dq / dk are
// accumulated over the group's heads in a fixed order.  dla receives the
// in-chunk reverse cumulative sums; dcs_sum[bh*N + c] the chunk totals.
template <int NBK, int NBV>
__global__ void __launch_bounds__(NT, 2) k_chunk_grad(
    const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
    const float *__restrict__ la, const float *__restrict__ dout, const float *__restrict__ Hst,
    const float *__restrict__ dXst, float *__restrict__ dq, float *__restrict__ dk,
    float *__restrict__ dv, float *__restrict__ dla, float *__restrict__ dcs_sum, Geo g) {
  extern __shared__ __align__(16) float smem[];
  float *Pm = smem;                   // [t][s]  decayed, masked scores
  float *dPm = Pm + CMAX * LDT;       // [t][s]  decayed, masked dout.v
  float *dPmT = dPm + CMAX * LDT;     // [s][t]
  float *As = dPmT + CMAX * LDT;      // [KS][LDT]
  float *Bs = As + KS * LDT;          // [KS][ldn(max(NBK,NBV))]
  constexpr int NBM = NBK > NBV ? NBK : NBV;
  float *cs = Bs + KS * ldn(NBM);
  float *w = cs + CMAX, *e = w + CMAX, *dcq = e + CMAX, *dck = dcq + CMAX;

  const int64_t c = blockIdx.x, grp = blockIdx.y, b = blockIdx.z;
  const int64_t t0 = c * g.C;
  const int len = (int)(g.L - t0 < g.C ? g.L - t0 : g.C);
  const int64_t ldqk = g.G * g.dk, ldv = g.H * g.dv;
  const float *qs = q + qk_off(g, b, t0, grp);
  const float *ks = k + qk_off(g, b, t0, grp);
  float *dqs = dq + qk_off(g, b, t0, grp);
  float *dks = dk + qk_off(g, b, t0, grp);
  const int64_t aqk = n_qk(g) - qk_off(g, b, t0, grp);

  float sraw[4][4];
  chunk_scores(sraw, qs, ks, aqk, As, Bs, g, len);

  for (int hh = 0; hh < g.hpg; ++hh) {
    const int64_t h = grp * g.hpg + hh, bh = b * g.H + h;
    chunk_cumsum64(la, n_la(g), la_off(g, b, t0, h), g.H, len, cs);
    const float A = cs[len - 1];
    if (threadIdx.x < len) {
      w[threadIdx.x] = expf(A - cs[threadIdx.x]);
      e[threadIdx.x] = expf(cs[threadIdx.x]);
    }
    const float *vs = v + v_off(g, b, t0, h);
    const float *dos = dout + v_off(g, b, t0, h);
    const float *Hc = Hst + st_off(g, bh, c);
    const float *dXc = dXst + st_off(g, bh, c);
    const int64_t av = n_v(g) - v_off(g, b, t0, h), ast = n_st(g) - st_off(g, bh, c);

    // dP[t][s] = dout_t . v_s, then the decayed, causally masked tiles
    {
      float dp[4][4];
      zero_acc<1, 1>(dp);
      for (int j0 = 0; j0 < g.dv; j0 += KS) {
        stage<false>(As, LDT, dos + j0, av - j0, 1, ldv, 0, (int)g.dv - j0, len, nullptr, nullptr);
        stage<false>(Bs, LDT, vs + j0, av - j0, 1, ldv, 0, (int)g.dv - j0, len, nullptr, nullptr);
        __syncthreads();
        mma_slice<1, 1>(dp, As, LDT, Bs, LDT, min(KS, (int)g.dv - j0));
        __syncthreads();
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int t = row_of(r);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int s = col_of(cc);
          float d = 0.f;
          if (t < len && s <= t) d = expf(cs[t] - cs[s]);
          Pm[t * LDT + s] = d * sraw[r][cc];
          dPm[t * LDT + s] = d * dp[r][cc];
          dPmT[s * LDT + t] = d * dp[r][cc];
        }
      }
      __syncthreads();
    }

    // dq_h[t][i] = sum_s dPm[t][s] k_s[i] + e_t sum_j dout_t[j] H[i][j]
    {
      float acc[4][4 * NBK];
      zero_acc<1, NBK>(acc);
      for (int s0 = 0; s0 < len; s0 += KS) {
        stage<true>(Bs, ldn(NBK), ks, aqk, ldqk, 1, s0, len, (int)g.dk, nullptr, nullptr);
        __syncthreads();
        mma_slice<1, NBK>(acc, dPmT + s0 * LDT, LDT, Bs, ldn(NBK), min(KS, len - s0));
        __syncthreads();
      }
      for (int j0 = 0; j0 < g.dv; j0 += KS) {
        stage<false>(As, LDT, dos + j0, av - j0, 1, ldv, 0, (int)g.dv - j0, len, nullptr, e);
        stage<false>(Bs, ldn(NBK), Hc + j0, ast - j0, 1, g.dv, 0, (int)g.dv - j0, (int)g.dk, nullptr, nullptr);
        __syncthreads();
        mma_slice<1, NBK>(acc, As, LDT, Bs, ldn(NBK), min(KS, (int)g.dv - j0));
        __syncthreads();
      }
      row_dots<NBK>(acc, qs, aqk, ldqk, len, (int)g.dk, dcq);
      store_or_add<NBK>(acc, dqs, aqk, ldqk, len, (int)g.dk, hh > 0);
    }

    // dk_h[s][i] = sum_t dPm[t][s] q_t[i] + w_s sum_j v_s[j] dX[i][j]
    {
      float acc[4][4 * NBK];
      zero_acc<1, NBK>(acc);
      for (int r0 = 0; r0 < len; r0 += KS) {
        stage<true>(Bs, ldn(NBK), qs, aqk, ldqk, 1, r0, len, (int)g.dk, nullptr, nullptr);
        __syncthreads();
        mma_slice<1, NBK>(acc, dPm + r0 * LDT, LDT, Bs, ldn(NBK), min(KS, len - r0));
        __syncthreads();
      }
      for (int j0 = 0; j0 < g.dv; j0 += KS) {
        stage<false>(As, LDT, vs + j0, av - j0, 1, ldv, 0, (int)g.dv - j0, len, nullptr, w);
        stage<false>(Bs, ldn(NBK), dXc + j0, ast - j0, 1, g.dv, 0, (int)g.dv - j0, (int)g.dk, nullptr, nullptr);
        __syncthreads();
        mma_slice<1, NBK>(acc, As, LDT, Bs, ldn(NBK), min(KS, (int)g.dv - j0));
        __syncthreads();
      }
      row_dots<NBK>(acc, ks, aqk, ldqk, len, (int)g.dk, dck);
      store_or_add<NBK>(acc, dks, aqk, ldqk, len, (int)g.dk, hh > 0);
    }

    // dv[s][j] = sum_t Pm[t][s] dout_t[j] + w_s sum_i k_s[i] dX[i][j]
    {
      float acc[4][4 * NBV];
      zero_acc<1, NBV>(acc);
      for (int r0 = 0; r0 < len; r0 += KS) {
        stage<true>(Bs, ldn(NBV), dos, av, ldv, 1, r0, len, (int)g.dv, nullptr, nullptr);
        __syncthreads();
        mma_slice<1, NBV>(acc, Pm + r0 * LDT, LDT, Bs, ldn(NBV), min(KS, len - r0));
        __syncthreads();
      }
      for (int i0 = 0; i0 < g.dk; i0 += KS) {
        stage<false>(As, LDT, ks + i0, aqk - i0, 1, ldqk, 0, (int)g.dk - i0, len, nullptr, w);
        stage<true>(Bs, ldn(NBV), dXc + (int64_t)i0 * g.dv, ast - (int64_t)i0 * g.dv, g.dv, 1, 0, (int)g.dk - i0,
                    (int)g.dv, nullptr, nullptr);
        __syncthreads();
        mma_slice<1, NBV>(acc, As, LDT, Bs, ldn(NBV), min(KS, (int)g.dk - i0));
        __syncthreads();
      }
      store_or_add<NBV>(acc, dv + v_off(g, b, t0, h), av, ldv, len, (int)g.dv, false);
    }
    __syncthreads();

    // in-chunk reverse cumulative sum of dcs_t = q_t.dq_h[t] - k_t.dk_h[t]
    if (threadIdx.x < 32) {
      const int l = threadIdx.x;
      // lane l owns steps 2l, 2l+1; reverse inclusive scan over lanes
      double x0 = (2 * l < len) ? (double)dcq[2 * l] - (double)dck[2 * l] : 0.0;
      double x1 = (2 * l + 1 < len) ? (double)dcq[2 * l + 1] - (double)dck[2 * l + 1] : 0.0;
      double pair = x0 + x1, incl = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        double y = __shfl_down_sync(0xffffffffu, incl, o);
        if (l + o < 32) incl += y;
      }
      double after = incl - pair;  // sum over steps > 2l+1
      const int64_t dl = la_off(g, b, t0, h), nla = n_la(g);
      if (2 * l < len) STC(dla, dl + (int64_t)(2 * l) * g.H, nla, (float)(after + pair));
      if (2 * l + 1 < len) STC(dla, dl + (int64_t)(2 * l + 1) * g.H, nla, (float)(after + x1));
      if (l == 0) STC(dcs_sum, bh * g.N + c, g.B * g.H * g.N, (float)incl);
    }
    __syncthreads();
  }
}

// dla[t] += sum of the totals of all later chunks (fp64 carry), plus
// <dhT, hT> when the final state has a cotangent (both given, [dk x dv] per
// head).  grid (B*H)
__global__ void __launch_bounds__(NT) k_dla_carry(float *__restrict__ dla,
                                                  const float *__restrict__ dcs_sum,
                                                  const float *__restrict__ dhT,
                                                  const float *__restrict__ hT, Geo g) {
  __shared__ double sh[NT], ex[NT];
  __shared__ double carry_in;
  const int64_t bh = blockIdx.x, b = bh / g.H, h = bh % g.H;
  {
    double part = 0.0;
    if (dhT) {
      const int64_t sz = g.dk * g.dv;
      for (int64_t e = threadIdx.x; e < sz; e += NT)
        part += (double)LDC(dhT, bh * sz + e, n_h(g)) * (double)LDC(hT, bh * sz + e, n_h(g));
    }
    sh[threadIdx.x] = part;
    __syncthreads();
    for (int o = NT / 2; o > 0; o >>= 1) {
      if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
      __syncthreads();
    }
    if (threadIdx.x == 0) carry_in = sh[0];
    __syncthreads();
  }
  // walk chunk blocks from the end; within a block, an exclusive suffix scan
  for (int64_t hi = g.N; hi > 0; hi -= NT) {
    const int64_t lo = hi - NT > 0 ? hi - NT : 0;
    const int64_t c = lo + threadIdx.x;
    double x = (c < hi) ? (double)LDC(dcs_sum, bh * g.N + c, g.B * g.H * g.N) : 0.0;
    sh[threadIdx.x] = x;
    __syncthreads();
    // inclusive suffix scan (Hillis-Steele) over the block
    for (int o = 1; o < NT; o <<= 1) {
      double y = (threadIdx.x + o < NT) ? sh[threadIdx.x + o] : 0.0;
      __syncthreads();
      sh[threadIdx.x] += y;
      __syncthreads();
    }
    ex[threadIdx.x] = sh[threadIdx.x] - x + carry_in;  // carry into chunk c
    __syncthreads();
    // every token of chunks lo..hi-1 gets its chunk's carry, all threads, the
    // loads of 8 tokens per thread in flight before their stores
    const int64_t ntok = (hi - lo) * g.C;
    for (int64_t i0 = threadIdx.x; i0 < ntok; i0 += 8 * NT) {
      float cur[8];
      int64_t off[8];
      bool in[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = i0 + (int64_t)u * NT, t = lo * g.C + i;
        in[u] = i < ntok && t < g.L;
        off[u] = in[u] ? la_off(g, b, t, h) : 0;
        cur[u] = in[u] ? LDC(dla, off[u], n_la(g)) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (in[u]) STC(dla, off[u], n_la(g), (float)((double)cur[u] + ex[(i0 + (int64_t)u * NT) / g.C]));
    }
    __syncthreads();
    if (threadIdx.x == 0) carry_in += sh[0];
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Host launchers.

static size_t grad_smem(int nbk, int nbv) {
  const int nbm = nbk > nbv ? nbk : nbv;
  return sizeof(float) * (3 * CMAX * LDT + KS * LDT + KS * ldn(nbm) + 5 * CMAX);
}

template <int MA, int NB, bool QUERY>
static void launch_state(const float *X, const float *Y, const float *la, float *st, float *Adec,
                         const Geo &g, cudaStream_t s) {
  dim3 grid((unsigned)g.N, (unsigned)g.H, (unsigned)g.B);
  LaunchTrace lt(QUERY ? "simt.query_state" : "simt.chunk_state", s);
  k_chunk_state<MA, NB, QUERY><<<grid, NT, 0, s>>>(X, Y, la, st, Adec, g);
}

template <bool QUERY>
static void dispatch_state(const float *X, const float *Y, const float *la, float *st,
                           float *Adec, const Geo &g, cudaStream_t s) {
  const int ma = g.dk > 64 ? 2 : 1, nb = g.dv > 64 ? 2 : 1;
  if (ma == 1 && nb == 1) launch_state<1, 1, QUERY>(X, Y, la, st, Adec, g, s);
  else if (ma == 1) launch_state<1, 2, QUERY>(X, Y, la, st, Adec, g, s);
  else if (nb == 1) launch_state<2, 1, QUERY>(X, Y, la, st, Adec, g, s);
  else launch_state<2, 2, QUERY>(X, Y, la, st, Adec, g, s);
}

static void launch_scan_fwd(float *st, const float *Adec, const float *h0, float *fin,
                            const Geo &g, cudaStream_t s) {
  launch_scan<false>(st, Adec, h0, fin, g, s, "simt.state_scan_fwd");
}

size_t fwd_workspace_bytes(const Geo &g) {
  return sizeof(float) * (size_t)(g.B * g.H * g.N * g.dk * g.dv + g.B * g.H * g.N);
}

// Two chunk-state arrays, their decays and chunk totals, and room for the
// final state (used only when it has a cotangent).
size_t bwd_workspace_bytes(const Geo &g) {
  return sizeof(float) * (size_t)(2 * g.B * g.H * g.N * g.dk * g.dv + 2 * g.B * g.H * g.N +
                                  g.B * g.H * g.dk * g.dv);
}

cudaError_t fwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                float *out, float *hT, const Geo &g, void *ws, cudaStream_t s) {
  float *st = static_cast<float *>(ws);
  float *Adec = st + g.B * g.H * g.N * g.dk * g.dv;
  dispatch_state<false>(k, v, la, st, Adec, g, s);
  launch_scan_fwd(st, Adec, h0, hT, g, s);
  dim3 grid((unsigned)g.N, (unsigned)g.H, (unsigned)g.B);
  LaunchTrace lt("simt.chunk_out", s);
  if (g.dv > 64) k_chunk_out<2><<<grid, NT, 0, s>>>(q, k, v, la, st, out, g);
  else k_chunk_out<1><<<grid, NT, 0, s>>>(q, k, v, la, st, out, g);
  return cudaGetLastError();
}

template <int NBK, int NBV>
static cudaError_t launch_grad(const float *q, const float *k, const float *v, const float *la,
                               const float *dout, const float *Hst, const float *dXst, float *dq,
                               float *dk, float *dv, float *dla, float *dcs_sum, const Geo &g,
                               cudaStream_t s) {
  const size_t smem = grad_smem(NBK, NBV);
  cudaError_t err = cudaFuncSetAttribute(k_chunk_grad<NBK, NBV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)g.N, (unsigned)g.G, (unsigned)g.B);
  LaunchTrace lt("simt.chunk_grad", s);
  k_chunk_grad<NBK, NBV><<<grid, NT, smem, s>>>(q, k, v, la, dout, Hst, dXst, dq, dk, dv, dla,
                                                 dcs_sum, g);
  return cudaGetLastError();
}

cudaError_t bwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                const float *dout, const float *dhT, float *dq, float *dk, float *dv, float *dla,
                float *dh0, const Geo &g, void *ws, cudaStream_t s) {
  const int64_t nst = g.B * g.H * g.N * g.dk * g.dv;
  float *Hst = static_cast<float *>(ws);
  float *dXst = Hst + nst;
  float *Adec = dXst + nst;
  float *dcs_sum = Adec + g.B * g.H * g.N;
  float *hT = dhT ? dcs_sum + g.B * g.H * g.N : nullptr;
  // forward states entering each chunk (recomputed; nothing is saved by fwd)
  dispatch_state<false>(k, v, la, Hst, Adec, g, s);
  launch_scan_fwd(Hst, Adec, h0, hT, g, s);
  // query contributions, then the reverse state-gradient pass
  dispatch_state<true>(q, dout, la, dXst, nullptr, g, s);
  launch_scan<true>(dXst, Adec, dhT, dh0, g, s, "simt.state_scan_rev");
  cudaError_t err;
  const bool bk = g.dk > 64, bv = g.dv > 64;
  if (bk && bv) err = launch_grad<2, 2>(q, k, v, la, dout, Hst, dXst, dq, dk, dv, dla, dcs_sum, g, s);
  else if (bk) err = launch_grad<2, 1>(q, k, v, la, dout, Hst, dXst, dq, dk, dv, dla, dcs_sum, g, s);
  else if (bv) err = launch_grad<1, 2>(q, k, v, la, dout, Hst, dXst, dq, dk, dv, dla, dcs_sum, g, s);
  else err = launch_grad<1, 1>(q, k, v, la, dout, Hst, dXst, dq, dk, dv, dla, dcs_sum, g, s);
  if (err != cudaSuccess) return err;
  {
    LaunchTrace lt("simt.dla_carry", s);
    k_dla_carry<<<(unsigned)(g.B * g.H), NT, 0, s>>>(dla, dcs_sum, dhT, hT, g);
  }
  return cudaGetLastError();
}

cudaError_t read_and_clear_error(unsigned int *word) {
  *word = 0;
#ifdef SSD_CHECK
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(word, g_check_word, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_check_word, &zero, sizeof(unsigned int));
#else
  return cudaSuccess;
#endif
}

}  // namespace simt
}  // namespace ssd
