// Tensor-core path of the chunked SSD scan (tcgen05.mma kind::tf32, fp32
// accumulators in tensor memory, TMA-fed shared-memory operands).
//
// The op is the recurrence S_t = exp(la_t) S_{t-1} + k_t v_t^T, out_t = S_t^T q_t
// timed as impl "chunked" on the "kernel_ssd_gpu.json" benchmark page.
//
// Everything is built from one "scan pass" on operands (q', k', v'):
//   causal       out'_r = sum_{u<=r} exp(cs_r - cs_u)(q'_r.k'_u) v'_u + exp(cs_r) S^T q'_r
//   anti-causal  out'_r = sum_{u>=r} exp(cs_u - cs_r)(q'_r.k'_u) v'_u + exp(A_c - cs_r) G^T q'_r
// (cs the in-chunk inclusive prefix of la, A_c its total; S / G the state
// entering the chunk from the left / right).  The forward is the causal pass
// on (q, k, v).  The gradients of <dout, out> are passes too, because the
// adjoint of a linear scan is a linear scan:
//   dq_h = causal(q' = dout, k' = v, v' = k, initial state h0^T)
//   dk_h = anti-causal(q' = v, k' = dout, v' = q, initial state dhT^T)
//   dv   = anti-causal(q' = k, k' = q, v' = dout, initial state dhT), whose
//          leftmost state is dh0
// and dla_t = sum_{t'>=t} (q_t'.dq_h[t'] - k_t'.dk_h[t']) + <dhT, hT>, where
// dhT is the cotangent of the final state hT (zero unless given).
//
// A pass cuts every (batch, head) sequence into segments of Ls tokens (a
// multiple of the 64-token chunk) so that B*H*nseg CTAs work at once:
//   k_seg_state  each segment's zero-initial-state contribution (one contraction)
//   k_seg_scan   the states entering every segment (sequential over segments)
//   k_walk       each segment's chunks in order, the running state resident in
//                tensor memory
//
// Operands the tensor cores must see transposed (anything contracted over
// tokens) are made by the threads from the TMA-loaded tiles: into tensor
// memory as the A operand (k'^T, v'^T) or into shared memory in the K-major
// 128-byte-swizzled layout (w * k'^T, P).  Operands written by threads are
// rounded to TF32 to nearest; TMA-fed ones are truncated by the tensor core.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/ssd.h"
#include "common.cuh"
#include "tc.h"
#include "tc_common.cuh"

namespace ssd {
namespace tc {

constexpr int C = 64;     // chunk length of the tensor-core path
constexpr int NTH = 128;  // threads per CTA: one per tensor-memory lane
constexpr int NT2 = 256;  // two threads per tensor-memory lane (column halves)

__host__ __device__ constexpr int rup(int x, int m) { return (x + m - 1) / m * m; }
__host__ __device__ inline int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// 2^x, hardware approximation (relative error ~2^-22)
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Inclusive prefix sums over n <= 64 tokens of la, given as the two values
// each lane holds (lane l: tokens 2l and 2l + 1, zero past n), accumulated in
// fp64 by one warp and rounded once to fp32 into cs, plus `carry` added before
// rounding.  Returns the sum of the n values.
__device__ inline double warp_cumsum64_regs(double x0, double x1, int n, double carry, float *cs) {
  const int l = threadIdx.x & 31;
  double pair = x0 + x1, incl = pair;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (l >= o) incl += y;
  }
  const double excl = incl - pair;
  if (cs) {
    if (2 * l < n) cs[2 * l] = (float)(carry + excl + x0);
    if (2 * l + 1 < n) cs[2 * l + 1] = (float)(carry + incl);
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}

// The same, loading la[first + t * stride] for t < n itself.
__device__ inline double warp_cumsum64(const float *__restrict__ la, int64_t first,
                                       int64_t stride, int n, double carry, float *cs) {
  const int l = threadIdx.x & 31;
  const double x0 = (2 * l < n) ? (double)la[first + (int64_t)(2 * l) * stride] : 0.0;
  const double x1 = (2 * l + 1 < n) ? (double)la[first + (int64_t)(2 * l + 1) * stride] : 0.0;
  return warp_cumsum64_regs(x0, x1, n, carry, cs);
}

// ===========================================================================
// Geometry of one scan pass on operands (q', k', v').
struct PassGeo {
  int64_t B, L, H;
  int hpg;
  int dk, dv;          // feature dims of q'/k' and of v' (= out')
  int dkp, dkn;        // dk rounded up to 32 (TMA column blocks) / 16 (MMA N)
  int dvp, dvn;        // dv rounded up to 32 / 16
  int qk_per_head;     // q', k' indexed by head (1) or by group (0)
  int v_per_head;      // v' indexed by head (1) or by group (0)
  int Ls, nseg;        // segment length (multiple of C) and segments per sequence
};

// Output of a walk: out'[b, t, slot, 0:dv] with slot = h (out_slots == H) or
// h / hpg (out_slots == G, summed over the group's heads by atomic adds);
// optionally dcs[b, t, h] = y[b, t, h / hpg, :] . (the inter-chunk part of
// out'_t, the term carried by the state entering the chunk).
struct OutArgs {
  float *out;
  int out_slots;
  const float *y;
  float *dcs;
};

__device__ __forceinline__ int qk_slot(const PassGeo &p, int64_t h) {
  return (int)(p.qk_per_head ? h : h / p.hpg);
}
__device__ __forceinline__ int v_slot(const PassGeo &p, int64_t h) {
  return (int)(p.v_per_head ? h : h / p.hpg);
}

// ===========================================================================
// Segment contraction, the zero-initial-state contribution of one segment:
//   causal      D = sum_u exp(A_seg - cs_u) k'_u v'_u^T   (evaluated at its end)
//   anti-causal D = sum_u exp(cs_u) k'_u v'_u^T           (evaluated at its start)
// with cs the in-segment inclusive prefix of la and A_seg its total (also
// written).  grid (nseg, H, B), 256 threads: thread (quarter q, lane l, half f)
// owns tensor-memory lane 32q + l and token half f of each 32-token slice.
// The segment is streamed in 32-token slices through a two-stage TMA ring,
// loaded two slices ahead.  Tensor memory (256 columns): D [0,128), A operand
// k'^T double-buffered at [128,160) / [160,192).  Shared memory: two stages of
// k' and v' tiles, and the B operand (sc * v')^T [dvn x 32], double-buffered.
constexpr int SL = 32;  // slice length of the segment contraction
template <bool REV>
__global__ void __launch_bounds__(NT2, 2) k_seg_state(const __grid_constant__ CUtensorMap tmK,
                                                      const __grid_constant__ CUtensorMap tmV,
                                                      const float *__restrict__ la,
                                                      float *__restrict__ states,
                                                      float *__restrict__ Aseg, PassGeo p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_align1024(smem_raw);
  const int ncbk = p.dkp / 32, ncbv = p.dvp / 32;
  const uint32_t xbytes = (uint32_t)ncbk * 4096, ybytes = (uint32_t)ncbv * 4096;
  const uint32_t stage = xbytes + ybytes;
  const uint32_t bbytes = (uint32_t)rup(p.dvn * 128, 1024);
  uint8_t *tiles = smem;                      // [2][k' tile 32 x dkp | v' tile 32 x dvp]
  uint8_t *Bb = smem + 2 * stage;             // [2][dvn x 32] K-major
  float *scb = (float *)(Bb + 2 * bbytes);    // [256] per-token weights of 8 slices
  __shared__ double wtot[8];
  __shared__ uint64_t bar_tma[2], bar_mma[2];
  __shared__ uint32_t tmem_base;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, hf = warp >> 2, L = qd * 32 + lane;
  const int64_t seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t bh = b * p.H + h;
  const int64_t s_begin = seg * (int64_t)p.Ls;
  const int64_t s_end = imin64(p.L, s_begin + p.Ls);
  const int nsl = (int)cdiv(s_end - s_begin, SL);
  const int kslot = qk_slot(p, h), vslot = v_slot(p, h);

  // thread 0 issues the MMAs; lane 0 of warp 1 / warp 2 loads the k' / v'
  // slices (two arrivals complete a stage's load phase)
  const bool ldk = tid == 32, ldv = tid == 64;
  if (warp == 0) tmem_alloc(&tmem_base, 256);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_tma[i], 2);
      mbar_init(&bar_mma[i], 1);
    }
    fence_mbar_init();
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  __syncthreads();
  int pend[2] = {-1, -1};  // slice in flight per stage (each loader's view)
  auto issue_tma = [&](int n) {  // the calling loader's half of slice n
    const int st = n & 1;
    pend[st] = n;
    const int row = (int)(b * p.L + s_begin + (int64_t)n * SL);
    uint8_t *Xt = tiles + st * stage, *Yt = Xt + xbytes;
    if (ldk) {
      mbar_expect_tx(&bar_tma[st], xbytes);
      for (int cb = 0; cb < ncbk; ++cb) tma_load_3d(Xt + cb * 4096, &tmK, &bar_tma[st], cb * 32, kslot, row);
    } else {
      mbar_expect_tx(&bar_tma[st], ybytes);
      for (int cb = 0; cb < ncbv; ++cb) tma_load_3d(Yt + cb * 4096, &tmV, &bar_tma[st], cb * 32, vslot, row);
    }
  };
  if (ldk || ldv) {
    issue_tma(0);
    if (nsl > 1) issue_tma(1);
  }
  // segment total of la: all threads, fp64
  __shared__ double wsum[8];
  {
    double part = 0.0;
    for (int64_t t = s_begin + tid; t < s_end; t += NT2) part += (double)la[(b * p.L + t) * p.H + h];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) wsum[warp] = part;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  double tot = 0.0;
#pragma unroll
  for (int w2 = 0; w2 < 8; ++w2) tot += wsum[w2];
  const float Af = (float)tot;
  if (tid == 0) Aseg[bh * p.nseg + seg] = Af;
  const uint32_t tmem = tmem_base;
  const uint32_t lb = (uint32_t)(qd * 32) << 16;
  double carry = 0.0;
  bool ok = true;
  // all threads: weights of the 256 tokens from slice n on (one per thread),
  // continuing the running in-segment prefix (fp64 block scan); each thread's
  // la value of the next batch is loaded one batch ahead
  auto la_at = [&](int64_t t) { return t < s_end ? (double)la[(b * p.L + t) * p.H + h] : 0.0; };
  double la_next = la_at(s_begin + tid);
  auto batch_weights = [&](int n) {
    const int64_t t = s_begin + (int64_t)n * SL + tid;
    double x = la_next;
    la_next = la_at(t + 8 * SL);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    double before = carry, all = carry;
#pragma unroll
    for (int w2 = 0; w2 < 8; ++w2) {
      if (w2 < warp) before += wtot[w2];
      all += wtot[w2];
    }
    const float csf = (float)(before + x);
    scb[tid] = t < s_end ? expf(REV ? csf : Af - csf) : 0.f;
    carry = all;
    __syncthreads();
  };

  for (int n = 0; n < nsl; ++n) {
    const int st = n & 1;
    const int64_t t0 = s_begin + (int64_t)n * SL;
    const int len = (int)imin64(SL, s_end - t0);
    if ((n & 7) == 0) batch_weights(n);
    const float *sc = scb + (n & 7) * SL;
    const uint8_t *Xt = tiles + st * stage, *Yt = Xt + xbytes;
    uint8_t *Bs = Bb + st * bbytes;
    ok = mbar_wait(&bar_tma[st], (n >> 1) & 1) && ok;
    if (ok) pend[st] = -1;
    if (n >= 2) ok = mbar_wait(&bar_mma[st], ((n >> 1) - 1) & 1) && ok;  // slice n-2 done
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    {  // A operand: k'^T, lane = feature, tokens [16 hf, 16 hf + 16)
      float v[16];
#pragma unroll
      for (int uu = 0; uu < 16; ++uu) {
        const int u = hf * 16 + uu;
        v[uu] = (L < p.dk && u < len) ? tf32r(*(const float *)(Xt + sw128_off(u, L, SL))) : 0.f;
      }
      tmem_st16(tmem + lb + 128 + st * 32 + hf * 16, v);
    }
    if (L < p.dvn) {  // B operand: (sc v')^T, row = feature
#pragma unroll
      for (int uu = 0; uu < 16; uu += 4) {
        const int u = hf * 16 + uu;
        float f[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
          f[r] = L < p.dv ? tf32r(*(const float *)(Yt + sw128_off(u + r, L, SL)) * sc[u + r]) : 0.f;
        *reinterpret_cast<float4 *>(Bs + sw128_off(L, u, p.dvn)) = make_float4(f[0], f[1], f[2], f[3]);
      }
    }
    tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((ldk || ldv) && n + 2 < nsl) issue_tma(n + 2);  // this stage's tiles are consumed
    if (tid == 0) {
      const uint32_t bsm = smem_u32(Bs);
      const uint32_t id = idesc_tf32(128, p.dvn);
#pragma unroll
      for (int kk = 0; kk < SL / 8; ++kk)
        mma_ts(tmem, tmem + 128 + st * 32 + kk * 8, sdesc(bsm + kk * 32), id, (n > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&bar_mma[st]);
    }
  }
  if (ok) {
    for (int n = (nsl >= 2 ? nsl - 2 : 0); n < nsl; ++n) ok = mbar_wait(&bar_mma[n & 1], (n >> 1) & 1) && ok;
  }
  const bool fail = __syncthreads_or(!ok);
  tc_fence_after();
  if (!fail) {
    // stage D [dk x dv] through the (now idle) tile buffers in the swizzled
    // column-block layout, then write it out coalesced
    uint8_t *Ds = tiles;  // needs dk * dvp * 4 <= 2 * stage bytes
    const int dkr = rup(p.dk, 8);
    for (int c0 = hf * 64; c0 < hf * 64 + 64; c0 += 32) {
      if (c0 >= p.dvn) break;  // warp-uniform
      float v[32];
      tmem_ld32(tmem + lb + c0, v);
      if (L < p.dk) {
#pragma unroll
        for (int jj = 0; jj < 32; jj += 4)
          if (c0 + jj < p.dvp)
            *reinterpret_cast<float4 *>(Ds + sw128_off(L, c0 + jj, dkr)) =
                make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
      }
    }
    __syncthreads();
    float *dst = states + (bh * p.nseg + seg) * (int64_t)p.dk * p.dv;
    const int n4 = p.dk * p.dv / 4;
    for (int m = tid; m < n4; m += NT2) {
      const int e = 4 * m, i = e / p.dv, j = e - i * p.dv;
      *reinterpret_cast<float4 *>(dst + e) = *reinterpret_cast<const float4 *>(Ds + sw128_off(i, j, dkr));
    }
  } else if (ldk || ldv) {
    // tiles of up to two slices may still be in flight: wait for them
    for (int st = 0; st < 2; ++st)
      if (pend[st] >= 0) mbar_wait(&bar_tma[st], (pend[st] >> 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ===========================================================================
// State passing over segments, in place (each thread owns 4 consecutive state
// elements and loads up to SU segments of them at once, so a pass costs about
// one memory round trip per SU segments).
//   causal:      st[s] <- state entering segment s from the left; the first is
//                init, or 0; the state right of the last segment goes to fin
//   anti-causal: st[s] <- state entering segment s from the right; the one
//                entering the last is init, or 0; the state left of segment 0
//                goes to fin
// init is read, and fin (if given) written, transposed when TRANS.  When stT
// is given, every result is also written there transposed.
// grid (B*H, ceil(dk*dv / (4*128))), dk*dv a multiple of 4
constexpr int SU = 10;
template <bool REV, bool TRANS>
__global__ void __launch_bounds__(NTH) k_seg_scan(float *__restrict__ st,
                                                  const float *__restrict__ Aseg,
                                                  const float *__restrict__ init,
                                                  float *__restrict__ fin,
                                                  float *__restrict__ stT, PassGeo p) {
  const int64_t bh = blockIdx.x;
  const int64_t e0 = 4 * ((int64_t)blockIdx.y * NTH + threadIdx.x);
  const int64_t sz = (int64_t)p.dk * p.dv;
  if (e0 >= sz) return;
  auto tpos = [&](int64_t e) { return (e % p.dv) * p.dk + e / p.dv; };  // transposed position
  float4 *q = reinterpret_cast<float4 *>(st + bh * p.nseg * sz + e0);
  const int64_t sz4 = sz / 4;
  const float *a = Aseg + bh * p.nseg;
  float run[4] = {0.f, 0.f, 0.f, 0.f};
  if (init) {
#pragma unroll
    for (int j = 0; j < 4; ++j) run[j] = init[bh * sz + (TRANS ? tpos(e0 + j) : e0 + j)];
  }
  for (int k0 = 0; k0 < p.nseg; k0 += SU) {
    float4 x[SU];
    float d[SU];
#pragma unroll
    for (int u = 0; u < SU; ++u) {
      const int k = k0 + u;
      if (k < p.nseg) {
        const int s = REV ? p.nseg - 1 - k : k;
        x[u] = q[(int64_t)s * sz4];
        d[u] = expf(a[s]);
      }
    }
#pragma unroll
    for (int u = 0; u < SU; ++u) {
      const int k = k0 + u;
      if (k < p.nseg) {
        const int s = REV ? p.nseg - 1 - k : k;
        q[(int64_t)s * sz4] = make_float4(run[0], run[1], run[2], run[3]);
        if (stT) {
#pragma unroll
          for (int j = 0; j < 4; ++j) stT[bh * p.nseg * sz + (int64_t)s * sz + tpos(e0 + j)] = run[j];
        }
        run[0] = fmaf(d[u], run[0], x[u].x);
        run[1] = fmaf(d[u], run[1], x[u].y);
        run[2] = fmaf(d[u], run[2], x[u].z);
        run[3] = fmaf(d[u], run[3], x[u].w);
      }
    }
  }
  if (fin) {
#pragma unroll
    for (int j = 0; j < 4; ++j) fin[bh * sz + (TRANS ? tpos(e0 + j) : e0 + j)] = run[j];
  }
}

// ===========================================================================
// Walk over the chunks of one segment (left to right, or right to left when
// REV) with the running state resident in tensor memory.  grid (nseg, H, B),
// 256 threads: thread (quarter q, lane l, half f) owns tensor-memory lane
// 32q + l and column half f of each 64-column block; two CTAs per SM.
//
// Tensor memory (256 columns):
//   X   [0,64)    S = q' k'^T (M = 64: rows 16q..16q+15 in lanes 32q..), then
//                 out'^T (lane j = feature, column = token)
//   VT  [64,128)  v'^T of the chunk (A operand)
//   HT  [128,256) running state, transposed (A operand): lane j, column i
// Shared memory: q' tile (scaled in place to the B operand of the inter term),
// k' tile (then reused for w * k'^T, the B operand of the state update), v'
// tile (then reused for P).
// The entering state is read from Hseg as [dk x dv] (or [dv x dk] when
// HT_SRC_T).
template <bool REV, bool ATOMIC>
__global__ void __launch_bounds__(NT2, 2) k_walk(const __grid_constant__ CUtensorMap tmQ,
                                              const __grid_constant__ CUtensorMap tmK,
                                              const __grid_constant__ CUtensorMap tmV,
                                              const __grid_constant__ CUtensorMap tmO,
                                              const float *__restrict__ la,
                                              const float *__restrict__ Hseg, int hseg_t,
                                              OutArgs oa, PassGeo p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_align1024(smem_raw);
  const int ncbk = p.dkp / 32, ncbv = p.dvp / 32;
  const uint32_t vbytes = (uint32_t)max(ncbv * 8192, 16384);
  uint8_t *Qb = smem;
  uint8_t *Kb = Qb + ncbk * 8192;
  uint8_t *Vb = Kb + ncbk * 8192;
  // per-chunk factors, double-buffered: in-chunk prefix of la times log2(e),
  // exp(cs), exp(A - cs); computed one chunk ahead by warp 4
  float *cs2b = (float *)(Vb + vbytes);  // [2][64]
  float *ewb = cs2b + 2 * C, *wwb = ewb + 2 * C;
  float *red = wwb + 2 * C;  // [4][64]
  float *scr = red + 4 * C;  // [64] scratch of warp 4
  __shared__ uint64_t bar_tma, bar_s, bar_i, bar_o, bar_h;
  __shared__ uint32_t tmem_base;
  __shared__ float a_chunk[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, hf = warp >> 2, L = qd * 32 + lane;
  const int64_t seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t bh = b * p.H + h;
  const int64_t s_begin = seg * (int64_t)p.Ls;
  const int64_t s_end = imin64(p.L, s_begin + p.Ls);
  const int nc = (int)cdiv(s_end - s_begin, C);
  const int kslot = qk_slot(p, h), vslot = v_slot(p, h);
  const int dk = p.dk, dv = p.dv, dkn = p.dkn;
  const int oslot = oa.out_slots == p.H ? (int)h : (int)(h / p.hpg);
  constexpr float LOG2E = 1.4426950408889634f;

  // Serial issue work is spread over warps: thread 0 issues the MMAs, lane 0
  // of warps 1, 2, 3 the q', v' and k' tile loads (three arrivals complete a
  // load phase), warp 4 computes the next chunk's decay factors.
  const bool ldq = tid == 32, ldv = tid == 64, ldk = tid == 96;
  if (warp == 0) tmem_alloc(&tmem_base, 256);
  if (tid == 0) {
    mbar_init(&bar_tma, 3);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_i, 1);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_h, 1);
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t lb = (uint32_t)(qd * 32) << 16;
  int tma_pending = -1;  // barrier phase of this loader's loads not yet waited for
  // chunk c's tiles; `use` counts the barrier's phases (chunks in walk order).
  // Each loader thread arrives once per phase with its own byte count; the
  // k' tile may be issued later than the q' and v' tiles.
  auto tma_q = [&](int c, int use) {
    const int row = (int)(b * p.L + s_begin + (int64_t)c * C);
    mbar_expect_tx(&bar_tma, (uint32_t)ncbk * 8192);
    for (int cb = 0; cb < ncbk; ++cb) tma_load_3d(Qb + cb * 8192, &tmQ, &bar_tma, cb * 32, kslot, row);
    tma_pending = use;
  };
  auto tma_v = [&](int c, int use) {
    const int row = (int)(b * p.L + s_begin + (int64_t)c * C);
    mbar_expect_tx(&bar_tma, (uint32_t)ncbv * 8192);
    for (int cb = 0; cb < ncbv; ++cb) tma_load_3d(Vb + cb * 8192, &tmV, &bar_tma, cb * 32, vslot, row);
    tma_pending = use;
  };
  auto tma_k = [&](int c, int use) {
    const int row = (int)(b * p.L + s_begin + (int64_t)c * C);
    mbar_expect_tx(&bar_tma, (uint32_t)ncbk * 8192);
    for (int cb = 0; cb < ncbk; ++cb) tma_load_3d(Kb + cb * 8192, &tmK, &bar_tma, cb * 32, kslot, row);
    tma_pending = use;
  };
  auto issue_first_loads = [&]() {
    const int c0 = REV ? nc - 1 : 0;
    if (ldq) tma_q(c0, 0);
    if (ldv) tma_v(c0, 0);
    if (ldk) tma_k(c0, 0);
  };

  if (!hseg_t) issue_first_loads();

  // warp 4: the factors of chunk c into buffer bf, from la values loaded one
  // chunk ahead (la_x0, la_x1: this lane's two tokens of chunk c)
  double la_x0 = 0.0, la_x1 = 0.0;
  auto la_prefetch = [&](int c) {
    const int64_t t0 = s_begin + (int64_t)c * C;
    const int len = (int)imin64(C, s_end - t0);
    const float *lp = la + (b * p.L + t0) * p.H + h;
    la_x0 = (2 * lane < len) ? (double)lp[(int64_t)(2 * lane) * p.H] : 0.0;
    la_x1 = (2 * lane + 1 < len) ? (double)lp[(int64_t)(2 * lane + 1) * p.H] : 0.0;
  };
  auto chunk_factors = [&](int c, int bf) {
    const int64_t t0 = s_begin + (int64_t)c * C;
    const int len = (int)imin64(C, s_end - t0);
    const double tot = warp_cumsum64_regs(la_x0, la_x1, len, 0.0, scr);
    __syncwarp();
    const float tot2 = (float)tot * LOG2E;
    for (int t = lane; t < C; t += 32) {
      const float x = t < len ? scr[t] * LOG2E : 0.f;
      cs2b[bf * C + t] = x;
      ewb[bf * C + t] = t < len ? ex2f(x) : 0.f;
      wwb[bf * C + t] = t < len ? ex2f(tot2 - x) : 0.f;
    }
    if (lane == 0) a_chunk[bf] = ex2f(tot2);
    __syncwarp();
  };
  if (warp == 4) {
    la_prefetch(REV ? nc - 1 : 0);
    chunk_factors(REV ? nc - 1 : 0, 0);
  }

  {  // running state, transposed: lane j, column i = state[i][j]
    const float *H0 = Hseg + (bh * p.nseg + seg) * (int64_t)dk * dv;
    if (hseg_t) {
      // the entering state is stored transposed ([dv x dk]): read it coalesced
      // into the idle tile buffers ([dv rows x (dk + 1)]), then by rows
      float *Ts = reinterpret_cast<float *>(Qb);
      const int n = dv * dk;
      for (int e = tid; e < n; e += NT2) {
        const int r = e / dk, cc = e - r * dk;
        Ts[r * (dk + 1) + cc] = H0[e];
      }
      __syncthreads();
      for (int c0 = hf * 64; c0 < hf * 64 + 64 && c0 < rup(dk, 32); c0 += 32) {
        float hv[32];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
          const int i = c0 + ii;
          hv[ii] = (L < dv && i < dk) ? Ts[L * (dk + 1) + i] : 0.f;
        }
        tmem_st32(tmem + lb + 128 + c0, hv);
      }
      __syncthreads();  // the tile buffers are about to receive the first loads
      issue_first_loads();
    } else {
      for (int c0 = hf * 64; c0 < hf * 64 + 64 && c0 < rup(dk, 32); c0 += 32) {
        float hv[32];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
          const int i = c0 + ii;
          hv[ii] = (L < dv && i < dk) ? H0[(int64_t)i * dv + L] : 0.f;
        }
        tmem_st32(tmem + lb + 128 + c0, hv);
      }
    }
    tmem_st_wait();
  }

  bool ok = true;
  const bool split = oa.dcs != nullptr;
  // The resident state is kept as Hs with the true state = alpha * Hs.  While
  // alpha stays in [2^-40, 2^40] a chunk's decay is folded into alpha (the
  // inter term scales q' by alpha, the update scales w k' by 1 / alpha), so
  // the update MMA issues with the output MMAs and no rescale pass runs;
  // otherwise the threads rescale Hs explicitly and alpha returns to 1.
  float alpha = 1.f;
  int hphase = 0;  // completions of bar_h so far (the explicit path only)
  // HT += v'^T (w k')   (M = dv lanes, N = dkn, K = 64 tokens); thread 0
  auto issue_update = [&]() {
    const uint32_t kwa = smem_u32(Kb);
    const uint32_t id = idesc_tf32(128, dkn);
#pragma unroll
    for (int kk = 0; kk < C / 8; ++kk)
      mma_ts(tmem + 128, tmem + 64 + kk * 8, sdesc(kwa + (kk >> 2) * (dkn * 128) + (kk & 3) * 32),
             id, 1u);
  };
  for (int ci = 0; ci < nc; ++ci) {
    const int c = REV ? nc - 1 - ci : ci;
    const int64_t t0 = s_begin + (int64_t)c * C;
    const int len = (int)imin64(C, s_end - t0);
    const int cnext = REV ? c - 1 : c + 1;
    const int fb = ci & 1;
    const float *cs2 = cs2b + fb * C, *ew = ewb + fb * C, *ww = wwb + fb * C;
    if (warp == 4 && ci + 1 < nc) la_prefetch(cnext);  // used by chunk_factors below
    ok = mbar_wait(&bar_tma, ci & 1) && ok;
    if (ok) tma_pending = -1;
    // S = q' k'^T (M = 64, N = 64, K = dk), issued as soon as the tiles are
    // in, before the CTA barrier: the issuing warp then starts its passes
    // with the others instead of 16 MMA issues behind them.  (The previous
    // chunk's output was read from these columns before its final barrier.)
    if (tid == 0 && ok) {
      tc_fence_after();
      const uint32_t qa = smem_u32(Qb), ka = smem_u32(Kb);
      const uint32_t id = idesc_tf32(64, 64);
      for (int kk = 0; kk < dk / 8; ++kk) {
        const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
        mma_ss(tmem, sdesc(qa + off), sdesc(ka + off), id, kk > 0 ? 1u : 0u);
      }
      mma_commit(&bar_s);
    }
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    // inter-term factor of a query row, state-update weight of a key column
    const float *interf = REV ? ww : ew;
    const float *statew = REV ? ew : ww;
    const float a_c = a_chunk[fb], an = alpha * a_c;
    const bool lazy = a_c >= 0x1p-30f && an >= 0x1p-40f && an <= 0x1p40f;
    const float kscale = lazy ? 1.f / an : 1.f;
    {  // v'^T into tensor memory: lane = feature, tokens [32 hf, 32 hf + 32)
      float v[32];
#pragma unroll
      for (int uu = 0; uu < 32; ++uu) {
        const int u = hf * 32 + uu;
        v[uu] = (L < dv && u < len) ? tf32r(*(const float *)(Vb + sw128_off(u, L, C))) : 0.f;
      }
      tmem_st32(tmem + lb + 64 + hf * 32, v);
    }
    float kw[32];  // w_u * k'[u][L], tokens [32 hf, 32 hf + 32)
    {
      const float4 *sw4 = reinterpret_cast<const float4 *>(statew + hf * 32);
#pragma unroll
      for (int u4 = 0; u4 < 8; ++u4) {
        const float4 wv = sw4[u4];
        const float wq[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int uu = 4 * u4 + e, u = hf * 32 + uu;
          kw[uu] = (L < dk) ? tf32r(*(const float *)(Kb + sw128_off(u, L, C)) * (wq[e] * kscale)) : 0.f;
        }
      }
    }
    ok = mbar_wait(&bar_s, ci & 1) && ok;
    tc_fence_after();
    float sr[32];
    tmem_ld32(tmem + lb + hf * 32, sr);
    tc_fence_before();
    __syncthreads();  // every read of the v' and k' tiles and of S is done
    {  // P into the v' tile's space.  S row r sits in lane r % 16 (M = 64); the
       // lane 16 above it takes the upper 16 of the warp's 32 tokens
      const int r = qd * 16 + (lane & 15), up = lane >> 4;
      const int ub = hf * 32 + 16 * up;  // first token of this lane's 16
      float s16[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float hi = __shfl_sync(0xffffffffu, sr[16 + i], lane & 15);
        s16[i] = up ? hi : sr[i];
      }
      const float cr = cs2[r];
      uint8_t *P = Vb;
#pragma unroll
      for (int uu = 0; uu < 16; uu += 4) {
        float f[4];
        const float4 c4 = *reinterpret_cast<const float4 *>(cs2 + ub + uu);
        const float cu[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int u = ub + uu + e;
          const bool valid = r < len && u < len && (REV ? u >= r : u <= r);
          f[e] = valid ? tf32r(ex2f(REV ? cu[e] - cr : cr - cu[e]) * s16[uu + e]) : 0.f;
        }
        *reinterpret_cast<float4 *>(P + sw128_off(r, ub + uu, C)) = make_float4(f[0], f[1], f[2], f[3]);
      }
    }
    if (L < dkn) {  // w * k'^T into the k' tile's space (B operand, dkn rows)
#pragma unroll
      for (int uu = 0; uu < 32; uu += 4)
        *reinterpret_cast<float4 *>(Kb + sw128_off(L, hf * 32 + uu, dkn)) =
            make_float4(kw[uu], kw[uu + 1], kw[uu + 2], kw[uu + 3]);
    }
    {  // q' rows scaled by the inter-term factor, in place (4 threads per row)
      const int r = tid & 63, part = tid >> 6;
      const float e = interf[r] * alpha;
      const int cols = p.dkp / 4;
      for (int col = part * cols; col < (part + 1) * cols; col += 4) {
        float4 *q4 = reinterpret_cast<float4 *>(Qb + sw128_off(r, col, C));
        float4 f = *q4;
        f.x = tf32r(f.x * e); f.y = tf32r(f.y * e); f.z = tf32r(f.z * e); f.w = tf32r(f.w * e);
        *q4 = f;
      }
    }
    tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    if (tid == 0) {  // out'^T = HT (f q')^T  [+ v'^T P^T]
      const uint32_t qa = smem_u32(Qb), pa = smem_u32(Vb);
      const uint32_t id = idesc_tf32(128, 64);
      for (int kk = 0; kk < dk / 8; ++kk)
        mma_ts(tmem, tmem + 128 + kk * 8, sdesc(qa + (kk >> 2) * 8192 + (kk & 3) * 32), id,
               kk > 0 ? 1u : 0u);
      if (split) {
        mma_commit(&bar_i);
      } else {
#pragma unroll
        for (int kk = 0; kk < C / 8; ++kk)
          mma_ts(tmem, tmem + 64 + kk * 8, sdesc(pa + (kk >> 2) * 8192 + (kk & 3) * 32), id, 1u);
        if (lazy) issue_update();
        mma_commit(&bar_o);
      }
    }
    if (warp == 4 && ci + 1 < nc) chunk_factors(cnext, fb ^ 1);
    if (split) {
      // dcs[t] = y_t . (inter-chunk part of out'_t), reduced over the 128 lanes
      float yv[32];
      {
        const int64_t ldy = (int64_t)(p.H / p.hpg) * dv;
        const float *ys = oa.y + ((b * p.L + t0) * (p.H / p.hpg) + h / p.hpg) * (int64_t)dv + L;
#pragma unroll
        for (int tt = 0; tt < 32; ++tt) {
          const int t = hf * 32 + tt;
          yv[tt] = (L < dv && t < len) ? ys[t * ldy] : 0.f;
        }
      }
      ok = mbar_wait(&bar_i, ci & 1) && ok;
      tc_fence_after();
      float o[32];
      tmem_ld32(tmem + lb + hf * 32, o);
      // every thread has its inter part: let the intra MMA accumulate on top
      // while the dot products are reduced
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {  // + v'^T P^T
        const uint32_t pa = smem_u32(Vb);
        const uint32_t id = idesc_tf32(128, 64);
#pragma unroll
        for (int kk = 0; kk < C / 8; ++kk)
          mma_ts(tmem, tmem + 64 + kk * 8, sdesc(pa + (kk >> 2) * 8192 + (kk & 3) * 32), id, 1u);
        if (lazy) issue_update();
        mma_commit(&bar_o);
      }
#pragma unroll
      for (int tt = 0; tt < 32; ++tt) o[tt] *= yv[tt];
#pragma unroll
      for (int off = 16, n = 32; off >= 1; off >>= 1, n >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int k2 = 0; k2 < n / 2; ++k2) {
          const float mine = up ? o[n / 2 + k2] : o[k2];
          const float send = up ? o[k2] : o[n / 2 + k2];
          o[k2] = mine + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      red[qd * C + hf * 32 + lane] = o[0];
      __syncthreads();
      if (tid < len)
        oa.dcs[(b * p.L + t0 + tid) * p.H + h] = red[tid] + red[C + tid] + red[2 * C + tid] + red[3 * C + tid];
    }
    ok = mbar_wait(&bar_o, ci & 1) && ok;
    tc_fence_after();
    // q' and v' tiles are free now (and k' too when the update ran): next loads.
    // A full chunk's output is staged in the v' tile and stored by TMA first,
    // so its next v' tile is loaded after that store has read the buffer.
    const bool staged = len == C;
    if (ok && ci + 1 < nc) {
      if (ldq) tma_q(cnext, ci + 1);
      if (ldv && !staged) tma_v(cnext, ci + 1);
      if (ldk && lazy) tma_k(cnext, ci + 1);
    }
    {
      float o[32];
      tmem_ld32(tmem + lb + hf * 32, o);
      if (staged) {  // out'[t][L] into the v' tile, in the layout a load of tmO gives
        if (L < p.dvp) {
#pragma unroll
          for (int tt = 0; tt < 32; ++tt)
            *reinterpret_cast<float *>(Vb + sw128_off(hf * 32 + tt, L, C)) = o[tt];
        }
      } else if (L < dv) {
        const int64_t ld = (int64_t)oa.out_slots * dv;
        float *os = oa.out + ((b * p.L + t0) * oa.out_slots + oslot) * (int64_t)dv + L;
#pragma unroll
        for (int tt = 0; tt < 32; ++tt) {
          const int t = hf * 32 + tt;
          if (t < len) {
            if (ATOMIC) atomicAdd(os + t * ld, o[tt]);
            else os[t * ld] = o[tt];
          }
        }
      }
    }
    if (staged) {
      fence_async_smem();
      __syncthreads();
      if (ldv) {  // store (or add, for a group's heads) the chunk's output rows
        const int row = (int)(b * p.L + t0);
        for (int cb = 0; cb < ncbv; ++cb) {
          if (ATOMIC) tma_reduce_add_3d(&tmO, Vb + cb * 8192, cb * 32, oslot, row);
          else tma_store_3d(&tmO, Vb + cb * 8192, cb * 32, oslot, row);
        }
        bulk_commit_group();
        bulk_wait_read_all();
        if (ok && ci + 1 < nc) tma_v(cnext, ci + 1);
      }
    }
    if (lazy) {
      alpha = an;
    } else {
      // Hs <- alpha exp(A_c) Hs (the true state, decayed), then the update
      for (int c0 = hf * 64; c0 < hf * 64 + 64 && c0 < rup(dk, 32); c0 += 32) {
        float hv[32];
        tmem_ld32(tmem + lb + 128 + c0, hv);
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) hv[ii] *= an;
        tmem_st32(tmem + lb + 128 + c0, hv);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
        issue_update();
        mma_commit(&bar_h);
      }
      ok = mbar_wait(&bar_h, hphase & 1) && ok;
      ++hphase;
      tc_fence_after();
      if (ldk && ok && ci + 1 < nc) tma_k(cnext, ci + 1);
      alpha = 1.f;
    }
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
  }
  __syncthreads();
  if ((ldq || ldv || ldk) && tma_pending >= 0) mbar_wait(&bar_tma, tma_pending & 1);
  if (ldv) bulk_wait_all();  // the output stores have landed
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ===========================================================================
// Intra-chunk part of dlog_alpha, per (chunk, group), for each head h of the
// group:
//   B_t = sum_{t' >= t, s < t, both in the chunk} exp(cs_t' - cs_s) (q_t'.k_s)(dout_t'.v_s)
// (the block of M = D o (q k^T) o (dout v^T) below row t and left of column
// t), from the row and column sums of M's strictly lower triangle.  q k^T is
// computed once; dout v^T per head.  Both score MMAs have M = 64
// (rows 16w..16w+15 in lanes 32w..) and share one two-tile shared-memory
// buffer; the next head's tiles load while the current head's sums run.
// grid (N chunks, G, B), 128 threads, three CTAs per SM.
__global__ void __launch_bounds__(NTH) k_dla_intra(const __grid_constant__ CUtensorMap tmQ,
                                                   const __grid_constant__ CUtensorMap tmK,
                                                   const __grid_constant__ CUtensorMap tmV,
                                                   const __grid_constant__ CUtensorMap tmD,
                                                   const float *__restrict__ la,
                                                   float *__restrict__ Bt, PassGeo p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_align1024(smem_raw);
  const int dk = p.dk, dv = p.dv;  // here dk = q/k features, dv = v/dout features
  const int ncbk = p.dkp / 32, ncbv = p.dvp / 32, ncbm = ncbk > ncbv ? ncbk : ncbv;
  uint8_t *T1 = smem, *T2 = smem + ncbm * 8192;
  float *R = (float *)(T2 + ncbm * 8192);  // [4][64] column partials, [64] row sums
  float *cs = R + 5 * C;                  // [64]
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t c = blockIdx.x, grp = blockIdx.y, b = blockIdx.z;
  const int64_t t0 = c * C;
  const int len = (int)imin64(C, p.L - t0);
  const int row = (int)(b * p.L + t0);
  const int hpg = p.hpg;

  auto load_dv = [&](int64_t h) {  // dout -> T1, v -> T2
    mbar_expect_tx(&bar_tma, (uint32_t)(2 * ncbv) * 8192);
    for (int cb = 0; cb < ncbv; ++cb) {
      tma_load_3d(T1 + cb * 8192, &tmD, &bar_tma, cb * 32, (int)h, row);
      tma_load_3d(T2 + cb * 8192, &tmV, &bar_tma, cb * 32, (int)h, row);
    }
  };
  if (warp == 0) tmem_alloc(&tmem_base, 128);
  if (tid == 0) {
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    mbar_expect_tx(&bar_tma, (uint32_t)(2 * ncbk) * 8192);
    for (int cb = 0; cb < ncbk; ++cb) {
      tma_load_3d(T1 + cb * 8192, &tmQ, &bar_tma, cb * 32, (int)grp, row);
      tma_load_3d(T2 + cb * 8192, &tmK, &bar_tma, cb * 32, (int)grp, row);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t lb = (uint32_t)(warp * 32) << 16;
  bool ok = true;
  int pending = 1;  // loads in flight (thread 0's view)
  // Score rows live in lanes 0-15 of each warp (M = 64); the lane 16 above a
  // row works on its upper 32 columns, so every lane holds 32 columns:
  // u = 32 * up + i.
  const int up = lane >> 4;
  float sq[32];  // q k^T, this lane's half row
  // phase 0: q k^T; phase 1 + hh: dout v^T of head hh
  for (int ph = 0; ph <= hpg; ++ph) {
    const int ncb = ph == 0 ? ncbk : ncbv;
    const int kdim = ph == 0 ? dk : dv;
    const int64_t h = grp * hpg + (ph == 0 ? 0 : ph - 1);
    if (ph >= 1 && warp == 0) {  // in-chunk prefix of la, times log2(e)
      warp_cumsum64(la, (b * p.L + t0) * p.H + h, p.H, len, 0.0, cs);
      __syncwarp();
      for (int t = lane; t < C; t += 32) cs[t] = t < len ? cs[t] * 1.4426950408889634f : 0.f;
    }
    ok = mbar_wait(&bar_tma, ph & 1) && ok;
    if (tid == 0 && ok) pending = 0;
    if (__syncthreads_or(!ok)) break;
    {  // round both tiles to TF32 (nearest) in place
      const int r = tid & 63, half = tid >> 6;
      const int cols = ncb * 16;
      for (int col = half * cols; col < (half + 1) * cols; col += 4) {
        float4 *a4 = reinterpret_cast<float4 *>(T1 + sw128_off(r, col, C));
        float4 *b4 = reinterpret_cast<float4 *>(T2 + sw128_off(r, col, C));
        float4 x = *a4, y = *b4;
        x.x = tf32r(x.x); x.y = tf32r(x.y); x.z = tf32r(x.z); x.w = tf32r(x.w);
        y.x = tf32r(y.x); y.y = tf32r(y.y); y.z = tf32r(y.z); y.w = tf32r(y.w);
        *a4 = x;
        *b4 = y;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {  // phase 0 -> cols [0,64); later phases -> [64,128)
      const uint32_t a = smem_u32(T1), bb = smem_u32(T2);
      const uint32_t id = idesc_tf32(64, 64);
      for (int kk = 0; kk < kdim / 8; ++kk) {
        const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
        mma_ss(tmem + (ph == 0 ? 0 : 64), sdesc(a + off), sdesc(bb + off), id, kk > 0 ? 1u : 0u);
      }
      mma_commit(&bar_mma);
    }
    ok = mbar_wait(&bar_mma, ph & 1) && ok;
    tc_fence_after();
    if (tid == 0 && ok && ph < hpg) {  // the tiles are consumed: next head's loads
      load_dv(grp * hpg + ph);
      pending = 1;
    }
    if (ph == 0) {
      float lo[32], hi[32];
      tmem_ld32(tmem + lb, lo);
      tmem_ld32(tmem + lb + 32, hi);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float x = __shfl_sync(0xffffffffu, hi[i], lane & 15);
        sq[i] = up ? x : lo[i];
      }
      continue;
    }
    float dp[32];  // dout v^T of this head, this lane's half row
    {
      float lo[32], hi[32];
      tmem_ld32(tmem + lb + 64, lo);
      tmem_ld32(tmem + lb + 96, hi);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float x = __shfl_sync(0xffffffffu, hi[i], lane & 15);
        dp[i] = up ? x : lo[i];
      }
    }
    // B_t = B_{t+1} + rowpre_t - colsuf_t with rowpre_t = sum_{u<t} M[t][u]
    // (a row of the strictly lower triangle) and colsuf_t = sum_{r>t} M[r][t]
    // (a column of it).  Row r's two halves live in lanes r % 16 and
    // r % 16 + 16 of warp r / 16; the column sums are reduce-scattered over
    // each half-warp (lane l ends with columns 32 up + 2 (l % 16) + {0, 1}),
    // then added over the four warps in shared memory.
    {
      const int r = warp * 16 + (lane & 15);
      const bool rowok = r < len;
      const float cr = cs[rowok ? r : 0];
      float *m = dp;  // M's half row, in place of dout v^T's
      float rp0 = 0.f, rp1 = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int u = 32 * up + i;
        m[i] = (rowok && u < r) ? ex2f(cr - cs[u]) * sq[i] * dp[i] : 0.f;
        if (i & 1) rp1 += m[i];
        else rp0 += m[i];
      }
      float rp = rp0 + rp1;
      rp += __shfl_xor_sync(0xffffffffu, rp, 16);  // both halves of the row
#pragma unroll
      for (int off = 8, n = 32; off >= 1; off >>= 1, n >>= 1) {
        const bool hiL = (lane & off) != 0;
#pragma unroll
        for (int k2 = 0; k2 < n / 2; ++k2) {
          const float mine = hiL ? m[n / 2 + k2] : m[k2];
          const float send = hiL ? m[k2] : m[n / 2 + k2];
          m[k2] = mine + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      const int u0 = 32 * up + 2 * (lane & 15);
      R[warp * C + u0] = m[0];
      R[warp * C + u0 + 1] = m[1];
      if (rowok && up == 0) R[4 * C + r] = rp;
    }
    __syncthreads();
    if (warp == 0) {  // suffix sums of rowpre - colsuf; lane l owns t = 2l, 2l + 1
      float dd[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int t = 2 * lane + j;
        dd[j] = t < len ? R[4 * C + t] - (R[t] + R[C + t] + R[2 * C + t] + R[3 * C + t]) : 0.f;
      }
      float x = dd[0] + dd[1];  // inclusive suffix over lanes of the pair sums
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x += y;
      }
      const float b1 = x - dd[0];  // B_{2l+1} = suffix from 2l+1
      const float b0 = x;          // B_{2l}
      float *bt = Bt + (b * p.L + t0) * p.H + h;
      if (2 * lane < len) bt[(int64_t)(2 * lane) * p.H] = b0;
      if (2 * lane + 1 < len) bt[(int64_t)(2 * lane + 1) * p.H] = b1;
    }
    __syncthreads();  // R and cs are reused by the next head
  }
  if (tid == 0 && pending) mbar_wait(&bar_tma, 0);  // best effort after a failure
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// ===========================================================================
// dlog_alpha of one segment:
//   dla_t = B_t + sum_{t' >= t in the segment} (rq_t' - rk_t') + <G_end, S_end>
// where B_t is the intra-chunk block sum, rq / rk the inter-chunk terms
// q_t.dq_inter(t) and k_t.dk_inter(t), G_end the gradient of the state at the
// segment's end (from its right) and S_end that state (the state entering the
// next segment); both are given in the same layout (each transposed, sz
// elements).  For the last segment G_end is the final state's cotangent and
// S_end the final state: Gfin and Sfin, both [dk x dv] per head, or no term
// when Gfin is NULL.  grid (nseg, H, B).
constexpr int DT = 256;
__global__ void __launch_bounds__(DT) k_dla(const float *__restrict__ Bt,
                                            const float *__restrict__ rq,
                                            const float *__restrict__ rk,
                                            const float *__restrict__ Gst,
                                            const float *__restrict__ Sst,
                                            const float *__restrict__ Gfin,
                                            const float *__restrict__ Sfin, float *__restrict__ dla,
                                            int64_t L, int64_t H, int64_t sz, int Ls, int nseg) {
  __shared__ double wred[DT / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t bh = b * H + h;
  // carry = <G_end, S_end>: float4 loads, fp32 partial sums, fp64 across threads
  float part = 0.f;
  const float4 *G = nullptr, *S = nullptr;
  if (seg + 1 < nseg) {
    G = reinterpret_cast<const float4 *>(Gst + (bh * nseg + seg) * sz);
    S = reinterpret_cast<const float4 *>(Sst + (bh * nseg + seg + 1) * sz);
  } else if (Gfin) {
    G = reinterpret_cast<const float4 *>(Gfin + bh * sz);
    S = reinterpret_cast<const float4 *>(Sfin + bh * sz);
  }
  if (G) {
    for (int64_t e = tid; e < sz / 4; e += DT) {
      const float4 g = G[e], x = S[e];
      part = fmaf(g.x, x.x, fmaf(g.y, x.y, fmaf(g.z, x.z, fmaf(g.w, x.w, part))));
    }
  }
  double dp = part;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) dp += __shfl_xor_sync(0xffffffffu, dp, o);
  if (lane == 0) wred[warp] = dp;
  __syncthreads();
  double carry = 0.0;
#pragma unroll
  for (int w2 = 0; w2 < DT / 32; ++w2) carry += wred[w2];
  __syncthreads();
  // suffix sums of rq - rk over the segment, 256 tokens at a time from its end
  const int64_t s_begin = seg * (int64_t)Ls;
  const int64_t s_end = imin64(L, s_begin + Ls);
  for (int64_t hi = s_end; hi > s_begin; hi -= DT) {
    const int64_t t = hi - DT + tid;  // thread tid owns token t (valid if t >= s_begin)
    const bool ok = t >= s_begin;
    const int64_t idx = (b * L + t) * H + h;
    double x = ok ? (double)rq[idx] - (double)rk[idx] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {  // inclusive suffix within the warp
      const double y = __shfl_down_sync(0xffffffffu, x, o);
      if (lane + o < 32) x += y;
    }
    if (lane == 0) wred[warp] = x;  // warp total
    __syncthreads();
    double after = carry;  // everything right of this warp
#pragma unroll
    for (int w2 = 0; w2 < DT / 32; ++w2)
      if (w2 > warp) after += wred[w2];
    if (ok) dla[idx] = (float)((double)Bt[idx] + x + after);
#pragma unroll
    for (int w2 = 0; w2 < DT / 32; ++w2) carry += wred[w2];
    __syncthreads();
  }
}

// ===========================================================================
// Host side.

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                        cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// 3-D view [rows, slots, d] of a row-major fp32 tensor; box = 32 features x
// 1 slot x box_rows rows, 128-byte swizzle, zero fill out of bounds.
cudaError_t make_map(CUtensorMap *m, const float *base, int64_t rows, int64_t slots, int64_t d,
                     int box_rows = C) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)slots, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)(d * 4), (cuuint64_t)(slots * d * 4)};
  cuuint32_t box[3] = {32, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

// Segment length: as many segments as fit one wave of the segment kernels
// (two CTAs per SM), so no partial second wave trails behind; measured
// faster than two full waves (1.032 -> 0.996 ms per fwd+bwd step at
// B=4, H=8, L=8192) and than 1.6 waves (1.195 ms).
void choose_segments(const Geo &g, int *Ls, int *nseg) {
  const int64_t bh = g.B * g.H;
  const int64_t want = std::max<int64_t>(1, (2 * (int64_t)num_sms()) / bh);
  int64_t ls = cdiv(cdiv(g.L, want), C) * C;
  if (ls < C) ls = C;
  *Ls = (int)std::min<int64_t>(ls, 1 << 30);
  *nseg = (int)cdiv(g.L, *Ls);
}

PassGeo make_pass(const Geo &g, int dk, int dv, bool qk_head, bool v_head) {
  PassGeo p;
  p.B = g.B; p.L = g.L; p.H = g.H; p.hpg = g.hpg;
  p.dk = dk; p.dv = dv;
  p.dkp = rup(dk, 32); p.dkn = rup(dk, 16);
  p.dvp = rup(dv, 32); p.dvn = rup(dv, 16);
  p.qk_per_head = qk_head ? 1 : 0;
  p.v_per_head = v_head ? 1 : 0;
  choose_segments(g, &p.Ls, &p.nseg);
  return p;
}

size_t state_floats(const PassGeo &p) {
  return (size_t)(p.B * p.H * p.nseg) * (size_t)p.dk * p.dv;
}

size_t seg_state_smem(const PassGeo &p) {
  return (size_t)(p.dkp / 32 + p.dvp / 32) * 4096 * 2 + (size_t)rup(p.dvn * 128, 1024) * 2 +
         NT2 * 4 + 1024;
}
size_t walk_smem(const PassGeo &p) {
  return (size_t)(p.dkp / 32) * 2 * 8192 + std::max(p.dvp / 32 * 8192, 16384) + 11 * C * 4 + 1024;
}

size_t dla_intra_smem(const PassGeo &p) {
  const int ncbm = std::max(p.dkp, p.dvp) / 32;
  return (size_t)ncbm * 2 * 8192 + (size_t)(6 * C) * 4 + 1024;  // three CTAs per SM fit
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Segment contributions and state passing of one pass: on return `states`
// holds the state entering every segment (from the left, or from the right
// when REV).
//   k' : [B*L, qk_slots, dk]   v' : [B*L, v_slots, dv]
template <bool REV>
cudaError_t run_states(const PassGeo &p, const float *kp, const float *vp, const float *la,
                       const float *h0, bool trans, float *fin, float *states, float *Aseg,
                       float *statesT, cudaStream_t s, const char *name_state) {
  cudaError_t e;
  const int64_t rows = p.B * p.L;
  const int64_t G = p.H / p.hpg;
  CUtensorMap mk, mv;
  if ((e = make_map(&mk, kp, rows, p.qk_per_head ? p.H : G, p.dk, SL)) != cudaSuccess) return e;
  if ((e = make_map(&mv, vp, rows, p.v_per_head ? p.H : G, p.dv, SL)) != cudaSuccess) return e;
  const dim3 grid((unsigned)p.nseg, (unsigned)p.H, (unsigned)p.B);
  {
    const size_t sm = seg_state_smem(p);
    if ((e = set_smem(k_seg_state<REV>, sm)) != cudaSuccess) return e;
    LaunchTrace lt(name_state, s);
    k_seg_state<REV><<<grid, NT2, sm, s>>>(mk, mv, la, states, Aseg, p);
  }
  {
    LaunchTrace lt("tc.seg_scan", s);
    const dim3 sg((unsigned)(p.B * p.H), (unsigned)cdiv((int64_t)p.dk * p.dv, 4 * NTH));
    if (trans) k_seg_scan<REV, true><<<sg, NTH, 0, s>>>(states, Aseg, h0, fin, statesT, p);
    else k_seg_scan<REV, false><<<sg, NTH, 0, s>>>(states, Aseg, h0, fin, statesT, p);
  }
  return cudaGetLastError();
}

// The walk of one pass over every segment, from the entering states.
//   q', k' : [B*L, qk_slots, dk]   v' : [B*L, v_slots, dv]
template <bool REV>
cudaError_t run_walk(const PassGeo &p, const float *qp, const float *kp, const float *vp,
                     const float *la, const float *states, bool states_t, const OutArgs &oa,
                     bool atomic, cudaStream_t s, const char *name_walk) {
  cudaError_t e;
  const int64_t rows = p.B * p.L;
  const int64_t G = p.H / p.hpg;
  CUtensorMap mq, mk, mv, mo;
  if ((e = make_map(&mq, qp, rows, p.qk_per_head ? p.H : G, p.dk)) != cudaSuccess) return e;
  if ((e = make_map(&mk, kp, rows, p.qk_per_head ? p.H : G, p.dk)) != cudaSuccess) return e;
  if ((e = make_map(&mv, vp, rows, p.v_per_head ? p.H : G, p.dv)) != cudaSuccess) return e;
  if ((e = make_map(&mo, oa.out, rows, oa.out_slots, p.dv)) != cudaSuccess) return e;
  const dim3 grid((unsigned)p.nseg, (unsigned)p.H, (unsigned)p.B);
  const size_t sm = walk_smem(p);
  LaunchTrace lt(name_walk, s);
  if (atomic) {
    if ((e = set_smem(k_walk<REV, true>, sm)) != cudaSuccess) return e;
    k_walk<REV, true><<<grid, NT2, sm, s>>>(mq, mk, mv, mo, la, states, states_t ? 1 : 0, oa, p);
  } else {
    if ((e = set_smem(k_walk<REV, false>, sm)) != cudaSuccess) return e;
    k_walk<REV, false><<<grid, NT2, sm, s>>>(mq, mk, mv, mo, la, states, states_t ? 1 : 0, oa, p);
  }
  return cudaGetLastError();
}

// A second stream of the library's own per device, on which the backward runs
// its anti-causal passes (dk, dv) while the caller's stream runs the causal one
// (dq) and the intra-chunk dlog_alpha sums: each kernel fills one wave, and the
// other pass's kernels take the SM slots its tail leaves and overlap its short
// scans.  Fork and join are events; the lock makes the enqueue of one backward
// atomic with respect to others on other host threads (the events are reused).
struct Side {
  cudaStream_t s2 = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
Side g_side[64];
std::atomic<bool> g_overlap{true};

cudaError_t get_side(Side **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  Side &sd = g_side[dev];
  if (!sd.s2) {
    if ((e = cudaStreamCreateWithFlags(&sd.s2, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &sd;
  return cudaSuccess;
}

}  // namespace

bool set_overlap(bool on) { return g_overlap.exchange(on); }
bool get_overlap() { return g_overlap.load(); }

int check_shape(int64_t dk, int64_t dv, int64_t chunk) {
  if (chunk != C) return SSD_ERR_CHUNK;
  if (dk % 8 || dv % 8 || dk > 128 || dv > 128) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

size_t fwd_workspace_bytes(const Geo &g) {
  const PassGeo p = make_pass(g, (int)g.dk, (int)g.dv, false, true);
  return sizeof(float) * (state_floats(p) + (size_t)(g.B * g.H * p.nseg));
}

// Two passes' states (both kept for dlog_alpha), their decays, three
// per-token arrays, and the final state (used only when it has a cotangent).
size_t bwd_workspace_bytes(const Geo &g) {
  const PassGeo p = make_pass(g, (int)g.dk, (int)g.dv, false, true);
  const size_t nst = state_floats(p), na = (size_t)(g.B * g.H * p.nseg);
  return sizeof(float) * (2 * nst + 2 * na + 3 * (size_t)(g.B * g.L * g.H) +
                          (size_t)(g.B * g.H * g.dk * g.dv)) + 256;
}

cudaError_t fwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                float *out, float *hT, const Geo &g, void *ws, cudaStream_t s) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  if (g.B * g.L >= (int64_t)1 << 31) return cudaErrorNotSupported;
  const PassGeo p = make_pass(g, (int)g.dk, (int)g.dv, false, true);
  float *st = static_cast<float *>(ws);
  float *Aseg = st + state_floats(p);
  if ((e = run_states<false>(p, k, v, la, h0, false, hT, st, Aseg, nullptr, s, "tc.seg_state")) != cudaSuccess)
    return e;
  OutArgs oa{out, (int)g.H, nullptr, nullptr};
  return run_walk<false>(p, q, k, v, la, st, false, oa, false, s, "tc.walk_out");
}

cudaError_t bwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                const float *dout, const float *dhT, float *dq, float *dk, float *dv, float *dla,
                float *dh0, const Geo &g, void *ws, cudaStream_t s) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  if (g.B * g.L >= (int64_t)1 << 31) return cudaErrorNotSupported;
  const int DK = (int)g.dk, DV = (int)g.dv;
  // dq_h = scan(q' = dout, k' = v, v' = k; causal; initial state h0^T)
  const PassGeo pa = make_pass(g, DV, DK, true, false);
  // dk_h = anti-causal scan(q' = v, k' = dout, v' = q)
  const PassGeo pb = make_pass(g, DV, DK, true, false);
  // dv = anti-causal scan(q' = k, k' = q, v' = dout).  Its states are the
  // transposes of pass B's (read transposed by its walk), and its leftmost
  // state is dh0.
  const PassGeo pc = make_pass(g, DK, DV, false, true);
  const size_t nst = state_floats(pa), na = (size_t)(g.B * g.H * pa.nseg);
  float *stA = static_cast<float *>(ws);
  float *stB = stA + nst;
  float *aA = stB + nst;
  float *aB = aA + na;
  float *rq = aB + na;
  float *rk = rq + g.B * g.L * g.H;
  float *Bt = rk + g.B * g.L * g.H;
  // the final state, [dk x dv] per head, needed for dlog_alpha only when it
  // has a cotangent
  float *hT = nullptr;
  if (dhT) {  // 16-byte aligned for the float4 reads of k_dla
    const uintptr_t a = reinterpret_cast<uintptr_t>(Bt + g.B * g.L * g.H);
    hT = reinterpret_cast<float *>((a + 15) & ~uintptr_t(15));
  }
  const bool grouped = g.hpg > 1;
  if (grouped) {
    if ((e = cudaMemsetAsync(dq, 0, sizeof(float) * g.B * g.L * g.G * g.dk, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dk, 0, sizeof(float) * g.B * g.L * g.G * g.dk, s)) != cudaSuccess) return e;
  }
  const int oslots = grouped ? (int)g.G : (int)g.H;
  // The dk / dv passes (pass B's states, both anti-causal walks) run on the
  // side stream, forked from s after the memsets and joined before k_dla
  // (or on s itself when overlap is off).
  const bool overlap = g_overlap.load();
  std::unique_lock<std::mutex> lock(g_side_mu, std::defer_lock);
  Side *sd = nullptr;
  if (overlap) {
    lock.lock();
    if ((e = get_side(&sd)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(sd->fork, s)) == cudaErrorInvalidResourceHandle ||
        e == cudaErrorContextIsDestroyed) {
      // the cached handles died with a device reset: make new ones once
      cudaGetLastError();
      *sd = Side{};
      if ((e = get_side(&sd)) != cudaSuccess) return e;
      e = cudaEventRecord(sd->fork, s);
    }
    if (e != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(sd->s2, sd->fork, 0)) != cudaSuccess) return e;
  }
  cudaStream_t s2 = overlap ? sd->s2 : s;
  cudaError_t eb = run_states<true>(pb, dout, q, la, dhT, true, dh0, stB, aB, nullptr, s2, "tc.seg_state_dk");
  OutArgs okk{dk, oslots, k, rk};
  if (eb == cudaSuccess) eb = run_walk<true>(pb, v, dout, q, la, stB, false, okk, grouped, s2, "tc.walk_dk");
  OutArgs ov{dv, (int)g.H, nullptr, nullptr};
  if (eb == cudaSuccess) eb = run_walk<true>(pc, k, q, dout, la, stB, true, ov, false, s2, "tc.walk_dv");
  // whatever was enqueued on s2 is joined back into s before this returns,
  // even after an error (the caller frees the workspace on s)
  cudaError_t ej = overlap ? cudaEventRecord(sd->join, s2) : cudaSuccess;
  auto join = [&]() -> cudaError_t {
    if (!overlap || ej != cudaSuccess) return ej;
    return cudaStreamWaitEvent(s, sd->join, 0);
  };
  if (eb != cudaSuccess) {
    join();
    return eb;
  }
  // pass A and the intra-chunk sums on s, meanwhile
  auto on_s = [&]() -> cudaError_t {
    cudaError_t ea = run_states<false>(pa, v, k, la, h0, true, hT, stA, aA, nullptr, s, "tc.seg_state_dq");
    if (ea != cudaSuccess) return ea;
    OutArgs oq{dq, oslots, q, rq};
    if ((ea = run_walk<false>(pa, dout, v, k, la, stA, false, oq, grouped, s, "tc.walk_dq")) != cudaSuccess)
      return ea;
    // intra-chunk block sums of dlog_alpha
    const PassGeo pi = make_pass(g, DK, DV, false, true);
    CUtensorMap mq, mk, mv, md;
    const int64_t rows = g.B * g.L;
    if ((ea = make_map(&mq, q, rows, g.G, DK)) != cudaSuccess) return ea;
    if ((ea = make_map(&mk, k, rows, g.G, DK)) != cudaSuccess) return ea;
    if ((ea = make_map(&mv, v, rows, g.H, DV)) != cudaSuccess) return ea;
    if ((ea = make_map(&md, dout, rows, g.H, DV)) != cudaSuccess) return ea;
    const size_t sm = dla_intra_smem(pi);
    if ((ea = set_smem(k_dla_intra, sm)) != cudaSuccess) return ea;
    LaunchTrace lt("tc.dla_intra", s);
    k_dla_intra<<<dim3((unsigned)g.N, (unsigned)g.G, (unsigned)g.B), NTH, sm, s>>>(mq, mk, mv, md,
                                                                                  la, Bt, pi);
    return cudaGetLastError();
  };
  const cudaError_t ea = on_s();
  if ((e = join()) != cudaSuccess) return e;
  if (ea != cudaSuccess) return ea;
  {  // pass A's states are S^T, pass B's are G^T: the carry is their plain dot
    LaunchTrace lt("tc.dla", s);
    k_dla<<<dim3((unsigned)pa.nseg, (unsigned)g.H, (unsigned)g.B), DT, 0, s>>>(
        Bt, rq, rk, stB, stA, dhT, hT, dla, g.L, g.H, DK * DV, pa.Ls, pa.nseg);
  }
  return cudaGetLastError();
}

cudaError_t read_and_clear_error(unsigned int *word) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned int));
}

}  // namespace tc
}  // namespace ssd
