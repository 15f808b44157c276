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
// multiple of the 64-token chunk), about one segment per SM in all:
//   k_seg_state  each segment's zero-initial-state contribution (one contraction)
//   k_seg_scan   the states entering every segment (sequential over segments)
//   k_walk       each segment's chunks in order, the running state resident in
//                tensor memory
//
// Operand layouts.  A product that contracts over features (q' k'^T, the
// state times q') takes K-major operands: TMA tiles in the 128-byte swizzle.
// A product that contracts over tokens (P v', the state update v'^T (w k'))
// takes MN-major operands: TMA tiles in the 128-byte swizzle with 32-byte
// atoms, the only layout in which the tensor cores read fp32 operands
// transposed.  So no operand is ever transposed by the threads; they only
// scale (w k') and mask (P).  TMA-fed operands are truncated to TF32 by the
// tensor core; operands written by threads are rounded to nearest.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <utility>

#include <cudaTypedefs.h>

#include "../../include/ssd.h"
#include "common.cuh"
#include "tc.h"
#include "tc_common.cuh"

namespace ssd {
namespace tc {

constexpr int C = 64;     // chunk length of the tensor-core path
constexpr int NTH = 128;  // threads per CTA of the small kernels
constexpr float LOG2E = 1.4426950408889634f;
constexpr double LOG2E_D = 1.4426950408889634;

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
// (n_la: elements of la, for the debug build's index checks)
__device__ inline double warp_cumsum64(const float *__restrict__ la, int64_t n_la, int64_t first,
                                       int64_t stride, int n, double carry, float *cs) {
  const int l = threadIdx.x & 31;
  const double x0 = (2 * l < n) ? (double)LDC(la, first + (int64_t)(2 * l) * stride, n_la) : 0.0;
  const double x1 = (2 * l + 1 < n) ? (double)LDC(la, first + (int64_t)(2 * l + 1) * stride, n_la) : 0.0;
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
  int wide_k, wide_v;  // the q'/k' (v') maps load all feature blocks of a row in one box
};

// The feature blocks [0, nblk) of a 64-row tile, 8 KB apart in shared memory
// (the layout of one 32-feature box per block): one 4-D box when the map is
// wide, else one 3-D box per block.  Fewer, larger boxes: the load unit's
// issue rate, not DRAM, bounds the walks' tile loads.
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *map, uint64_t *bar, int nblk,
                                          int slot, int row, int wide) {
  if (wide) {
    tma_load_4d(dst, map, bar, 0, row, 0, slot);
  } else {
    for (int cb = 0; cb < nblk; ++cb) tma_load_3d(dst + cb * 8192, map, bar, cb * 32, slot, row);
  }
}

__device__ __forceinline__ int qk_slot(const PassGeo &p, int64_t h) {
  return (int)(p.qk_per_head ? h : h / p.hpg);
}
__device__ __forceinline__ int v_slot(const PassGeo &p, int64_t h) {
  return (int)(p.v_per_head ? h : h / p.hpg);
}

// ===========================================================================
// Segment contraction, the zero-initial-state contribution of one segment,
// stored as the pass's state [dk' x dv'] (row-major):
//   causal      D = sum_u exp(A_seg - cs_u) k'_u v'_u^T   (evaluated at its end)
//   anti-causal D = sum_u exp(cs_u) k'_u v'_u^T           (evaluated at its start)
// with cs the in-segment inclusive prefix of la and A_seg its total (also
// written).  grid (nseg, H, B), one CTA per SM, 192 threads.  Per 64-token
// slice, both products on the tensor cores, operands straight from TMA:
//   T^T  = v'^T W           (W = diag(w) of the slice, K-major in shared memory)
//   D^T += T^T k'           (T^T from tensor memory, k' MN-major)
// so that no thread pass touches the k' / v' tiles (thread reads of shared
// memory are slow while the tensor cores stream from it).  Warp 0 issues the
// TMA loads (three-stage ring; no L2 prefetches: the load unit issues their
// boxes at the rate of loads, and the ring alone was faster), warp 1 the MMAs,
// warps 2-5 compute the weights into W (double-buffered; only its diagonal is
// rewritten) and finally stage D in shared memory for one bulk store.  Tensor memory: D^T [0,128) (lane = v'
// feature, column = k' feature), T^T [128,256) (two buffers).
constexpr int SL = 64;          // slice length
constexpr int SS_STAGES = 3;    // slices in flight
constexpr int SS_THREADS = 192;
template <bool REV>
__global__ void __launch_bounds__(SS_THREADS, 1) k_seg_state(const __grid_constant__ CUtensorMap tmK,
                                                             const __grid_constant__ CUtensorMap tmV,
                                                             const float *__restrict__ la,
                                                             float *__restrict__ states,
                                                             float *__restrict__ Aseg, PassGeo p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_align1024(smem_raw);
  const int ncbk = p.dkp / 32, ncbv = p.dvp / 32;
  constexpr uint32_t BLK = SL * 128;           // one 32-feature block of a slice
  const uint32_t kbytes = (uint32_t)ncbk * BLK;
  const uint32_t stage = kbytes + 4 * BLK;     // k' blocks, then all four v' blocks
  auto Kt = [&](int st) { return smem + st * stage; };
  auto Vt = [&](int st) { return smem + st * stage + kbytes; };
  uint8_t *Wb = smem + SS_STAGES * stage;      // [2][SL x SL] K-major, 2 column blocks each
  __shared__ uint64_t full[SS_STAGES], empty[SS_STAGES], w_full[2], w_free[2], done;
  __shared__ uint32_t tmem_base;
  __shared__ double wred[4];
  __shared__ int abort_flag;
  volatile int *ab = &abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t bh = b * p.H + h;
  const int64_t s_begin = seg * (int64_t)p.Ls;
  const int64_t s_end = imin64(p.L, s_begin + p.Ls);
  const int nsl = (int)cdiv(s_end - s_begin, SL);
  const int kslot = qk_slot(p, h), vslot = v_slot(p, h);
  const int64_t n_la = p.B * p.L * p.H, n_seg = p.B * p.H * p.nseg;

  if (warp == 1) tmem_alloc(&tmem_base, 256);
  if (tid == 0) {
    for (int i = 0; i < SS_STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {  // (W buffers)
      mbar_init(&w_full[i], 32);
      mbar_init(&w_free[i], 1);
    }
    mbar_init(&done, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  // v' blocks past dv' are read by the M = 128 MMAs: keep them zero; W is
  // zero off its diagonal
  for (int st = 0; st < SS_STAGES; ++st)
    for (int e = ncbv * (int)BLK / 16 + tid; e < 4 * (int)BLK / 16; e += SS_THREADS)
      reinterpret_cast<float4 *>(Vt(st))[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int e = tid; e < 2 * 2 * (int)BLK / 16; e += SS_THREADS)
    reinterpret_cast<float4 *>(Wb)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t T_D = tmem, T_T = tmem + 128;

  if (warp == 0) {
    if (lane == 0) {  // producer
      int last[SS_STAGES];
      for (int i = 0; i < SS_STAGES; ++i) last[i] = -1;
      for (int n = 0; n < nsl; ++n) {
        const int st = n % SS_STAGES, use = n / SS_STAGES;
        if (use > 0 && !mbar_wait(&empty[st], (use - 1) & 1, ab)) break;
        const int row = (int)(b * p.L + s_begin + (int64_t)n * SL);
        mbar_expect_tx(&full[st], kbytes + (uint32_t)ncbv * BLK);
        load_tile(Kt(st), &tmK, &full[st], ncbk, kslot, row, p.wide_k);
        load_tile(Vt(st), &tmV, &full[st], ncbv, vslot, row, p.wide_v);
        last[st] = n;
      }
      // loads still in flight must land before the CTA exits
      for (int st = 0; st < SS_STAGES; ++st)
        if (last[st] >= 0) mbar_wait(&full[st], (last[st] / SS_STAGES) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t id_t = idesc_tf32(128, SL, 1, 0);       // T^T = v'^T W
      const uint32_t id_d = idesc_tf32(128, p.dkp, 0, 1);    // D^T += T^T k'
      // T^T of slice n goes to buffer n & 1, and the D MMAs of slice n - 1 are
      // issued after the T MMAs of slice n: consecutive MMA groups never wait
      // for each other's results in tensor memory
      auto issue_d = [&](int n) {
        const int st = n % SS_STAGES;
        const uint64_t dk_ = sdesc_mn(smem_u32(Kt(st)), BLK);
#pragma unroll
        for (int kk = 0; kk < SL / 8; ++kk)
          mma_ts(T_D, T_T + (n & 1) * SL + kk * 8, dk_ + (uint64_t)(kk * 64), id_d, (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&empty[st]);
      };
      bool ok = true;
      for (int n = 0; n < nsl; ++n) {
        const int st = n % SS_STAGES, use = n / SS_STAGES, wb = n & 1;
        if (!mbar_wait(&full[st], use & 1, ab)) { ok = false; break; }
        if (!mbar_wait(&w_full[wb], (n >> 1) & 1, ab)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dv_ = sdesc_mn(smem_u32(Vt(st)), BLK);
        const uint64_t dw = sdesc(smem_u32(Wb + wb * 2 * BLK));
#pragma unroll
        for (int kk = 0; kk < SL / 8; ++kk)
          mma_ss(T_T + wb * SL, dv_ + (uint64_t)(kk * 64), dw + (uint64_t)((kk >> 2) * (BLK >> 4) + (kk & 3) * 2),
                 id_t, kk > 0 ? 1u : 0u);
        mma_commit(&w_free[wb]);
        if (n > 0) issue_d(n - 1);
      }
      if (ok && nsl > 0) issue_d(nsl - 1);
      mma_commit(&done);  // every MMA issued above has completed when this arrives
      mbar_wait(&done, 0);
    }
  } else {  // warps 2-5: weights into W, then the result
    const int wt = tid - 64, wq = warp & 3;
    static_assert(SL == 64, "two tokens per lane");
    // (warp 2, lane l: tokens 2l and 2l + 1 of slice n)
    auto la_of = [&](int n, int u) {
      const int64_t t = s_begin + (int64_t)n * SL + u;
      return (n < nsl && t < s_end) ? (double)LDC(la, (b * p.L + t) * p.H + h, n_la) : 0.0;
    };
    // la of the next WLA slices is in flight while the current WLA slices'
    // weights are made: an L2 round trip takes longer than a slice's MMAs.
    // The first ones are requested before the segment sum below.
    constexpr int WLA = 4;
    double xc0[WLA], xc1[WLA];
    if (warp == 2) {
#pragma unroll
      for (int u = 0; u < WLA; ++u) {
        xc0[u] = la_of(u, 2 * lane);
        xc1[u] = la_of(u, 2 * lane + 1);
      }
    }
    // The causal weights exp(A_seg - cs_u) need the segment's total first
    // (all four warps, one batch of loads per thread); the anti-causal ones
    // do not, and their total is the weights warp's running sum at the end.
    double tot = 0.0;
    if (!REV) {
      double part = 0.0;
#pragma unroll 16
      for (int64_t t = s_begin + wt; t < s_end; t += 128) part += (double)LDC(la, (b * p.L + t) * p.H + h, n_la);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == 0) wred[warp - 2] = part;
      named_sync(1, 128);
      tot = wred[0] + wred[1] + wred[2] + wred[3];
      if (wt == 0) STC(Aseg, bh * p.nseg + seg, n_seg, (float)tot);
    }
    bool ok = true;
    if (warp == 2) {  // one warp writes the diagonal: lane l owns tokens 2l, 2l + 1
      double carry = 0.0;
      double xn0[WLA], xn1[WLA];
      for (int n0 = 0; ok && n0 < nsl; n0 += WLA) {
#pragma unroll
        for (int u = 0; u < WLA; ++u) {
          xn0[u] = la_of(n0 + WLA + u, 2 * lane);
          xn1[u] = la_of(n0 + WLA + u, 2 * lane + 1);
        }
#pragma unroll
        for (int u = 0; u < WLA; ++u) {
          const int n = n0 + u;
          if (n >= nsl) break;
          const int wb = n & 1;
          const int64_t t0 = s_begin + (int64_t)n * SL;
          const int len = (int)imin64(SL, s_end - t0);
          const double x0 = xc0[u], x1 = xc1[u];
          double incl = x0 + x1;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const double cs1 = carry + incl, cs0 = cs1 - x1;
          carry += __shfl_sync(0xffffffffu, incl, 31);
          const float w0 = 2 * lane < len ? exp2f((float)((REV ? cs0 : tot - cs0) * LOG2E_D)) : 0.f;
          const float w1 = 2 * lane + 1 < len ? exp2f((float)((REV ? cs1 : tot - cs1) * LOG2E_D)) : 0.f;
          if (n >= 2 && !mbar_wait_all(&w_free[wb], ((n >> 1) - 1) & 1, ab)) { ok = false; break; }
          float *W = reinterpret_cast<float *>(Wb + wb * 2 * BLK);
          STC(W, sw128_off(2 * lane, 2 * lane, SL) / 4, 2 * BLK / 4, tf32r(w0));
          STC(W, sw128_off(2 * lane + 1, 2 * lane + 1, SL) / 4, 2 * BLK / 4, tf32r(w1));
          fence_async_smem();
          mbar_arrive(&w_full[wb]);
        }
#pragma unroll
        for (int u = 0; u < WLA; ++u) {
          xc0[u] = xn0[u];
          xc1[u] = xn1[u];
        }
      }
      if (REV && ok && lane == 0) STC(Aseg, bh * p.nseg + seg, n_seg, (float)carry);
    }
    // warps 2-5 take the decision together (a barrier that ORs their
    // failures), since the store below meets at a named barrier: a give-up of
    // the weights warp, or a wait that ran out, leaves all four out of it
    const bool fin = ok && mbar_wait_all(&done, 0, ab);  // (ok is uniform over each warp)
    if (!named_sync_or(1, 128, !fin)) {
      tc_fence_after();
      // D^T in tensor memory (lane j = v' feature, column i = k' feature) ->
      // the state [dk' x dv'] in the free stage-0 buffer (every slice's MMAs
      // have completed), then one bulk copy to global memory
      const int j = 32 * wq + lane;
      const int64_t sz = (int64_t)p.dk * p.dv, dst = (bh * p.nseg + seg) * sz;
      float *Dst = reinterpret_cast<float *>(Kt(0));  // sz <= dkp * 128 floats fit a stage
      for (int c0 = 0; c0 < p.dkp; c0 += 32) {
        float v[32];
        tmem_ld32(T_D + ((uint32_t)(32 * wq) << 16) + c0, v);
        if (j < p.dv) {
#pragma unroll
          for (int ii = 0; ii < 32; ++ii)
            if (c0 + ii < p.dk) STC(Dst, (int64_t)(c0 + ii) * p.dv + j, sz, v[ii]);
        }
      }
      fence_async_smem();
      named_sync(1, 128);
      if (wt == 0) {  // (dst and sz are multiples of 64 floats: 16-byte aligned)
        bulk_store(states + dst, Dst, (uint32_t)(sz * 4));
        bulk_commit_group();
        bulk_wait_all();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 256);
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
// is given, every result is also written there transposed.  With tfast (the
// block's 4*NTH elements are R = 4*NTH/dv whole rows, R a multiple of 4 that
// divides dk) every transposed read or write (init, fin, stT) goes through a
// shared-memory tile, so that each thread moves four consecutive elements of
// one transposed row as a float4; otherwise element by element.
// grid (B*H, ceil(dk*dv / (4*128))), dk*dv a multiple of 4
constexpr int SU = 10;
template <bool REV, bool TRANS>
__global__ void __launch_bounds__(NTH) k_seg_scan(float *__restrict__ st,
                                                  const float *__restrict__ Aseg,
                                                  const float *__restrict__ init,
                                                  float *__restrict__ fin,
                                                  float *__restrict__ stT, PassGeo p, int tfast) {
  __shared__ float4 tile[NTH];
  const int64_t bh = blockIdx.x;
  const int64_t e0 = 4 * ((int64_t)blockIdx.y * NTH + threadIdx.x);
  const int64_t sz = (int64_t)p.dk * p.dv;
  if (e0 >= sz) return;  // (never with tfast: the blocks cover sz exactly)
  auto tpos = [&](int64_t e) { return (e % p.dv) * p.dk + e / p.dv; };  // transposed position
  float4 *q = reinterpret_cast<float4 *>(st);
  const int64_t sz4 = sz / 4, qb = (bh * p.nseg * sz + e0) / 4;  // (sz and e0 multiples of 4)
  const int64_t n_st = p.B * p.H * p.nseg * sz, n_a = p.B * p.H * p.nseg, n_h = p.B * p.H * sz;
  // tfast: this thread's float4 of the transposed block is column jj, rows
  // i0 + 4 r4 .. + 3 (offset tq from a matrix's start); the tile holds the
  // block row-major, thread t's own four elements at tile[t]
  const int R = tfast ? 4 * NTH / p.dv : 4, nq = R / 4;
  const int jj = (int)threadIdx.x / nq, r4 = (int)threadIdx.x % nq;
  const int64_t tq = (int64_t)jj * p.dk + (int64_t)blockIdx.y * R + 4 * r4;
  float *tf = reinterpret_cast<float *>(tile);
  auto col_of_tile = [&]() {
    return make_float4(tf[(4 * r4) * p.dv + jj], tf[(4 * r4 + 1) * p.dv + jj], tf[(4 * r4 + 2) * p.dv + jj],
                       tf[(4 * r4 + 3) * p.dv + jj]);
  };
  float4 x[SU];
  float d[SU];
  auto load_batch = [&](int k0) {
#pragma unroll
    for (int u = 0; u < SU; ++u) {
      const int k = k0 + u;
      if (k < p.nseg) {
        const int s = REV ? p.nseg - 1 - k : k;
        x[u] = LDC(q, qb + (int64_t)s * sz4, n_st / 4);
        d[u] = expf(LDC(Aseg, bh * p.nseg + s, n_a));
      }
    }
  };
  load_batch(0);  // (in flight while the initial state is fetched)
  float run[4] = {0.f, 0.f, 0.f, 0.f};
  if (init && TRANS && tfast) {  // a float4 of the transposed block, turned round in the tile
    const float4 t4 = LDC(reinterpret_cast<const float4 *>(init), (bh * sz + tq) / 4, n_h / 4);
    tf[(4 * r4) * p.dv + jj] = t4.x;
    tf[(4 * r4 + 1) * p.dv + jj] = t4.y;
    tf[(4 * r4 + 2) * p.dv + jj] = t4.z;
    tf[(4 * r4 + 3) * p.dv + jj] = t4.w;
    __syncthreads();
    const float4 r = tile[threadIdx.x];
    run[0] = r.x, run[1] = r.y, run[2] = r.z, run[3] = r.w;
  } else if (init && TRANS) {
#pragma unroll
    for (int j = 0; j < 4; ++j) run[j] = LDC(init, bh * sz + tpos(e0 + j), n_h);
  } else if (init) {
    const float4 r = LDC(reinterpret_cast<const float4 *>(init), (bh * sz + e0) / 4, n_h / 4);
    run[0] = r.x, run[1] = r.y, run[2] = r.z, run[3] = r.w;
  }
  for (int k0 = 0; k0 < p.nseg; k0 += SU) {
    if (k0 > 0) load_batch(k0);
#pragma unroll
    for (int u = 0; u < SU; ++u) {
      const int k = k0 + u;
      if (k < p.nseg) {
        const int s = REV ? p.nseg - 1 - k : k;
        STC(q, qb + (int64_t)s * sz4, n_st / 4, make_float4(run[0], run[1], run[2], run[3]));
        if (stT && tfast) {
          __syncthreads();  // the tile's previous contents are read
          tile[threadIdx.x] = make_float4(run[0], run[1], run[2], run[3]);
          __syncthreads();
          STC(reinterpret_cast<float4 *>(stT), (bh * p.nseg * sz + (int64_t)s * sz + tq) / 4, n_st / 4,
              col_of_tile());
        } else if (stT) {
#pragma unroll
          for (int j = 0; j < 4; ++j) STC(stT, bh * p.nseg * sz + (int64_t)s * sz + tpos(e0 + j), n_st, run[j]);
        }
        run[0] = fmaf(d[u], run[0], x[u].x);
        run[1] = fmaf(d[u], run[1], x[u].y);
        run[2] = fmaf(d[u], run[2], x[u].z);
        run[3] = fmaf(d[u], run[3], x[u].w);
      }
    }
  }
  if (fin && TRANS && tfast) {
    __syncthreads();
    tile[threadIdx.x] = make_float4(run[0], run[1], run[2], run[3]);
    __syncthreads();
    STC(reinterpret_cast<float4 *>(fin), (bh * sz + tq) / 4, n_h / 4, col_of_tile());
  } else if (fin && TRANS) {
#pragma unroll
    for (int j = 0; j < 4; ++j) STC(fin, bh * sz + tpos(e0 + j), n_h, run[j]);
  } else if (fin) {
    STC(reinterpret_cast<float4 *>(fin), (bh * sz + e0) / 4, n_h / 4, make_float4(run[0], run[1], run[2], run[3]));
  }
}

// ===========================================================================
// Walk over the chunks of one segment (left to right, or right to left when
// REV) with the running state resident in tensor memory.  grid (nseg, H, B),
// one CTA per SM, 384 threads (512 when SPLIT) in warp-specialised roles:
//   warp 0      TMA producer: q', k' (K-major) and v' (MN-major) tiles of each
//               chunk into a two-stage ring
//   warp 1      state-chain MMAs of chunk c:  X = S^T q'^T (inter term),
//               Y = v'^T P^T (intra term), S^T += v'^T (w k') (update)
//   warp 2      score MMAs  Sc = q' k'^T  of the next chunk
//   warp 3      decay factors of each chunk (fp64 in-chunk prefix of la, the
//               lazy state scale) into a four-slot ring
//   warps 4-7   mask: v' rounded to TF32 in place, P = D o Sc into shared
//               memory (K-major), and k' turned in place into w k'
//               (MN-major, scaled by the state weights, rounded to TF32)
//   warps 8-11  epilogue: out'_t = f_t X_t + Y_t to global memory (atomic
//               add over a group's heads when ATOMIC), dcs_t = y_t . f_t X_t
//               when SPLIT, and the occasional explicit state rescale
//   warps 12-15 (SPLIT) a second epilogue group: each group takes two of a
//               chunk's four 16-token steps
// so the next chunk's scores and mask overlap the current chunk's products.
//
// Tensor memory (512 columns): S^T [0,128) (lane j = v' feature, column i =
// k' feature), Sc [128,256) two 64-column buffers (M = 64: row r in lane
// 32(r/16) + r%16), X [256,384) and Y [384,512) two buffers each (lane j,
// column = token).  Shared memory per stage: q' tile (128-byte swizzle,
// K-major), k' tile (the same, later w k' in the 32-byte-atom layout),
// v' tile (32-byte-atom layout, all four 32-feature blocks so that the M = 128
// MMAs read zeros past dv'); one P tile [64 x 64].
//
// The stored state is kept as Hs with the true state = alpha * Hs.  While
// alpha stays in [2^-40, 2^40] a chunk's decay is folded into alpha (the
// inter term takes f_t * alpha, the update w / alpha'), so no pass over the
// state runs; otherwise the epilogue warps rescale Hs to the true decayed state
// between the chunk's inter product and its update, and alpha returns to 1.
//
// The entering state is read from Hseg as [dk' x dv'] (or [dv' x dk'] when
// hseg_t).
constexpr int WT = 384;
// The walks with per-token dots (SPLIT) add a second epilogue warpgroup
// (warps 12-15): each group takes half of every chunk's tokens, since their
// epilogue, not the state chain, paced those walks.  All roles still fit 128
// registers a thread at 512 threads.
__host__ __device__ constexpr int walk_threads(bool split) { return split ? 512 : WT; }
struct Fac {     // decay factors of one chunk, walk order
  float cs2[C];  // in-chunk inclusive prefix of la, times log2(e) (0 past the end)
  float qf[C];   // inter-term factor of query row t times the state scale
  float kw[C];   // state-update weight of key row s over the new state scale
  float an;      // the rescale factor (state scale times the chunk's decay)
  int rescale;   // 1: rescale the stored state before this chunk's update
};
struct WalkOut {
  float *out;       // out'[b, t, slot, 0:dv']
  int out_slots;    // H (slot = head) or G (slot = group, summed by atomic adds)
  const float *y;   // SPLIT: y[b, t, h / hpg, 0:dv']
  float *dcs;       // SPLIT: dcs[b, t, h] = y_t . (inter-chunk part of out'_t)
};

template <bool REV, bool ATOMIC, bool SPLIT>
__global__ void __launch_bounds__(walk_threads(SPLIT), 1) k_walk(const __grid_constant__ CUtensorMap tmQ,
                                              const __grid_constant__ CUtensorMap tmK,
                                              const __grid_constant__ CUtensorMap tmV,
                                              const float *__restrict__ la,
                                              const float *__restrict__ Hseg, int hseg_t,
                                              WalkOut oa, PassGeo p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_align1024(smem_raw);
  const int ncbk = p.dkp / 32, ncbv = p.dvp / 32;
  constexpr uint32_t BLK = C * 128;  // one 32-feature block of a 64-row tile
  const uint32_t qkbytes = (uint32_t)ncbk * BLK;
  const uint32_t stage = 2 * qkbytes + 4 * BLK;
  auto Qs = [&](int st) { return smem + st * stage; };
  auto Ks = [&](int st) { return smem + st * stage + qkbytes; };
  auto Vs = [&](int st) { return smem + st * stage + 2 * qkbytes; };
  uint8_t *P = smem + 2 * stage;
  Fac *fac = reinterpret_cast<Fac *>(P + 2 * BLK);
  float *red = reinterpret_cast<float *>(fac + 4);  // [4][64]

  __shared__ uint64_t full[2], empty[2], s_full[2], s_empty[2], xy_full[2], x_empty[2];
  // The mask signals P (p_full) before it turns k' into w k' (wk_full, one
  // barrier per stage), so that the intra-term MMAs issue during the turn
  __shared__ uint64_t p_full, p_empty, rescaled, st_init, drain_s, drain_m, wk_full[2];
  __shared__ uint64_t fac_full[4], fac_empty[4];
  // never: a barrier nothing arrives on (the failure-path test waits on it)
  __shared__ uint64_t never;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  volatile int *ab = &abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t bh = b * p.H + h;
  const int64_t s_begin = seg * (int64_t)p.Ls;
  const int64_t s_end = imin64(p.L, s_begin + p.Ls);
  const int nc = (int)cdiv(s_end - s_begin, C);
  const int kslot = qk_slot(p, h), vslot = v_slot(p, h);
  const int dk = p.dk, dv = p.dv;
  auto chunk_of = [&](int ci) { return REV ? nc - 1 - ci : ci; };
  const int64_t n_la = p.B * p.L * p.H;  // element counts (debug-build index checks)
  constexpr int NEG = SPLIT ? 2 : 1;     // epilogue warpgroups

  if (warp == 1) tmem_alloc(&tmem_base, 512);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 128);
      mbar_init(&xy_full[i], 1);
      mbar_init(&x_empty[i], 128 * NEG);
      mbar_init(&wk_full[i], 128);
    }
    mbar_init(&p_full, 128);
    mbar_init(&p_empty, 1);
    mbar_init(&rescaled, 128);
    mbar_init(&st_init, 128);
    mbar_init(&drain_s, 1);
    mbar_init(&drain_m, 1);
    mbar_init(&never, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&fac_full[i], 32);
      mbar_init(&fac_empty[i], 129 + 128 * NEG);
    }
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  // v' blocks past dv' are read by the M = 128 MMAs: keep them zero
  for (int st = 0; st < 2; ++st)
    for (int e = ncbv * (int)BLK / 16 + tid; e < 4 * (int)BLK / 16; e += WT)
      reinterpret_cast<float4 *>(Vs(st))[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t T_ST = tmem, T_SC = tmem + 128, T_X = tmem + 256, T_Y = tmem + 384;

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------
    if (lane == 0) {
      int last[2] = {-1, -1};
      for (int ci = 0; ci < nc; ++ci) {
        const int st = ci & 1;
        if (ci >= 2 && !mbar_wait(&empty[st], ((ci >> 1) - 1) & 1, ab)) break;
        const int row = (int)(b * p.L + s_begin + (int64_t)chunk_of(ci) * C);
        mbar_expect_tx(&full[st], 2 * qkbytes + (uint32_t)ncbv * BLK);
        load_tile(Qs(st), &tmQ, &full[st], ncbk, kslot, row, p.wide_k);
        load_tile(Ks(st), &tmK, &full[st], ncbk, kslot, row, p.wide_k);
        load_tile(Vs(st), &tmV, &full[st], ncbv, vslot, row, p.wide_v);
        last[st] = ci;
        // (No L2 prefetch of later chunks: the tensor-memory-access unit
        // issues prefetch boxes at the same rate as loads, and the walks ran
        // 15 % faster without them; a chunk's loads are requested one chunk
        // ahead, which covers their latency.)
      }
      for (int st = 0; st < 2; ++st)  // loads in flight must land before the CTA exits
        if (last[st] >= 0) mbar_wait(&full[st], (last[st] >> 1) & 1);
    }
  } else if (warp == 1) {
    // ---- state-chain MMAs ----------------------------------------------------
    if (lane == 0) {
      const uint32_t id_x = idesc_tf32(128, 64), id_y = idesc_tf32(128, 64, 1, 0);
      const uint32_t id_u = idesc_tf32(128, p.dkp, 1, 1);  // N a whole number of 32-wide atoms
      const uint64_t dp = sdesc(smem_u32(P));
      int nres = 0;
      if (mbar_wait(&st_init, 0, ab)) {
        for (int ci = 0; ci < nc; ++ci) {
          const int st = ci & 1, xb = ci & 1, slot = ci & 3;
          if (!mbar_wait(&full[st], (ci >> 1) & 1, ab)) break;
          if (ci >= 2 && !mbar_wait(&x_empty[xb], ((ci >> 1) - 1) & 1, ab)) break;
          tc_fence_after();
          // descriptors advance by adds in 16-byte units: K-major K steps are
          // 32 B inside a 128-byte row and BLK between column blocks, MN-major
          // K steps are 8 rows (1024 B)
          const uint64_t dq = sdesc(smem_u32(Qs(st))), dkm = sdesc_mn(smem_u32(Ks(st)), BLK);
          const uint64_t dvm = sdesc_mn(smem_u32(Vs(st)), BLK);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)  // X = S^T q'^T
            if (kk < dk / 8)
              mma_ts(T_X + xb * 64, T_ST + kk * 8, dq + (uint64_t)((kk >> 2) * (BLK >> 4) + (kk & 3) * 2),
                     id_x, kk > 0 ? 1u : 0u);
          if (!mbar_wait(&p_full, ci & 1, ab)) break;  // P is in place
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C / 8; ++kk)  // Y = v'^T P^T
            mma_ss(T_Y + xb * 64, dvm + (uint64_t)(kk * 64), dp + (uint64_t)((kk >> 2) * (BLK >> 4) + (kk & 3) * 2),
                   id_y, kk > 0 ? 1u : 0u);
          mma_commit(&xy_full[xb]);
          mma_commit(&p_empty);
          if (!mbar_wait(&fac_full[slot], (ci >> 2) & 1, ab)) break;
          const int resc = fac[slot].rescale;
          mbar_arrive(&fac_empty[slot]);
          if (!mbar_wait(&wk_full[st], (ci >> 1) & 1, ab)) break;  // w k' is in place
          if (resc) {
            if (!mbar_wait(&rescaled, nres & 1, ab)) break;
            ++nres;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C / 8; ++kk)  // S^T += v'^T (w k')
            mma_ss(T_ST, dvm + (uint64_t)(kk * 64), dkm + (uint64_t)(kk * 64), id_u, 1u);
          mma_commit(&empty[st]);
        }
      }
      mma_commit(&drain_m);  // arrives once every MMA issued above has completed
      mbar_wait(&drain_m, 0);
    }
  } else if (warp == 2) {
    // ---- score MMAs ----------------------------------------------------------
    if (lane == 0) {
      const uint32_t id_s = idesc_tf32(64, 64);
      for (int ci = 0; ci < nc; ++ci) {
        const int st = ci & 1, sb = ci & 1;
        if (!mbar_wait(&full[st], (ci >> 1) & 1, ab)) break;
        if (ci >= 2 && !mbar_wait(&s_empty[sb], ((ci >> 1) - 1) & 1, ab)) break;
        tc_fence_after();
        const uint64_t dq = sdesc(smem_u32(Qs(st))), dkk = sdesc(smem_u32(Ks(st)));
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          if (kk < dk / 8) {
            const uint64_t off = (uint64_t)((kk >> 2) * (BLK >> 4) + (kk & 3) * 2);
            mma_ss(T_SC + sb * 64, dq + off, dkk + off, id_s, kk > 0 ? 1u : 0u);
          }
        mma_commit(&s_full[sb]);
      }
      mma_commit(&drain_s);
      mbar_wait(&drain_s, 0);
    }
  } else if (warp == 3) {
    // ---- decay factors ---------------------------------------------------------
    double x0 = 0.0, x1 = 0.0;
    auto la_load = [&](int ci) {
      const int64_t t0 = s_begin + (int64_t)chunk_of(ci) * C;
      const int len = (int)imin64(C, s_end - t0);
      const int64_t l0 = (b * p.L + t0) * p.H + h;
      x0 = (2 * lane < len) ? (double)LDC(la, l0 + (int64_t)(2 * lane) * p.H, n_la) : 0.0;
      x1 = (2 * lane + 1 < len) ? (double)LDC(la, l0 + (int64_t)(2 * lane + 1) * p.H, n_la) : 0.0;
    };
    la_load(0);
    float alpha = 1.f;
    for (int ci = 0; ci < nc; ++ci) {
      const int slot = ci & 3;
      const int64_t t0 = s_begin + (int64_t)chunk_of(ci) * C;
      const int len = (int)imin64(C, s_end - t0);
      const double cx0 = x0, cx1 = x1;
      if (ci + 1 < nc) la_load(ci + 1);
      if (ci >= 4 && !mbar_wait_all(&fac_empty[slot], ((ci >> 2) - 1) & 1, ab)) break;
      Fac &F = fac[slot];
      const double tot = warp_cumsum64_regs(cx0, cx1, len, 0.0, F.cs2);
      __syncwarp();
      const float tot2 = (float)(tot * LOG2E_D);
      const float a_c = ex2f(tot2), an = alpha * a_c;
      const bool lazy = a_c >= 0x1p-30f && an >= 0x1p-40f && an <= 0x1p40f;
      const float kscale = lazy ? 1.f / an : 1.f;
      for (int t = lane; t < C; t += 32) {
        const bool in = t < len;
        const float x = in ? F.cs2[t] * LOG2E : 0.f;
        const float e = in ? ex2f(x) : 0.f;             // exp(cs_t)
        const float wgt = in ? ex2f(tot2 - x) : 0.f;    // exp(A_c - cs_t)
        F.cs2[t] = x;
        F.qf[t] = (REV ? wgt : e) * alpha;
        F.kw[t] = (REV ? e : wgt) * kscale;
      }
      if (lane == 0) {
        F.an = an;
        F.rescale = lazy ? 0 : 1;
      }
      alpha = lazy ? an : 1.f;
      __syncwarp();
      mbar_arrive(&fac_full[slot]);
    }
  } else if (warp < 8) {
    // ---- mask: P and w k' ------------------------------------------------------
    // The loops below run 8 columns per step: the roles' hot loops together
    // must fit the instruction cache, so nothing long is unrolled.
    const int wt = tid - 128, wq = warp & 3;
    const uint32_t lb = (uint32_t)(32 * wq) << 16;
    for (int ci = 0; ci < nc; ++ci) {
      const int slot = ci & 3, sb = ci & 1, st = ci & 1;
      const int64_t t0 = s_begin + (int64_t)chunk_of(ci) * C;
      const int len = (int)imin64(C, s_end - t0);
      if (!mbar_wait_all(&fac_full[slot], (ci >> 2) & 1, ab)) break;
      // The chunk's factors, two per lane (tokens lane and lane + 32), handed
      // around with shuffles: thread reads of shared memory are slow while
      // the tensor cores stream their operands from it.
      const Fac &F = fac[slot];
      const float csA = F.cs2[lane], csB = F.cs2[lane + 32];
      const float kwA = F.kw[lane], kwB = F.kw[lane + 32];
      // Round the chunk's v' tile to TF32 in place while its score MMAs run:
      // the tensor core truncates what it reads, and v' feeds the state
      // update of every chunk, whose bias would accumulate along the walk
      // (Y and the update read v' only after p_full, below)
      if (!mbar_wait_all(&full[st], (ci >> 1) & 1, ab)) break;
      {
        float4 *V4 = reinterpret_cast<float4 *>(Vs(st));
        const int n4 = ncbv * (int)BLK / 16;  // a multiple of 4 * 128
#pragma unroll 1
        for (int e0 = wt; e0 < n4; e0 += 4 * 128) {
          float4 x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) x[u] = LDC(V4, e0 + u * 128, n4);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            x[u].x = tf32r(x[u].x); x[u].y = tf32r(x[u].y); x[u].z = tf32r(x[u].z); x[u].w = tf32r(x[u].w);
            STC(V4, e0 + u * 128, n4, x[u]);
          }
        }
      }
      if (!mbar_wait_all(&s_full[sb], (ci >> 1) & 1, ab)) break;
      if (ci >= 1 && !mbar_wait_all(&p_empty, (ci - 1) & 1, ab)) break;
      tc_fence_after();
      // score row r = 16 wq + lane % 16 sits in lane lane % 16 (M = 64); the
      // lane 16 above it takes the row's upper 32 columns
      const int r = 16 * wq + (lane & 15), up = lane >> 4, ub = 32 * up;
      const float cr = __shfl_sync(0xffffffffu, wq < 2 ? csA : csB, r & 31);
#pragma unroll 1
      for (int g = 0; g < 2; ++g) {  // 16 of this lane's 32 columns per step
        float lo[16], hi[16];
        tmem_ld16x2(T_SC + sb * 64 + 16 * g + lb, T_SC + sb * 64 + 32 + 16 * g + lb, lo, hi);
        if (g == 1) {
          tc_fence_before();
          mbar_arrive(&s_empty[sb]);
        }
        float f[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float hv = __shfl_sync(0xffffffffu, hi[i], lane & 15);
          const float s_ = up ? hv : lo[i];
          const float a = __shfl_sync(0xffffffffu, csA, 16 * g + i), bb = __shfl_sync(0xffffffffu, csB, 16 * g + i);
          const float cu = up ? bb : a;
          const int u = ub + 16 * g + i;
          const bool valid = r < len && u < len && (REV ? u >= r : u <= r);
          f[i] = valid ? tf32r(ex2f(REV ? cu - cr : cr - cu) * s_) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          STC(reinterpret_cast<float4 *>(P), sw128_off(r, ub + 16 * g + i, C) / 16, 2 * BLK / 16,
              make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]));
      }
      fence_async_smem();
      mbar_arrive(&p_full);
      // k' (K-major, 128-byte swizzle) -> w k' (MN-major, 32-byte atoms), in
      // place: both layouts keep row s in the same 128 bytes of its block, so
      // each row is permuted within itself (8 threads per row, one 16-byte
      // chunk each; a warp holds 4 whole rows)
      // (one column block per iteration: its four 16-row passes load first)
      float4 *K4 = reinterpret_cast<float4 *>(Ks(st));
      const int n_k4 = (int)(qkbytes / 16);
      const int ch = wt & 7;
      float wr4[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        wr4[q4] = __shfl_sync(0xffffffffu, q4 < 2 ? kwA : kwB, (q4 * 16 + (wt >> 3)) & 31);
#pragma unroll 1
      for (int blk = 0; blk < ncbk; ++blk) {
        float4 v[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int row = q4 * 16 + (wt >> 3);
          v[q4] = LDC(K4, (blk * BLK + row * 128 + ((ch ^ (row & 7)) << 4)) / 16, n_k4);
        }
        __syncwarp();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int row = q4 * 16 + (wt >> 3);
          const float wr = wr4[q4];
          float4 x = v[q4];
          x.x = tf32r(x.x * wr); x.y = tf32r(x.y * wr); x.z = tf32r(x.z * wr); x.w = tf32r(x.w * wr);
          STC(K4, (blk * BLK + row * 128 + ((((ch >> 1) ^ (row & 3)) << 5) | ((ch & 1) << 4))) / 16, n_k4, x);
        }
      }
      fence_async_smem();
      mbar_arrive(&wk_full[st]);
      mbar_arrive(&fac_empty[slot]);
    }
  } else {
    // ---- epilogue --------------------------------------------------------------
    // group eg (one with NEG = 1) takes steps g_lo .. g_hi - 1 (16 tokens
    // each) of every chunk; group 0 also loads the entering state and does
    // the occasional rescale
    const int et = (tid - 256) & 127, eg = (tid - 256) >> 7, wq = warp & 3;
    const int g_lo = eg * (4 / NEG), g_hi = g_lo + 4 / NEG;
    const int j = 32 * wq + lane;  // v' feature of this lane
    const uint32_t lb = (uint32_t)(32 * wq) << 16;
    if (eg == 0) {  // entering state into tensor memory: lane j, column i = state[i][j]
      const int64_t sz = (int64_t)dk * dv, h0 = (bh * p.nseg + seg) * sz, n_h = p.B * p.H * p.nseg * sz;
      for (int c0 = 0; c0 < p.dkp; c0 += 32) {
        float hv[32];
        if (!SPLIT && hseg_t) {  // lane j reads its row as float4s (h0, j dk, c0 multiples of 4; dk of 8)
          const float4 *H4 = reinterpret_cast<const float4 *>(Hseg);
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const int i = c0 + 4 * i4;
            const float4 x = (j < dv && i < dk) ? LDC(H4, (h0 + (int64_t)j * dk + i) / 4, n_h / 4)
                                                : make_float4(0.f, 0.f, 0.f, 0.f);
            hv[4 * i4] = x.x;
            hv[4 * i4 + 1] = x.y;
            hv[4 * i4 + 2] = x.z;
            hv[4 * i4 + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int ii = 0; ii < 32; ++ii) {
            const int i = c0 + ii;
            hv[ii] = (j < dv && i < dk) ? LDC(Hseg, h0 + (hseg_t ? (int64_t)j * dk + i : (int64_t)i * dv + j), n_h) : 0.f;
          }
        }
        tmem_st32(T_ST + lb + c0, hv);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&st_init);
    }
    const int oslot = oa.out_slots == p.H ? (int)h : (int)(h / p.hpg);
    const int64_t ld = (int64_t)oa.out_slots * dv;
    const int64_t ldy = (int64_t)(p.H / p.hpg) * dv;
    const int64_t n_out = p.B * p.L * ld, n_y = p.B * p.L * ldy;
    // SPLIT: the y values of 16-token step (chunk cy, step g), loaded two steps
    // before they are used (yr0: this step, yr1: the next; the ring runs
    // across chunks), so the loads' latency hides behind the steps between.
    // A lane pair (features fb, fb + 1) loads float2s: the even lane tokens
    // 0-7 of the step, the odd lane tokens 8-15 (dst[2i], dst[2i + 1] = the
    // two features of token i of its half); the step swaps the halves' other
    // feature between the pair, so each load instruction brings two rows.
    float yr0[SPLIT ? 16 : 1], yr1[SPLIT ? 16 : 1];
    auto load_y = [&](float (&dst)[SPLIT ? 16 : 1], int cy, int g) {
      if constexpr (SPLIT) {
        const int64_t ty = s_begin + (int64_t)chunk_of(cy < nc ? cy : 0) * C;
        const int leny = cy < nc ? (int)imin64(C, s_end - ty) : 0;
        const int odd = lane & 1, fb = j - odd;  // (dv is even: a pair is inside or past dv)
        const int64_t y0 = ((b * p.L + ty) * (p.H / p.hpg) + h / p.hpg) * (int64_t)dv + fb;
        const float2 *y2 = reinterpret_cast<const float2 *>(oa.y);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = 16 * g + 8 * odd + i;
          const float2 v2 = (fb < dv && t < leny) ? LDC(y2, (y0 + (int64_t)t * ldy) / 2, n_y / 2)
                                                  : make_float2(0.f, 0.f);
          dst[2 * i] = v2.x;
          dst[2 * i + 1] = v2.y;
        }
      }
    };
    load_y(yr0, 0, g_lo);
    load_y(yr1, 0, g_lo + 1);
    const int stall_at = g_test_stall ? (nc > 1 ? 1 : 0) : -1;
    for (int ci = 0; ci < nc; ++ci) {
      const int slot = ci & 3, xb = ci & 1;
      const int64_t t0 = s_begin + (int64_t)chunk_of(ci) * C;
      const int len = (int)imin64(C, s_end - t0);
      if constexpr (SPLIT) {
        // the four epilogue warps meet at named barrier 2 for the token sums
        // below, so they take the give-up decision together (a barrier that
        // ORs the threads' failures), never one warp alone; this barrier also
        // keeps red from being rewritten before the last chunk's sums are read
        bool ok = mbar_wait(&fac_full[slot], (ci >> 2) & 1, ab);
        if (ok && ci == stall_at) ok = mbar_wait(&never, 0, ab);
        if (ok) ok = mbar_wait(&xy_full[xb], (ci >> 1) & 1, ab);
        if (named_sync_or(2 + eg, 128, !ok)) break;
        __syncwarp();
      } else {
        if (!mbar_wait_all(&fac_full[slot], (ci >> 2) & 1, ab)) break;
        if (ci == stall_at) {
          if (!mbar_wait_all(&never, 0, ab)) break;
        }
        if (!mbar_wait_all(&xy_full[xb], (ci >> 1) & 1, ab)) break;
      }
      tc_fence_after();
      const Fac &F = fac[slot];
      if (F.rescale && eg == 0) {  // Hs <- alpha exp(A_c) Hs before the update is issued
        const float an = F.an;
        for (int c0 = 0; c0 < p.dkp; c0 += 32) {
          float hv[32];
          tmem_ld32(T_ST + lb + c0, hv);
#pragma unroll
          for (int ii = 0; ii < 32; ++ii) hv[ii] *= an;
          tmem_st32(T_ST + lb + c0, hv);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&rescaled);
      }
      const float qfA = F.qf[lane], qfB = F.qf[lane + 32];  // shuffled below (see the mask)
      const int64_t o0 = ((b * p.L + t0) * oa.out_slots + oslot) * (int64_t)dv + j;
      auto step = [&](const int g) {  // tokens 16 g .. 16 g + 15
        float xa[16], ya[16];
        tmem_ld16x2(T_X + xb * 64 + 16 * g + lb, T_Y + xb * 64 + 16 * g + lb, xa, ya);
        if (g == g_hi - 1) {
          tc_fence_before();
          mbar_arrive(&x_empty[xb]);
        }
        // all sixteen values first: a shuffle cannot move past a branch, so
        // interleaving them with the (conditional) stores would serialise the
        // shuffle latencies
        const float qsrc = g < 2 ? qfA : qfB;
        float yv[SPLIT ? 16 : 1];  // this lane's feature of the step's 16 tokens
        if constexpr (SPLIT) {
          const bool odd = (lane & 1) != 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float keep = odd ? yr0[2 * i + 1] : yr0[2 * i];
            const float got = __shfl_xor_sync(0xffffffffu, odd ? yr0[2 * i] : yr0[2 * i + 1], 1);
            yv[i] = odd ? got : keep;
            yv[8 + i] = odd ? keep : got;
          }
        }
        float o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float xi = __shfl_sync(0xffffffffu, qsrc, (16 * g + i) & 31) * xa[i];
          o[i] = xi + ya[i];
          if constexpr (SPLIT) xa[i] = xi * yv[i];
        }
        if constexpr (SPLIT) {  // shift the ring and load two steps ahead
#pragma unroll
          for (int i = 0; i < 16; ++i) yr0[i] = yr1[i];
          // (two steps ahead in this group's sequence of steps)
          if (NEG == 2) load_y(yr1, ci + 1, g);
          else load_y(yr1, g + 2 < 4 ? ci : ci + 1, (g + 2) & 3);
        }
        if (j < dv) {
          const int64_t o16 = o0 + (int64_t)(16 * g) * ld;
          if (16 * g + 16 <= len) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (ATOMIC) ADDC(oa.out, o16 + i * ld, n_out, o[i]);
              else STC(oa.out, o16 + i * ld, n_out, o[i]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (16 * g + i < len) {
                if (ATOMIC) ADDC(oa.out, o16 + i * ld, n_out, o[i]);
                else STC(oa.out, o16 + i * ld, n_out, o[i]);
              }
          }
        }
        if constexpr (SPLIT) {
          // sum the 16 products over the warp's 32 lanes: four halving
          // exchanges leave each lane one value (index (lane >> 1) & 15)
          // summed over 16 lanes, one butterfly finishes the sum
#pragma unroll
          for (int off = 16, n = 16; off >= 2; off >>= 1, n >>= 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int k2 = 0; k2 < n / 2; ++k2) {
              const float mine = upper ? xa[n / 2 + k2] : xa[k2];
              const float send = upper ? xa[k2] : xa[n / 2 + k2];
              xa[k2] = mine + __shfl_xor_sync(0xffffffffu, send, off);
            }
          }
          xa[0] += __shfl_xor_sync(0xffffffffu, xa[0], 1);
          if ((lane & 1) == 0) red[wq * C + 16 * g + (lane >> 1)] = xa[0];
        }
      };
#pragma unroll 1
      for (int g = g_lo; g < g_hi; ++g) step(g);
      if constexpr (SPLIT) {
        named_sync(2 + eg, 128);
        // this group's tokens: 16 g_lo .. 16 g_hi - 1
        const int tk = 16 * g_lo + et;
        if (et < 16 * (g_hi - g_lo) && tk < len)
          STC(oa.dcs, (b * p.L + t0 + tk) * p.H + h, n_la, red[tk] + red[C + tk] + red[2 * C + tk] + red[3 * C + tk]);
      }
      mbar_arrive(&fac_empty[slot]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
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
//
// Persistent: each CTA holds DI_WG independent workers of 128 threads (one
// warpgroup each: its own tiles, barriers, named barrier and 128 tensor-memory
// columns), and worker w of CTA c takes the (chunk, group, batch) items
// w + DI_WG c, w + DI_WG (c + grid), ...  Beside the backward's walks the grid
// is the SMs the walks leave idle, and a CTA fills its SM (shared memory),
// so that no walk or contraction CTA lands beside it; otherwise the grid
// covers the GPU.
constexpr int DI_WG = 3;
__global__ void __launch_bounds__(DI_WG * NTH, 1) k_dla_intra(const __grid_constant__ CUtensorMap tmQ,
                                                             const __grid_constant__ CUtensorMap tmK,
                                                             const __grid_constant__ CUtensorMap tmV,
                                                             const __grid_constant__ CUtensorMap tmD,
                                                             const float *__restrict__ la,
                                                             float *__restrict__ Bt, PassGeo p, int64_t N,
                                                             int64_t G, uint32_t wbytes) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int dk = p.dk, dv = p.dv;  // here dk = q/k features, dv = v/dout features
  const int ncbk = p.dkp / 32, ncbv = p.dvp / 32, ncbm = ncbk > ncbv ? ncbk : ncbv;
  __shared__ uint64_t bars[2 * DI_WG];
  __shared__ uint32_t tmem_base;
  const int wg = threadIdx.x / NTH;  // this worker
  const int tid = threadIdx.x % NTH, warp = tid >> 5, lane = tid & 31;
  const int bid = 1 + wg;            // its named barrier
  uint8_t *smem = smem_align1024(smem_raw) + (size_t)wg * wbytes;
  uint8_t *T1 = smem, *T2 = smem + ncbm * 8192;
  float *R = (float *)(T2 + ncbm * 8192);  // [4][64] column partials, [64] row sums
  float *cs = R + 5 * C;                  // [64]
  uint64_t *bar_tma = &bars[2 * wg], *bar_mma = &bars[2 * wg + 1];
  const int hpg = p.hpg;
  const int64_t n_items = N * G * p.B;

  if (threadIdx.x < 32) tmem_alloc(&tmem_base, 512);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * DI_WG; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmD);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base + (uint32_t)(128 * wg);
  const uint32_t lb = (uint32_t)(warp * 32) << 16;  // (warp w of a warpgroup reaches lanes 32w..)
  // thread 0's view of what is in flight: whether a tile load, and an MMA
  // group, have been issued and not yet seen to complete (and the parity of
  // the phase each completes); both are drained before the tensor memory is
  // freed, also after a failure.  kt / km count the phases of the two
  // barriers waited for so far.
  bool tma_out = false, mma_out = false;
  uint32_t kt = 0, km = 0, tma_par = 0, mma_par = 0;
  bool ok = true;
  // Score rows live in lanes 0-15 of each warp (M = 64); the lane 16 above a
  // row works on its upper 32 columns, so every lane holds 32 columns:
  // u = 32 * up + i.
  const int up = lane >> 4;
  for (int64_t item = wg + (int64_t)DI_WG * blockIdx.x; ok && item < n_items;
       item += (int64_t)DI_WG * gridDim.x) {
    const int64_t c = item % N, grp = (item / N) % G, b = item / (N * G);
    const int64_t t0 = c * C;
    const int len = (int)imin64(C, p.L - t0);
    const int row = (int)(b * p.L + t0);
    if (tid == 0) {  // q -> T1, k -> T2
      mbar_expect_tx(bar_tma, (uint32_t)(2 * ncbk) * 8192);
      load_tile(T1, &tmQ, bar_tma, ncbk, (int)grp, row, p.wide_k);
      load_tile(T2, &tmK, bar_tma, ncbk, (int)grp, row, p.wide_k);
      tma_out = true;
      tma_par = kt & 1;
    }
    float sq[32];  // q k^T, this lane's half row
    // phase 0: q k^T; phase 1 + hh: dout v^T of head hh
    for (int ph = 0; ph <= hpg; ++ph) {
      const int ncb = ph == 0 ? ncbk : ncbv;
      const int kdim = ph == 0 ? dk : dv;
      const int64_t h = grp * hpg + (ph == 0 ? 0 : ph - 1);
      if (ph >= 1 && warp == 0) {  // in-chunk prefix of la, times log2(e)
        warp_cumsum64(la, p.B * p.L * p.H, (b * p.L + t0) * p.H + h, p.H, len, 0.0, cs);
        __syncwarp();
        for (int t = lane; t < C; t += 32) cs[t] = t < len ? cs[t] * 1.4426950408889634f : 0.f;
      }
      ok = mbar_wait(bar_tma, kt & 1) && ok;
      if (tid == 0 && ok) tma_out = false;
      ++kt;
      if (named_sync_or(bid, NTH, !ok)) {
        ok = false;
        break;
      }
      {  // round both tiles to TF32 (nearest) in place
        const int r = tid & 63, half = tid >> 6;
        const int cols = ncb * 16;
        float4 *a4 = reinterpret_cast<float4 *>(T1), *b4 = reinterpret_cast<float4 *>(T2);
        const int n4 = ncbm * 8192 / 16;
        for (int col = half * cols; col < (half + 1) * cols; col += 4) {
          const int i4 = sw128_off(r, col, C) / 16;
          float4 x = LDC(a4, i4, n4), y = LDC(b4, i4, n4);
          x.x = tf32r(x.x); x.y = tf32r(x.y); x.z = tf32r(x.z); x.w = tf32r(x.w);
          y.x = tf32r(y.x); y.y = tf32r(y.y); y.z = tf32r(y.z); y.w = tf32r(y.w);
          STC(a4, i4, n4, x);
          STC(b4, i4, n4, y);
        }
      }
      fence_async_smem();
      tc_fence_before();
      named_sync(bid, NTH);
      tc_fence_after();
      if (tid == 0) {  // phase 0 -> cols [0,64); later phases -> [64,128)
        const uint32_t a = smem_u32(T1), bb = smem_u32(T2);
        const uint32_t id = idesc_tf32(64, 64);
        for (int kk = 0; kk < kdim / 8; ++kk) {
          const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
          mma_ss(tmem + (ph == 0 ? 0 : 64), sdesc(a + off), sdesc(bb + off), id, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_mma);
        mma_out = true;
        mma_par = km & 1;
      }
      ok = mbar_wait(bar_mma, km & 1) && ok;
      if (tid == 0 && ok) mma_out = false;
      ++km;
      tc_fence_after();
      if (tid == 0 && ok && ph < hpg) {  // the tiles are consumed: next head's loads
        const int64_t hn = grp * hpg + ph;
        mbar_expect_tx(bar_tma, (uint32_t)(2 * ncbv) * 8192);
        load_tile(T1, &tmD, bar_tma, ncbv, (int)hn, row, p.wide_v);  // dout -> T1, v -> T2
        load_tile(T2, &tmV, bar_tma, ncbv, (int)hn, row, p.wide_v);
        tma_out = true;
        tma_par = kt & 1;
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
      named_sync(bid, NTH);
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
        const int64_t bt = (b * p.L + t0) * p.H + h, n_bt = p.B * p.L * p.H;
        if (2 * lane < len) STC(Bt, bt + (int64_t)(2 * lane) * p.H, n_bt, b0);
        if (2 * lane + 1 < len) STC(Bt, bt + (int64_t)(2 * lane + 1) * p.H, n_bt, b1);
      }
      named_sync(bid, NTH);  // R and cs are reused by the next head
    }
    // the MMA waits above may have given up on some threads only: the
    // worker leaves (or goes on) as a whole
    if (named_sync_or(bid, NTH, !ok)) ok = false;
  }
  if (tid == 0) {
    if (mma_out) mbar_wait(bar_mma, mma_par);
    if (tma_out) mbar_wait(bar_tma, tma_par);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tmem_base, 512);
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
// The carry comes from k_dla_carry.  The segment is taken in tiles of
// DT * DTPT tokens from its end; thread tid owns DTPT consecutive tokens of a
// tile, and all of a tile's loads are issued together, so a tile costs one
// memory round trip.  The suffix sums run in double-float arithmetic (an
// unevaluated pair hi + lo of fp32 values, added by Knuth's two-sum): about
// fp64's accuracy on the fp32 pipes, since this part's fp64 rate is low.
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_two_sum(float a, float b) {  // a + b exactly, as hi + lo
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const FF t = ff_two_sum(a.hi, b.hi);
  const float lo = __fadd_rn(t.lo, __fadd_rn(a.lo, b.lo));
  return ff_two_sum(t.hi, lo);
}
__device__ __forceinline__ FF ff_neg(FF a) { return {-a.hi, -a.lo}; }
constexpr int DT = 256;
constexpr int DTPT = 8;
// The segment carries <G_end, S_end> (defined above), one per (segment, head,
// batch) into carry[(b H + h) nseg + seg]: float4 loads eight pairs per thread
// at a time, fp32 partial sums, fp64 across threads.  They need only the two
// passes' scanned states, so the backward computes them on a side stream
// beside the walks.  grid (nseg, H, B).
__global__ void __launch_bounds__(DT) k_dla_carry(const float *__restrict__ Gst, const float *__restrict__ Sst,
                                                  const float *__restrict__ Gfin, const float *__restrict__ Sfin,
                                                  double *__restrict__ carry, int64_t H, int64_t sz, int nseg) {
  __shared__ double wred[DT / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t bh = b * H + h;
  float part = 0.f;
  const float4 *G = nullptr, *S = nullptr;
  int64_t g0 = 0, s0 = 0;        // float4 offsets of G and S
  [[maybe_unused]] int64_t n4 = 0;  // float4 count of their buffers (index checks)
  if (seg + 1 < nseg) {
    G = reinterpret_cast<const float4 *>(Gst);
    S = reinterpret_cast<const float4 *>(Sst);
    g0 = (bh * nseg + seg) * sz / 4;
    s0 = (bh * nseg + seg + 1) * sz / 4;
    n4 = (int64_t)gridDim.z * H * nseg * sz / 4;
  } else if (Gfin) {
    G = reinterpret_cast<const float4 *>(Gfin);
    S = reinterpret_cast<const float4 *>(Sfin);
    g0 = s0 = bh * sz / 4;
    n4 = (int64_t)gridDim.z * H * sz / 4;
  }
  if (G) {
    constexpr int U = 8;  // float4 pairs in flight per thread
    for (int64_t e0 = tid; e0 < sz / 4; e0 += (int64_t)U * DT) {
      float4 g[U], x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t e = e0 + (int64_t)u * DT;
        g[u] = e < sz / 4 ? LDC(G, g0 + e, n4) : make_float4(0.f, 0.f, 0.f, 0.f);
        x[u] = e < sz / 4 ? LDC(S, s0 + e, n4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        part = fmaf(g[u].x, x[u].x, fmaf(g[u].y, x[u].y, fmaf(g[u].z, x[u].z, fmaf(g[u].w, x[u].w, part))));
    }
  }
  double dp = part;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) dp += __shfl_xor_sync(0xffffffffu, dp, o);
  if (lane == 0) wred[warp] = dp;
  __syncthreads();
  if (tid == 0) {
    double c = 0.0;
#pragma unroll
    for (int w2 = 0; w2 < DT / 32; ++w2) c += wred[w2];
    STC(carry, bh * nseg + seg, (int64_t)gridDim.z * H * nseg, c);
  }
}

__global__ void __launch_bounds__(DT) k_dla(const float *__restrict__ Bt,
                                            const float *__restrict__ rq,
                                            const float *__restrict__ rk,
                                            const double *__restrict__ carry_in, float *__restrict__ dla,
                                            int64_t L, int64_t H, int Ls, int nseg) {
  constexpr int TILE = DT * DTPT;
  __shared__ FF wred[DT / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t bh = b * H + h;
  const int64_t n_tok = (int64_t)gridDim.z * L * H;  // element counts (debug-build index checks)
  const int64_t s_begin = seg * (int64_t)Ls;
  const int64_t s_end = imin64(L, s_begin + Ls);
  float xq[DTPT], xk[DTPT], xb[DTPT];
  auto load_tile = [&](int64_t hi) {  // tokens hi - TILE + tid DTPT + u (those >= s_begin)
    const int64_t t0 = hi - TILE + (int64_t)tid * DTPT;
#pragma unroll
    for (int u = 0; u < DTPT; ++u) {
      const bool ok = t0 + u >= s_begin;
      const int64_t idx = (b * L + t0 + u) * H + h;
      xq[u] = ok ? LDC(rq, idx, n_tok) : 0.f;
      xk[u] = ok ? LDC(rk, idx, n_tok) : 0.f;
      xb[u] = ok ? LDC(Bt, idx, n_tok) : 0.f;
    }
  };
  load_tile(s_end);
  FF carry;
  {
    const double c = LDC(carry_in, bh * nseg + seg, (int64_t)gridDim.z * H * nseg);
    carry.hi = (float)c;
    carry.lo = (float)(c - (double)carry.hi);
  }
  for (int64_t hi = s_end; hi > s_begin; hi -= TILE) {
    if (hi != s_end) load_tile(hi);
    FF suf[DTPT], tot = {0.f, 0.f};  // suffix sums over this thread's tokens
#pragma unroll
    for (int u = DTPT - 1; u >= 0; --u) {
      tot = ff_add(tot, ff_two_sum(xq[u], -xk[u]));
      suf[u] = tot;
    }
    FF x = tot;  // inclusive suffix of the thread totals within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const FF y = {__shfl_down_sync(0xffffffffu, x.hi, o), __shfl_down_sync(0xffffffffu, x.lo, o)};
      if (lane + o < 32) x = ff_add(x, y);
    }
    if (lane == 0) wred[warp] = x;  // warp total
    __syncthreads();
    FF after = ff_add(carry, ff_add(x, ff_neg(tot)));  // everything right of this thread's tokens
#pragma unroll
    for (int w2 = 0; w2 < DT / 32; ++w2)
      if (w2 > warp) after = ff_add(after, wred[w2]);
    const int64_t t0 = hi - TILE + (int64_t)tid * DTPT;
#pragma unroll
    for (int u = 0; u < DTPT; ++u)
      if (t0 + u >= s_begin) {
        const FF r = ff_add(ff_add(suf[u], after), FF{xb[u], 0.f});
        STC(dla, (b * L + t0 + u) * H + h, n_tok, __fadd_rn(r.hi, r.lo));
      }
#pragma unroll
    for (int w2 = 0; w2 < DT / 32; ++w2) carry = ff_add(carry, wred[w2]);
    __syncthreads();
  }
}

// ===========================================================================
// Deterministic group sums: out[r, :] = sum over hh = 0 .. hpg - 1, in that
// order, of in[r hpg + hh, :] for every (batch, token, group) row r of
// d4 float4s (in: [B, L, H, dk], out: [B, L, G, dk], H = G hpg).
__global__ void __launch_bounds__(NTH) k_group_sum(const float *__restrict__ in, float *__restrict__ out,
                                                   int64_t rows, int hpg, int d4) {
  const float4 *i4 = reinterpret_cast<const float4 *>(in);
  float4 *o4 = reinterpret_cast<float4 *>(out);
  const int64_t n = rows * d4, n_in = n * hpg;
  for (int64_t e = (int64_t)blockIdx.x * NTH + threadIdx.x; e < n; e += (int64_t)gridDim.x * NTH) {
    const int64_t r = e / d4, c = e - r * d4;
    float4 acc = LDC(i4, (r * hpg) * d4 + c, n_in);
    for (int hh = 1; hh < hpg; ++hh) {
      const float4 x = LDC(i4, (r * hpg + hh) * d4 + c, n_in);
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    STC(o4, e, n, acc);
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
// 1 slot x box_rows rows, zero fill out of bounds.  K-major operands use the
// plain 128-byte swizzle, MN-major ones the 128-byte swizzle with 32-byte
// atoms (sdesc / sdesc_mn).
// A tensor [rows][slots][d] (fp32, row-major) as 64-row tiles of 32-feature
// blocks.  Narrow: dims (d, slots, rows), box (32, 1, box_rows), one load per
// block.  Wide (d a multiple of 32): dims (32, rows, d / 32, slots) with the
// block as its own dimension (stride 128 B), box (32, box_rows, d / 32, 1):
// one load brings every block, each landing where its own narrow box would.
cudaError_t make_map(CUtensorMap *m, const float *base, int64_t rows, int64_t slots, int64_t d,
                     int box_rows, bool mn_major, bool wide) {
  const CUtensorMapSwizzle sw = mn_major ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r;
  if (wide) {
    if (d % 32) return cudaErrorInvalidValue;
    cuuint64_t dims[4] = {32, (cuuint64_t)rows, (cuuint64_t)(d / 32), (cuuint64_t)slots};
    cuuint64_t strides[3] = {(cuuint64_t)(slots * d * 4), 128, (cuuint64_t)(d * 4)};
    cuuint32_t box[4] = {32, (cuuint32_t)box_rows, (cuuint32_t)(d / 32), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(base), dims, strides, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)slots, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)(d * 4), (cuuint64_t)(slots * d * 4)};
    cuuint32_t box[3] = {32, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
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

// Segment length: the walk runs one CTA per SM, so as many segments per
// sequence as keep every (batch, head, segment) walk in one wave.
void choose_segments(const Geo &g, int *Ls, int *nseg) {
  const int64_t bh = g.B * g.H;
  const int64_t want = std::max<int64_t>(1, (int64_t)num_sms() / bh);
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
  p.wide_k = dk % 32 == 0;
  p.wide_v = dv % 32 == 0;
  return p;
}

size_t state_floats(const PassGeo &p) {
  return (size_t)(p.B * p.H * p.nseg) * (size_t)p.dk * p.dv;
}

size_t seg_state_smem(const PassGeo &p) {
  return (size_t)SS_STAGES * ((size_t)(p.dkp / 32) * SL * 128 + 4 * SL * 128) + 2 * 2 * SL * 128 + 1024;
}
// At least 120 KB, so that a walk CTA (which takes all 512 tensor-memory
// columns) never shares its SM with a second one.
size_t walk_smem(const PassGeo &p) {
  const size_t stage = (size_t)(p.dkp / 32) * 2 * C * 128 + 4 * C * 128;
  const size_t need = 2 * stage + 2 * C * 128 + 4 * sizeof(Fac) + 4 * C * 4 + 1024;
  return std::max<size_t>(need, 120 * 1024);
}

// Shared memory of one k_dla_intra worker (two tiles, the partial sums and
// the prefix of la; a multiple of 1024 B for the 128-byte swizzle), and of a
// CTA: at least 112 KB, so that no walk (at least 120 KB) or contraction CTA
// ever shares an SM with it (they need all of an SM's tensor memory).
uint32_t dla_intra_worker_bytes(const PassGeo &p) {
  const int ncbm = std::max(p.dkp, p.dvp) / 32;
  return (uint32_t)rup(ncbm * 2 * 8192 + 6 * C * 4, 1024);
}
size_t dla_intra_smem(const PassGeo &p) {
  return std::max<size_t>((size_t)DI_WG * dla_intra_worker_bytes(p) + 1024, 112 * 1024);
}

// Launch helper (grid, block, dynamic shared memory, stream, kernel arguments).
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
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
  if ((e = make_map(&mk, kp, rows, p.qk_per_head ? p.H : G, p.dk, SL, true, p.wide_k)) != cudaSuccess) return e;
  if ((e = make_map(&mv, vp, rows, p.v_per_head ? p.H : G, p.dv, SL, true, p.wide_v)) != cudaSuccess) return e;
  const dim3 grid((unsigned)p.nseg, (unsigned)p.H, (unsigned)p.B);
  {
    const size_t sm = seg_state_smem(p);
    if ((e = set_smem(k_seg_state<REV>, sm)) != cudaSuccess) return e;
    LaunchTrace lt(name_state, s);
    if ((e = launch(k_seg_state<REV>, grid, dim3(SS_THREADS), sm, s, mk, mv, la, states, Aseg, p)) != cudaSuccess)
      return e;
  }
  {
    LaunchTrace lt("tc.seg_scan", s);
    const dim3 sg((unsigned)(p.B * p.H), (unsigned)cdiv((int64_t)p.dk * p.dv, 4 * NTH));
    const int R = (4 * NTH) % p.dv == 0 ? 4 * NTH / p.dv : 0;
    const int tfast = (R > 0 && R % 4 == 0 && p.dk % R == 0) ? 1 : 0;
    e = trans ? launch(k_seg_scan<REV, true>, sg, dim3(NTH), 0, s, states, Aseg, h0, fin, statesT, p, tfast)
              : launch(k_seg_scan<REV, false>, sg, dim3(NTH), 0, s, states, Aseg, h0, fin, statesT, p, tfast);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

template <bool REV, bool ATOMIC, bool SPLIT>
cudaError_t launch_walk(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                        const PassGeo &p, const float *la, const float *states, bool states_t,
                        const WalkOut &oa, cudaStream_t s) {
  cudaError_t e;
  const size_t sm = walk_smem(p);
  if ((e = set_smem(k_walk<REV, ATOMIC, SPLIT>, sm)) != cudaSuccess) return e;
  const dim3 grid((unsigned)p.nseg, (unsigned)p.H, (unsigned)p.B);
  return launch(k_walk<REV, ATOMIC, SPLIT>, grid, dim3(walk_threads(SPLIT)), sm, s, mq, mk, mv, la, states,
                states_t ? 1 : 0, oa, p);
}

// The walk of one pass over every segment, from the entering states.
//   q', k' : [B*L, qk_slots, dk]   v' : [B*L, v_slots, dv]
// atomic: out' is summed over the heads of a group; oa.dcs given: the per-token
// inter-term dots are written too.
template <bool REV>
cudaError_t run_walk(const PassGeo &p, const float *qp, const float *kp, const float *vp,
                     const float *la, const float *states, bool states_t, const WalkOut &oa,
                     bool atomic, cudaStream_t s, const char *name_walk) {
  cudaError_t e;
  const int64_t rows = p.B * p.L;
  const int64_t G = p.H / p.hpg;
  CUtensorMap mq, mk, mv;
  if ((e = make_map(&mq, qp, rows, p.qk_per_head ? p.H : G, p.dk, C, false, p.wide_k)) != cudaSuccess) return e;
  if ((e = make_map(&mk, kp, rows, p.qk_per_head ? p.H : G, p.dk, C, false, p.wide_k)) != cudaSuccess) return e;
  if ((e = make_map(&mv, vp, rows, p.v_per_head ? p.H : G, p.dv, C, true, p.wide_v)) != cudaSuccess) return e;
  LaunchTrace lt(name_walk, s);
  const bool split = oa.dcs != nullptr;
  if (atomic) {
    e = split ? launch_walk<REV, true, true>(mq, mk, mv, p, la, states, states_t, oa, s)
              : launch_walk<REV, true, false>(mq, mk, mv, p, la, states, states_t, oa, s);
  } else {
    e = split ? launch_walk<REV, false, true>(mq, mk, mv, p, la, states, states_t, oa, s)
              : launch_walk<REV, false, false>(mq, mk, mv, p, la, states, states_t, oa, s);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// A second stream of the library's own per device, on which the backward runs
// its anti-causal passes (dk, dv) while the caller's stream runs the causal one
// (dq) and the intra-chunk dlog_alpha sums: each kernel fills one wave, and the
// other pass's kernels take the SM slots its tail leaves and overlap its short
// scans.  Fork and join are events; the lock makes the enqueue of one backward
// atomic with respect to others on other host threads (the events are reused).
struct Side {
  cudaStream_t s2 = nullptr, s3 = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, join3 = nullptr;
  cudaEvent_t scanA = nullptr, scanB = nullptr, walkA = nullptr, walkB = nullptr;  // a pass's scan / dot walk done
};
std::mutex g_side_mu;
Side g_side[64];
std::atomic<bool> g_overlap{true};
std::atomic<bool> g_det{false};

cudaError_t get_side(Side **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  Side &sd = g_side[dev];
  if (!sd.s2) {
    if ((e = cudaStreamCreateWithFlags(&sd.s2, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&sd.s3, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&sd.join3, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&sd.scanA, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&sd.scanB, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&sd.walkA, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&sd.walkB, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &sd;
  return cudaSuccess;
}

}  // namespace

bool set_overlap(bool on) { return g_overlap.exchange(on); }
bool get_overlap() { return g_overlap.load(); }
bool set_deterministic(bool on) { return g_det.exchange(on); }
bool get_deterministic() { return g_det.load(); }

int check_shape(int64_t dk, int64_t dv, int64_t chunk) {
  if (chunk != C) return SSD_ERR_CHUNK;
  if (dk % 8 || dv % 8 || dk > 128 || dv > 128) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

// The dq pass's states (its layout: [dv x dk] per head and segment) are the
// forward's own states transposed; the forward can leave them for the backward.
size_t saved_floats(const Geo &g) { return state_floats(make_pass(g, (int)g.dv, (int)g.dk, true, false)); }

size_t fwd_workspace_bytes(const Geo &g) {
  const PassGeo p = make_pass(g, (int)g.dk, (int)g.dv, false, true);
  return sizeof(float) * (state_floats(p) + (size_t)(g.B * g.H * p.nseg));
}

// Two passes' states (both kept for dlog_alpha), their decays, three
// per-token arrays, and the final state (used only when it has a cotangent).
size_t bwd_workspace_bytes(const Geo &g, bool det) {
  const PassGeo p = make_pass(g, (int)g.dk, (int)g.dv, false, true);
  const size_t nst = state_floats(p), na = (size_t)(g.B * g.H * p.nseg);
  // deterministic group sums: per-head dq_h and dk_h, [B, L, H, dk] each
  const size_t per_head = (det && g.hpg > 1) ? 2 * (size_t)(g.B * g.L * g.H * g.dk) + 4 : 0;
  // + the segment carries (fp64), 16-byte aligned after the rest
  return sizeof(float) * (2 * nst + 2 * na + 3 * (size_t)(g.B * g.L * g.H) +
                          (size_t)(g.B * g.H * g.dk * g.dv) + per_head) + 256 + sizeof(double) * na + 16;
}

cudaError_t fwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                float *out, float *hT, float *saved, const Geo &g, void *ws, cudaStream_t s) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  if (g.B * g.L >= (int64_t)1 << 31) return cudaErrorNotSupported;
  const PassGeo p = make_pass(g, (int)g.dk, (int)g.dv, false, true);
  float *st = static_cast<float *>(ws);
  float *Aseg = st + state_floats(p);
  // (saved: the scan also writes every segment's entering state transposed,
  // the dq pass's states)
  if ((e = run_states<false>(p, k, v, la, h0, false, hT, st, Aseg, saved, s, "tc.seg_state")) != cudaSuccess)
    return e;
  WalkOut oa{out, (int)g.H, nullptr, nullptr};
  return run_walk<false>(p, q, k, v, la, st, false, oa, false, s, "tc.walk_out");
}

cudaError_t bwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                const float *dout, const float *dhT, float *dq, float *dk, float *dv, float *dla,
                float *dh0, const float *saved, const float *hT_saved, const Geo &g, bool det, void *ws,
                cudaStream_t s) {
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
  // A group's per-head dq / dk: summed by atomic adds into dq / dk, or (det)
  // written per head into the workspace and summed in head order afterwards
  const bool atomic = grouped && !det;
  float *dqh = nullptr, *dkh = nullptr;
  if (grouped && det) {  // after hT's slot, 16-byte aligned for the float4 sums
    const uintptr_t a = reinterpret_cast<uintptr_t>(Bt + g.B * g.L * g.H + g.B * g.H * g.dk * g.dv);
    dqh = reinterpret_cast<float *>((a + 15) & ~uintptr_t(15));
    dkh = dqh + g.B * g.L * g.H * g.dk;
  }
  // the segment carries of dlog_alpha, fp64, after everything above
  double *carry = nullptr;
  {
    const float *end = dkh ? dkh + g.B * g.L * g.H * g.dk : Bt + g.B * g.L * g.H + g.B * g.H * g.dk * g.dv + 4;
    carry = reinterpret_cast<double *>((reinterpret_cast<uintptr_t>(end) + 15) & ~uintptr_t(15));
  }
  // pass A's states and final state: recomputed below into the workspace, or
  // the forward's (saved; then hT_saved is the final state whenever dhT is
  // given)
  const float *stA_r = saved ? saved : stA;
  const float *hT_r = saved ? hT_saved : hT;
  const int oslots = atomic ? (int)g.G : (int)g.H;
  // The dk / dv passes (pass B's states, both anti-causal walks) run on one
  // side stream (s2) and the intra-chunk dlog_alpha sums (inputs only) on
  // another (s3), both forked from s and joined back into s before this
  // returns (or all on s when overlap is off); the rest of dlog_alpha follows
  // on s3 (below).  The walks take one CTA per SM and leave the rest of the
  // SMs to the other streams' kernels.
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
    if ((e = cudaStreamWaitEvent(sd->s3, sd->fork, 0)) != cudaSuccess) return e;
  }
  cudaStream_t s2 = overlap ? sd->s2 : s, s3 = overlap ? sd->s3 : s;
  // intra-chunk block sums of dlog_alpha, on s3
  cudaError_t ei = cudaSuccess;
  {
    const PassGeo pi = make_pass(g, DK, DV, false, true);
    CUtensorMap mq, mk, mv, md;
    const int64_t rows = g.B * g.L;
    if (ei == cudaSuccess) ei = make_map(&mq, q, rows, g.G, DK, C, false, pi.wide_k);
    if (ei == cudaSuccess) ei = make_map(&mk, k, rows, g.G, DK, C, false, pi.wide_k);
    if (ei == cudaSuccess) ei = make_map(&mv, v, rows, g.H, DV, C, false, pi.wide_v);
    if (ei == cudaSuccess) ei = make_map(&md, dout, rows, g.H, DV, C, false, pi.wide_v);
    const size_t sm = dla_intra_smem(pi);
    // Beside the walks (overlap on), the kernel takes the SMs that the walks
    // (one CTA per SM) leave idle, if its work fits in the time of the
    // backward's three walks there: about one (chunk, head) phase per worker
    // per walk chunk.  Otherwise it takes the whole GPU.
    const int64_t sms = num_sms(), items = g.N * g.G * g.B;
    const int64_t spare = sms - g.B * g.H * pa.nseg;
    const int64_t per_worker = cdiv(items * (g.hpg + 1), std::max<int64_t>(1, spare) * DI_WG);
    const int64_t grid = (overlap && spare >= 8 && per_worker <= 3 * cdiv(pa.Ls, C))
                             ? spare
                             : std::min<int64_t>(sms, cdiv(items, DI_WG));
    if (ei == cudaSuccess) ei = set_smem(k_dla_intra, sm);
    if (ei == cudaSuccess) {
      LaunchTrace lt("tc.dla_intra", s3);
      ei = launch(k_dla_intra, dim3((unsigned)grid), dim3(DI_WG * NTH), sm, s3, mq, mk, mv, md, la, Bt, pi,
                  (int64_t)g.N, (int64_t)g.G, dla_intra_worker_bytes(pi));
    }
  }
  // s3 is joined through join3, recorded after its last kernel: the
  // dlog_alpha sums once both dot walks are done, or right away if the call
  // stops early (whatever is enqueued on s3 is joined back before this returns)
  bool rec3 = false;
  cudaError_t ej3 = cudaSuccess;
  auto record3 = [&]() {
    if (overlap && !rec3) {
      ej3 = cudaEventRecord(sd->join3, s3);
      rec3 = true;
    }
  };
  // (where dlog_alpha's segment carries run: see below)
  const bool carry_on_s2 = overlap && saved;
  // (dq / dk are zeroed for the atomic group sums on the stream of the pass
  // that adds into them, after the fork, so that the two fills overlap)
  cudaError_t eb = atomic ? cudaMemsetAsync(dk, 0, sizeof(float) * g.B * g.L * g.G * g.dk, s2) : cudaSuccess;
  if (eb == cudaSuccess)
    eb = run_states<true>(pb, dout, q, la, dhT, true, dh0, stB, aB, nullptr, s2, "tc.seg_state_dk");
  if (eb == cudaSuccess && overlap) eb = cudaEventRecord(sd->scanB, s2);
  WalkOut okk{dkh ? dkh : dk, oslots, k, rk};
  if (eb == cudaSuccess) eb = run_walk<true>(pb, v, dout, q, la, stB, false, okk, atomic, s2, "tc.walk_dk");
  if (eb == cudaSuccess && overlap && !carry_on_s2) eb = cudaEventRecord(sd->walkB, s2);
  WalkOut ov{dv, (int)g.H, nullptr, nullptr};
  if (eb == cudaSuccess) eb = run_walk<true>(pc, k, q, dout, la, stB, true, ov, false, s2, "tc.walk_dv");
  // dlog_alpha's segment carries <G_end, S_end> (pass B's states against pass
  // A's).  With overlap on and the forward's states given, k_dla_intra on s3
  // outlasts the 128-SM chain, so they run here, at the end of the chain
  // (pass A's states exist from the start); otherwise on s3 beside the walks,
  // or on s in turn (below).
  if (eb == cudaSuccess && carry_on_s2) {
    LaunchTrace lt("tc.dla_carry", s2);
    eb = launch(k_dla_carry, dim3((unsigned)pa.nseg, (unsigned)g.H, (unsigned)g.B), dim3(DT), 0, s2, stB, stA_r,
                dhT, hT_r, carry, g.H, (int64_t)(DK * DV), pa.nseg);
  }
  if (eb == cudaSuccess && carry_on_s2) eb = cudaEventRecord(sd->walkB, s2);
  // whatever was enqueued on s2 is joined back into s before this returns,
  // even after an error (the caller frees the workspace on s)
  cudaError_t ej = overlap ? cudaEventRecord(sd->join, s2) : cudaSuccess;
  auto join = [&]() -> cudaError_t {
    if (!overlap) return cudaSuccess;
    record3();
    if (ej != cudaSuccess) return ej;
    if (ej3 != cudaSuccess) return ej3;
    cudaError_t e1 = cudaStreamWaitEvent(s, sd->join, 0);
    cudaError_t e2 = cudaStreamWaitEvent(s, sd->join3, 0);
    return e1 != cudaSuccess ? e1 : e2;
  };
  if (eb != cudaSuccess || ei != cudaSuccess) {
    join();
    return eb != cudaSuccess ? eb : ei;
  }
  // pass A on s, meanwhile
  auto on_s = [&]() -> cudaError_t {
    cudaError_t ea = atomic ? cudaMemsetAsync(dq, 0, sizeof(float) * g.B * g.L * g.G * g.dk, s) : cudaSuccess;
    if (ea == cudaSuccess && !saved)
      ea = run_states<false>(pa, v, k, la, h0, true, hT, stA, aA, nullptr, s, "tc.seg_state_dq");
    if (ea == cudaSuccess && overlap) ea = cudaEventRecord(sd->scanA, s);
    if (ea != cudaSuccess) return ea;
    WalkOut oq{dqh ? dqh : dq, oslots, q, rq};
    return run_walk<false>(pa, dout, v, k, la, stA_r, false, oq, atomic, s, "tc.walk_dq");
  };
  cudaError_t ea = on_s();
  // dlog_alpha: the segment carries once both scans are done (on s3 beside
  // the walks, or on s in turn, unless they ran on s2 above), then the
  // in-segment suffix sums once both dot walks have written rq / rk, on s3
  // after k_dla_intra (beside the dv walk, on the SMs it leaves).
  if (ea == cudaSuccess && !carry_on_s2) {
    if (overlap) {
      ea = cudaStreamWaitEvent(s3, sd->scanA, 0);
      if (ea == cudaSuccess) ea = cudaStreamWaitEvent(s3, sd->scanB, 0);
    }
    if (ea == cudaSuccess) {
      LaunchTrace lt("tc.dla_carry", s3);
      ea = launch(k_dla_carry, dim3((unsigned)pa.nseg, (unsigned)g.H, (unsigned)g.B), dim3(DT), 0, s3, stB, stA_r,
                  dhT, hT_r, carry, g.H, (int64_t)(DK * DV), pa.nseg);
    }
  }
  if (ea == cudaSuccess) {
    if (overlap) ea = cudaEventRecord(sd->walkA, s);  // the dq walk done
    if (ea == cudaSuccess && overlap) {
      ea = cudaStreamWaitEvent(s3, sd->walkA, 0);
      if (ea == cudaSuccess) ea = cudaStreamWaitEvent(s3, sd->walkB, 0);
    }
    if (ea == cudaSuccess) {
      LaunchTrace lt("tc.dla", s3);
      ea = launch(k_dla, dim3((unsigned)pa.nseg, (unsigned)g.H, (unsigned)g.B), dim3(DT), 0, s3, Bt, rq, rk,
                  (const double *)carry, dla, g.L, g.H, pa.Ls, pa.nseg);
    }
  }
  if ((e = join()) != cudaSuccess) return e;
  if (ea != cudaSuccess) return ea;
  if (dqh) {  // the group sums, heads in order
    const int64_t n4 = g.B * g.L * g.G * g.dk / 4;
    const dim3 grid((unsigned)std::min<int64_t>(cdiv(n4, NTH), 65535 * 8));
    for (int i = 0; i < 2; ++i) {
      LaunchTrace lt("tc.group_sum", s);
      if ((e = launch(k_group_sum, grid, dim3(NTH), 0, s, i == 0 ? dqh : dkh, i == 0 ? dq : dk, g.B * g.L * g.G,
                      (int)g.hpg, (int)(g.dk / 4))) != cudaSuccess)
        return e;
    }
  }
  return cudaGetLastError();
}

cudaError_t read_and_clear_error(unsigned int *word) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if ((e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned int))) != cudaSuccess) return e;
#ifdef SSD_CHECK
  unsigned int cw = 0;
  if ((e = cudaMemcpyFromSymbol(&cw, g_check_word, sizeof(unsigned int))) != cudaSuccess) return e;
  *word |= cw;
  if ((e = cudaMemcpyToSymbol(g_check_word, &zero, sizeof(unsigned int))) != cudaSuccess) return e;
#endif
  return cudaSuccess;
}

cudaError_t set_test_stall(int on) {
  const int v = on ? 1 : 0;
  return cudaMemcpyToSymbol(g_test_stall, &v, sizeof(int));
}

}  // namespace tc
}  // namespace ssd
