// Shared definitions of the libssd kernels (host and device).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace ssd {

// ---- debug build: device-side index checks ---------------------------------
// Built with -DSSD_CHECK, the kernels' global (and staged shared-memory)
// accesses test their index against the buffer's element count first; an
// index outside [0, n) sets bit 1 of the translation unit's check word (read
// and cleared by the unit's read_and_clear_error) and the access is skipped (a
// skipped load reads zero).  Without the flag the macros are the plain access.
#ifdef SSD_CHECK
static __device__ unsigned int g_check_word;
__device__ __forceinline__ bool chk_idx(int64_t i, int64_t n) {
  const bool ok = i >= 0 && i < n;
  if (!ok) atomicOr(&g_check_word, 2u);
  return ok;
}
#define SSD_OK_IDX(i, n) ::ssd::chk_idx((int64_t)(i), (int64_t)(n))
#else
#define SSD_OK_IDX(i, n) ((void)(i), (void)(n), true)
#endif
#define LDC(a, i, n) (SSD_OK_IDX(i, n) ? (a)[i] : std::decay_t<decltype((a)[0])>{})
#define STC(a, i, n, v) \
  do {                                  \
    if (SSD_OK_IDX(i, n)) (a)[i] = (v); \
  } while (0)
#define ADDC(a, i, n, v) \
  do {                                           \
    if (SSD_OK_IDX(i, n)) atomicAdd((a) + (i), (v)); \
  } while (0)

// Geometry of one call.  Sizes that index memory are 64-bit.
struct Geo {
  int64_t B, L, G, H, dk, dv;
  int C;      // chunk length
  int64_t N;  // number of chunks, ceil(L / C)
  int hpg;    // heads per group, H / G
};

__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Element offsets of the row-major layouts.
__host__ __device__ inline int64_t qk_off(const Geo &g, int64_t b, int64_t t, int64_t grp) {
  return ((b * g.L + t) * g.G + grp) * g.dk;
}
__host__ __device__ inline int64_t v_off(const Geo &g, int64_t b, int64_t t, int64_t h) {
  return ((b * g.L + t) * g.H + h) * g.dv;
}
__host__ __device__ inline int64_t la_off(const Geo &g, int64_t b, int64_t t, int64_t h) {
  return (b * g.L + t) * g.H + h;
}
// Per-chunk state buffers [B, H, N, dk, dv].
__host__ __device__ inline int64_t st_off(const Geo &g, int64_t bh, int64_t c) {
  return (bh * g.N + c) * g.dk * g.dv;
}
// Element counts of q / k, of v / dout / out, of la / dla, of the per-chunk
// state buffers and of one state per head (h0, hT, dh0, dhT).
__host__ __device__ inline int64_t n_qk(const Geo &g) { return g.B * g.L * g.G * g.dk; }
__host__ __device__ inline int64_t n_v(const Geo &g) { return g.B * g.L * g.H * g.dv; }
__host__ __device__ inline int64_t n_la(const Geo &g) { return g.B * g.L * g.H; }
__host__ __device__ inline int64_t n_st(const Geo &g) { return g.B * g.H * g.N * g.dk * g.dv; }
__host__ __device__ inline int64_t n_h(const Geo &g) { return g.B * g.H * g.dk * g.dv; }

// Inclusive prefix sums of log_alpha over one chunk, for one (b, h), written
// to cs[0 .. len).  Accumulated in fp64 by warp 0 (lane l owns steps
// 2l, 2l+1; len <= 64) and rounded once to fp32.  All threads must call.
__device__ inline void chunk_cumsum64(const float *__restrict__ la, int64_t n_la, int64_t first,
                                      int64_t stride, int len, float *cs) {
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    double x0 = (2 * l < len) ? (double)LDC(la, first + (int64_t)(2 * l) * stride, n_la) : 0.0;
    double x1 = (2 * l + 1 < len) ? (double)LDC(la, first + (int64_t)(2 * l + 1) * stride, n_la) : 0.0;
    double pair = x0 + x1, incl = pair;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (l >= o) incl += y;
    }
    double excl = incl - pair;
    if (2 * l < len) cs[2 * l] = (float)(excl + x0);
    if (2 * l + 1 < len) cs[2 * l + 1] = (float)(excl + pair);
  }
  __syncthreads();
}

}  // namespace ssd

namespace ssd {
// Scope around one kernel launch: counts it and, when tracing is enabled,
// records CUDA events before and after it on stream s (trace.cu).
class LaunchTrace {
 public:
  LaunchTrace(const char *name, cudaStream_t s);
  ~LaunchTrace();
  LaunchTrace(const LaunchTrace &) = delete;
  LaunchTrace &operator=(const LaunchTrace &) = delete;
  // While one of these lives on a thread, launches on that thread are only
  // counted: no events are created or recorded and nothing is appended to
  // the trace (both allocate), whether or not tracing is enabled.
  class Quiet {
   public:
    Quiet();
    ~Quiet();
    Quiet(const Quiet &) = delete;
    Quiet &operator=(const Quiet &) = delete;

   private:
    bool prev_;
  };

 private:
  const char *name_;
  cudaStream_t s_;
  void *a_;
};
}  // namespace ssd
