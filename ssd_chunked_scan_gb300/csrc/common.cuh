// Shared definitions of the libssd kernels (host and device).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

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

// Inclusive prefix sums of log_alpha over one chunk, for one (b, h), written
// to cs[0 .. len).  Accumulated in fp64 by warp 0 (lane l owns steps
// 2l, 2l+1; len <= 64) and rounded once to fp32.  All threads must call.
__device__ inline void chunk_cumsum64(const float *__restrict__ la, int64_t first,
                                      int64_t stride, int len, float *cs) {
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    double x0 = (2 * l < len) ? (double)la[first + (int64_t)(2 * l) * stride] : 0.0;
    double x1 = (2 * l + 1 < len) ? (double)la[first + (int64_t)(2 * l + 1) * stride] : 0.0;
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

 private:
  const char *name_;
  cudaStream_t s_;
  void *a_;
};
}  // namespace ssd
