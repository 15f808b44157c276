// Host entry points of the Mamba-1 selective-scan kernels (mamba.cu).
#pragma once
#include "common.cuh"

namespace ssd {
namespace mamba {

// Workspace bytes of fwd / bwd for (B, L, D, N); N <= 16.
size_t fwd_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N);
size_t bwd_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N);

// Enqueue on stream s; Dk (and dD) may be NULL.  Returns the first launch error.
cudaError_t fwd(const float *x, const float *dt, const float *A, const float *Bm, const float *Cm,
                const float *Dk, float *y, int64_t B, int64_t L, int64_t D, int64_t N, void *ws,
                cudaStream_t s);
cudaError_t bwd(const float *x, const float *dt, const float *A, const float *Bm, const float *Cm,
                const float *Dk, const float *dy, float *dx, float *ddt, float *dA, float *dB,
                float *dC, float *dD, int64_t B, int64_t L, int64_t D, int64_t N, void *ws,
                cudaStream_t s);

}  // namespace mamba
}  // namespace ssd
