// Host entry points of the all-fp32 CUDA-core path (simt.cu).
#pragma once
#include "common.cuh"

namespace ssd {
namespace simt {

// Workspace bytes needed by fwd / bwd for geometry g.
size_t fwd_workspace_bytes(const Geo &g);
size_t bwd_workspace_bytes(const Geo &g);

// Enqueue the forward / backward on stream s.  hT (final state, written) and
// dhT (its cotangent, read) may be NULL.  ws must hold the bytes above
// (256-byte aligned).  Returns the first launch error.
cudaError_t fwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                float *out, float *hT, const Geo &g, void *ws, cudaStream_t s);
cudaError_t bwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                const float *dout, const float *dhT, float *dq, float *dk, float *dv, float *dla,
                float *dh0, const Geo &g, void *ws, cudaStream_t s);

// Reads and clears this path's check word (bit 1: a failed index check; only
// debug builds set it, otherwise the word reads 0).
cudaError_t read_and_clear_error(unsigned int *word);

}  // namespace simt
}  // namespace ssd
