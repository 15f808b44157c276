// Host entry points of the sequential (chunk = 1) kernels (seq.cu).
#pragma once
#include "common.cuh"

namespace ssd {
namespace seq {

// Workspace bytes needed by fwd (none) / bwd for geometry g.
size_t fwd_workspace_bytes(const Geo &g);
size_t bwd_workspace_bytes(const Geo &g);

// Enqueue on stream s; hT (written) and dhT (read) may be NULL.  1 <= dk, dv
// <= 128.  Returns the first launch error.
cudaError_t fwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                float *out, float *hT, const Geo &g, cudaStream_t s);
cudaError_t bwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                const float *dout, const float *dhT, float *dq, float *dk, float *dv, float *dla,
                float *dh0, const Geo &g, void *ws, cudaStream_t s);

}  // namespace seq
}  // namespace ssd
