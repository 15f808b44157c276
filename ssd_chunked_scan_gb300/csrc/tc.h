// Host entry points of the tensor-core path (tc.cu).
#pragma once
#include "common.cuh"

namespace ssd {
namespace tc {

// 0 when the tensor-core path supports (dk, dv, chunk), else an ssd_status.
int check_shape(int64_t dk, int64_t dv, int64_t chunk);

size_t fwd_workspace_bytes(const Geo &g);
// det: the deterministic group sums (see set_deterministic); the same value
// must be given to bwd.
size_t bwd_workspace_bytes(const Geo &g, bool det);

// Floats of the states the forward can leave for the backward (see fwd).
size_t saved_floats(const Geo &g);

// hT (final state, written) and dhT (its cotangent, read) may be NULL.
// saved (saved_floats(g), may be NULL): fwd also writes there the states
// entering each segment, transposed, which are the backward's dq-pass states;
// bwd then reads them instead of recomputing them, and hT_saved is the final
// state fwd wrote (needed when dhT is given).
cudaError_t fwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                float *out, float *hT, float *saved, const Geo &g, void *ws, cudaStream_t s);
cudaError_t bwd(const float *q, const float *k, const float *v, const float *la, const float *h0,
                const float *dout, const float *dhT, float *dq, float *dk, float *dv, float *dla,
                float *dh0, const float *saved, const float *hT_saved, const Geo &g, bool det, void *ws,
                cudaStream_t s);

// Whether bwd runs its dk / dv passes on a side stream (see ssd_set_overlap);
// set_overlap returns the previous setting.
bool set_overlap(bool on);
bool get_overlap();

// Whether bwd sums a group's per-head dq / dk in a fixed order (per-head
// results in the workspace, then one summing kernel) instead of by atomic
// adds (see ssd_set_deterministic); set_deterministic returns the previous
// setting.
bool set_deterministic(bool on);
bool get_deterministic();

// Reads and clears the device error word of the current device: bit 0 is set
// by a bounded wait that gave up, bit 1 by a failed index check (debug
// builds).
cudaError_t read_and_clear_error(unsigned int *word);

// Failure-path test switch (see ssd_test_stall_walks).
cudaError_t set_test_stall(int on);

}  // namespace tc
}  // namespace ssd
