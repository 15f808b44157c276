/*
 * ssd_mamba.h -- Mamba-1 selective scan in libssd.so (C ABI).
 *
 * The second workload of the benchmark pages: "kernel_mamba_cpu.json"
 * (https://www.mackelab.org/probjax/benchmarks/), impls "scan" / "chunked",
 * modes "fwd" and "fwd_bwd", state 16.  The pages give shapes and argument
 * byte counts only (x, delta [B,L,D]; A [D,N]; B, C [B,L,N]; D [D] fit them
 * exactly); the recurrence this library fixes is the Mamba selective scan:
 *
 *   per batch b, channel d, state n < N, h_{-1} = 0:
 *     h_t[d,n] = exp(delta[b,t,d] A[d,n]) h_{t-1}[d,n] + delta[b,t,d] B[b,t,n] x[b,t,d]
 *     y[b,t,d] = sum_n C[b,t,n] h_t[d,n] + D[d] x[b,t,d]
 *
 * delta is used as given (any softplus is the caller's).  ssd_mamba_bwd
 * returns the gradients of <dy, y> for all six arguments.
 *
 * Layouts: contiguous row-major fp32 in device memory,
 *   x, delta, y, dy, dx, ddelta  [B, L, D]
 *   A, dA                        [D, N]
 *   Bm, Cm, dB, dC               [B, L, N]
 *   Dk, dD                       [D]      (Dk NULL: no skip term; dD then
 *                                          not written and may be NULL)
 * Conventions as in ssd.h: caller-owned buffers, outputs fully overwritten,
 * no aliasing, 16-byte aligned pointers (SSD_ERR_ALIGN), asynchronous on
 * `stream` with workspace from cudaMallocAsync, status codes.  1 <= N <= 16
 * (SSD_ERR_UNSUPPORTED otherwise), D >= 1, L == 0 or B == 0 is an empty
 * problem (ssd_mamba_bwd then zero-fills dA and dD).  Arithmetic is fp32 on
 * the CUDA cores whatever ssd_set_path selected.  dA, dB, dC and dD are
 * sums formed with fp32 atomic adds, so their last bits may vary from run
 * to run.
 */
#ifndef SSD_MAMBA_H_
#define SSD_MAMBA_H_

#include "ssd.h"

#ifdef __cplusplus
extern "C" {
#endif

SSD_API int ssd_mamba_fwd(const float *x, const float *delta, const float *A, const float *Bm,
                          const float *Cm, const float *Dk, float *y, int64_t B, int64_t L,
                          int64_t D, int64_t N, ssd_stream_t stream);

SSD_API int ssd_mamba_bwd(const float *x, const float *delta, const float *A, const float *Bm,
                          const float *Cm, const float *Dk, const float *dy, float *dx,
                          float *ddelta, float *dA, float *dB, float *dC, float *dD, int64_t B,
                          int64_t L, int64_t D, int64_t N, ssd_stream_t stream);

/* Workspace bytes ssd_mamba_fwd (bwd == 0) or ssd_mamba_bwd (bwd != 0)
 * takes; same shape checks as the calls.  bytes must not be NULL. */
SSD_API int ssd_mamba_workspace_bytes(int bwd, int64_t B, int64_t L, int64_t D, int64_t N,
                                      size_t *bytes);

#ifdef __cplusplus
}
#endif

#endif /* SSD_MAMBA_H_ */
