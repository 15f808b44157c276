/*
 * ssd.h -- C ABI of the GB300 (sm_103a) chunked SSD scan library, libssd.so.
 *
 * The operation is the gated linear-attention ("SSD") scan benchmarked by the
 * "kernel_ssd_gpu.json" and "kernel_ssd_cpu.json" benchmark pages
 * (https://www.mackelab.org/probjax/benchmarks/, their `results` tables, impl
 * "chunked", modes "fwd" and "fwd_bwd").  Those pages give only shapes, byte
 * counts and timings; the recurrence below is the one this library fixes:
 *
 *   per batch b, head h, group g = h / (H / G)   (heads split evenly and
 *   contiguously over the groups)
 *     S_{-1} = h0[b,h]                                        dk x dv
 *     S_t    = exp(log_alpha[b,t,h]) * S_{t-1} + k[b,t,g] v[b,t,h]^T
 *     out[b,t,h,:] = S_t^T q[b,t,g]        (inclusive state, q unscaled)
 *
 * ssd_bwd returns the gradients of the scalar <dout, out> with respect to
 * q, k, v, log_alpha and h0 (the pages' fwd_bwd records return gradients for
 * all five arguments: their output bytes equal the argument bytes plus a
 * scalar).  dq and dk are summed over the heads that share a group.
 *
 * Layouts: every tensor is contiguous, row-major, fp32, in device memory
 * (the pages' argument byte counts fix these shapes exactly):
 *   q, k, dq, dk        [B, L, G, dk]
 *   v, dv, out, dout    [B, L, H, dv]
 *   log_alpha, dlog_alpha [B, L, H]
 *   h0, dh0             [B, H, dk, dv]
 *
 * Conventions for every entry point:
 *   - The caller owns every buffer.  Outputs are fully overwritten (dq and dk
 *     are not accumulated into).  Inputs are never written.  Outputs must not
 *     alias inputs or each other.
 *   - h0 == NULL means a zero initial state; dh0 == NULL means "not wanted".
 *   - Every pointer must be 16-byte aligned (SSD_ERR_ALIGN otherwise).
 *   - L == 0 (or B == 0) is a valid empty problem: nothing is launched,
 *     except that ssd_bwd zero-fills dh0 when it is given.
 *   - Any L >= 1 is accepted; a last chunk shorter than `chunk` is handled.
 *   - log_alpha must be finite (a documented precondition that the device
 *     does not check; use a large negative finite value such as -1e4 for
 *     "forget everything").
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream):
 *     argument checks happen on the host before anything is enqueued; the
 *     call returns without synchronising.  Temporary device workspace is
 *     taken with cudaMallocAsync and released with cudaFreeAsync on the same
 *     stream.  Calls on different streams may run concurrently.
 *   - No function throws or aborts; each returns an ssd_status code.
 *
 * Two arithmetic paths implement the chunked evaluation (ssd_set_path), and
 * chunk == 1 selects a third, sequential one:
 *   SSD_PATH_TC   tensor-core path: tcgen05.mma (kind::tf32) with the
 *                 accumulators in tensor memory; operands rounded to TF32
 *                 (to nearest), accumulation and state passing in fp32.
 *                 Supports chunk == 64, dk and dv multiples of 8 up to 128,
 *                 B*L < 2^31.  In ssd_bwd the group sums of dq and dk are
 *                 formed with fp32 atomic adds when H > G, so their last
 *                 bits may differ from run to run.
 *   SSD_PATH_SIMT all-fp32 CUDA-core path.  Supports chunk in {16, 32, 64},
 *                 1 <= dk, dv <= 128.  Its workspace holds every chunk's
 *                 state (B*H*ceil(L/chunk)*dk*dv floats per pass), where
 *                 the tensor-core path keeps one state per segment (about
 *                 one segment per SM in all, whatever L); see
 *                 ssd_fwd_workspace_bytes.  The tensor-core backward runs
 *                 part of its work on streams of the library's own, forked
 *                 from and joined back into `stream` within the call (see
 *                 ssd_set_overlap).
 *   chunk == 1    (either path) the sequential evaluation: the recurrence one
 *                 token at a time, the state in registers, all fp32, no
 *                 workspace in the forward (suits decoding a few tokens with
 *                 h0 / hT).  1 <= dk, dv <= 128.  Its backward forms dq and
 *                 dk with fp32 atomic adds (last bits may vary run to run).
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Matches the runtime's opaque stream handle (cudaStream_t). */
typedef struct CUstream_st *ssd_stream_t;

typedef enum ssd_status {
  SSD_OK = 0,
  SSD_ERR_ARG = 1,          /* a size <= 0 where >= 1 is needed, H % G != 0,
                               a required pointer is NULL, or unknown path */
  SSD_ERR_ALIGN = 2,        /* a pointer is not 16-byte aligned */
  SSD_ERR_CHUNK = 3,        /* chunk length not supported by the active path */
  SSD_ERR_UNSUPPORTED = 4,  /* dk / dv outside what the active path supports */
  SSD_ERR_ALLOC = 5,        /* workspace allocation failed (nothing launched) */
  SSD_ERR_LAUNCH = 6,       /* a kernel launch failed */
  SSD_ERR_TIMEOUT = 7,      /* a device-side bounded wait gave up (see
                               ssd_last_device_error) */
  SSD_ERR_CUDA = 8,         /* another CUDA runtime error (no device, ...) */
  SSD_ERR_SCRATCH = 9,      /* the problem needs more scratch than
                               ssd_fwd_noalloc's fixed buffer holds */
  SSD_ERR_CHECK = 10        /* a device-side index check failed (libraries
                               built with SSD_CHECK only; see
                               ssd_last_device_error) */
} ssd_status;

typedef enum ssd_path { SSD_PATH_TC = 0, SSD_PATH_SIMT = 1 } ssd_path;

/*
 * Forward: out = the inclusive-state outputs of the recurrence above.
 *   q, k       [B,L,G,dk]   read
 *   v          [B,L,H,dv]   read
 *   log_alpha  [B,L,H]      read (finite)
 *   h0         [B,H,dk,dv]  read, or NULL for zeros
 *   out        [B,L,H,dv]   written
 *   chunk      the chunk length of the chunked evaluation (1: sequential);
 *              results do not depend on it beyond rounding.
 */
SSD_API int ssd_fwd(const float *q, const float *k, const float *v,
            const float *log_alpha, const float *h0, float *out,
            int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk,
            int64_t dv, int64_t chunk, ssd_stream_t stream);

/*
 * Backward: gradients of <dout, out>, recomputing every intermediate from the
 * inputs (nothing is saved by ssd_fwd).
 *   dout        [B,L,H,dv]   read
 *   dq, dk      [B,L,G,dk]   written (summed over the heads of each group)
 *   dv          [B,L,H,dv]   written
 *   dlog_alpha  [B,L,H]      written
 *   dh0         [B,H,dk,dv]  written, or NULL when not wanted
 * h0 may be NULL (zeros).  Other arguments as for ssd_fwd.
 */
SSD_API int ssd_bwd(const float *q, const float *k, const float *v,
            const float *log_alpha, const float *h0, const float *dout,
            float *dq, float *dk, float *dv, float *dlog_alpha, float *dh0,
            int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk_dim,
            int64_t dv_dim, int64_t chunk, ssd_stream_t stream);

/*
 * Final state and its cotangent.  A sequence can be processed in pieces:
 * running [0, L1) and then [L1, L) with the first piece's final state as h0
 * gives the outputs of one run over [0, L) (up to rounding), and the backward
 * of the pieces chains through dhT / dh0 the same way.  The benchmark pages
 * time only out (fwd) and the five argument gradients (fwd_bwd); these entry
 * points add the final state S_{L-1} of the same recurrence as an output.
 *
 * ssd_fwd_ex: as ssd_fwd, and also writes
 *   hT   [B,H,dk,dv]  the final state S_{L-1} (h0, or zeros, when L == 0),
 *                     or NULL when not wanted (then identical to ssd_fwd).
 * ssd_bwd_ex: as ssd_bwd for the scalar <dout, out> + <dhT, hT>:
 *   dhT  [B,H,dk,dv]  read, or NULL for zeros (then identical to ssd_bwd).
 *                     When L == 0, dh0 = dhT.
 * Same checks, errors, alignment, path support and stream behaviour as
 * ssd_fwd / ssd_bwd; hT must not alias any other argument.
 */
SSD_API int ssd_fwd_ex(const float *q, const float *k, const float *v,
                       const float *log_alpha, const float *h0, float *out, float *hT,
                       int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk,
                       int64_t dv, int64_t chunk, ssd_stream_t stream);
SSD_API int ssd_bwd_ex(const float *q, const float *k, const float *v,
                       const float *log_alpha, const float *h0, const float *dout,
                       const float *dhT, float *dq, float *dk, float *dv,
                       float *dlog_alpha, float *dh0, int64_t B, int64_t L, int64_t G,
                       int64_t H, int64_t dk_dim, int64_t dv_dim, int64_t chunk,
                       ssd_stream_t stream);

/*
 * Saved segment states, for a training step (forward, then backward on the
 * same inputs).  On the tensor-core path the backward's dq pass needs the
 * forward recurrence's state entering every segment of the sequence (the
 * chunked scan's passed states at segment boundaries, about one segment per
 * SM in all), which ssd_bwd / ssd_bwd_ex recompute from k, v, log_alpha and
 * h0: a contraction over the whole sequence and a scan, the same work the
 * forward did.  ssd_fwd_save keeps the forward's copy in a caller buffer and
 * ssd_bwd_saved reads it there instead.  The benchmark pages' chunked
 * records keep nothing between the forward and the backward (residual 0 MB),
 * as ssd_fwd / ssd_bwd do; this pair is an option for callers that can spare
 * the buffer.
 *
 * ssd_saved_bytes: the size of that buffer for the active path and the
 *   current device (it depends on the SM count, like the workspace):
 *   B*H*nseg*dk*dv*4 bytes on the tensor-core path (8 MiB at B=4, H=8,
 *   L=8192, dk=dv=128 on 152 SMs), 0 on the CUDA-core and sequential
 *   evaluations, whose backward always recomputes.  Same checks and return
 *   values as ssd_fwd_workspace_bytes.
 * ssd_fwd_save: as ssd_fwd_ex, and also writes
 *   saved  ssd_saved_bytes bytes, 16-byte aligned: the states entering every
 *          segment, transposed ([B, H, nseg, dv, dk]); may be NULL when
 *          ssd_saved_bytes gives 0 (then identical to ssd_fwd_ex).
 * ssd_bwd_saved: as ssd_bwd_ex, reading
 *   saved  as ssd_fwd_save wrote it for the same q, k, v, log_alpha, h0,
 *          shapes and chunk, on the same path and device, or NULL (then
 *          identical to ssd_bwd_ex); the library does not check that it
 *          matches, and a stale buffer gives wrong gradients.
 *   hT     [B,H,dk,dv] the final state that ssd_fwd_save wrote; required
 *          (SSD_ERR_ARG otherwise) when both saved and dhT are given,
 *          ignored otherwise.
 * Results equal those of ssd_bwd_ex up to rounding (the states come from the
 * forward's products instead of the backward's own).  saved is only read, and
 * must be complete in the stream order of the ssd_bwd_saved call.
 */
SSD_API int ssd_saved_bytes(int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk, int64_t dv,
                            int64_t chunk, size_t *bytes);
SSD_API int ssd_fwd_save(const float *q, const float *k, const float *v,
                         const float *log_alpha, const float *h0, float *out, float *hT,
                         float *saved, int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk,
                         int64_t dv, int64_t chunk, ssd_stream_t stream);
SSD_API int ssd_bwd_saved(const float *q, const float *k, const float *v,
                          const float *log_alpha, const float *h0, const float *dout,
                          const float *dhT, const float *hT, const float *saved, float *dq,
                          float *dk, float *dv, float *dlog_alpha, float *dh0, int64_t B,
                          int64_t L, int64_t G, int64_t H, int64_t dk_dim, int64_t dv_dim,
                          int64_t chunk, ssd_stream_t stream);

/*
 * Allocation-free forward.  The benchmark pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory at call
 * time -- code whose memory is fully reserved up front by a framework's own
 * caching allocator (so a further cudaMalloc fails), real-time loops that
 * must not allocate once running, and hooks that run inside an allocator and
 * so must not call back into it.
 *
 * Same arguments, layouts and result as ssd_fwd, always on the all-fp32
 * CUDA-core path (chunk in {16, 32, 64}, 1 <= dk, dv <= 128), whatever
 * ssd_set_path selected.  Its scratch is one fixed array of
 * ssd_fwd_noalloc_scratch_bytes() bytes (32 MiB) that the library holds in
 * the memory of every GPU on which it is loaded, until the process exits.
 * The problem must fit: B*H*ceil(L/chunk)*(dk*dv + 1)*4 bytes at most
 * (for example B*H*L <= 32768 at dk = dv = 128, chunk 64); larger problems
 * return SSD_ERR_SCRATCH before anything is enqueued.
 *   - It never calls cudaMalloc, cudaFree or any allocating routine.  Its
 *     launches are counted by ssd_launch_count but never traced: it records
 *     no events even while ssd_trace_enable(1) is in force.
 *   - Its argument checks are ssd_fwd's (the same code, in the same order),
 *     with chunk == 1 (the sequential kernels) refused as SSD_ERR_CHUNK.
 *   - The first call on a device looks up the array's device address on that
 *     device; make that first call before any stream capture.
 *   - Every call on a device shares the one array: calls that overlap on the
 *     GPU (different streams, or different host threads without ordering)
 *     race and give wrong results.  Nothing in the array needs clearing;
 *     each call writes all the scratch it reads.
 */
SSD_API int ssd_fwd_noalloc(const float *q, const float *k, const float *v,
                            const float *log_alpha, const float *h0, float *out,
                            int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk,
                            int64_t dv, int64_t chunk, ssd_stream_t stream);
SSD_API size_t ssd_fwd_noalloc_scratch_bytes(void);

/*
 * Memory.  The op keeps nothing between calls: besides the caller's tensors a
 * call needs only its temporary workspace, which these report for the active
 * path and the current device (the tensor-core path sizes its segment states
 * by the device's SM count; without a device a count of 148 is assumed).
 *   ssd_fwd_workspace_bytes  bytes ssd_fwd / ssd_fwd_ex take for this problem
 *   ssd_bwd_workspace_bytes  bytes ssd_bwd / ssd_bwd_ex take for this problem
 * Each returns the status the call itself would return from its shape checks
 * (pointers are not involved) and writes 0 for an empty problem.  `bytes`
 * must not be NULL.
 *
 * ssd_pool_high_water: the high-water mark, in bytes, of the current device's
 * default stream-ordered memory pool (the pool the workspace comes from; it
 * also counts anything else the process took from that pool with
 * cudaMallocAsync).  bytes may be NULL; reset != 0 then lowers the mark to the
 * memory in use now.  Returns SSD_ERR_CUDA without a usable device.
 */
SSD_API int ssd_fwd_workspace_bytes(int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk,
                                    int64_t dv, int64_t chunk, size_t *bytes);
SSD_API int ssd_bwd_workspace_bytes(int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk,
                                    int64_t dv, int64_t chunk, size_t *bytes);
SSD_API int ssd_pool_high_water(int reset, size_t *bytes);

/* Select the arithmetic path for later calls in this process (all threads).
 * Returns SSD_ERR_ARG for an unknown value.  The initial path is SSD_PATH_TC,
 * or the value of the environment variable SSD_PATH ("tc" / "simt") read at
 * the first call. */
SSD_API int ssd_set_path(int path);
SSD_API int ssd_get_path(void);

/* Overlap of the tensor-core backward's independent passes (process-wide,
 * all threads; on by default).  When on, ssd_bwd / ssd_bwd_ex run the dk and
 * dv passes on a stream of the library's own (one per device, created at the
 * first backward), forked from and joined back into the caller's stream
 * inside the call, so the call stays ordered on `stream` like any other; the
 * intra-chunk dlog_alpha sums run on a second stream of the library's, and
 * the causal dq pass on `stream`, meanwhile.  With overlap on, the
 * intra-chunk sums take the SMs the one-CTA-per-SM passes leave idle (when
 * their work fits in the passes' time there), so they run beside them.  Off
 * runs every kernel on `stream` in turn (the same results up to the order of
 * the float atomic adds that sum a group's heads; for profiling one kernel
 * at a time).  The SIMT and sequential paths are not affected.
 * ssd_set_overlap returns the previous setting. */
SSD_API int ssd_set_overlap(int on);
SSD_API int ssd_get_overlap(void);

/* Deterministic group sums in the tensor-core backward (process-wide, off
 * by default).  When H > G, dq and dk are sums over the heads of a group.
 * Off, every head's walk adds its share into dq / dk with fp32 atomic adds,
 * whose order (and so the last bits of the sums) may differ from run to run.
 * On, every head's share is written to the workspace and one more kernel
 * adds them in head order, so that the same inputs give bitwise the same dq
 * and dk on every run; the workspace grows by 2*B*L*H*dk floats and the step
 * by that kernel.  ssd_bwd_workspace_bytes reports the size for the current
 * setting (change it only between calls).  The SIMT path always sums heads
 * in order; the sequential kernels (chunk == 1) use atomic adds either way.
 * Returns the previous setting. */
SSD_API int ssd_set_deterministic(int on);
SSD_API int ssd_get_deterministic(void);

/* Static description of a status code; never NULL. */
SSD_API const char *ssd_strerror(int status);

/* Synchronises `stream`, then reads and clears the library's device error
 * words on the current device.  Returns SSD_ERR_TIMEOUT when a bounded
 * device-side wait gave up since the last check (the affected outputs are
 * then unspecified), SSD_ERR_CHECK when (in a library built with -DSSD_CHECK,
 * whose kernels test every global index against its buffer's size) an index
 * check failed and its access was skipped, SSD_ERR_CUDA when the
 * synchronisation itself failed, SSD_OK otherwise. */
SSD_API int ssd_last_device_error(ssd_stream_t stream);

/* Test switch for the failure path of the tensor-core kernels' bounded waits
 * (not needed for the op).  While `on` is nonzero, the epilogue of every
 * tensor-core walk CTA waits, at its second chunk, on a barrier that nothing
 * completes.  That wait gives up after its limit (about 2^31 SM cycles, about
 * a second), every role of the CTA leaves its loop, the tile loads and MMAs
 * still in flight are drained, tensor memory is freed and the kernel returns;
 * ssd_last_device_error then reports SSD_ERR_TIMEOUT and the outputs of the
 * calls made meanwhile are unspecified.  It writes a device variable of the
 * current device with a synchronous copy, so it applies to calls enqueued
 * after it returns.  Returns SSD_ERR_CUDA when that copy fails. */
SSD_API int ssd_test_stall_walks(int on);

/* Launch accounting and tracing (for profiling; not needed for the op).
 * ssd_launch_count: kernels launched by this library in this process so far.
 * ssd_trace_enable(1): from now on, bracket every launch with two CUDA events
 *   on its stream (adds a few microseconds of device time per launch).
 * ssd_trace_collect: waits for the traced launches, folds them into
 *   per-kernel totals, returns the number of distinct kernel names (or a
 *   negated ssd_status on failure).
 * ssd_trace_get(i, ...): name (NUL-terminated, truncated to name_len),
 *   launch count and total device milliseconds of kernel i.
 * ssd_trace_reset: drops all records and totals. */
SSD_API long long ssd_launch_count(void);
SSD_API int ssd_trace_enable(int on);
SSD_API int ssd_trace_collect(void);
SSD_API int ssd_trace_get(int i, char *name, int name_len, long long *launches,
                          double *total_ms);
SSD_API int ssd_trace_reset(void);

/* Library version as major*10000 + minor*100 + patch (0.2.0 added the
 * final-state entry points, 0.3.0 ssd_set_overlap / ssd_get_overlap, 0.4.0
 * ssd_set_deterministic / ssd_get_deterministic, ssd_test_stall_walks and
 * SSD_ERR_CHECK). */
SSD_API int ssd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H_ */
