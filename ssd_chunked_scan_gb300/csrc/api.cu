// C ABI of libssd (declared in include/ssd.h): argument checks, workspace,
// path selection and dispatch.  No kernel arithmetic lives here.
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "../../include/ssd.h"
#include "../../include/ssd_mamba.h"
#include "common.cuh"
#include "mamba.h"
#include "seq.h"
#include "api_checks.h"
#include "simt.h"
#include "tc.h"

namespace {

using ssd::abi::check_common;
using ssd::abi::check_path_shape;
using ssd::abi::from_cuda;
using ssd::abi::make_geo;
using ssd::abi::misaligned;

std::atomic<int> g_path{-1};

int current_path() {
  int p = g_path.load(std::memory_order_relaxed);
  if (p < 0) {
    p = SSD_PATH_TC;
    const char *e = std::getenv("SSD_PATH");
    if (e && (std::strcmp(e, "simt") == 0 || std::strcmp(e, "SIMT") == 0)) p = SSD_PATH_SIMT;
    int expected = -1;
    if (!g_path.compare_exchange_strong(expected, p)) p = expected;
  }
  return p;
}

// Host-side fault injection for tests of the error path: with
// SSD_FAULT_ALLOC=1 in the environment every workspace request fails before
// anything is enqueued.
bool alloc_fault_injected() {
  const char *e = std::getenv("SSD_FAULT_ALLOC");
  return e && e[0] == '1';
}

// Which kernels serve a call: chunk == 1 is the sequential evaluation on every
// path; otherwise the selected path's chunked kernels.
enum class Impl { TC, SIMT, SEQ };
Impl impl_of(int path, int64_t chunk) {
  if (chunk == 1) return Impl::SEQ;
  return path == SSD_PATH_SIMT ? Impl::SIMT : Impl::TC;
}

// Stream-ordered workspace.  The first use on a device raises that device's
// default memory pool release threshold so freed workspace is kept for the
// next call instead of being returned to the driver at every synchronisation.
int ws_alloc(void **p, size_t bytes, cudaStream_t s) {
  *p = nullptr;
  if (bytes == 0) return SSD_OK;
  if (alloc_fault_injected()) return SSD_ERR_ALLOC;
  static std::atomic<unsigned long long> tuned{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSD_ERR_CUDA;
  if (dev < 64 && !(tuned.load() & (1ull << dev))) {
    cudaMemPool_t pool;
    if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
      uint64_t thr = ~0ull;
      cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    }
    tuned.fetch_or(1ull << dev);
  }
  cudaError_t e = cudaMallocAsync(p, bytes, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return e == cudaErrorMemoryAllocation ? SSD_ERR_ALLOC : from_cuda(e);
  }
  return SSD_OK;
}

// ssd_fwd_ex / ssd_fwd_save: saved (may be NULL) is written by the
// tensor-core path only.
int fwd_impl(const float *q, const float *k, const float *v, const float *log_alpha, const float *h0,
             float *out, float *hT, float *saved, int64_t B, int64_t L, int64_t G, int64_t H,
             int64_t dk, int64_t dv, int64_t chunk, ssd_stream_t stream) {
  int rc = check_common(B, L, G, H, dk, dv, chunk);
  if (rc) return rc;
  const int path = current_path();
  rc = check_path_shape(path, B, L, dk, dv, chunk);
  if (rc) return rc;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(log_alpha) ||
      misaligned(h0) || misaligned(out) || misaligned(hT) || misaligned(saved))
    return SSD_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (B == 0 || L == 0) {  // the final state is the initial one
    if (!hT || B == 0) return SSD_OK;
    const size_t bytes = sizeof(float) * B * H * dk * dv;
    return from_cuda(h0 ? cudaMemcpyAsync(hT, h0, bytes, cudaMemcpyDeviceToDevice, s)
                        : cudaMemsetAsync(hT, 0, bytes, s));
  }
  if (!q || !k || !v || !log_alpha || !out) return SSD_ERR_ARG;
  const ssd::Geo g = make_geo(B, L, G, H, dk, dv, chunk);
  const Impl im = impl_of(path, chunk);
  if (im == Impl::SEQ) return from_cuda(ssd::seq::fwd(q, k, v, log_alpha, h0, out, hT, g, s));
  const size_t wsb = im == Impl::SIMT ? ssd::simt::fwd_workspace_bytes(g)
                                      : ssd::tc::fwd_workspace_bytes(g);
  void *ws = nullptr;
  rc = ws_alloc(&ws, wsb, s);
  if (rc) return rc;
  cudaError_t e = im == Impl::SIMT ? ssd::simt::fwd(q, k, v, log_alpha, h0, out, hT, g, ws, s)
                                   : ssd::tc::fwd(q, k, v, log_alpha, h0, out, hT, saved, g, ws, s);
  if (ws) cudaFreeAsync(ws, s);
  return from_cuda(e);
}

// ssd_bwd_ex / ssd_bwd_saved: saved (may be NULL) is read by the tensor-core
// path only, with hT_saved the final state when dhT is given.
int bwd_impl(const float *q, const float *k, const float *v, const float *log_alpha, const float *h0,
             const float *dout, const float *dhT, const float *hT_saved, const float *saved, float *dq,
             float *dk, float *dv, float *dlog_alpha, float *dh0, int64_t B, int64_t L, int64_t G,
             int64_t H, int64_t dk_dim, int64_t dv_dim, int64_t chunk, ssd_stream_t stream) {
  int rc = check_common(B, L, G, H, dk_dim, dv_dim, chunk);
  if (rc) return rc;
  const int path = current_path();
  rc = check_path_shape(path, B, L, dk_dim, dv_dim, chunk);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(log_alpha) ||
      misaligned(h0) || misaligned(dout) || misaligned(dhT) || misaligned(dq) ||
      misaligned(dk) || misaligned(dv) || misaligned(dlog_alpha) || misaligned(dh0) ||
      misaligned(hT_saved) || misaligned(saved))
    return SSD_ERR_ALIGN;
  if (B == 0 || L == 0) {  // dh0 = dhT (or zero)
    if (!dh0 || B == 0) return SSD_OK;
    const size_t bytes = sizeof(float) * B * H * dk_dim * dv_dim;
    return from_cuda(dhT ? cudaMemcpyAsync(dh0, dhT, bytes, cudaMemcpyDeviceToDevice, s)
                         : cudaMemsetAsync(dh0, 0, bytes, s));
  }
  if (!q || !k || !v || !log_alpha || !dout || !dq || !dk || !dv || !dlog_alpha)
    return SSD_ERR_ARG;
  const ssd::Geo g = make_geo(B, L, G, H, dk_dim, dv_dim, chunk);
  const Impl im = impl_of(path, chunk);
  if (im == Impl::TC && saved && dhT && !hT_saved) return SSD_ERR_ARG;
  const bool det = ssd::tc::get_deterministic();  // read once: sizes the workspace and steers the call
  const size_t wsb = im == Impl::SEQ    ? ssd::seq::bwd_workspace_bytes(g)
                     : im == Impl::SIMT ? ssd::simt::bwd_workspace_bytes(g)
                                        : ssd::tc::bwd_workspace_bytes(g, det);
  void *ws = nullptr;
  rc = ws_alloc(&ws, wsb, s);
  if (rc) return rc;
  cudaError_t e;
  if (im == Impl::SEQ)
    e = ssd::seq::bwd(q, k, v, log_alpha, h0, dout, dhT, dq, dk, dv, dlog_alpha, dh0, g, ws, s);
  else if (im == Impl::SIMT)
    e = ssd::simt::bwd(q, k, v, log_alpha, h0, dout, dhT, dq, dk, dv, dlog_alpha, dh0, g, ws, s);
  else
    e = ssd::tc::bwd(q, k, v, log_alpha, h0, dout, dhT, dq, dk, dv, dlog_alpha, dh0, saved, hT_saved, g, det,
                     ws, s);
  if (ws) cudaFreeAsync(ws, s);
  return from_cuda(e);
}

}  // namespace

extern "C" {

int ssd_version(void) { return 400; }

const char *ssd_strerror(int status) {
  switch (status) {
    case SSD_OK: return "ok";
    case SSD_ERR_ARG: return "invalid argument (size, H % G, null pointer or unknown path)";
    case SSD_ERR_ALIGN: return "pointer not 16-byte aligned";
    case SSD_ERR_CHUNK: return "chunk length not supported by the active path";
    case SSD_ERR_UNSUPPORTED: return "shape not supported by the active path";
    case SSD_ERR_ALLOC: return "workspace allocation failed";
    case SSD_ERR_LAUNCH: return "kernel launch failed";
    case SSD_ERR_TIMEOUT: return "a device-side bounded wait timed out";
    case SSD_ERR_CUDA: return "CUDA runtime error";
    case SSD_ERR_SCRATCH: return "problem too large for the fixed scratch of ssd_fwd_noalloc";
    case SSD_ERR_CHECK: return "a device-side index check failed (debug build)";
    default: return "unknown status";
  }
}

int ssd_set_path(int path) {
  if (path != SSD_PATH_TC && path != SSD_PATH_SIMT) return SSD_ERR_ARG;
  g_path.store(path);
  return SSD_OK;
}

int ssd_get_path(void) { return current_path(); }

int ssd_set_overlap(int on) { return ssd::tc::set_overlap(on != 0) ? 1 : 0; }

int ssd_get_overlap(void) { return ssd::tc::get_overlap() ? 1 : 0; }

int ssd_set_deterministic(int on) { return ssd::tc::set_deterministic(on != 0) ? 1 : 0; }

int ssd_get_deterministic(void) { return ssd::tc::get_deterministic() ? 1 : 0; }

int ssd_fwd_ex(const float *q, const float *k, const float *v, const float *log_alpha,
               const float *h0, float *out, float *hT, int64_t B, int64_t L, int64_t G, int64_t H,
               int64_t dk, int64_t dv, int64_t chunk, ssd_stream_t stream) {
  return fwd_impl(q, k, v, log_alpha, h0, out, hT, nullptr, B, L, G, H, dk, dv, chunk, stream);
}

int ssd_fwd_save(const float *q, const float *k, const float *v, const float *log_alpha,
                 const float *h0, float *out, float *hT, float *saved, int64_t B, int64_t L, int64_t G,
                 int64_t H, int64_t dk, int64_t dv, int64_t chunk, ssd_stream_t stream) {
  return fwd_impl(q, k, v, log_alpha, h0, out, hT, saved, B, L, G, H, dk, dv, chunk, stream);
}

int ssd_fwd(const float *q, const float *k, const float *v, const float *log_alpha,
            const float *h0, float *out, int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk,
            int64_t dv, int64_t chunk, ssd_stream_t stream) {
  return ssd_fwd_ex(q, k, v, log_alpha, h0, out, nullptr, B, L, G, H, dk, dv, chunk, stream);
}

int ssd_bwd_ex(const float *q, const float *k, const float *v, const float *log_alpha,
               const float *h0, const float *dout, const float *dhT, float *dq, float *dk,
               float *dv, float *dlog_alpha, float *dh0, int64_t B, int64_t L, int64_t G,
               int64_t H, int64_t dk_dim, int64_t dv_dim, int64_t chunk, ssd_stream_t stream) {
  return bwd_impl(q, k, v, log_alpha, h0, dout, dhT, nullptr, nullptr, dq, dk, dv, dlog_alpha, dh0, B, L, G, H,
                  dk_dim, dv_dim, chunk, stream);
}

int ssd_bwd_saved(const float *q, const float *k, const float *v, const float *log_alpha,
                  const float *h0, const float *dout, const float *dhT, const float *hT,
                  const float *saved, float *dq, float *dk, float *dv, float *dlog_alpha, float *dh0,
                  int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk_dim, int64_t dv_dim,
                  int64_t chunk, ssd_stream_t stream) {
  return bwd_impl(q, k, v, log_alpha, h0, dout, dhT, hT, saved, dq, dk, dv, dlog_alpha, dh0, B, L, G, H, dk_dim,
                  dv_dim, chunk, stream);
}

int ssd_bwd(const float *q, const float *k, const float *v, const float *log_alpha,
            const float *h0, const float *dout, float *dq, float *dk, float *dv,
            float *dlog_alpha, float *dh0, int64_t B, int64_t L, int64_t G, int64_t H,
            int64_t dk_dim, int64_t dv_dim, int64_t chunk, ssd_stream_t stream) {
  return ssd_bwd_ex(q, k, v, log_alpha, h0, dout, nullptr, dq, dk, dv, dlog_alpha, dh0, B, L, G,
                    H, dk_dim, dv_dim, chunk, stream);
}

int ssd_fwd_workspace_bytes(int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk, int64_t dv,
                            int64_t chunk, size_t *bytes) {
  if (!bytes) return SSD_ERR_ARG;
  *bytes = 0;
  int rc = check_common(B, L, G, H, dk, dv, chunk);
  if (rc) return rc;
  const int path = current_path();
  rc = check_path_shape(path, B, L, dk, dv, chunk);
  if (rc) return rc;
  if (B == 0 || L == 0) return SSD_OK;
  const ssd::Geo g = make_geo(B, L, G, H, dk, dv, chunk);
  const Impl im = impl_of(path, chunk);
  *bytes = im == Impl::SEQ    ? ssd::seq::fwd_workspace_bytes(g)
           : im == Impl::SIMT ? ssd::simt::fwd_workspace_bytes(g)
                              : ssd::tc::fwd_workspace_bytes(g);
  return SSD_OK;
}

int ssd_bwd_workspace_bytes(int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk, int64_t dv,
                            int64_t chunk, size_t *bytes) {
  if (!bytes) return SSD_ERR_ARG;
  *bytes = 0;
  int rc = check_common(B, L, G, H, dk, dv, chunk);
  if (rc) return rc;
  const int path = current_path();
  rc = check_path_shape(path, B, L, dk, dv, chunk);
  if (rc) return rc;
  if (B == 0 || L == 0) return SSD_OK;
  const ssd::Geo g = make_geo(B, L, G, H, dk, dv, chunk);
  const Impl im = impl_of(path, chunk);
  *bytes = im == Impl::SEQ    ? ssd::seq::bwd_workspace_bytes(g)
           : im == Impl::SIMT ? ssd::simt::bwd_workspace_bytes(g)
                              : ssd::tc::bwd_workspace_bytes(g, ssd::tc::get_deterministic());
  return SSD_OK;
}

int ssd_saved_bytes(int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk, int64_t dv, int64_t chunk,
                    size_t *bytes) {
  if (!bytes) return SSD_ERR_ARG;
  *bytes = 0;
  int rc = check_common(B, L, G, H, dk, dv, chunk);
  if (rc) return rc;
  const int path = current_path();
  rc = check_path_shape(path, B, L, dk, dv, chunk);
  if (rc) return rc;
  if (B == 0 || L == 0 || impl_of(path, chunk) != Impl::TC) return SSD_OK;
  *bytes = sizeof(float) * ssd::tc::saved_floats(make_geo(B, L, G, H, dk, dv, chunk));
  return SSD_OK;
}

int ssd_pool_high_water(int reset, size_t *bytes) {
  if (bytes) *bytes = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SSD_ERR_CUDA; }
  cudaMemPool_t pool;
  if (cudaDeviceGetDefaultMemPool(&pool, dev) != cudaSuccess) { cudaGetLastError(); return SSD_ERR_CUDA; }
  if (bytes) {
    uint64_t v = 0;
    if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &v) != cudaSuccess) {
      cudaGetLastError();
      return SSD_ERR_CUDA;
    }
    *bytes = (size_t)v;
  }
  if (reset) {
    uint64_t zero = 0;  // resets the mark to the memory in use now
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &zero) != cudaSuccess) {
      cudaGetLastError();
      return SSD_ERR_CUDA;
    }
  }
  return SSD_OK;
}

static int mamba_check(int64_t B, int64_t L, int64_t D, int64_t N) {
  if (B < 0 || L < 0 || D < 1 || N < 1) return SSD_ERR_ARG;
  if (N > 16) return SSD_ERR_UNSUPPORTED;
  // grid limits: batch on grid z, segments (at most 1024 tokens each) on grid y
  if (B > 65535 || (D + 15) / 16 > 0x7fffffffLL || L > (int64_t)65535 * 1024)
    return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

int ssd_mamba_workspace_bytes(int bwd, int64_t B, int64_t L, int64_t D, int64_t N,
                              size_t *bytes) {
  if (!bytes) return SSD_ERR_ARG;
  *bytes = 0;
  int rc = mamba_check(B, L, D, N);
  if (rc) return rc;
  if (B == 0 || L == 0) return SSD_OK;
  *bytes = bwd ? ssd::mamba::bwd_workspace_bytes(B, L, D, N)
               : ssd::mamba::fwd_workspace_bytes(B, L, D, N);
  return SSD_OK;
}

int ssd_mamba_fwd(const float *x, const float *delta, const float *A, const float *Bm,
                  const float *Cm, const float *Dk, float *y, int64_t B, int64_t L, int64_t D,
                  int64_t N, ssd_stream_t stream) {
  int rc = mamba_check(B, L, D, N);
  if (rc) return rc;
  if (misaligned(x) || misaligned(delta) || misaligned(A) || misaligned(Bm) || misaligned(Cm) ||
      misaligned(Dk) || misaligned(y))
    return SSD_ERR_ALIGN;
  if (B == 0 || L == 0) return SSD_OK;
  if (!x || !delta || !A || !Bm || !Cm || !y) return SSD_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void *ws = nullptr;
  rc = ws_alloc(&ws, ssd::mamba::fwd_workspace_bytes(B, L, D, N), s);
  if (rc) return rc;
  cudaError_t e = ssd::mamba::fwd(x, delta, A, Bm, Cm, Dk, y, B, L, D, N, ws, s);
  if (ws) cudaFreeAsync(ws, s);
  return from_cuda(e);
}

int ssd_mamba_bwd(const float *x, const float *delta, const float *A, const float *Bm,
                  const float *Cm, const float *Dk, const float *dy, float *dx, float *ddelta,
                  float *dA, float *dB, float *dC, float *dD, int64_t B, int64_t L, int64_t D,
                  int64_t N, ssd_stream_t stream) {
  int rc = mamba_check(B, L, D, N);
  if (rc) return rc;
  if (misaligned(x) || misaligned(delta) || misaligned(A) || misaligned(Bm) || misaligned(Cm) ||
      misaligned(Dk) || misaligned(dy) || misaligned(dx) || misaligned(ddelta) ||
      misaligned(dA) || misaligned(dB) || misaligned(dC) || misaligned(dD))
    return SSD_ERR_ALIGN;
  if (!dA || (Dk && !dD)) return SSD_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (B == 0 || L == 0) {
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * D * N, s);
    if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, sizeof(float) * D, s);
    return from_cuda(e);
  }
  if (!x || !delta || !A || !Bm || !Cm || !dy || !dx || !ddelta || !dB || !dC)
    return SSD_ERR_ARG;
  void *ws = nullptr;
  rc = ws_alloc(&ws, ssd::mamba::bwd_workspace_bytes(B, L, D, N), s);
  if (rc) return rc;
  cudaError_t e = ssd::mamba::bwd(x, delta, A, Bm, Cm, Dk, dy, dx, ddelta, dA, dB, dC,
                                  Dk ? dD : nullptr, B, L, D, N, ws, s);
  if (ws) cudaFreeAsync(ws, s);
  return from_cuda(e);
}

int ssd_last_device_error(ssd_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  unsigned int word = 0, sw = 0;
  if (ssd::tc::read_and_clear_error(&word) != cudaSuccess) return SSD_ERR_CUDA;
  if (ssd::simt::read_and_clear_error(&sw) != cudaSuccess) return SSD_ERR_CUDA;
  word |= sw;
  if (word & 1u) return SSD_ERR_TIMEOUT;
  return word ? SSD_ERR_CHECK : SSD_OK;
}

int ssd_test_stall_walks(int on) {
  return ssd::tc::set_test_stall(on) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
