// Allocation-free forward entry point (ssd_fwd_noalloc in include/ssd.h).
//
// For callers that cannot allocate device memory when they call us: the
// forward's scratch (per-chunk states and decays) lives in one fixed
// file-scope device array instead of a cudaMallocAsync workspace.  The
// kernels are the all-fp32 path's forward kernels, unchanged.
#include <atomic>
#include <mutex>

#include "../../include/ssd.h"
#include "api_checks.h"
#include "common.cuh"
#include "simt.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

// Held in every GPU's memory once this library's module is loaded there.
static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mu;

// Device address of g_fwd_scratch on the current device, looked up once per
// device.  In host code the array's name is only a host-side stand-in; the
// kernels must be given this address.
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_fwd_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" {

SSD_API size_t ssd_fwd_noalloc_scratch_bytes(void) { return kScratchBytes; }

SSD_API int ssd_fwd_noalloc(const float *q, const float *k, const float *v,
                            const float *log_alpha, const float *h0, float *out, int64_t B,
                            int64_t L, int64_t G, int64_t H, int64_t dk, int64_t dv,
                            int64_t chunk, ssd_stream_t stream) {
  using namespace ssd::abi;
  // the same checks, in the same order, as ssd_fwd on the all-fp32 path
  int rc = check_common(B, L, G, H, dk, dv, chunk);
  if (rc) return rc;
  if (chunk == 1) return SSD_ERR_CHUNK;  // (ssd_fwd's sequential kernels are not served here)
  rc = check_path_shape(SSD_PATH_SIMT, B, L, dk, dv, chunk);
  if (rc) return rc;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(log_alpha) ||
      misaligned(h0) || misaligned(out))
    return SSD_ERR_ALIGN;
  if (B == 0 || L == 0) return SSD_OK;
  if (!q || !k || !v || !log_alpha || !out) return SSD_ERR_ARG;
  const ssd::Geo g = make_geo(B, L, G, H, dk, dv, chunk);
  // B*H*N*(dk*dv + 1) floats, checked without overflow
  const long double need = (long double)B * H * g.N * ((long double)dk * dv + 1) * 4;
  if (need > (long double)kScratchBytes || ssd::simt::fwd_workspace_bytes(g) > kScratchBytes)
    return SSD_ERR_SCRATCH;
  void *ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) {
    cudaGetLastError();
    return SSD_ERR_CUDA;
  }
  // no trace events here, even with tracing on: recording them allocates
  ssd::LaunchTrace::Quiet quiet;
  return from_cuda(ssd::simt::fwd(q, k, v, log_alpha, h0, out, nullptr, g, ws,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
