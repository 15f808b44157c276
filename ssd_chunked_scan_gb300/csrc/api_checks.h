// Argument checks, geometry and CUDA-error mapping shared by the C-ABI entry
// points (api.cu, noalloc.cu), so that every entry point takes the same
// decisions on the same arguments.
#pragma once

#include <stdint.h>

#include "../../include/ssd.h"
#include "common.cuh"
#include "tc.h"

namespace ssd {
namespace abi {

inline bool misaligned(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u); }

// Sizes every path needs: non-negative B and L, positive G, H, dk, dv and
// chunk, H a multiple of G, grid-sized B, H and G.
inline int check_common(int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk, int64_t dv,
                        int64_t chunk) {
  if (B < 0 || L < 0 || G < 1 || H < 1 || dk < 1 || dv < 1 || chunk < 1) return SSD_ERR_ARG;
  if (H % G != 0) return SSD_ERR_ARG;
  if (B > 65535 || H > 65535 || G > 65535) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

// Shape limits of the kernels that serve (path, chunk): chunk == 1 is the
// sequential evaluation on every path; otherwise the path's chunked kernels.
inline int check_path_shape(int path, int64_t B, int64_t L, int64_t dk, int64_t dv,
                            int64_t chunk) {
  if (chunk == 1) {
    if (dk > 128 || dv > 128) return SSD_ERR_UNSUPPORTED;
  } else if (path == SSD_PATH_SIMT) {
    if (chunk != 16 && chunk != 32 && chunk != 64) return SSD_ERR_CHUNK;
    if (dk > 128 || dv > 128) return SSD_ERR_UNSUPPORTED;
  } else {
    int rc = ssd::tc::check_shape(dk, dv, chunk);
    if (rc) return rc;
    if (B * L >= ((int64_t)1 << 31)) return SSD_ERR_UNSUPPORTED;  // 32-bit TMA row index
  }
  if (ssd::cdiv(L, chunk) > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

inline ssd::Geo make_geo(int64_t B, int64_t L, int64_t G, int64_t H, int64_t dk, int64_t dv,
                         int64_t chunk) {
  ssd::Geo g;
  g.B = B; g.L = L; g.G = G; g.H = H; g.dk = dk; g.dv = dv;
  g.C = (int)chunk;
  g.N = ssd::cdiv(L, chunk);
  g.hpg = (int)(H / G);
  return g;
}

inline int from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return SSD_OK;
  if (e == cudaErrorMemoryAllocation) return SSD_ERR_ALLOC;
  if (e == cudaErrorLaunchFailure || e == cudaErrorInvalidConfiguration ||
      e == cudaErrorLaunchOutOfResources || e == cudaErrorInvalidDeviceFunction ||
      e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidValue)
    return SSD_ERR_LAUNCH;
  return SSD_ERR_CUDA;
}

}  // namespace abi
}  // namespace ssd
