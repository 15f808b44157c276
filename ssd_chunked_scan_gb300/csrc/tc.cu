// Tensor-core (tcgen05) path of the chunked SSD scan.
#include "../../include/ssd.h"
#include "common.cuh"
#include "tc.h"

namespace ssd {
namespace tc {

// Device error word: bit 0 = an mbarrier wait exceeded its iteration limit.
__device__ unsigned int g_error_word;

int check_shape(int64_t dk, int64_t dv, int64_t chunk) {
  if (chunk != 64) return SSD_ERR_CHUNK;
  if (dk % 8 || dv % 8 || dk > 128 || dv > 128) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}
size_t fwd_workspace_bytes(const Geo &) { return 0; }
size_t bwd_workspace_bytes(const Geo &) { return 0; }

cudaError_t fwd(const float *, const float *, const float *, const float *, const float *,
                float *, const Geo &, void *, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t bwd(const float *, const float *, const float *, const float *, const float *,
                const float *, float *, float *, float *, float *, float *, const Geo &, void *,
                cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t read_and_clear_error(unsigned int *word) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned int));
}

}  // namespace tc
}  // namespace ssd
