// Placeholder translation unit for the int8 prefill GEMM (tcgen05 version
// follows).  Until then the entry point reports TERN_ERR_CUDA-free
// "unsupported" through an invalid-value launch error.
#include "tern_internal.cuh"

namespace tern {

__device__ unsigned int g_gemm_error;

cudaError_t launch_gemm(const uint16_t*, const float*, const uint16_t*, const float*, int64_t,
                        int64_t, int64_t, uint16_t*, int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t gemm_read_clear_error(unsigned int* err) {
  cudaError_t e = cudaMemcpyFromSymbol(err, g_gemm_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(unsigned int));
}

}  // namespace tern
