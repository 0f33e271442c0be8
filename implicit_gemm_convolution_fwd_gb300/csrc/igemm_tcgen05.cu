// Placeholder translation unit for the tensor-core implicit GEMM; the tcgen05
// kernel replaces it.
#include <cuda_runtime.h>

#include "conv_internal.cuh"

namespace convfwd {

__device__ unsigned int g_device_status = 0;

bool igemm_supported(const Geom &, const char **why) {
  *why = "tensor-core path not built";
  return false;
}

cudaError_t launch_igemm_3xtf32(const float *, const float *, const float *, float *, const Geom &,
                                cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t read_and_clear_device_status(unsigned *flags) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
  *flags = v;
  return e;
}

}  // namespace convfwd
