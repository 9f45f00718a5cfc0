// Device side of the seeded input generator (see moe_gen.h): fills device
// buffers with the same values the host side produces.  Holds none of the
// layer's arithmetic; used by tests and the benchmark to build full-size
// layers without a host round trip.
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gen.h"

namespace {

__global__ void fill_f32_kernel(float* out, uint64_t n, uint64_t key, float sigma,
                                uint64_t offset) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = __fmul_rn(moe_gen_normal(key, offset + i), sigma);
}

__global__ void fill_bf16_kernel(uint16_t* out, uint64_t n, uint64_t key, float sigma,
                                 uint64_t offset) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = moe_gen_bf16_rne(__fmul_rn(moe_gen_normal(key, offset + i), sigma));
}

int grid_for(uint64_t n) {
  uint64_t b = (n + 255) / 256;
  return (int)(b > 152 * 16 ? 152 * 16 : (b == 0 ? 1 : b));
}

}  // namespace

extern "C" int moe_gen_fill_f32_dev(float* out, uint64_t n, uint64_t key, float sigma,
                                    uint64_t offset, void* stream) {
  if (n == 0) return 0;
  fill_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(out, n, key, sigma, offset);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

extern "C" int moe_gen_fill_bf16_dev(uint16_t* out, uint64_t n, uint64_t key, float sigma,
                                     uint64_t offset, void* stream) {
  if (n == 0) return 0;
  fill_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(out, n, key, sigma, offset);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}
