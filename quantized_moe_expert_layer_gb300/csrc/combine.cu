// Gate-weighted combine of the expert outputs: out[t] = sum_j g[t,j] * y[row(t,j)]
// + y_shared[t], j in order (a fixed fmaf chain, deterministic).  Used after
// the expert kernels that write y rows to global memory (tensor-core path,
// streaming path for more than a few tokens); the few-token path combines in
// shared memory inside its down kernel.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- combine
// out[t] = sum_j gates[t,j] * y[row(t,j)] + y_shared[t], j in order.
__global__ void __launch_bounds__(256) combine_kernel(ExpertParams p, const float* gates,
                                                      const int* inv, float* out) {
  griddep_launch();
  griddep_wait();
  const int H4 = p.H / 4, S = p.T * p.k;
  const float4* y4 = reinterpret_cast<const float4*>(p.ybuf);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)p.T * H4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H4), h = (int)(i % H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float gs[kMaxK];
    int rows[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < p.k) {
        gs[j] = gates[(size_t)t * p.k + j];
        rows[j] = inv[(size_t)t * p.k + j];
      }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < p.k) {
        const float4 yv = y4[(size_t)rows[j] * H4 + h];
        acc.x = fmaf(gs[j], yv.x, acc.x);
        acc.y = fmaf(gs[j], yv.y, acc.y);
        acc.z = fmaf(gs[j], yv.z, acc.z);
        acc.w = fmaf(gs[j], yv.w, acc.w);
      }
    if (p.shared) {
      const float4 yv = y4[(size_t)(S + t) * H4 + h];
      acc.x += yv.x; acc.y += yv.y; acc.z += yv.z; acc.w += yv.w;
    }
    reinterpret_cast<float4*>(out)[i] = acc;
  }
}

}  // namespace

cudaError_t launch_combine(const ExpertParams& p, const float* gates, const int* inv, float* out,
                           bool pdl, cudaStream_t st) {
  const int64_t n = (int64_t)p.T * (p.H / 4);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  return launch_k(combine_kernel, dim3(blocks), dim3(256), 0, st, pdl, p, gates, inv, out);
}

}  // namespace moe
