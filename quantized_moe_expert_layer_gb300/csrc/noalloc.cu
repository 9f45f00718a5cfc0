// Router logits + top-k for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at run time: a serving runtime that
// plans all of the GPU's memory at start-up and hands it out only from its own
// pool (a stray allocation can fail when HBM is full, or goes around the
// pool's accounting), or a plug-in running inside such a runtime.  For them
// this entry point needs nothing but its inputs and outputs: the one piece of
// scratch memory the router uses -- the partial dot products of its K-split,
// which the top-k step adds up -- lives in a fixed file-scope device array
// that is part of the library image.  Every GPU that loads the library holds
// that array (4 MiB) until the process exits.
//
// In host code the array's name is only a host-side stand-in, never a device
// address; the device address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernels.
#include <mutex>

#include "../../include/moe.h"
#include "kernels.cuh"

namespace moe {
int record_error(int code, const char* fmt, ...);
}

namespace {

constexpr size_t kScratchFloats = size_t(1) << 20;  // 4 MiB of fp32 partial sums
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_route_scratch[kScratchFloats];

std::mutex g_mu;
float* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device; the first call
// on a device looks it up (and sets the router kernels' shared-memory limit).
int scratch_for_current_device(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return moe::record_error(MOE_ECUDA, "moe_route_noalloc: cudaGetDevice: %s", cudaGetErrorName(e));
  if (dev < 0 || dev >= kMaxDevices)
    return moe::record_error(MOE_EINVAL, "moe_route_noalloc: device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || !p)
      return moe::record_error(MOE_ECUDA, "moe_route_noalloc: cudaGetSymbolAddress: %s",
                               cudaGetErrorName(e));
    e = moe::route_kernels_init();
    if (e != cudaSuccess)
      return moe::record_error(MOE_ECUDA, "moe_route_noalloc: kernel set-up: %s", cudaGetErrorName(e));
    g_scratch[dev] = static_cast<float*>(p);
  }
  *out = g_scratch[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_route_noalloc(const uint16_t* x, int T, int H, const uint16_t* wr,
                                 const float* bias, int E, int k, float* logits, int32_t* idx,
                                 float* gates, void* stream) {
  if (!x || !wr || !logits || !idx || !gates)
    return moe::record_error(MOE_EINVAL, "moe_route_noalloc: null argument");
  if (T < 1 || H < 64 || H % 64 || H > 65536 || E < 1 || E > moe::kMaxE || k < 1 || k > E ||
      k > moe::kMaxK)
    return moe::record_error(MOE_EINVAL, "moe_route_noalloc: bad sizes T=%d H=%d E=%d k=%d", T, H,
                             E, k);
  // the router grid has ceil(T / 8) token groups in its y dimension
  if ((T + moe::kTokTile - 1) / moe::kTokTile > 65535)
    return moe::record_error(MOE_EINVAL, "moe_route_noalloc: T=%d above %d", T, 65535 * moe::kTokTile);
  if (((uintptr_t)x | (uintptr_t)wr) & 15u)
    return moe::record_error(MOE_EINVAL, "moe_route_noalloc: x and wr must be 16-byte aligned");
  const int ksplit = moe::router_ksplit(T, H, E);
  const size_t need = (size_t)ksplit * T * E;
  if (need > kScratchFloats)
    return moe::record_error(MOE_EINVAL,
                             "moe_route_noalloc: T=%d, E=%d needs %zu floats of scratch; the static "
                             "array holds %zu (T * E <= %zu always fits)",
                             T, E, need, kScratchFloats, kScratchFloats / moe::kMaxKsplitHost);
  float* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  moe::RouteParams p{};
  p.x = x;
  p.wr = wr;
  p.bias = bias;
  p.T = T;
  p.H = H;
  p.E = E;
  p.k = k;
  p.ksplit = ksplit;
  // Every partial sum the top-k step reads is written first by the router
  // kernel of the same call, so nothing in the array has to start at zero.
  p.partial = scratch;
  p.logits = logits;
  p.idx = idx;
  p.gates = gates;
  cudaStream_t st = (cudaStream_t)stream;
  // Launched without programmatic dependent launch: x, wr and bias are the
  // caller's and may be written by the kernel just before this call, so the
  // router reads nothing before that kernel has finished.
  cudaError_t e = moe::launch_router(p, st, false);
  if (e == cudaSuccess) e = moe::launch_topk(p, false, st);
  if (e != cudaSuccess)
    return moe::record_error(MOE_ECUDA, "moe_route_noalloc: kernel launch: %s", cudaGetErrorName(e));
  return MOE_OK;
}
