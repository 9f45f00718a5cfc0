// The whole layer for a few tokens (T <= 8) in one cooperative launch.
//
// A decode step is a chain of three small dependent steps -- routing, gate/up
// over the selected experts, down + combine -- each of which moves only a few
// MB, so launch boundaries and per-kernel latency chains cost as much as the
// weight traffic.  Here one CTA per SM runs all of it, with two grid-wide
// barriers:
//   phase 1: router partial sums (K split over CTAs), and, on the CTAs left
//            over, the shared expert's gate/up (it needs no routing);
//   barrier;
//   phase 2: every CTA computes top-k, gates and the dispatch itself (a few
//            hundred bytes of partial sums; no further barrier needed), asks
//            L2 for the down-projection tiles it will need, and runs its share
//            of the routed gate/up tasks;
//   barrier;
//   phase 3: down projection + j-ordered combine, one 16-row tile of H per CTA.
// The arithmetic of every step is the one the stand-alone kernels use (same
// device functions, same order), so both paths give the same numbers.
// Co-residency of all CTAs is guaranteed by the cooperative launch; every
// barrier wait is bounded and records MOE_ETIMEOUT in the status word if it
// gives up.
#include "common.cuh"
#include "expert_dev.cuh"
#include "kernels.cuh"
#include "layout.cuh"
#include "route_dev.cuh"

namespace moe {
namespace {

constexpr int kDecThreads = 256;
constexpr long long kBarrierBudget = 2000000000LL;  // ~1 s of clock64

struct DecodeShared {
  int4 entries[kSmallSlots];
  int n_entries;
  int inv[kSmallSlots];
  int row_token[kSmallSlots + kTokTile];
  float gates[kSmallSlots];
  int sidx[kSmallSlots];
  uint32_t ck[8 * kMaxK];
  int ci[8 * kMaxK];
  float red[kDecThreads * 8];
  int disp[64 + kMaxE];  // dispatch scratch: scan space + per-expert counts
  int timed_out;
};

// Grid-wide barrier: the last CTA to arrive resets the count and advances the
// generation the others wait on.  Bounded: gives up after kBarrierBudget.
__device__ void grid_barrier(unsigned* count, unsigned* gen, int* status, int* timed_out) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned g = *reinterpret_cast<volatile unsigned*>(gen);
    __threadfence();
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
      atomicExch(count, 0u);
      __threadfence();
      atomicAdd(gen, 1u);
    } else {
      const long long t0 = clock64();
      while (*reinterpret_cast<volatile unsigned*>(gen) == g) {
        if (clock64() - t0 > kBarrierBudget) {
          *timed_out = 1;
          *status = -5;  // MOE_ETIMEOUT
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
  }
  __syncthreads();
}

template <int FMT>
__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(RouteParams rp, ExpertParams ep,
                                                                float* out, unsigned* bar) {
  extern __shared__ uint4 dsm[];  // router staging (phase 1), y tiles (phase 3)
  __shared__ DecodeShared sh;
  const int cta = blockIdx.x, ncta = gridDim.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int T = rp.T, S = T * rp.k;
  if (threadIdx.x == 0) sh.timed_out = 0;
  // expert params whose routing outputs live in this CTA's shared memory
  ExpertParams el = ep;
  el.entries = sh.entries;
  el.n_entries = &sh.n_entries;
  el.row_token = sh.row_token;
  const int tpc = tiles_per_cta(n_halves(mat_geom(FMT, ep.H)));
  const int n_pg = (ep.I / 16 + tpc - 1) / tpc;

  // ---------------------------------------------------------------- phase 1
  const int n_router = ((rp.E + 15) / 16) * rp.ksplit;
  const int n_shared = ep.shared ? n_pg : 0;
  for (int task = cta; task < n_router + n_shared; task += ncta) {
    if (task < n_router)
      router_partials(rp, task / rp.ksplit, 0, task % rp.ksplit, dsm);
    else
      gateup_task<FMT>(el, ep.E, S, T, task - n_router, tpc, sh.red);  // shared expert: x itself
    __syncthreads();
  }
  grid_barrier(&bar[0], &bar[1], rp.status, &sh.timed_out);

  // ---------------------------------------------------------------- phase 2
  // top-k, gates and dispatch in every CTA; CTA 0 also publishes them
  RouteParams rl = rp;
  rl.entries = sh.entries;
  rl.n_entries = &sh.n_entries;
  rl.inv = sh.inv;
  rl.row_token = sh.row_token;
  if (cta != 0) {
    rl.logits = nullptr;
    rl.idx = nullptr;
    rl.gates = nullptr;
    rl.counts = nullptr;
    rl.offsets = nullptr;
    rl.perm = nullptr;
  }
  if (T == 1) {  // one token: all 8 warps share its top-k (E/8 experts each)
    if (rp.E <= 256)
      topk_token_cta<1, 8>(rl, 0, sh.sidx, sh.ck, sh.ci, sh.gates);
    else if (rp.E <= 512)
      topk_token_cta<2, 8>(rl, 0, sh.sidx, sh.ck, sh.ci, sh.gates);
    else
      topk_token_cta<4, 8>(rl, 0, sh.sidx, sh.ck, sh.ci, sh.gates);
  } else {
    if (warp < T) topk_token(rl, warp, lane, sh.sidx, sh.gates);
    __syncthreads();
  }
  dispatch_small(rl, sh.disp, sh.sidx);
  __syncthreads();
  if (cta == 0) {  // the routing outputs the debug hooks read
    for (int i = threadIdx.x; i < sh.n_entries; i += kDecThreads) rp.entries[i] = sh.entries[i];
    for (int i = threadIdx.x; i < S; i += kDecThreads) rp.inv[i] = sh.inv[i];
    for (int i = threadIdx.x; i < S + T; i += kDecThreads) rp.row_token[i] = sh.row_token[i];
    if (threadIdx.x == 0) *rp.n_entries = sh.n_entries;
  }
  for (int tile = cta; tile < ep.H / 16; tile += ncta) down_prefetch<FMT>(el, tile);
  const int nsh = ep.shared ? 1 : 0;
  const int n_routed = sh.n_entries * n_pg;
  for (int task = cta; task < n_routed; task += ncta) {
    const int y = nsh + task / n_pg;
    int expert, row, n;
    if (get_entry(el, y, expert, row, n)) gateup_task<FMT>(el, expert, row, n, task % n_pg, tpc, sh.red);
    __syncthreads();
  }
  grid_barrier(&bar[2], &bar[3], rp.status, &sh.timed_out);

  // ---------------------------------------------------------------- phase 3
  float* ys = reinterpret_cast<float*>(dsm);
  for (int tile = cta; tile < ep.H / 16; tile += ncta) {
    DownPreload none;
    down_combine_task<FMT>(el, tile, sh.gates, sh.inv, out, ys, none, false);
    __syncthreads();
  }
}

size_t decode_smem(const RouteParams& rp, const ExpertParams& ep) {
  const int C = rp.H / 64;
  const int max_klen = ((C + rp.ksplit - 1) / rp.ksplit) * 64;
  const size_t router = (size_t)kTokTile * (max_klen + 8) * 2 + kDecThreads * 4 * sizeof(float);
  const size_t ys = ((size_t)ep.T * ep.k + (ep.shared ? ep.T : 0)) * 16 * sizeof(float);
  return router > ys ? router : ys;
}

int g_num_sms = 0;

}  // namespace

bool decode_ok(int fmt, int T, int k, int shared, int H) {
  (void)fmt;
  (void)H;
  return T <= kTokTile && T * k + (shared ? T : 0) <= kSmallSlots;
}

cudaError_t launch_decode(const RouteParams& rp, const ExpertParams& ep, float* out, unsigned* bar,
                          cudaStream_t st) {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g_num_sms);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = decode_smem(rp, ep);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (ep.fmt == FMT_NVFP4) return cudaLaunchKernelEx(&cfg, decode_kernel<FMT_NVFP4>, rp, ep, out, bar);
  return cudaLaunchKernelEx(&cfg, decode_kernel<FMT_FP6>, rp, ep, out, bar);
}

cudaError_t decode_kernels_init() {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<FMT_NVFP4>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_kernel<FMT_FP6>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           64 * 1024);
  if (e != cudaSuccess) return e;
  // one CTA per SM must fit for the cooperative launch
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<FMT_NVFP4>, kDecThreads,
                                                    64 * 1024);
  if (e == cudaSuccess && n < 1) e = cudaErrorCooperativeLaunchTooLarge;
  return e;
}

}  // namespace moe
