// Expert kernels: fused dequant + gate/up GEMM + SwiGLU, dequant + down GEMM,
// and the gate-weighted combine.
//
// Work unit: an entry = (expert, first row, up to 8 tokens) from dispatch, or
// one of the leading shared-expert entries.  Each CTA takes one entry and one
// group of 16-row weight tiles; its 4 warps split the tiles and/or the K
// dimension.  Weights stream from HBM with 16-byte per-lane loads in the order
// the packed layout stores them (layout.cuh) and are dequantised in registers
// straight into m16n8k16 A fragments: NVFP4 code * e4m3 block scale is exact
// in f16; FP6 e2m3 codes are exact in f16 and the power-of-two block scale is
// applied to an fp32 per-block accumulator.  The activations (x, or the SwiGLU
// output a) are the B operand, staged once per CTA in shared memory as f16.
// The fp32 tensor scale is applied in the epilogue.  Partial sums over K are
// added in a fixed warp order, so results are deterministic and each token's
// value does not depend on which other tokens share its entry.
//
// SwiGLU: a = silu(g) * u with g = W_gate x, u = W_up x, silu(v) = v / (1 + e^-v);
// y = W_down a.  The fused gate|up and separate down split follows the expert
// kernels of "Strata on an Intel Arc" and of the nextsycl README ("the
// experts' gate | up" / "down projection").
#include "common.cuh"
#include "expert_dev.cuh"
#include "kernels.cuh"
#include "layout.cuh"
#include "route_dev.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- gate/up + SwiGLU
template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) gateup_kernel(ExpertParams p, int tpc) {
  const int y = blockIdx.y;
  // Shared-expert entries need no routing.  Routed ones wait for it, and only
  // then let the next kernel start: once every CTA here has triggered, the
  // routing outputs (work entries) are complete and the next kernel may read
  // them before its own wait.
  if (y >= p.nsh) griddep_wait();
  griddep_launch();
  int expert, row, n;
  if (!get_entry(p, y, expert, row, n)) return;
  __shared__ float red[kThreads * 8];
  gateup_task<FMT>(p, expert, row, n, blockIdx.x, tpc, red);
}

// Gate/up for T <= 8 tokens that routes itself: every routed CTA takes the
// top-k and the dispatch from the router's partial sums (a few KB through
// L2) instead of waiting for a routing kernel and reading its work entries;
// CTA (0, first routed) also publishes the routing.  The shared expert's CTAs
// run at once.
template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) gateup_routed_kernel(ExpertParams p, RouteParams rp, int tpc) {
  const int y = blockIdx.y;
  __shared__ float red[kThreads * 8];
  if (y < p.nsh) {
    int expert, row, n;
    if (get_entry(p, y, expert, row, n)) gateup_task<FMT>(p, expert, row, n, blockIdx.x, tpc, red);
    return;
  }
  __shared__ SmallRoute rt;
  griddep_wait();  // the router's partial sums
  const bool pub = y == p.nsh && blockIdx.x == 0;
  route_small_cta(rp, rt, pub);
  griddep_launch();  // the next kernel routes itself from the same partial sums
  const int d = y - p.nsh;
  if (d < rt.n_entries) {
    const int4 e = rt.entries[d];
    ExpertParams el = p;  // the routed rows' tokens from shared memory
    el.row_token = rt.row_token;
    gateup_task<FMT>(el, e.x, e.y, e.z, blockIdx.x, tpc, red);
  }
  if (pub) publish_counts(rp, rt);
}

// ---------------------------------------------------------------- down
template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) down_kernel(ExpertParams p, int tpc) {
  griddep_wait();
  int expert, row, n;
  if (!get_entry(p, blockIdx.y, expert, row, n)) return;
  __shared__ float red[kThreads * 8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int nks = kWarps / tpc;
  const int tile = blockIdx.x * tpc + (warp % tpc), ks = warp / tpc;
  const bool valid = tile < p.H / 16;
  const MatGeom g = mat_geom(FMT, p.I);
  const uint8_t* const tiles[1] = {p.arena + (size_t)expert * p.expert_bytes + p.gu_bytes +
                                   (size_t)tile * p.dn_tile_bytes};
  const uint16_t* brow = gi < n ? p.abuf + (size_t)(row + gi) * p.I : nullptr;
  float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
  if (valid) {
    prefetch_tile(FMT, tiles[0], g, ks + nks, nks);
    tiles_mma<FMT, 1>(tiles, g, ks, nks, brow, false, acc);
  }
  float v[4] = {acc[0][0], acc[0][1], acc[0][2], acc[0][3]};
  reduce_ksplit<4>(red, v, tpc, nks);
  if (ks != 0 || !valid) return;
  const float ts = p.tscale[expert * 3 + 2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 16 * tile + gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
    if (col < n) p.ybuf[(size_t)(row + col) * p.H + r] = ts * v[i];
  }
}

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

// ---------------------------------------------------------------- down + combine for a few tokens
// CTA = one 16-row tile of H for every work entry of the forward (one warp per
// entry); y of all rows stays in shared memory and the CTA writes
// out[:, tile] = sum_j g_j y_j + y_s with the same j-ordered fmaf chain as
// combine_kernel, so both paths agree bit for bit.  The tile's weights are
// known once routing is done, so they are requested from L2 before waiting
// for gate/up.
constexpr int kDcMaxWarps = 12;

template <int FMT>
__global__ void __launch_bounds__(kDcMaxWarps * 32) down_combine_kernel(ExpertParams p,
                                                                         const float* gates,
                                                                         const int* inv, float* out) {
  // routing is complete here (gate/up triggered this launch only after its wait):
  // the weights are read before waiting for gate/up
  DownPreload pre;
  bool have = false;
  if (FMT == FMT_NVFP4 && p.I <= 512) have = down_preload(p, blockIdx.x, threadIdx.x >> 5, pre);
  down_prefetch<FMT>(p, blockIdx.x);  // (the rest: into L2)
  griddep_wait();  // gate/up complete: abuf holds every row
  extern __shared__ float ys[];  // [rows x 16]
  down_combine_task<FMT>(p, blockIdx.x, gates, inv, out, ys, pre, have);
}

// The same for T <= 8 with routing in the CTA: the router finished before
// gate/up let this launch start, so its partial sums are final; the top-k,
// the dispatch and the weights all come before waiting for gate/up.
template <int FMT>
__global__ void __launch_bounds__(kDcMaxWarps * 32) down_combine_routed_kernel(ExpertParams p,
                                                                                RouteParams rp,
                                                                                float* out) {
  __shared__ SmallRoute rt;
  route_small_cta(rp, rt, false);
  ExpertParams el = p;
  el.entries = rt.entries;
  el.n_entries = &rt.n_entries;
  el.row_token = rt.row_token;
  DownPreload pre;
  bool have = false;
  if (FMT == FMT_NVFP4 && p.I <= 512) have = down_preload(el, blockIdx.x, threadIdx.x >> 5, pre);
  down_prefetch<FMT>(el, blockIdx.x);
  griddep_wait();  // gate/up complete: abuf holds every row
  extern __shared__ float ys[];
  down_combine_task<FMT>(el, blockIdx.x, rt.gates, rt.inv, out, ys, pre, have);
}

size_t down_combine_smem(int T, int k, int shared) {
  return ((size_t)T * k + (shared ? T : 0)) * 16 * sizeof(float);
}



}  // namespace

cudaError_t launch_gateup(const ExpertParams& p, int grid_y, bool pdl, cudaStream_t st) {
  const int tpc = tiles_per_cta(n_halves(mat_geom(p.fmt, p.H)));
  const int pairs = p.I / 16;
  dim3 grid((pairs + tpc - 1) / tpc, grid_y);
  if (p.fmt == FMT_NVFP4)
    return launch_k(gateup_kernel<FMT_NVFP4>, grid, dim3(kThreads), 0, st, pdl, p, tpc);
  return launch_k(gateup_kernel<FMT_FP6>, grid, dim3(kThreads), 0, st, pdl, p, tpc);
}

cudaError_t launch_down(const ExpertParams& p, int grid_y, bool pdl, cudaStream_t st) {
  const int tpc = tiles_per_cta(n_halves(mat_geom(p.fmt, p.I)));
  const int tiles = p.H / 16;
  dim3 grid((tiles + tpc - 1) / tpc, grid_y);
  if (p.fmt == FMT_NVFP4)
    return launch_k(down_kernel<FMT_NVFP4>, grid, dim3(kThreads), 0, st, pdl, p, tpc);
  return launch_k(down_kernel<FMT_FP6>, grid, dim3(kThreads), 0, st, pdl, p, tpc);
}

cudaError_t launch_combine(const ExpertParams& p, const float* gates, const int* inv, float* out,
                           bool pdl, cudaStream_t st) {
  const int64_t n = (int64_t)p.T * (p.H / 4);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  return launch_k(combine_kernel, dim3(blocks), dim3(256), 0, st, pdl, p, gates, inv, out);
}

bool down_combine_ok(int T, int k, int shared, int I) {
  (void)I;
  return T <= kTokTile && down_combine_smem(T, k, shared) <= 48 * 1024;
}

cudaError_t launch_down_combine(const ExpertParams& p, const float* gates, const int* inv,
                                float* out, bool pdl, cudaStream_t st) {
  // one warp per work entry (the routed entries are at most T*k for T <= 8)
  int warps = p.nsh + (p.T * p.k < p.E ? p.T * p.k : p.E);
  if (warps > kDcMaxWarps) warps = kDcMaxWarps;
  const size_t smem = down_combine_smem(p.T, p.k, p.shared);
  if (p.fmt == FMT_NVFP4)
    return launch_k(down_combine_kernel<FMT_NVFP4>, dim3(p.H / 16), dim3(32 * warps), smem, st,
                    pdl, p, gates, inv, out);
  return launch_k(down_combine_kernel<FMT_FP6>, dim3(p.H / 16), dim3(32 * warps), smem, st, pdl, p,
                  gates, inv, out);
}

bool small_route_ok(int T, int k) { return T <= kTokTile && T * k <= kSmallSlots; }

cudaError_t launch_gateup_routed(const ExpertParams& p, const RouteParams& rp, int grid_y,
                                 cudaStream_t st) {
  const int tpc = tiles_per_cta(n_halves(mat_geom(p.fmt, p.H)));
  const int pairs = p.I / 16;
  dim3 grid((pairs + tpc - 1) / tpc, grid_y);
  if (p.fmt == FMT_NVFP4)
    return launch_k(gateup_routed_kernel<FMT_NVFP4>, grid, dim3(kThreads), 0, st, true, p, rp, tpc);
  return launch_k(gateup_routed_kernel<FMT_FP6>, grid, dim3(kThreads), 0, st, true, p, rp, tpc);
}

cudaError_t launch_down_combine_routed(const ExpertParams& p, const RouteParams& rp, float* out,
                                       cudaStream_t st) {
  // one warp per work entry, at least 8 warps (the routing wants the slots covered)
  int warps = p.nsh + (p.T * p.k < p.E ? p.T * p.k : p.E);
  if (warps > kDcMaxWarps) warps = kDcMaxWarps;
  if (warps < 8) warps = 8;
  const size_t smem = down_combine_smem(p.T, p.k, p.shared);
  if (p.fmt == FMT_NVFP4)
    return launch_k(down_combine_routed_kernel<FMT_NVFP4>, dim3(p.H / 16), dim3(32 * warps), smem, st,
                    true, p, rp, out);
  return launch_k(down_combine_routed_kernel<FMT_FP6>, dim3(p.H / 16), dim3(32 * warps), smem, st, true,
                  p, rp, out);
}

cudaError_t expert_kernels_init() { return cudaSuccess; }

}  // namespace moe
