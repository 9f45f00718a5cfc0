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
// SMEM: the NVFP4 tile pair through shared memory (gateup_task_nv, one tile
// pair per CTA, several CTAs per SM); otherwise registers (gateup_task).
template <int FMT, bool SMEM>
__global__ void __launch_bounds__(kThreads, SMEM ? 3 : 2) gateup_kernel(ExpertParams p, int tpc) {
  const int y = blockIdx.y;
  // Shared-expert entries need no routing.  Routed ones wait for it, and only
  // then let the next kernel start: once every CTA here has triggered, the
  // routing outputs (work entries) are complete and the next kernel may read
  // them before its own wait.  With quantised activations (W4A4) every entry
  // reads the quantised x, written before the router: all of them wait.
  if (y >= p.nsh || p.ts_x) griddep_wait();
  griddep_launch();
  int expert, row, n;
  if (!get_entry(p, y, expert, row, n)) return;
  __shared__ float red[kThreads * 8];
  if constexpr (SMEM) {
    extern __shared__ __align__(16) uint8_t gu_smem[];
    gateup_task_nv(p, expert, row, n, blockIdx.x, gu_smem, red, false);
  } else {
    gateup_task<FMT>(p, expert, row, n, blockIdx.x, tpc, red);
  }
}

// Gate/up for T <= 8 tokens that routes itself: every routed CTA takes the
// top-k and the dispatch from the router's partial sums (a few KB through
// L2) instead of waiting for a routing kernel and reading its work entries;
// CTA (0, first routed) also publishes the routing for the down kernel (which
// reads it after its wait).  Every CTA, once its gate/up weights have landed,
// asks L2 for its share of its expert's down matrix, so the down kernel reads
// its weights from L2.  The shared expert's CTAs run at once.
// PATH 0: registers (gateup_task); 1: the NVFP4 tile pair through shared
// memory (gateup_task_nv); 3: the same for tile pairs blockIdx.x * tpc ...
// + tpc - 1 one after another (when one pair per CTA would not fit the GPU at
// once: a CTA then routes once for several tile pairs); 2: streamed tile
// pairs (stream_task, FP6).
template <int FMT, int PATH>
__device__ __forceinline__ void gateup_any_task(const ExpertParams& p, int expert, int row, int n,
                                                int tpc, uint8_t* smem, float* red) {
  if constexpr (PATH == 1) {
    gateup_task_nv(p, expert, row, n, blockIdx.x, smem, red, true);
  } else if constexpr (PATH == 3) {
    const int pairs = p.I / 16, end = min(pairs, (int)(blockIdx.x + 1) * tpc);
    for (int pair = blockIdx.x * tpc; pair < end; ++pair) {
      gateup_task_nv(p, expert, row, n, pair, smem, red, true);
      __syncthreads();  // warp 0 has read `red`, every warp is done with its stages
    }
  }
  else if constexpr (PATH == 2)
    stream_task<FMT, 0, 2>(p, expert, row, n, blockIdx.x, smem);
  else
    gateup_task<FMT>(p, expert, row, n, blockIdx.x, tpc, red);
}

template <int FMT, int PATH>
__global__ void __launch_bounds__(kThreads, PATH == 1 || PATH == 3 ? 3 : 2) gateup_routed_kernel(ExpertParams p, RouteParams rp, int tpc) {
  const int y = blockIdx.y;
  __shared__ float red[kThreads * 8];
  extern __shared__ __align__(16) uint8_t gu_smem[];
  if (y < p.nsh) {
    if (p.ts_x) griddep_wait();  // W4A4: the quantised x (written before the router)
    griddep_launch();
    int expert, row, n;
    if (get_entry(p, y, expert, row, n)) gateup_any_task<FMT, PATH>(p, expert, row, n, tpc, gu_smem, red);
    return;
  }
  __shared__ SmallRoute rt;
  griddep_wait();  // the router's partial sums and f16 copy of x
  const bool pub = y == p.nsh && blockIdx.x == 0;
  route_small_cta(rp, rt, pub);
  griddep_launch();
  const int d = y - p.nsh;
  if (d < rt.n_entries) {
    const int4 e = rt.entries[d];
    ExpertParams el = p;  // the routed rows' tokens from shared memory
    el.row_token = rt.row_token;
    gateup_any_task<FMT, PATH>(el, e.x, e.y, e.z, tpc, gu_smem, red);
  }
  if (pub) publish_counts(rp, rt);
}

// ---------------------------------------------------------------- streamed GEMVs
// NVFP4 for 8 < T, FP6 at every T.  MODE 0: gate/up + SwiGLU (shared-expert
// entries run ahead of the router); MODE 1: down.  See stream_task.
template <int FMT, int MODE>
__global__ void __launch_bounds__(kThreads, 2) stream_kernel(ExpertParams p) {
  const int y = blockIdx.y;
  if (MODE == 1 || y >= p.nsh || p.ts_x) griddep_wait();
  griddep_launch();
  int expert, row, n;
  if (!get_entry(p, y, expert, row, n)) return;
  extern __shared__ __align__(16) uint8_t stream_smem_buf[];
  stream_task<FMT, MODE>(p, expert, row, n, blockIdx.x, stream_smem_buf);
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
  const uint8_t* const tiles[1] = {expert_base(p, expert) + p.gu_bytes +
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
    if (col < n) p.ybuf[(size_t)(row + col) * p.H + r] = (ts * a_scale(p, row + col)) * v[i];
  }
}

// ---------------------------------------------------------------- combine
// out[t] = sum_j gates[t,j] * y[row(t,j)] + y_shared[t], j in order.  One
// warp per (token, slice of 32U float4s of the row): lane j < k reads gate j
// and row j once and hands them out by shuffle; each lane accumulates U
// float4s (h, h + 32, ...), so every step of the j loop has U independent
// row loads in flight (U = 1 when there are too few tokens to fill the GPU).
template <int U>
__global__ void __launch_bounds__(256) combine_kernel(ExpertParams p, const float* gates,
                                                      const int* inv, float* out) {
  griddep_launch();
  griddep_wait();
  const int H4 = p.H / 4, S = p.T * p.k, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const float4* y4 = reinterpret_cast<const float4*>(p.ybuf);
  float4* o4 = reinterpret_cast<float4*>(out);
  const int ns = (H4 + 32 * U - 1) / (32 * U);  // slices per row
  for (int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < p.T * ns; item += nwarps) {
    const int t = item / ns;
    const float g_l = lane < p.k ? gates[(size_t)t * p.k + lane] : 0.f;
    const int r_l = lane < p.k ? inv[(size_t)t * p.k + lane] : 0;
    {
      const int h0 = (item - t * ns) * 32 * U + lane;
      float4 acc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
      for (int j = 0; j < p.k; ++j) {
        const float g = __shfl_sync(0xffffffffu, g_l, j);
        const float4* yr = y4 + (size_t)__shfl_sync(0xffffffffu, r_l, j) * H4;
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (h0 + 32 * u < H4) {
            const float4 yv = yr[h0 + 32 * u];
            acc[u].x = fmaf(g, yv.x, acc[u].x);
            acc[u].y = fmaf(g, yv.y, acc[u].y);
            acc[u].z = fmaf(g, yv.z, acc[u].z);
            acc[u].w = fmaf(g, yv.w, acc[u].w);
          }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int h = h0 + 32 * u;
        if (h >= H4) continue;
        if (p.shared) {
          const float4 yv = y4[(size_t)(S + t) * H4 + h];
          acc[u].x += yv.x; acc[u].y += yv.y; acc[u].z += yv.z; acc[u].w += yv.w;
        }
        o4[(size_t)t * H4 + h] = acc[u];
      }
    }
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

// WAIT_FIRST: the routing is published by the kernel before this one (the
// self-routed gate/up), so nothing is read before the wait; the weights come
// from L2, where gate/up asked for them.  Otherwise the routing is complete
// before gate/up starts, and the first entry's tile is loaded into registers
// and the others requested from L2 before the wait.  Either way the next
// kernel may start at once (it waits for this whole grid before it reads
// anything this one writes).
// LONGK (NVFP4, I > 512): one-row entries stream their tile through a ring
template <int FMT, bool WAIT_FIRST, bool LONGK = false>
__global__ void __launch_bounds__(kDcMaxWarps * 32) down_combine_kernel(ExpertParams p,
                                                                         const float* gates,
                                                                         const int* inv, float* out) {
  griddep_launch();
  DownPreload pre;
  bool have = false;
  const bool preload = FMT == FMT_NVFP4 && p.I <= 512;
  if (!WAIT_FIRST) {
    if (preload) have = down_preload(p, blockIdx.x, threadIdx.x >> 5, pre);
    down_prefetch<FMT>(p, blockIdx.x);  // (the rest: into L2)
  } else if (preload) {
    // Speculative: the routing this grid reads is published by the gate/up
    // grid long before that grid ends, so the entry read now is almost always
    // the final one.  It is checked again after the wait; a stale or torn
    // read only costs a reload (every address it forms is bounds-checked).
    have = down_preload(p, blockIdx.x, threadIdx.x >> 5, pre, true);
  }
  griddep_wait();  // gate/up complete: abuf holds every row
  __shared__ float sg[kTokTile * kMaxK];
  __shared__ int si[kTokTile * kMaxK];
  if (WAIT_FIRST) {
    // the warp's entry read again now that it is final: the speculative
    // tile stays if it is this entry's expert, else every entry's tile is
    // requested at once; then the combine's gates and rows
    if (preload) {
      int e, r, n;
      const bool ok = get_entry(p, threadIdx.x >> 5, e, r, n);
      if (!ok) {
        have = false;
      } else if (have && e == pre.expert) {
        pre.row = r;
        pre.n = n;
      } else {
        have = down_preload(p, blockIdx.x, threadIdx.x >> 5, pre);
      }
    }
    for (int i = threadIdx.x; i < p.T * p.k; i += blockDim.x) {
      sg[i] = gates[i];
      si[i] = inv[i];
    }
    gates = sg;  // read after the task's barrier
    inv = si;
  }
  extern __shared__ float ys[];  // [rows x 16], then (FP6) the warps' unit rings
  const int rows = p.T * p.k + (p.shared ? p.T : 0);
  down_combine_task<FMT, LONGK>(p, blockIdx.x, gates, inv, out, ys, smem_u32(ys + rows * 16), pre,
                                have);
}

// ys (rows x 16 floats); the FP6 unit rings come on top (down_combine_ring)
size_t down_combine_smem(int T, int k, int shared) {
  return ((size_t)T * k + (shared ? T : 0)) * 16 * sizeof(float);
}
size_t down_combine_ring(int fmt, int I, int warps) {
  if (fmt == FMT_FP6) return (size_t)warps * 2 * kDcFp6Stage;
  return I > 512 ? (size_t)warps * kDcNvStages * kDcNvStage : 0;
}



}  // namespace

// Dynamic shared memory the NVFP4 tile-pair gate/up kernels may use (set in
// expert_kernels_init); larger shapes take the register kernels.
constexpr int kNvMaxDyn = 160 * 1024;

// The tile-pair task (one pair per CTA, warps splitting K) for T <= 8 only:
// for larger batches it would stage every entry's token rows once per tile
// pair, and the streamed kernels (a warp per pair over the whole K, rows
// staged once per CTA) take over.
bool gateup_smem_ok(const ExpertParams& p) {
  return p.fmt == FMT_NVFP4 && p.T <= kTokTile && gateup_nv_smem(p.H, p.T) <= kNvMaxDyn;
}

// Streamed GEMVs: NVFP4 for T > 8 (T <= 8 keeps the tile-pair gate/up and
// the fused down + combine), FP6 at every T; within the dynamic shared-memory
// budget.
constexpr int kStreamMaxDyn = 200 * 1024;
bool stream_ok(const ExpertParams& p, int mode) {
  if (p.fmt == FMT_NVFP4 && p.T <= kTokTile) return false;
  return stream_smem(p.fmt, 2, mode == 0 ? p.H : p.I, p.T, 2) <= kStreamMaxDyn;
}

template <int MODE>
cudaError_t launch_stream(const ExpertParams& p, int grid_y, bool pdl, cudaStream_t st) {
  // a warp per gate/up tile pair (I/16 of them) or per two down tiles (H/32)
  const int items = MODE == 0 ? p.I / 16 : p.H / 32;
  const dim3 grid((items + kWarps - 1) / kWarps, grid_y);
  const size_t smem = stream_smem(p.fmt, 2, MODE == 0 ? p.H : p.I, p.T, 2);
  if (p.fmt == FMT_NVFP4)
    return launch_k(stream_kernel<FMT_NVFP4, MODE>, grid, dim3(kThreads), smem, st, pdl, p);
  return launch_k(stream_kernel<FMT_FP6, MODE>, grid, dim3(kThreads), smem, st, pdl, p);
}

cudaError_t launch_gateup(const ExpertParams& p, int grid_y, bool pdl, cudaStream_t st) {
  const int pairs = p.I / 16;
  if (stream_ok(p, 0)) return launch_stream<0>(p, grid_y, pdl, st);
  if (gateup_smem_ok(p))
    return launch_k(gateup_kernel<FMT_NVFP4, true>, dim3(pairs, grid_y), dim3(kThreads),
                    gateup_nv_smem(p.H, p.T), st, pdl, p, 1);
  const int tpc = tiles_per_cta(n_halves(mat_geom(p.fmt, p.H)));
  dim3 grid((pairs + tpc - 1) / tpc, grid_y);
  if (p.fmt == FMT_NVFP4)
    return launch_k(gateup_kernel<FMT_NVFP4, false>, grid, dim3(kThreads), 0, st, pdl, p, tpc);
  return launch_k(gateup_kernel<FMT_FP6, false>, grid, dim3(kThreads), 0, st, pdl, p, tpc);
}

cudaError_t launch_down(const ExpertParams& p, int grid_y, bool pdl, cudaStream_t st) {
  if (stream_ok(p, 1)) return launch_stream<1>(p, grid_y, pdl, st);
  const int tpc = tiles_per_cta(n_halves(mat_geom(p.fmt, p.I)));
  const int tiles = p.H / 16;
  dim3 grid((tiles + tpc - 1) / tpc, grid_y);
  if (p.fmt == FMT_NVFP4)
    return launch_k(down_kernel<FMT_NVFP4>, grid, dim3(kThreads), 0, st, pdl, p, tpc);
  return launch_k(down_kernel<FMT_FP6>, grid, dim3(kThreads), 0, st, pdl, p, tpc);
}

cudaError_t launch_combine(const ExpertParams& p, const float* gates, const int* inv, float* out,
                           bool pdl, cudaStream_t st) {
  // a warp per item; 4 float4s per lane once that still gives every SM 16 warps
  const int64_t items4 = (int64_t)p.T * ((p.H / 4 + 127) / 128);
  const bool wide = items4 >= 152 * 16;
  const int64_t items = wide ? items4 : (int64_t)p.T * ((p.H / 4 + 31) / 32);
  int blocks = (int)((items + 7) / 8);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (wide) return launch_k(combine_kernel<4>, dim3(blocks), dim3(256), 0, st, pdl, p, gates, inv, out);
  return launch_k(combine_kernel<1>, dim3(blocks), dim3(256), 0, st, pdl, p, gates, inv, out);
}

bool down_combine_ok(int T, int k, int shared, int I) {
  (void)I;
  return T <= kTokTile && down_combine_smem(T, k, shared) <= 48 * 1024;
}

cudaError_t launch_down_combine(const ExpertParams& p, const float* gates, const int* inv,
                                float* out, bool pdl, bool wait_first, cudaStream_t st) {
  // one warp per work entry (the routed entries are at most T*k for T <= 8)
  int warps = p.nsh + (p.T * p.k < p.E ? p.T * p.k : p.E);
  if (warps > kDcMaxWarps) warps = kDcMaxWarps;
  const size_t smem = down_combine_smem(p.T, p.k, p.shared) + down_combine_ring(p.fmt, p.I, warps);
  const dim3 grid(p.H / 16), block(32 * warps);
  if (p.fmt == FMT_NVFP4 && p.I > 512)
    return wait_first
               ? launch_k(down_combine_kernel<FMT_NVFP4, true, true>, grid, block, smem, st, pdl, p, gates, inv, out)
               : launch_k(down_combine_kernel<FMT_NVFP4, false, true>, grid, block, smem, st, pdl, p, gates, inv, out);
  if (p.fmt == FMT_NVFP4)
    return wait_first
               ? launch_k(down_combine_kernel<FMT_NVFP4, true>, grid, block, smem, st, pdl, p, gates, inv, out)
               : launch_k(down_combine_kernel<FMT_NVFP4, false>, grid, block, smem, st, pdl, p, gates, inv, out);
  return wait_first
             ? launch_k(down_combine_kernel<FMT_FP6, true>, grid, block, smem, st, pdl, p, gates, inv, out)
             : launch_k(down_combine_kernel<FMT_FP6, false>, grid, block, smem, st, pdl, p, gates, inv, out);
}

bool small_route_ok(int T, int k) { return T <= kTokTile && T * k <= kSmallSlots; }

cudaError_t launch_gateup_routed(const ExpertParams& p, const RouteParams& rp, int grid_y,
                                 cudaStream_t st) {
  const int pairs = p.I / 16;
  if (gateup_smem_ok(p)) {
    // tile pairs per CTA: enough that the grid fits the GPU at once (CTAs
    // per SM from the shared memory a CTA holds: dynamic + 23.6 KB static)
    const size_t dyn = gateup_nv_smem(p.H, p.T);
    int per_sm = (int)((228u * 1024u) / (dyn + 25u * 1024u));
    per_sm = per_sm < 1 ? 1 : (per_sm > 3 ? 3 : per_sm);
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long slots = (long)sms * per_sm, ctas = (long)pairs * grid_y;
    if (ctas <= slots)
      return launch_k(gateup_routed_kernel<FMT_NVFP4, 1>, dim3(pairs, grid_y), dim3(kThreads), dyn,
                      st, true, p, rp, 1);
    const int ppc = (int)((ctas + slots - 1) / slots);
    return launch_k(gateup_routed_kernel<FMT_NVFP4, 3>, dim3((pairs + ppc - 1) / ppc, grid_y),
                    dim3(kThreads), dyn, st, true, p, rp, ppc);
  }
  if (p.fmt == FMT_FP6 && stream_ok(p, 0))
    return launch_k(gateup_routed_kernel<FMT_FP6, 2>, dim3((pairs + kWarps - 1) / kWarps, grid_y),
                    dim3(kThreads), stream_smem(p.fmt, 2, p.H, p.T, 2), st, true, p, rp, 1);
  const int tpc = tiles_per_cta(n_halves(mat_geom(p.fmt, p.H)));
  dim3 grid((pairs + tpc - 1) / tpc, grid_y);
  if (p.fmt == FMT_NVFP4)
    return launch_k(gateup_routed_kernel<FMT_NVFP4, 0>, grid, dim3(kThreads), 0, st, true, p, rp, tpc);
  return launch_k(gateup_routed_kernel<FMT_FP6, 0>, grid, dim3(kThreads), 0, st, true, p, rp, tpc);
}

cudaError_t expert_kernels_init() {
  cudaError_t e = cudaFuncSetAttribute(gateup_kernel<FMT_NVFP4, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kNvMaxDyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gateup_routed_kernel<FMT_NVFP4, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kNvMaxDyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gateup_routed_kernel<FMT_NVFP4, 3>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kNvMaxDyn);
  // (the routed kernel also holds 23.6 KB of static shared memory)
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gateup_routed_kernel<FMT_FP6, 2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamMaxDyn);

  // ys (at most 48 KB: down_combine_ok) and up to kDcMaxWarps warps' rings
  // (12 x 4 x 3072 bytes NVFP4 with I > 512, 12 x 2 x 3712 FP6): 195 KB at most
  constexpr int kDcMaxDyn = 200 * 1024;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(down_combine_kernel<FMT_NVFP4, true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kDcMaxDyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(down_combine_kernel<FMT_NVFP4, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kDcMaxDyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(down_combine_kernel<FMT_FP6, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kDcMaxDyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(down_combine_kernel<FMT_FP6, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kDcMaxDyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_kernel<FMT_NVFP4, 0>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamMaxDyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_kernel<FMT_NVFP4, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamMaxDyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_kernel<FMT_FP6, 0>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamMaxDyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_kernel<FMT_FP6, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamMaxDyn);
  return e;
}

}  // namespace moe
