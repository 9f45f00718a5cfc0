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
#include "kernels.cuh"
#include "layout.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float ue8m0_to_f32(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// The 16 f16 activations of this lane's token row at column `col` (two
// 16-byte reads, kept in L1: the warps of a CTA share them), or zeros.
// A bf16 source row (b_bf16) is converted to f16 in registers: the shared
// expert's CTAs start before the router has written the f16 copy of x.
__device__ __forceinline__ void load_b(const uint16_t* brow, int col, bool b_bf16,
                                       uint32_t (&xw)[8]) {
  if (brow) {
    const uint4* px = reinterpret_cast<const uint4*>(brow + col);
    const uint4 q0 = px[0], q1 = px[1];
    xw[0] = q0.x; xw[1] = q0.y; xw[2] = q0.z; xw[3] = q0.w;
    xw[4] = q1.x; xw[5] = q1.y; xw[6] = q1.z; xw[7] = q1.w;
    if (b_bf16) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(xw[i] << 16),
                                            __uint_as_float(xw[i] & 0xFFFF0000u));
        xw[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) xw[i] = 0u;
  }
}

// Work is split along K in units of 256 columns: 4 NVFP4 chunks of 64 or 2
// FP6 blocks of 128.  A warp handles units h0, h0 + dh, ...; per unit it keeps
// all weight vectors and activation fragments in flight before doing the math.
__host__ __device__ __forceinline__ int n_halves(const MatGeom& g) { return (g.K + 255) / 256; }

// NT NVFP4 tiles (same K) times the activations.
// brow: this lane's B row (f16, K long), null when the lane's column is empty.
template <int NT>
__device__ __forceinline__ void tiles_nvfp4(const uint8_t* const (&tile)[NT], const MatGeom& g,
                                            int h0, int dh, const uint16_t* brow, bool b_bf16,
                                            float (&acc)[NT][4]) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int nh = n_halves(g);
  for (int hh = h0; hh < nh; hh += dh) {
    const int s = hh >> 1, jb = (hh & 1) * 4;
    const int nc = min(4, sc_units(g, s) - jb);
    uint4 sv[NT], cv[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const uint8_t* b = tile[i] + (size_t)s * g.sc_bytes + 16 * lane;
      sv[i] = ldg_stream(b);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < nc) cv[i][j] = ldg_stream(b + 512 * (1 + jb + j));
    }
    uint32_t xb[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < nc) load_b(brow, 64 * (8 * s + jb + j) + 16 * t, b_bf16, xb[j]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j < nc) {
        const int jj = jb + j;  // chunk within the super-chunk
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const uint32_t sp = e4m3x2_to_f16x2((u4get(sv[i], jj >> 1) >> (16 * (jj & 1))) & 0xFFFFu);
          const uint32_t s_lo = dup_lo(sp), s_hi = dup_hi(sp);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint32_t h[4];
            e2m1x8_to_f16x8(u4get(cv[i][j], w), h);
            const uint32_t a[4] = {hmul2(h[0], s_lo), hmul2(h[1], s_hi), hmul2(h[2], s_lo),
                                   hmul2(h[3], s_hi)};
            mma_f16(acc[i], a, xb[j][2 * w], xb[j][2 * w + 1]);
          }
        }
      }
    }
  }
}

__device__ __forceinline__ void fp6_unpack(uint32_t Ha, uint32_t Hb, uint32_t L, uint32_t (&c)[4]) {
  c[0] = ((Ha << 2) & 0x3C3C3C3Cu) | (L & 0x03030303u);
  c[1] = ((Ha >> 2) & 0x3C3C3C3Cu) | ((L >> 2) & 0x03030303u);
  c[2] = ((Hb << 2) & 0x3C3C3C3Cu) | ((L >> 4) & 0x03030303u);
  c[3] = ((Hb >> 2) & 0x3C3C3C3Cu) | ((L >> 6) & 0x03030303u);
}

// NT FP6 tiles; a unit is 2 blocks (pairs of 64-column chunks) of 128 columns.
template <int NT>
__device__ __forceinline__ void tiles_fp6(const uint8_t* const (&tile)[NT], const MatGeom& g,
                                          int h0, int dh, const uint16_t* brow, bool b_bf16,
                                          float (&acc)[NT][4]) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int nh = n_halves(g);
  for (int hh = h0; hh < nh; hh += dh) {
    const int s = hh >> 2, j0 = (hh & 3) * 2;
    const int np = sc_units(g, s);
    uint32_t ew[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) ew[i] = ldg_stream_u32(tile[i] + (size_t)s * g.sc_bytes + 4 * lane);
    uint4 cv[NT][2][3];
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
        if (j0 + jj < np)
#pragma unroll
          for (int v = 0; v < 3; ++v)
            cv[i][jj][v] = ldg_stream(tile[i] + (size_t)s * g.sc_bytes + 128 + 1536 * (j0 + jj) +
                                      512 * v + 16 * lane);
    uint32_t xb[2][2][8];  // activation fragments of the 2 blocks, both chunks
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
      if (j0 + jj < np)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          load_b(brow, 128 * (8 * s + j0 + jj) + 64 * h + 16 * t, b_bf16, xb[jj][h]);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      if (j0 + jj < np) {
        const int j = j0 + jj;
        float blk[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
          for (int r = 0; r < 4; ++r) blk[i][r] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            const uint32_t words[12] = {cv[i][jj][0].x, cv[i][jj][0].y, cv[i][jj][0].z,
                                        cv[i][jj][0].w, cv[i][jj][1].x, cv[i][jj][1].y,
                                        cv[i][jj][1].z, cv[i][jj][1].w, cv[i][jj][2].x,
                                        cv[i][jj][2].y, cv[i][jj][2].z, cv[i][jj][2].w};
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint32_t c[4];
              fp6_unpack(words[h * 6 + q * 3], words[h * 6 + q * 3 + 1], words[h * 6 + q * 3 + 2], c);
#pragma unroll
              for (int ww = 0; ww < 2; ++ww) {
                const int w = 2 * q + ww;
                uint32_t u[2], v[2];
                e2m3x4_to_f16x4(c[2 * ww], u);      // rows g, g+8 at columns 4w, 4w+1
                e2m3x4_to_f16x4(c[2 * ww + 1], v);  // rows g, g+8 at columns 4w+2, 4w+3
                const uint32_t a[4] = {u[0], u[1], v[0], v[1]};
                mma_f16(blk[i], a, xb[jj][h][2 * w], xb[jj][h][2 * w + 1]);
              }
            }
          }
        }
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const uint32_t e = __shfl_sync(0xffffffffu, ew[i], (gi << 2) | (j >> 1));
          const float f0 = ue8m0_to_f32((e >> (16 * (j & 1))) & 0xFFu);
          const float f1 = ue8m0_to_f32((e >> (16 * (j & 1) + 8)) & 0xFFu);
          acc[i][0] = fmaf(blk[i][0], f0, acc[i][0]);
          acc[i][1] = fmaf(blk[i][1], f0, acc[i][1]);
          acc[i][2] = fmaf(blk[i][2], f1, acc[i][2]);
          acc[i][3] = fmaf(blk[i][3], f1, acc[i][3]);
        }
      }
    }
  }
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// Ask L2 for every 16-byte vector this lane will read from one tile's halves
// h0, h0+dh, ... (fire and forget: no registers, no waiting).
__device__ __forceinline__ void prefetch_tile(int fmt, const uint8_t* tile, const MatGeom& g,
                                              int h0, int dh) {
  const int lane = threadIdx.x & 31;
  for (int hh = h0; hh < n_halves(g); hh += dh) {
    if (fmt == FMT_NVFP4) {
      const int s = hh >> 1, jb = (hh & 1) * 4;
      const uint8_t* b = tile + (size_t)s * g.sc_bytes;
      const int u = min(4, sc_units(g, s) - jb);
      prefetch_l2(b + 16 * lane);
      for (int j = 0; j < u; ++j) prefetch_l2(b + 512 * (1 + jb + j) + 16 * lane);
    } else {
      const int s = hh >> 2, jb = (hh & 3) * 2;
      const uint8_t* b = tile + (size_t)s * g.sc_bytes;
      const int u = min(2, sc_units(g, s) - jb);
      prefetch_l2(b + 4 * lane);
      for (int j = 0; j < 3 * u; ++j) prefetch_l2(b + 128 + 1536 * jb + 512 * j + 16 * lane);
    }
  }
}

template <int FMT, int NT>
__device__ __forceinline__ void tiles_mma(const uint8_t* const (&tile)[NT], const MatGeom& g,
                                          int s0, int ds, const uint16_t* brow, bool b_bf16,
                                          float (&acc)[NT][4]) {
  if (FMT == FMT_NVFP4)
    tiles_nvfp4<NT>(tile, g, s0, ds, brow, b_bf16, acc);
  else
    tiles_fp6<NT>(tile, g, s0, ds, brow, b_bf16, acc);
}

// Entry y of the launch: the first p.nsh are the shared expert's token groups
// (known without routing); the rest come from dispatch.
__device__ __forceinline__ bool get_entry(const ExpertParams& p, int y, int& expert, int& row,
                                          int& n) {
  const int S = p.T * p.k;
  if (y < p.nsh) {
    expert = p.E;
    row = S + kTokTile * y;
    n = min(kTokTile, p.T - kTokTile * y);
    return true;
  }
  const int r = y - p.nsh;
  const int4 e = p.entries[r];  // read together with the count (the slot always exists)
  if (r >= *p.n_entries) return false;
  expert = e.x;
  row = e.y;
  n = e.z;
  if (expert < 0 || expert >= p.E || n < 1 || n > kTokTile || row < 0 || row + n > S) {
    *p.status = -1;  // MOE_EINVAL: corrupt entry, skip it
    return false;
  }
  return true;
}

// Sum the per-warp partials of warps sharing a tile (fixed order) into warp ks == 0.
template <int NV>
__device__ __forceinline__ void reduce_ksplit(float* red, float (&v)[NV], int tpc, int nks) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (nks == 1) return;
#pragma unroll
  for (int i = 0; i < NV; ++i) red[(warp * 32 + lane) * NV + i] = v[i];
  __syncthreads();
  if (warp / tpc == 0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = 0.f;
    for (int ks = 0; ks < nks; ++ks) {
      const int w2 = ks * tpc + warp;
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] += red[(w2 * 32 + lane) * NV + i];
    }
  }
}

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
  const int S = p.T * p.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int nks = kWarps / tpc;
  const int pair = blockIdx.x * tpc + (warp % tpc), ks = warp / tpc;
  const bool valid = pair < p.I / 16;
  const MatGeom g = mat_geom(FMT, p.H);
  const uint8_t* eb = p.arena + (size_t)expert * p.expert_bytes;
  const uint8_t* const tiles[2] = {eb + (size_t)(2 * pair) * p.gu_tile_bytes,
                                   eb + (size_t)(2 * pair + 1) * p.gu_tile_bytes};
  // routed entries read the router's f16 copy of x; the shared expert's
  // entries run ahead of the router and read (and convert) x itself
  const bool shared_entry = expert == p.E;
  const uint16_t* brow = nullptr;
  if (gi < n) {
    const int tok = shared_entry ? row - S + gi : p.row_token[row + gi];
    brow = (shared_entry ? p.x : p.xh) + (size_t)tok * p.H;
  }
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  if (valid) {
    // the warp's later K-units are requested from L2 now, so their loads do not wait on HBM
    prefetch_tile(FMT, tiles[0], g, ks + nks, nks);
    prefetch_tile(FMT, tiles[1], g, ks + nks, nks);
    tiles_mma<FMT, 2>(tiles, g, ks, nks, brow, shared_entry, acc);
  }
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = acc[0][i];
    v[4 + i] = acc[1][i];
  }
  reduce_ksplit<8>(red, v, tpc, nks);
  if (ks != 0 || !valid) return;
  const float ts_g = p.tscale[expert * 3 + 0], ts_u = p.tscale[expert * 3 + 1];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 16 * pair + gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
    if (col < n) {
      const float G = ts_g * v[i], U = ts_u * v[4 + i];
      const float a = G / (1.0f + expf(-G)) * U;
      p.abuf[(size_t)(row + col) * p.I + r] = __half_as_ushort(__float2half_rn(a));
    }
  }
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
  const int tile = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int gi = lane >> 2, t = lane & 3;
  const int S = p.T * p.k, rows_total = S + (p.shared ? p.T : 0);
  const MatGeom g = mat_geom(FMT, p.I);
  // routing is complete here (gate/up triggered this launch only after its wait)
  const int n_entries = p.nsh + *p.n_entries;
  const uint8_t* tile_base = p.arena + p.gu_bytes + (size_t)tile * p.dn_tile_bytes;
  for (int y = warp; y < n_entries; y += nw) {
    const int expert = (y < p.nsh) ? p.E : p.entries[y - p.nsh].x;
    if (expert >= 0 && expert <= p.E)
      prefetch_tile(FMT, tile_base + (size_t)expert * p.expert_bytes, g, 0, 1);
  }
  griddep_wait();  // gate/up complete: abuf holds every row
  extern __shared__ float ys[];  // [rows_total x 16]
  for (int y = warp; y < n_entries; y += nw) {
    int expert, row, n;
    if (!get_entry(p, y, expert, row, n)) continue;
    const uint8_t* const tiles[1] = {tile_base + (size_t)expert * p.expert_bytes};
    const uint16_t* brow = gi < n ? p.abuf + (size_t)(row + gi) * p.I : nullptr;
    float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    tiles_mma<FMT, 1>(tiles, g, 0, 1, brow, false, acc);
    const float ts = p.tscale[expert * 3 + 2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
      if (col < n) ys[(row + col) * 16 + r] = ts * acc[0][i];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < p.T * 16; i += blockDim.x) {
    const int tk = i / 16, h = i % 16;
    float a = 0.f;
    for (int j = 0; j < p.k; ++j)
      a = fmaf(gates[(size_t)tk * p.k + j], ys[inv[(size_t)tk * p.k + j] * 16 + h], a);
    if (p.shared) a += ys[(S + tk) * 16 + h];
    out[(size_t)tk * p.H + 16 * tile + h] = a;
  }
  (void)rows_total;
}

size_t down_combine_smem(int T, int k, int shared) {
  return ((size_t)T * k + (shared ? T : 0)) * 16 * sizeof(float);
}

// Warps of a CTA: kWarps / tpc of them split K, tpc tile groups side by side.
// Each warp takes about two 256-column units (the second one requested from
// L2 up front), which keeps the decode grid within one wave at two CTAs per SM.
int tiles_per_cta(int units) {
  int nks = 1;
  while (nks * 2 <= kWarps && nks * 2 <= units / 2) nks *= 2;
  return kWarps / nks;
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

cudaError_t expert_kernels_init() { return cudaSuccess; }

}  // namespace moe
