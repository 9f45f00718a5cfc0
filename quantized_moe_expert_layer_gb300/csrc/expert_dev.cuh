// Device code of the expert GEMMs (dequantise packed tiles into m16n8k16 A
// fragments, activations as B), shared by the stand-alone expert kernels and
// the decode megakernel.
#pragma once

#include "async.cuh"
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

// Warps of a CTA: kWarps / tpc of them split K, tpc tile groups side by side.
// Each warp takes about two 256-column units (the second one requested from
// L2 up front), which keeps the decode grid within one wave at two CTAs per SM.
__host__ __device__ __forceinline__ int tiles_per_cta(int units) {
  int nks = 1;
  while (nks * 2 <= kWarps && nks * 2 <= units / 2) nks *= 2;
  return kWarps / nks;
}

// NT NVFP4 tiles (same K) times the activations.
// brow: this lane's B row (f16, K long), null when the lane's column is empty.
template <int NT>
__device__ __forceinline__ void tiles_nvfp4(const uint8_t* const (&tile)[NT], const MatGeom& g,
                                            int h0, int dh, const uint16_t* brow, bool b_bf16,
                                            float (&acc)[NT][4]) {
  const int lane = threadIdx.x & 31, t = lane & 3;
  const int nh = n_halves(g);
  float acc2[NT][2][4] = {};  // even / odd chunks: two shorter mma chains per tile
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
            mma_f16(acc2[i][jj & 1], a, xb[j][2 * w], xb[j][2 * w + 1]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[i][r] += acc2[i][0][r] + acc2[i][1][r];
}

// Byte containers for cvt.rn.f16x2.e2m3x2 from the 4-bit and 2-bit planes:
// bits 2-5 of each byte from the 4-bit plane, bits 0-1 from the 2-bit plane.
// cvt reads only bits 0-5 of a container (checked on sm_103a over every
// 16-bit input), so bits 6-7 may keep whatever the 2-bit plane's shift left
// there and each container is one bit-select.
__device__ __forceinline__ uint32_t sel_bits(uint32_t hi4, uint32_t lo2) {
  constexpr uint32_t M = 0x3C3C3C3Cu;
  return (hi4 & M) | (lo2 & ~M);
}
__device__ __forceinline__ void fp6_unpack(uint32_t Ha, uint32_t Hb, uint32_t L, uint32_t (&c)[4]) {
  c[0] = sel_bits(Ha << 2, L);
  c[1] = sel_bits(Ha >> 2, L >> 2);
  c[2] = sel_bits(Hb << 2, L >> 4);
  c[3] = sel_bits(Hb >> 2, L >> 6);
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
// quiet: a read that may race with the writer (speculation): an entry that
// fails the checks is skipped without setting the status word.
__device__ __forceinline__ bool get_entry(const ExpertParams& p, int y, int& expert, int& row,
                                          int& n, bool quiet = false) {
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
    if (!quiet) *p.status = kStatusInvalid;  // corrupt entry: skip it
    return false;
  }
  return true;
}

// W4A4: the activation tensor scale of token `tok`, and of row `row` of a
// (1 otherwise; ts * 1.0f is ts exactly, so the W4A16 path keeps its bits).
__device__ __forceinline__ float x_scale(const ExpertParams& p, int tok) {
  return p.ts_x ? p.ts_x[tok] : 1.0f;
}
__device__ __forceinline__ float a_scale(const ExpertParams& p, int row) {
  return p.ts_a ? p.ts_a[row] : 1.0f;
}
// Token of row `row` of abuf: the shared expert's rows S..S+T-1 are tokens 0..T-1.
__device__ __forceinline__ int row_tok(const ExpertParams& p, int row) {
  const int S = p.T * p.k;
  return row >= S ? row - S : p.row_token[row];
}
// The SwiGLU output a of (row, column r): f16 for the down kernels, or fp32
// for the W4A4 quantiser.
__device__ __forceinline__ void store_a(const ExpertParams& p, size_t row, int r, float a) {
  if (p.af)
    p.af[row * p.I + r] = a;
  else
    p.abuf[row * p.I + r] = a_to_f16(a, p.status);
}
// Shared-expert entries run ahead of the router and convert x themselves,
// unless x was quantised (W4A4): then every entry reads the quantised copy.
__device__ __forceinline__ bool convert_x(const ExpertParams& p, bool shared_entry) {
  return shared_entry && !p.ts_x;
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
// One CTA-level task: tile pairs group*tpc .. +tpc of `expert`, for the n
// tokens of rows row..row+n-1; red: kThreads x 8 floats of shared memory.
template <int FMT>
__device__ __forceinline__ void gateup_task(const ExpertParams& p, int expert, int row, int n,
                                            int group, int tpc, float* red) {
  const int S = p.T * p.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int nks = kWarps / tpc;
  const int pair = group * tpc + (warp % tpc), ks = warp / tpc;
  const bool valid = pair < p.I / 16;
  const MatGeom g = mat_geom(FMT, p.H);
  const uint8_t* eb = expert_base(p, expert);
  const uint8_t* const tiles[2] = {eb + (size_t)(2 * pair) * p.gu_tile_bytes,
                                   eb + (size_t)(2 * pair + 1) * p.gu_tile_bytes};
  // routed entries read the router's f16 copy of x; the shared expert's
  // entries run ahead of the router and read (and convert) x itself
  const bool shared_entry = expert == p.E, cvt = convert_x(p, shared_entry);
  const uint16_t* brow = nullptr;
  if (gi < n) {
    const int tok = shared_entry ? row - S + gi : p.row_token[row + gi];
    brow = (cvt ? p.x : p.xh) + (size_t)tok * p.H;
  }
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  if (valid) {
    // the warp's later K-units are requested from L2 now, so their loads do not wait on HBM
    prefetch_tile(FMT, tiles[0], g, ks + nks, nks);
    prefetch_tile(FMT, tiles[1], g, ks + nks, nks);
    tiles_mma<FMT, 2>(tiles, g, ks, nks, brow, cvt, acc);
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
      const float sx = x_scale(p, row_tok(p, row + col));
      const float G = (ts_g * sx) * v[i], U = (ts_u * sx) * v[4 + i];
      const float a = G / (1.0f + expf(-G)) * U;
      store_a(p, row + col, r, a);
    }
  }
}


// ---------------------------------------------------------------- NVFP4 gate/up through shared memory
// A CTA takes one tile pair over the whole K; warp w takes the 256-column
// units w, w + 8, ... of both tiles (per unit and tile: the scale vector and
// up to 4 code vectors, 2.5 KB) together with the entry's token rows over the
// same 256 columns.  The warp copies them into its own stage of shared memory
// with cp.async, so no registers wait on HBM: a CTA needs few of them,
// several CTAs share an SM, and a decode step has every weight byte requested
// at once.  Each warp starts its math as soon as its own copies have landed
// (no CTA-wide barrier before the K-split reduction).  For T <= 8 tokens:
// the staged token rows (f16, or bf16 converted on read for the shared
// expert's entries) sit in slot = token, so an entry may hold any number of
// rows (e.g. a token that picked one expert twice); rows are padded by 16
// bytes so that the B-fragment reads of 8 slots hit distinct banks.
constexpr int kNvUnitBytes = 2 * 5 * 512;
constexpr int kNvXStride = 256 + 8;  // halfs per staged token-row slice

__host__ __device__ __forceinline__ int gateup_nv_stages(int K) {
  return (K + 255) / 256 > kWarps ? 2 : 1;
}
__host__ __device__ __forceinline__ int gateup_nv_stage_bytes(int T) {
  return kNvUnitBytes + T * kNvXStride * 2;
}
__host__ __device__ __forceinline__ size_t gateup_nv_smem(int K, int T) {
  return (size_t)kWarps * gateup_nv_stages(K) * gateup_nv_stage_bytes(T);
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

// cp.async of unit hh of NT tiles (per tile: its scale vector and up to 4
// code vectors, 2560 bytes) into the stage at `dst`.
template <int NT>
__device__ __forceinline__ void nv_units_copy(const uint8_t* const* tile, const MatGeom& g, int hh,
                                              uint32_t dst) {
  const int lane = threadIdx.x & 31;
  const int s = hh >> 1, jb = (hh & 1) * 4;
  const int nc = min(4, sc_units(g, s) - jb);
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const uint8_t* b = tile[i] + (size_t)s * g.sc_bytes + 16 * lane;
    const uint32_t d = dst + i * 2560 + 16 * lane;
    cp_async16(d, b);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < nc) cp_async16(d + 512 * (1 + j), b + 512 * (1 + jb + j));
  }
}

// cp.async of unit hh (both tiles, and the token rows over its columns) into
// the stage at `dst`.  tok_of(r): token of row r of the entry.
template <typename TokOf>
__device__ __forceinline__ void nv_unit_copy(const uint8_t* const (&tile)[2], const MatGeom& g,
                                             int hh, uint32_t dst, const uint16_t* xsrc, int H,
                                             int n, int T, TokOf tok_of) {
  const int lane = threadIdx.x & 31;
  const int s = hh >> 1, jb = (hh & 1) * 4;
  const int nc = min(4, sc_units(g, s) - jb);
  nv_units_copy<2>(tile, g, hh, dst);
  const int pieces = nc * 8, col0 = 256 * hh;  // 16-byte pieces of a row slice
  for (int i = lane; i < n * pieces; i += 32) {
    const int r = i / pieces, c = i - r * pieces;
    const int tok = tok_of(r);
    if ((unsigned)tok < (unsigned)T)
      cp_async16(dst + kNvUnitBytes + 2 * (tok * kNvXStride + 8 * c),
                 xsrc + (size_t)tok * H + col0 + 8 * c);
  }
}

// Unit hh of NT tiles (staged at `st`) times this lane's staged token row
// (xrow: its shared-memory address at the unit's first column; has_x false:
// an empty column), into two accumulators per tile (even / odd chunks:
// shorter mma chains).
template <int NT>
__device__ __forceinline__ void nv_units_mma(const MatGeom& g, int hh, uint32_t st, uint32_t xrow,
                                             bool has_x, bool b_bf16, float (&acc)[NT][2][4]) {
  const int lane = threadIdx.x & 31, t = lane & 3;
  const int s = hh >> 1, jb = (hh & 1) * 4;
  const int nc = min(4, sc_units(g, s) - jb);
  uint4 sv[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) sv[i] = lds128(st + i * 2560 + 16 * lane);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j < nc) {
      const int jj = jb + j;
      uint32_t xb[8];
      if (has_x) {
        const uint32_t xa = xrow + 2 * (64 * j + 16 * t);
        const uint4 q0 = lds128(xa), q1 = lds128(xa + 16);
        xb[0] = q0.x; xb[1] = q0.y; xb[2] = q0.z; xb[3] = q0.w;
        xb[4] = q1.x; xb[5] = q1.y; xb[6] = q1.z; xb[7] = q1.w;
        if (b_bf16) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const __half2 h = __floats2half2_rn(__uint_as_float(xb[q] << 16),
                                                __uint_as_float(xb[q] & 0xFFFF0000u));
            xb[q] = *reinterpret_cast<const uint32_t*>(&h);
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) xb[q] = 0u;
      }
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const uint4 cv = lds128(st + i * 2560 + 512 * (1 + j) + 16 * lane);
        const uint32_t sp = e4m3x2_to_f16x2((u4get(sv[i], jj >> 1) >> (16 * (jj & 1))) & 0xFFFFu);
        const uint32_t s_lo = dup_lo(sp), s_hi = dup_hi(sp);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t h[4];
          e2m1x8_to_f16x8(u4get(cv, w), h);
          const uint32_t a[4] = {hmul2(h[0], s_lo), hmul2(h[1], s_hi), hmul2(h[2], s_lo),
                                 hmul2(h[3], s_hi)};
          mma_f16(acc[i][j & 1], a, xb[2 * w], xb[2 * w + 1]);
        }
      }
    }
  }
}

// Tile pair `pair` of `expert` for the n tokens of rows row..row+n-1, T <= 8.
// smem: gateup_nv_smem(H, T) bytes (16-byte aligned); red: kThreads x 8 floats.  prefetch_down: also ask L2 for this tile pair's share (1/(I/16)) of
// the expert's down matrix, for a down kernel that starts after this one.
__device__ __forceinline__ void gateup_task_nv(const ExpertParams& p, int expert, int row, int n,
                                               int pair, uint8_t* smem, float* red,
                                               bool prefetch_down) {
  const int S = p.T * p.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const MatGeom g = mat_geom(FMT_NVFP4, p.H);
  const int nh = n_halves(g), nst = gateup_nv_stages(p.H);
  const int sbytes = gateup_nv_stage_bytes(p.T);
  const uint8_t* eb = expert_base(p, expert);
  const uint8_t* const tiles[2] = {eb + (size_t)(2 * pair) * p.gu_tile_bytes,
                                   eb + (size_t)(2 * pair + 1) * p.gu_tile_bytes};
  const uint32_t wst = smem_u32(smem) + warp * nst * sbytes;
  const bool shared_entry = expert == p.E, cvt = convert_x(p, shared_entry);
  const uint16_t* xsrc = cvt ? p.x : p.xh;
  auto tok_of = [&](int r) { return shared_entry ? row - S + r : p.row_token[row + r]; };
  if (warp < nh) nv_unit_copy(tiles, g, warp, wst, xsrc, p.H, n, p.T, tok_of);
  cp_async_commit();
  if (nst > 1 && warp + kWarps < nh)
    nv_unit_copy(tiles, g, warp + kWarps, wst + sbytes, xsrc, p.H, n, p.T, tok_of);
  cp_async_commit();
  int xslot = -1;  // this lane's staged slot (B operand), or none
  if (gi < n) {
    const int tok = tok_of(gi);
    if ((unsigned)tok < (unsigned)p.T) xslot = tok;
  }
  float acc[2][2][4] = {};
  int u = 0;
  for (int hh = warp; hh < nh; hh += kWarps, ++u) {
    const uint32_t st = wst + (u & 1) * sbytes;
    cp_async_wait<1>();
    __syncwarp();  // the other lanes' token-row pieces of this stage
    nv_units_mma<2>(g, hh, st, st + kNvUnitBytes + 2 * (xslot > 0 ? xslot : 0) * kNvXStride,
                    xslot >= 0, cvt, acc);
    __syncwarp();  // every lane is done with the stage before it is refilled
    if (hh + 2 * kWarps < nh)
      nv_unit_copy(tiles, g, hh + 2 * kWarps, st, xsrc, p.H, n, p.T, tok_of);
    cp_async_commit();
  }
  cp_async_wait<0>();
  if (prefetch_down) {
    const size_t len = (size_t)(p.H / 16) * p.dn_tile_bytes;
    const size_t npairs = (size_t)(p.I / 16);
    const size_t b0 = len * pair / npairs, b1 = len * (pair + 1) / npairs;
    const uint8_t* dn = eb + p.gu_bytes;
    for (size_t o = (b0 & ~(size_t)127) + 128 * threadIdx.x; o < b1; o += 128 * kThreads)
      prefetch_l2(dn + o);
  }
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = acc[0][0][i] + acc[0][1][i];
    v[4 + i] = acc[1][0][i] + acc[1][1][i];
  }
  reduce_ksplit<8>(red, v, 1, kWarps);
  if (warp != 0) return;
  const float ts_g = p.tscale[expert * 3 + 0], ts_u = p.tscale[expert * 3 + 1];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 16 * pair + gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
    if (col < n) {
      const float sx = x_scale(p, row_tok(p, row + col));
      const float G = (ts_g * sx) * v[i], U = (ts_u * sx) * v[4 + i];
      const float a = G / (1.0f + expf(-G)) * U;
      store_a(p, row + col, r, a);
    }
  }
}

// ---------------------------------------------------------------- streamed expert GEMVs
// CTA = (work entry of up to 8 tokens, group of kWarps tile pairs for gate/up
// or kWarps tiles for down).  The entry's B rows (x for gate/up, a for down;
// f16) are staged once in shared memory over the whole K and shared by the 8
// warps.  Warp w streams its own tile pair (tile) over the whole K through a
// two-stage cp.async ring of 256-column units, so it always has the next unit
// in flight and owns its sums: no K-split reduction and no CTA barrier after
// the staging.  Staged rows are padded by 16 bytes (bank-conflict-free
// B-fragment reads of 8 rows).  NVFP4 (T > 8; decode keeps the tile-pair
// path) and FP6 (every T).
__host__ __device__ __forceinline__ int stream_xstride(int K) { return K + 8; }
// bytes of one tile's 256-column unit in a stage
__host__ __device__ __forceinline__ int stream_unit_bytes(int fmt) {
  return fmt == FMT_NVFP4 ? 2560 : 3200;
}
__host__ __device__ __forceinline__ int stream_rows(int T) { return T < kTokTile ? T : kTokTile; }
// ns: ring stages per warp (2 or 3)
__host__ __device__ __forceinline__ size_t stream_smem(int fmt, int nt, int K, int T, int ns) {
  return (size_t)stream_rows(T) * stream_xstride(K) * 2 +
         (size_t)kWarps * ns * nt * stream_unit_bytes(fmt);
}

// cp.async of FP6 unit hh of NT tiles (per tile: the super-chunk's 128-byte
// exponent vector and the code vectors of up to 2 blocks, 3200 bytes).
template <int NT>
__device__ __forceinline__ void fp6_units_copy(const uint8_t* const* tile, const MatGeom& g, int hh,
                                               uint32_t dst) {
  const int lane = threadIdx.x & 31;
  const int s = hh >> 2, j0 = (hh & 3) * 2, np = sc_units(g, s);
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const uint8_t* b = tile[i] + (size_t)s * g.sc_bytes;
    const uint32_t d = dst + i * 3200;
    if (lane < 8) cp_async16(d + 16 * lane, b + 16 * lane);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
      if (j0 + jj < np)
#pragma unroll
        for (int v = 0; v < 3; ++v)
          cp_async16(d + 128 + 1536 * jj + 512 * v + 16 * lane,
                     b + 128 + 1536 * (j0 + jj) + 512 * v + 16 * lane);
  }
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// FP6 unit hh of NT tiles (staged at `st`) times this lane's B row: per
// 128-column block an fp32 block sum, times the block's power-of-two scale,
// into acc[i][block parity].  ldx(col, xb): this lane's 16 f16 B values at
// column `col` of the unit (its 16-column block of the m16n8k16 k-permutation).
template <int NT, typename LdX>
__device__ __forceinline__ void fp6_units_mma(const MatGeom& g, int hh, uint32_t st, LdX ldx,
                                              float (&acc)[NT][2][4]) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int s = hh >> 2, j0 = (hh & 3) * 2, np = sc_units(g, s);
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    if (j0 + jj < np) {
      const int j = j0 + jj;
      uint32_t xb[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h) ldx(128 * jj + 64 * h + 16 * t, xb[h]);
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const uint32_t tb = st + i * 3200;
        const uint4 c0 = lds128(tb + 128 + 1536 * jj + 16 * lane);
        const uint4 c1 = lds128(tb + 128 + 1536 * jj + 512 + 16 * lane);
        const uint4 c2 = lds128(tb + 128 + 1536 * jj + 1024 + 16 * lane);
        const uint32_t words[12] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y,
                                    c1.z, c1.w, c2.x, c2.y, c2.z, c2.w};
        float blk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
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
              mma_f16(blk, a, xb[h][2 * w], xb[h][2 * w + 1]);
            }
          }
        }
        // exponent bytes of rows g and g+8 for block j (the layout of tiles_fp6)
        const uint32_t e = lds32(tb + 4 * ((gi << 2) | (j >> 1)));
        const float f0 = ue8m0_to_f32((e >> (16 * (j & 1))) & 0xFFu);
        const float f1 = ue8m0_to_f32((e >> (16 * (j & 1) + 8)) & 0xFFu);
        acc[i][jj][0] = fmaf(blk[0], f0, acc[i][jj][0]);
        acc[i][jj][1] = fmaf(blk[1], f0, acc[i][jj][1]);
        acc[i][jj][2] = fmaf(blk[2], f1, acc[i][jj][2]);
        acc[i][jj][3] = fmaf(blk[3], f1, acc[i][jj][3]);
      }
    }
  }
}

// MODE 0: gate/up + SwiGLU of tile pair group*kWarps + w into abuf; MODE 1:
// down tiles 2i and 2i + 1 (i = group*kWarps + w) into ybuf, the two tiles
// sharing the warp's B fragments like a gate/up pair.  NS ring stages per
// warp.  smem: stream_smem bytes (nt = 2).
template <int FMT, int MODE, int NS = 2>
__device__ __forceinline__ void stream_task(const ExpertParams& p, int expert, int row, int n,
                                            int group, uint8_t* smem) {
  constexpr int NT = 2;
  constexpr int SB = FMT == FMT_NVFP4 ? 2560 : 3200;  // stream_unit_bytes
  const int S = p.T * p.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int K = MODE == 0 ? p.H : p.I;
  const MatGeom g = mat_geom(FMT, K);
  const int nh = n_halves(g), xs = stream_xstride(K);
  const int idx = group * kWarps + warp;  // tile pair (gate/up) or pair of down tiles
  const bool valid = idx < (MODE == 0 ? p.I / 16 : p.H / 32);
  const uint8_t* eb = expert_base(p, expert);
  const uint8_t* tiles[2];
  if (MODE == 0) {
    tiles[0] = eb + (size_t)(2 * idx) * p.gu_tile_bytes;
    tiles[1] = eb + (size_t)(2 * idx + 1) * p.gu_tile_bytes;
  } else {
    tiles[0] = eb + p.gu_bytes + (size_t)(2 * idx) * p.dn_tile_bytes;
    tiles[1] = eb + p.gu_bytes + (size_t)(2 * idx + 1) * p.dn_tile_bytes;
  }
  auto copy_unit = [&](int hh, uint32_t dst) {
    if (FMT == FMT_NVFP4)
      nv_units_copy<NT>(tiles, g, hh, dst);
    else
      fp6_units_copy<NT>(tiles, g, hh, dst);
  };
  const uint32_t xs_base = smem_u32(smem);
  const uint32_t st_base = xs_base + stream_rows(p.T) * xs * 2 + warp * NS * NT * SB;
  // The B rows first (one cp.async group), then the warp's first NS units.
  // Gate/up rows are tokens; with T <= 8 a row sits in slot = its token (an
  // entry may hold one token twice, e.g. from a given routing), else in slot
  // = its row of the entry (n <= 8).  Down rows are rows of a, in slot = row;
  // with T <= 8 (FP6 only) an entry of more rows than slots (a token that
  // picked one expert twice) reads a from global memory instead.
  const bool shared_entry = MODE == 0 && expert == p.E;
  const bool by_token = MODE == 0 && p.T <= kTokTile;
  const bool b_global = MODE == 1 && n > stream_rows(p.T);
  auto tok_of = [&](int r) { return shared_entry ? row - S + r : p.row_token[row + r]; };
  const int pieces = K / 8;  // 16-byte pieces of a row
  for (int i = threadIdx.x; i < (b_global ? 0 : n) * pieces; i += kThreads) {
    const int r = i / pieces, c = i - r * pieces;
    const int tok = MODE == 0 ? tok_of(r) : 0;
    if (MODE == 0 && (unsigned)tok >= (unsigned)p.T) continue;
    const uint32_t dst = xs_base + 2 * ((by_token ? tok : r) * xs + 8 * c);
    if (MODE == 1) {
      cp_async16(dst, p.abuf + (size_t)(row + r) * p.I + 8 * c);
    } else if (!convert_x(p, shared_entry)) {
      cp_async16(dst, p.xh + (size_t)tok * p.H + 8 * c);
    } else {  // the shared expert's entries run ahead of the router: convert x here
      const uint4 q = *reinterpret_cast<const uint4*>(p.x + (size_t)tok * p.H + 8 * c);
      uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w[k2] << 16),
                                            __uint_as_float(w[k2] & 0xFFFF0000u));
        w[k2] = *reinterpret_cast<const uint32_t*>(&h);
      }
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(w[0]), "r"(w[1]),
                   "r"(w[2]), "r"(w[3])
                   : "memory");
    }
  }
  cp_async_commit();
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    if (valid && u < nh) copy_unit(u, st_base + u * NT * SB);
    cp_async_commit();
  }
  cp_async_wait<NS>();  // this thread's B-row pieces
  __syncthreads();      // everyone's
  float acc[NT][2][4] = {};
  if (valid) {
    int slot = gi < n ? gi : -1;  // this lane's staged row (B column), or none
    if (MODE == 0 && gi < n) {
      const int tok = tok_of(gi);
      slot = (unsigned)tok >= (unsigned)p.T ? -1 : (by_token ? tok : gi);
    }
    const uint32_t xrow = xs_base + 2 * (slot > 0 ? slot : 0) * xs;
    for (int hh = 0; hh < nh; ++hh) {
      const uint32_t st = st_base + (hh % NS) * NT * SB;
      cp_async_wait<NS - 1>();
      __syncwarp();  // the other lanes' pieces of this stage
      if (FMT == FMT_NVFP4)
        nv_units_mma<NT>(g, hh, st, xrow + 2 * 256 * hh, slot >= 0, false, acc);
      else
        fp6_units_mma<NT>(g, hh, st, [&](int col, uint32_t(&xb)[8]) {
          if (b_global) {
            load_b(gi < n ? p.abuf + (size_t)(row + gi) * p.I : nullptr, 256 * hh + col, false, xb);
          } else if (slot >= 0) {
            const uint32_t xa = xrow + 2 * (256 * hh + col);
            const uint4 q0 = lds128(xa), q1 = lds128(xa + 16);
            xb[0] = q0.x; xb[1] = q0.y; xb[2] = q0.z; xb[3] = q0.w;
            xb[4] = q1.x; xb[5] = q1.y; xb[6] = q1.z; xb[7] = q1.w;
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) xb[q] = 0u;
          }
        }, acc);
      __syncwarp();  // every lane is done with the stage before it is refilled
      if (hh + NS < nh) copy_unit(hh + NS, st);
      cp_async_commit();
    }
  }
  cp_async_wait<0>();
  if (!valid) return;
  if (MODE == 0) {
    const float ts_g = p.tscale[expert * 3 + 0], ts_u = p.tscale[expert * 3 + 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 16 * idx + gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
      if (col < n) {
        const float sx = x_scale(p, row_tok(p, row + col));
        const float G = (ts_g * sx) * (acc[0][0][i] + acc[0][1][i]);
        const float U = (ts_u * sx) * (acc[NT - 1][0][i] + acc[NT - 1][1][i]);
        const float a = G / (1.0f + expf(-G)) * U;
        store_a(p, row + col, r, a);
      }
    }
  } else {
    const float ts = p.tscale[expert * 3 + 2];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 16 * (2 * idx + q) + gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
        if (col < n)
          p.ybuf[(size_t)(row + col) * p.H + r] = (ts * a_scale(p, row + col)) * (acc[q][0][i] + acc[q][1][i]);
      }
  }
}

// Requests from L2 the down tile `tile` of every work entry (fire and forget).
template <int FMT>
__device__ __forceinline__ void down_prefetch(const ExpertParams& p, int tile) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const MatGeom g = mat_geom(FMT, p.I);
  const int n_entries = p.nsh + *p.n_entries;
  const size_t tile_off = p.gu_bytes + (size_t)tile * p.dn_tile_bytes;
  for (int y = warp; y < n_entries; y += nw) {
    const int expert = (y < p.nsh) ? p.E : p.entries[y - p.nsh].x;
    if (expert >= 0 && expert <= p.E)
      prefetch_tile(FMT, expert_base(p, expert) + tile_off, g, 0, 1);
  }
}

// The down tile of one work entry, loaded into registers before the kernel
// waits for gate/up: the weights do not depend on it (NVFP4, K <= 512: one
// super-chunk of at most 8 chunks).
struct DownPreload {
  int expert, row, n;
  float ts;
  uint4 sv, cv[8];
};

__device__ __forceinline__ bool down_preload(const ExpertParams& p, int tile, int y, DownPreload& d,
                                             bool quiet = false) {
  const int lane = threadIdx.x & 31;
  if (!get_entry(p, y, d.expert, d.row, d.n, quiet)) return false;  // (reads the count and the entry together)
  const uint8_t* b = expert_base(p, d.expert) + p.gu_bytes +
                     (size_t)tile * p.dn_tile_bytes + 16 * lane;
  const int nc = p.I / 64;
  d.sv = ldg_stream(b);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < nc) d.cv[j] = ldg_stream(b + 512 * (1 + j));
  d.ts = p.tscale[d.expert * 3 + 2];
  return true;
}

// The preloaded tile times the entry's rows of a (which gate/up wrote).
__device__ __forceinline__ void down_preloaded_mma(const ExpertParams& p, const DownPreload& d,
                                                   float (&acc)[4]) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int nc = p.I / 64;
  const uint16_t* brow = gi < d.n ? p.abuf + (size_t)(d.row + gi) * p.I : nullptr;
  float acc2[2][4] = {};  // even / odd chunks: two shorter mma chains
#pragma unroll
  for (int j0 = 0; j0 < 8; j0 += 4) {
    uint32_t xb[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j0 + j < nc) load_b(brow, 64 * (j0 + j) + 16 * t, false, xb[j]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int jj = j0 + j;
      if (jj < nc) {
        const uint32_t sp = e4m3x2_to_f16x2((u4get(d.sv, jj >> 1) >> (16 * (jj & 1))) & 0xFFFFu);
        const uint32_t s_lo = dup_lo(sp), s_hi = dup_hi(sp);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t h[4];
          e2m1x8_to_f16x8(u4get(d.cv[jj], w), h);
          const uint32_t a[4] = {hmul2(h[0], s_lo), hmul2(h[1], s_hi), hmul2(h[2], s_lo),
                                 hmul2(h[3], s_hi)};
          mma_f16(acc2[jj & 1], a, xb[j][2 * w], xb[j][2 * w + 1]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] += acc2[0][i] + acc2[1][i];
}

// y of tile `tile` (16 rows of H) for every work entry, one warp per entry,
// into ys [rows x 16] (shared memory), then out[:, tile] = sum_j g_j y_j + y_s
// in j order (the same fmaf chain as combine_kernel).  `pre`: the warp's first
// entry, preloaded (when have_pre).
// FP6: `ring` is a shared-memory ring of 2 stages of kDcFp6Stage bytes per
// warp; NVFP4 with I > 512: kDcNvStages stages of kDcNvStage bytes.
constexpr int kDcFp6Stage = 3200 + 512;  // a unit's weights and one row of a over its columns
constexpr int kDcNvStages = 4;
constexpr int kDcNvStage = 2560 + 512;
template <int FMT, bool LONGK = false>
__device__ __forceinline__ void down_combine_task(const ExpertParams& p, int tile, const float* gates,
                                                  const int* inv, float* out, float* ys,
                                                  uint32_t ring, const DownPreload& pre,
                                                  bool have_pre) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int gi = lane >> 2, t = lane & 3;
  const int S = p.T * p.k;
  const MatGeom g = mat_geom(FMT, p.I);
  const int n_entries = p.nsh + *p.n_entries;
  const size_t tile_off = p.gu_bytes + (size_t)tile * p.dn_tile_bytes;
  for (int y = warp; y < n_entries; y += nw) {
    if (have_pre && y == warp) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      down_preloaded_mma(p, pre, acc);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
        if (col < pre.n) ys[(pre.row + col) * 16 + r] = (pre.ts * a_scale(p, pre.row + col)) * acc[i];
      }
      continue;
    }
    int expert, row, n;
    if (!get_entry(p, y, expert, row, n)) continue;
    const uint8_t* const tiles[1] = {expert_base(p, expert) + tile_off};
    const uint16_t* brow = gi < n ? p.abuf + (size_t)(row + gi) * p.I : nullptr;
    float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    if (FMT == FMT_FP6) {
      // The tile's units through this warp's two-stage cp.async ring (`ring`,
      // kDcFp6Stage bytes a stage).  A one-row entry (every entry of a
      // self-routed token) copies its row of a over the unit's columns into
      // the same stage; other entries read a from global memory.
      const bool b_smem = n == 1;
      const uint16_t* arow = p.abuf + (size_t)row * p.I;
      const int nh = n_halves(g);
      const uint32_t wr = ring + warp * 2 * kDcFp6Stage;
      auto copy_unit = [&](int hh, uint32_t dst) {
        fp6_units_copy<1>(tiles, g, hh, dst);
        if (b_smem && 256 * hh + 8 * lane < p.I)
          cp_async16(dst + 3200 + 16 * lane, arow + 256 * hh + 8 * lane);
      };
      copy_unit(0, wr);
      cp_async_commit();
      if (nh > 1) copy_unit(1, wr + kDcFp6Stage);
      cp_async_commit();
      float a2[1][2][4] = {};
      for (int hh = 0; hh < nh; ++hh) {
        const uint32_t st = wr + (hh & 1) * kDcFp6Stage;
        cp_async_wait<1>();
        __syncwarp();
        fp6_units_mma<1>(g, hh, st, [&](int col, uint32_t(&xb)[8]) {
          if (!b_smem) {
            load_b(brow, 256 * hh + col, false, xb);
          } else if (gi == 0) {
            const uint4 q0 = lds128(st + 3200 + 2 * col), q1 = lds128(st + 3200 + 2 * col + 16);
            xb[0] = q0.x; xb[1] = q0.y; xb[2] = q0.z; xb[3] = q0.w;
            xb[4] = q1.x; xb[5] = q1.y; xb[6] = q1.z; xb[7] = q1.w;
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) xb[q] = 0u;
          }
        }, a2);
        __syncwarp();
        if (hh + 2 < nh) copy_unit(hh + 2, st);
        cp_async_commit();
      }
      cp_async_wait<0>();
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[0][i] = a2[0][0][i] + a2[0][1][i];
    } else if (LONGK && n == 1) {
      // NVFP4 with a long K (the fused decode down of wide experts), one row:
      // the tile's units and the row of a through this warp's kDcNvStages-
      // stage cp.async ring, several units in flight instead of one at a time
      const uint16_t* arow = p.abuf + (size_t)row * p.I;
      const int nh = n_halves(g);
      const uint32_t wr = ring + warp * kDcNvStages * kDcNvStage;
      auto copy_unit = [&](int hh, uint32_t dst) {
        nv_units_copy<1>(tiles, g, hh, dst);
        if (256 * hh + 8 * lane < p.I) cp_async16(dst + 2560 + 16 * lane, arow + 256 * hh + 8 * lane);
      };
#pragma unroll
      for (int u = 0; u < kDcNvStages; ++u) {
        if (u < nh) copy_unit(u, wr + u * kDcNvStage);
        cp_async_commit();
      }
      float a2[1][2][4] = {};
      for (int hh = 0; hh < nh; ++hh) {
        const uint32_t st = wr + (hh % kDcNvStages) * kDcNvStage;
        cp_async_wait<kDcNvStages - 1>();
        __syncwarp();
        nv_units_mma<1>(g, hh, st, st + 2560, gi == 0, false, a2);
        __syncwarp();
        if (hh + kDcNvStages < nh) copy_unit(hh + kDcNvStages, st);
        cp_async_commit();
      }
      cp_async_wait<0>();
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[0][i] = a2[0][0][i] + a2[0][1][i];
    } else {
      tiles_mma<FMT, 1>(tiles, g, 0, 1, brow, false, acc);
    }
    const float ts = p.tscale[expert * 3 + 2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
      if (col < n) ys[(row + col) * 16 + r] = (ts * a_scale(p, row + col)) * acc[0][i];
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
}

}  // namespace
}  // namespace moe
