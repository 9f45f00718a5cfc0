// Small-batch expert path (work entries of up to 8 tokens): the packed expert
// weights stream from HBM through a shared-memory ring of bulk async copies.
//
// A launch is one CTA per SM over a list of work items.  An item is one work
// entry (an expert and up to eight of its token rows) times one weight group:
// a gate/up tile pair (16 rows of W_gate and the same 16 rows of W_up), or one
// 16-row tile of W_down.  A producer warp copies each item stage by stage into
// the ring with cp.async.bulk, the bytes counted on the stage's mbarrier; a
// stage is a run of units (NVFP4: 64-column chunks, FP6: 128-column pairs) of
// one super-chunk of every tile of the group, with its scale vector, plus the
// same columns of the item's activation rows.  The eight consumer warps take
// the stage's (tile, unit) pairs round-robin, dequantise them in registers
// into m16n8k16 A fragments (the layout of layout.cuh) and accumulate in fp32.
// At the end of an item the eight partial sums are added in warp order
// (deterministic, and independent of the other tokens of the entry) and one
// warp applies the epilogue: SwiGLU into a (gate/up), y (down), or y into
// shared memory for the gate-weighted combine of a few tokens.  The producer
// keeps the whole ring in flight whatever the arithmetic is doing, which is
// what streaming weight bytes at HBM bandwidth needs: 16-byte per-thread loads
// left too few bytes in flight per SM (the "Strata on an Intel Arc" pages
// found the same for their decode matvecs: "The engine itself on Intel",
// "Planned", item 5).
//
// Decode variants (T <= 8) route in every CTA from the router's partial sums
// (route_small_cta): no routing kernel and no hand-off of work entries through
// global memory sits between the router and the experts.  The shared
// expert's items need no routing and are streamed while the router is still
// running; the down kernel routes and issues its weight copies while gate/up
// is still running, so after gate/up only the activations' arrival, the
// arithmetic and the combine remain.
//
// Every wait is bounded: on a timeout the kernel records MOE_ETIMEOUT in the
// status word, stops issuing, drains the copies it issued and returns.
#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"
#include "layout.cuh"
#include "route_dev.cuh"

namespace moe {
namespace {

constexpr int kSW = 8;                     // consumer warps
constexpr int kSThreads = (kSW + 1) * 32;  // + the producer warp
constexpr int kSMaxStages = 16;

// ue8m0 byte b -> 2^(b - 127); b = 0 gives the subnormal 2^-127
__device__ __forceinline__ float ue8m0_to_f32(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// Byte containers of 4 FP6 codes each from the 4+2 bit planes of the layout
// (high nibbles in Ha / Hb, low 2 bits in L; layout.cuh)
__device__ __forceinline__ void fp6_unpack(uint32_t Ha, uint32_t Hb, uint32_t L, uint32_t (&c)[4]) {
  c[0] = ((Ha << 2) & 0x3C3C3C3Cu) | (L & 0x03030303u);
  c[1] = ((Ha >> 2) & 0x3C3C3C3Cu) | ((L >> 2) & 0x03030303u);
  c[2] = ((Hb << 2) & 0x3C3C3C3Cu) | ((L >> 4) & 0x03030303u);
  c[3] = ((Hb >> 2) & 0x3C3C3C3Cu) | ((L >> 6) & 0x03030303u);
}

// header of a ring stage, written by the producer before it arms the stage
enum : int { ST_LAST = 1, ST_BF16 = 2, ST_TILE_END = 4, ST_END = 8, ST_SHARED = 16 };
struct StageHdr {
  int row;         // first row (of a / y) of the item's entry
  int n;           // token rows
  int tile;        // gate/up: tile pair; down: 16-row tile of H
  int flags;
  int mask;        // tiles of the group in the stage (bit t: tile t)
  int sa, sb;      // super-chunks [sa, sb) of each of those tiles
  int part;        // bytes of one tile's part of the stage
  float ts0, ts1;  // fp32 tensor scales: gate and up, or down
};

struct StreamShared {
  uint64_t full[kSMaxStages];
  uint64_t empty[kSMaxStages];
  uint64_t cons;   // barrier of the eight consumer warps (bounded waits, unlike bar.sync)
  uint64_t red_full[2];  // an item's eight partial sums are in its slot (count 8)
  uint64_t red_free[2];  // the owner has read them (count 1)
  uint64_t bonce;  // the activation rows staged once per CTA have landed
  uint64_t tsbar;  // the tensor-scale table has landed
  StageHdr hdr[kSMaxStages];
  int abort;
};

// One work item as the producer issues it.
struct ItemDesc {
  const uint8_t* tile0;  // first tile of the group
  int expert, row, n, tile, flags;
  float ts0, ts1;
  int tok[kTokTile];     // gate/up, activations per stage: token of each row
};

// Work entries in shared memory (routed in this CTA) or in global memory
// (written by the dispatch kernel, read through L2), after the leading
// shared-expert entries, which follow from T.
struct Entries {
  const int4* e;   // routed entries
  const int* tok;  // token of each routed row
  int n;           // routed entries
  int nsh;         // leading shared-expert entries
  bool global;
};

// MODE 0: item (y, tile pair) of gate/up; MODE 1: item (y, 16-row tile of H) of down.
template <int MODE>
__device__ __forceinline__ ItemDesc describe(const ExpertParams& p, const Entries& en, const float* sts, int y,
                                             int tile) {
  ItemDesc d;
  const int S = p.T * p.k;
  d.tile = tile;
  d.flags = 0;
  if (y < en.nsh) {
    d.expert = p.E;
    d.row = S + kTokTile * y;
    d.n = min(kTokTile, p.T - kTokTile * y);
    d.flags = ST_SHARED | (MODE == 0 ? ST_BF16 : 0);  // the shared expert's rows: x itself
  } else {
    const int4 e = en.global ? __ldcg(en.e + (y - en.nsh)) : en.e[y - en.nsh];
    d.expert = e.x;
    d.row = e.y;
    d.n = e.z;
    if (d.expert < 0 || d.expert >= p.E || d.n < 1 || d.n > kTokTile || d.row < 0 || d.row + d.n > S) {
      *p.status = -1;  // MOE_EINVAL: corrupt entry, skipped
      d.expert = 0;
      d.n = 0;
      d.row = 0;
    }
  }
  const uint8_t* eb = p.arena + (size_t)d.expert * p.expert_bytes;
  if (MODE == 0) {
    d.tile0 = eb + (size_t)(2 * tile) * p.gu_tile_bytes;
    d.ts0 = sts[d.expert * 3 + 0];
    d.ts1 = sts[d.expert * 3 + 1];
#pragma unroll
    for (int r = 0; r < kTokTile; ++r)
      d.tok[r] = (y >= en.nsh && r < d.n) ? (en.global ? __ldcg(en.tok + d.row + r) : en.tok[d.row + r]) : 0;
  } else {
    d.tile0 = eb + p.gu_bytes + (size_t)tile * p.dn_tile_bytes;
    d.ts0 = sts[d.expert * 3 + 2];
    d.ts1 = 0.f;
  }
  return d;
}

// bytes of super-chunks [a, b) of one tile (only the last super-chunk can be short)
__device__ __forceinline__ int run_bytes(const StreamGeom& g, int a, int b) {
  if (b < g.nsc) return (b - a) * g.sc_bytes;
  return (b - 1 - a) * g.sc_bytes + g.hdr_bytes + (g.units - 8 * (g.nsc - 1)) * g.unit_bytes;
}

// ---------------------------------------------------------------- producer
// One lane issues every copy.  Stages are taken in order; stage q waits until
// the consumers have released its previous use.  Each stage is one contiguous
// copy of weights (a whole gate/up tile pair, or a run of super-chunks of one
// tile): small copies are slow, a streaming multiprocessor keeps only a few
// bulk copies in flight.
struct Producer {
  const ExpertParams& p;
  const StreamGeom& g;
  StreamShared& sh;
  uint8_t* ring;
  uint64_t pol;
  int q;  // stages issued
  bool ok;
  bool bonce_armed;  // the staged-once activations were requested by this producer
  const float* sts;  // the fp32 tensor scales, staged in shared memory

  __device__ __forceinline__ Producer(const ExpertParams& p_, const StreamGeom& g_, StreamShared& sh_,
                                      uint8_t* ring_, int q_)
      : p(p_), g(g_), sh(sh_), ring(ring_), pol(l2_evict_first()), q(q_), ok(true), bonce_armed(false),
        sts(reinterpret_cast<const float*>(ring_ + (size_t)g_.n_stages * g_.stage_bytes + g_.b_bytes)) {}

  // the tensor-scale table into shared memory (lane 0, at the start)
  __device__ __forceinline__ void stage_ts() {
    mbar_arrive_expect(&sh.tsbar, (uint32_t)g.ts_bytes);
    bulk_g2s(const_cast<float*>(sts), p.tscale, (uint32_t)g.ts_bytes, &sh.tsbar);
  }

  // one copy of `bytes` activation bytes into the staged-once area
  __device__ __forceinline__ void stage_once(uint8_t* dst, const void* src, uint32_t bytes) {
    mbar_arrive_expect(&sh.bonce, bytes);
    bulk_g2s(dst, src, bytes, &sh.bonce);
    bonce_armed = true;
  }

  __device__ __forceinline__ uint8_t* stage_ptr(int st) const { return ring + (size_t)st * g.stage_bytes; }

  __device__ __forceinline__ bool take(int& st) {
    st = q % g.n_stages;
    if (!mbar_wait(&sh.empty[st], ((q / g.n_stages) & 1) ^ 1, &sh.abort)) {
      ok = false;
      return false;
    }
    return true;
  }

  // Activation columns of a stage (per-stage mode): x or the f16 copy of x
  // for gate/up (by token), a for down (by row); one copy per row.
  template <int MODE>
  __device__ __forceinline__ void copy_b(const ItemDesc& d, const StageHdr& h, int st) {
    const int c0 = h.sa * 8 * g.unit_cols, c1 = min(g.K, h.sb * 8 * g.unit_cols);
    const uint32_t bb = (uint32_t)(c1 - c0) * 2u;
    uint8_t* dst = stage_ptr(st) + g.w_cap;
    const int S = p.T * p.k;
#pragma unroll
    for (int r = 0; r < kTokTile; ++r) {  // unrolled: d.tok stays in registers
      if (r >= h.n) break;
      const uint16_t* src;
      if (MODE != 0)
        src = p.abuf + (size_t)(h.row + r) * p.I;
      else if (h.flags & ST_SHARED)
        src = p.x + (size_t)(h.row - S + r) * p.H;
      else
        src = p.xh + (size_t)d.tok[r] * p.H;
      bulk_g2s(dst + r * g.b_stride, src + c0, bb, &sh.full[st]);
    }
  }

  __device__ __forceinline__ bool stage(const ItemDesc& d, int mask, int sa, int sb, bool last,
                                        const uint8_t* src, int part, int nparts, bool with_b,
                                        int mode) {
    int st;
    if (!take(st)) return false;
    StageHdr h;
    h.row = d.row;
    h.n = d.n;
    h.tile = d.tile;
    h.flags = d.flags | (last ? ST_LAST : 0);
    h.mask = mask;
    h.sa = sa;
    h.sb = sb;
    h.part = part;
    h.ts0 = d.ts0;
    h.ts1 = d.ts1;
    sh.hdr[st] = h;
    uint32_t bytes = (uint32_t)(part * nparts);
    if (with_b)
      bytes += (uint32_t)(d.n * (min(g.K, sb * 8 * g.unit_cols) - sa * 8 * g.unit_cols) * 2);
    mbar_arrive_expect(&sh.full[st], bytes);
    bulk_g2s_hint(stage_ptr(st), src, (uint32_t)(part * nparts), &sh.full[st], pol);
    if (with_b) {
      if (mode == 0)
        copy_b<0>(d, h, st);
      else
        copy_b<1>(d, h, st);
    }
    ++q;
    return true;
  }

  // The stages of one item.
  template <int MODE>
  __device__ __forceinline__ void item(const ItemDesc& d) {
    const bool with_b = !g.b_once;
    if (g.pair_stage) {  // both tiles, every super-chunk: one copy
      stage(d, 3, 0, g.nsc, true, d.tile0, g.tile_bytes, 2, with_b, MODE);
      return;
    }
    for (int t = 0; t < g.tiles && ok; ++t)
      for (int a = 0; a < g.nsc && ok; a += g.sc_run) {
        const int b = min(g.nsc, a + g.sc_run);
        stage(d, 1 << t, a, b, t == g.tiles - 1 && b == g.nsc,
              d.tile0 + (size_t)t * g.tile_bytes + (size_t)a * g.sc_bytes, run_bytes(g, a, b), 1,
              with_b, MODE);
      }
  }

  // a stage that carries no data and tells the consumers to leave their loop
  __device__ __forceinline__ void end_marker() {
    int st;
    if (!take(st)) return;
    StageHdr h{};
    h.flags = ST_END;
    sh.hdr[st] = h;
    mbar_arrive(&sh.full[st]);
    ++q;
  }

  // before exit after a timeout: wait (bounded) for the copies still landing
  __device__ __forceinline__ void drain() {
    const int n = min(q, g.n_stages);
    for (int i = 1; i <= n; ++i) {
      const int qq = q - i, st = qq % g.n_stages;
      mbar_drain(&sh.full[st], (qq / g.n_stages) & 1);
    }
    if (bonce_armed) mbar_drain(&sh.bonce, 0);
    mbar_drain(&sh.tsbar, 0);
  }
};

// ---------------------------------------------------------------- consumers
// 16 activations (f16, or bf16 converted to f16) at column `col` of an
// activation row in shared memory, or zeros (no row).
__device__ __forceinline__ void b_frag(const uint8_t* brow, int col, bool bf16, uint32_t (&xw)[8]) {
  if (brow) {
    const uint4* px = reinterpret_cast<const uint4*>(brow + 2 * col);
    const uint4 q0 = px[0], q1 = px[1];
    xw[0] = q0.x; xw[1] = q0.y; xw[2] = q0.z; xw[3] = q0.w;
    xw[4] = q1.x; xw[5] = q1.y; xw[6] = q1.z; xw[7] = q1.w;
    if (bf16) {
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

// NVFP4 unit j of the super-chunk at `sc` (64 columns from column c0 + 64 j,
// one e4m3 scale per 16 columns and row).  The four 16-column steps go to
// four accumulators: independent MMAs instead of one dependent chain.
__device__ __forceinline__ void unit_nvfp4(const uint8_t* sc, int j, const uint8_t* brow, int c0, bool bf16,
                                           float (&acc)[4][4]) {
  const int lane = threadIdx.x & 31, t = lane & 3;
  // the lane's two scale bytes of chunk j (rows g, g + 8): one 4-byte read
  const uint32_t sw = *reinterpret_cast<const uint32_t*>(sc + 16 * lane + 4 * (j >> 1));
  const uint4 cv = *reinterpret_cast<const uint4*>(sc + 512 * (1 + j) + 16 * lane);
  uint32_t xb[8];
  b_frag(brow, c0 + 64 * j + 16 * t, bf16, xb);
  const uint32_t sp = e4m3x2_to_f16x2((sw >> (16 * (j & 1))) & 0xFFFFu);
  const uint32_t s_lo = dup_lo(sp), s_hi = dup_hi(sp);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4];
    e2m1x8_to_f16x8(u4get(cv, q), h);
    const uint32_t a[4] = {hmul2(h[0], s_lo), hmul2(h[1], s_hi), hmul2(h[2], s_lo), hmul2(h[3], s_hi)};
    mma_f16(acc[q], a, xb[2 * q], xb[2 * q + 1]);
  }
}

// FP6 unit j of the super-chunk at `sc`: a pair of 64-column chunks from
// column c0 + 128 j, one power-of-two scale per 128 columns and row.  All
// lanes take part (shuffle).
__device__ __forceinline__ void unit_fp6(const uint8_t* sc, int j, const uint8_t* brow, int c0, bool bf16,
                                         float (&acc)[4][4]) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const uint32_t ew = *reinterpret_cast<const uint32_t*>(sc + 4 * lane);
  uint4 cv[3];
#pragma unroll
  for (int v = 0; v < 3; ++v) cv[v] = *reinterpret_cast<const uint4*>(sc + 128 + 1536 * j + 512 * v + 16 * lane);
  const uint32_t words[12] = {cv[0].x, cv[0].y, cv[0].z, cv[0].w, cv[1].x, cv[1].y,
                              cv[1].z, cv[1].w, cv[2].x, cv[2].y, cv[2].z, cv[2].w};
  float blk[4][4];  // per 16-column step: independent MMAs
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int r = 0; r < 4; ++r) blk[q][r] = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t xb[8];
    b_frag(brow, c0 + 128 * j + 64 * h + 16 * t, bf16, xb);
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      uint32_t c[4];
      fp6_unpack(words[h * 6 + qq * 3], words[h * 6 + qq * 3 + 1], words[h * 6 + qq * 3 + 2], c);
#pragma unroll
      for (int ww = 0; ww < 2; ++ww) {
        const int step = 2 * qq + ww;
        uint32_t uu[2], vv[2];
        e2m3x4_to_f16x4(c[2 * ww], uu);
        e2m3x4_to_f16x4(c[2 * ww + 1], vv);
        const uint32_t a[4] = {uu[0], uu[1], vv[0], vv[1]};
        mma_f16(blk[step], a, xb[2 * step], xb[2 * step + 1]);
      }
    }
  }
  const uint32_t e = __shfl_sync(0xffffffffu, ew, (gi << 2) | (j >> 1));
  const float f0 = ue8m0_to_f32((e >> (16 * (j & 1))) & 0xFFu);
  const float f1 = ue8m0_to_f32((e >> (16 * (j & 1) + 8)) & 0xFFu);
  // the pair's sum (steps in order), scaled by its power of two
  float b[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) b[r] = ((blk[0][r] + blk[1][r]) + blk[2][r]) + blk[3][r];
  acc[0][0] = fmaf(b[0], f0, acc[0][0]);
  acc[0][1] = fmaf(b[1], f0, acc[0][1]);
  acc[0][2] = fmaf(b[2], f1, acc[0][2]);
  acc[0][3] = fmaf(b[3], f1, acc[0][3]);
}

// Bounded wait of a whole warp: lane 0 polls, then every lane acquires the
// completed phase itself (one try_wait each).  Returns false on timeout.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) ok = mbar_wait(bar, parity, abort);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_test(bar, parity);
  return ok != 0;
}

// State of a consumer warp across stages and items.
struct Consumer {
  int q;      // stages consumed
  int items;  // items finished
  int syncs;  // consumer barriers passed
  float acc[2][4][4];  // [tile][16-column step or pair slot][m16n8 fragment]
};

// Barrier of the eight consumer warps on an mbarrier (count 8), so that a warp
// that gave up after a timeout cannot leave the others waiting for ever.
__device__ __forceinline__ bool consumer_sync(StreamShared& sh, Consumer& c) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.cons);
  const bool ok = warp_wait(&sh.cons, c.syncs & 1, &sh.abort);
  ++c.syncs;
  return ok;
}

// The units of super-chunks [sa, sb) of the tiles in a stage, round-robin over
// the warps (warp w: unit w, w + 8, ... of every super-chunk).  For a tile
// pair the two tiles' units of two super-chunks are issued in one block, with
// independent accumulators, so that their loads, conversions and MMAs overlap.
template <int FMT>
__device__ __forceinline__ void run_units(const StreamGeom& g, const uint8_t* stage, const StageHdr& h,
                                          const uint8_t* brow, bool bf16, float (&acc)[2][4][4]) {
  const int warp = threadIdx.x >> 5;
  if (FMT == FMT_NVFP4 && h.mask == 3) {
    const uint8_t* p1 = stage + h.part;
    int s = h.sa;
    for (; s + 1 < h.sb; s += 2) {  // two full super-chunks (only the last can be short)
      const int off = (s - h.sa) * g.sc_bytes, c0 = 8 * s * g.unit_cols;
      for (int j = warp; j < 8; j += kSW) {
        unit_nvfp4(stage + off, j, brow, c0, bf16, acc[0]);
        unit_nvfp4(p1 + off, j, brow, c0, bf16, acc[1]);
        unit_nvfp4(stage + off + g.sc_bytes, j, brow, c0 + 8 * g.unit_cols, bf16, acc[0]);
        unit_nvfp4(p1 + off + g.sc_bytes, j, brow, c0 + 8 * g.unit_cols, bf16, acc[1]);
      }
    }
    if (s < h.sb) {
      const int off = (s - h.sa) * g.sc_bytes, c0 = 8 * s * g.unit_cols;
      for (int j = warp; j < min(8, g.units - 8 * s); j += kSW) {
        unit_nvfp4(stage + off, j, brow, c0, bf16, acc[0]);
        unit_nvfp4(p1 + off, j, brow, c0, bf16, acc[1]);
      }
    }
    return;
  }
  const uint8_t* p0 = stage;
  const uint8_t* p1 = stage + ((h.mask & 1) ? h.part : 0);
  for (int s = h.sa; s < h.sb; ++s) {
    const int off = (s - h.sa) * g.sc_bytes;
    const int us = min(8, g.units - 8 * s), c0 = 8 * s * g.unit_cols;
    for (int j = warp; j < us; j += kSW) {
      if (FMT == FMT_NVFP4) {
        if (h.mask & 1) unit_nvfp4(p0 + off, j, brow, c0, bf16, acc[0]);
        if (h.mask & 2) unit_nvfp4(p1 + off, j, brow, c0, bf16, acc[1]);
      } else {
        if (h.mask & 1) unit_fp6(p0 + off, j, brow, c0, bf16, acc[0]);
        if (h.mask & 2) unit_fp6(p1 + off, j, brow, c0, bf16, acc[1]);
      }
    }
  }
}

// MODE 0: gate/up + SwiGLU -> a;  MODE 1: down -> y;  MODE 2: down -> y tile in
// shared memory, combined per 16-row tile of H into out.  Activation rows:
// staged once (`bonce` area; gate/up: by token, rtok = routed rows' tokens;
// down: by row) or with every stage.  Returns at the end marker (or on a
// timeout).
template <int FMT, int MODE>
__device__ __forceinline__ void consume(const ExpertParams& p, const StreamGeom& g, StreamShared& sh,
                                        uint8_t* ring, const uint8_t* bonce, const int* rtok, Consumer& c,
                                        float4 (*red)[kSW][2][32], float* ys, const float* gates,
                                        const int* inv, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int S = p.T * p.k;
  while (true) {
    const int st = c.q % g.n_stages;
    if (!warp_wait(&sh.full[st], (c.q / g.n_stages) & 1, &sh.abort)) return;
    const StageHdr h = sh.hdr[st];
    const uint8_t* stage = ring + (size_t)st * g.stage_bytes;
    ++c.q;
    if (h.flags & ST_END) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[st]);
      return;
    }
    // this lane's activation row (column-addressed), or none
    const uint8_t* brow = nullptr;
    if (gi < h.n) {
      if (g.b_once) {
        const int r = MODE != 0 ? h.row + gi : ((h.flags & ST_SHARED) ? h.row - S + gi : rtok[h.row + gi]);
        brow = bonce + (size_t)r * g.b_stride;
      } else {
        brow = stage + g.w_cap + gi * g.b_stride - 2 * (h.sa * 8 * g.unit_cols);
      }
    }
    const bool bf16 = !g.b_once && (h.flags & ST_BF16);
    run_units<FMT>(g, stage, h, brow, bf16, c.acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[st]);
    if (!(h.flags & ST_LAST)) continue;

    // ---- item complete: the eight partial sums (warp order) in warp `owner`.
    // Two slots; a warp writes an item's partials once the owner of the item
    // two before has read that slot, and only the owner waits for the eight.
    const int slot = c.items & 1, owner = c.items % kSW, use = c.items >> 1;
    if (use > 0 && !warp_wait(&sh.red_free[slot], (use - 1) & 1, &sh.abort)) return;
    {  // the four accumulators in order, then zeroed (16-byte stores: no bank conflicts)
      float s0[4], s1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s0[i] = ((c.acc[0][0][i] + c.acc[0][1][i]) + c.acc[0][2][i]) + c.acc[0][3][i];
        s1[i] = ((c.acc[1][0][i] + c.acc[1][1][i]) + c.acc[1][2][i]) + c.acc[1][3][i];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          c.acc[0][q][i] = 0.f;
          c.acc[1][q][i] = 0.f;
        }
      }
      red[slot][warp][0][lane] = make_float4(s0[0], s0[1], s0[2], s0[3]);
      red[slot][warp][1][lane] = make_float4(s1[0], s1[1], s1[2], s1[3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.red_full[slot]);
    ++c.items;
    if (warp == owner) {
      if (!warp_wait(&sh.red_full[slot], use & 1, &sh.abort)) return;
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
#pragma unroll
      for (int w = 0; w < kSW; ++w) {
        const float4 a0 = red[slot][w][0][lane], a1 = red[slot][w][1][lane];
        v[0] += a0.x; v[1] += a0.y; v[2] += a0.z; v[3] += a0.w;
        v[4] += a1.x; v[5] += a1.y; v[6] += a1.z; v[7] += a1.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.red_free[slot]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rl = gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
        if (col >= h.n) continue;
        if (MODE == 0) {
          const float G = h.ts0 * v[i], U = h.ts1 * v[4 + i];
          const float a = G / (1.0f + expf(-G)) * U;
          p.abuf[(size_t)(h.row + col) * p.I + 16 * h.tile + rl] = __half_as_ushort(__float2half_rn(a));
        } else if (MODE == 1) {
          p.ybuf[(size_t)(h.row + col) * p.H + 16 * h.tile + rl] = h.ts0 * v[i];
        } else {
          ys[(h.row + col) * 16 + rl] = h.ts0 * v[i];
        }
      }
    }
    if (MODE == 2 && (h.flags & ST_TILE_END)) {
      // every entry of this tile of H is in ys: out = sum_j g_j y_j + y_shared, j in order
      if (!consumer_sync(sh, c)) return;
      for (int i = threadIdx.x; i < p.T * 16; i += kSW * 32) {
        const int tk = i / 16, hh = i % 16;
        float a = 0.f;
        for (int j = 0; j < p.k; ++j) a = fmaf(gates[tk * p.k + j], ys[inv[tk * p.k + j] * 16 + hh], a);
        if (p.shared) a += ys[(S + tk) * 16 + hh];
        out[(size_t)tk * p.H + 16 * h.tile + hh] = a;
      }
    }
  }
}

// The activation rows staged once: consumers wait for them and, for x, turn
// the bf16 values into f16 in place (then a barrier, before any use).
__device__ __forceinline__ bool consumer_take_bonce(StreamShared& sh, Consumer& c, uint8_t* bonce, int n16,
                                                    bool convert) {
  if (!warp_wait(&sh.bonce, 0, &sh.abort)) return false;
  if (!convert) return true;
  uint32_t* w = reinterpret_cast<uint32_t*>(bonce);
  for (int i = threadIdx.x; i < n16 / 2; i += kSW * 32) {
    const uint32_t v = w[i];
    const __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return consumer_sync(sh, c);
}

struct StreamArgs {
  ExpertParams p;
  RouteParams rp;  // routing in the CTA (decode variants)
  StreamGeom g;
  float* out;      // MODE 2
};

__device__ __forceinline__ void stream_setup(StreamShared& sh, const StreamGeom& g) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < g.n_stages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kSW);
    }
    mbar_init(&sh.cons, kSW);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.red_full[i], kSW);
      mbar_init(&sh.red_free[i], 1);
    }
    mbar_init(&sh.bonce, 1);
    mbar_init(&sh.tsbar, 1);
    sh.abort = 0;
    mbar_init_fence();
  }
  __syncthreads();
}

__device__ __forceinline__ int stages_per_item(const StreamGeom& g) {
  return g.pair_stage ? 1 : g.tiles * ((g.nsc + g.sc_run - 1) / g.sc_run);
}

__device__ __forceinline__ void item_range(int n_items, int& i0, int& i1) {
  i0 = (int)((long long)n_items * blockIdx.x / gridDim.x);
  i1 = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x);
}

// Producer loop over items [i0, i1), run by the whole producer warp: the 32
// lanes describe 32 items at once (their global reads overlap), lane 0 issues
// them.  map(i, y, tile, flags) gives item i's entry, weight group and extra
// flags.  With `pre` set, lane 0 issues weights only while the ring is free,
// then waits for the kernels before this one and calls after_wait() (which
// stages activations) before it goes on.
template <int MODE, typename Map, typename AfterWait>
__device__ __forceinline__ void produce_items(Producer& pr, const ExpertParams& p, const Entries& en, int i0,
                                              int i1, ItemDesc* sdesc, Map map, bool pre,
                                              AfterWait after_wait) {
  const int lane = threadIdx.x & 31;
  const float* sts = pr.sts;
  const int per_item = stages_per_item(pr.g);
  int ok = warp_wait(&pr.sh.tsbar, 0, &pr.sh.abort);
  for (int base = i0; base < i1 && ok; base += 32) {
    if (base + lane < i1) {
      int y, tile, flags;
      map(base + lane, y, tile, flags);
      ItemDesc d = describe<MODE>(p, en, sts, y, tile);
      d.flags |= flags;
      sdesc[lane] = d;
    }
    __syncwarp();
    if (lane == 0) {
      for (int l = 0; l < 32 && base + l < i1 && pr.ok; ++l) {
        if (pre && pr.q + per_item > pr.g.n_stages) {  // the ring is full: now the wait
          pre = false;
          after_wait();
        }
        pr.item<MODE>(sdesc[l]);
      }
      ok = pr.ok;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
  }
  if (lane == 0 && pre) after_wait();
}

// ---------------------------------------------------------------- gate/up
// ROUTE 1 (T <= 8): x staged once per CTA, shared-expert items before the
// router has finished, then routing in the CTA, then the routed items.
// ROUTE 0: work entries from the dispatch kernel, activation rows with every
// stage.  Items are (entry y, tile pair) in y-major order; the list is cut
// into equal contiguous ranges, one per CTA (for ROUTE 1 by its upper bound,
// every routed expert one entry, so that the cut is known before the routing
// is).
template <int FMT, int ROUTE>
__global__ void __launch_bounds__(kSThreads, 2) stream_gateup_kernel(StreamArgs a) {
  // local copies: fields read in the loops stay in registers
  const ExpertParams p = a.p;
  const StreamGeom g = a.g;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ StreamShared sh;
  __shared__ float4 red[2][kSW][2][32];
  __shared__ SmallRoute rt;
  __shared__ ItemDesc sdesc[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.I / 16;
  const int nsh = p.shared ? (p.T + kTokTile - 1) / kTokTile : 0;
  uint8_t* bonce = ring + (size_t)g.n_stages * g.stage_bytes;
  stream_setup(sh, g);
  Consumer c{0, 0, 0, {}};
  int i0, i1;
  if (ROUTE) {
    item_range((nsh + min(p.T * p.k, p.E)) * P, i0, i1);
    int q_pre = 0;  // stages the producer issued before the routing
    auto gu_map = [P](int i, int& y, int& tile, int& flags) {
      y = i / P;
      tile = i % P;
      flags = 0;
    };
    auto nothing = [] {};
    if (warp == kSW) {  // x once, then the shared-expert items: no routing needed
      Producer pr(p, g, sh, ring, 0);
      if (lane == 0) {
        pr.stage_ts();
        pr.stage_once(bonce, p.x, (uint32_t)(p.T * p.H * 2));
      }
      const Entries en{nullptr, nullptr, 0, nsh, false};
      produce_items<0>(pr, p, en, i0, min(i1, nsh * P), sdesc, gu_map, false, nothing);
      if (lane == 0) {
        pr.end_marker();
        q_pre = pr.q;
      }
      __syncwarp();
    } else {
      if (consumer_take_bonce(sh, c, bonce, p.T * p.H, true))
        consume<FMT, 0>(p, g, sh, ring, bonce, rt.row_token, c, red, nullptr, nullptr, nullptr, nullptr);
    }
    griddep_wait();  // the router's partial sums
    route_small_cta(a.rp, rt, blockIdx.x == 0);
    griddep_launch();
    if (warp == kSW) {
      q_pre = __shfl_sync(0xffffffffu, q_pre, 0);
      Producer pr(p, g, sh, ring, q_pre);
      pr.bonce_armed = true;  // x, requested before the routing
      const Entries er{rt.entries, rt.row_token, rt.n_entries, nsh, false};
      produce_items<0>(pr, p, er, max(i0, nsh * P), min(i1, (nsh + er.n) * P), sdesc, gu_map, false,
                       nothing);
      if (lane == 0) {
        pr.end_marker();
        if (!pr.ok) pr.drain();
      }
      __syncwarp();
    } else {
      consume<FMT, 0>(p, g, sh, ring, bonce, rt.row_token, c, red, nullptr, nullptr, nullptr, nullptr);
    }
    if (blockIdx.x == 0) {
      __syncthreads();
      publish_counts(a.rp, rt);
    }
  } else {
    griddep_wait();  // work entries from the dispatch kernel
    griddep_launch();
    const Entries en{p.entries, p.row_token, __ldcg(p.n_entries), nsh, true};
    item_range((nsh + en.n) * P, i0, i1);
    if (warp == kSW) {
      Producer pr(p, g, sh, ring, 0);
      if (lane == 0) pr.stage_ts();
      produce_items<0>(pr, p, en, i0, i1, sdesc, [P](int i, int& y, int& tile, int& flags) {
        y = i / P;
        tile = i % P;
        flags = 0;
      }, false, [] {});
      if (lane == 0) {
        pr.end_marker();
        if (!pr.ok) pr.drain();
      }
      __syncwarp();
    } else {
      consume<FMT, 0>(p, g, sh, ring, nullptr, nullptr, c, red, nullptr, nullptr, nullptr, nullptr);
    }
  }
  if (sh.abort && threadIdx.x == 0) *p.status = -5;  // MOE_ETIMEOUT
}

// ---------------------------------------------------------------- down
// ROUTE 1 (T <= 8, MODE 2): routing in the CTA before waiting for gate/up;
// each CTA owns a contiguous range of 16-row tiles of H and takes every entry
// of each (tile-major items), so the combine of a tile happens in shared
// memory; a (all rows, one copy) staged once after the wait when it fits.
// ROUTE 0 (MODE 1): entries from the dispatch kernel, items (entry, tile)
// entry-major, y to ybuf for the combine kernel.  Either way the weights of
// the first ring-full of stages are copied before waiting for gate/up.
template <int FMT, int ROUTE>
__global__ void __launch_bounds__(kSThreads, 2) stream_down_kernel(StreamArgs a) {
  const ExpertParams p = a.p;
  const StreamGeom g = a.g;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ StreamShared sh;
  __shared__ float4 red[2][kSW][2][32];
  __shared__ SmallRoute rt;
  __shared__ ItemDesc sdesc[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HT = p.H / 16;
  const int nsh = p.shared ? (p.T + kTokTile - 1) / kTokTile : 0;
  const int S = p.T * p.k;
  // the next kernel (the next layer's router) may start reading its weights
  griddep_launch();
  stream_setup(sh, g);
  if (threadIdx.x == kSW * 32) {  // the tensor-scale table, while the CTA routes
    mbar_arrive_expect(&sh.tsbar, (uint32_t)g.ts_bytes);
    bulk_g2s(ring + (size_t)g.n_stages * g.stage_bytes + g.b_bytes, p.tscale, (uint32_t)g.ts_bytes, &sh.tsbar);
  }
  Consumer c{0, 0, 0, {}};
  Entries en;
  if (ROUTE) {
    // the router finished before gate/up let this launch start: its partial
    // sums are final
    route_small_cta(a.rp, rt, false);
    en = Entries{rt.entries, rt.row_token, rt.n_entries, nsh, false};
  } else {
    // dispatch finished before gate/up let this launch start
    en = Entries{p.entries, p.row_token, __ldcg(p.n_entries), nsh, true};
  }
  const int Y = nsh + en.n;
  int i0, i1;
  if (ROUTE) {
    int h0, h1;
    item_range(HT, h0, h1);
    i0 = h0 * Y;
    i1 = h1 * Y;
  } else {
    item_range(Y * HT, i0, i1);
  }
  uint8_t* bonce = ring + (size_t)g.n_stages * g.stage_bytes;
  float* ys = reinterpret_cast<float*>(bonce + g.b_bytes + g.ts_bytes);
  if (warp == kSW) {
    Producer pr(p, g, sh, ring, 0);
    auto dn_map = [Y, HT](int i, int& y, int& tile, int& flags) {
      y = ROUTE ? i % Y : i / HT;
      tile = ROUTE ? i / Y : i % HT;
      flags = (ROUTE && y == Y - 1) ? ST_TILE_END : 0;
    };
    // staged-once activations: weights of the first stages before the wait
    // for gate/up (the ring is free: no waits), then a; otherwise the wait first
    auto after_wait = [&] {
      griddep_wait();  // a from gate/up
      if (g.b_once) pr.stage_once(bonce, p.abuf, (uint32_t)((S + p.T) * p.I * 2));
    };
    if (!g.b_once && lane == 0) griddep_wait();
    produce_items<1>(pr, p, en, i0, i1, sdesc, dn_map, g.b_once, after_wait);
    if (lane == 0) {
      pr.end_marker();
      if (!pr.ok) pr.drain();
    }
    __syncwarp();
  } else {
    if (!g.b_once || consumer_take_bonce(sh, c, bonce, 0, false)) {
      if (ROUTE)
        consume<FMT, 2>(p, g, sh, ring, bonce, nullptr, c, red, ys, rt.gates, rt.inv, a.out);
      else
        consume<FMT, 1>(p, g, sh, ring, bonce, nullptr, c, red, nullptr, nullptr, nullptr, nullptr);
    }
  }
  if (sh.abort && threadIdx.x == 0) *p.status = -5;  // MOE_ETIMEOUT
}

int g_sms = 0;

int num_sms() {
  if (g_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      g_sms = 148;
  }
  return g_sms;
}

template <typename K>
cudaError_t set_smem(K kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamMaxDyn);
}

constexpr int kStageTarget = 40 * 1024;  // weight bytes of a stage at most, when it can be split

}  // namespace

// Geometry of a streaming launch: reduction length K, `tiles` weight tiles
// per item, up to n_max activation rows per item; `b_rows` > 0 stages that
// many activation rows (K columns) once per CTA instead of with every stage.
StreamGeom stream_geom(int fmt, int K, int tiles, int n_max, int b_rows, int ring_bytes, int n_experts) {
  StreamGeom g{};
  g.ts_bytes = tscale_bytes(n_experts);
  const MatGeom m = mat_geom(fmt, K);
  const bool nv = fmt == FMT_NVFP4;
  g.fmt = fmt;
  g.K = K;
  g.tiles = tiles;
  g.units = m.units;
  g.nsc = m.nsc;
  g.sc_bytes = m.sc_bytes;
  g.tile_bytes = m.tile_bytes;
  g.unit_cols = nv ? 64 : 128;
  g.unit_bytes = nv ? 512 : 1536;
  g.hdr_bytes = nv ? 512 : 128;
  g.pair_stage = tiles == 2 && 2 * m.tile_bytes <= kStageTarget;
  if (g.pair_stage) {
    g.sc_run = m.nsc;
    g.w_cap = 2 * m.tile_bytes;
  } else {
    g.sc_run = kStageTarget / m.sc_bytes;
    if (g.sc_run < 1) g.sc_run = 1;
    if (g.sc_run > m.nsc) g.sc_run = m.nsc;
    g.w_cap = g.sc_run * m.sc_bytes < m.tile_bytes ? g.sc_run * m.sc_bytes : m.tile_bytes;
  }
  g.n_max = n_max;
  g.b_once = b_rows > 0 && (size_t)b_rows * K * 2 <= (size_t)kStreamOnceMax;
  int b_area = 0;
  if (g.b_once) {
    g.b_stride = K * 2;
    g.b_bytes = (b_rows * K * 2 + 127) / 128 * 128;
  } else {
    const int cols = g.sc_run * 8 * g.unit_cols < K ? g.sc_run * 8 * g.unit_cols : K;
    g.b_stride = cols * 2 + 16;
    g.b_bytes = 0;
    b_area = n_max * g.b_stride;
  }
  g.stage_bytes = (g.w_cap + b_area + 127) / 128 * 128;
  int ns = ring_bytes / g.stage_bytes;
  if (ns > kSMaxStages) ns = kSMaxStages;
  if (ns < 2) ns = 2;
  g.n_stages = ns;
  return g;
}

size_t stream_smem(const StreamGeom& g, int ys_rows) {
  return (size_t)g.n_stages * g.stage_bytes + g.b_bytes + g.ts_bytes + (size_t)ys_rows * 16 * sizeof(float);
}

bool stream_small_ok(int T, int k) { return T <= kTokTile && T * k <= kSmallSlots; }

cudaError_t launch_stream_gateup(const ExpertParams& p, const RouteParams& rp, const StreamGeom& g,
                                 bool route, cudaStream_t st) {
  if (route && !g.b_once) return cudaErrorInvalidValue;  // the routed variant stages x once
  StreamArgs a{p, rp, g, nullptr};
  const size_t smem = stream_smem(g, 0);
  if (smem > (size_t)kStreamMaxDyn) return cudaErrorInvalidValue;
  dim3 grid(num_sms());
  if (p.fmt == FMT_NVFP4)
    return route ? launch_k(stream_gateup_kernel<FMT_NVFP4, 1>, grid, dim3(kSThreads), smem, st, true, a)
                 : launch_k(stream_gateup_kernel<FMT_NVFP4, 0>, grid, dim3(kSThreads), smem, st, true, a);
  return route ? launch_k(stream_gateup_kernel<FMT_FP6, 1>, grid, dim3(kSThreads), smem, st, true, a)
               : launch_k(stream_gateup_kernel<FMT_FP6, 0>, grid, dim3(kSThreads), smem, st, true, a);
}

cudaError_t launch_stream_down(const ExpertParams& p, const RouteParams& rp, const StreamGeom& g,
                               bool route, float* out, cudaStream_t st) {
  StreamArgs a{p, rp, g, out};
  const size_t smem = stream_smem(g, route ? p.T * p.k + p.T : 0);
  if (smem > (size_t)kStreamMaxDyn) return cudaErrorInvalidValue;
  int ctas = num_sms();
  if (route && ctas > p.H / 16) ctas = p.H / 16;  // one tile of H per CTA at least
  dim3 grid(ctas);
  if (p.fmt == FMT_NVFP4)
    return route ? launch_k(stream_down_kernel<FMT_NVFP4, 1>, grid, dim3(kSThreads), smem, st, true, a)
                 : launch_k(stream_down_kernel<FMT_NVFP4, 0>, grid, dim3(kSThreads), smem, st, true, a);
  return route ? launch_k(stream_down_kernel<FMT_FP6, 1>, grid, dim3(kSThreads), smem, st, true, a)
               : launch_k(stream_down_kernel<FMT_FP6, 0>, grid, dim3(kSThreads), smem, st, true, a);
}

cudaError_t stream_kernels_init() {
  cudaError_t e;
  if ((e = set_smem(stream_gateup_kernel<FMT_NVFP4, 0>)) != cudaSuccess) return e;
  if ((e = set_smem(stream_gateup_kernel<FMT_NVFP4, 1>)) != cudaSuccess) return e;
  if ((e = set_smem(stream_gateup_kernel<FMT_FP6, 0>)) != cudaSuccess) return e;
  if ((e = set_smem(stream_gateup_kernel<FMT_FP6, 1>)) != cudaSuccess) return e;
  if ((e = set_smem(stream_down_kernel<FMT_NVFP4, 0>)) != cudaSuccess) return e;
  if ((e = set_smem(stream_down_kernel<FMT_NVFP4, 1>)) != cudaSuccess) return e;
  if ((e = set_smem(stream_down_kernel<FMT_FP6, 0>)) != cudaSuccess) return e;
  return set_smem(stream_down_kernel<FMT_FP6, 1>);
}

}  // namespace moe
