// Small-batch expert path (work entries of up to 8 tokens): the packed expert
// weights stream from HBM through a shared-memory ring of bulk async copies.
//
// A launch is one CTA per SM over a list of work items.  An item is one work
// entry (an expert and up to eight of its token rows) times one weight group:
// a gate/up tile pair (16 rows of W_gate and the same 16 rows of W_up), or one
// 16-row tile of W_down.  A producer warp copies each item super-chunk by
// super-chunk (up to 512 NVFP4 or 1024 FP6 columns of every tile of the
// group) into the ring with cp.async.bulk, the bytes counted on the stage's
// mbarrier, together with the same columns of the item's activation rows.
// The eight consumer warps take one unit of every stage each (warp w: chunk
// or pair w of the super-chunk), dequantise it in registers into m16n8k16 A
// fragments (the layout of layout.cuh) and accumulate in fp32.  At the end of
// an item the eight partial sums are added in warp order (deterministic, and
// independent of the other tokens of the entry) and one warp applies the
// epilogue: SwiGLU into a (gate/up), y (down), or y into shared memory for
// the gate-weighted combine of a few tokens.  The copies keep the whole ring
// in flight whatever the arithmetic is doing, which is what streaming weight
// bytes at HBM bandwidth needs: 16-byte per-thread loads left too few bytes
// in flight per SM (the "Strata on an Intel Arc" pages found the same for
// their decode matvecs: "The engine itself on Intel", "Planned", item 5).
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
enum : int { ST_LAST = 1, ST_BF16 = 2, ST_TILE_END = 4, ST_END = 8 };
struct StageHdr {
  int expert;  // E: the shared expert
  int row;     // first row (of a / y) of the item's entry
  int n;       // token rows
  int tile;    // gate/up: tile pair; down: 16-row tile of H
  int u0;      // first unit of the stage within its super-chunk
  int nu;      // units in the stage
  int col0;    // first column of the stage
  int flags;
};

struct StreamShared {
  uint64_t full[kSMaxStages];
  uint64_t empty[kSMaxStages];
  uint64_t cons;  // barrier of the eight consumer warps (bounded waits, unlike bar.sync)
  StageHdr hdr[kSMaxStages];
  int abort;
};

// Item source: work entries in shared memory (routed in this CTA) or in
// global memory (written by the dispatch kernel), plus the leading shared-
// expert entries, which follow from T.
struct Entries {
  const int4* e;   // routed entries
  const int* tok;  // token of each routed row
  int n;           // routed entries
  int nsh;         // leading shared-expert entries
  bool global;     // e and tok in global memory (read through L2)
};

__device__ __forceinline__ void entry_of(const ExpertParams& p, const Entries& en, int y, int& expert,
                                         int& row, int& n) {
  const int S = p.T * p.k;
  if (y < en.nsh) {
    expert = p.E;
    row = S + kTokTile * y;
    n = min(kTokTile, p.T - kTokTile * y);
    return;
  }
  const int4 e = en.global ? __ldcg(en.e + (y - en.nsh)) : en.e[y - en.nsh];
  expert = e.x;
  row = e.y;
  n = e.z;
  if (expert < 0 || expert >= p.E || n < 1 || n > kTokTile || row < 0 || row + n > S) {
    *p.status = -1;  // MOE_EINVAL: corrupt entry, skipped
    n = 0;
  }
}

// ---------------------------------------------------------------- producer
// One lane issues every copy.  Stages are taken in order; stage q waits until
// the consumers have released its previous use.
struct Producer {
  const ExpertParams& p;
  const StreamGeom& g;
  StreamShared& sh;
  uint8_t* ring;
  uint64_t pol;
  int q;        // stages issued
  bool ok;
  // stages whose activation copies wait for the kernels before this one
  int deferred_from, deferred_to;

  __device__ Producer(const ExpertParams& p_, const StreamGeom& g_, StreamShared& sh_, uint8_t* ring_)
      : p(p_), g(g_), sh(sh_), ring(ring_), pol(l2_evict_first()), q(0), ok(true), deferred_from(0),
        deferred_to(0) {}

  __device__ uint8_t* stage_ptr(int st) const { return ring + (size_t)st * g.stage_bytes; }

  __device__ bool take(int& st) {
    st = q % g.n_stages;
    if (!mbar_wait(&sh.empty[st], ((q / g.n_stages) & 1) ^ 1, &sh.abort)) {
      ok = false;
      return false;
    }
    return true;
  }

  // units (chunks / pairs) of super-chunk s
  __device__ int sc_units_of(int s) const { return min(8, g.units - 8 * s); }

  // Activation row r of an item (its column origin): x / f16 copy of x for
  // gate/up, a for down.
  __device__ const uint16_t* brow(int mode, int expert, int row, int r, const Entries* en) const {
    const int S = p.T * p.k;
    if (mode != 0) return p.abuf + (size_t)(row + r) * p.I;
    if (expert == p.E) return p.x + (size_t)(row - S + r) * p.H;
    const int tk = en->global ? __ldcg(en->tok + row + r) : en->tok[row + r];
    return p.xh + (size_t)tk * p.H;
  }

  __device__ void copy_b(int mode, const StageHdr& h, uint8_t* dst, uint64_t* bar, const Entries* en) const {
    const uint32_t bb = (uint32_t)(h.nu * g.unit_cols) * 2u;
    for (int r = 0; r < h.n; ++r)
      bulk_g2s(dst + g.w_bytes + r * g.seg_stride, brow(mode, h.expert, h.row, r, en) + h.col0, bb, bar);
  }

  // Copies of one item, stage by stage (a stage: up to g.stage_units units
  // of one super-chunk of every tile of the group), each with its activation
  // columns unless `defer_b`.  tile0: first tile of the group.
  __device__ void item(int mode, const uint8_t* tile0, int expert, int row, int n, int tile, int flags,
                       const Entries* en, bool defer_b) {
    for (int s = 0; s < g.nsc && ok; ++s) {
      const int su = sc_units_of(s);
      for (int u0 = 0; u0 < su && ok; u0 += g.stage_units) {
        int st;
        if (!take(st)) return;
        uint8_t* dst = stage_ptr(st);
        StageHdr h;
        h.expert = expert;
        h.row = row;
        h.n = n;
        h.tile = tile;
        h.u0 = u0;
        h.nu = min(g.stage_units, su - u0);
        h.col0 = (8 * s + u0) * g.unit_cols;
        h.flags = flags | ((s == g.nsc - 1 && u0 + g.stage_units >= su) ? ST_LAST : 0);
        sh.hdr[st] = h;
        const uint32_t ub = (uint32_t)h.nu * g.unit_bytes;
        mbar_arrive_expect(&sh.full[st], g.tiles * (g.hdr_bytes + ub) + (uint32_t)(n * h.nu * g.unit_cols * 2));
        for (int tt = 0; tt < g.tiles; ++tt) {
          const uint8_t* sc = tile0 + (size_t)tt * g.tile_bytes + (size_t)s * g.sc_bytes;
          uint8_t* d = dst + tt * g.tile_w;
          if (u0 == 0) {  // scales and the units are contiguous
            bulk_g2s_hint(d, sc, g.hdr_bytes + ub, &sh.full[st], pol);
          } else {
            bulk_g2s_hint(d, sc, g.hdr_bytes, &sh.full[st], pol);
            bulk_g2s_hint(d + g.hdr_bytes, sc + g.hdr_bytes + u0 * g.unit_bytes, ub, &sh.full[st], pol);
          }
        }
        if (!defer_b) copy_b(mode, h, dst, &sh.full[st], en);
        ++q;
      }
    }
  }

  // activation copies of stages [from, to) issued earlier with defer_b
  __device__ void release_deferred(int mode, const Entries* en) {
    for (int qq = deferred_from; qq < deferred_to; ++qq) {
      const int st = qq % g.n_stages;
      copy_b(mode, sh.hdr[st], stage_ptr(st), &sh.full[st], en);
    }
  }

  // a stage that carries no data and tells the consumers to leave their loop
  __device__ void end_marker() {
    int st;
    if (!take(st)) return;
    StageHdr h{};
    h.flags = ST_END;
    sh.hdr[st] = h;
    mbar_arrive(&sh.full[st]);
    ++q;
  }

  // before exit after a timeout: wait (bounded) for the copies still landing
  __device__ void drain() {
    const int n = min(q, g.n_stages);
    for (int i = 1; i <= n; ++i) {
      const int qq = q - i, st = qq % g.n_stages;
      mbar_drain(&sh.full[st], (qq / g.n_stages) & 1);
    }
  }
};

// ---------------------------------------------------------------- consumers
// 16 activations (f16, or bf16 converted to f16) of row gi of a stage, or zeros.
__device__ __forceinline__ void b_frag(const uint8_t* stage, const StreamGeom& g, int gi, int n, int col,
                                       bool bf16, uint32_t (&xw)[8]) {
  if (gi < n) {
    const uint4* px = reinterpret_cast<const uint4*>(stage + g.w_bytes + gi * g.seg_stride + 2 * col);
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

// NVFP4 unit u of tile tt of a stage: chunk j = u0 + u of its super-chunk
// (64 columns, one e4m3 scale per 16 columns and row).
__device__ __forceinline__ void unit_nvfp4(const uint8_t* stage, const StreamGeom& g, int tt, int u,
                                           int j, int n, bool bf16, float (&acc)[4]) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const uint8_t* base = stage + tt * g.tile_w;
  const uint4 sv = *reinterpret_cast<const uint4*>(base + 16 * lane);
  const uint4 cv = *reinterpret_cast<const uint4*>(base + g.hdr_bytes + 512 * u + 16 * lane);
  uint32_t xb[8];
  b_frag(stage, g, gi, n, 64 * u + 16 * t, bf16, xb);
  const uint32_t sp = e4m3x2_to_f16x2((u4get(sv, j >> 1) >> (16 * (j & 1))) & 0xFFFFu);
  const uint32_t s_lo = dup_lo(sp), s_hi = dup_hi(sp);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4];
    e2m1x8_to_f16x8(u4get(cv, q), h);
    const uint32_t a[4] = {hmul2(h[0], s_lo), hmul2(h[1], s_hi), hmul2(h[2], s_lo), hmul2(h[3], s_hi)};
    mma_f16(acc, a, xb[2 * q], xb[2 * q + 1]);
  }
}

// FP6 unit u of tile tt of a stage: pair j = u0 + u of its super-chunk (two
// 64-column chunks, one power-of-two scale per 128 columns and row).  All
// lanes take part (shuffle).
__device__ __forceinline__ void unit_fp6(const uint8_t* stage, const StreamGeom& g, int tt, int u, int j,
                                         int n, bool bf16, float (&acc)[4]) {
  const int lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const uint8_t* base = stage + tt * g.tile_w;
  const uint32_t ew = *reinterpret_cast<const uint32_t*>(base + 4 * lane);
  uint4 cv[3];
#pragma unroll
  for (int v = 0; v < 3; ++v)
    cv[v] = *reinterpret_cast<const uint4*>(base + g.hdr_bytes + 1536 * u + 512 * v + 16 * lane);
  const uint32_t words[12] = {cv[0].x, cv[0].y, cv[0].z, cv[0].w, cv[1].x, cv[1].y,
                              cv[1].z, cv[1].w, cv[2].x, cv[2].y, cv[2].z, cv[2].w};
  float blk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t xb[8];
    b_frag(stage, g, gi, n, 128 * u + 64 * h + 16 * t, bf16, xb);
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
        mma_f16(blk, a, xb[2 * step], xb[2 * step + 1]);
      }
    }
  }
  const uint32_t e = __shfl_sync(0xffffffffu, ew, (gi << 2) | (j >> 1));
  const float f0 = ue8m0_to_f32((e >> (16 * (j & 1))) & 0xFFu);
  const float f1 = ue8m0_to_f32((e >> (16 * (j & 1) + 8)) & 0xFFu);
  acc[0] = fmaf(blk[0], f0, acc[0]);
  acc[1] = fmaf(blk[1], f0, acc[1]);
  acc[2] = fmaf(blk[2], f1, acc[2]);
  acc[3] = fmaf(blk[3], f1, acc[3]);
}

// Per-item state of the consumer warps.
struct Consumer {
  int q;      // stages consumed
  int items;  // items finished
  int syncs;  // consumer barriers passed
  float acc[2][4];
  __device__ Consumer() : q(0), items(0), syncs(0) { zero(); }
  __device__ void zero() {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  }
};

// Barrier of the eight consumer warps on an mbarrier (count 8), so that a warp
// that gave up after a timeout cannot leave the others waiting for ever.
// Returns false on timeout.
__device__ __forceinline__ bool consumer_sync(StreamShared& sh, Consumer& c) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane == 0) mbar_arrive(&sh.cons);
  const bool ok = mbar_wait(&sh.cons, c.syncs & 1, &sh.abort);
  ++c.syncs;
  __syncwarp();
  return ok;
}

// Sum the eight warps' partials of an item (warp order) in warp `owner`.
// Returns false on timeout (and sets `mine` false).
__device__ __forceinline__ bool reduce_item(StreamShared& sh, Consumer& c, float (*red)[kSW][32][8],
                                            int slot, int tiles, int owner, bool& mine,
                                            float (&v)[8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    red[slot][warp][lane][i] = c.acc[0][i];
    if (tiles == 2) red[slot][warp][lane][4 + i] = c.acc[1][i];
  }
  mine = false;
  if (!consumer_sync(sh, c)) return false;
  if (warp != owner) return true;
  mine = true;
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = 0.f;
  for (int w = 0; w < kSW; ++w)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] += red[slot][w][lane][i];
      if (tiles == 2) v[4 + i] += red[slot][w][lane][4 + i];
    }
  return true;
}

// MODE 0: gate/up + SwiGLU -> a;  MODE 1: down -> y;  MODE 2: down -> y tile in
// shared memory, combined per 16-row tile of H into out.
template <int FMT, int MODE>
__device__ void consume(const ExpertParams& p, const StreamGeom& g, StreamShared& sh, uint8_t* ring,
                        Consumer& c, float (*red)[kSW][32][8], float* ys, const float* gates,
                        const int* inv, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  while (true) {
    const int st = c.q % g.n_stages;
    if (!mbar_wait(&sh.full[st], (c.q / g.n_stages) & 1, &sh.abort)) return;
    const StageHdr h = sh.hdr[st];
    const uint8_t* stage = ring + (size_t)st * g.stage_bytes;
    ++c.q;
    if (h.flags & ST_END) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[st]);
      return;
    }
    {  // (tile, unit) combinations of the stage, round-robin over the warps
      const bool bf16 = (h.flags & ST_BF16) != 0;
      for (int cb = warp; cb < g.tiles * h.nu; cb += kSW) {
        const int tt = cb / h.nu, u = cb % h.nu;
        if (FMT == FMT_NVFP4)
          unit_nvfp4(stage, g, tt, u, h.u0 + u, h.n, bf16, c.acc[tt]);
        else
          unit_fp6(stage, g, tt, u, h.u0 + u, h.n, bf16, c.acc[tt]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[st]);
    if (!(h.flags & ST_LAST)) continue;

    // ---- item complete: reduce, epilogue
    float v[8];
    const int owner = c.items % kSW;
    bool mine;
    if (!reduce_item(sh, c, red, c.items & 1, g.tiles, owner, mine, v)) return;
    ++c.items;
    c.zero();
    if (mine && h.n > 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rl = gi + ((i & 2) ? 8 : 0), col = 2 * t + (i & 1);
        if (col >= h.n) continue;
        if (MODE == 0) {
          const float G = p.tscale[h.expert * 3 + 0] * v[i], U = p.tscale[h.expert * 3 + 1] * v[4 + i];
          const float a = G / (1.0f + expf(-G)) * U;
          p.abuf[(size_t)(h.row + col) * p.I + 16 * h.tile + rl] = __half_as_ushort(__float2half_rn(a));
        } else if (MODE == 1) {
          p.ybuf[(size_t)(h.row + col) * p.H + 16 * h.tile + rl] = p.tscale[h.expert * 3 + 2] * v[i];
        } else {
          ys[(h.row + col) * 16 + rl] = p.tscale[h.expert * 3 + 2] * v[i];
        }
      }
    }
    if (MODE == 2 && (h.flags & ST_TILE_END)) {
      // every entry of this tile of H is in ys: out = sum_j g_j y_j + y_shared, j in order
      if (!consumer_sync(sh, c)) return;
      const int S = p.T * p.k;
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

struct StreamArgs {
  ExpertParams p;
  RouteParams rp;   // routing in the CTA (decode variants)
  StreamGeom g;
  float* out;       // MODE 2
};

__device__ __forceinline__ void stream_setup(StreamShared& sh, const StreamGeom& g) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < g.n_stages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kSW);
    }
    mbar_init(&sh.cons, kSW);
    sh.abort = 0;
    mbar_init_fence();
  }
  __syncthreads();
}

__device__ __forceinline__ int stages_per_item(const StreamGeom& g) {
  int n = 0;
  for (int s = 0; s < g.nsc; ++s) n += (min(8, g.units - 8 * s) + g.stage_units - 1) / g.stage_units;
  return n;
}

__device__ __forceinline__ void item_range(int n_items, int& i0, int& i1) {
  i0 = (int)((long long)n_items * blockIdx.x / gridDim.x);
  i1 = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x);
}

// ---------------------------------------------------------------- gate/up
// ROUTE 1 (T <= 8): shared-expert items before the router has finished, then
// routing in the CTA, then the routed items.  ROUTE 0: work entries from the
// dispatch kernel.  Items are (entry y, tile pair) in y-major order; the list
// is cut into equal contiguous ranges, one per CTA (for ROUTE 1 by its upper
// bound, every routed expert one entry, so that the cut is known before the
// routing is).
template <int FMT, int ROUTE>
__global__ void __launch_bounds__(kSThreads, 2) stream_gateup_kernel(StreamArgs a) {
  const ExpertParams& p = a.p;
  const StreamGeom& g = a.g;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ StreamShared sh;
  __shared__ float red[2][kSW][32][8];
  __shared__ SmallRoute rt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.I / 16;
  const int nsh = p.shared ? (p.T + kTokTile - 1) / kTokTile : 0;
  stream_setup(sh, g);
  Consumer c;
  Producer pr(p, g, sh, ring);
  int i0, i1;
  if (ROUTE) {
    const int routed_max = min(p.T * p.k, p.E);
    item_range((nsh + routed_max) * P, i0, i1);
    // shared-expert items: no routing needed
    const int is1 = min(i1, nsh * P);
    Entries en{nullptr, nullptr, 0, nsh, false};
    if (warp == kSW) {
      if (lane == 0) {
        for (int i = i0; i < is1 && pr.ok; ++i) {
          int expert, row, n;
          entry_of(p, en, i / P, expert, row, n);
          const uint8_t* tile0 = p.arena + (size_t)expert * p.expert_bytes + (size_t)(2 * (i % P)) * p.gu_tile_bytes;
          pr.item(0, tile0, expert, row, n, i % P, ST_BF16, &en, false);
        }
        pr.end_marker();
      }
      __syncwarp();
    } else {
      consume<FMT, 0>(p, g, sh, ring, c, red, nullptr, nullptr, nullptr, nullptr);
    }
    griddep_wait();  // the router's partial sums
    RouteParams rp = a.rp;
    if (blockIdx.x != 0) {  // only CTA 0 publishes the routing
      rp.logits = nullptr;
      rp.idx = nullptr;
      rp.gates = nullptr;
      rp.perm = nullptr;
      rp.inv = nullptr;
      rp.row_token = nullptr;
      rp.entries = nullptr;
      rp.n_entries = nullptr;
    }
    route_small_cta(rp, rt);
    griddep_launch();
    Entries er{rt.entries, rt.row_token, rt.n_entries, nsh, false};
    if (warp == kSW) {
      if (lane == 0) {
        const int iend = min(i1, (nsh + er.n) * P);
        for (int i = max(i0, nsh * P); i < iend && pr.ok; ++i) {
          int expert, row, n;
          entry_of(p, er, i / P, expert, row, n);
          const uint8_t* tile0 = p.arena + (size_t)expert * p.expert_bytes + (size_t)(2 * (i % P)) * p.gu_tile_bytes;
          pr.item(0, tile0, expert, row, n, i % P, 0, &er, false);
        }
        pr.end_marker();
        if (!pr.ok) pr.drain();
      }
      __syncwarp();
    } else {
      consume<FMT, 0>(p, g, sh, ring, c, red, nullptr, nullptr, nullptr, nullptr);
    }
    if (blockIdx.x == 0) {
      __syncthreads();
      publish_counts(a.rp, rt);
    }
  } else {
    griddep_wait();  // work entries from the dispatch kernel
    griddep_launch();
    const int n_routed = __ldcg(p.n_entries);
    Entries en{p.entries, p.row_token, n_routed, nsh, true};
    item_range((nsh + n_routed) * P, i0, i1);
    if (warp == kSW) {
      if (lane == 0) {
        for (int i = i0; i < i1 && pr.ok; ++i) {
          int expert, row, n;
          entry_of(p, en, i / P, expert, row, n);
          const uint8_t* tile0 = p.arena + (size_t)expert * p.expert_bytes + (size_t)(2 * (i % P)) * p.gu_tile_bytes;
          pr.item(0, tile0, expert, row, n, i % P, expert == p.E ? ST_BF16 : 0, &en, false);
        }
        pr.end_marker();
        if (!pr.ok) pr.drain();
      }
      __syncwarp();
    } else {
      consume<FMT, 0>(p, g, sh, ring, c, red, nullptr, nullptr, nullptr, nullptr);
    }
  }
  if (sh.abort && threadIdx.x == 0) *p.status = -5;  // MOE_ETIMEOUT
}

// ---------------------------------------------------------------- down
// ROUTE 1 (T <= 8, MODE 2): routing in the CTA before waiting for gate/up;
// each CTA owns a contiguous range of 16-row tiles of H and takes every entry
// of each (tile-major items), so the combine of a tile happens in shared
// memory.  ROUTE 0 (MODE 1): entries from the dispatch kernel, items
// (entry, tile) entry-major, y to ybuf for the combine kernel.  Either way the
// weight copies of the first ring-full of stages are issued before waiting
// for gate/up; their activation copies follow the wait.
template <int FMT, int ROUTE>
__global__ void __launch_bounds__(kSThreads, 2) stream_down_kernel(StreamArgs a) {
  const ExpertParams& p = a.p;
  const StreamGeom& g = a.g;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ StreamShared sh;
  __shared__ float red[2][kSW][32][8];
  __shared__ SmallRoute rt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HT = p.H / 16;
  const int nsh = p.shared ? (p.T + kTokTile - 1) / kTokTile : 0;
  // the next kernel (the next layer's router) may start reading its weights
  griddep_launch();
  stream_setup(sh, g);
  Consumer c;
  Producer pr(p, g, sh, ring);
  Entries en;
  if (ROUTE) {
    // the router finished before gate/up let this launch start: its partial
    // sums are final
    RouteParams rp = a.rp;
    rp.logits = nullptr;
    rp.idx = nullptr;
    rp.gates = nullptr;
    rp.perm = nullptr;
    rp.inv = nullptr;
    rp.row_token = nullptr;
    rp.entries = nullptr;
    rp.n_entries = nullptr;
    route_small_cta(rp, rt);
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
  float* ys = reinterpret_cast<float*>(ring + (size_t)g.n_stages * g.stage_bytes);
  if (warp == kSW) {
    if (lane == 0) {
      // weights of the first stages now; their activations after the wait
      pr.deferred_from = 0;
      int i = i0;
      const int per_item = stages_per_item(g);
      for (; i < i1 && pr.ok && pr.q + per_item <= g.n_stages; ++i) {
        const int y = ROUTE ? i % Y : i / HT, tile = ROUTE ? i / Y : i % HT;
        int expert, row, n;
        entry_of(p, en, y, expert, row, n);
        const uint8_t* tile0 = p.arena + (size_t)expert * p.expert_bytes + p.gu_bytes + (size_t)tile * p.dn_tile_bytes;
        const int fl = (ROUTE && y == Y - 1) ? ST_TILE_END : 0;
        pr.item(1, tile0, expert, row, n, tile, fl, &en, true);
      }
      pr.deferred_to = pr.q;
      griddep_wait();  // a from gate/up
      pr.release_deferred(1, &en);
      for (; i < i1 && pr.ok; ++i) {
        const int y = ROUTE ? i % Y : i / HT, tile = ROUTE ? i / Y : i % HT;
        int expert, row, n;
        entry_of(p, en, y, expert, row, n);
        const uint8_t* tile0 = p.arena + (size_t)expert * p.expert_bytes + p.gu_bytes + (size_t)tile * p.dn_tile_bytes;
        const int fl = (ROUTE && y == Y - 1) ? ST_TILE_END : 0;
        pr.item(1, tile0, expert, row, n, tile, fl, &en, false);
      }
      pr.end_marker();
      if (!pr.ok) pr.drain();
    }
    __syncwarp();
  } else {
    if (ROUTE)
      consume<FMT, 2>(p, g, sh, ring, c, red, ys, rt.gates, rt.inv, a.out);
    else
      consume<FMT, 1>(p, g, sh, ring, c, red, nullptr, nullptr, nullptr, nullptr);
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

}  // namespace

StreamGeom stream_geom(int fmt, int K, int tiles, int n_max, int stage_units, int ring_bytes) {
  StreamGeom g{};
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
  g.stage_units = stage_units < m.units ? stage_units : m.units;
  g.tile_w = g.hdr_bytes + g.stage_units * g.unit_bytes;
  g.w_bytes = tiles * g.tile_w;
  g.seg_stride = g.stage_units * g.unit_cols * 2 + 16;
  g.n_max = n_max;
  g.stage_bytes = ((g.w_bytes + n_max * g.seg_stride) + 127) / 128 * 128;
  int ns = ring_bytes / g.stage_bytes;
  if (ns > kSMaxStages) ns = kSMaxStages;
  if (ns < 2) ns = 2;
  g.n_stages = ns;
  return g;
}

size_t stream_smem(const StreamGeom& g, int ys_rows) {
  return (size_t)g.n_stages * g.stage_bytes + (size_t)ys_rows * 16 * sizeof(float);
}

bool stream_small_ok(int T, int k) { return T <= kTokTile && T * k <= kSmallSlots; }

cudaError_t launch_stream_gateup(const ExpertParams& p, const RouteParams& rp, const StreamGeom& g,
                                 bool route, cudaStream_t st) {
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
