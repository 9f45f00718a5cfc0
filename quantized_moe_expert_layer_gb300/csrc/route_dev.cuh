// Device code of the routing step (router partial sums, top-k, dispatch),
// shared by the routing kernels and the small-batch expert kernels, which
// route a few tokens themselves.
#pragma once

#include <climits>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kRouterThreads = 256;
constexpr int kFinishThreads = 1024;
constexpr int kMaxKsplit = kMaxKsplitHost;  // router K slices at most

// ---------------------------------------------------------------- router logits
// ---------------------------------------------------------------- router logits
// Router partial sums of expert tile `tile` (16 experts), token group `group`
// (8 tokens) and K slice `ks` of p.ksplit, by the whole CTA (any number of
// warps); warp 0 writes them to p.partial.  smem: 8 x (K/ksplit + 8) bf16 +
// blockDim.x x 4 floats.
__device__ __forceinline__ void router_partials(const RouteParams& p, int tile, int group, int ks,
                                                uint4* smem_u4) {
  const int t0 = group * kTokTile;
  const int nwarps = blockDim.x >> 5;
  const int n = min(kTokTile, p.T - t0);
  const int C = p.H / 64;
  const int c_begin = C * ks / p.ksplit, c_end = C * (ks + 1) / p.ksplit;
  const int kbase = c_begin * 64, klen = (c_end - c_begin) * 64;
  const int stride = klen + 8;  // +16 bytes per row: conflict-free 16-byte reads
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem_u4);
  float* red = reinterpret_cast<float*>(xs + kTokTile * stride);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t = lane & 3;
  const int e0 = 16 * tile + gi, e1 = e0 + 8;
  const uint16_t* r0 = p.wr + (size_t)min(e0, p.E - 1) * p.H;
  const uint16_t* r1 = p.wr + (size_t)min(e1, p.E - 1) * p.H;
  // The router weights do not depend on earlier kernels: the warp's first
  // chunk is loaded, and the rest requested from L2, before waiting for them.
  auto load_a = [&](int c, uint32_t (&ra)[8], uint32_t (&rb)[8]) {
    const int kc = 64 * c + 16 * t;
    uint4 a00 = ldg_stream(r0 + kc), a01 = ldg_stream(r0 + kc + 8);
    uint4 a10 = ldg_stream(r1 + kc), a11 = ldg_stream(r1 + kc + 8);
    if (e0 >= p.E) a00 = a01 = make_uint4(0, 0, 0, 0);
    if (e1 >= p.E) a10 = a11 = make_uint4(0, 0, 0, 0);
    ra[0] = a00.x; ra[1] = a00.y; ra[2] = a00.z; ra[3] = a00.w;
    ra[4] = a01.x; ra[5] = a01.y; ra[6] = a01.z; ra[7] = a01.w;
    rb[0] = a10.x; rb[1] = a10.y; rb[2] = a10.z; rb[3] = a10.w;
    rb[4] = a11.x; rb[5] = a11.y; rb[6] = a11.z; rb[7] = a11.w;
  };
  uint32_t ra[8], rb[8];
  int c = c_begin + warp;
  if (c < c_end) load_a(c, ra, rb);
  for (int cc = c + nwarps; cc < c_end; cc += nwarps) {
    prefetch_l2(r0 + 64 * cc + 16 * t);
    prefetch_l2(r1 + 64 * cc + 16 * t);
  }
  // x (and everything written below) waits for the kernels before this one;
  // the next kernel may start once every CTA is past this point
  griddep_wait();
  griddep_launch();
  const bool write_xh = p.xh != nullptr && tile == 0;
  for (int i = threadIdx.x; i < n * (klen / 8); i += blockDim.x) {
    const int r = i / (klen / 8), v = i % (klen / 8);
    const size_t off = (size_t)(t0 + r) * p.H + kbase + 8 * v;
    const uint4 raw = *reinterpret_cast<const uint4*>(p.x + off);
    *reinterpret_cast<uint4*>(xs + r * stride + 8 * v) = raw;
    if (write_xh) {  // the f16 copy the expert kernels read (exact for |x| in [2^-14, 65504])
      const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t o[4];
      bool bad = false;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2 h = __floats2half2_rn(__uint_as_float(in[q] << 16),
                                            __uint_as_float(in[q] & 0xFFFF0000u));
        o[q] = *reinterpret_cast<const uint32_t*>(&h);
        bad |= f16x2_nonfinite(o[q]);
      }
      *reinterpret_cast<uint4*>(p.xh + off) = make_uint4(o[0], o[1], o[2], o[3]);
      if (bad && p.status) *p.status = kStatusRange;  // |x| beyond f16's range
    }
  }
  __syncthreads();

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (; c < c_end; c += nwarps) {
    const int kc = 64 * c + 16 * t;
    uint32_t xw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (gi < n) {
      const uint4* px = reinterpret_cast<const uint4*>(xs + gi * stride + (kc - kbase));
      const uint4 q0 = px[0], q1 = px[1];
      xw[0] = q0.x; xw[1] = q0.y; xw[2] = q0.z; xw[3] = q0.w;
      xw[4] = q1.x; xw[5] = q1.y; xw[6] = q1.z; xw[7] = q1.w;
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t a[4] = {ra[2 * w], rb[2 * w], ra[2 * w + 1], rb[2 * w + 1]};
      mma_bf16(acc, a, xw[2 * w], xw[2 * w + 1]);
    }
    if (c + nwarps < c_end) load_a(c + nwarps, ra, rb);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) red[(warp * 32 + lane) * 4 + i] = acc[i];
  __syncthreads();
  if (warp == 0) {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    for (int w = 0; w < nwarps; ++w)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[i] += red[(w * 32 + lane) * 4 + i];
    float* out = p.partial + (size_t)ks * p.T * p.E;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = (i < 2) ? e0 : e1, col = 2 * t + (i & 1);
      if (e < p.E && col < n) out[(size_t)(t0 + col) * p.E + e] = s[i];
    }
  }
}

// ---------------------------------------------------------------- top-k (one warp per token)
// The sigmoid router's score of a logit (fp32).
__device__ __forceinline__ float sigmoid_score(float l) { return 1.0f / (1.0f + expf(-l)); }

// Order-preserving map of an fp32 value to a uint32 key (larger value, larger
// key).  -0 and +0 compare equal, so both get the key of +0: a tie between
// them goes to the lower expert id like any other tie.
__device__ __forceinline__ uint32_t f32_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One top-k round over a lane's V slots: the largest key of the warp, ties to
// the lower expert id (slot i of lane l holds expert id[i]); the winner's slot
// is cleared.  Returns (key, expert id) of the winner in every lane.
template <int V>
__device__ __forceinline__ void warp_argmax_round(uint32_t (&key)[V], const int (&id)[V],
                                                  uint32_t& best, int& win) {
  uint32_t bk = key[0];
  int bi = id[0];
#pragma unroll
  for (int i = 1; i < V; ++i) {  // ids ascend with i, so '>' keeps the lower id on ties
    const bool take = key[i] > bk;
    bk = take ? key[i] : bk;
    bi = take ? id[i] : bi;
  }
  best = __reduce_max_sync(0xffffffffu, bk);
  win = (int)__reduce_min_sync(0xffffffffu, bk == best ? (uint32_t)bi : 0xFFFFFFFFu);
#pragma unroll
  for (int i = 0; i < V; ++i) key[i] = (id[i] == win) ? 0u : key[i];
}

// Logits of token t for experts e = e0 + lane + 32 i (i < V, e < e_end): the
// router's K-split slices added in order, then the bias; written to p.logits.
template <int V>
__device__ __forceinline__ void load_logits(const RouteParams& p, int t, int e0, int e_end,
                                            int lane, uint32_t (&key)[V], int (&id)[V],
                                            bool pub = true) {
  float v[V];
#pragma unroll
  for (int i = 0; i < V; ++i) v[i] = 0.f;
  if constexpr (V <= 4) {  // few slots: every slice requested at once
    float part[kMaxKsplit][V];
#pragma unroll
    for (int s = 0; s < kMaxKsplit; ++s)
#pragma unroll
      for (int i = 0; i < V; ++i) {  // written by other CTAs: read through L2
        const float* ps = p.partial + ((size_t)s * p.T + t) * p.E;
        part[s][i] = (s < p.ksplit && e0 + lane + 32 * i < e_end) ? __ldcg(ps + e0 + lane + 32 * i) : 0.f;
      }
#pragma unroll
    for (int s = 0; s < kMaxKsplit; ++s)  // slices added in order
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (s < p.ksplit) v[i] += part[s][i];
  } else {
    for (int s = 0; s < p.ksplit; ++s) {
      const float* ps = p.partial + ((size_t)s * p.T + t) * p.E;
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (e0 + lane + 32 * i < e_end) v[i] += __ldcg(ps + e0 + lane + 32 * i);
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = e0 + lane + 32 * i;
    id[i] = e;
    if (e < e_end) {
      float l = v[i];
      if (p.mode == ROUTER_SIGMOID) {  // score sigmoid(l); the bias moves the selection only
        if (pub && p.logits) p.logits[(size_t)t * p.E + e] = l;
        const float s = sigmoid_score(l);
        key[i] = f32_key(p.bias ? s + p.bias[e] : s);
      } else {
        if (p.bias) l = l + p.bias[e];
        if (pub && p.logits) p.logits[(size_t)t * p.E + e] = l;
        key[i] = f32_key(l);
      }
    } else {
      key[i] = 0u;  // below every real key
    }
  }
}

// Gates (lane j < k holds pick j): the softmax of the k selected logits, or
// for the sigmoid router the selected scores renormalised (each score
// recomputed from the router's K slices, in the order the selection used).
__device__ __forceinline__ void write_gates(const RouteParams& p, int t, int lane, uint32_t my_key,
                                            int my_i, int* sidx, float* sgates = nullptr,
                                            bool pub = true) {
  const int k = p.k;
  float ex;
  if (p.mode == ROUTER_SIGMOID) {
    ex = 0.f;
    if (lane < k) {
      float l = 0.f;
      for (int s = 0; s < p.ksplit; ++s) l += __ldcg(p.partial + ((size_t)s * p.T + t) * p.E + my_i);
      ex = sigmoid_score(l);
    }
  } else {
    const float my_v = key_f32(my_key);
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    ex = (lane < k) ? expf(my_v - top) : 0.f;
  }
  float sum = ex;
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    if (pub && p.idx) p.idx[(size_t)t * k + lane] = my_i;
    if (pub && p.gates) p.gates[(size_t)t * k + lane] = ex / sum;
    if (sidx) sidx[t * k + lane] = my_i;
    if (sgates) sgates[t * k + lane] = ex / sum;
  }
}

// Top-k of token t by one warp: k rounds of arg-max (largest logit, ties to
// the lower expert index), then the softmax of the k selected logits.
template <int V>
__device__ void topk_token_v(const RouteParams& p, int t, int lane, int* sidx,
                             float* sgates = nullptr, bool pub = true) {
  uint32_t key[V];
  int id[V];
  load_logits<V>(p, t, 0, p.E, lane, key, id, pub);
  uint32_t my_key = 0;
  int my_i = 0;
  for (int j = 0; j < p.k; ++j) {
    uint32_t best;
    int win;
    warp_argmax_round<V>(key, id, best, win);
    if (lane == j) {
      my_key = best;
      my_i = win;
    }
  }
  write_gates(p, t, lane, my_key, my_i, sidx, sgates, pub);
}

__device__ void topk_token(const RouteParams& p, int t, int lane, int* sidx,
                           float* sgates = nullptr, bool pub = true) {
  if (p.E <= 256)
    topk_token_v<8>(p, t, lane, sidx, sgates, pub);
  else if (p.E <= 512)
    topk_token_v<16>(p, t, lane, sidx, sgates, pub);
  else
    topk_token_v<32>(p, t, lane, sidx, sgates, pub);
}

// Top-k of token t by all warps of the CTA: each of the NW warps takes a
// contiguous share of the experts (V1 slots per lane) and finds its own k
// best; warp 0 then picks the k best of those NW*k candidates (V2 slots per
// lane, NW*k <= 32*V2) by the same rule, which gives the global top-k.
// ck / ci: NW * kMaxK entries of shared memory.
template <int V1, int V2>
__device__ void topk_token_cta(const RouteParams& p, int t, int* sidx, uint32_t* ck, int* ci,
                               float* sgates = nullptr, bool pub = true) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, k = p.k, NW = blockDim.x >> 5;
  const int q = (p.E + NW - 1) / NW;
  uint32_t key[V1];
  int id[V1];
  load_logits<V1>(p, t, warp * q, min(p.E, (warp + 1) * q), lane, key, id, pub);
  uint32_t c_key = 0;  // lane j keeps the warp's pick j
  int c_id = 0x7FFFFFFF;
  for (int j = 0; j < k; ++j) {
    uint32_t best;
    int win;
    warp_argmax_round<V1>(key, id, best, win);
    if (lane == j) {
      c_key = best;
      c_id = win;
    }
  }
  if (lane < k) {  // candidates packed: warp w's picks at w * k ...
    ck[warp * k + lane] = c_key;
    ci[warp * k + lane] = c_id;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t k2[V2];
    int i2[V2];
#pragma unroll
    for (int i = 0; i < V2; ++i) {  // candidate c = lane + 32 i
      const int c = lane + 32 * i;
      const bool ok = c < NW * k;
      k2[i] = ok ? ck[c] : 0u;
      i2[i] = ok ? ci[c] : 0x7FFFFFFF;
    }
    // order each lane's slots by expert id so that ties keep the lower id
#pragma unroll
    for (int a = 0; a < V2; ++a)
#pragma unroll
      for (int b = a + 1; b < V2; ++b) {
        const bool sw = i2[b] < i2[a];
        const uint32_t tk = sw ? k2[b] : k2[a];
        const int ti = sw ? i2[b] : i2[a];
        k2[b] = sw ? k2[a] : k2[b];
        i2[b] = sw ? i2[a] : i2[b];
        k2[a] = tk;
        i2[a] = ti;
      }
    uint32_t my_key = 0;
    int my_i = 0;
    for (int j = 0; j < k; ++j) {
      uint32_t best;
      int win;
      warp_argmax_round<V2>(k2, i2, best, win);
      if (lane == j) {
        my_key = best;
        my_i = win;
      }
    }
    write_gates(p, t, lane, my_key, my_i, sidx, sgates, pub);
  }
  __syncthreads();
}

// ---------------------------------------------------------------- dispatch (one CTA of 1024 threads)
// exclusive scan of v over the block; *total gets the sum
__device__ int block_excl_scan(int v, int* sc, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sc[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = (lane < (int)(blockDim.x >> 5)) ? sc[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sc[32 + lane] = s;  // inclusive warp-total prefix
  }
  __syncthreads();
  const int before = (w > 0) ? sc[32 + w - 1] : 0;
  *total = sc[32 + (blockDim.x >> 5) - 1];
  const int r = before + x - v;
  __syncthreads();
  return r;
}

__device__ __forceinline__ int checked_expert(const RouteParams& p, int e) {
  if (e < 0 || e >= p.E) {
    *p.status = kStatusInvalid;
    return 0;
  }
  return e;
}

// The shared rows' tokens and the work entries, by every thread of the block
// (blockDim.x >= E): thread e < E holds expert e's slot count c and first row
// excl.  Routed entries: ceil(c / 8) per expert, expert-major; tensor-core
// entries (when p.tc_entries): ceil(c / 128).
__device__ void write_entries(const RouteParams& p, int c, int excl, int* sc) {
  const int tid = threadIdx.x, E = p.E, S = p.T * p.k;
  for (int i = tid; i < p.T; i += blockDim.x) p.row_token[S + i] = i;
  const int nch = (tid < E) ? (c + kTokTile - 1) / kTokTile : 0;
  int n_total;
  const int ebase = block_excl_scan(nch, sc, &n_total);
  if (tid < E)
    for (int i = 0; i < nch; ++i)
      p.entries[ebase + i] = make_int4(tid, excl + kTokTile * i, min(kTokTile, c - kTokTile * i), 0);
  if (tid == 0) *p.n_entries = n_total;
  if (p.tc_entries) {
    const int ntc = (tid < E) ? (c + kTcMaxN - 1) / kTcMaxN : 0;
    int tc_total;
    const int tbase = block_excl_scan(ntc, sc, &tc_total);
    if (tid < E)
      for (int i = 0; i < ntc; ++i)
        p.tc_entries[tbase + i] = make_int4(tid, excl + kTcMaxN * i, min(kTcMaxN, c - kTcMaxN * i), 0);
    if (tid == 0) *p.n_tc_entries = tc_total;
  }
}

__device__ void dispatch_block(const RouteParams& p, int* hist, int* sc) {
  const int S = p.T * p.k, E = p.E;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, NW = blockDim.x >> 5;
  for (int i = tid; i < NW * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int per = (S + NW - 1) / NW;
  const int sb = min(S, w * per), se = min(S, sb + per);
  for (int s = sb + lane; s < se; s += 32) atomicAdd(&hist[w * E + checked_expert(p, p.idx[s])], 1);
  __syncthreads();
  int c = 0;
  if (tid < E)
    for (int ww = 0; ww < NW; ++ww) c += hist[ww * E + tid];
  int total;
  const int excl = block_excl_scan(tid < E ? c : 0, sc, &total);
  if (tid < E) {
    p.counts[tid] = c;
    p.offsets[tid] = excl;
    int run = excl;
    for (int ww = 0; ww < NW; ++ww) {
      const int h = hist[ww * E + tid];
      hist[ww * E + tid] = run;
      run += h;
    }
  }
  if (tid == 0) p.offsets[E] = total;
  __syncthreads();
  // stable placement: each warp walks its slot range in order, 32 at a time
  for (int base = sb; base < se; base += 32) {
    const int s = base + lane;
    const bool valid = s < se;
    const int e = valid ? checked_expert(p, p.idx[s]) : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (valid) {
      const int pos = hist[w * E + e] + __popc(peers & lanemask_lt());
      p.perm[pos] = s;
      p.inv[s] = pos;
      p.row_token[pos] = s / p.k;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) hist[w * E + e] += __popc(peers);
    __syncwarp();
  }
  write_entries(p, c, excl, sc);
}

// Dispatch of T <= 64 tokens whose k picks are distinct (the top-k's), by
// one CTA with a thread per expert: expert e's rows are its tokens in
// ascending order (its slots in slot order), so slot (t, j) of expert e lands
// at offsets[e] + (tokens below t in e's 64-bit token mask).  The rows come
// out the same as dispatch_block's.  Ends synchronised.
__device__ void dispatch_block_t64(const RouteParams& p, unsigned long long* mask, int* sc) {
  const int E = p.E, k = p.k, S = p.T * k, tid = threadIdx.x;
  int* off = reinterpret_cast<int*>(mask + E);
  for (int e = tid; e < E; e += blockDim.x) mask[e] = 0ull;
  __syncthreads();
  for (int s = tid; s < S; s += blockDim.x)
    atomicOr(&mask[checked_expert(p, p.idx[s])], 1ull << (s / k));
  __syncthreads();
  const int c = tid < E ? __popcll(mask[tid]) : 0;
  int total;
  const int excl = block_excl_scan(c, sc, &total);
  if (tid < E) {
    p.counts[tid] = c;
    p.offsets[tid] = excl;
    off[tid] = excl;
  }
  if (tid == 0) p.offsets[E] = total;
  __syncthreads();
  for (int s = tid; s < S; s += blockDim.x) {
    const int e = checked_expert(p, p.idx[s]), t = s / k;
    const int pos = off[e] + __popcll(mask[e] & ((1ull << t) - 1ull));
    p.perm[pos] = s;
    p.inv[s] = pos;
    p.row_token[pos] = t;
  }
  write_entries(p, c, excl, sc);
}

// slots of the few-token path (T * k at most)// slots of the few-token path (T * k at most)
constexpr int kSmallSlots = 256;

// ---------------------------------------------------------------- routing of a few tokens by one CTA
// For T <= kTokTile tokens no expert can receive more than kTokTile slots, so
// every routed expert is exactly one work entry.  The small-batch expert
// kernels route in every CTA from the router's partial sums (a few KB read
// through L2) instead of waiting for a separate routing kernel.
struct SmallRoute {
  int4 entries[kSmallSlots];  // {expert, first row, tokens, 0}, expert order
  int inv[kSmallSlots];       // row of each slot
  int row_token[kSmallSlots + kTokTile];
  float gates[kSmallSlots];
  int sidx[kSmallSlots];      // expert of each slot
  int lt[kSmallSlots];        // per slot: slots with a smaller expert id
  int cnt[kSmallSlots];       // per slot: slots with the same expert
  int lead[kSmallSlots];      // per slot: first slot of its expert
  uint32_t ck[16 * kMaxK];    // per-warp top-k candidates (T == 1)
  int ci[16 * kMaxK];
  int n_entries;
};

// Top-k, gates and the stable expert-major dispatch of T <= kTokTile tokens,
// T * k <= min(kSmallSlots, blockDim.x), by every thread of the block (at most
// 16 warps); results in r, and, when `pub`, in the global outputs of p
// (logits, idx, gates, perm, inv, row_token, entries, n_entries).  Row of slot
// s: pos(s) = #{q : e_q < e_s} + #{q < s : e_q == e_s}, which is the dispatch
// of dispatch_block.  Ends synchronised.
template <int V2>
__device__ void topk_one_token_cta(const RouteParams& p, SmallRoute& r, bool pub) {
  const int NW = blockDim.x >> 5, q = (p.E + NW - 1) / NW;
  if (q <= 32)
    topk_token_cta<1, V2>(p, 0, r.sidx, r.ck, r.ci, r.gates, pub);
  else if (q <= 64)
    topk_token_cta<2, V2>(p, 0, r.sidx, r.ck, r.ci, r.gates, pub);
  else
    topk_token_cta<4, V2>(p, 0, r.sidx, r.ck, r.ci, r.gates, pub);
}

__device__ __noinline__ void route_small_cta(const RouteParams& p, SmallRoute& r, bool pub) {
  const int T = p.T, k = p.k, S = T * k;
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31, NW = nt >> 5;
  if (T == 1) {  // all warps share the token: E / NW experts each, then one merge
    if (NW * k <= 32 * 3)
      topk_one_token_cta<3>(p, r, pub);
    else if (NW * k <= 32 * 9)
      topk_one_token_cta<9>(p, r, pub);
    else
      topk_one_token_cta<16>(p, r, pub);
  } else {  // one warp per token
    for (int t = warp; t < T; t += NW) topk_token(p, t, lane, r.sidx, r.gates, pub);
    __syncthreads();
  }
  if (T == 1) {  // k distinct experts, one row each: the entries are the picks sorted by id
    if (warp == 0) {
      const int e = lane < k ? r.sidx[lane] : INT_MAX;
      int rank = 0;
      for (int l = 0; l < k; ++l) rank += __shfl_sync(0xffffffffu, e, l) < e;
      if (lane < k) {
        r.inv[lane] = rank;
        r.row_token[rank] = 0;
        r.entries[rank] = make_int4(e, rank, 1, 0);
        if (pub) {
          p.perm[rank] = lane;
          p.inv[lane] = rank;
          p.row_token[rank] = 0;
          p.entries[rank] = make_int4(e, rank, 1, 0);
        }
      }
      if (lane == 0) {
        r.row_token[k] = 0;  // the shared expert's row
        r.n_entries = k;
        if (pub) {
          p.row_token[k] = 0;
          *p.n_entries = k;
        }
      }
    }
    __syncthreads();
    return;
  }
  int is_lead = 0;
  for (int s = tid; s < S; s += nt) {
    const int e = r.sidx[s];
    int lt = 0, before = 0, cnt = 0;
    for (int q = 0; q < S; ++q) {
      const int f = r.sidx[q];
      lt += f < e;
      cnt += f == e;
      before += (f == e) & (q < s);
    }
    const int pos = lt + before;
    r.inv[s] = pos;
    r.row_token[pos] = s / k;
    r.lt[s] = lt;
    r.cnt[s] = cnt;
    r.lead[s] = before == 0;
    is_lead = before == 0;
    if (pub) {
      p.perm[pos] = s;
      p.inv[s] = pos;
      p.row_token[pos] = s / k;
    }
  }
  for (int t = tid; t < T; t += nt) {
    r.row_token[S + t] = t;
    if (pub) p.row_token[S + t] = t;
  }
  const int n_ent = __syncthreads_count(is_lead);  // one slot per thread at most
  for (int s = tid; s < S; s += nt) {
    if (!r.lead[s]) continue;
    const int e = r.sidx[s];
    int d = 0;
    for (int q = 0; q < S; ++q) d += r.lead[q] & (r.sidx[q] < e);
    const int4 en = make_int4(e, r.lt[s], r.cnt[s], 0);
    r.entries[d] = en;
    if (pub) p.entries[d] = en;
  }
  if (tid == 0) {
    r.n_entries = n_ent;
    if (pub) *p.n_entries = n_ent;
  }
  __syncthreads();
}

// counts[E] and offsets[E + 1] of a routing held in r (diagnostic outputs).
__device__ __noinline__ void publish_counts(const RouteParams& p, const SmallRoute& r) {
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    int c = 0, off = 0;
    for (int d = 0; d < r.n_entries; ++d) {
      const int4 en = r.entries[d];
      c += en.x == e ? en.z : 0;
      off += en.x < e ? en.z : 0;
    }
    if (p.counts) p.counts[e] = c;
    if (p.offsets) p.offsets[e] = off;
  }
  if (threadIdx.x == 0 && p.offsets) p.offsets[p.E] = p.T * p.k;
}

}  // namespace
}  // namespace moe
