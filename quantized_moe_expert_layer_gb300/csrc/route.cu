// Routing: router logits, softmax / top-k / renormalise, and the expert-sorted
// dispatch (counts, offsets, stable permutation, per-expert work entries).
//
// The router and top-k are the "router_top10" kernel of "Strata on an Intel
// Arc", "The engine itself on Intel: the SYCL port"; grouping tokens by expert
// on the device instead of the host follows that page's device-built plan
// ("resident_plan", "Decode round 2"), where host grouping cost 9% of prompt
// time.  Readings where the pages are silent: logit = (x . Wr_e) + bias_e with
// the dot product in fp32; top-k on the logits (softmax is monotone), ties to
// the lower expert index; the k gates are the softmax over the k selected
// logits (equal to softmax -> top-k -> renormalise); dispatch order is
// expert-major, then slot id t*k + j (stable).
#include <climits>

#include "common.cuh"
#include "kernels.cuh"
#include "route_dev.cuh"

namespace moe {
namespace {

// grid (ceil(E/16) expert tiles, ceil(T/8) token groups, ksplit); the 8 warps
// split the CTA's 64-column chunks; tensor cores take bf16 x bf16 -> fp32.
// Each (ksplit slice, token, expert) partial sum goes to p.partial; the top-k
// step adds the slices in a fixed order.
__global__ void __launch_bounds__(kRouterThreads) router_kernel(RouteParams p) {
  extern __shared__ uint4 smem_u4[];
  router_partials(p, blockIdx.x, blockIdx.y, blockIdx.z, smem_u4);
}

// One token per CTA: the 8 warps take E/8 experts each and find their k best,
// warp 0 merges the 8k candidates (topk_token_cta); a warp per token would
// run k arg-max rounds over E/32 slots per lane, a longer serial chain.
template <int V1, int V2>
__device__ __forceinline__ void topk_cta_task(const RouteParams& p, uint32_t* ck, int* ci) {
  topk_token_cta<V1, V2>(p, blockIdx.x, nullptr, ck, ci);
}

__global__ void __launch_bounds__(256) topk_kernel(RouteParams p) {
  griddep_launch();
  griddep_wait();
  __shared__ uint32_t ck[8 * kMaxK];
  __shared__ int ci[8 * kMaxK];
  const int q = (p.E + 7) / 8;  // experts per warp (E <= 1024: q <= 128)
  if (8 * p.k <= 96) {
    if (q <= 32) topk_cta_task<1, 3>(p, ck, ci);
    else if (q <= 64) topk_cta_task<2, 3>(p, ck, ci);
    else topk_cta_task<4, 3>(p, ck, ci);
  } else {
    if (q <= 32) topk_cta_task<1, 8>(p, ck, ci);
    else if (q <= 64) topk_cta_task<2, 8>(p, ck, ci);
    else topk_cta_task<4, 8>(p, ck, ci);
  }
}

// Top-k of many tokens (T >= kTopkWarpMinT): one warp per token, 8 tokens per
// CTA; each lane holds E/32 logits, all requested at once, and takes k
// arg-max rounds (topk_token).  Same picks, order and gates as topk_kernel.
constexpr int kTopkWarpMinT = 1024;
__global__ void __launch_bounds__(256) topk_warp_kernel(RouteParams p) {
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t < p.T) topk_token(p, t, threadIdx.x & 31, nullptr);
}

// Top-k of one token per CTA (the two levels of topk_kernel over blockDim / 32
// warps), then the dispatch by the CTA that finishes last: every CTA makes its
// picks visible and takes a ticket; the one that draws the last ticket runs
// dispatch_block over all the picks and clears the ticket for the next
// forward.  No CTA waits for another.  One launch instead of two for
// 16 < T with T*k <= kDispOneCtaMax and E <= 512 (dispatch_block needs a
// thread per expert).
template <int V2>
__global__ void __launch_bounds__(512) topk_dispatch_kernel(RouteParams p) {
  griddep_launch();
  griddep_wait();
  extern __shared__ int smem_td[];  // keys, ids [warps x kMaxK each], scan scratch [64], histograms
  const int NW = blockDim.x >> 5;
  uint32_t* ck = reinterpret_cast<uint32_t*>(smem_td);
  int* ci = smem_td + NW * kMaxK;
  int* sc = ci + NW * kMaxK;
  __shared__ int last;
  topk_token_cta<1, V2>(p, blockIdx.x, nullptr, ck, ci);  // (ends synchronised)
  __threadfence();  // this CTA's picks, before its ticket
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(p.ticket, 1) == p.T - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();  // every other CTA's picks, after the last ticket
  if (p.T <= 64)  // (the top-k's picks of a token are distinct)
    dispatch_block_t64(p, reinterpret_cast<unsigned long long*>(sc + 64), sc);
  else
    dispatch_block(p, sc + 64, sc);
  if (threadIdx.x == 0) *p.ticket = 0;
}

__global__ void __launch_bounds__(kFinishThreads) route_finish_kernel(RouteParams p, int do_topk) {
  griddep_launch();
  griddep_wait();
  extern __shared__ int smem_i[];
  if (do_topk) {
    for (int t = threadIdx.x >> 5; t < p.T; t += kFinishThreads / 32)
      topk_token(p, t, threadIdx.x & 31, nullptr);
    __syncthreads();
  }
  dispatch_block(p, smem_i + 64, smem_i);
}

// ---------------------------------------------------------------- dispatch over several CTAs
// For many slots the one-CTA dispatch walks them serially; here CTA b of the
// count and place kernels takes slots [b * kDispChunk, (b + 1) * kDispChunk)
// (one per thread), and one CTA scans the per-chunk counts in between.  The
// rows come out the same as dispatch_block's: expert-major, ascending slot
// within an expert.

// Per-chunk expert counts into p.blk[b * E + e].
__global__ void __launch_bounds__(kDispChunk) dispatch_count_kernel(RouteParams p) {
  griddep_launch();
  griddep_wait();
  extern __shared__ int hist_c[];  // [E]
  const int b = blockIdx.x, tid = threadIdx.x, E = p.E, S = p.T * p.k;
  for (int i = tid; i < E; i += blockDim.x) hist_c[i] = 0;
  __syncthreads();
  const int s = b * kDispChunk + tid;
  if (s < S) atomicAdd(&hist_c[checked_expert(p, p.idx[s])], 1);
  __syncthreads();
  for (int i = tid; i < E; i += blockDim.x) p.blk[(size_t)b * E + i] = hist_c[i];
}

// Stable placement of chunk b (one slot per thread): row = offsets[e] + rows
// of e in earlier chunks + rows of e in earlier warps of this chunk + rank
// among the warp's lanes.  Every CTA sums the per-chunk counts itself
// (thread e < E reads expert e's column: its rows in all chunks and in the
// chunks before b; 16 loads in flight) and scans them over the experts, so no
// single CTA walks the chunks; CTA 0 also writes counts, offsets, the work
// entries and the shared expert's rows.  Needs blockDim.x >= E.
__global__ void __launch_bounds__(kDispChunk) dispatch_place_kernel(RouteParams p, int nb) {
  griddep_launch();
  griddep_wait();
  extern __shared__ int hist_p[];  // [warps][E], then 64 ints of scan scratch
  const int b = blockIdx.x, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int E = p.E, S = p.T * p.k, NW = blockDim.x >> 5;
  int* sc = hist_p + NW * E;
  int before = 0, total = 0;
  if (tid < E) {
    for (int b0 = 0; b0 < nb; b0 += 16) {
      int v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = (b0 + u < nb) ? p.blk[(size_t)(b0 + u) * E + tid] : 0;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        before += (b0 + u < b) ? v[u] : 0;
        total += v[u];
      }
    }
  }
  int all;
  const int excl = block_excl_scan(tid < E ? total : 0, sc, &all);
  if (b == 0) {  // (uniform in the CTA: write_entries synchronises every thread)
    if (tid < E) {
      p.counts[tid] = total;
      p.offsets[tid] = excl;
    }
    if (tid == 0) p.offsets[E] = all;
    write_entries(p, total, excl, sc);
  }
  for (int i = tid; i < NW * E; i += blockDim.x) hist_p[i] = 0;
  __syncthreads();
  const int s = b * kDispChunk + tid;
  const bool valid = s < S;
  const int e = valid ? checked_expert(p, p.idx[s]) : -1 - lane;
  const uint32_t peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & lanemask_lt());
  if (valid && lane == __ffs(peers) - 1) hist_p[w * E + e] = __popc(peers);
  __syncthreads();
  if (tid < E) {
    const int x = tid;
    int run = excl + before;
    for (int ww = 0; ww < NW; ++ww) {
      const int v = hist_p[ww * E + x];
      hist_p[ww * E + x] = run;
      run += v;
    }
  }
  __syncthreads();
  if (valid) {
    const int pos = hist_p[w * E + e] + rank;
    p.perm[pos] = s;
    p.inv[s] = pos;
    p.row_token[pos] = s / p.k;
  }
}

// The f16 copy of x the expert kernels read: exact for |x| in [2^-14, 65504]
// (bf16 has 8 significant bits, f16 11); an element beyond 65504 (or not
// finite) records MOE_ERANGE in the status word.
__global__ void convert_x_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ xh, long n8,
                                 int* status) {
  bool bad = false;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long)gridDim.x * blockDim.x) {
    const uint4 raw = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 h = __floats2half2_rn(__uint_as_float(in[q] << 16),
                                          __uint_as_float(in[q] & 0xFFFF0000u));
      o[q] = *reinterpret_cast<const uint32_t*>(&h);
      bad |= f16x2_nonfinite(o[q]);
    }
    reinterpret_cast<uint4*>(xh)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (bad) *status = kStatusRange;
}

}  // namespace

cudaError_t launch_convert_x(const uint16_t* x, uint16_t* xh, long n, int* status, cudaStream_t st) {
  const long n8 = n / 8;
  long blocks = (n8 + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  convert_x_kernel<<<(int)blocks, 256, 0, st>>>(x, xh, n8, status);
  return cudaGetLastError();
}

// K slices of the router: about 128 CTAs up to 16 tokens (their top-k reads
// the slices with a warp per token, a serial loop over them), about 1024 above
// (the CTA-per-token top-k requests every slice at once; each router warp
// then has one or two 64-column chunks instead of a serial chain of them)
int router_ksplit(int T, int H, int E) {
  const int tiles = (E + 15) / 16, groups = (T + kTokTile - 1) / kTokTile;
  const int C = H / 64, target = T <= 2 * kTokTile ? 128 : 1024;
  int ks = (target + tiles * groups - 1) / (tiles * groups);
  if (ks > kMaxKsplitHost) ks = kMaxKsplitHost;
  if (ks > C) ks = C;
  // a slice's 8 staged token rows must fit the kernel's shared memory
  // (launch_router: 8 x (slice + 8) bf16 + 4 KB <= 200 KB): at most 12288 columns
  const int min_ks = (H + 12287) / 12288;
  if (ks < min_ks) ks = min_ks;
  if (ks < 1) ks = 1;
  return ks;
}

size_t route_finish_smem(int E) { return (size_t)(64 + (kFinishThreads / 32) * E) * sizeof(int); }

cudaError_t launch_router(const RouteParams& p, cudaStream_t st, bool pdl) {
  const int C = p.H / 64;
  const int max_klen = ((C + p.ksplit - 1) / p.ksplit) * 64;
  const size_t smem = (size_t)kTokTile * (max_klen + 8) * 2 + kRouterThreads * 4 * sizeof(float);
  dim3 grid((p.E + 15) / 16, (p.T + kTokTile - 1) / kTokTile, p.ksplit);
  // with pdl, launched early: only the weight reads run before the previous kernels finish
  return launch_k(router_kernel, grid, dim3(kRouterThreads), smem, st, pdl, p);
}

cudaError_t launch_topk(const RouteParams& p, bool pdl, cudaStream_t st) {
  if (p.T >= kTopkWarpMinT)
    return launch_k(topk_warp_kernel, dim3((p.T + 7) / 8), dim3(256), 0, st, pdl, p);
  return launch_k(topk_kernel, dim3(p.T), dim3(256), 0, st, pdl, p);
}

cudaError_t launch_route_finish(const RouteParams& p, bool do_topk, bool pdl, cudaStream_t st) {
  return launch_k(route_finish_kernel, dim3(1), dim3(kFinishThreads), route_finish_smem(p.E), st,
                  pdl, p, do_topk ? 1 : 0);
}

int dispatch_launches(int S) { return S > kDispOneCtaMax ? 2 : 1; }

// a thread per expert (at least 8 warps), at most 512
static int topk_dispatch_threads(int E) { return E <= 256 ? 256 : 512; }

bool topk_dispatch_ok(int T, int k, int E) {
  return T > 16 && T < kTopkWarpMinT && (long)T * k <= kDispOneCtaMax && E <= 512;
}

cudaError_t launch_topk_dispatch(const RouteParams& p, bool pdl, cudaStream_t st) {
  const int threads = topk_dispatch_threads(p.E), NW = threads / 32;
  const size_t smem = ((size_t)2 * NW * kMaxK + 64 + (size_t)NW * p.E) * sizeof(int);
  // warp 0 merges NW * k candidates, V2 per lane
  if (NW * p.k <= 96)
    return launch_k(topk_dispatch_kernel<3>, dim3(p.T), dim3(threads), smem, st, pdl, p);
  if (NW * p.k <= 256)
    return launch_k(topk_dispatch_kernel<8>, dim3(p.T), dim3(threads), smem, st, pdl, p);
  return launch_k(topk_dispatch_kernel<16>, dim3(p.T), dim3(threads), smem, st, pdl, p);
}

cudaError_t launch_dispatch(const RouteParams& p, bool pdl, cudaStream_t st) {
  const int S = p.T * p.k;
  if (S <= kDispOneCtaMax) return launch_route_finish(p, false, pdl, st);
  const int nb = (S + kDispChunk - 1) / kDispChunk;
  cudaError_t e = launch_k(dispatch_count_kernel, dim3(nb), dim3(kDispChunk), p.E * sizeof(int),
                           st, pdl, p);
  if (e == cudaSuccess)
    e = launch_k(dispatch_place_kernel, dim3(nb), dim3(kDispChunk),
                 ((size_t)(kDispChunk / 32) * p.E + 64) * sizeof(int), st, pdl, p, nb);
  return e;
}

cudaError_t route_kernels_init() {
  cudaError_t e = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       200 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(dispatch_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           ((kDispChunk / 32) * kMaxE + 64) * (int)sizeof(int));
  if (e != cudaSuccess) return e;
  for (auto f : {(const void*)topk_dispatch_kernel<3>, (const void*)topk_dispatch_kernel<8>,
                 (const void*)topk_dispatch_kernel<16>}) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)((2 * 16 * kMaxK + 64 + 16 * 512) * sizeof(int)));
    if (e != cudaSuccess) return e;
  }
  return cudaFuncSetAttribute(route_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)route_finish_smem(kMaxE));
}

}  // namespace moe
