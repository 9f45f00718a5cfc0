// Prefill path: grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05 kind::f16, fp32 accumulators in tensor memory).
//
// Per work item (expert e, 128-row block of W, up to 128 tokens routed to e):
//   D[128 x N] (TMEM, fp32) = sum over K of A[128 x 64] . B[N x 64]^T
// A = the weights, dequantised exactly to f16 (e2m1 code * e4m3 block scale is
// an f16) by four producer warps from the packed NVFP4 tiles and written to
// shared memory in the 128-byte-swizzled K-major layout the MMA reads; B = the
// token rows (x, gathered through the dispatch permutation and converted from
// bf16 to f16, or the SwiGLU output a), written the same way.  One thread
// issues the MMAs; stages are handed over with mbarriers; tcgen05.commit frees
// a stage when the MMAs reading it are done.  The epilogue warps read D from
// TMEM (warp w owns lanes 32w..32w+31) and apply the fp32 tensor scale and
// SwiGLU (gate/up) or write y rows (down).
//
// MODE 2 is the router for large T: a plain bf16 GEMM, logits[t][e] =
// x[t] . Wr[e], with 128 experts as M and 128 tokens as N; both operands are
// copied straight into the swizzled stages (no dequantisation).
//
// The weights stay the M operand and the token count the N operand (N is 80 on
// average for 4096 tokens over 512 experts), as the survey of the prompt paths
// suggests: experts with few tokens keep the decoded weights as the wide side.
// Every wait is bounded: on a timeout the kernel records MOE_ETIMEOUT in the
// status word, stops issuing work, waits (bounded) for its MMAs, frees its
// TMEM and returns.
#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"
#include "layout.cuh"

namespace moe {
namespace {

constexpr int kTcM = 128;            // rows of W per work item
constexpr int kTcK = 64;             // K per pipeline stage (one packed chunk)
constexpr int kTcStages = 6;
constexpr int kTcLookahead = kTcStages - 2;  // chunks in flight; one stage of slack for the MMAs
constexpr int kTcProducers = 256;    // warps 0-7: producers, then epilogue
constexpr int kTcThreads = 288;      // + warp 8: TMEM allocation and MMA issue
constexpr int kTcAStageBytes = kTcM * kTcK * 2;     // 16 KB of dequantised f16 weights
constexpr int kTcRawStageBytes = 8 * 512;           // 4 KB of packed codes (8 tiles)
constexpr int kTcBStageBytes = kTcMaxN * kTcK * 2;  // 16 KB of f16 token rows

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {  // one full warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // the same warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// arrive on `bar` once every MMA issued so far by this thread has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 TMEM lanes (one per thread of the warp) x 32 consecutive fp32 columns
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the stage bases are 1024-byte aligned).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: D fp32, A and B f16, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// byte offset of the 16-byte chunk c16 of row r in a 128B-swizzled K-major tile
__device__ __forceinline__ uint32_t swz(int r, int c16) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c16 ^ (r & 7)) << 4));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

struct TcShared {
  uint64_t full[kTcStages];
  uint64_t empty[kTcStages];
  uint64_t acc_full;
  uint32_t tmem_base;
  int abort;
  int tok[kTcMaxN];
};

// Work item y of a tc launch: leading shared-expert items, then routed ones.
__device__ __forceinline__ bool tc_entry(const ExpertParams& p, int y, int& expert, int& row, int& n) {
  const int S = p.T * p.k;
  if (y < p.nsh_tc) {
    expert = p.E;
    row = S + kTcMaxN * y;
    n = min(kTcMaxN, p.T - kTcMaxN * y);
    return true;
  }
  const int r = y - p.nsh_tc;
  if (r >= *p.n_tc_entries) return false;
  const int4 e = p.tc_entries[r];
  expert = e.x;
  row = e.y;
  n = e.z;
  if (expert < 0 || expert >= p.E || n < 1 || n > kTcMaxN || row < 0 || row + n > S) {
    *p.status = -1;  // MOE_EINVAL
    return false;
  }
  return true;
}

// The shared skeleton of the GEMMs.  MODE 0: gate/up + SwiGLU -> abuf;
// MODE 1: down -> ybuf; MODE 2: router logits (bf16 x bf16) -> logits_out.
//
// Producer thread u (of 256) owns packed vector u of each chunk: tile u/32,
// lane u%32 of the 16-row tile layout, i.e. rows 16*(u/32) + (u%32)/4 (+8) and
// 16 columns.  Chunk c's raw codes and token rows are copied with cp.async
// kTcLookahead chunks ahead; at chunk c the thread waits for its own copies,
// dequantises its vector into the swizzled A stage, fences the async proxy and
// arrives on full[c % stages].
template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(ExpertParams p) {
  griddep_wait();
  int expert, row0, n;
  if (MODE == 2) {  // token tile blockIdx.y of the router GEMM
    expert = 0;
    row0 = kTcMaxN * blockIdx.y;
    n = min(kTcMaxN, p.T - row0);
    if (n <= 0) return;
  } else if (!tc_entry(p, blockIdx.y, expert, row0, n)) {
    return;
  }
  extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~(uintptr_t)1023);
  const int n_pad = (n + 15) & ~15;
  const int b_stage = n_pad * kTcK * 2;  // multiple of 2 KB: stages stay 1024-byte aligned
  uint8_t* A = base;
  uint8_t* B = A + kTcStages * kTcAStageBytes;
  uint8_t* RAW = B + kTcStages * kTcBStageBytes;
  TcShared* sh = reinterpret_cast<TcShared*>(RAW + kTcStages * kTcRawStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.T * p.k;
  const int K = MODE == 1 ? p.I : p.H;
  const int KC = K / kTcK;
  const int mb = blockIdx.x;
  const uint32_t ncols = n_pad <= 32 ? 32 : (n_pad <= 64 ? 64 : 128);
  const uint8_t* eb = p.arena + (size_t)expert * p.expert_bytes;
  const MatGeom g = mat_geom(FMT_NVFP4, K);

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&sh->full[s], kTcProducers);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->acc_full, 1);
    sh->abort = 0;
    mbar_init_fence();
  }
  for (int i = tid; i < n_pad; i += kTcThreads) {
    int tk = 0;
    if (i < n) tk = (MODE == 0) ? ((expert == p.E) ? row0 - S + i : p.row_token[row0 + i]) : row0 + i;
    sh->tok[i] = tk;  // MODE 0 / 2: token index into x; MODE 1: row of abuf
  }
  // token-row padding stays zero in every stage (cp.async never writes it)
  for (int i = tid; i < kTcStages * (n_pad - n) * 8; i += kTcThreads) {
    const int st = i / ((n_pad - n) * 8), rem = i % ((n_pad - n) * 8);
    const int r = n + rem / 8, c16 = rem % 8;
    *reinterpret_cast<uint4*>(B + st * b_stage + swz(r, c16)) = make_uint4(0, 0, 0, 0);
  }
  if (warp == 8) tmem_alloc(&sh->tmem_base, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp < 8) {
    // ---------------------------------------------------------------- producers
    const int u = tid, ti = u >> 5, ln = u & 31, gi = ln >> 2, t = ln & 3;
    const uint8_t* tile = (MODE == 0) ? eb + (size_t)(8 * mb + ti) * p.gu_tile_bytes
                                      : eb + p.gu_bytes + (size_t)(8 * mb + ti) * p.dn_tile_bytes;
    const uint16_t* bsrc = (MODE == 0) ? p.xh : (MODE == 1 ? p.abuf : p.x);
    const int bld = (MODE == 1) ? p.I : p.H;
    const uint16_t* arow = p.wr + (size_t)kTcM * mb * p.H;  // MODE 2: 128 router rows
    // ask L2 for everything this CTA will read
    if (MODE == 2) {
      for (int i = tid; i < kTcM * (K / 64); i += kTcProducers)
        prefetch_l2(arow + (size_t)(i / (K / 64)) * p.H + 64 * (i % (K / 64)));
    } else {
      for (int s = 0; s < g.nsc; ++s)
        for (int j = 0; j <= sc_units(g, s); ++j)
          prefetch_l2(tile + (size_t)s * g.sc_bytes + 512 * j + 16 * ln);
    }
    for (int i = tid; i < n * (K / 64); i += kTcProducers)
      prefetch_l2(bsrc + (size_t)sh->tok[i / (K / 64)] * bld + 64 * (i % (K / 64)));
    const uint32_t a_s = smem_u32(A), b_s = smem_u32(B), raw_s = smem_u32(RAW);
    auto issue = [&](int c) {  // chunk c's copies into stage c % stages
      const int stage = c % kTcStages, s = c >> 3, j = c & 7;
      if (MODE == 2) {  // router rows straight into the swizzled A stage
        for (int v = tid; v < kTcM * 8; v += kTcProducers) {
          const int r = v >> 3, c16 = v & 7;
          cp_async16(a_s + stage * kTcAStageBytes + swz(r, c16),
                     arow + (size_t)r * p.H + c * kTcK + 8 * c16);
        }
      } else {
        cp_async16(raw_s + stage * kTcRawStageBytes + 16 * u,
                   tile + (size_t)s * g.sc_bytes + 512 * (1 + j) + 16 * ln);
      }
      const uint32_t bs = b_s + stage * b_stage;
      for (int v = tid; v < n * 8; v += kTcProducers) {
        const int r = v >> 3, c16 = v & 7;
        cp_async16(bs + swz(r, c16), bsrc + (size_t)sh->tok[r] * bld + c * kTcK + 8 * c16);
      }
    };
    for (int c = 0; c < kTcLookahead; ++c) {
      if (c < KC) issue(c);
      cp_async_commit();
    }
    uint4 sv = make_uint4(0, 0, 0, 0), sv_next = sv;
    if (MODE != 2) sv = sv_next = ldg_stream(tile + 16 * ln);
    for (int c = 0; c < KC; ++c) {
      const int stage = c % kTcStages, s = c >> 3, j = c & 7;
      if (MODE != 2) {
        if (j == 0 && c > 0) sv = sv_next;
        if (j == 4 && s + 1 < g.nsc) sv_next = ldg_stream(tile + (size_t)(s + 1) * g.sc_bytes + 16 * ln);
      }
      cp_async_wait<kTcLookahead - 1>();  // this thread's copies of chunk c have landed
      if (MODE == 2) {  // nothing to dequantise
        fence_async_smem();
        mbar_arrive(&sh->full[stage]);
        const int cn = c + kTcLookahead;
        if (cn < KC) {
          if (!mbar_wait(&sh->empty[cn % kTcStages], ((cn / kTcStages) & 1) ^ 1, abort)) break;
          issue(cn);
        }
        cp_async_commit();
        continue;
      }
      const uint4 cv = *reinterpret_cast<const uint4*>(RAW + stage * kTcRawStageBytes + 16 * u);
      const uint32_t sp = e4m3x2_to_f16x2((u4get(sv, j >> 1) >> (16 * (j & 1))) & 0xFFFFu);
      const uint32_t s_lo = dup_lo(sp), s_hi = dup_hi(sp);
      uint32_t r0[8], r1[8];  // rows gi and gi+8 of tile ti: 16 f16 each
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t hh[4];
        e2m1x8_to_f16x8(u4get(cv, w), hh);
        r0[2 * w] = hmul2(hh[0], s_lo);
        r0[2 * w + 1] = hmul2(hh[2], s_lo);
        r1[2 * w] = hmul2(hh[1], s_hi);
        r1[2 * w + 1] = hmul2(hh[3], s_hi);
      }
      const int ra = 16 * ti + gi, rb = ra + 8;
      const uint32_t as = a_s + stage * kTcAStageBytes;
      st_shared_v4(as + swz(ra, 2 * t), r0[0], r0[1], r0[2], r0[3]);
      st_shared_v4(as + swz(ra, 2 * t + 1), r0[4], r0[5], r0[6], r0[7]);
      st_shared_v4(as + swz(rb, 2 * t), r1[0], r1[1], r1[2], r1[3]);
      st_shared_v4(as + swz(rb, 2 * t + 1), r1[4], r1[5], r1[6], r1[7]);
      fence_async_smem();
      mbar_arrive(&sh->full[stage]);
      // refill: chunk c + lookahead goes to the stage the MMAs of chunk c - 1 free
      const int cn = c + kTcLookahead;
      if (cn < KC) {
        if (!mbar_wait(&sh->empty[cn % kTcStages], ((cn / kTcStages) & 1) ^ 1, abort)) break;
        issue(cn);
      }
      cp_async_commit();
    }
    cp_async_wait<0>();
  } else {
    if (lane == 0) {
    // ---------------------------------------------------------------- MMA issue
    const uint32_t idesc = idesc_f16(kTcM, n_pad) | (MODE == 2 ? (1u << 7) | (1u << 10) : 0u);  // bf16
    const uint32_t a_s = smem_u32(A), b_s = smem_u32(B);
    for (int c = 0; c < KC; ++c) {
      const int stage = c % kTcStages;
      if (!mbar_wait(&sh->full[stage], (c / kTcStages) & 1, abort)) break;
      tc_fence_after();
      const uint64_t ad = sw128_desc(a_s + stage * kTcAStageBytes);
      const uint64_t bd = sw128_desc(b_s + stage * b_stage);
#pragma unroll
      for (int kk = 0; kk < kTcK / 16; ++kk)  // +32 bytes per 16-column step
        umma_f16(tmem_d, ad + 2 * kk, bd + 2 * kk, idesc, (c | kk) != 0);
      umma_commit(&sh->empty[stage]);
    }
    umma_commit(&sh->acc_full);  // fires once every issued MMA is done
    }
    __syncwarp();  // the other lanes of the MMA warp idle here instead of polling
  }

  // ---------------------------------------------------------------- epilogue
  // (the MMA warp goes straight to the final barrier: the epilogue warps only
  // pass it once acc_full says every MMA has completed)
  bool ok = true;
  if (warp < 8) ok = mbar_wait(&sh->acc_full, 0, abort);
  if (warp < 8 && !ok) {
    // wait (bounded) for the MMAs already in flight before freeing TMEM
    mbar_drain(&sh->acc_full, 0);
  }
  tc_fence_after();
  if (warp < 8 && ok && !*abort) {
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    const int r = 32 * q + lane;         // row of the 128-row block
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    if (MODE == 0) {
      const int pair = 4 * mb + q, i = 16 * pair + (lane & 15);
      const float ts_g = p.tscale[expert * 3 + 0], ts_u = p.tscale[expert * 3 + 1];
      for (int c0 = 32 * (warp >> 2); c0 < n_pad; c0 += 64) {
        uint32_t v[32];
        tmem_ld32(tmem_d + lane_addr + c0, v);
#pragma unroll
        for (int qq = 0; qq < 32; ++qq) {
          const float mine = __uint_as_float(v[qq]);
          const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
          const int col = c0 + qq;
          if (lane < 16 && col < n) {
            const float G = ts_g * mine, U = ts_u * other;
            const float a = G / (1.0f + expf(-G)) * U;
            p.abuf[(size_t)(row0 + col) * p.I + i] = __half_as_ushort(__float2half_rn(a));
          }
        }
      }
    } else if (MODE == 2) {
      const int e = kTcM * mb + r;
      for (int c0 = 32 * (warp >> 2); c0 < n_pad; c0 += 64) {
        uint32_t v[32];
        tmem_ld32(tmem_d + lane_addr + c0, v);
#pragma unroll
        for (int qq = 0; qq < 32; ++qq) {
          const int col = c0 + qq;
          if (col < n) p.logits_out[(size_t)(row0 + col) * p.E + e] = __uint_as_float(v[qq]);
        }
      }
    } else {
      const float ts = p.tscale[expert * 3 + 2];
      const int h = kTcM * mb + r;
      for (int c0 = 32 * (warp >> 2); c0 < n_pad; c0 += 64) {
        uint32_t v[32];
        tmem_ld32(tmem_d + lane_addr + c0, v);
#pragma unroll
        for (int qq = 0; qq < 32; ++qq) {
          const int col = c0 + qq;
          if (col < n) p.ybuf[(size_t)(row0 + col) * p.H + h] = ts * __uint_as_float(v[qq]);
        }
      }
    }
  }
  if (*abort && tid == 0) *p.status = -5;  // MOE_ETIMEOUT
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem_d, ncols);
  }
}

size_t tc_smem() {
  return 1024 + (size_t)kTcStages * (kTcAStageBytes + kTcBStageBytes + kTcRawStageBytes) +
         sizeof(TcShared);
}

}  // namespace

bool tc_path_ok(int fmt, int T, int k, int E, int H, int I) {
  // NVFP4 only; enough tokens per expert for a dense contraction; tile shapes
  return fmt == FMT_NVFP4 && (long)T * k >= 16L * E && H % kTcM == 0 && (2 * I) % kTcM == 0 &&
         H % kTcK == 0 && I % kTcK == 0;
}

int max_tc_entries(int T, int E, int k) {
  const long S = (long)T * k;
  const long m = S < E ? S : E;
  return (int)(m + S / kTcMaxN + 1);
}

cudaError_t launch_tc_gateup(const ExpertParams& p, int grid_y, cudaStream_t st) {
  dim3 grid((2 * p.I) / kTcM, grid_y);
  return launch_k(tc_gemm_kernel<0>, grid, dim3(kTcThreads), tc_smem(), st, true, p);
}

cudaError_t launch_tc_down(const ExpertParams& p, int grid_y, cudaStream_t st) {
  dim3 grid(p.H / kTcM, grid_y);
  return launch_k(tc_gemm_kernel<1>, grid, dim3(kTcThreads), tc_smem(), st, true, p);
}

bool tc_router_ok(int E, int H) { return E % kTcM == 0 && H % kTcK == 0; }

// logits_out gets the fp32 dot products (one K slice: the top-k step adds the bias)
cudaError_t launch_tc_router(const ExpertParams& p, cudaStream_t st) {
  dim3 grid(p.E / kTcM, (p.T + kTcMaxN - 1) / kTcMaxN);
  return launch_k(tc_gemm_kernel<2>, grid, dim3(kTcThreads), tc_smem(), st, true, p);
}

cudaError_t tc_kernels_init() {
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc_smem());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc_smem());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tc_smem());
}

}  // namespace moe
