// Prefill path: grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05, fp32 accumulators in tensor memory), and the router as a bf16
// GEMM.  Three forms of the expert GEMMs:
//   * tc_tmem_kernel (W4A16, H and I multiples of 128): the weights
//     dequantised into tensor memory, two MMA-issuing pipelines per SM (see
//     its section below);
//   * tc_fp4_kernel (W4A4): both operands NVFP4 on kind::mxf4nvf4;
//   * tc_expert_kernel (the other shapes): the weights dequantised into
//     shared memory, described here.
//
// Expert GEMMs (tc_expert_kernel): per work item (expert e, up to 128 tokens
// routed to e) and group of G 128-row blocks of W,
//   D_m[128 x N] (TMEM, fp32) = sum over K of A_m[128 x 64] . B[N x 64]^T
// A = the weights, dequantised exactly to f16 (e2m1 code * e4m3 block scale is
// an f16) by the producer warps from the packed NVFP4 tiles, which the Tensor
// Memory Accelerator brings in, and written to shared memory in the
// 128-byte-swizzled K-major layout the MMA reads; B = the token rows (x,
// gathered through the dispatch permutation, or the SwiGLU output a), copied
// the same way.  One thread issues the MMAs; stages are handed over with
// mbarriers; tcgen05.commit frees a stage when the MMAs reading it are done.
// The epilogue warps read D from TMEM (warp w owns lanes 32(w%4)..+31) and
// apply the fp32 tensor scale and SwiGLU (gate/up) or write y rows (down).
//
// The weights stay the M operand and the token count the N operand (N is 80 on
// average for 4096 tokens over 512 experts): an expert with few tokens keeps
// its decoded weights on the 128-row side of the MMA.
// Every wait is bounded: on a timeout the kernel records MOE_ETIMEOUT in the
// status word, stops issuing work, waits (bounded) for its MMAs and copies,
// frees its TMEM and returns.
#include <cuda.h>  // CUtensorMap: the tile map of the packed arena
#include <cudaTypedefs.h>

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
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

struct TcShared {
  uint64_t full[kTcStages];
  uint64_t empty[kTcStages];
  uint64_t acc_full;
  uint32_t tmem_base;
  int abort;
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
    *p.status = kStatusInvalid;
    return false;
  }
  return true;
}

// The router GEMM for large T: logits[t][e] = x[t] . Wr[e] (bf16 x bf16 ->
// fp32), 128 experts as M and up to 128 tokens as N per CTA.  The 8 copy
// warps bring the router rows and the token rows of each 64-column chunk
// straight into 128B-swizzled stages with cp.async, kTcLookahead chunks ahead,
// fence the async proxy and arrive on full[c % stages]; one thread issues the
// MMAs and commits each stage back; the copy warps then read D from TMEM.
__global__ void __launch_bounds__(kTcThreads, 1) tc_router_kernel(ExpertParams p) {
  griddep_wait();
  const int row0 = kTcMaxN * blockIdx.y;  // token tile
  const int n = min(kTcMaxN, p.T - row0);
  if (n <= 0) return;
  extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~(uintptr_t)1023);
  const int n_pad = (n + 15) & ~15;
  const int b_stage = n_pad * kTcK * 2;  // multiple of 2 KB: stages stay 1024-byte aligned
  uint8_t* A = base;
  uint8_t* B = A + kTcStages * kTcAStageBytes;
  TcShared* sh = reinterpret_cast<TcShared*>(B + kTcStages * kTcBStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = p.H, KC = K / kTcK, mb = blockIdx.x;
  const uint32_t ncols = n_pad <= 32 ? 32 : (n_pad <= 64 ? 64 : 128);

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&sh->full[s], kTcProducers);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->acc_full, 1);
    sh->abort = 0;
    mbar_init_fence();
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
    // ---------------------------------------------------------------- copies
    const uint16_t* arow = p.wr + (size_t)kTcM * mb * p.H;  // 128 router rows
    for (int i = tid; i < kTcM * KC; i += kTcProducers)     // ask L2 for everything
      prefetch_l2(arow + (size_t)(i / KC) * p.H + 64 * (i % KC));
    const uint32_t a_s = smem_u32(A), b_s = smem_u32(B);
    auto issue = [&](int c) {  // chunk c's copies into stage c % stages
      const int stage = c % kTcStages;
      for (int v = tid; v < kTcM * 8; v += kTcProducers) {
        const int r = v >> 3, c16 = v & 7;
        cp_async16(a_s + stage * kTcAStageBytes + swz(r, c16), arow + (size_t)r * p.H + c * kTcK + 8 * c16);
      }
      const uint32_t bs = b_s + stage * b_stage;
      for (int v = tid; v < n * 8; v += kTcProducers) {
        const int r = v >> 3, c16 = v & 7;
        cp_async16(bs + swz(r, c16), p.x + (size_t)(row0 + r) * p.H + c * kTcK + 8 * c16);
      }
    };
    for (int c = 0; c < kTcLookahead; ++c) {
      if (c < KC) issue(c);
      cp_async_commit();
    }
    for (int c = 0; c < KC; ++c) {
      cp_async_wait<kTcLookahead - 1>();  // this thread's copies of chunk c have landed
      fence_async_smem();
      mbar_arrive(&sh->full[c % kTcStages]);
      const int cn = c + kTcLookahead;
      if (cn < KC) {
        if (!mbar_wait(&sh->empty[cn % kTcStages], ((cn / kTcStages) & 1) ^ 1, abort, p.wait_budget)) break;
        issue(cn);
      }
      cp_async_commit();
    }
    cp_async_wait<0>();
  } else {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issue
      const uint32_t idesc = idesc_f16(kTcM, n_pad) | (1u << 7) | (1u << 10);  // A and B bf16
      const uint32_t a_s = smem_u32(A), b_s = smem_u32(B);
      for (int c = 0; c < KC; ++c) {
        const int stage = c % kTcStages;
        if (!mbar_wait(&sh->full[stage], (c / kTcStages) & 1, abort, p.wait_budget)) break;
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
    __syncwarp();
  }

  // ---------------------------------------------------------------- epilogue
  bool ok = true;
  if (warp < 8) ok = mbar_wait(&sh->acc_full, 0, abort, p.wait_budget);
  if (warp < 8 && !ok) mbar_drain(&sh->acc_full, 0);  // MMAs in flight finish before TMEM is freed
  tc_fence_after();
  if (warp < 8 && ok && !*abort) {
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int e = kTcM * mb + 32 * q + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    for (int c0 = 32 * (warp >> 2); c0 < n_pad; c0 += 64) {
      uint32_t v[32];
      tmem_ld32(tmem_d + lane_addr + c0, v);
#pragma unroll
      for (int qq = 0; qq < 32; ++qq) {
        const int col = c0 + qq;
        if (col < n) p.logits_out[(size_t)(row0 + col) * p.E + e] = __uint_as_float(v[qq]);
      }
    }
  }
  if (*abort && tid == 0) *p.status = kStatusTimeout;
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem_d, ncols);
  }
}

size_t tc_smem() {
  return 1024 + (size_t)kTcStages * (kTcAStageBytes + kTcBStageBytes) + sizeof(TcShared);
}

// ---------------------------------------------------------------- expert GEMMs with TMA-fed tiles
// The expert GEMMs (MODE 0 gate/up + SwiGLU, MODE 1 down) with the packed
// codes brought in by the Tensor Memory Accelerator and G M-blocks per CTA.
//
// Work item (expert, up to 128 tokens) x group of G 128-row M-blocks.  Per
// 64-column K-chunk c:
//   * one TMA load (warp 9) brings the code vectors of the group's 8G tiles
//     (box {512 B, 1 piece, 8G tiles} of the arena's tile map, 4G KB) into a
//     4-stage ring (the scale vectors, 1/8 of the bytes, each producer thread
//     reads for its tiles straight into registers, a super-chunk ahead).  The
//     tile map views the packed layout as
//     [expert][tile][512-byte piece][512 B], so a box is 8G pieces at the same
//     offset of consecutive tiles: one bulk copy instead of 8G small ones,
//     and several chunks in flight per SM.
//   * the 8 producer warps copy the chunk's token rows (B, gathered through
//     the dispatch, 64 columns each) with cp.async three chunks ahead into a
//     5-stage ring, and dequantise each M-block's codes into a 128B-swizzled
//     f16 A slot (a 4-slot ring, one slot per M-block);
//   * one thread issues, per M-block, 4 MMAs into that M-block's TMEM
//     accumulator (G accumulators of N columns side by side) and commits the
//     A slot back; after the last M-block it commits the B stage back.
// A token chunk is read once for G M-blocks (G = 4 where the matrix has 4k
// M-blocks), which cuts the L2 traffic of the token rows by G.
constexpr int kTxNA = 8;             // A slots (16 KB each): two chunks of a 4-M-block group
constexpr int kTxNB = 3;             // B stages (up to 16 KB each)
constexpr int kTxLB = 2;             // B chunks in flight ahead of the dequantisation
constexpr int kTxNR = 3;             // code stages (4 KB per M-block)
constexpr int kTxPW = 16;            // producer (and epilogue) warps
constexpr int kTxThreads = 32 * (kTxPW + 2);  // + warp 16: MMA issue, warp 17: TMA issue
constexpr int kTxMaxG = 4;

struct TxShared {
  uint64_t a_full[kTxNA], a_empty[kTxNA];
  uint64_t b_empty[kTxNB];
  uint64_t r_full[kTxNR], r_empty[kTxNR];
  uint64_t acc_full;
  uint32_t tmem_base;
  int abort;
  int tok[kTcMaxN];
};

__host__ __device__ constexpr size_t tx_smem_bytes(int G) {
  return 1024 + (size_t)kTxNA * kTcAStageBytes + (size_t)kTxNB * kTcBStageBytes +
         (size_t)kTxNR * 4096 * G + sizeof(TxShared);
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

// 4-D tiled TMA load of the tile map box at (0, piece, tile, expert) into
// shared memory, counted on `bar`.
__device__ __forceinline__ void tma_load_tiles(uint32_t dst, const CUtensorMap* map, int piece,
                                               int tile, int expert, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(piece), "r"(tile), "r"(expert),
      "r"(smem_u32(bar))
      : "memory");
}

// Epilogue of the expert GEMMs, by the 16 producer warps (warp w reads TMEM
// lanes 32(w%4)..+31 and every fourth group of 32 columns): G accumulators of
// npc columns side by side, row r of M-block m in lane r.  MODE 0: rows 32q..
// 32q+15 of quadrant q are a gate tile and 32q+16.. the matching up tile;
// a = silu(ts_g * g) * (ts_u * u) (times the token's scale in W4A4) goes to
// af (fp32) or abuf (f16).  MODE 1: y rows (times the row's scale in W4A4).
template <int MODE>
__device__ __forceinline__ void tx_epilogue(const ExpertParams& p, int expert, int row0, int n,
                                            int n_pad, int npc, int G, uint32_t tmem_d,
                                            const int* tok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3;             // TMEM lane quadrant of this warp
  const int r = 32 * qd + lane;        // row of the 128-row block
  const uint32_t lane_addr = (uint32_t)(32 * qd) << 16;
  for (int m = 0; m < G; ++m) {
    const int mb = G * blockIdx.x + m;  // M-block of the matrix
    const uint32_t acc = tmem_d + lane_addr + (uint32_t)(m * npc);
    if (MODE == 0) {
      const int pair = 4 * mb + qd, i = 16 * pair + (lane & 15);
      const float ts_g = p.tscale[expert * 3 + 0], ts_u = p.tscale[expert * 3 + 1];
      for (int c0 = 32 * (warp >> 2); c0 < n_pad; c0 += 32 * (kTxPW / 4)) {
        uint32_t v[32];
        tmem_ld32(acc + c0, v);
#pragma unroll
        for (int qq = 0; qq < 32; ++qq) {
          const float mine = __uint_as_float(v[qq]);
          const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
          const int col = c0 + qq;
          if (lane < 16 && col < n) {
            const float sx = p.ts_x ? p.ts_x[tok[col]] : 1.0f;  // W4A4: the token's scale
            const float Gv = (ts_g * sx) * mine, U = (ts_u * sx) * other;
            const float a = Gv / (1.0f + expf(-Gv)) * U;
            if (p.af)
              p.af[(size_t)(row0 + col) * p.I + i] = a;
            else
              p.abuf[(size_t)(row0 + col) * p.I + i] = a_to_f16(a, p.status);
          }
        }
      }
    } else {
      const float ts = p.tscale[expert * 3 + 2];
      const int h = kTcM * mb + r;
      for (int c0 = 32 * (warp >> 2); c0 < n_pad; c0 += 32 * (kTxPW / 4)) {
        uint32_t v[32];
        tmem_ld32(acc + c0, v);
#pragma unroll
        for (int qq = 0; qq < 32; ++qq) {
          const int col = c0 + qq;
          if (col < n) {
            const float sa = p.ts_a ? p.ts_a[row0 + col] : 1.0f;  // W4A4: the row's scale
            p.ybuf[(size_t)(row0 + col) * p.H + h] = (ts * sa) * __uint_as_float(v[qq]);
          }
        }
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kTxThreads, 1)
    tc_expert_kernel(ExpertParams p, const __grid_constant__ CUtensorMap tmap, int G) {
  griddep_wait();
  int expert, row0, n;
  if (!tc_entry(p, blockIdx.y, expert, row0, n)) return;
  extern __shared__ __align__(1024) uint8_t tx_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tx_smem_raw) + 1023) & ~(uintptr_t)1023);
  const int RB = 4096 * G;               // bytes of one code stage (8G tiles x 512 B)
  const int n_pad = (n + 15) & ~15;
  const int b_stage = n_pad * kTcK * 2;  // multiple of 2 KB: stages stay 1024-byte aligned
  uint8_t* A = base;
  uint8_t* B = A + kTxNA * kTcAStageBytes;
  uint8_t* R = B + kTxNB * kTcBStageBytes;
  TxShared* sh = reinterpret_cast<TxShared*>(R + kTxNR * RB);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.T * p.k;
  const int K = MODE == 1 ? p.I : p.H;
  const int KC = K / kTcK;
  const int tile0 = 8 * G * blockIdx.x;  // first 16-row tile of this CTA's M-blocks
  const int npc = n_pad <= 32 ? 32 : (n_pad <= 64 ? 64 : 128);  // TMEM columns per accumulator
  const uint32_t ncols = (uint32_t)(G * npc);

  if (tid == 0) {
    // producer warps arrive once each (lane 0, after a __syncwarp): 256
    // single-thread arrivals on one barrier serialise on its shared word
    for (int i = 0; i < kTxNA; ++i) {
      mbar_init(&sh->a_full[i], 8);  // the 8 warps of an M-block's half
      mbar_init(&sh->a_empty[i], 1);
    }
    for (int i = 0; i < kTxNB; ++i) mbar_init(&sh->b_empty[i], 1);
    for (int i = 0; i < kTxNR; ++i) {
      mbar_init(&sh->r_full[i], 1);
      mbar_init(&sh->r_empty[i], kTxPW);
    }
    mbar_init(&sh->acc_full, 1);
    sh->abort = 0;
    mbar_init_fence();
  }
  for (int i = tid; i < n_pad; i += kTxThreads) {
    int tk = 0;
    if (i < n) tk = (MODE == 0) ? ((expert == p.E) ? row0 - S + i : p.row_token[row0 + i]) : row0 + i;
    sh->tok[i] = tk;  // MODE 0: token index into x; MODE 1: row of abuf
  }
  // token-row padding stays zero in every stage (cp.async never writes it)
  for (int i = tid; i < kTxNB * (n_pad - n) * 8; i += kTxThreads) {
    const int st = i / ((n_pad - n) * 8), rem = i % ((n_pad - n) * 8);
    const int r = n + rem / 8, c16 = rem % 8;
    *reinterpret_cast<uint4*>(B + st * b_stage + swz(r, c16)) = make_uint4(0, 0, 0, 0);
  }
  if (warp == kTxPW) tmem_alloc(&sh->tmem_base, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = sh->tmem_base;
  volatile int* abort = &sh->abort;
  const uint32_t a_s = smem_u32(A), b_s = smem_u32(B), r_s = smem_u32(R);

  if (warp < kTxPW) {
    // ---------------------------------------------------------------- producers
    // warp pw: tile pw%8 of the M-blocks m = pw/8, pw/8 + 2 (of the group's G),
    // lane ln of that tile's 16-byte vectors; the warps of half 0 also copy the
    // token rows (so that their a_full arrivals for M-block 0 publish them)
    const int half = warp >> 3, ti = warp & 7, ln = lane, gi = ln >> 2, t = ln & 3;
    const uint16_t* bsrc = (MODE == 0) ? p.xh : p.abuf;
    const int bld = (MODE == 0) ? p.H : p.I;
    auto issue_b = [&](int c) {  // chunk c's token rows into B stage c % kTxNB
      if (half != 0) return;
      const uint32_t bs = b_s + (c % kTxNB) * b_stage;
      for (int v = tid; v < n * 8; v += 256) {
        const int r = v >> 3, c16 = v & 7;
        cp_async16(bs + swz(r, c16), bsrc + (size_t)sh->tok[r] * bld + c * kTcK + 8 * c16);
      }
    };
    for (int c = 0; c < kTxLB; ++c) {
      if (c < KC) issue_b(c);
      cp_async_commit();
    }
    // my tiles' scale vectors, a super-chunk ahead
    const MatGeom g = mat_geom(FMT_NVFP4, K);
    const uint8_t* tiles = expert_base(p, expert) + (MODE == 1 ? p.gu_bytes : 0);
    const size_t tb = MODE == 1 ? (size_t)p.dn_tile_bytes : (size_t)p.gu_tile_bytes;
    const uint8_t* mine = tiles + (size_t)(tile0 + ti) * tb + 16 * ln;
    uint4 sv[2], sv_next[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int m = half + 2 * i;
      if (m < G) sv[i] = sv_next[i] = ldg_stream(mine + (size_t)m * 8 * tb);
    }
    for (int c = 0; c < KC; ++c) {
      const int s = c >> 3, j = c & 7;
      if (j == 0 && c > 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) sv[i] = sv_next[i];
      }
      if (j == 4 && s + 1 < g.nsc) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int m = half + 2 * i;
          if (m < G) sv_next[i] = ldg_stream(mine + (size_t)m * 8 * tb + (size_t)(s + 1) * g.sc_bytes);
        }
      }
      // (waits are made warp-uniform: the warps arrive with one lane after a __syncwarp)
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(&sh->r_full[c % kTxNR], (c / kTxNR) & 1, abort, p.wait_budget))) break;
      uint4 cv[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int m = half + 2 * i;
        if (m < G) cv[i] = lds128(r_s + (c % kTxNR) * RB + (m * 8 + ti) * 512 + 16 * ln);
      }
      __syncwarp();
      if (ln == 0) mbar_arrive(&sh->r_empty[c % kTxNR]);
      cp_async_wait<kTxLB - 1>();  // this thread's token-row pieces of chunk c have landed
      bool ok = true;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int m = half + 2 * i;
        if (m >= G) break;
        const int q = c * G + m, slot = q % kTxNA;
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(&sh->a_empty[slot], ((q / kTxNA) & 1) ^ 1, abort, p.wait_budget))) {
          ok = false;
          break;
        }
        const uint32_t sp = e4m3x2_to_f16x2((u4get(sv[i], j >> 1) >> (16 * (j & 1))) & 0xFFFFu);
        const uint32_t s_lo = dup_lo(sp), s_hi = dup_hi(sp);
        uint32_t r0[8], r1[8];  // rows gi and gi+8 of tile ti: 16 f16 each
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t hh[4];
          e2m1x8_to_f16x8(u4get(cv[i], w), hh);
          r0[2 * w] = hmul2(hh[0], s_lo);
          r0[2 * w + 1] = hmul2(hh[2], s_lo);
          r1[2 * w] = hmul2(hh[1], s_hi);
          r1[2 * w + 1] = hmul2(hh[3], s_hi);
        }
        const int ra = 16 * ti + gi, rb = ra + 8;
        const uint32_t as = a_s + slot * kTcAStageBytes;
        st_shared_v4(as + swz(ra, 2 * t), r0[0], r0[1], r0[2], r0[3]);
        st_shared_v4(as + swz(ra, 2 * t + 1), r0[4], r0[5], r0[6], r0[7]);
        st_shared_v4(as + swz(rb, 2 * t), r1[0], r1[1], r1[2], r1[3]);
        st_shared_v4(as + swz(rb, 2 * t + 1), r1[4], r1[5], r1[6], r1[7]);
        fence_async_smem();  // (for half 0 also publishes the token rows of chunk c)
        __syncwarp();
        if (ln == 0) mbar_arrive(&sh->a_full[slot]);
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      // refill: chunk c + kTxLB goes to the B stage the MMAs of chunk c + kTxLB - kTxNB freed
      const int cn = c + kTxLB;
      if (cn < KC && half == 0) {
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(&sh->b_empty[cn % kTxNB], ((cn / kTxNB) & 1) ^ 1, abort, p.wait_budget)))
          break;
        issue_b(cn);
      }
      cp_async_commit();
    }
    cp_async_wait<0>();
  } else if (warp == kTxPW) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issue
      const uint32_t idesc = idesc_f16(kTcM, n_pad);
      bool ok = true;
      for (int c = 0; c < KC && ok; ++c) {
        const uint64_t bd = sw128_desc(b_s + (c % kTxNB) * b_stage);
        for (int m = 0; m < G; ++m) {
          const int q = c * G + m, slot = q % kTxNA;
          if (!mbar_wait_sleep(&sh->a_full[slot], (q / kTxNA) & 1, abort, p.wait_budget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_desc(a_s + slot * kTcAStageBytes);
#pragma unroll
          for (int kk = 0; kk < kTcK / 16; ++kk)  // +32 bytes per 16-column step
            umma_f16(tmem_d + m * npc, ad + 2 * kk, bd + 2 * kk, idesc, (c | kk) != 0);
          umma_commit(&sh->a_empty[slot]);
        }
        if (ok) umma_commit(&sh->b_empty[c % kTxNB]);
      }
      umma_commit(&sh->acc_full);  // fires once every issued MMA is done
    }
    __syncwarp();
  } else {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA issue
      const CUtensorMap* map = &tmap;
      int issued = 0;  // code chunks issued
      for (int c = 0; c < KC; ++c) {
        const int s = c >> 3, j = c & 7;
        if (!mbar_wait_sleep(&sh->r_empty[c % kTxNR], ((c / kTxNR) & 1) ^ 1, abort, p.wait_budget)) break;
        mbar_arrive_expect(&sh->r_full[c % kTxNR], (uint32_t)RB);
        tma_load_tiles(r_s + (c % kTxNR) * RB, map, 9 * s + 1 + j, tile0, expert,
                       &sh->r_full[c % kTxNR]);
        ++issued;
      }
      if (*abort) {  // let the copies in flight land before the CTA exits (bounded waits)
        for (int c = (issued > kTxNR ? issued - kTxNR : 0); c < issued; ++c)
          mbar_drain(&sh->r_full[c % kTxNR], (c / kTxNR) & 1);
      }
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- epilogue
  bool ok = true;
  if (warp < kTxPW) ok = mbar_wait_sleep(&sh->acc_full, 0, abort, p.wait_budget);
  if (warp < kTxPW && !ok) mbar_drain(&sh->acc_full, 0);  // MMAs in flight finish before TMEM is freed
  tc_fence_after();
  if (warp < kTxPW && ok && !*abort) tx_epilogue<MODE>(p, expert, row0, n, n_pad, npc, G, tmem_d, sh->tok);
  if (*abort && tid == 0) *p.status = kStatusTimeout;
  tc_fence_before();
  __syncthreads();
  if (warp == kTxPW) {
    tc_fence_after();
    tmem_dealloc(tmem_d, ncols);
  }
}

// ---------------------------------------------------------------- W4A4: the block-scaled FP4 MMA
// With the activations quantised to NVFP4 per row (x per token, a per
// (token, expert) row), both operands of the expert GEMMs are e2m1 codes with
// an e4m3 scale per 16 columns, and the products run on tcgen05.mma
// kind::mxf4nvf4 (scale_vec::4X: four block scales per row and K = 64 step;
// fp32 accumulators in TMEM).  The weights come from their MMA layout
// (layout.cuh) and the activations from rows in expert-sorted order (x
// quantised into the rows of its slots after the dispatch; a in slot order),
// so every operand byte arrives by the Tensor Memory Accelerator.
//
// Persistent: one CTA per SM walks the work units u = blockIdx.x,
// blockIdx.x + gridDim.x, ...; unit u = (work item u / M-blocks: an expert
// and up to 128 of its tokens, 128-row M-block u % M-blocks).  The stage ring
// (kFqNS stages of 256 columns of K) runs on across units, and the
// accumulators are double-buffered, so a unit's epilogue overlaps the next
// unit's loads and MMAs.  Per stage:
//   * the TMA warp loads the M-block's codes (one 128-byte x 128-row box, 16
//     contiguous KB of the layout, 128B-swizzled: the K-major layout the MMA
//     reads) and block scales (2 KB, one bulk copy), and the item's 128 token
//     rows: codes (one 128-byte x 128-row box, 128B-swizzled) and block
//     scales (16 bytes a row); rows past the item's tokens hold other rows'
//     values and only reach accumulator columns the epilogue never reads;
//   * warps 0-3 (a row per thread) move the token rows' scales into the
//     512-byte groups tcgen05.cp reads (row l of a group: the 4 scales of
//     rows l, l+32, l+64 and l+96 for one K-step);
//   * one thread each (warps 14 and 15) moves the stage's block scales of A
//     and of B into tensor memory with tcgen05.cp 32x128b.warpx4 (a group
//     lands in lanes l of all four lane quadrants, one 32-bit column per
//     32-row group) and commits them to the slot's mbarrier: a copy takes
//     about as long to issue as an MMA, so three threads share the issuing;
//   * the MMA thread (warp 12) waits for both and issues the stage's 4 MMAs;
//   * warps 4-11 read a finished unit's accumulators (the activation scales
//     of their columns loaded before the wait) and hand the buffer back.
constexpr int kFqThreads = 32 * 16;
constexpr int kFqEpi0 = 4;                // epilogue warps 4-11
constexpr int kFqMmaWarp = 12, kFqTmaWarp = 13, kFqSfaWarp = 14, kFqSfbWarp = 15;
static_assert(32 * (kFqSfbWarp + 1) == kFqThreads, "warp roles");
constexpr int kFqK = 256;                 // K per stage (4 steps of 64)
constexpr int kFqNS = 5;                  // stages in flight
constexpr int kFqList = 128;              // units a CTA keeps in its list
constexpr int kFqAStage = kTcM * 128;     // 16 KB of weight codes
constexpr int kFqBStage = kTcMaxN * 128;  // 16 KB of token-row codes
constexpr int kFqSf = 4 * 512;            // block scales of a stage: 4 K-steps x 128 rows x 4
constexpr int kFqStage = kFqAStage + kFqBStage + 3 * kFqSf;  // + A scales, B scales, B scales as loaded
// TMEM columns: two accumulators of 128, then 16 columns of A scales and 16
// of B scales per stage slot
constexpr uint32_t kFqSfaCol = 256;
constexpr uint32_t kFqSfbCol = kFqSfaCol + 16 * kFqNS;
static_assert(kFqSfbCol + 16 * kFqNS <= 512, "tensor memory columns");

struct FqShared {
  uint64_t full_a[kFqNS];   // weight codes and scales of the slot (transaction bytes)
  uint64_t full_bt[kFqNS];  // token-row codes and scales of the slot (transaction bytes)
  uint64_t full_b[kFqNS];   // the token rows' scales regrouped (4 warp arrivals)
  uint64_t sfa[kFqNS];      // the slot's A scales are in tensor memory
  uint64_t sfb[kFqNS];      // the slot's B scales are in tensor memory
  uint64_t empty[kFqNS];    // the MMAs reading the slot are done
  uint64_t acc_full[2], acc_empty[2];
  uint64_t fin, fin2[2];
  uint32_t tmem_base;
  int abort;
};

__host__ __device__ constexpr size_t fq_smem_bytes() {
  return 1024 + (size_t)kFqNS * kFqStage + sizeof(FqShared) + 16 + 16 * kFqList;  // + the unit list
}

// Instruction descriptor of kind::mxf4nvf4: A and B e2m1 (format 1), both
// K-major, e4m3 block scales (scale format 0), D fp32 (implied), M x N; the
// scale-factor ids stay 0 (at scale_vec::4X all four bytes of a column count).
__device__ __forceinline__ uint32_t idesc_mxf4nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem));
}

// Shared-memory descriptor of a 512-byte group of 32 rows x 16 bytes without
// swizzle: 8-row core matrices of 128 contiguous bytes, 128 bytes apart (both
// offsets 128, so the group is read as one contiguous block either way).
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  return d;
}

// lanes l of all four TMEM lane quadrants, 4 columns from taddr <- row l of the group
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// tiled TMA load of the MMA layout's box at (row y, stage s, expert e), counted on `bar`
__device__ __forceinline__ void tma_load_codes(uint32_t dst, const CUtensorMap* map, int y, int s, int e,
                                               uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(s), "r"(e), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned), counted on `bar`
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// 2-D tiled TMA load of the box at (x, row y) of an activation-row map, counted on `bar`
__device__ __forceinline__ void tma_load_rows(uint32_t dst, const CUtensorMap* map, int x, int y,
                                              uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// y rows from a 32-column accumulator chunk (lane l = row h0 + l of the
// M-block, v[c] = column c0 + c): 4 x 4 transposes within lane quads (two
// shuffle rounds) give lane 4a + b the rows h0 + 4a .. + 3 of column c0 + 4m + b,
// so each store instruction writes 4 rows of y x 128 bytes (16 bytes a lane)
// instead of one.  y = (ts * column scale) * D.
__device__ __forceinline__ void store_y_chunk(const ExpertParams& p, const uint32_t (&v)[32], int row0,
                                              int c0, int n, int h0, float ts, float sc_lane) {
  const int lane = threadIdx.x & 31;
  const bool b1 = lane & 1, b2 = lane & 2;
  float* yb = p.ybuf + h0 + 4 * (lane >> 2);
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    float w0 = __uint_as_float(v[4 * m]), w1 = __uint_as_float(v[4 * m + 1]);
    float w2 = __uint_as_float(v[4 * m + 2]), w3 = __uint_as_float(v[4 * m + 3]);
    float s0 = b2 ? w0 : w2, s1 = b2 ? w1 : w3;
    float r0 = __shfl_xor_sync(0xffffffffu, s0, 2), r1 = __shfl_xor_sync(0xffffffffu, s1, 2);
    if (b2) {
      w0 = r0;
      w1 = r1;
    } else {
      w2 = r0;
      w3 = r1;
    }
    s0 = b1 ? w0 : w1;
    s1 = b1 ? w2 : w3;
    r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
    r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
    if (b1) {
      w0 = r0;
      w2 = r1;
    } else {
      w1 = r0;
      w3 = r1;
    }
    const int cq = 4 * m + (lane & 3), col = c0 + cq;
    const float sc = ts * __shfl_sync(0xffffffffu, sc_lane, cq);
    if (col < n)
      *reinterpret_cast<float4*>(yb + (size_t)(row0 + col) * p.H) = make_float4(sc * w0, sc * w1, sc * w2, sc * w3);
  }
}

struct FqUnit {
  int expert, row0, n, mb;
};

// Unit i of this CTA (u = blockIdx.x + i * gridDim.x): false past the last.
// The first kFqList come from the CTA's list in shared memory (filled at the
// start), later ones are read from the work entries.  A unit whose entry
// fails its bounds check gets n = 0 (every role skips it).
__device__ __forceinline__ bool fq_unit(const ExpertParams& p, const int4* list, int i, int n_units,
                                        int mblocks, FqUnit& w) {
  const int u = blockIdx.x + i * gridDim.x;
  if (u >= n_units) return false;
  if (i < kFqList) {
    const int4 v = list[i];
    w.expert = v.x;
    w.row0 = v.y;
    w.n = v.z;
    w.mb = v.w;
    return true;
  }
  if (!tc_entry(p, u / mblocks, w.expert, w.row0, w.n)) w.n = 0;
  w.mb = u % mblocks;
  return true;
}

template <int MODE>
__global__ void __launch_bounds__(kFqThreads, 1)
    tc_fp4_kernel(ExpertParams p, const __grid_constant__ CUtensorMap tmap,
                  const __grid_constant__ CUtensorMap bmap_c, const __grid_constant__ CUtensorMap bmap_s,
                  int max_items) {
  griddep_wait();
  extern __shared__ __align__(1024) uint8_t fq_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(fq_smem_raw) + 1023) & ~(uintptr_t)1023);
  // per stage slot: A codes (16 KB), B codes (16 KB), A scales, B scales, B scales as loaded (2 KB each)
  FqShared* sh = reinterpret_cast<FqShared*>(base + kFqNS * kFqStage);
  int4* list = reinterpret_cast<int4*>((reinterpret_cast<uintptr_t>(sh + 1) + 15) & ~(uintptr_t)15);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.T * p.k;
  const int K = MODE == 1 ? p.I : p.H;
  const int KC = K / 64, KS = (K + kFqK - 1) / kFqK;
  const int mblocks = (MODE == 1 ? p.H : 2 * p.I) / kTcM;
  const int items = min(p.nsh_tc + *p.n_tc_entries, max_items);
  const int n_units = mblocks * max(items, 0);
  const uint32_t s0 = smem_u32(base);
  auto a_addr = [&](int slot) { return s0 + slot * kFqStage; };
  auto b_addr = [&](int slot) { return s0 + slot * kFqStage + kFqAStage; };
  auto sa_addr = [&](int slot) { return s0 + slot * kFqStage + kFqAStage + kFqBStage; };
  auto sb_addr = [&](int slot) { return sa_addr(slot) + kFqSf; };
  auto sn_addr = [&](int slot) { return sa_addr(slot) + 2 * kFqSf; };

  if (tid == 0) {
    for (int i = 0; i < kFqNS; ++i) {
      mbar_init(&sh->full_a[i], 1);
      mbar_init(&sh->full_bt[i], 1);
      mbar_init(&sh->full_b[i], 4);
      mbar_init(&sh->sfa[i], 1);
      mbar_init(&sh->sfb[i], 1);
      mbar_init(&sh->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->acc_full[i], 1);
      mbar_init(&sh->acc_empty[i], 8);  // the 8 epilogue warps
    }
    mbar_init(&sh->fin, 1);
    mbar_init(&sh->fin2[0], 1);
    mbar_init(&sh->fin2[1], 1);
    sh->abort = 0;
    mbar_init_fence();
  }
  if (warp == 0) {  // the unit list: {expert, first row, tokens, M-block}
    for (int i = lane; i < kFqList; i += 32) {
      const int u = blockIdx.x + i * gridDim.x;
      int4 v = make_int4(0, 0, 0, 0);
      if (u < n_units) {
        int e, r0, n;
        v = tc_entry(p, u / mblocks, e, r0, n) ? make_int4(e, r0, n, u % mblocks)
                                               : make_int4(0, 0, 0, u % mblocks);
      }
      list[i] = v;
    }
  }
  if (warp == kFqMmaWarp) tmem_alloc(&sh->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp < kFqEpi0) {
    // ---------------------------------------------------------------- token-row scales into groups
    const int r = tid;  // row of the stage (0..127)
    int gs = 0;
    FqUnit cur;
    bool ok = true;
    for (int i = 0; ok && fq_unit(p, list, i, n_units, mblocks, cur); ++i) {
      if (cur.n == 0) continue;
      for (int s = 0; s < KS; ++s, ++gs) {
        const int slot = gs % kFqNS;
        // (sleeping waits: the spinning MMA and TMA threads share these warps' schedulers)
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(&sh->full_bt[slot], (gs / kFqNS) & 1, abort,
                                                     p.wait_budget))) {
          ok = false;
          break;
        }
        const uint4 w4 = lds128(sn_addr(slot) + 16 * r);  // the row's scales of K-steps 0..3
        const uint32_t g = sb_addr(slot) + (r & 31) * 16 + (r >> 5) * 4;
        st_shared_u32(g, w4.x);
        st_shared_u32(g + 512, w4.y);
        st_shared_u32(g + 1024, w4.z);
        st_shared_u32(g + 1536, w4.w);
        fence_async_smem();  // (for tcgen05.cp)
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->full_b[slot]);
      }
    }
  } else if (warp < kFqMmaWarp) {
    // ---------------------------------------------------------------- epilogue
    // warp 4 + 4h + q: TMEM lane quadrant q (rows 32q..32q+31), columns 64h..64h+63
    const int qd = warp & 3, ch = (warp - kFqEpi0) >> 2;
    const uint32_t lane_addr = (uint32_t)(32 * qd) << 16;
    // row of x (MODE 0: the token) behind column r of a unit
    auto tok = [&](const FqUnit& w, int r) -> size_t {
      return (size_t)(w.expert == p.E ? w.row0 - S + r : p.row_token[w.row0 + r]);
    };
    FqUnit cur;
    int uk = 0;
    for (int i = 0; fq_unit(p, list, i, n_units, mblocks, cur); ++i) {
      if (cur.n == 0) continue;
      const int n_pad = (cur.n + 15) & ~15, buf = uk & 1;
      // the unit's tensor scales, read before the accumulator wait (an L2 round
      // trip under this load takes about a microsecond)
      const float ts_g = p.tscale[cur.expert * 3 + (MODE == 1 ? 2 : 0)];
      const float ts_u = MODE == 0 ? p.tscale[cur.expert * 3 + 1] : 0.0f;
      float sc_lane[2] = {1.0f, 1.0f};  // W4A4 scales of columns 64h + 32c + lane
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col = 64 * ch + 32 * c + lane;
        if (col < cur.n) {
          if (MODE == 0 && p.ts_x) sc_lane[c] = p.ts_x[tok(cur, col)];
          if (MODE == 1 && p.ts_a) sc_lane[c] = p.ts_a[cur.row0 + col];
        }
      }
      if (!mbar_wait_sleep(&sh->acc_full[buf], (uk >> 1) & 1, abort, p.wait_budget)) break;
      tc_fence_after();
      const uint32_t acc = tmem_d + lane_addr + (uint32_t)(128 * buf);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int c0 = 64 * ch + 32 * c;
        if (c0 >= n_pad) break;
        uint32_t v[32];
        tmem_ld32(acc + c0, v);
        if (MODE == 0) {
          // lanes 0-15 hold gate rows, 16-31 the matching up rows: lane l < 16
          // computes columns 0-15 of its row, lane l + 16 columns 16-31
          const int i = 16 * (4 * cur.mb + qd) + (lane & 15);
          const bool hi = lane >= 16;
#pragma unroll
          for (int qq = 0; qq < 16; ++qq) {
            const float lo_v = __uint_as_float(v[qq]), hi_v = __uint_as_float(v[16 + qq]);
            const float recv = __shfl_xor_sync(0xffffffffu, hi ? lo_v : hi_v, 16);
            const int cq = hi ? 16 + qq : qq;
            const float gv = hi ? recv : lo_v, uv = hi ? hi_v : recv;
            const float sx = __shfl_sync(0xffffffffu, sc_lane[c], cq);
            const int col = c0 + cq;
            if (col < cur.n) {
              const float Gv = (ts_g * sx) * gv, U = (ts_u * sx) * uv;
              const float a = Gv / (1.0f + expf(-Gv)) * U;
              if (p.af)
                p.af[(size_t)(cur.row0 + col) * p.I + i] = a;
              else
                p.abuf[(size_t)(cur.row0 + col) * p.I + i] = a_to_f16(a, p.status);
            }
          }
        } else {
          store_y_chunk(p, v, cur.row0, c0, cur.n, kTcM * cur.mb + 32 * qd, ts_g, sc_lane[c]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[buf]);
      ++uk;
    }
  } else if (warp == kFqMmaWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issue
      FqUnit cur;
      int gs = 0, uk = 0;
      bool ok = true;
      for (int i = 0; ok && fq_unit(p, list, i, n_units, mblocks, cur); ++i) {
        if (cur.n == 0) continue;
        const int n_pad = (cur.n + 15) & ~15, buf = uk & 1;
        const uint32_t idesc = idesc_mxf4nvf4(kTcM, n_pad);
        // the epilogue of the unit before the previous one has read this accumulator
        if (!mbar_wait_fast(&sh->acc_empty[buf], ((uk >> 1) & 1) ^ 1, abort, p.wait_budget)) break;
        tc_fence_after();
        for (int s = 0; s < KS; ++s, ++gs) {
          const int nsub = min(4, KC - 4 * s), slot = gs % kFqNS, ph = (gs / kFqNS) & 1;
          // the scales in tensor memory: their threads committed them after
          // observing the operands' barriers (weight codes, token rows), so
          // the operands are in too (release / acquire through the commits)
          if (!mbar_wait_fast(&sh->sfa[slot], ph, abort, p.wait_budget) ||
              !mbar_wait_fast(&sh->sfb[slot], ph, abort, p.wait_budget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa = tmem_d + kFqSfaCol + 16 * slot, sfb = tmem_d + kFqSfbCol + 16 * slot;
          const uint64_t ad = sw128_desc(a_addr(slot)), bd = sw128_desc(b_addr(slot));
          for (int kk = 0; kk < nsub; ++kk)  // +32 bytes (64 codes) per K-step
            umma_mxf4nvf4(tmem_d + 128 * buf, ad + 2 * kk, bd + 2 * kk, idesc, sfa + 4 * kk,
                          sfb + 4 * kk, (s | kk) != 0);
          umma_commit(&sh->empty[slot]);
        }
        if (ok) umma_commit(&sh->acc_full[buf]);
        ++uk;
      }
      umma_commit(&sh->fin);  // every MMA issued before TMEM is freed
      mbar_drain(&sh->fin, 0);
    }
    __syncwarp();
  } else if (warp == kFqTmaWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA issue
      const CUtensorMap* map = &tmap;
      const uint64_t sc_off = MODE == 1 ? p.mma_dn_sc : p.mma_gu_sc;
      const uint64_t wpol = l2_evict_first(), apol = l2_evict_last();
      int issued = 0;  // stages issued
      FqUnit cur;
      bool ok = true;
      for (int i = 0; ok && fq_unit(p, list, i, n_units, mblocks, cur); ++i) {
        if (cur.n == 0) continue;
        const uint8_t* scales = p.mma + (size_t)cur.expert * p.mma_expert_bytes + sc_off;
        for (int s = 0; s < KS; ++s) {
          const int slot = issued % kFqNS;
          if (!mbar_wait(&sh->empty[slot], ((issued / kFqNS) & 1) ^ 1, abort, p.wait_budget)) {
            ok = false;
            break;
          }
          mbar_arrive_expect(&sh->full_a[slot], (uint32_t)(kFqAStage + kFqSf));
          tma_load_codes(a_addr(slot), map, kTcM * cur.mb, s, cur.expert, &sh->full_a[slot], wpol);
          bulk_load(sa_addr(slot), scales + ((size_t)s * mblocks + cur.mb) * kFqSf, (uint32_t)kFqSf,
                    &sh->full_a[slot], wpol);
          mbar_arrive_expect(&sh->full_bt[slot], (uint32_t)(kFqBStage + kFqSf));
          tma_load_rows(b_addr(slot), &bmap_c, 16 * s, cur.row0, &sh->full_bt[slot], apol);
          tma_load_rows(sn_addr(slot), &bmap_s, 2 * s, cur.row0, &sh->full_bt[slot], apol);
          ++issued;
        }
      }
      if (*abort) {  // let the copies in flight land before the CTA exits (bounded waits)
        for (int c = (issued > kFqNS ? issued - kFqNS : 0); c < issued; ++c) {
          mbar_drain(&sh->full_a[c % kFqNS], (c / kFqNS) & 1);
          mbar_drain(&sh->full_bt[c % kFqNS], (c / kFqNS) & 1);
        }
      }
    }
    __syncwarp();
  } else {
    if (lane == 0) {
      // ---------------------------------------------------------------- scale copies (A: warp 14, B: 15)
      const bool is_a = warp == kFqSfaWarp;
      FqUnit cur;
      int gs = 0;
      bool ok = true;
      for (int i = 0; ok && fq_unit(p, list, i, n_units, mblocks, cur); ++i) {
        if (cur.n == 0) continue;
        for (int s = 0; s < KS; ++s, ++gs) {
          const int nsub = min(4, KC - 4 * s), slot = gs % kFqNS, ph = (gs / kFqNS) & 1;
          if (!mbar_wait_sleep(is_a ? &sh->full_a[slot] : &sh->full_b[slot], ph, abort, p.wait_budget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dst = tmem_d + (is_a ? kFqSfaCol : kFqSfbCol) + 16 * slot;
          const uint32_t src = is_a ? sa_addr(slot) : sb_addr(slot);
          for (int kk = 0; kk < nsub; ++kk) tmem_cp_sf(dst + 4 * kk, sf_desc(src + 512 * kk));
          umma_commit(is_a ? &sh->sfa[slot] : &sh->sfb[slot]);
        }
      }
      umma_commit(&sh->fin2[is_a ? 0 : 1]);  // (its copies done before TMEM is freed)
      mbar_drain(&sh->fin2[is_a ? 0 : 1], 0);
    }
    __syncwarp();
  }

  if (*abort && tid == 0) *p.status = kStatusTimeout;
  tc_fence_before();
  __syncthreads();
  if (warp == kFqMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_d, 512);
  }
}

// ---------------------------------------------------------------- W4A16: the weights in tensor memory
// The expert GEMMs of the W4A16 prefill (f16 activations) with the
// dequantised weights kept in tensor memory: producer warps write each weight
// row's f16 values (e2m1 code x e4m3 block scale, exact in f16) with
// tcgen05.st, and the MMA takes A from there (tcgen05.mma kind::f16 [d], [a],
// b_desc), so only the token rows pass through shared memory.
//
// Persistent like tc_fp4_kernel: a CTA per SM walks units (work item, 128-row
// M-block), its unit list in shared memory.  One thread issuing MMAs into one
// accumulator reaches a fraction of the tensor core's rate (each further
// issuing thread with its own accumulator adds about as much again), so the
// CTA runs two pipelines: pipeline q takes the CTA's units q, q + 2, ..., with
// its own MMA thread, accumulator (128 TMEM columns), two TMA warps, four
// producer warps, a ring of kTmNB token-row stages of 128 columns of K (each
// with a 64-column A slot in TMEM) and a deeper ring of kTmNC code stages, so
// that the codes (from HBM) and their conversion run ahead of the token rows
// and off the path that sets the stage rate.  The epilogue warps serve both
// pipelines, unit after unit, so one pipeline's epilogue overlaps the other's
// MMAs.  Per stage of a pipeline:
//   * its code TMA warp loads the M-block's code vectors of the stage's two
//     64-column chunks (one box of the arena's tile map: the same two 512-byte
//     pieces of 8 consecutive 16-row tiles, 8 KB), at the first chunk of a
//     super-chunk also the tiles' scale vectors (4 KB);
//   * its row TMA warp loads the stage's 128 columns of the item's 128 token
//     rows (two 16 KB boxes, 128B-swizzled: the K-major layout the MMA reads)
//     from rows in slot order: x gathered into them by gather_rows_kernel
//     (gate/up), or a (down); rows past the item's tokens belong to other
//     items and only reach accumulator columns the epilogue never reads;
//   * its producer warps (warp w: TMEM lane quadrant w % 4) rebuild their
//     row's codes from the tile's fragment order (one byte permute per 8
//     codes), convert and scale them to f16 and store 64 TMEM columns, then
//     arrive once per warp;
//   * its MMA thread issues the stage's 8 MMAs (K = 16 each) and commits the
//     stage (its shared memory and its A slot) back;
//   * epilogue warps 8-15 read a finished unit's accumulator (SwiGLU into a,
//     or y rows) and hand it back to its pipeline.
constexpr int kTmPipes = 2;                        // pipelines (MMA issuers)
constexpr int kTmProd = 4;                         // producer warps per pipeline
constexpr int kTmEpi0 = kTmPipes * kTmProd;        // epilogue warps 8-15
constexpr int kTmMmaWarp = kTmEpi0 + 8;            // MMA warps 16 + q
constexpr int kTmTmaWarp = kTmMmaWarp + kTmPipes;  // TMA warps: token rows 18 + q, codes 20 + q
constexpr int kTmThreads = 32 * (kTmTmaWarp + 2 * kTmPipes);
constexpr int kTmK = 128;                      // K per stage: two 64-column chunks
constexpr int kTmNB = 2;                       // token-row stages (and A slots) per pipeline
constexpr int kTmNC = 3;                       // code stages per pipeline
constexpr int kTmB = 2 * kTcMaxN * 128;        // token rows of a stage: 2 x (128 rows x 64 f16)
constexpr int kTmCodes = 2 * 8 * 512;          // two 512-byte pieces of 8 tiles
constexpr int kTmScales = 8 * 512;             // the scale vectors of 8 tiles
constexpr int kTmCStage = kTmCodes + kTmScales;
constexpr uint32_t kTmACol = 256;              // A slots (64 columns each) after the two accumulators
static_assert(kTmACol + 64 * kTmPipes * kTmNB <= 512, "tensor memory columns");
static_assert(kTmB % 1024 == 0 && kTmCStage % 1024 == 0, "stages stay 1024-byte aligned");

struct TmShared {
  uint64_t bfull[kTmPipes * kTmNB];   // the stage's token rows landed (transaction bytes)
  uint64_t afull[kTmPipes * kTmNB];   // the stage's A slot is written (the pipeline's producer warps)
  uint64_t empty[kTmPipes * kTmNB];   // the MMAs reading the token rows and the A slot are done
  uint64_t cfull[kTmPipes * kTmNC];   // the stage's codes (+ scales) landed (transaction bytes)
  uint64_t cempty[kTmPipes * kTmNC];  // the producers have read them
  uint64_t acc_full[kTmPipes], acc_empty[kTmPipes];
  uint64_t fin[kTmPipes];
  uint32_t tmem_base;
  int abort;
};

constexpr int kTmStaging = 8 * 1024;  // the epilogue warps' a tiles (gate/up): 32 columns x 16 rows of f16 each
constexpr size_t kTmRings = (size_t)kTmPipes * (kTmNB * kTmB + kTmNC * kTmCStage);

__host__ __device__ constexpr size_t tm_smem_bytes() {
  return 1024 + kTmRings + kTmStaging + sizeof(TmShared) + 16 + 16 * kFqList;
}

// 4-D tiled TMA load of the tile map box at (0, piece, tile, expert) with an L2 policy
__device__ __forceinline__ void tma_load_tiles_pol(uint32_t dst, const CUtensorMap* map, int piece,
                                                   int tile, int expert, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(piece), "r"(tile), "r"(expert),
      "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}


// 32 TMEM lanes (one per thread of the warp) x 32 consecutive 32-bit columns
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D (TMEM) += A (TMEM, 128 lanes x 8 columns of f16 pairs) . B (shared memory)^T
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// One row's 16-column block from a lane's 16-byte code vector of the packed
// tile (word w: bytes [(g, 4w..4w+1), (g+8, 4w..4w+1), (g, 4w+2..), (g+8, 4w+2..)],
// two codes a byte): `sel` picks row g's bytes (0x6420) or row g+8's (0x7531)
// in column order; each f16 pair is multiplied by the block scale `sc` (both
// halves the scale).
__device__ __forceinline__ void tm_block(const uint4& cv, uint32_t sel, uint32_t sc, uint32_t* out) {
  uint32_t hh[4];
  e2m1x8_to_f16x8(prmt(cv.x, cv.y, sel), hh);
#pragma unroll
  for (int k = 0; k < 4; ++k) out[k] = hmul2(hh[k], sc);
  e2m1x8_to_f16x8(prmt(cv.z, cv.w, sel), hh);
#pragma unroll
  for (int k = 0; k < 4; ++k) out[4 + k] = hmul2(hh[k], sc);
}

// The token rows of the gate/up GEMM in slot order: row r of xs = x's row of
// token row_token[r] (r < T*k), or of token r - T*k (the shared expert's
// rows), converted from bf16 to f16 (exact for |x| in [2^-14, 65504]; an
// element beyond 65504, or not finite, records MOE_ERANGE); a warp per row.
// from_f16: copied from the f16 copy of x instead (x in host memory mapped
// for the device: read once by the conversion, not once per row here).
__global__ void __launch_bounds__(256) gather_rows_kernel(ExpertParams p, int rows, uint16_t* xs,
                                                          int from_f16) {
  griddep_wait();
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int S = p.T * p.k;
  const int t = r >= S ? r - S : p.row_token[r];
  if (t < 0 || t >= p.T) {
    if (lane == 0) *p.status = kStatusInvalid;
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)r * p.H);
  const int n16 = p.H / 8;  // 16-byte vectors of a row; 4 of a lane's in flight at once
  if (from_f16) {
    const uint4* h = reinterpret_cast<const uint4*>(p.xh + (size_t)t * p.H);
    for (int v0 = lane; v0 < n16; v0 += 128) {
      uint4 w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < n16) w[u] = h[v0 + 32 * u];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < n16) dst[v0 + 32 * u] = w[u];
    }
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H);
  bool bad = false;
  for (int v0 = lane; v0 < n16; v0 += 128) {
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (v0 + 32 * u < n16) raw[u] = src[v0 + 32 * u];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (v0 + 32 * u >= n16) break;
      const uint32_t in[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2 h = __floats2half2_rn(__uint_as_float(in[q] << 16), __uint_as_float(in[q] & 0xFFFF0000u));
        o[q] = *reinterpret_cast<const uint32_t*>(&h);
        bad |= f16x2_nonfinite(o[q]);
      }
      dst[v0 + 32 * u] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  if (bad) *p.status = kStatusRange;
}

template <int MODE>
__global__ void __launch_bounds__(kTmThreads, 1)
    tc_tmem_kernel(ExpertParams p, const __grid_constant__ CUtensorMap tmap,
                   const __grid_constant__ CUtensorMap smap, const __grid_constant__ CUtensorMap bmap,
                   int max_items) {
  griddep_wait();
  extern __shared__ __align__(1024) uint8_t tm_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tm_smem_raw) + 1023) & ~(uintptr_t)1023);
  TmShared* sh = reinterpret_cast<TmShared*>(base + kTmRings + kTmStaging);
  int4* list = reinterpret_cast<int4*>((reinterpret_cast<uintptr_t>(sh + 1) + 15) & ~(uintptr_t)15);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = MODE == 1 ? p.I : p.H;
  const int KC = K / kTmK;  // stages per unit
  const int mblocks = (MODE == 1 ? p.H : 2 * p.I) / kTcM;
  const int items = min(p.nsh_tc + *p.n_tc_entries, max_items);
  const int n_units = mblocks * max(items, 0);
  const uint32_t s0 = smem_u32(base);
  // token-row slot r = q * kTmNB + b; code slot r = q * kTmNC + c (all 1024-byte aligned)
  auto b_addr = [&](int r) { return s0 + r * kTmB; };
  auto c_addr = [&](int r) { return s0 + kTmPipes * kTmNB * kTmB + r * kTmCStage; };  // [tile][piece 0..1][512 B]
  auto v_addr = [&](int r) { return c_addr(r) + kTmCodes; };  // [tile][512 B]

  if (tid == 0) {
    for (int i = 0; i < kTmPipes * kTmNB; ++i) {
      mbar_init(&sh->bfull[i], 1);
      mbar_init(&sh->afull[i], kTmProd);  // the pipeline's producer warps
      mbar_init(&sh->empty[i], 1);
    }
    for (int i = 0; i < kTmPipes * kTmNC; ++i) {
      mbar_init(&sh->cfull[i], 1);
      mbar_init(&sh->cempty[i], kTmProd);
    }
    for (int i = 0; i < kTmPipes; ++i) {
      mbar_init(&sh->acc_full[i], 1);
      mbar_init(&sh->acc_empty[i], 8);  // the 8 epilogue warps
      mbar_init(&sh->fin[i], 1);
    }
    sh->abort = 0;
    mbar_init_fence();
  }
  if (warp == 0) {  // the unit list: {expert, first row, tokens, M-block}
    for (int i = lane; i < kFqList; i += 32) {
      const int u = blockIdx.x + i * gridDim.x;
      int4 v = make_int4(0, 0, 0, 0);
      if (u < n_units) {
        int e, r0, n;
        v = tc_entry(p, u / mblocks, e, r0, n) ? make_int4(e, r0, n, u % mblocks)
                                               : make_int4(0, 0, 0, u % mblocks);
      }
      list[i] = v;
    }
  }
  if (warp == kTmMmaWarp) tmem_alloc(&sh->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = sh->tmem_base;
  volatile int* abort = &sh->abort;
  // (every role walks the CTA's units in the same order; uk counts the units
  // with tokens, and unit uk belongs to pipeline uk % 2)

  if (warp < kTmEpi0) {
    // ---------------------------------------------------------------- producers: A into TMEM
    // row r of the M-block = TMEM lane r: tile r / 16, row g or g + 8 of it
    const int q = warp / kTmProd, qd = warp & 3;
    const int r = 32 * qd + lane, tile = r >> 4, g8 = lane & 7, hi = (lane >> 3) & 1;
    const uint32_t sel = hi ? 0x7531u : 0x6420u;
    // the lanes (g8, t) of the tile's vectors hold this row's 16-column block t
    // of every chunk (scales: byte 2j + hi of the scale vector, chunk j)
    const uint32_t loff = (uint32_t)(tile * 512 + 64 * g8);
    const uint32_t tdst = tmem_d + ((uint32_t)(32 * qd) << 16) + kTmACol;
    uint4 sv[4];  // the super-chunk's scale vectors of lanes (g8, 0..3)
#pragma unroll
    for (int t = 0; t < 4; ++t) sv[t] = make_uint4(0, 0, 0, 0);
    int gs = 0, uk = 0;
    FqUnit cur;
    bool ok = true;
    for (int i = 0; ok && fq_unit(p, list, i, n_units, mblocks, cur); ++i) {
      if (cur.n == 0) continue;
      if ((uk++ & 1) != q) continue;
      for (int c = 0; c < KC; ++c, ++gs) {
        const int rb = q * kTmNB + gs % kTmNB, rc = q * kTmNC + gs % kTmNC;
        const int j0 = 2 * (c & 3);  // chunks j0, j0 + 1 of the super-chunk
        // the stage's codes landed; the MMAs that last read the A slot are done
        if (!__all_sync(0xffffffffu, mbar_wait_fast(&sh->cfull[rc], (gs / kTmNC) & 1, abort, p.wait_budget) &&
                                          mbar_wait_fast(&sh->empty[rb], ((gs / kTmNB) & 1) ^ 1, abort,
                                                         p.wait_budget))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (j0 == 0) {  // the super-chunk's scale vectors, kept for its 8 chunks
#pragma unroll
          for (int t = 0; t < 4; ++t) sv[t] = lds128(v_addr(rc) + loff + 16 * t);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // the stage's two chunks
          const int sb = 2 * (j0 + hh) + hi;
          uint32_t v[32];
#pragma unroll
          for (int t = 0; t < 4; ++t) {  // 16-column block t: TMEM columns 8t .. 8t + 7 of the chunk
            const uint4 cv = lds128(c_addr(rc) + tile * 1024 + hh * 512 + 64 * g8 + 16 * t);
            const uint32_t e = (u4get(sv[t], sb >> 2) >> (8 * (sb & 3))) & 0xFFu;
            const uint32_t sp = e4m3x2_to_f16x2(e | (e << 8));
            tm_block(cv, sel, sp, v + 8 * t);
          }
          tmem_st32(tdst + 64 * rb + 32 * hh, v);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->cempty[rc]);  // (every lane's code reads are done)
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->afull[rb]);
      }
    }
  } else if (warp < kTmMmaWarp) {
    // ---------------------------------------------------------------- epilogue
    // warp 8 + 4h + q: TMEM lane quadrant q (rows 32q..32q+31), columns 64h..64h+63
    const int qd = warp & 3, ch = (warp - kTmEpi0) >> 2;
    const uint32_t lane_addr = (uint32_t)(32 * qd) << 16;
    const uint32_t tile = s0 + (uint32_t)kTmRings + (warp - kTmEpi0) * 1024;
    FqUnit cur;
    int uk = 0;
    for (int i = 0; fq_unit(p, list, i, n_units, mblocks, cur); ++i) {
      if (cur.n == 0) continue;
      const int n_pad = (cur.n + 15) & ~15, buf = uk & 1;  // (the unit's pipeline)
      // the unit's tensor scales, read before the accumulator wait (an L2 round
      // trip under this load takes about a microsecond)
      const float ts_g = p.tscale[cur.expert * 3 + (MODE == 1 ? 2 : 0)];
      const float ts_u = MODE == 0 ? p.tscale[cur.expert * 3 + 1] : 0.0f;
      if (!mbar_wait_sleep(&sh->acc_full[buf], (uk >> 1) & 1, abort, p.wait_budget)) break;
      tc_fence_after();
      const uint32_t acc = tmem_d + lane_addr + (uint32_t)(128 * buf);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int c0 = 64 * ch + 32 * c;
        if (c0 >= n_pad) break;
        uint32_t v[32];
        tmem_ld32(acc + c0, v);
        if (MODE == 0) {
          // lanes 0-15 hold gate rows, 16-31 the matching up rows: lane l < 16
          // computes columns 0-15 of its row, lane l + 16 columns 16-31.  The
          // f16 values go through the warp's tile [32 columns][16 rows of a],
          // so that a store instruction writes 16 columns x 32 bytes of a.
          const bool hi = lane >= 16;
          bool bad = false;
#pragma unroll
          for (int qq = 0; qq < 16; ++qq) {
            const float lo_v = __uint_as_float(v[qq]), hi_v = __uint_as_float(v[16 + qq]);
            const float recv = __shfl_xor_sync(0xffffffffu, hi ? lo_v : hi_v, 16);
            const int cq = hi ? 16 + qq : qq;
            const float gv = hi ? recv : lo_v, uv = hi ? hi_v : recv;
            const float Gv = ts_g * gv, U = ts_u * uv;
            // (the fast exponential and division: a becomes f16, 11 bits, so their few
            // ulps of fp32 error do not show; the epilogue stays short of the MMAs)
            const float a = __fdividef(Gv, 1.0f + __expf(-Gv)) * U;
            const uint16_t h = __half_as_ushort(__float2half_rn(a));
            // (columns past the item's tokens hold stale accumulators: never stored, never flagged)
            bad |= c0 + cq < cur.n && f16_nonfinite(h);
            st_shared_u16(tile + cq * 32 + (lane & 15) * 2, h);
          }
          if (bad) *p.status = kStatusRange;
          __syncwarp();
          // lane j: column 16g + j / 2 of the chunk, rows 8 (j % 2) .. + 7 of the 16
          const int i0 = 16 * (4 * cur.mb + qd);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int cq = 16 * g + (lane >> 1), col = c0 + cq;
            const uint4 w = lds128(tile + cq * 32 + (lane & 1) * 16);
            if (col < cur.n)
              *reinterpret_cast<uint4*>(p.abuf + (size_t)(cur.row0 + col) * p.I + i0 + 8 * (lane & 1)) = w;
          }
          __syncwarp();  // (the next chunk rewrites the tile)
        } else {
          store_y_chunk(p, v, cur.row0, c0, cur.n, kTcM * cur.mb + 32 * qd, ts_g, 1.0f);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[buf]);
      ++uk;
    }
  } else if (warp < kTmTmaWarp) {
    const int q = warp - kTmMmaWarp;
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issue (pipeline q)
      FqUnit cur;
      int gs = 0, uk = 0;
      bool ok = true;
      for (int i = 0; ok && fq_unit(p, list, i, n_units, mblocks, cur); ++i) {
        if (cur.n == 0) continue;
        const int me = uk++;
        if ((me & 1) != q) continue;
        const int n_pad = (cur.n + 15) & ~15;
        const uint32_t idesc = idesc_f16(kTcM, n_pad);
        // the epilogue has read this pipeline's accumulator (its previous unit)
        if (!mbar_wait_fast(&sh->acc_empty[q], ((me >> 1) & 1) ^ 1, abort, p.wait_budget)) break;
        tc_fence_after();
        for (int c = 0; c < KC; ++c, ++gs) {
          const int rs = q * kTmNB + gs % kTmNB;
          const uint32_t ph = (gs / kTmNB) & 1;
          if (!mbar_wait_fast(&sh->afull[rs], ph, abort, p.wait_budget) ||
              !mbar_wait_fast(&sh->bfull[rs], ph, abort, p.wait_budget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = sw128_desc(b_addr(rs));
          const uint32_t a0 = tmem_d + kTmACol + 64 * rs;
#pragma unroll
          for (int kk = 0; kk < kTmK / 16; ++kk)  // A: +8 columns per K-step of 16; B: +32 bytes
            // within a 64-column box, the second box 16 KB on
            umma_f16_tmem_a(tmem_d + 128 * q, a0 + 8 * kk, bd + 2 * (kk & 3) + (kk >> 2) * (kTcMaxN * 128 >> 4),
                            idesc, (c | kk) != 0);
          umma_commit(&sh->empty[rs]);
        }
        if (ok) umma_commit(&sh->acc_full[q]);
      }
      umma_commit(&sh->fin[q]);  // every MMA issued before TMEM is freed
      mbar_drain(&sh->fin[q], 0);
    }
    __syncwarp();
  } else {
    const int q = (warp - kTmTmaWarp) % kTmPipes;
    const bool rows = warp < kTmTmaWarp + kTmPipes;  // token rows, else codes
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA issue (pipeline q)
      const CUtensorMap* map = &tmap;
      const uint64_t wpol = l2_evict_first(), apol = l2_evict_last();
      const int depth = rows ? kTmNB : kTmNC;
      uint64_t* full = rows ? sh->bfull + q * kTmNB : sh->cfull + q * kTmNC;
      uint64_t* empty = rows ? sh->empty + q * kTmNB : sh->cempty + q * kTmNC;
      int gs = 0, uk = 0;
      FqUnit cur;
      bool ok = true;
      for (int i = 0; ok && fq_unit(p, list, i, n_units, mblocks, cur); ++i) {
        if (cur.n == 0) continue;
        if ((uk++ & 1) != q) continue;
        for (int c = 0; c < KC; ++c, ++gs) {
          const int slot = gs % depth, j0 = 2 * (c & 3), sc = c >> 2;
          if (!mbar_wait_sleep(&empty[slot], ((gs / depth) & 1) ^ 1, abort, p.wait_budget)) {
            ok = false;
            break;
          }
          if (rows) {
            const uint32_t dst = b_addr(q * kTmNB + slot);
            mbar_arrive_expect(&full[slot], (uint32_t)kTmB);
            tma_load_rows(dst, &bmap, kTmK * c, cur.row0, &full[slot], apol);
            tma_load_rows(dst + kTcMaxN * 128, &bmap, kTmK * c + kTcK, cur.row0, &full[slot], apol);
          } else {
            const int r = q * kTmNC + slot;
            mbar_arrive_expect(&full[slot], (uint32_t)kTmCodes + (j0 == 0 ? (uint32_t)kTmScales : 0u));
            tma_load_tiles_pol(c_addr(r), map, 9 * sc + 1 + j0, 8 * cur.mb, cur.expert, &full[slot], wpol);
            if (j0 == 0) tma_load_tiles_pol(v_addr(r), &smap, 9 * sc, 8 * cur.mb, cur.expert, &full[slot], wpol);
          }
        }
      }
      if (*abort) {  // let this warp's copies in flight land before the CTA exits (bounded waits)
        for (int c = (gs > depth ? gs - depth : 0); c < gs; ++c) mbar_drain(&full[c % depth], (c / depth) & 1);
      }
    }
    __syncwarp();
  }

  if (*abort && tid == 0) *p.status = kStatusTimeout;
  tc_fence_before();
  __syncthreads();
  if (warp == kTmMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_d, 512);
  }
}

}  // namespace

// M-blocks per CTA of the TMA-fed expert GEMMs: 4 where they divide the matrix
int tc_group(int mblocks) { return mblocks % 4 == 0 ? 4 : (mblocks % 2 == 0 ? 2 : 1); }

cudaError_t tc_make_tile_map(void* map, const uint8_t* region, int n_experts, int tiles,
                             uint64_t tile_bytes, uint64_t expert_bytes, int box_tiles, int box_pieces) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // [expert][tile][512-byte piece][64 x 8 bytes]; a box: box_pieces consecutive
  // pieces of box_tiles consecutive tiles
  const cuuint64_t dims[4] = {64, (cuuint64_t)(tile_bytes / 512), (cuuint64_t)tiles,
                              (cuuint64_t)n_experts};
  const cuuint64_t strides[3] = {512, tile_bytes, expert_bytes};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_pieces, (cuuint32_t)box_tiles, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = encode(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT64, 4,
                            const_cast<uint8_t*>(region), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// [expert][stage][row][128 B] codes of the MMA layout; a box: the 128 bytes
// (256 codes) of box_rows consecutive rows of a stage, 128B-swizzled as the
// MMA reads them
cudaError_t tc_make_mma_map(void* map, const uint8_t* codes, int n_experts, int rows, int stages,
                            uint64_t expert_stride, int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // (the bytes viewed as 8-byte elements: 16 to a 128-byte row)
  const cuuint64_t dims[4] = {16, (cuuint64_t)rows, (cuuint64_t)stages, (cuuint64_t)n_experts};
  const cuuint64_t strides[3] = {128, (cuuint64_t)rows * 128, expert_stride};
  const cuuint32_t box[4] = {16, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = encode(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT64, 4,
                            const_cast<uint8_t*>(codes), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// [rows][row_bytes] activation rows; a box: 128 rows of 128 bytes (codes,
// 128B-swizzled) or of 16 bytes (scales, as they are)
cudaError_t tc_make_rows_map(void* map, const uint8_t* base, size_t rows, int row_bytes, bool codes) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // (8-byte elements: 16 to a 128-byte box row, 2 to a 16-byte one)
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes / 8, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {codes ? 16u : 2u, (cuuint32_t)kTcMaxN};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT64, 2,
                            const_cast<uint8_t*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE,
                            codes ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

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

cudaError_t launch_tc_gateup(const ExpertParams& p, int grid_y, const void* tile_map,
                             cudaStream_t st) {
  const int mblocks = (2 * p.I) / kTcM, G = tc_group(mblocks);
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(tile_map);
  return launch_k(tc_expert_kernel<0>, dim3(mblocks / G, grid_y), dim3(kTxThreads),
                  tx_smem_bytes(G), st, true, p, map, G);
}

cudaError_t launch_tc_down(const ExpertParams& p, int grid_y, const void* tile_map,
                           cudaStream_t st) {
  const int mblocks = p.H / kTcM, G = tc_group(mblocks);
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(tile_map);
  return launch_k(tc_expert_kernel<1>, dim3(mblocks / G, grid_y), dim3(kTxThreads),
                  tx_smem_bytes(G), st, true, p, map, G);
}

// M-blocks per work unit of the block-scaled FP4 GEMMs (one: the accumulators are double-buffered)
int tc_fp4_group(int) { return 1; }

// persistent grid: one CTA per SM, or one per unit when there are fewer
static int fq_grid(int units) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      sms = 1;
  }
  return units < sms ? (units > 0 ? units : 1) : sms;
}

cudaError_t launch_tc_fp4_gateup(const ExpertParams& p, int items, const void* tile_map,
                                 const void* bmap_c, const void* bmap_s, cudaStream_t st) {
  const int mblocks = (2 * p.I) / kTcM;
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(tile_map);
  const CUtensorMap& bc = *reinterpret_cast<const CUtensorMap*>(bmap_c);
  const CUtensorMap& bs = *reinterpret_cast<const CUtensorMap*>(bmap_s);
  return launch_k(tc_fp4_kernel<0>, dim3(fq_grid(mblocks * items)), dim3(kFqThreads),
                  fq_smem_bytes(), st, true, p, map, bc, bs, items);
}

cudaError_t launch_tc_fp4_down(const ExpertParams& p, int items, const void* tile_map,
                               const void* bmap_c, const void* bmap_s, cudaStream_t st) {
  const int mblocks = p.H / kTcM;
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(tile_map);
  const CUtensorMap& bc = *reinterpret_cast<const CUtensorMap*>(bmap_c);
  const CUtensorMap& bs = *reinterpret_cast<const CUtensorMap*>(bmap_s);
  return launch_k(tc_fp4_kernel<1>, dim3(fq_grid(mblocks * items)), dim3(kFqThreads),
                  fq_smem_bytes(), st, true, p, map, bc, bs, items);
}

// [rows][cols] f16 rows in slot order (x gathered, or a); a box: 64 columns
// of 128 rows, 128B-swizzled
cudaError_t tc_make_rows16_map(void* map, const uint16_t* base, size_t rows, int cols) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTcK, (cuuint32_t)kTcMaxN};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                            const_cast<uint16_t*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gather_rows(const ExpertParams& p, int rows, uint16_t* xs, bool from_f16, cudaStream_t st) {
  const int blocks = (rows + 7) / 8;
  return launch_k(gather_rows_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, st, true, p, rows, xs,
                  from_f16 ? 1 : 0);
}

bool tc_tm_ok(int H, int I) { return H % kTmK == 0 && I % kTmK == 0; }

cudaError_t launch_tc_tm_gateup(const ExpertParams& p, int items, const void* code_map,
                                const void* scale_map, const void* xmap, cudaStream_t st) {
  const int mblocks = (2 * p.I) / kTcM;
  const CUtensorMap& cm = *reinterpret_cast<const CUtensorMap*>(code_map);
  const CUtensorMap& sm = *reinterpret_cast<const CUtensorMap*>(scale_map);
  const CUtensorMap& bm = *reinterpret_cast<const CUtensorMap*>(xmap);
  return launch_k(tc_tmem_kernel<0>, dim3(fq_grid(mblocks * items)), dim3(kTmThreads),
                  tm_smem_bytes(), st, true, p, cm, sm, bm, items);
}

cudaError_t launch_tc_tm_down(const ExpertParams& p, int items, const void* code_map,
                              const void* scale_map, const void* amap, cudaStream_t st) {
  const int mblocks = p.H / kTcM;
  const CUtensorMap& cm = *reinterpret_cast<const CUtensorMap*>(code_map);
  const CUtensorMap& sm = *reinterpret_cast<const CUtensorMap*>(scale_map);
  const CUtensorMap& bm = *reinterpret_cast<const CUtensorMap*>(amap);
  return launch_k(tc_tmem_kernel<1>, dim3(fq_grid(mblocks * items)), dim3(kTmThreads),
                  tm_smem_bytes(), st, true, p, cm, sm, bm, items);
}

bool tc_router_ok(int E, int H) { return E % kTcM == 0 && H % kTcK == 0; }

// logits_out gets the fp32 dot products (one K slice: the top-k step adds the bias)
cudaError_t launch_tc_router(const ExpertParams& p, cudaStream_t st) {
  dim3 grid(p.E / kTcM, (p.T + kTcMaxN - 1) / kTcMaxN);
  return launch_k(tc_router_kernel, grid, dim3(kTcThreads), tc_smem(), st, true, p);
}

cudaError_t tc_kernels_init() {
  cudaError_t e = cudaFuncSetAttribute(tc_expert_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tx_smem_bytes(kTxMaxG));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_expert_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tx_smem_bytes(kTxMaxG));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_fp4_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)fq_smem_bytes());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_fp4_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)fq_smem_bytes());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_tmem_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tm_smem_bytes());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_tmem_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tm_smem_bytes());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tc_smem());
}

}  // namespace moe
