// Launchers of the layer's kernels (implemented in quant_pack.cu, route.cu, expert.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

constexpr int kTokTile = 8;     // tokens per expert entry (the n of m16n8k16)
constexpr int kTcMaxN = 128;    // tokens per entry of the tensor-core path
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxKsplitHost = 8;  // router K slices at most (router_ksplit)

// Everything the expert kernels read or write for one forward.
struct ExpertParams {
  const uint8_t* arena;
  const uint8_t* const* eptr;  // [E + shared] base of each expert, or null: arena + e * expert_bytes
  uint64_t expert_bytes;
  uint64_t gu_bytes;
  int gu_tile_bytes, dn_tile_bytes;
  const float* tscale;   // [(E + shared) * 3]
  int fmt, H, I, E, T, k, shared;
  int nsh;               // leading shared-expert entries: ceil(T / 8) or 0
  int nsh_tc;            // leading shared-expert entries of the tensor-core path: ceil(T / 256)
  const int4* tc_entries;  // routed entries of up to kTcMaxN tokens
  const int* n_tc_entries;
  const int4* entries;   // routed entries {expert, first row, tokens, 0}
  const int* n_entries;  // number of routed entries
  const int* row_token;  // [T*k + T] token of each row of abuf / ybuf
  const uint16_t* x;     // bf16 [T x H]
  const uint16_t* xh;    // f16 copy of x [T x H] (written by the router)
  uint16_t* abuf;        // f16 bits [(T*k + T) x I]: silu(g) * u per row
  float* ybuf;           // [(T*k + T) x H]: ts_down * (W_down a) per row
  const uint16_t* wr;    // router weights bf16 [E x H] (tensor-core router only)
  const float* rbias;    // router bias [E] or null (tensor-core router only)
  float* logits_out;     // router logits [T x E] (tensor-core router only)
  int* status;
  long long wait_budget; // clock64 cycles one bounded wait of the tensor-core kernels may take
  // W4A4 (activations quantised to NVFP4 per row), else all null: the f16
  // copies of x (xh) and of a (abuf) then hold the activations' e2m1 code x
  // e4m3 block scale (exact in f16) and these fp32 tensor scales multiply the
  // accumulators; the gate/up kernels write a in fp32 to af for the quantiser
  const float* ts_x;     // [T] per token
  const float* ts_a;     // [T*k + T] per row of abuf
  float* af;             // [(T*k + T) x I] fp32 a before quantisation
  // the weights in the MMA layout (layout.cuh): per expert mma_expert_bytes,
  // the gate/up and down block scales at mma_gu_sc and mma_dn_sc
  const uint8_t* mma;
  uint64_t mma_expert_bytes, mma_gu_sc, mma_dn_sc;
};

#ifdef __CUDACC__
// First byte of expert e's packed matrices: in the arena, or wherever the
// per-expert table puts it (an HBM slot or the pinned host mirror).
__device__ __forceinline__ const uint8_t* expert_base(const ExpertParams& p, int e) {
  return p.eptr ? p.eptr[e] : p.arena + (size_t)e * p.expert_bytes;
}
#endif

// Router modes: softmax over the logits (the bias is part of the logit), or
// sigmoid scores with the bias deciding the selection only.
enum { ROUTER_SOFTMAX = 0, ROUTER_SIGMOID = 1 };

struct RouteParams {
  const uint16_t* x;      // bf16 [T x H]
  uint16_t* xh;           // f16 copy of x, written by the router (may be null)
  const uint16_t* wr;     // bf16 [E x H]
  const float* bias;      // [E] or null
  int T, H, E, k, shared, ksplit;
  int mode;               // ROUTER_SOFTMAX or ROUTER_SIGMOID
  float* partial;         // [ksplit x T x E] router partial dot products
  float* logits;          // [T x E]
  int* idx;               // [T x k]
  float* gates;           // [T x k]
  int* counts;            // [E]
  int* offsets;           // [E + 1]
  int* perm;              // [T*k] slot ids in expert-sorted order
  int* inv;               // [T*k] row of each slot
  int* row_token;         // [T*k + T]
  int4* entries;
  int* n_entries;
  int4* tc_entries;       // optional: entries of up to kTcMaxN tokens (tensor-core path)
  int* n_tc_entries;
  int* blk;               // [ceil(T*k / kDispChunk) x E] per-chunk expert counts, then bases
  int* ticket;            // CTAs of the fused top-k + dispatch done so far (0 between forwards)
  int* status;
};

// Slots per CTA of the several-CTA dispatch (count, then scan + place), used when
// T*k is above kDispOneCtaMax; below it one CTA does the whole dispatch.
constexpr int kDispChunk = 1024;
constexpr int kDispOneCtaMax = 8192;

cudaError_t launch_quantize_nvfp4(const float* W, int rows, int K, uint8_t* codes,
                                  uint8_t* scales, float* tscale, cudaStream_t st);
cudaError_t launch_quantize_fp6(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps,
                                cudaStream_t st);
cudaError_t launch_quantize_mxfp4(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps,
                                  cudaStream_t st);
cudaError_t launch_mx_to_tile_scales(const uint8_t* codes, const uint8_t* exps, int rows, int K,
                                     uint8_t* nv_scales, float* ts_dst, int* bad, cudaStream_t st);
cudaError_t launch_pack(int fmt, const uint8_t* codes, const uint8_t* scales, int rows, int K,
                        uint8_t* dst, uint64_t tile_stride, const float* ts_src, float ts_val,
                        float* ts_dst, cudaStream_t st);
cudaError_t launch_debug_dequant(int fmt, const uint8_t* src, uint64_t tile_stride, int rows,
                                 int K, const float* ts_ptr, float* out, cudaStream_t st);
// The packed NVFP4 tiles of one matrix region (src_off into each expert,
// rows M, K columns) of n_experts experts into the MMA layout (layout.cuh) at
// dst (dst_expert_bytes per expert; the region's codes and scales at
// codes_off and scales_off).
cudaError_t launch_to_mma_layout(const uint8_t* arena, uint64_t expert_bytes, uint64_t src_off,
                                 int tile_bytes, int M, int K, int n_experts, uint8_t* dst,
                                 uint64_t dst_expert_bytes, uint64_t codes_off, uint64_t scales_off,
                                 cudaStream_t st);
// Activations to NVFP4 per row (the weights' recipe with one tensor scale per
// row): in [rows x K] bf16 (in_bf16) or fp32; optional outputs: canonical
// codes (rows cpitch bytes apart, default K/2) and e4m3 scales (spitch apart,
// default K/16), the f16 values e2m1 code x e4m3 scale [rows x K] (exact), and
// the tensor scales ts [rows].  With inv, input row t's codes and scales go to
// the kd output rows inv[t*kd + j] and, if shared_base >= 0, to row
// shared_base + t.  A row whose amax is not finite records MOE_ERANGE in
// *status (if status).  pdl: may start while the previous kernel drains.
cudaError_t launch_quantize_act(const void* in, bool in_bf16, int rows, int K, uint8_t* codes,
                                uint8_t* scales, uint16_t* out_f16, float* ts, int* status,
                                bool pdl, cudaStream_t st, int cpitch = 0, int spitch = 0,
                                const int* inv = nullptr, int kd = 0, int shared_base = -1);

// routing
int router_ksplit(int T, int H, int E);
// pdl: may start while the previous kernel on the stream drains (it then reads
// the router weights before its wait: they must not be written by that kernel)
cudaError_t launch_router(const RouteParams& p, cudaStream_t st, bool pdl = true);
cudaError_t launch_route_finish(const RouteParams& p, bool do_topk, bool pdl, cudaStream_t st);
// Dispatch of p.idx (top-k done): one CTA, or count and scan + place kernels
// for T*k > kDispOneCtaMax.  dispatch_launches: how many kernels that is.
cudaError_t launch_dispatch(const RouteParams& p, bool pdl, cudaStream_t st);
int dispatch_launches(int S);
cudaError_t launch_topk(const RouteParams& p, bool pdl, cudaStream_t st);
// Top-k and dispatch in one launch (topk_dispatch_kernel) when topk_dispatch_ok.
bool topk_dispatch_ok(int T, int k, int E);
cudaError_t launch_topk_dispatch(const RouteParams& p, bool pdl, cudaStream_t st);
size_t route_finish_smem(int E);
cudaError_t route_kernels_init();

// experts
cudaError_t launch_gateup(const ExpertParams& p, int grid_y, bool pdl, cudaStream_t st);
cudaError_t launch_down(const ExpertParams& p, int grid_y, bool pdl, cudaStream_t st);
cudaError_t launch_combine(const ExpertParams& p, const float* gates, const int* inv, float* out,
                           bool pdl, cudaStream_t st);
bool down_combine_ok(int T, int k, int shared, int I);
cudaError_t launch_down_combine(const ExpertParams& p, const float* gates, const int* inv,
                                float* out, bool pdl, bool wait_first, cudaStream_t st);

// T <= 8: gate/up that routes itself and publishes the routing (expert.cu)
bool small_route_ok(int T, int k);
cudaError_t launch_gateup_routed(const ExpertParams& p, const RouteParams& rp, int grid_y,
                                 cudaStream_t st);
cudaError_t expert_kernels_init();
// the f16 copy of x (n elements); MOE_ERANGE in *status for |x| beyond f16's range
cudaError_t launch_convert_x(const uint16_t* x, uint16_t* xh, long n, int* status, cudaStream_t st);

// tensor-core (tcgen05) prefill path
bool tc_path_ok(int fmt, int T, int k, int E, int H, int I);
int max_tc_entries(int T, int E, int k);
// tile_map: the CUtensorMap (128 bytes, 64-byte aligned) of the matrix region,
// made by tc_make_tile_map with box_tiles = 8 * tc_group(M-blocks of the matrix)
int tc_group(int mblocks);
cudaError_t tc_make_tile_map(void* map, const uint8_t* region, int n_experts, int tiles,
                             uint64_t tile_bytes, uint64_t expert_bytes, int box_tiles,
                             int box_pieces = 1);
cudaError_t launch_tc_gateup(const ExpertParams& p, int grid_y, const void* tile_map,
                             cudaStream_t st);
cudaError_t launch_tc_down(const ExpertParams& p, int grid_y, const void* tile_map,
                           cudaStream_t st);
// W4A4: the same GEMMs on the block-scaled FP4 MMA (kind::mxf4nvf4), both
// operands NVFP4, the weights read from their MMA layout; tile_map: the
// CUtensorMap of the region's codes made by tc_make_mma_map with
// box_rows = 128 * tc_fp4_group(M-blocks of the matrix).  grid: a CTA per SM.
int tc_fp4_group(int mblocks);
cudaError_t tc_make_mma_map(void* map, const uint8_t* codes, int n_experts, int rows, int stages,
                            uint64_t expert_stride, int box_rows);
cudaError_t launch_tc_fp4_gateup(const ExpertParams& p, int items, const void* tile_map,
                                 const void* bmap_c, const void* bmap_s, cudaStream_t st);
cudaError_t launch_tc_fp4_down(const ExpertParams& p, int items, const void* tile_map,
                               const void* bmap_c, const void* bmap_s, cudaStream_t st);
// the maps of the activation rows the block-scaled GEMMs read (B operands):
// [rows][row_bytes], codes (128-byte boxes, 128B-swizzled) or scales (16-byte boxes)
// W4A16 expert GEMMs with the dequantised weights in tensor memory (H and I
// multiples of 128: tc_tm_ok): code_map made by tc_make_tile_map with
// box_tiles = 8 and box_pieces = 2, scale_map with box_tiles = 8; xmap / amap by
// tc_make_rows16_map over x gathered into slot order (xs, written by
// launch_gather_rows: rows = T*k + T) / the rows of a.  grid: a CTA per SM.
cudaError_t tc_make_rows16_map(void* map, const uint16_t* base, size_t rows, int cols);
cudaError_t launch_gather_rows(const ExpertParams& p, int rows, uint16_t* xs, bool from_f16,
                               cudaStream_t st);
bool tc_tm_ok(int H, int I);
cudaError_t launch_tc_tm_gateup(const ExpertParams& p, int items, const void* code_map,
                                const void* scale_map, const void* xmap, cudaStream_t st);
cudaError_t launch_tc_tm_down(const ExpertParams& p, int items, const void* code_map,
                              const void* scale_map, const void* amap, cudaStream_t st);
cudaError_t tc_make_rows_map(void* map, const uint8_t* base, size_t rows, int row_bytes, bool codes);
bool tc_router_ok(int E, int H);
cudaError_t launch_tc_router(const ExpertParams& p, cudaStream_t st);
cudaError_t tc_kernels_init();

// launch helper: optional programmatic dependent launch on the previous kernel in the stream
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}


}  // namespace moe
