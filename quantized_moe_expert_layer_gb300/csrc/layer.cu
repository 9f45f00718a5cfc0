// The C ABI of include/moe.h: layer lifetime, weight packing, the forward
// pass (router -> top-k / dispatch -> gate/up + SwiGLU -> down -> combine,
// chained with programmatic dependent launch) and the test hooks.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/moe.h"
#include "kernels.cuh"
#include "layout.cuh"

using namespace moe;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(const char* op, cudaError_t e) {
  return fail(MOE_ECUDA, "%s: %s (%s)", op, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define CK(op, call)                                 \
  do {                                               \
    cudaError_t e_ = (call);                         \
    if (e_ != cudaSuccess) return cuda_fail(op, e_); \
  } while (0)

// Makes the layer's device current for the scope of an entry point.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Test hook of moe_debug_fail_alloc: the countdown to the allocation that
// fails (0: none).  Every device or pinned-host allocation the library makes
// goes through alloc_dev / alloc_host.
std::atomic<int> g_fail_alloc{0};

bool injected_failure() {
  int n = g_fail_alloc.load();
  while (n > 0 && !g_fail_alloc.compare_exchange_weak(n, n - 1)) {
  }
  return n == 1;
}

cudaError_t alloc_dev(void** p, size_t bytes) {
  *p = nullptr;
  if (injected_failure()) return cudaErrorMemoryAllocation;
  return cudaMalloc(p, bytes);
}

cudaError_t alloc_host(void** p, size_t bytes, unsigned flags) {
  *p = nullptr;
  if (injected_failure()) return cudaErrorMemoryAllocation;
  return cudaHostAlloc(p, bytes, flags);
}

// Guard regions around the workspace buffers: 256 bytes of this value each.
constexpr unsigned char kCanary = 0xA5;
constexpr size_t kGuard = 256;

// Upper bound on routed entries (ceil(count/8) summed over experts) for T tokens.
int max_routed_entries(int T, int E, int k) {
  const long S = (long)T * k;
  const long m = S < E ? S : E;
  long b = (S + 7 * m) / kTokTile;
  if (b > S) b = S;
  return (int)b;
}

}  // namespace

namespace moe {
// Records the message of a failure for moe_last_error(); used by entry points
// implemented in other translation units.
int record_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}
}  // namespace moe

struct moe_layer {
  int device = 0;
  int fmt = 0, H = 0, I = 0, E = 0, k = 0, shared = 0;
  int dev_fmt = 0;  // layout of the packed tiles (MXFP4 is packed as NVFP4)
  ExpertGeom geom{};
  // TMA tile maps (CUtensorMap) of the gate/up and down regions of the arena,
  // for the tensor-core path; maps_ok false when they could not be made
  alignas(64) unsigned char map_gu[128] = {};
  alignas(64) unsigned char map_dn[128] = {};
  bool maps_ok = false;
  // the same with a box of one M-block (8 tiles), and the maps of the f16
  // token rows in slot order (x gathered into the y buffer, which the down
  // GEMM writes only after gate/up; the rows of a) for the W4A16 GEMMs with
  // the weights in tensor memory
  alignas(64) unsigned char map_gu8[128] = {};   // code boxes: 2 pieces of 8 tiles
  alignas(64) unsigned char map_dn8[128] = {};
  alignas(64) unsigned char map_gu8s[128] = {};  // scale boxes: 1 piece of 8 tiles
  alignas(64) unsigned char map_dn8s[128] = {};
  alignas(64) unsigned char map_xs[128] = {};
  alignas(64) unsigned char map_ab[128] = {};
  bool tm_maps_ok = false;
  bool rows_maps_ok = false;
  // W4A4 on the tensor-core path: the packed tiles again in the MMA layout
  // (layout.cuh), rebuilt from the arena before the first forward after any
  // change to it, and the TMA maps of its code regions
  uint8_t* mma = nullptr;
  uint64_t mma_expert_bytes = 0;
  bool mma_dirty = true;
  alignas(64) unsigned char map_gu_mma[128] = {};
  alignas(64) unsigned char map_dn_mma[128] = {};
  bool mma_maps_ok = false;
  // ... and their B operands: x quantised into its expert-sorted rows (xg) and
  // the rows of a (aqb), codes then scales, each row padded (act_pitches),
  // with the TMA maps of their codes and scales
  uint8_t* xg = nullptr;
  uint8_t* aqb = nullptr;
  alignas(64) unsigned char map_bx_c[128] = {};
  alignas(64) unsigned char map_bx_s[128] = {};
  alignas(64) unsigned char map_ba_c[128] = {};
  alignas(64) unsigned char map_ba_s[128] = {};
  bool bmaps_ok = false;
  uint8_t* arena = nullptr;      // HBM: every expert in order, or the HBM slots of a split placement
  uint64_t arena_bytes = 0;
  // Split placement (moe_place_experts): experts without an HBM slot live in a
  // pinned, device-mapped host mirror and the kernels read them there through
  // the per-expert table.  eptr is null while every expert sits in the arena
  // in expert order.
  uint8_t* mirror = nullptr;
  uint64_t mirror_bytes = 0;
  const uint8_t** eptr = nullptr;           // device [E + shared]
  std::vector<const uint8_t*> eptr_host;    // the same table, host copy
  std::vector<uint8_t> in_hbm;              // [E + shared] 1: HBM slot, 0: host mirror
  float* tscale = nullptr;
  uint16_t* router = nullptr;
  float* bias = nullptr;
  bool has_bias = false;
  bool router_set = false;
  int router_mode = ROUTER_SOFTMAX;
  int* status = nullptr;
  long long wait_budget = 0;     // bounded-wait budget of the tensor-core kernels (0: default)
  int act_fmt = MOE_ACT_BF16;    // MOE_ACT_NVFP4: W4A4, activations quantised per row
  // workspace
  int T_max = 0;
  void* ws = nullptr;
  float* partial = nullptr;
  float* logits = nullptr;
  int* idx = nullptr;
  float* gates = nullptr;
  int* counts = nullptr;
  int* offsets = nullptr;
  int* perm = nullptr;
  int* inv = nullptr;
  int* row_token = nullptr;
  int4* entries = nullptr;
  int* n_entries = nullptr;
  int4* tc_entries = nullptr;    // entries of up to 256 tokens (tensor-core path)
  int* n_tc_entries = nullptr;
  int* blk = nullptr;            // per-chunk expert counts of the several-CTA dispatch
  uint16_t* xh = nullptr;        // f16 copy of x
  uint16_t* abuf = nullptr;
  float* ybuf = nullptr;
  uint16_t* x_stage = nullptr;
  float* out_stage = nullptr;
  float* ts_x = nullptr;         // W4A4: per-token activation tensor scales
  float* ts_a = nullptr;         // W4A4: per-row tensor scales of a
  int* ticket = nullptr;         // the fused top-k + dispatch's CTA count (0 between forwards)
  std::vector<size_t> guards;    // byte offsets of the workspace's guard regions
  size_t ws_bytes = 0;
  int last_T = 0;
  bool last_has_logits = false;
  bool x_mapped = false;         // this forward's x is pinned host memory read in place
};

namespace {

// The TMA tile maps of the tensor-core path view the arena as
// [expert][tile][piece]: only while every expert sits there in expert order.
void make_mma_maps(moe_layer* L);

void make_tile_maps(moe_layer* L) {
  L->maps_ok = false;
  L->mma_dirty = true;
  if (L->eptr || L->dev_fmt != FMT_NVFP4 || L->H % 128 || (2 * L->I) % 128) return;
  const ExpertGeom& g = L->geom;
  const int n_total = L->E + L->shared, gu_tiles = 2 * L->I / 16, dn_tiles = L->H / 16;
  L->maps_ok =
      tc_make_tile_map(L->map_gu, L->arena, n_total, gu_tiles, g.gu.tile_bytes, g.expert_bytes,
                       8 * tc_group(gu_tiles / 8)) == cudaSuccess &&
      tc_make_tile_map(L->map_dn, L->arena + g.gu_bytes, n_total, dn_tiles, g.dn.tile_bytes,
                       g.expert_bytes, 8 * tc_group(dn_tiles / 8)) == cudaSuccess;
  L->tm_maps_ok =
      L->maps_ok && tc_tm_ok(L->H, L->I) &&
      tc_make_tile_map(L->map_gu8, L->arena, n_total, gu_tiles, g.gu.tile_bytes, g.expert_bytes, 8, 2) ==
          cudaSuccess &&
      tc_make_tile_map(L->map_dn8, L->arena + g.gu_bytes, n_total, dn_tiles, g.dn.tile_bytes,
                       g.expert_bytes, 8, 2) == cudaSuccess &&
      tc_make_tile_map(L->map_gu8s, L->arena, n_total, gu_tiles, g.gu.tile_bytes, g.expert_bytes, 8, 1) ==
          cudaSuccess &&
      tc_make_tile_map(L->map_dn8s, L->arena + g.gu_bytes, n_total, dn_tiles, g.dn.tile_bytes,
                       g.expert_bytes, 8, 1) == cudaSuccess;
  make_mma_maps(L);
}

// the MMA layout's regions within an expert: gate/up codes, scales, down codes, scales
void mma_geoms(const moe_layer* L, MmaGeom& gu, MmaGeom& dn) {
  gu = mma_geom(2 * L->I, L->H);
  dn = mma_geom(L->H, L->I);
}

void make_mma_maps(moe_layer* L) {
  L->mma_maps_ok = false;
  if (!L->mma || !L->maps_ok) return;
  MmaGeom gu, dn;
  mma_geoms(L, gu, dn);
  const int n_total = L->E + L->shared;
  L->mma_maps_ok =
      tc_make_mma_map(L->map_gu_mma, L->mma, n_total, gu.M, gu.KS, L->mma_expert_bytes,
                      128 * tc_fp4_group(gu.M / 128)) == cudaSuccess &&
      tc_make_mma_map(L->map_dn_mma, L->mma + gu.codes + gu.scales, n_total, dn.M, dn.KS,
                      L->mma_expert_bytes, 128 * tc_fp4_group(dn.M / 128)) == cudaSuccess;
}

// rows of the block-scaled GEMMs' B operands: codes padded to 128-byte
// multiples (one TMA box of a stage), scales to 16-byte multiples
int act_cpitch(int K) { return (K / 2 + 127) / 128 * 128; }
int act_spitch(int K) { return (K / 16 + 15) / 16 * 16; }
size_t act_rows_cap(const moe_layer* L) { return (size_t)L->T_max * L->k + (L->shared ? L->T_max : 0); }

uint16_t* xs_rows(const moe_layer* L) { return reinterpret_cast<uint16_t*>(L->ybuf); }

void make_rows_maps(moe_layer* L) {
  L->rows_maps_ok = L->ybuf && L->abuf &&
                    tc_make_rows16_map(L->map_xs, xs_rows(L), act_rows_cap(L), L->H) == cudaSuccess &&
                    tc_make_rows16_map(L->map_ab, L->abuf, act_rows_cap(L), L->I) == cudaSuccess;
}

void make_b_maps(moe_layer* L) {
  L->bmaps_ok = false;
  if (!L->xg || !L->aqb) return;
  const size_t rows = act_rows_cap(L);
  const int cH = act_cpitch(L->H), sH = act_spitch(L->H), cI = act_cpitch(L->I), sI = act_spitch(L->I);
  L->bmaps_ok =
      tc_make_rows_map(L->map_bx_c, L->xg, rows, cH, true) == cudaSuccess &&
      tc_make_rows_map(L->map_bx_s, L->xg + rows * cH, rows, sH, false) == cudaSuccess &&
      tc_make_rows_map(L->map_ba_c, L->aqb, rows, cI, true) == cudaSuccess &&
      tc_make_rows_map(L->map_ba_s, L->aqb + rows * cI, rows, sI, false) == cudaSuccess;
}

// the MMA layout from the arena (every expert in it, in order), when the arena changed
int refresh_mma(moe_layer* L, cudaStream_t st) {
  if (!L->mma_dirty) return MOE_OK;
  MmaGeom gu, dn;
  mma_geoms(L, gu, dn);
  const ExpertGeom& g = L->geom;
  const int n_total = L->E + L->shared;
  CK("MMA-layout conversion (gate/up)",
     launch_to_mma_layout(L->arena, g.expert_bytes, 0, g.gu.tile_bytes, gu.M, gu.K, n_total, L->mma,
                          L->mma_expert_bytes, 0, gu.codes, st));
  CK("MMA-layout conversion (down)",
     launch_to_mma_layout(L->arena, g.expert_bytes, g.gu_bytes, g.dn.tile_bytes, dn.M, dn.K, n_total,
                          L->mma, L->mma_expert_bytes, gu.codes + gu.scales,
                          gu.codes + gu.scales + dn.codes, st));
  L->mma_dirty = false;
  return MOE_OK;
}

// Device address of expert e's packed matrices, wherever they are placed.
const uint8_t* expert_ptr(const moe_layer* L, int e) {
  return L->eptr ? L->eptr_host[e] : L->arena + (size_t)e * L->geom.expert_bytes;
}

RouteParams route_params(moe_layer* L, const uint16_t* x, int T) {
  RouteParams p{};
  p.mode = L->router_mode;
  p.x = x;
  p.wr = L->router;
  p.bias = L->has_bias ? L->bias : nullptr;
  p.T = T;
  p.H = L->H;
  p.E = L->E;
  p.k = L->k;
  p.shared = L->shared;
  const bool tc = L->maps_ok && tc_path_ok(L->dev_fmt, T, L->k, L->E, L->H, L->I);
  // the tensor-core router writes the whole dot product: one K slice
  p.ksplit = tc && tc_router_ok(L->E, L->H) ? 1 : router_ksplit(T, L->H, L->E);
  p.partial = L->partial;
  p.logits = L->logits;
  p.idx = L->idx;
  p.gates = L->gates;
  p.counts = L->counts;
  p.offsets = L->offsets;
  p.perm = L->perm;
  p.inv = L->inv;
  p.row_token = L->row_token;
  p.entries = L->entries;
  p.n_entries = L->n_entries;
  p.xh = L->act_fmt == MOE_ACT_NVFP4 ? nullptr : L->xh;  // W4A4: the quantiser writes it
  p.tc_entries = tc ? L->tc_entries : nullptr;
  p.n_tc_entries = tc ? L->n_tc_entries : nullptr;
  p.blk = L->blk;
  p.ticket = L->ticket;
  p.status = L->status;
  return p;
}

ExpertParams expert_params(moe_layer* L, const uint16_t* x, int T) {
  ExpertParams p{};
  p.arena = L->arena;
  p.eptr = L->eptr;
  p.expert_bytes = L->geom.expert_bytes;
  p.gu_bytes = L->geom.gu_bytes;
  p.gu_tile_bytes = L->geom.gu.tile_bytes;
  p.dn_tile_bytes = L->geom.dn.tile_bytes;
  p.tscale = L->tscale;
  p.fmt = L->dev_fmt;
  p.H = L->H;
  p.I = L->I;
  p.E = L->E;
  p.T = T;
  p.k = L->k;
  p.shared = L->shared;
  p.nsh = L->shared ? (T + kTokTile - 1) / kTokTile : 0;
  p.nsh_tc = L->shared ? (T + kTcMaxN - 1) / kTcMaxN : 0;
  p.tc_entries = L->tc_entries;
  p.n_tc_entries = L->n_tc_entries;
  p.xh = L->xh;
  p.entries = L->entries;
  p.n_entries = L->n_entries;
  p.row_token = L->row_token;
  p.x = x;
  p.abuf = L->abuf;
  p.ybuf = L->ybuf;
  p.wr = L->router;
  p.rbias = L->has_bias ? L->bias : nullptr;
  p.status = L->status;
  p.wait_budget = L->wait_budget > 0 ? L->wait_budget : 2000000000LL;
  if (L->act_fmt == MOE_ACT_NVFP4) {
    p.ts_x = L->ts_x;
    p.ts_a = L->ts_a;
    p.af = L->ybuf;  // a in fp32 until quantised; the down kernels write y after that
    if (L->mma) {
      MmaGeom gu, dn;
      mma_geoms(L, gu, dn);
      p.mma = L->mma;
      p.mma_expert_bytes = L->mma_expert_bytes;
      p.mma_gu_sc = gu.codes;
      p.mma_dn_sc = gu.codes + gu.scales + dn.codes;
    }
  }
  return p;
}

int check_forward_args(moe_layer* L, const void* x, int T, const void* out) {
  if (!L) return fail(MOE_EINVAL, "moe_forward: null layer");
  if (!x || !out) return fail(MOE_EINVAL, "moe_forward: null x or out");
  if (((uintptr_t)x | (uintptr_t)out) & 15u)
    return fail(MOE_EINVAL, "moe_forward: x and out must be 16-byte aligned");
  if (T < 1) return fail(MOE_EINVAL, "moe_forward: T = %d < 1", T);
  if (!L->ws || T > L->T_max)
    return fail(MOE_ESTATE, "moe_forward: T = %d exceeds the reserved T_max = %d", T, L->T_max);
  if (!L->router_set) return fail(MOE_ESTATE, "moe_forward: router weights not set");
  const long grid_y = (L->shared ? (T + kTokTile - 1) / kTokTile : 0) +
                      max_routed_entries(T, L->E, L->k);
  if (grid_y > 65535)
    return fail(MOE_EINVAL, "moe_forward: T = %d needs %ld expert work entries (> 65535)", T, grid_y);
  return MOE_OK;
}

// experts + combine, after routing has filled idx / gates / dispatch
// Top-k inside the one-CTA dispatch kernel up to this many tokens (one warp
// each, no extra launch); more tokens take the top-k kernel (8 tokens per CTA)
constexpr int kFusedTopkMaxT = 16;

bool fused_down(moe_layer* L, int T) { return down_combine_ok(T, L->k, L->shared, L->I); }

bool tc_path(moe_layer* L, int T) {
  return L->maps_ok && tc_path_ok(L->dev_fmt, T, L->k, L->E, L->H, L->I);
}

// prefill routing: logits as one bf16 GEMM on the tensor cores, then top-k and
// dispatch as usual (the GEMM's output is the one K slice the top-k reads)
bool tc_router(moe_layer* L, int T) { return tc_path(L, T) && tc_router_ok(L->E, L->H); }

bool w4a4(const moe_layer* L) { return L->act_fmt == MOE_ACT_NVFP4; }

// W4A4 on the tensor-core path: the expert GEMMs on the block-scaled FP4 MMA
bool fq_path(moe_layer* L, int T) {
  return w4a4(L) && tc_path(L, T) && L->mma_maps_ok && L->bmaps_ok;
}

// the tensor-core path's f16 GEMMs with the weights in tensor memory (W4A16:
// W4A4 keeps a in fp32 in the y buffer, where these read x's rows)
bool tm_path(moe_layer* L, int T) {
  return !w4a4(L) && tc_path(L, T) && L->tm_maps_ok && L->rows_maps_ok;
}

// x's rows in slot order (the gate/up GEMM's token rows), after the dispatch
int launch_row_gather(moe_layer* L, const ExpertParams& ep, int T, cudaStream_t st) {
  CK("row gather kernel launch",
     launch_gather_rows(ep, T * L->k + (L->shared ? T : 0), xs_rows(L), L->x_mapped, st));
  return MOE_OK;
}

int launch_tm_gateup(moe_layer* L, const ExpertParams& ep, int T, cudaStream_t st) {
  const int gy = ep.nsh_tc + max_tc_entries(T, L->E, L->k);
  CK("tensor-core gate/up kernel launch",
     launch_tc_tm_gateup(ep, gy, L->map_gu8, L->map_gu8s, L->map_xs, st));
  return MOE_OK;
}

// top-k then dispatch: one fused launch where it applies, else two (or three)
int launch_topk_and_dispatch(moe_layer* L, const RouteParams& rp, int T, bool pdl, cudaStream_t st) {
  if (topk_dispatch_ok(T, L->k, L->E)) {
    CK("top-k + dispatch kernel launch", launch_topk_dispatch(rp, pdl, st));
    return MOE_OK;
  }
  CK("top-k kernel launch", launch_topk(rp, pdl, st));
  CK("dispatch kernel launch", launch_dispatch(rp, pdl, st));
  return MOE_OK;
}

// W4A4: x quantised per token, with the per-token tensor scales, into the
// f16 copy the expert kernels read (e2m1 code x e4m3 block scale), or, for the
// block-scaled FP4 GEMMs, into codes and block scales in the same space
int launch_quant_x(moe_layer* L, const uint16_t* x, int T, cudaStream_t st) {
  CK("activation quantiser launch (x)", launch_quantize_act(x, true, T, L->H, nullptr, nullptr, L->xh,
                                                             L->ts_x, L->status, true, st));
  return MOE_OK;
}

// W4A4 on the block-scaled GEMMs: x quantised per token into each of its
// expert-sorted rows of xg (after the dispatch: the rows come from inv)
int launch_quant_x_rows(moe_layer* L, const uint16_t* x, int T, cudaStream_t st) {
  const size_t rows = act_rows_cap(L);
  const int c = act_cpitch(L->H), sc = act_spitch(L->H);
  CK("activation quantiser launch (x rows)",
     launch_quantize_act(x, true, T, L->H, L->xg, L->xg + rows * c, nullptr, L->ts_x, L->status,
                         true, st, c, sc, L->inv, L->k, L->shared ? T * L->k : -1));
  return MOE_OK;
}

// W4A4: the rows of a (fp32, written by gate/up) quantised into abuf (f16
// values, or codes and block scales for the FP4 GEMMs) and ts_a
int launch_quant_a(moe_layer* L, int T, cudaStream_t st) {
  const int rows = T * L->k + (L->shared ? T : 0);
  if (fq_path(L, T)) {
    const size_t cap = act_rows_cap(L);
    const int c = act_cpitch(L->I), sc = act_spitch(L->I);
    CK("activation quantiser launch (a rows)",
       launch_quantize_act(L->ybuf, false, rows, L->I, L->aqb, L->aqb + cap * c, nullptr, L->ts_a,
                           L->status, true, st, c, sc));
    return MOE_OK;
  }
  CK("activation quantiser launch (a)", launch_quantize_act(L->ybuf, false, rows, L->I, nullptr,
                                                             nullptr, L->abuf, L->ts_a, L->status,
                                                             true, st));
  return MOE_OK;
}

int launch_tc_routing_gemm(moe_layer* L, const uint16_t* x, int T, cudaStream_t st) {
  ExpertParams ep = expert_params(L, x, T);
  ep.logits_out = L->partial;
  // (W4A4: the quantiser wrote the f16 copy before the router; the GEMMs with
  // the weights in tensor memory convert x while gathering its rows)
  // (x in mapped host memory: converted once here, and the gather copies the
  // f16 rows instead of reading x over the link once per row)
  if (!w4a4(L) && (!tm_path(L, T) || L->x_mapped))
    CK("x conversion kernel launch", launch_convert_x(x, L->xh, (long)T * L->H, L->status, st));
  CK("tensor-core router kernel launch", launch_tc_router(ep, st));
  return MOE_OK;
}

int run_experts(moe_layer* L, const uint16_t* x, int T, float* out, cudaStream_t st) {
  ExpertParams ep = expert_params(L, x, T);
  if (fq_path(L, T)) {
    const int gy = ep.nsh_tc + max_tc_entries(T, L->E, L->k);
    if (refresh_mma(L, st)) return MOE_ECUDA;
    if (launch_quant_x_rows(L, x, T, st)) return MOE_ECUDA;
    CK("FP4 tensor-core gate/up kernel launch",
       launch_tc_fp4_gateup(ep, gy, L->map_gu_mma, L->map_bx_c, L->map_bx_s, st));
    if (launch_quant_a(L, T, st)) return MOE_ECUDA;
    CK("FP4 tensor-core down kernel launch",
       launch_tc_fp4_down(ep, gy, L->map_dn_mma, L->map_ba_c, L->map_ba_s, st));
    CK("combine kernel launch", launch_combine(ep, L->gates, L->inv, out, true, st));
    return MOE_OK;
  }
  if (tc_path(L, T)) {
    const int gy = ep.nsh_tc + max_tc_entries(T, L->E, L->k);
    if (tm_path(L, T)) {
      int rc = launch_row_gather(L, ep, T, st);
      if (!rc) rc = launch_tm_gateup(L, ep, T, st);
      if (rc) return rc;
    } else {
      CK("tensor-core gate/up kernel launch", launch_tc_gateup(ep, gy, L->map_gu, st));
    }
    if (w4a4(L) && launch_quant_a(L, T, st)) return MOE_ECUDA;
    if (tm_path(L, T))
      CK("tensor-core down kernel launch",
         launch_tc_tm_down(ep, gy, L->map_dn8, L->map_dn8s, L->map_ab, st));
    else
      CK("tensor-core down kernel launch", launch_tc_down(ep, gy, L->map_dn, st));
    CK("combine kernel launch", launch_combine(ep, L->gates, L->inv, out, true, st));
    return MOE_OK;
  }
  const int grid_y = ep.nsh + max_routed_entries(T, L->E, L->k);
  CK("gate/up kernel launch", launch_gateup(ep, grid_y, true, st));
  if (w4a4(L) && launch_quant_a(L, T, st)) return MOE_ECUDA;
  if (fused_down(L, T)) {
    CK("down+combine kernel launch", launch_down_combine(ep, L->gates, L->inv, out, true, false, st));
    return MOE_OK;
  }
  CK("down kernel launch", launch_down(ep, grid_y, true, st));
  CK("combine kernel launch", launch_combine(ep, L->gates, L->inv, out, true, st));
  return MOE_OK;
}

// T <= 8: router partial sums; gate/up, which routes itself from them and
// publishes the routing; down + combine (three launches, chained)
bool small_path(moe_layer* L, int T) { return small_route_ok(T, L->k) && fused_down(L, T); }

// kernels one forward of T tokens launches
int forward_launches(moe_layer* L, int T) {
  // W4A4: the quantiser of a, and of x (in place of the x conversion before the tensor-core router)
  const int q = w4a4(L) ? 1 + (tc_router(L, T) ? 0 : 1) : 0;
  if (small_path(L, T)) return 3 + q;
  // (convert x, tc router | router), top-k, dispatch (1 or 2 kernels); T <= 16: router, top-k + dispatch
  const int dispatch = dispatch_launches(T * L->k);
  // top-k + dispatch: one kernel (T <= 16, or the fused one), else top-k then dispatch
  const int topk_disp = topk_dispatch_ok(T, L->k, L->E) ? 1 : 1 + dispatch;
  const int routing = tc_router(L, T) ? 2 + topk_disp : (T <= kFusedTopkMaxT ? 2 : 1 + topk_disp);
  // (the GEMMs with the weights in tensor memory: + the row gather, which
  // replaces the x conversion before the tensor-core router)
  if (tc_path(L, T)) return routing + 3 + q + (tm_path(L, T) && !tc_router(L, T) ? 1 : 0);
  return routing + (fused_down(L, T) ? 2 : 3) + q;
}

int forward_impl(moe_layer* L, const uint16_t* x, int T, float* out, cudaStream_t st) {
  RouteParams rp = route_params(L, x, T);
  L->last_T = T;
  L->last_has_logits = true;
  if (w4a4(L) && !fq_path(L, T)) {  // (the block-scaled path quantises x after the dispatch)
    const int rc = launch_quant_x(L, x, T, st);
    if (rc) return rc;
  }
  if (small_path(L, T)) {
    ExpertParams ep = expert_params(L, x, T);
    CK("router kernel launch", launch_router(rp, st));
    CK("gate/up kernel launch",
       launch_gateup_routed(ep, rp, ep.nsh + max_routed_entries(T, L->E, L->k), st));
    if (w4a4(L) && launch_quant_a(L, T, st)) return MOE_ECUDA;
    CK("down+combine kernel launch", launch_down_combine(ep, L->gates, L->inv, out, true, true, st));
    return MOE_OK;
  }
  if (tc_router(L, T)) {
    const int rc = launch_tc_routing_gemm(L, x, T, st);
    if (rc) return rc;
    const int rc2 = launch_topk_and_dispatch(L, rp, T, true, st);
    if (rc2) return rc2;
  } else if (T <= kFusedTopkMaxT) {
    CK("router kernel launch", launch_router(rp, st));
    CK("top-k/dispatch kernel launch", launch_route_finish(rp, true, true, st));
  } else {
    CK("router kernel launch", launch_router(rp, st));
    const int rc2 = launch_topk_and_dispatch(L, rp, T, true, st);
    if (rc2) return rc2;
  }
  L->last_T = T;
  L->last_has_logits = true;
  return run_experts(L, x, T, out, st);
}

}  // namespace

extern "C" {

const char* moe_last_error(void) { return g_last_error.c_str(); }

int moe_layer_create(int format, int H, int I, int E, int k, int shared, moe_layer** out) {
  if (!out) return fail(MOE_EINVAL, "moe_layer_create: null out");
  *out = nullptr;
  if (format != MOE_FMT_NVFP4 && format != MOE_FMT_FP6_E2M3 && format != MOE_FMT_MXFP4)
    return fail(MOE_EINVAL, "moe_layer_create: unknown format %d", format);
  const int mult = format == MOE_FMT_FP6_E2M3 ? 128 : 64;
  const int dev_fmt = format == MOE_FMT_FP6_E2M3 ? FMT_FP6 : FMT_NVFP4;
  if (H <= 0 || I <= 0 || H % mult || I % mult)
    return fail(MOE_EINVAL, "moe_layer_create: H=%d and I=%d must be positive multiples of %d", H,
                I, mult);
  if (H > 65536 || I > 65536)
    return fail(MOE_EINVAL, "moe_layer_create: H=%d and I=%d must be at most 65536", H, I);
  if (E < 1 || E > kMaxE) return fail(MOE_EINVAL, "moe_layer_create: E=%d not in [1, %d]", E, kMaxE);
  if (k < 1 || k > E || k > kMaxK)
    return fail(MOE_EINVAL, "moe_layer_create: k=%d not in [1, min(E, %d)]", k, kMaxK);
  if (shared != 0 && shared != 1) return fail(MOE_EINVAL, "moe_layer_create: shared must be 0 or 1");
  moe_layer* L = new moe_layer();
  L->fmt = format;
  L->dev_fmt = dev_fmt;
  L->H = H;
  L->I = I;
  L->E = E;
  L->k = k;
  L->shared = shared;
  L->geom = expert_geom(dev_fmt, H, I);
  L->in_hbm.assign(E + shared, 1);
  cudaError_t e = cudaGetDevice(&L->device);
  if (e == cudaSuccess) e = route_kernels_init();
  if (e == cudaSuccess) e = expert_kernels_init();
  if (e == cudaSuccess) e = tc_kernels_init();
  if (e != cudaSuccess) {
    delete L;
    return cuda_fail("moe_layer_create: device set-up", e);
  }
  const int n_total = E + shared;
  L->arena_bytes = (uint64_t)n_total * L->geom.expert_bytes;
  if (alloc_dev((void**)&L->arena, L->arena_bytes) != cudaSuccess ||
      alloc_dev((void**)&L->tscale, sizeof(float) * 3 * n_total) != cudaSuccess ||
      alloc_dev((void**)&L->router, sizeof(uint16_t) * (size_t)E * H) != cudaSuccess ||
      alloc_dev((void**)&L->bias, sizeof(float) * E) != cudaSuccess ||
      alloc_dev((void**)&L->status, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    const double mb = (double)L->arena_bytes / 1e6;
    moe_layer_destroy(L);
    return fail(MOE_ENOMEM, "moe_layer_create: device allocation failed (arena %.1f MB)", mb);
  }
  if (cudaMemset(L->arena, 0, L->arena_bytes) != cudaSuccess ||
      cudaMemset(L->tscale, 0, sizeof(float) * 3 * n_total) != cudaSuccess ||
      cudaMemset(L->status, 0, sizeof(int)) != cudaSuccess) {
    moe_layer_destroy(L);
    return fail(MOE_ECUDA, "moe_layer_create: cudaMemset failed");
  }
  make_tile_maps(L);
  *out = L;
  return MOE_OK;
}

int moe_layer_reserve(moe_layer* L, int T_max) {
  if (!L) return fail(MOE_EINVAL, "moe_layer_reserve: null layer");
  if (T_max < 1) return fail(MOE_EINVAL, "moe_layer_reserve: T_max = %d < 1", T_max);
  if (T_max <= L->T_max) return MOE_OK;
  DeviceGuard dg(L->device);
  const size_t S = (size_t)T_max * L->k, E = L->E;
  size_t partial = 0;
  for (int T = 1; T <= T_max; ++T) {
    size_t v = (size_t)router_ksplit(T, L->H, L->E) * T * E;
    if (v > partial) partial = v;
  }
  const size_t n_entries = (size_t)max_routed_entries(T_max, L->E, L->k);
  const size_t sizes[] = {
      partial * 4,                       // partial
      (size_t)T_max * E * 4,             // logits
      S * 4, S * 4,                      // idx, gates
      E * 4, (E + 1) * 4,                // counts, offsets
      S * 4, S * 4,                      // perm, inv
      (S + T_max) * 4,                   // row_token
      n_entries * 16, 16,                // entries, n_entries
      (size_t)max_tc_entries(T_max, L->E, L->k) * 16, 16,  // tc_entries, n_tc_entries
      (size_t)T_max * L->H * 2,          // xh
      (S + T_max) * L->I * 2,            // abuf
      (S + T_max) * (size_t)(L->H > L->I ? L->H : L->I) * 4,  // ybuf (W4A4: fp32 a first)
      (size_t)T_max * L->H * 2,          // x_stage
      (size_t)T_max * L->H * 4,          // out_stage
      ((S + kDispChunk - 1) / kDispChunk) * E * 4,  // blk
      (size_t)T_max * 4,                 // ts_x
      (S + T_max) * 4,                   // ts_a
      4,                                 // ticket
      // W4A4 block-scaled GEMMs: x's and a's NVFP4 rows (codes, then scales)
      (S + (L->shared ? T_max : 0)) * (size_t)(act_cpitch(L->H) + act_spitch(L->H)),  // xg
      (S + (L->shared ? T_max : 0)) * (size_t)(act_cpitch(L->I) + act_spitch(L->I)),  // aqb
  };
  const int n = (int)(sizeof(sizes) / sizeof(sizes[0]));
  // [guard][buffer 0][guard][buffer 1] ... [guard]: moe_debug_check_workspace
  // finds a kernel that wrote past the end of its buffer
  size_t total = kGuard;
  for (int i = 0; i < n; ++i) total += align_up(sizes[i], 256) + kGuard;
  void* ws = nullptr;
  if (alloc_dev(&ws, total) != cudaSuccess) {
    cudaGetLastError();
    return fail(MOE_ENOMEM, "moe_layer_reserve: device allocation of %.1f MB failed", total / 1e6);
  }
  if (L->ws) {
    cudaDeviceSynchronize();
    cudaFree(L->ws);
  }
  L->ws = ws;
  L->ws_bytes = total;
  L->guards.clear();
  char* p = static_cast<char*>(ws);
  void* ptrs[24];
  for (int i = 0; i < n; ++i) {
    L->guards.push_back((size_t)(p - static_cast<char*>(ws)));
    p += kGuard;
    ptrs[i] = p;
    p += align_up(sizes[i], 256);
  }
  L->guards.push_back((size_t)(p - static_cast<char*>(ws)));
  L->partial = (float*)ptrs[0];
  L->logits = (float*)ptrs[1];
  L->idx = (int*)ptrs[2];
  L->gates = (float*)ptrs[3];
  L->counts = (int*)ptrs[4];
  L->offsets = (int*)ptrs[5];
  L->perm = (int*)ptrs[6];
  L->inv = (int*)ptrs[7];
  L->row_token = (int*)ptrs[8];
  L->entries = (int4*)ptrs[9];
  L->n_entries = (int*)ptrs[10];
  L->tc_entries = (int4*)ptrs[11];
  L->n_tc_entries = (int*)ptrs[12];
  L->xh = (uint16_t*)ptrs[13];
  L->abuf = (uint16_t*)ptrs[14];
  L->ybuf = (float*)ptrs[15];
  L->x_stage = (uint16_t*)ptrs[16];
  L->out_stage = (float*)ptrs[17];
  L->blk = (int*)ptrs[18];
  L->ts_x = (float*)ptrs[19];
  L->ts_a = (float*)ptrs[20];
  L->ticket = (int*)ptrs[21];
  L->xg = (uint8_t*)ptrs[22];
  L->aqb = (uint8_t*)ptrs[23];
  L->T_max = T_max;
  make_b_maps(L);
  make_rows_maps(L);
  CK("moe_layer_reserve: clear workspace", cudaMemset(ws, 0, total));
  for (size_t off : L->guards)
    CK("moe_layer_reserve: guard regions", cudaMemset(static_cast<char*>(ws) + off, kCanary, kGuard));
  return MOE_OK;
}

void moe_layer_destroy(moe_layer* L) {
  if (!L) return;
  DeviceGuard dg(L->device);
  cudaDeviceSynchronize();
  cudaFree(L->arena);
  cudaFreeHost(L->mirror);
  cudaFree(L->eptr);
  cudaFree(L->mma);
  cudaFree(L->tscale);
  cudaFree(L->router);
  cudaFree(L->bias);
  cudaFree(L->status);
  cudaFree(L->ws);
  delete L;
}

int moe_layer_status(moe_layer* L, int reset, int* status) {
  if (!L || !status) return fail(MOE_EINVAL, "moe_layer_status: null argument");
  DeviceGuard dg(L->device);
  CK("moe_layer_status: synchronize", cudaDeviceSynchronize());
  CK("moe_layer_status: read", cudaMemcpy(status, L->status, sizeof(int), cudaMemcpyDeviceToHost));
  if (reset) CK("moe_layer_status: reset", cudaMemset(L->status, 0, sizeof(int)));
  return MOE_OK;
}

int moe_forward_launches(moe_layer* L, int T) {
  if (!L || T < 1) return fail(MOE_EINVAL, "moe_forward_launches: bad argument");
  return forward_launches(L, T);
}

int moe_forward_path(moe_layer* L, int T) {
  if (!L || T < 1) return fail(MOE_EINVAL, "moe_forward_path: bad argument");
  if (small_path(L, T)) return MOE_PATH_DECODE;
  if (fq_path(L, T)) return MOE_PATH_TC_FP4;
  if (tc_path(L, T)) return MOE_PATH_TC_F16;
  return MOE_PATH_STREAM;
}

int moe_place_experts(moe_layer* L, const uint8_t* in_hbm) {
  if (!L || !in_hbm) return fail(MOE_EINVAL, "moe_place_experts: null argument");
  DeviceGuard dg(L->device);
  const int n_total = L->E + L->shared;
  const uint64_t eb = L->geom.expert_bytes;
  int n_hbm = 0;
  for (int e = 0; e < n_total; ++e) n_hbm += in_hbm[e] != 0;
  const int n_host = n_total - n_hbm;
  CK("moe_place_experts: synchronize", cudaDeviceSynchronize());
  uint8_t* arena = nullptr;
  uint8_t* mirror = nullptr;
  uint8_t* mirror_dev = nullptr;
  const uint8_t** eptr = nullptr;
  cudaError_t err = cudaSuccess;
  if (n_hbm) err = alloc_dev((void**)&arena, (size_t)n_hbm * eb);
  if (err == cudaSuccess && n_host)
    err = alloc_host((void**)&mirror, (size_t)n_host * eb, cudaHostAllocMapped | cudaHostAllocPortable);
  if (err == cudaSuccess && n_host) err = cudaHostGetDevicePointer(&mirror_dev, mirror, 0);
  if (err == cudaSuccess && n_host) err = alloc_dev((void**)&eptr, sizeof(uint8_t*) * n_total);
  if (err != cudaSuccess) {
    cudaGetLastError();
    cudaFree(arena);
    cudaFreeHost(mirror);
    cudaFree(eptr);
    return fail(MOE_ENOMEM, "moe_place_experts: %d HBM slots + %d host experts of %.1f MB: %s",
                n_hbm, n_host, eb / 1e6, cudaGetErrorName(err));
  }
  // HBM slots in expert order, then the mirror in expert order
  std::vector<const uint8_t*> table(n_total);
  for (int e = 0, ih = 0, im = 0; e < n_total; ++e)
    table[e] = in_hbm[e] ? arena + (size_t)(ih++) * eb : mirror_dev + (size_t)(im++) * eb;
  for (int e = 0; e < n_total && err == cudaSuccess; ++e)
    err = cudaMemcpy(const_cast<uint8_t*>(table[e]), expert_ptr(L, e), eb, cudaMemcpyDefault);
  if (err == cudaSuccess && n_host)
    err = cudaMemcpy(eptr, table.data(), sizeof(uint8_t*) * n_total, cudaMemcpyHostToDevice);
  if (err != cudaSuccess) {
    cudaFree(arena);
    cudaFreeHost(mirror);
    cudaFree(eptr);
    return cuda_fail("moe_place_experts: move the experts", err);
  }
  cudaFree(L->arena);
  cudaFreeHost(L->mirror);
  cudaFree(L->eptr);
  L->arena = arena;
  L->arena_bytes = (uint64_t)n_hbm * eb;
  L->mirror = mirror;
  L->mirror_bytes = (uint64_t)n_host * eb;
  L->eptr = eptr;
  if (n_host)
    L->eptr_host = table;
  else
    L->eptr_host.clear();
  for (int e = 0; e < n_total; ++e) L->in_hbm[e] = in_hbm[e] != 0;
  make_tile_maps(L);
  return MOE_OK;
}

int moe_layer_placement(moe_layer* L, uint8_t* in_hbm, uint64_t* hbm_bytes, uint64_t* host_bytes) {
  if (!L) return fail(MOE_EINVAL, "moe_layer_placement: null layer");
  if (in_hbm)
    for (int e = 0; e < L->E + L->shared; ++e) in_hbm[e] = L->in_hbm[e];
  if (hbm_bytes) *hbm_bytes = L->arena_bytes;
  if (host_bytes) *host_bytes = L->mirror_bytes;
  return MOE_OK;
}

int moe_layer_info(moe_layer* L, uint64_t* arena_bytes, uint64_t* expert_bytes) {
  if (!L) return fail(MOE_EINVAL, "moe_layer_info: null layer");
  if (arena_bytes) *arena_bytes = L->arena_bytes;
  if (expert_bytes) *expert_bytes = L->geom.expert_bytes;
  return MOE_OK;
}

int moe_set_router(moe_layer* L, const uint16_t* wr_bf16, const float* bias, int where) {
  if (!L || !wr_bf16) return fail(MOE_EINVAL, "moe_set_router: null argument");
  DeviceGuard dg(L->device);
  const cudaMemcpyKind kind = where == MOE_DEVICE ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
  CK("moe_set_router: copy weights",
     cudaMemcpy(L->router, wr_bf16, sizeof(uint16_t) * (size_t)L->E * L->H, kind));
  L->has_bias = bias != nullptr;
  if (bias) CK("moe_set_router: copy bias", cudaMemcpy(L->bias, bias, sizeof(float) * L->E, kind));
  L->router_set = true;
  return MOE_OK;
}

int moe_set_router_mode(moe_layer* L, int mode) {
  if (!L) return fail(MOE_EINVAL, "moe_set_router_mode: null layer");
  if (mode != MOE_ROUTER_SOFTMAX && mode != MOE_ROUTER_SIGMOID)
    return fail(MOE_EINVAL, "moe_set_router_mode: unknown mode %d", mode);
  L->router_mode = mode == MOE_ROUTER_SIGMOID ? ROUTER_SIGMOID : ROUTER_SOFTMAX;
  return MOE_OK;
}

int moe_pack_matrix(moe_layer* L, int expert, int matrix, const uint8_t* codes,
                    const uint8_t* scales, const float* tscale, int where, void* stream) {
  if (!L || !codes || !scales) return fail(MOE_EINVAL, "moe_pack_matrix: null argument");
  if (L->fmt == MOE_FMT_NVFP4 && !tscale)
    return fail(MOE_EINVAL, "moe_pack_matrix: NVFP4 needs a tensor scale");
  if (expert < 0 || expert >= L->E + L->shared)
    return fail(MOE_EINVAL, "moe_pack_matrix: expert %d out of range", expert);
  if (matrix < 0 || matrix > 2) return fail(MOE_EINVAL, "moe_pack_matrix: matrix %d", matrix);
  DeviceGuard dg(L->device);
  cudaStream_t st = (cudaStream_t)stream;
  L->mma_dirty = true;  // (the MMA layout follows the arena)
  const int rows = matrix == MOE_DOWN ? L->H : L->I, K = matrix == MOE_DOWN ? L->I : L->H;
  const bool fp4 = L->dev_fmt == FMT_NVFP4, mx = L->fmt == MOE_FMT_MXFP4;
  const size_t code_bytes = fp4 ? (size_t)rows * K / 2 : (size_t)rows * K;
  const size_t scale_bytes =
      mx ? (size_t)rows * K / 32 : (fp4 ? (size_t)rows * K / 16 : (size_t)rows * K / 128);
  // MXFP4: the converted e4m3 scales and a range flag, on the device
  const size_t tile_scale_bytes = mx ? (size_t)rows * K / 16 : 0;
  const size_t tmp_bytes = (where != MOE_DEVICE ? code_bytes + scale_bytes : 0) +
                           (mx ? tile_scale_bytes + 16 : 0);
  const uint8_t* c = codes;
  const uint8_t* s = scales;
  uint8_t* tmp = nullptr;
  if (tmp_bytes && alloc_dev((void**)&tmp, tmp_bytes) != cudaSuccess) {
    cudaGetLastError();
    return fail(MOE_ENOMEM, "moe_pack_matrix: staging allocation of %zu bytes failed", tmp_bytes);
  }
  size_t used = 0;
  if (where != MOE_DEVICE) {
    cudaError_t e = cudaMemcpy(tmp, codes, code_bytes, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(tmp + code_bytes, scales, scale_bytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      cudaFree(tmp);
      CK("moe_pack_matrix: copy codes and scales", e);
    }
    c = tmp;
    s = tmp + code_bytes;
    used = code_bytes + scale_bytes;
    st = 0;
  }
  const ExpertGeom& g = L->geom;
  uint8_t* dst = const_cast<uint8_t*>(expert_ptr(L, expert)) + tile_offset(g, matrix, 0);
  const uint64_t stride = matrix == MOE_DOWN ? (uint64_t)g.dn.tile_bytes : 2u * g.gu.tile_bytes;
  float* ts_dst = L->tscale + expert * 3 + matrix;
  cudaError_t e = cudaSuccess;
  int* bad = nullptr;
  if (mx) {  // MXFP4 -> NVFP4 tile scales and the tensor scale, then the NVFP4 packer
    uint8_t* tile_scales = tmp + used;
    bad = reinterpret_cast<int*>(tmp + used + tile_scale_bytes);
    e = cudaMemsetAsync(bad, 0, sizeof(int), st);
    if (e == cudaSuccess) e = launch_mx_to_tile_scales(c, s, rows, K, tile_scales, ts_dst, bad, st);
    if (e == cudaSuccess)
      e = launch_pack(FMT_NVFP4, c, tile_scales, rows, K, dst, stride, nullptr, 1.0f, nullptr, st);
  } else {
    const float* ts_src = (fp4 && where == MOE_DEVICE) ? tscale : nullptr;
    const float ts_val = (fp4 && where != MOE_DEVICE) ? *tscale : 1.0f;
    e = launch_pack(L->dev_fmt, c, s, rows, K, dst, stride, ts_src, ts_val, ts_dst, st);
  }
  int bad_h = 0;
  if (tmp) {
    cudaError_t e2 = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = e2;
    if (e == cudaSuccess && bad) e = cudaMemcpy(&bad_h, bad, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(tmp);
  }
  CK("moe_pack_matrix: pack kernel", e);
  if (bad_h)
    return fail(MOE_EINVAL,
                "moe_pack_matrix: MXFP4 block exponents span more than 17 binades (or a NaN "
                "scale); the tile layout holds them as e4m3 powers of two 2^-9..2^8");
  return MOE_OK;
}

int moe_pack_weights(moe_layer* L, const uint16_t* wr_bf16, const float* bias,
                     const moe_canonical_matrix* mats) {
  if (!L || !wr_bf16 || !mats) return fail(MOE_EINVAL, "moe_pack_weights: null argument");
  int rc = moe_set_router(L, wr_bf16, bias, MOE_HOST);
  if (rc) return rc;
  for (int e = 0; e < L->E + L->shared; ++e)
    for (int m = 0; m < 3; ++m) {
      const moe_canonical_matrix& M = mats[e * 3 + m];
      rc = moe_pack_matrix(L, e, m, M.codes, M.scales, &M.tscale, MOE_HOST, nullptr);
      if (rc) return rc;
    }
  return MOE_OK;
}

int moe_quantize_nvfp4(const float* W, int rows, int K, uint8_t* codes, uint8_t* scales,
                       float* tscale, void* stream) {
  if (!W || !codes || !scales || !tscale) return fail(MOE_EINVAL, "moe_quantize_nvfp4: null argument");
  if (rows < 1 || K < 16 || K % 16) return fail(MOE_EINVAL, "moe_quantize_nvfp4: bad shape %dx%d", rows, K);
  if (((uintptr_t)W | (uintptr_t)codes) & 15u)
    return fail(MOE_EINVAL, "moe_quantize_nvfp4: W and codes must be 16-byte aligned");
  CK("moe_quantize_nvfp4", launch_quantize_nvfp4(W, rows, K, codes, scales, tscale,
                                                 (cudaStream_t)stream));
  return MOE_OK;
}

int moe_quantize_fp6(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps, void* stream) {
  if (!W || !codes || !exps) return fail(MOE_EINVAL, "moe_quantize_fp6: null argument");
  if (rows < 1 || K < 128 || K % 128) return fail(MOE_EINVAL, "moe_quantize_fp6: bad shape %dx%d", rows, K);
  if (((uintptr_t)W | (uintptr_t)codes) & 15u)
    return fail(MOE_EINVAL, "moe_quantize_fp6: W and codes must be 16-byte aligned");
  CK("moe_quantize_fp6", launch_quantize_fp6(W, rows, K, codes, exps, (cudaStream_t)stream));
  return MOE_OK;
}

int moe_quantize_mxfp4(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps, void* stream) {
  if (!W || !codes || !exps) return fail(MOE_EINVAL, "moe_quantize_mxfp4: null argument");
  if (rows < 1 || K < 32 || K % 32) return fail(MOE_EINVAL, "moe_quantize_mxfp4: bad shape %dx%d", rows, K);
  if (((uintptr_t)W | (uintptr_t)codes) & 15u)
    return fail(MOE_EINVAL, "moe_quantize_mxfp4: W and codes must be 16-byte aligned");
  CK("moe_quantize_mxfp4", launch_quantize_mxfp4(W, rows, K, codes, exps, (cudaStream_t)stream));
  return MOE_OK;
}

int moe_forward(moe_layer* L, const uint16_t* x, int T, float* out, void* stream) {
  int rc = check_forward_args(L, x, T, out);
  if (rc) return rc;
  DeviceGuard dg(L->device);
  return forward_impl(L, x, T, out, (cudaStream_t)stream);
}

int moe_forward_host(moe_layer* L, const uint16_t* x_host, int T, float* out_host, void* stream) {
  if (!L || !x_host || !out_host) return fail(MOE_EINVAL, "moe_forward_host: null argument");
  if (!L->ws) return fail(MOE_ESTATE, "moe_forward_host: no workspace (moe_layer_reserve first)");
  int rc = check_forward_args(L, L->x_stage, T, L->out_stage);
  if (rc) return rc;
  DeviceGuard dg(L->device);
  cudaStream_t st = (cudaStream_t)stream;
  // Page-locked, device-mapped buffers (cudaHostAlloc, cudaHostRegister): the
  // kernels read x and write out through the CPU-GPU link themselves, with no
  // separate copies.  Other host memory goes through the staging buffers.
  cudaPointerAttributes ax{}, ao{};
  if (cudaPointerGetAttributes(&ax, x_host) == cudaSuccess && ax.type == cudaMemoryTypeHost &&
      ax.devicePointer && cudaPointerGetAttributes(&ao, out_host) == cudaSuccess &&
      ao.type == cudaMemoryTypeHost && ao.devicePointer &&
      !(((uintptr_t)ax.devicePointer | (uintptr_t)ao.devicePointer) & 15u)) {
    L->x_mapped = true;
    rc = forward_impl(L, static_cast<const uint16_t*>(ax.devicePointer), T,
                      static_cast<float*>(ao.devicePointer), st);
    L->x_mapped = false;
    if (rc) return rc;
    CK("moe_forward_host: synchronize", cudaStreamSynchronize(st));
    return MOE_OK;
  }
  cudaGetLastError();  // (pageable memory: the attribute query's status is not an error here)
  CK("moe_forward_host: copy x", cudaMemcpyAsync(L->x_stage, x_host, (size_t)T * L->H * 2,
                                                 cudaMemcpyHostToDevice, st));
  rc = forward_impl(L, L->x_stage, T, L->out_stage, st);
  if (rc) return rc;
  CK("moe_forward_host: copy out", cudaMemcpyAsync(out_host, L->out_stage, (size_t)T * L->H * 4,
                                                   cudaMemcpyDeviceToHost, st));
  CK("moe_forward_host: synchronize", cudaStreamSynchronize(st));
  return MOE_OK;
}

int moe_forward_routed(moe_layer* L, const uint16_t* x, int T, const int32_t* idx,
                       const float* gates, float* out, void* stream) {
  int rc = check_forward_args(L, x, T, out);
  if (rc) return rc;
  if (!idx || !gates) return fail(MOE_EINVAL, "moe_forward_routed: null idx or gates");
  DeviceGuard dg(L->device);
  cudaStream_t st = (cudaStream_t)stream;
  const size_t S = (size_t)T * L->k;
  CK("moe_forward_routed: copy idx", cudaMemcpyAsync(L->idx, idx, S * 4, cudaMemcpyDeviceToDevice, st));
  CK("moe_forward_routed: copy gates",
     cudaMemcpyAsync(L->gates, gates, S * 4, cudaMemcpyDeviceToDevice, st));
  if (w4a4(L)) {
    if (!fq_path(L, T) && (rc = launch_quant_x(L, x, T, st))) return rc;
  } else if (!tm_path(L, T)) {
    CK("x conversion kernel launch", launch_convert_x(x, L->xh, (long)T * L->H, L->status, st));
  }
  RouteParams rp = route_params(L, x, T);
  CK("dispatch kernel launch", launch_dispatch(rp, false, st));
  L->last_T = T;
  L->last_has_logits = false;
  return run_experts(L, x, T, out, st);
}

int moe_set_act_format(moe_layer* L, int fmt) {
  if (!L) return fail(MOE_EINVAL, "moe_set_act_format: null layer");
  if (fmt != MOE_ACT_BF16 && fmt != MOE_ACT_NVFP4)
    return fail(MOE_EINVAL, "moe_set_act_format: unknown activation format %d", fmt);
  if (fmt == MOE_ACT_NVFP4 && L->dev_fmt == FMT_NVFP4 && !L->mma && L->H % 128 == 0 &&
      (2 * L->I) % 128 == 0) {
    // the block-scaled GEMMs' copy of the weights in the MMA layout (built before the next forward)
    DeviceGuard dg(L->device);
    MmaGeom gu, dn;
    mma_geoms(L, gu, dn);
    const uint64_t eb = gu.codes + gu.scales + dn.codes + dn.scales;
    const size_t bytes = (size_t)eb * (L->E + L->shared);
    uint8_t* mma = nullptr;
    if (alloc_dev((void**)&mma, bytes) != cudaSuccess) {
      cudaGetLastError();
      return fail(MOE_ENOMEM, "moe_set_act_format: allocation of the MMA-layout weights (%zu bytes) failed",
                  bytes);
    }
    const cudaError_t e = cudaMemset(mma, 0, bytes);
    if (e != cudaSuccess) {
      cudaFree(mma);
      CK("moe_set_act_format: clear the MMA-layout weights", e);
    }
    L->mma = mma;
    L->mma_expert_bytes = eb;
    L->mma_dirty = true;
    make_mma_maps(L);
  }
  L->act_fmt = fmt;
  return MOE_OK;
}

int moe_quantize_act_nvfp4(const void* in, int in_bf16, int rows, int K, uint8_t* codes,
                           uint8_t* scales, float* tscale, void* stream) {
  if (!in || !codes || !scales || !tscale)
    return fail(MOE_EINVAL, "moe_quantize_act_nvfp4: null argument");
  if (rows < 1 || K < 16 || K % 16) return fail(MOE_EINVAL, "moe_quantize_act_nvfp4: bad shape %dx%d", rows, K);
  if (((uintptr_t)in | (uintptr_t)codes) & 15u)
    return fail(MOE_EINVAL, "moe_quantize_act_nvfp4: in and codes must be 16-byte aligned");
  CK("moe_quantize_act_nvfp4", launch_quantize_act(in, in_bf16 != 0, rows, K, codes, scales, nullptr,
                                                   tscale, nullptr, false, (cudaStream_t)stream));
  return MOE_OK;
}

int moe_set_wait_budget(moe_layer* L, int64_t cycles) {
  if (!L) return fail(MOE_EINVAL, "moe_set_wait_budget: null layer");
  L->wait_budget = cycles > 0 ? (long long)cycles : 0;
  return MOE_OK;
}

int moe_debug_fail_alloc(int n) {
  if (n < 0) return fail(MOE_EINVAL, "moe_debug_fail_alloc: n = %d < 0", n);
  g_fail_alloc.store(n);
  return MOE_OK;
}

int moe_debug_check_workspace(moe_layer* L, int* bad_bytes) {
  if (!L || !bad_bytes) return fail(MOE_EINVAL, "moe_debug_check_workspace: null argument");
  if (!L->ws) return fail(MOE_ESTATE, "moe_debug_check_workspace: no workspace");
  DeviceGuard dg(L->device);
  CK("moe_debug_check_workspace: synchronize", cudaDeviceSynchronize());
  std::vector<unsigned char> buf(kGuard);
  int bad = 0;
  for (size_t off : L->guards) {
    CK("moe_debug_check_workspace: read guard",
       cudaMemcpy(buf.data(), static_cast<char*>(L->ws) + off, kGuard, cudaMemcpyDeviceToHost));
    for (unsigned char b : buf) bad += b != kCanary;
  }
  *bad_bytes = bad;
  return MOE_OK;
}

int moe_debug_dequant(moe_layer* L, int expert, int matrix, float* out, void* stream) {
  if (!L || !out) return fail(MOE_EINVAL, "moe_debug_dequant: null argument");
  if (expert < 0 || expert >= L->E + L->shared || matrix < 0 || matrix > 2)
    return fail(MOE_EINVAL, "moe_debug_dequant: expert %d matrix %d out of range", expert, matrix);
  DeviceGuard dg(L->device);
  const ExpertGeom& g = L->geom;
  const int rows = matrix == MOE_DOWN ? L->H : L->I, K = matrix == MOE_DOWN ? L->I : L->H;
  const uint8_t* src = expert_ptr(L, expert) + tile_offset(g, matrix, 0);
  const uint64_t stride = matrix == MOE_DOWN ? (uint64_t)g.dn.tile_bytes : 2u * g.gu.tile_bytes;
  CK("moe_debug_dequant", launch_debug_dequant(L->dev_fmt, src, stride, rows, K,
                                               L->tscale + expert * 3 + matrix, out,
                                               (cudaStream_t)stream));
  return MOE_OK;
}

int moe_debug_routing(moe_layer* L, float* logits, int32_t* idx, float* gates, int32_t* counts,
                      int32_t* offsets, int32_t* perm, void* stream) {
  if (!L) return fail(MOE_EINVAL, "moe_debug_routing: null layer");
  if (!L->last_T) return fail(MOE_ESTATE, "moe_debug_routing: no forward has run");
  DeviceGuard dg(L->device);
  cudaStream_t st = (cudaStream_t)stream;
  const size_t T = L->last_T, S = T * L->k, E = L->E;
  const cudaMemcpyKind d2d = cudaMemcpyDeviceToDevice;
  if (logits) {
    if (!L->last_has_logits) return fail(MOE_ESTATE, "moe_debug_routing: last call was routed");
    CK("moe_debug_routing: logits", cudaMemcpyAsync(logits, L->logits, T * E * 4, d2d, st));
  }
  if (idx) CK("moe_debug_routing: idx", cudaMemcpyAsync(idx, L->idx, S * 4, d2d, st));
  if (gates) CK("moe_debug_routing: gates", cudaMemcpyAsync(gates, L->gates, S * 4, d2d, st));
  if (counts) CK("moe_debug_routing: counts", cudaMemcpyAsync(counts, L->counts, E * 4, d2d, st));
  if (offsets)
    CK("moe_debug_routing: offsets", cudaMemcpyAsync(offsets, L->offsets, (E + 1) * 4, d2d, st));
  if (perm) CK("moe_debug_routing: perm", cudaMemcpyAsync(perm, L->perm, S * 4, d2d, st));
  return MOE_OK;
}

int moe_debug_run_phase(moe_layer* L, int phase, const uint16_t* x, int T, float* out,
                        void* stream) {
  int rc = check_forward_args(L, x, T, out);
  if (rc) return rc;
  if (L->last_T != T || !L->last_has_logits)
    return fail(MOE_ESTATE, "moe_debug_run_phase: needs a moe_forward with T = %d first", T);
  DeviceGuard dg(L->device);
  cudaStream_t st = (cudaStream_t)stream;
  RouteParams rp = route_params(L, x, T);
  ExpertParams ep = expert_params(L, x, T);
  const int grid_y = ep.nsh + max_routed_entries(T, L->E, L->k);
  // W4A4: the x quantiser runs with the routing phase, the a quantiser with the down phase
  if (w4a4(L) && phase == 0 && !fq_path(L, T) && (rc = launch_quant_x(L, x, T, st))) return rc;
  if (w4a4(L) && phase == 3 && (rc = launch_quant_a(L, T, st))) return rc;
  if (small_path(L, T)) {  // router; gate/up (routing inside); down + combine (routing inside)
    if (phase < 0 || phase > 4) return fail(MOE_EINVAL, "moe_debug_run_phase: phase %d", phase);
    if (phase == 0) CK("router", launch_router(rp, st));
    if (phase == 2)
      CK("gate/up", launch_gateup_routed(ep, rp, ep.nsh + max_routed_entries(T, L->E, L->k), st));
    if (phase == 3) CK("down+combine", launch_down_combine(ep, L->gates, L->inv, out, false, true, st));
    return MOE_OK;
  }
  const bool fused = fused_down(L, T);
  switch (phase) {
    case 0:
      if (tc_router(L, T)) {
        const int rc = launch_tc_routing_gemm(L, x, T, st);
        if (rc) return rc;
      } else {
        CK("router", launch_router(rp, st));
      }
      break;
    case 1:
      if (T <= kFusedTopkMaxT && !tc_router(L, T)) {
        CK("top-k/dispatch", launch_route_finish(rp, true, false, st));
      } else if ((rc = launch_topk_and_dispatch(L, rp, T, false, st))) {
        return rc;
      }
      // the token rows in slot order for the tensor-core GEMMs (a4 gather): x
      // gathered (W4A16), or quantised into its rows (W4A4)
      if (tm_path(L, T) && (rc = launch_row_gather(L, ep, T, st))) return rc;
      if (fq_path(L, T) && ((rc = refresh_mma(L, st)) || (rc = launch_quant_x_rows(L, x, T, st))))
        return rc;
      break;
    case 2:
      if (fq_path(L, T))
        CK("gate/up", launch_tc_fp4_gateup(ep, ep.nsh_tc + max_tc_entries(T, L->E, L->k), L->map_gu_mma,
                                           L->map_bx_c, L->map_bx_s, st));
      else if (tm_path(L, T)) {
        if ((rc = launch_tm_gateup(L, ep, T, st))) return rc;
      }
      else if (tc_path(L, T))
        CK("gate/up", launch_tc_gateup(ep, ep.nsh_tc + max_tc_entries(T, L->E, L->k), L->map_gu, st));
      else
        CK("gate/up", launch_gateup(ep, grid_y, false, st));
      break;
    case 3:
      if (fq_path(L, T) && (rc = refresh_mma(L, st))) return rc;
      if (fq_path(L, T))
        CK("down", launch_tc_fp4_down(ep, ep.nsh_tc + max_tc_entries(T, L->E, L->k), L->map_dn_mma,
                                      L->map_ba_c, L->map_ba_s, st));
      else if (tm_path(L, T))
        CK("down", launch_tc_tm_down(ep, ep.nsh_tc + max_tc_entries(T, L->E, L->k), L->map_dn8,
                                     L->map_dn8s, L->map_ab, st));
      else if (tc_path(L, T))
        CK("down", launch_tc_down(ep, ep.nsh_tc + max_tc_entries(T, L->E, L->k), L->map_dn, st));
      else if (fused)
        CK("down+combine", launch_down_combine(ep, L->gates, L->inv, out, false, false, st));
      else
        CK("down", launch_down(ep, grid_y, false, st));
      break;
    case 4:
      if (!fused) CK("combine", launch_combine(ep, L->gates, L->inv, out, false, st));
      break;
    default: return fail(MOE_EINVAL, "moe_debug_run_phase: phase %d", phase);
  }
  return MOE_OK;
}

}  // extern "C"
