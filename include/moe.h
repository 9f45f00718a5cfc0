/*
 * moe.h -- C ABI of the GB300 (sm_103a) quantized mixture-of-experts FFN layer.
 *
 * The layer step: router logits, softmax / top-k with renormalised gates,
 * token-to-expert dispatch, per-expert SwiGLU  y = W_down (silu(W_gate x) * (W_up x))
 * with the expert weights dequantised on the fly from NVFP4 (e2m1 codes, an
 * e4m3 scale per 16 weights, an fp32 tensor scale) or FP6 e2m3 (a power-of-two
 * scale per 128 weights), the gate-weighted combine, and an always-on shared
 * expert.  The formats are those of the knivesysl README, "formats" (six-bit
 * e2m3 values with a power-of-two scale per 128 weights; four-bit values with
 * a scale per 16); the router with top-k and the shared expert are the
 * "router_top10" / "shared_expert" kernels of "Strata on an Intel Arc",
 * "The engine itself on Intel: the SYCL port".
 *
 * Conventions for every entry point:
 *   - return 0 (MOE_OK) on success, a negative moe_status on failure; the
 *     message of the last failure on the calling thread is moe_last_error();
 *   - `stream` is a cudaStream_t passed as void* (0 = the legacy default stream);
 *     device-side work is asynchronous on that stream unless stated;
 *   - "device pointer" means memory of the layer's CUDA device that the caller
 *     owns and keeps alive until the stream has finished with it;
 *   - the library owns the packed weights, router copy and workspace of a layer;
 *   - one layer is used from one stream at a time (its workspace is shared).
 * Dimensions: H hidden size, I expert intermediate size, E routed experts,
 * k experts per token, T tokens.  H and I are multiples of 64 (NVFP4, MXFP4)
 * or of 128 (FP6), at most 65536; 1 <= E <= 1024; 1 <= k <= min(E, 32).
 *
 * Value range.  The expert kernels multiply f16 copies of x and of the SwiGLU
 * output a = silu(g) * u (every product is exact, the sums are fp32): the
 * copies are exact to bf16's 8 bits for |x| in [2^-14, 65504] and keep 11 bits
 * of a in the same range.  Below 2^-14 an element keeps an absolute precision
 * of 2^-25 (f16 subnormals).  An element of x or a above 65504 in magnitude
 * (or not finite) records MOE_ERANGE in the layer's status word
 * (moe_layer_status); that forward's output is then not valid.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_layer moe_layer; /* opaque */

enum moe_format { MOE_FMT_NVFP4 = 1, MOE_FMT_FP6_E2M3 = 2, MOE_FMT_MXFP4 = 3 };

enum moe_status {
  MOE_OK = 0,
  MOE_EINVAL = -1,   /* bad argument (null pointer, size, alignment) */
  MOE_ENOMEM = -2,   /* device allocation failed */
  MOE_ECUDA = -3,    /* a CUDA call failed; moe_last_error() names it */
  MOE_ESTATE = -4,   /* call out of order (forward before pack / reserve) */
  MOE_ETIMEOUT = -5, /* a bounded device wait gave up (see moe_layer_status) */
  MOE_ERANGE = -6    /* x or a beyond the f16 range the experts compute in (status word only) */
};

enum moe_matrix { MOE_GATE = 0, MOE_UP = 1, MOE_DOWN = 2 };

/* where a pointer argument lives */
enum moe_where { MOE_HOST = 0, MOE_DEVICE = 1 };

/* ------------------------------------------------------------------ lifetime */

/* Create a layer on the current CUDA device.  format: moe_format; shared: 0 or 1
 * (one always-on shared expert of intermediate size I, weight 1: the
 * "shared_expert" kernel of "Strata on an Intel Arc", parity table of "Where
 * it stands").  Allocates the packed-weight arena (zero-filled) and the
 * tensor-scale table.  *out gets the handle, or NULL on failure (MOE_ENOMEM
 * when an allocation fails; nothing stays allocated). */
int moe_layer_create(int format, int H, int I, int E, int k, int shared, moe_layer** out);

/* Size the forward workspace for up to T_max tokens per call (reserved at
 * start-up so the forward never allocates, as the knivesysl README reserves
 * its buffers at initialisation, "runtime diagnostics").  May be called again
 * to grow it, never while a forward is in flight.  moe_forward allocates
 * nothing, so a forward can be captured into a CUDA graph after this call.
 * MOE_ENOMEM leaves the previous workspace in place.  The workspace buffers
 * are separated by guard regions (see moe_debug_check_workspace). */
int moe_layer_reserve(moe_layer* L, int T_max);

/* Free everything the layer owns (synchronises its device first).  NULL is a no-op. */
void moe_layer_destroy(moe_layer* L);

/* Message of the last failure on this thread ("" if none): the operation and,
 * for MOE_ECUDA, the CUDA error name. */
const char* moe_last_error(void);

/* Read the layer's device status word into *status: 0, or the negative
 * moe_status a kernel recorded: MOE_EINVAL from a device-side bounds check on
 * an expert id or work entry, MOE_ETIMEOUT from a bounded wait that gave up
 * (every device wait is capped, as the bounded spins of "Strata on an Intel
 * Arc" are), MOE_ERANGE from a value beyond f16's range (see "Value range").
 * Synchronises the device; clears the word when reset != 0.  Returns MOE_OK,
 * or an error if the read itself failed. */
int moe_layer_status(moe_layer* L, int reset, int* status);

/* Number of kernels one moe_forward of T tokens launches (>= 0), or an error. */
int moe_forward_launches(moe_layer* L, int T);

/* The expert path one moe_forward of T tokens takes with the layer's current
 * format, placement and activation format (>= 0), or an error. */
enum moe_path {
  MOE_PATH_DECODE = 0,    /* T <= 8: gate/up routes itself; fused down + combine */
  MOE_PATH_STREAM = 1,    /* streamed GEMVs over expert-sorted token groups */
  MOE_PATH_TC_F16 = 2,    /* tcgen05 kind::f16 GEMMs on exactly dequantised weights (held in
                             tensor memory when H and I are multiples of 128) */
  MOE_PATH_TC_FP4 = 3     /* W4A4: tcgen05 kind::mxf4nvf4 block-scaled GEMMs */
};
int moe_forward_path(moe_layer* L, int T);

/* Budget of each bounded wait in the tensor-core kernels, in SM clock cycles
 * (clock64); cycles <= 0 restores the default of 2e9 (about one second).  A
 * wait that runs out stops its CTA's work: the CTA lets its copies and MMAs in
 * flight finish (those drains keep the default budget), frees its tensor
 * memory, records MOE_ETIMEOUT in the status word and returns, leaving the
 * context usable.  Applies to the following forwards. */
int moe_set_wait_budget(moe_layer* L, int64_t cycles);

/* Bytes of the packed arena and of one packed expert (gate + up + down, without
 * its three fp32 tensor scales). */
int moe_layer_info(moe_layer* L, uint64_t* arena_bytes, uint64_t* expert_bytes);

/* ------------------------------------------------------------------ placement */

/* Two memory tiers for the packed experts: HBM, and a pinned host mirror that
 * the kernels read in place over the CPU-GPU link (NVLink-C2C on Grace
 * systems).  This is the host mirror of "Strata on an Intel Arc" ("Planned",
 * item 2: experts without a VRAM slot are read straight from pinned host
 * memory by the expert kernels) and the placement tiers of the Colibri page
 * ("Core techniques and measured findings": fast memory changes speed, not
 * results).
 *
 * in_hbm: host array [E + shared] (the shared expert last); nonzero = the
 * expert gets an HBM slot, zero = it lives in the host mirror.  Moves every
 * expert's packed bytes (and nothing else: tensor scales, router and workspace
 * stay in HBM) to its new place, frees the old storage, and rebuilds the
 * per-expert address table the kernels read.  Results do not depend on the
 * placement: every path runs the same arithmetic on the same bytes, so the
 * output is bit-identical.  With any expert on the host, forwards take the
 * non-tensor-core expert path (the TMA tile maps need one contiguous arena).
 * Synchronises the device; invalidates CUDA graphs captured before it (they
 * hold the old addresses).  May be called before or after packing, and again
 * to move experts.  MOE_ENOMEM if the HBM slots or the pinned mirror cannot be
 * allocated (the old placement then stays). */
int moe_place_experts(moe_layer* L, const uint8_t* in_hbm);

/* The current placement: in_hbm [E + shared] (may be NULL) gets 1 for an HBM
 * slot and 0 for the host mirror; *hbm_bytes / *host_bytes (may be NULL) the
 * packed-expert bytes held in each tier. */
int moe_layer_placement(moe_layer* L, uint8_t* in_hbm, uint64_t* hbm_bytes, uint64_t* host_bytes);

/* ------------------------------------------------------------------ weights */

/* Router weights Wr [E x H] as bf16 bits (row-major) and an optional fp32 bias
 * [E] (NULL = none), host or device memory per `where`.  Copied; synchronous.
 * The router with top-k is the "router_top10" kernel of "Strata on an Intel
 * Arc" (parity table of "Where it stands"). */
int moe_set_router(moe_layer* L, const uint16_t* wr_bf16, const float* bias, int where);

/* Router mode (default MOE_ROUTER_SOFTMAX):
 *   MOE_ROUTER_SOFTMAX: logit = x . Wr_e + bias_e; the k largest logits (ties
 *     to the lower expert index); gates = softmax over the k selected logits.
 *   MOE_ROUTER_SIGMOID: score s_e = sigmoid(x . Wr_e); the k largest s_e +
 *     bias_e are selected (the bias decides the selection only); gates =
 *     s_j / (sum of the selected s).  The logits reported by
 *     moe_debug_routing are then x . Wr_e without the bias.
 * Applies to the following forwards.  MOE_EINVAL for an unknown mode. */
enum moe_router_mode { MOE_ROUTER_SOFTMAX = 0, MOE_ROUTER_SIGMOID = 1 };
int moe_set_router_mode(moe_layer* L, int mode);

/* Activation format of the following forwards (default MOE_ACT_BF16):
 *   MOE_ACT_BF16: W4A16, the activations x and a = silu(g) * u stay exact
 *     (bf16 x, fp32 a; multiplied as f16 copies, see "Value range");
 *   MOE_ACT_NVFP4: W4A4, the knivesysl README's nvfp4 tier with four-bit
 *     activations ("nvfp4 w4a4 for every projection", the table of supported
 *     service formats): x of each token before gate/up, and a of each
 *     (token, expert) row (fp32) before down, are quantised to NVFP4 per row
 *     with the weights' recipe (one fp32 tensor scale per row,
 *     moe_quantize_act_nvfp4), and the products take the dequantised values.
 *     The router keeps bf16 x.  The values stay within f16 (|code x block
 *     scale| <= 2688) and the tensor scales multiply the fp32 accumulators,
 *     so x and a have no f16 range limit in this mode.  On the tensor-core
 *     path (MOE_PATH_TC_FP4) the products run on the block-scaled FP4 MMA
 *     (tcgen05 kind::mxf4nvf4, both operands' e4m3 scales applied by the
 *     tensor core); on the other paths on f16 copies of the exact values.
 * MOE_EINVAL for an unknown format. */
enum moe_act_format { MOE_ACT_BF16 = 0, MOE_ACT_NVFP4 = 1 };
int moe_set_act_format(moe_layer* L, int fmt);

/* Pack one expert matrix from the canonical quantised format into the layer's
 * device layout.  The formats are those of the knivesysl README, the
 * paragraph under the table of supported service formats (e2m3 with a
 * power-of-two scale per 128 weights; four-bit values with a scale per 16).  expert in [0, E) for routed experts, E for the shared one;
 * matrix: moe_matrix (gate and up are [I x H], down is [H x I]; row-major,
 * blocks run along the row).
 *   NVFP4: codes [rows x K/2] bytes, two e2m1 codes per byte, the even column
 *          in the low nibble; scales [rows x K/16] e4m3 bytes; *tscale the fp32
 *          tensor scale (dequantised weight = (e2m1 * e4m3) * tscale).
 *   FP6:   codes [rows x K] bytes, one e2m3 code in the low 6 bits of each;
 *          scales [rows x K/128] ue8m0 exponent bytes (2^(b-127)); tscale
 *          ignored (may be NULL).
 *   MXFP4 (OCP MX FP4): codes as for NVFP4; scales [rows x K/32] ue8m0
 *          exponent bytes (weight = e2m1 * 2^(b-127)); tscale ignored.  The
 *          device layout is NVFP4's: each block's scale becomes the e4m3
 *          power of two 2^(b - b_max + 8) of both of its 16-column halves and
 *          the matrix gets the fp32 tensor scale 2^(b_max - 135), b_max the
 *          largest exponent of a block with a nonzero code.  That is exact
 *          while every such block is within 17 binades of b_max; otherwise
 *          MOE_EINVAL.  Synchronous (it checks that range on the device).
 * codes / scales / tscale are host or device pointers per `where`.  Device input is
 * consumed asynchronously on `stream`; host input is copied synchronously. */
int moe_pack_matrix(moe_layer* L, int expert, int matrix, const uint8_t* codes,
                    const uint8_t* scales, const float* tscale, int where, void* stream);

/* One matrix of the canonical format (see moe_pack_matrix). */
typedef struct moe_canonical_matrix {
  const uint8_t* codes;
  const uint8_t* scales;
  float tscale;
} moe_canonical_matrix;

/* Pack a whole layer from host memory: router (+ optional bias) and
 * mats[expert * 3 + matrix] for expert in [0, E + shared), each in the
 * canonical format of moe_pack_matrix.  Synchronous; the host arrays may be
 * freed when it returns. */
int moe_pack_weights(moe_layer* L, const uint16_t* wr_bf16, const float* bias,
                     const moe_canonical_matrix* mats);

/* Quantise fp32 weights W [rows x K] (device) to canonical NVFP4 on the device
 * (the knivesysl README's nvfp4, a scale per 16 weights, in the two-level
 * reading: an e4m3 block scale under an fp32 tensor scale):
 * tscale = amax(W) / (6 * 448); per 16 weights along K the e4m3 scale
 * s = rne((amax_16 / 6) / tscale); code = rne_e2m1(w / (s * tscale)); ties to
 * the even code, saturating, +0 for zero, s = 0 gives code 0; IEEE fp32
 * division.  Device outputs: codes [rows x K/2], scales [rows x K/16],
 * tscale [1].  K % 16 == 0.  Uses no workspace beyond its outputs. */
int moe_quantize_nvfp4(const float* W, int rows, int K, uint8_t* codes, uint8_t* scales,
                       float* tscale, void* stream);

/* Quantise activation rows to canonical NVFP4 on the device, one tensor scale
 * per row (the W4A4 activations of moe_set_act_format): in [rows x K] bf16
 * bits (in_bf16 != 0) or fp32, device; per row tscale = amax(row) / (6 * 448)
 * and the recipe of moe_quantize_nvfp4 per 16 values.  Device outputs codes
 * [rows x K/2], scales [rows x K/16], tscale [rows].  K % 16 == 0; in and
 * codes 16-byte aligned. */
int moe_quantize_act_nvfp4(const void* in, int in_bf16, int rows, int K, uint8_t* codes,
                           uint8_t* scales, float* tscale, void* stream);

/* Quantise fp32 weights W [rows x K] (device) to canonical FP6 e2m3 on the
 * device (the knivesysl README's fp6, a power-of-two scale per 128 weights): per 128 weights the exponent E = the smallest integer with
 * amax_128 <= 7.5 * 2^E (byte E + 127; 127 for an all-zero block) and
 * code = rne_e2m3(w / 2^E).  Device outputs codes [rows x K], exps [rows x K/128].
 * K % 128 == 0. */
int moe_quantize_fp6(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps,
                     void* stream);

/* Quantise fp32 weights W [rows x K] (device) to canonical MXFP4 (OCP
 * Microscaling v1.0, FP4 E2M1 elements) on the device: per 32 weights along K
 * the shared exponent E = floor(log2 amax_32) - 2, clamped to [-127, 127]
 * (byte E + 127; 127 for an all-zero block), code = rne_e2m1(w / 2^E), ties
 * to the even code, saturating at 6, +0 for zero.  Device outputs codes
 * [rows x K/2] (as NVFP4), exps [rows x K/32].  K % 32 == 0; W and codes
 * 16-byte aligned. */
int moe_quantize_mxfp4(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps,
                       void* stream);

/* ------------------------------------------------------------------ forward */

/* out[T x H] (fp32, device) = the layer applied to x[T x H] (bf16 bits, device):
 * router logits, top-k with renormalised gates ("router_top10"), the
 * expert-sorted dispatch, each selected expert's SwiGLU on weights dequantised
 * on the fly, the shared expert ("shared_expert"), and the gate-weighted
 * combine (the kernels of "Strata on an Intel Arc", parity table of "Where it
 * stands", over the formats of the knivesysl README).
 * 1 <= T <= the reserved T_max.  Asynchronous on `stream`; allocates nothing.
 * x and out must be 16-byte aligned.  Errors in the arguments return at once;
 * device-side errors land in the status word. */
int moe_forward(moe_layer* L, const uint16_t* x, int T, float* out, void* stream);

/* moe_forward with host buffers x (T x H bf16) and out (T x H fp32); returns
 * once `stream` has finished.  MOE_ESTATE before moe_layer_reserve.  Page-locked, device-mapped buffers
 * (cudaHostAlloc / cudaHostRegister, 16-byte aligned) are read and written by
 * the kernels in place over the CPU-GPU link; any other host memory is copied
 * through the layer's staging buffers. */
int moe_forward_host(moe_layer* L, const uint16_t* x_host, int T, float* out_host, void* stream);

/* The layer with the routing given instead of computed: idx [T x k] expert ids
 * (distinct within a token, each in [0, E)) and gates [T x k] fp32, device
 * pointers.  Dispatch, experts, shared expert and combine are the kernels
 * moe_forward runs.  An expert id out of range records MOE_EINVAL in the
 * status word and its slot is skipped. */
int moe_forward_routed(moe_layer* L, const uint16_t* x, int T, const int32_t* idx,
                       const float* gates, float* out, void* stream);

/* ------------------------------------------------------------------ test hooks */

/* Make the n-th following device or pinned-host allocation of the library
 * fail as if memory were exhausted (n = 0: none).  Process-wide.  It lets
 * tests drive every MOE_ENOMEM path (layer creation, workspace, staging of a
 * host pack, placement) on a GPU with memory to spare, as the knivesysl
 * README's regressions check allocation and error recovery. */
int moe_debug_fail_alloc(int n);

/* Check the guard regions between the workspace buffers: *bad_bytes gets the
 * number of guard bytes a kernel overwrote (0 when every kernel stayed inside
 * its buffers).  Synchronises the device.  MOE_ESTATE before
 * moe_layer_reserve. */
int moe_debug_check_workspace(moe_layer* L, int* bad_bytes);

/* Dequantise one packed matrix back to fp32 [rows x K] (device `out`) from the
 * packed device bytes, with the decode the expert kernels use. */
int moe_debug_dequant(moe_layer* L, int expert, int matrix, float* out, void* stream);

/* Copy the routing of the last forward into caller device buffers (any may be
 * NULL): logits [T x E] fp32 (moe_forward only), idx [T x k], gates [T x k],
 * counts [E], offsets [E + 1], perm [T x k] (slot ids t*k + j, expert-sorted,
 * stable). */
int moe_debug_routing(moe_layer* L, float* logits, int32_t* idx, float* gates, int32_t* counts,
                      int32_t* offsets, int32_t* perm, void* stream);

/* Re-run one phase of the last moe_forward on the same arguments, for timing a
 * kernel on its own: 0 router logits, 1 top-k + dispatch, 2 gate/up + SwiGLU,
 * 3 down, 4 combine.  For T <= 8 the expert kernels route themselves: 1 and 4
 * launch nothing, 2 includes top-k and dispatch, 3 includes them and the
 * combine.  The workspace must hold that forward's state (same x, T). */
int moe_debug_run_phase(moe_layer* L, int phase, const uint16_t* x, int T, float* out,
                        void* stream);

/* ------------------------------------------------------------------ no device allocation */

/* Router logits, top-k and gates for callers that cannot allocate device
 * memory.  The pages have no counterpart of this entry point.  It is for code
 * whose GPU memory belongs to someone else's allocator: a serving runtime that
 * plans all of HBM at start-up and hands memory out only from its own pool, or
 * a plug-in inside such a runtime.  For them a cudaMalloc could fail when HBM
 * is full, or would go around the pool's accounting.
 * It computes what moe_forward's routing step computes, with the same kernels:
 *   logits [T x E] fp32 = x [T x H] (bf16 bits) . wr [E x H]^T (bf16 bits) + bias [E]
 *   (bias may be NULL), idx [T x k] the top-k experts per token (ties to the
 *   lower index) and gates [T x k] their renormalised softmax.
 * All pointers are device pointers the caller owns; x and wr are 16-byte
 * aligned; H % 64 == 0, 64 <= H <= 65536, 1 <= E <= 1024, 1 <= k <= min(E, 32),
 * T <= 524280.  The router starts only when the previous work on `stream` has
 * finished, so x, wr and bias may be written by the kernel just before.
 * It allocates nothing.  Its only scratch, the router's K-split partial sums,
 * is a fixed 4 MiB device array inside the library, held by every GPU that
 * loads the library until the process exits.  Inputs that would need more
 * (ksplit(T, E) * T * E > 2^20 floats; always fine when T * E <= 131072) are
 * rejected with MOE_EINVAL.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) and sets the router kernels'
 * shared-memory limit; make that first call before any stream capture.  All
 * calls share the one array and it keeps the last call's contents: calls that
 * may overlap on the GPU (different streams, or several host threads) race on
 * it and must be serialised by the caller.  Asynchronous on `stream`. */
int moe_route_noalloc(const uint16_t* x, int T, int H, const uint16_t* wr, const float* bias,
                      int E, int k, float* logits, int32_t* idx, float* gates, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
