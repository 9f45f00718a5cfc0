// Device quantisers (fp32 -> canonical NVFP4 / FP6 e2m3 / MXFP4), the packer
// (canonical -> the tile layout of layout.cuh) and the debug dequantiser that
// reads the packed bytes back with the expert kernels' decode.
//
// Quantiser recipe (NVFP4 two-level scaling; FP6 "six-bit e2m3 values with a
// power-of-two scale per 128 weights", knivesysl README, "formats"):
//   NVFP4: ts = amax(W) / 2688; s = e4m3_rne((amax_16 / 6) / ts);
//          q = e2m1_rne(w / (s * ts)), ties to even, saturating, +0 for zero.
//   FP6:   E = min{E : amax_128 <= 7.5 * 2^E}; q = e2m3_rne(w * 2^-E).
// Every division is one IEEE fp32 division (byte-exact quantisers need a
// correctly rounded divide: "Strata on an Intel Arc", "The engine itself on
// Intel: the SYCL port").
#include "common.cuh"
#include "kernels.cuh"
#include "layout.cuh"

namespace moe {
namespace {

// e2m1 magnitude code of a >= 0 by round-to-nearest-even on the grid
// {0, .5, 1, 1.5, 2, 3, 4, 6}, saturating: count the decision points passed.
// A midpoint goes to the even code, so it counts as passed only when the
// code above it is even (0.75, 1.75, 3.5).
__device__ __forceinline__ uint32_t e2m1_code_rne(float a) {
  return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
         (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
         (uint32_t)(a > 5.0f);
}

// e2m3 magnitude code of a in [0, 7.5]: the grid has steps 1/8 on [0, 2),
// 1/4 on [2, 4), 1/2 on [4, 7.5]; rintf rounds half to even, and the code is
// the step count plus an even offset, so ties land on the even code.
__device__ __forceinline__ uint32_t e2m3_code_rne(float a) {
  if (a < 2.0f) return (uint32_t)rintf(a * 8.0f);          // 0..16
  if (a < 4.0f) return (uint32_t)rintf(a * 4.0f) + 8u;     // 16..24
  float n = rintf(a * 2.0f);                                // 8..15 (+saturation)
  return (uint32_t)fminf(n, 15.0f) + 16u;                   // 24..31
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  return __half2float(__ushort_as_half((unsigned short)(e4m3x2_to_f16x2(b) & 0xFFFFu)));
}

__global__ void amax_kernel(const float* __restrict__ W, uint64_t n, unsigned int* amax_bits) {
  float m = 0.0f;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(W[i]));
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));  // m >= 0: bit order = value order
}

// one thread per 16-weight block
__global__ void quant_nvfp4_kernel(const float* __restrict__ W, int rows, int K,
                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                   const unsigned int* amax_bits) {
  const int nb = K / 16;
  const uint64_t total = (uint64_t)rows * nb;
  const float A = __uint_as_float(*amax_bits);
  const float ts = (A > 0.0f) ? __fdiv_rn(A, 2688.0f) : 0.0f;
  for (uint64_t b = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b < total;
       b += (uint64_t)gridDim.x * blockDim.x) {
    const float4* w4 = reinterpret_cast<const float4*>(W + b * 16);
    float w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 v = w4[i];
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(w[i]));
    uint32_t s = 0;
    if (ts > 0.0f) s = f32_to_e4m3_satfinite(__fdiv_rn(__fdiv_rn(amax, 6.0f), ts));
    uint32_t packed[2] = {0u, 0u};
    if (s != 0) {
      const float denom = __fmul_rn(e4m3_to_f32(s), ts);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float v = __fdiv_rn(w[i], denom);
        uint32_t q = e2m1_code_rne(fabsf(v));
        if (v < 0.0f && q != 0u) q |= 8u;
        packed[i / 8] |= q << (4 * (i % 8));
      }
    }
    reinterpret_cast<uint2*>(codes)[b] = make_uint2(packed[0], packed[1]);
    scales[b] = (uint8_t)s;
  }
}

// Activation rows to NVFP4 with one tensor scale per row: one warp per row,
// 8 rows per CTA; lane l takes the 16-column blocks l, l + 32, ...
// The same arithmetic as quant_nvfp4_kernel (IEEE fp32 divisions, e4m3 and
// e2m1 round to nearest even), so a row gives the bytes the weight quantiser
// gives for a one-row matrix.  Codes and scales of output row r start at
// r * cpitch and r * spitch; with `inv`, input row t (a token) goes to the
// kd output rows inv[t * kd + j] (its expert-sorted slots) and, when
// shared_base >= 0, to row shared_base + t (its shared-expert row).
template <bool IN_BF16>
__global__ void __launch_bounds__(256) quant_act_kernel(const void* __restrict__ in, int rows, int K,
                                                        uint8_t* __restrict__ codes,
                                                        uint8_t* __restrict__ scales,
                                                        uint16_t* __restrict__ out_f16,
                                                        float* __restrict__ ts_out, int* status,
                                                        int cpitch, int spitch,
                                                        const int* __restrict__ inv, int kd,
                                                        int shared_base) {
  griddep_wait();
  griddep_launch();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= rows) return;
  auto load16 = [&](int b, float (&w)[16]) {
    if constexpr (IN_BF16) {
      const uint4* q = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(in) +
                                                      (size_t)row * K + 16 * b);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 v = q[h];
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          w[8 * h + 2 * i] = __uint_as_float(u[i] << 16);
          w[8 * h + 2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
        }
      }
    } else {
      const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(in) +
                                                        (size_t)row * K + 16 * b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = q[i];
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
    }
  };
  const int nb = K / 16;
  float m = 0.0f;
  for (int b = lane; b < nb; b += 32) {
    float w[16];
    load16(b, w);
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(w[i]));
  }
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float A = m;
  if (!(A <= 3.0e38f)) {  // inf or NaN in the row
    if (lane == 0 && status) *status = kStatusRange;
    A = 0.0f;
  }
  const float ts = (A > 0.0f) ? __fdiv_rn(A, 2688.0f) : 0.0f;
  if (lane == 0) ts_out[row] = ts;
  for (int b = lane; b < nb; b += 32) {  // (the row again, from L1)
    float w[16];
    load16(b, w);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(w[i]));
    uint32_t s = 0;
    if (ts > 0.0f) s = f32_to_e4m3_satfinite(__fdiv_rn(__fdiv_rn(amax, 6.0f), ts));
    uint32_t packed[2] = {0u, 0u};
    if (s != 0) {
      const float denom = __fmul_rn(e4m3_to_f32(s), ts);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float v = __fdiv_rn(w[i], denom);
        uint32_t q = e2m1_code_rne(fabsf(v));
        if (v < 0.0f && q != 0u) q |= 8u;
        packed[i / 8] |= q << (4 * (i % 8));
      }
    }
    auto put = [&](size_t r) {
      if (codes) *reinterpret_cast<uint2*>(codes + r * cpitch + 8 * b) = make_uint2(packed[0], packed[1]);
      if (scales) scales[r * spitch + b] = (uint8_t)s;
    };
    if (inv) {
      for (int j = 0; j < kd; ++j) put((size_t)inv[(size_t)row * kd + j]);
      if (shared_base >= 0) put((size_t)shared_base + row);
    } else {
      put((size_t)row);
    }
    if (out_f16) {  // e2m1 code x e4m3 scale: both exact in f16, so is the product
      const uint32_t sp = dup_lo(e4m3x2_to_f16x2(s));
      uint32_t h[8];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t f[4];
        e2m1x8_to_f16x8(packed[q], f);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[4 * q + i] = hmul2(f[i], sp);
      }
      uint4* o = reinterpret_cast<uint4*>(out_f16 + (size_t)row * K + 16 * b);
      o[0] = make_uint4(h[0], h[1], h[2], h[3]);
      o[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

__global__ void amax_to_tscale_kernel(float* tscale) {
  const float A = tscale[0];  // holds amax bits (a non-negative float)
  tscale[0] = (A > 0.0f) ? __fdiv_rn(A, 2688.0f) : 0.0f;
}

// one warp per 128-weight block
__global__ void quant_fp6_kernel(const float* __restrict__ W, int rows, int K,
                                 uint8_t* __restrict__ codes, uint8_t* __restrict__ exps) {
  const int nb = K / 128;
  const uint64_t total = (uint64_t)rows * nb;
  const int lane = threadIdx.x & 31;
  const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x / 32);
  for (uint64_t b = (uint64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; b < total;
       b += warps) {
    float4 v = reinterpret_cast<const float4*>(W + b * 128)[lane];
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int E = 0;
    if (amax > 0.0f) {
      int e2;
      float f = frexpf(amax, &e2);  // amax = f * 2^e2, f in [0.5, 1)
      E = (f <= 0.9375f) ? e2 - 3 : e2 - 2;
      if (E < -127) E = -127;
    }
    float w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float s = (amax > 0.0f) ? ldexpf(w[i], -E) : 0.0f;
      uint32_t q = e2m3_code_rne(fabsf(s));
      if (s < 0.0f && q != 0u) q |= 32u;
      out |= q << (8 * i);
    }
    reinterpret_cast<uint32_t*>(codes + b * 128)[lane] = out;
    if (lane == 0) exps[b] = (uint8_t)(E + 127);
  }
}

// MXFP4 (OCP MX FP4): one thread per 32-weight block.  X = 2^E with
// E = floor(log2 amax) - 2 (frexpf gives amax = f 2^e2, f in [0.5, 1), so
// floor(log2 amax) = e2 - 1), clamped to [-127, 127]; q = e2m1_rne(w / X)
// with w / X taken exactly (ldexpf by a power of two); all-zero block: byte
// 127, codes 0.
__global__ void quant_mxfp4_kernel(const float* __restrict__ W, int rows, int K,
                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ exps) {
  const uint64_t total = (uint64_t)rows * (K / 32);
  for (uint64_t b = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b < total;
       b += (uint64_t)gridDim.x * blockDim.x) {
    const float4* w4 = reinterpret_cast<const float4*>(W + b * 32);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = w4[i];
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    int E = 0;
    if (amax > 0.0f) {
      int e2;
      frexpf(amax, &e2);
      E = min(127, max(-127, e2 - 3));
    }
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    if (amax > 0.0f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = w4[i];
        const float w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float s = ldexpf(w[j], -E);
          uint32_t q = e2m1_code_rne(fabsf(s));
          if (s < 0.0f && q != 0u) q |= 8u;
          const int c = 4 * i + j;
          packed[c / 8] |= q << (4 * (c % 8));
        }
      }
    }
    reinterpret_cast<uint4*>(codes)[b] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    exps[b] = (uint8_t)(E + 127);
  }
}

// e4m3 byte of 2^p, p in [-9, 8] (normal for p >= -6, subnormal m/8 * 2^-6 below)
__device__ __forceinline__ uint32_t e4m3_pow2(int p) {
  return p >= -6 ? (uint32_t)(p + 7) << 3 : (1u << (p + 9));
}

// MXFP4 -> the NVFP4 tile layout: the shared scale 2^(E_b - 127) of a block of
// 32 becomes the e4m3 scale 2^(E_b - E_max + 8) of both its 16-column halves
// and the fp32 tensor scale 2^(E_max - 135), E_max = the largest exponent of
// a block with a nonzero code.  Exact while every such block lies within 17
// binades of E_max (e4m3 holds 2^-9 .. 2^8); otherwise *bad is set.  One CTA.
__global__ void __launch_bounds__(1024) mx_to_tile_scales_kernel(
    const uint8_t* __restrict__ codes, const uint8_t* __restrict__ exps, int rows, int K,
    uint8_t* __restrict__ nv_scales, float* ts_dst, int* bad) {
  __shared__ int s_max;
  const int64_t nb = (int64_t)rows * (K / 32);
  if (threadIdx.x == 0) s_max = -1;
  __syncthreads();
  int m = -1;
  for (int64_t b = threadIdx.x; b < nb; b += blockDim.x) {
    const uint4 c = reinterpret_cast<const uint4*>(codes)[b];
    const bool nz = ((c.x | c.y | c.z | c.w) & 0x77777777u) != 0u;  // a nonzero magnitude
    if (nz) m = max(m, (int)exps[b]);
  }
  atomicMax(&s_max, m);
  __syncthreads();
  const int emax = s_max < 0 ? 127 : s_max;
  for (int64_t b = threadIdx.x; b < nb; b += blockDim.x) {
    const uint4 c = reinterpret_cast<const uint4*>(codes)[b];
    const bool nz = ((c.x | c.y | c.z | c.w) & 0x77777777u) != 0u;
    uint32_t s = 0u;
    if (nz) {
      const int p = (int)exps[b] - emax + 8;
      if (p < -9 || exps[b] == 255) {
        *bad = 1;
      } else {
        s = e4m3_pow2(p);
      }
    }
    nv_scales[2 * b] = (uint8_t)s;
    nv_scales[2 * b + 1] = (uint8_t)s;
  }
  if (threadIdx.x == 0) *ts_dst = ldexpf(1.0f, emax - 135);
}

// ---------------------------------------------------------------- packer
// one thread per (tile, super-chunk, lane)
__global__ void pack_nvfp4_kernel(const uint8_t* __restrict__ codes,
                                  const uint8_t* __restrict__ scales, int rows, int K,
                                  uint8_t* __restrict__ dst, uint64_t tile_stride,
                                  const float* ts_src, float ts_val, float* ts_dst) {
  const MatGeom g = mat_geom(FMT_NVFP4, K);
  const int tiles = rows / 16;
  const int64_t total = (int64_t)tiles * g.nsc * 32;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0 && ts_dst) *ts_dst = ts_src ? *ts_src : ts_val;
  if (i >= total) return;
  const int lane = (int)(i % 32), s = (int)((i / 32) % g.nsc), r = (int)(i / (32 * g.nsc));
  const int gi = lane >> 2, t = lane & 3;
  const int row0 = 16 * r + gi, row1 = row0 + 8;
  const int nc = sc_units(g, s);
  uint8_t* base = dst + (uint64_t)r * tile_stride + (uint64_t)s * g.sc_bytes;
  uint8_t sv[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    int blk = 4 * (8 * s + j) + t;
    sv[2 * j] = j < nc ? scales[(int64_t)row0 * (K / 16) + blk] : 0;
    sv[2 * j + 1] = j < nc ? scales[(int64_t)row1 * (K / 16) + blk] : 0;
  }
  *reinterpret_cast<uint4*>(base + 16 * lane) = *reinterpret_cast<uint4*>(sv);
  for (int j = 0; j < nc; ++j) {
    const int k0 = 64 * (8 * s + j) + 16 * t;
    uint32_t wv[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int ka = (k0 + 4 * w) / 2, kb = (k0 + 4 * w + 2) / 2;  // byte columns
      uint32_t b0 = codes[(int64_t)row0 * (K / 2) + ka];
      uint32_t b1 = codes[(int64_t)row1 * (K / 2) + ka];
      uint32_t b2 = codes[(int64_t)row0 * (K / 2) + kb];
      uint32_t b3 = codes[(int64_t)row1 * (K / 2) + kb];
      wv[w] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
    *reinterpret_cast<uint4*>(base + 512 * (1 + j) + 16 * lane) =
        make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
}

__global__ void pack_fp6_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ exps,
                                int rows, int K, uint8_t* __restrict__ dst, uint64_t tile_stride,
                                float* ts_dst) {
  const MatGeom g = mat_geom(FMT_FP6, K);
  const int tiles = rows / 16;
  const int64_t total = (int64_t)tiles * g.nsc * 32;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0 && ts_dst) *ts_dst = 1.0f;
  if (i >= total) return;
  const int lane = (int)(i % 32), s = (int)((i / 32) % g.nsc), r = (int)(i / (32 * g.nsc));
  const int gi = lane >> 2, t = lane & 3;
  const int row0 = 16 * r + gi, row1 = row0 + 8;
  const int np = sc_units(g, s);
  const int P = K / 128;
  uint8_t* base = dst + (uint64_t)r * tile_stride + (uint64_t)s * g.sc_bytes;
  uint32_t ew = 0;
  for (int h = 0; h < 2; ++h) {
    int blk = 8 * s + 2 * t + h;
    if (2 * t + h < np && blk < P) {
      ew |= (uint32_t)exps[(int64_t)row0 * P + blk] << (16 * h);
      ew |= (uint32_t)exps[(int64_t)row1 * P + blk] << (16 * h + 8);
    }
  }
  *reinterpret_cast<uint32_t*>(base + 4 * lane) = ew;
  for (int j = 0; j < np; ++j) {
    uint32_t words[12];
#pragma unroll
    for (int m = 0; m < 12; ++m) words[m] = 0;
    for (int h = 0; h < 2; ++h) {
      const int kb = 128 * (8 * s + j) + 64 * h + 16 * t;
      for (int q = 0; q < 2; ++q) {
        uint32_t Ha = 0, Hb = 0, L = 0;
        for (int x = 0; x < 4; ++x) {       // container C_x
          const int w = 2 * q + (x >> 1);   // step
          const int dk = 4 * w + ((x & 1) ? 2 : 0);
          for (int bi = 0; bi < 4; ++bi) {  // byte of the container
            const int row = (bi < 2) ? row0 : row1;
            const uint32_t cd = codes[(int64_t)row * K + kb + dk + (bi & 1)] & 63u;
            const uint32_t hi = cd >> 2, lo = cd & 3u;
            if (x == 0) { Ha |= hi << (8 * bi); L |= lo << (8 * bi); }
            if (x == 1) { Ha |= hi << (8 * bi + 4); L |= lo << (8 * bi + 2); }
            if (x == 2) { Hb |= hi << (8 * bi); L |= lo << (8 * bi + 4); }
            if (x == 3) { Hb |= hi << (8 * bi + 4); L |= lo << (8 * bi + 6); }
          }
        }
        words[h * 6 + q * 3 + 0] = Ha;
        words[h * 6 + q * 3 + 1] = Hb;
        words[h * 6 + q * 3 + 2] = L;
      }
    }
    for (int v = 0; v < 3; ++v)
      *reinterpret_cast<uint4*>(base + 128 + 1536 * j + 512 * v + 16 * lane) =
          make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2], words[4 * v + 3]);
  }
}

// ---------------------------------------------------------------- debug dequant
// one thread per (tile, super-chunk, lane); the decode matches the expert kernels
__global__ void dequant_nvfp4_kernel(const uint8_t* __restrict__ src, uint64_t tile_stride,
                                     int rows, int K, const float* ts_ptr, float* __restrict__ out) {
  const MatGeom g = mat_geom(FMT_NVFP4, K);
  const int64_t total = (int64_t)(rows / 16) * g.nsc * 32;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int lane = (int)(i % 32), s = (int)((i / 32) % g.nsc), r = (int)(i / (32 * g.nsc));
  const int gi = lane >> 2, t = lane & 3;
  const int row0 = 16 * r + gi, row1 = row0 + 8;
  const float ts = *ts_ptr;
  const uint8_t* base = src + (uint64_t)r * tile_stride + (uint64_t)s * g.sc_bytes;
  const uint4 sv = *reinterpret_cast<const uint4*>(base + 16 * lane);
  for (int j = 0; j < sc_units(g, s); ++j) {
    const uint4 cv = *reinterpret_cast<const uint4*>(base + 512 * (1 + j) + 16 * lane);
    const uint32_t sp = e4m3x2_to_f16x2((u4get(sv, j >> 1) >> (16 * (j & 1))) & 0xFFFFu);
    const uint32_t s0 = dup_lo(sp), s1 = dup_hi(sp);
    const int k0 = 64 * (8 * s + j) + 16 * t;
    for (int w = 0; w < 4; ++w) {
      uint32_t h[4];
      e2m1x8_to_f16x8(u4get(cv, w), h);
      const uint32_t a[4] = {hmul2(h[0], s0), hmul2(h[1], s1), hmul2(h[2], s0), hmul2(h[3], s1)};
      const int rr[4] = {row0, row1, row0, row1};
      const int kk[4] = {k0 + 4 * w, k0 + 4 * w, k0 + 4 * w + 2, k0 + 4 * w + 2};
      for (int x = 0; x < 4; ++x) {
        __half2 hv = *reinterpret_cast<const __half2*>(&a[x]);
        out[(int64_t)rr[x] * K + kk[x]] = __fmul_rn(__low2float(hv), ts);
        out[(int64_t)rr[x] * K + kk[x] + 1] = __fmul_rn(__high2float(hv), ts);
      }
    }
  }
}

// Packed NVFP4 tiles of one matrix region (rows M, K columns) of every
// expert -> the MMA layout (layout.cuh): one thread per (expert, tile,
// super-chunk, lane), as the packer.  A code vector's word w holds bytes
// (row g: columns 4w, 4w+1), (row g+8: 4w, 4w+1), (g: 4w+2, 4w+3),
// (g+8: 4w+2, 4w+3) of the lane's 16 columns: two byte permutes give each
// row's 8 bytes in column order.
__global__ void to_mma_layout_kernel(const uint8_t* __restrict__ arena, uint64_t expert_bytes,
                                     uint64_t src_off, int tile_bytes, int M, int K, int n_experts,
                                     uint8_t* __restrict__ dst, uint64_t dst_expert_bytes,
                                     uint64_t codes_off, uint64_t scales_off) {
  const MatGeom g = mat_geom(FMT_NVFP4, K);
  const int tiles = M / 16;
  const int64_t total = (int64_t)n_experts * tiles * g.nsc * 32;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int lane = (int)(i % 32), s = (int)((i / 32) % g.nsc), r = (int)((i / (32 * g.nsc)) % tiles);
  const int64_t e = i / ((int64_t)32 * g.nsc * tiles);
  const int gi = lane >> 2, t = lane & 3;
  const int ra = 16 * r + gi, rb = ra + 8;
  const uint8_t* base = arena + (uint64_t)e * expert_bytes + src_off + (uint64_t)r * tile_bytes +
                        (uint64_t)s * g.sc_bytes;
  uint8_t* codes = dst + (uint64_t)e * dst_expert_bytes + codes_off;
  uint8_t* scl = dst + (uint64_t)e * dst_expert_bytes + scales_off;
  const uint4 sv = *reinterpret_cast<const uint4*>(base + 16 * lane);
  const int mblocks = M / 128;
  for (int j = 0; j < sc_units(g, s); ++j) {
    const int c = 8 * s + j;
    const uint4 cv = *reinterpret_cast<const uint4*>(base + 512 * (1 + j) + 16 * lane);
    // stage c / 4, bytes 32 (c % 4) + 8t of the row's 128
    const uint64_t at = ((uint64_t)(c / 4) * M) * 128 + 32 * (c % 4) + 8 * t;
    *reinterpret_cast<uint2*>(codes + at + (uint64_t)ra * 128) =
        make_uint2(__byte_perm(cv.x, cv.y, 0x6420), __byte_perm(cv.z, cv.w, 0x6420));
    *reinterpret_cast<uint2*>(codes + at + (uint64_t)rb * 128) =
        make_uint2(__byte_perm(cv.x, cv.y, 0x7531), __byte_perm(cv.z, cv.w, 0x7531));
    const uint32_t sp = u4get(sv, j >> 1) >> (16 * (j & 1));  // block 4c + t of rows ra, rb
    const int st = c / 4, kk = c % 4;
    const int rows[2] = {ra, rb};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int x = rows[h], mb = x / 128, rr = x % 128;
      scl[((uint64_t)(st * mblocks + mb) * 4 + kk) * 512 + (rr % 32) * 16 + (rr / 32) * 4 + t] =
          (uint8_t)((sp >> (8 * h)) & 0xFFu);
    }
  }
}

__device__ __forceinline__ float pow2_from_ue8m0(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

__device__ __forceinline__ void fp6_unpack_group(uint32_t Ha, uint32_t Hb, uint32_t L,
                                                 uint32_t (&c)[4]) {
  c[0] = ((Ha << 2) & 0x3C3C3C3Cu) | (L & 0x03030303u);
  c[1] = ((Ha >> 2) & 0x3C3C3C3Cu) | ((L >> 2) & 0x03030303u);
  c[2] = ((Hb << 2) & 0x3C3C3C3Cu) | ((L >> 4) & 0x03030303u);
  c[3] = ((Hb >> 2) & 0x3C3C3C3Cu) | ((L >> 6) & 0x03030303u);
}

__global__ void dequant_fp6_kernel(const uint8_t* __restrict__ src, uint64_t tile_stride, int rows,
                                   int K, float* __restrict__ out) {
  const MatGeom g = mat_geom(FMT_FP6, K);
  const int64_t total = (int64_t)(rows / 16) * g.nsc * 32;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int lane = (int)(i % 32), s = (int)((i / 32) % g.nsc), r = (int)(i / (32 * g.nsc));
  const int gi = lane >> 2, t = lane & 3;
  const int row0 = 16 * r + gi, row1 = row0 + 8;
  const uint8_t* base = src + (uint64_t)r * tile_stride + (uint64_t)s * g.sc_bytes;
  // the exponent word of lane (gi, j/2) holds block j's exponents; read it directly
  for (int j = 0; j < sc_units(g, s); ++j) {
    const uint32_t ew = *reinterpret_cast<const uint32_t*>(base + 4 * ((gi << 2) | (j >> 1)));
    const float f0 = pow2_from_ue8m0((ew >> (16 * (j & 1))) & 0xFFu);
    const float f1 = pow2_from_ue8m0((ew >> (16 * (j & 1) + 8)) & 0xFFu);
    uint32_t words[12];
    for (int v = 0; v < 3; ++v) {
      uint4 q = *reinterpret_cast<const uint4*>(base + 128 + 1536 * j + 512 * v + 16 * lane);
      words[4 * v] = q.x; words[4 * v + 1] = q.y; words[4 * v + 2] = q.z; words[4 * v + 3] = q.w;
    }
    for (int h = 0; h < 2; ++h)
      for (int q = 0; q < 2; ++q) {
        uint32_t c[4];
        fp6_unpack_group(words[h * 6 + q * 3], words[h * 6 + q * 3 + 1], words[h * 6 + q * 3 + 2], c);
        for (int x = 0; x < 4; ++x) {
          const int w = 2 * q + (x >> 1);
          const int kk = 128 * (8 * s + j) + 64 * h + 16 * t + 4 * w + ((x & 1) ? 2 : 0);
          uint32_t hv[2];
          e2m3x4_to_f16x4(c[x], hv);  // hv[0]: row0 (kk, kk+1); hv[1]: row1 (kk, kk+1)
          __half2 a0 = *reinterpret_cast<__half2*>(&hv[0]);
          __half2 a1 = *reinterpret_cast<__half2*>(&hv[1]);
          out[(int64_t)row0 * K + kk] = __low2float(a0) * f0;
          out[(int64_t)row0 * K + kk + 1] = __high2float(a0) * f0;
          out[(int64_t)row1 * K + kk] = __low2float(a1) * f1;
          out[(int64_t)row1 * K + kk + 1] = __high2float(a1) * f1;
        }
      }
  }
}

int blocks_for(int64_t n, int threads) {
  int64_t b = (n + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > 152 * 32) b = 152 * 32;
  return (int)b;
}

}  // namespace

cudaError_t launch_quantize_nvfp4(const float* W, int rows, int K, uint8_t* codes,
                                  uint8_t* scales, float* tscale, cudaStream_t st) {
  const uint64_t n = (uint64_t)rows * K;
  cudaError_t e = cudaMemsetAsync(tscale, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  unsigned int* amax_bits = reinterpret_cast<unsigned int*>(tscale);
  amax_kernel<<<blocks_for((int64_t)n, 256), 256, 0, st>>>(W, n, amax_bits);
  quant_nvfp4_kernel<<<blocks_for((int64_t)rows * (K / 16), 256), 256, 0, st>>>(
      W, rows, K, codes, scales, amax_bits);
  amax_to_tscale_kernel<<<1, 1, 0, st>>>(tscale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_act(const void* in, bool in_bf16, int rows, int K, uint8_t* codes,
                                uint8_t* scales, uint16_t* out_f16, float* ts, int* status,
                                bool pdl, cudaStream_t st, int cpitch, int spitch, const int* inv,
                                int kd, int shared_base) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid((rows + 7) / 8);
  if (cpitch <= 0) cpitch = K / 2;
  if (spitch <= 0) spitch = K / 16;
  if (in_bf16)
    return launch_k(quant_act_kernel<true>, grid, dim3(256), 0, st, pdl, in, rows, K, codes, scales,
                    out_f16, ts, status, cpitch, spitch, inv, kd, shared_base);
  return launch_k(quant_act_kernel<false>, grid, dim3(256), 0, st, pdl, in, rows, K, codes, scales,
                  out_f16, ts, status, cpitch, spitch, inv, kd, shared_base);
}

cudaError_t launch_quantize_fp6(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps,
                                cudaStream_t st) {
  const int64_t blocks = (int64_t)rows * (K / 128);
  quant_fp6_kernel<<<blocks_for(blocks * 32, 256), 256, 0, st>>>(W, rows, K, codes, exps);
  return cudaGetLastError();
}

cudaError_t launch_quantize_mxfp4(const float* W, int rows, int K, uint8_t* codes, uint8_t* exps,
                                  cudaStream_t st) {
  quant_mxfp4_kernel<<<blocks_for((int64_t)rows * (K / 32), 256), 256, 0, st>>>(W, rows, K, codes,
                                                                                exps);
  return cudaGetLastError();
}

cudaError_t launch_mx_to_tile_scales(const uint8_t* codes, const uint8_t* exps, int rows, int K,
                                     uint8_t* nv_scales, float* ts_dst, int* bad, cudaStream_t st) {
  mx_to_tile_scales_kernel<<<1, 1024, 0, st>>>(codes, exps, rows, K, nv_scales, ts_dst, bad);
  return cudaGetLastError();
}

cudaError_t launch_pack(int fmt, const uint8_t* codes, const uint8_t* scales, int rows, int K,
                        uint8_t* dst, uint64_t tile_stride, const float* ts_src, float ts_val,
                        float* ts_dst, cudaStream_t st) {
  const MatGeom g = mat_geom(fmt, K);
  const int64_t n = (int64_t)(rows / 16) * g.nsc * 32;
  const int blocks = (int)((n + 127) / 128);
  if (fmt == FMT_NVFP4)
    pack_nvfp4_kernel<<<blocks, 128, 0, st>>>(codes, scales, rows, K, dst, tile_stride, ts_src,
                                              ts_val, ts_dst);
  else
    pack_fp6_kernel<<<blocks, 128, 0, st>>>(codes, scales, rows, K, dst, tile_stride, ts_dst);
  return cudaGetLastError();
}

cudaError_t launch_to_mma_layout(const uint8_t* arena, uint64_t expert_bytes, uint64_t src_off,
                                 int tile_bytes, int M, int K, int n_experts, uint8_t* dst,
                                 uint64_t dst_expert_bytes, uint64_t codes_off, uint64_t scales_off,
                                 cudaStream_t st) {
  const MatGeom g = mat_geom(FMT_NVFP4, K);
  const int64_t n = (int64_t)n_experts * (M / 16) * g.nsc * 32;
  to_mma_layout_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
      arena, expert_bytes, src_off, tile_bytes, M, K, n_experts, dst, dst_expert_bytes, codes_off,
      scales_off);
  return cudaGetLastError();
}

cudaError_t launch_debug_dequant(int fmt, const uint8_t* src, uint64_t tile_stride, int rows,
                                 int K, const float* ts_ptr, float* out, cudaStream_t st) {
  const MatGeom g = mat_geom(fmt, K);
  const int64_t n = (int64_t)(rows / 16) * g.nsc * 32;
  const int blocks = (int)((n + 127) / 128);
  if (fmt == FMT_NVFP4)
    dequant_nvfp4_kernel<<<blocks, 128, 0, st>>>(src, tile_stride, rows, K, ts_ptr, out);
  else
    dequant_fp6_kernel<<<blocks, 128, 0, st>>>(src, tile_stride, rows, K, out);
  return cudaGetLastError();
}

}  // namespace moe
