/*
 * Seeded synthetic inputs for the quantized MoE expert layer.
 *
 * This header is the one piece of code that both the CPU oracle's tests and
 * the CUDA path's tests/bench use: it draws the layer's inputs (activations x,
 * router weights, fp32 expert weights) and holds none of the layer's own
 * arithmetic (no quantisation, routing, GEMM or activation).
 *
 * Generator: the SplitMix64 output function (Steele, Lea & Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014) applied to a
 * counter, so element i of a tensor is a pure function of (key, i) and any
 * slice can be produced independently on the host or on the device.
 *
 * Normal deviates: the Irwin-Hall construction -- the sum of 12 independent
 * uniforms minus its mean has unit variance and is close to N(0,1).  It is
 * done here in exact integer arithmetic (12 x 16-bit uniforms) followed by a
 * power-of-two scale, so host and device produce bit-identical floats with no
 * dependence on libm.  The support is [-6, 6] standard deviations.
 *
 * Scaling by sigma is a single IEEE fp32 multiply (correctly rounded on both
 * sides, nothing to contract); bf16 values are the round-to-nearest-even of
 * that fp32 value.
 */
#ifndef MOE_GEN_H
#define MOE_GEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define MOE_GEN_FN static __host__ __device__ __forceinline__
#else
#define MOE_GEN_FN static inline
#endif

/* tensor ids used to derive per-tensor stream keys */
enum {
  MOE_GEN_T_X = 1,       /* activations [T x H], bf16, N(0,1) */
  MOE_GEN_T_ROUTER = 2,  /* router weights [E x H], bf16, N(0, 0.02) */
  MOE_GEN_T_WEIGHT = 3,  /* expert matrix (expert, matrix), fp32, N(0, 0.02) */
  MOE_GEN_T_ZIPF = 4,    /* popularity ranks for the Zipf router bias */
  MOE_GEN_T_BIAS = 5     /* normal router bias, N(0, sigma) */
};

/* SplitMix64 output function (the "mix" step). */
MOE_GEN_FN uint64_t moe_gen_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* i-th output of the SplitMix64 sequence whose state starts at `key`. */
MOE_GEN_FN uint64_t moe_gen_u64(uint64_t key, uint64_t i) {
  return moe_gen_mix64(key + (i + 1u) * 0x9E3779B97F4A7C15ULL);
}

/* Stream key of one tensor: (seed, tensor id, a, b), e.g. a = expert, b = matrix. */
MOE_GEN_FN uint64_t moe_gen_key(uint64_t seed, uint32_t tensor, uint32_t a, uint32_t b) {
  uint64_t h = moe_gen_mix64(seed ^ 0x6A09E667F3BCC909ULL);
  h = moe_gen_mix64(h ^ (((uint64_t)tensor << 32) | (uint64_t)a));
  h = moe_gen_mix64(h ^ ((uint64_t)b * 0x9E3779B97F4A7C15ULL + 0x3C6EF372FE94F82BULL));
  return h;
}

/* Approximately N(0,1): Irwin-Hall over 12 uniforms of 16 bits each. */
MOE_GEN_FN float moe_gen_normal(uint64_t key, uint64_t i) {
  uint64_t r0 = moe_gen_u64(key, 3u * i);
  uint64_t r1 = moe_gen_u64(key, 3u * i + 1u);
  uint64_t r2 = moe_gen_u64(key, 3u * i + 2u);
  int32_t s = 0;
  for (int j = 0; j < 4; ++j) {
    s += (int32_t)((r0 >> (16 * j)) & 0xFFFFu);
    s += (int32_t)((r1 >> (16 * j)) & 0xFFFFu);
    s += (int32_t)((r2 >> (16 * j)) & 0xFFFFu);
  }
  /* 2*sum - 12*65535 has standard deviation ~131072 = 2^17: exact in fp32 */
  int32_t c = 2 * s - 786420;
  return (float)c * (1.0f / 131072.0f);
}

/* Uniform in [0, 1) with 53 bits (host-side helpers only). */
MOE_GEN_FN double moe_gen_uniform(uint64_t key, uint64_t i) {
  return (double)(moe_gen_u64(key, i) >> 11) * (1.0 / 9007199254740992.0);
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs). */
MOE_GEN_FN uint16_t moe_gen_bf16_rne(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

#endif /* MOE_GEN_H */
