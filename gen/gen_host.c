/*
 * Host side of the seeded input generator (see moe_gen.h): fills host
 * buffers, split over POSIX threads.  Holds none of the layer's arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#include "moe_gen.h"

typedef struct {
  void* out;
  uint64_t begin, end, key, offset;
  float sigma;
  int bf16;
} fill_job;

static void* fill_worker(void* p) {
  fill_job* j = (fill_job*)p;
  if (j->bf16) {
    uint16_t* o = (uint16_t*)j->out;
    for (uint64_t i = j->begin; i < j->end; ++i)
      o[i] = moe_gen_bf16_rne(moe_gen_normal(j->key, j->offset + i) * j->sigma);
  } else {
    float* o = (float*)j->out;
    for (uint64_t i = j->begin; i < j->end; ++i)
      o[i] = moe_gen_normal(j->key, j->offset + i) * j->sigma;
  }
  return NULL;
}

static void fill(void* out, uint64_t n, uint64_t key, float sigma, uint64_t offset, int bf16,
                 int threads) {
  if (threads < 1) threads = 1;
  if (threads > 64) threads = 64;
  if (n < (1u << 16)) threads = 1;
  fill_job jobs[64];
  pthread_t tid[64];
  uint64_t per = (n + (uint64_t)threads - 1) / (uint64_t)threads;
  int launched = 0;
  for (int t = 0; t < threads; ++t) {
    uint64_t b = per * (uint64_t)t, e = b + per;
    if (b >= n) break;
    if (e > n) e = n;
    jobs[t] = (fill_job){out, b, e, key, offset, sigma, bf16};
    if (threads == 1 || pthread_create(&tid[t], NULL, fill_worker, &jobs[t]) != 0) {
      fill_worker(&jobs[t]);
      tid[t] = 0;
    }
    launched = t + 1;
  }
  for (int t = 0; t < launched; ++t)
    if (tid[t]) pthread_join(tid[t], NULL);
}

uint64_t moe_gen_stream_key(uint64_t seed, uint32_t tensor, uint32_t a, uint32_t b) {
  return moe_gen_key(seed, tensor, a, b);
}

/* out[i] = N(0,1)-like deviate (key, offset + i) * sigma, fp32 */
void moe_gen_fill_f32(float* out, uint64_t n, uint64_t key, float sigma, uint64_t offset,
                      int threads) {
  fill(out, n, key, sigma, offset, 0, threads);
}

/* out[i] = bf16_rne(deviate(key, offset + i) * sigma), bf16 bits */
void moe_gen_fill_bf16(uint16_t* out, uint64_t n, uint64_t key, float sigma, uint64_t offset,
                       int threads) {
  fill(out, n, key, sigma, offset, 1, threads);
}

/* Zipf(s) popularity bias: bias[e] = scale * r_e^(-s), r = a seeded random
 * permutation of 1..E (ranks ordered by the stream's 64-bit draws). */
void moe_gen_zipf_bias(float* bias, int E, uint64_t key, double s, double scale) {
  uint64_t* draw = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)E);
  for (int e = 0; e < E; ++e) draw[e] = moe_gen_u64(key, (uint64_t)e);
  for (int e = 0; e < E; ++e) {
    int rank = 1;
    for (int f = 0; f < E; ++f)
      if (draw[f] < draw[e] || (draw[f] == draw[e] && f < e)) ++rank;
    bias[e] = (float)(scale * pow((double)rank, -s));
  }
  free(draw);
}
