/*
 * Host build of the seeded synthetic-input generator (see gen_common.h).
 * Compiled with -ffp-contract=off so that it produces the same bytes as the
 * device build and the same bytes on x86-64 and aarch64 hosts.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "gen_common.h"

/* ---- exported scalar helpers (used by the tests) ------------------------ */
float gen_ln_f(float u) { return gen_ln(u); }
void gen_cossin_f(float f, float* c, float* s) { gen_cossin_2pi(f, c, s); }
float gen_normal_f(uint64_t key, uint64_t i) { return gen_normal(key, i); }
uint64_t gen_key_u64(uint64_t seed, uint32_t wset, uint32_t layer,
                     uint32_t tensor, uint32_t expert) {
  return gen_key(seed, wset, layer, tensor, expert);
}
uint64_t gen_u64_at(uint64_t key, uint64_t n) { return gen_u64(key, n); }

void gen_f32_to_f16_array(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = gen_f32_to_f16_rn(in[i]);
}
void gen_f16_to_f32_array(const uint16_t* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = gen_f16_to_f32(in[i]);
}
void gen_f32_to_bf16_array(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = gen_f32_to_bf16_rn(in[i]);
}
uint16_t gen_quant_block(const float* w32, uint8_t* out16) {
  return gen_quant_block32(w32, out16);
}

/* ---- threaded matrix generators ---------------------------------------- */
typedef struct {
  uint64_t key;
  int rows, K;
  float sigma;
  uint8_t* q;
  uint16_t* s;
  float* f;
  uint16_t* bf;
  int r0, r1;
} gen_job;

static void* quant_rows(void* arg) {
  gen_job* j = (gen_job*)arg;
  float w[32];
  const int nb = j->K / 32;
  for (int r = j->r0; r < j->r1; ++r) {
    for (int b = 0; b < nb; ++b) {
      uint64_t base = (uint64_t)r * (uint64_t)j->K + (uint64_t)b * 32u;
      for (int i = 0; i < 32; ++i) w[i] = G_MUL(j->sigma, gen_normal(j->key, base + (uint64_t)i));
      j->s[(size_t)r * nb + b] =
          gen_quant_block32(w, j->q + (size_t)r * (j->K / 2) + (size_t)b * 16);
    }
  }
  return 0;
}

static void* f32_rows(void* arg) {
  gen_job* j = (gen_job*)arg;
  for (int r = j->r0; r < j->r1; ++r) {
    for (int k = 0; k < j->K; ++k) {
      uint64_t i = (uint64_t)r * (uint64_t)j->K + (uint64_t)k;
      float v = G_MUL(j->sigma, gen_normal(j->key, i));
      if (j->f) j->f[i] = v;
      if (j->bf) j->bf[i] = gen_f32_to_bf16_rn(v);
    }
  }
  return 0;
}

static void run_rows(void* (*fn)(void*), gen_job proto, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > proto.rows) nthreads = proto.rows > 0 ? proto.rows : 1;
  pthread_t th[256];
  int created[256];
  gen_job jobs[256];
  int per = (proto.rows + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].r0 = t * per;
    jobs[t].r1 = (t + 1) * per < proto.rows ? (t + 1) * per : proto.rows;
    if (jobs[t].r0 >= jobs[t].r1) break;
    /* chunk 0 runs on the calling thread; a chunk whose thread cannot be
     * created also runs there */
    created[t] = (t > 0) && pthread_create(&th[t], 0, fn, &jobs[t]) == 0;
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (!created[t]) fn(&jobs[t]);
  for (int t = 0; t < started; ++t)
    if (created[t]) pthread_join(th[t], 0);
}

/* Quantized matrix [rows][K] of sigma*N(0,1) for stream (seed, wset, layer,
 * tensor, expert): codes q[rows][K/2], scales s[rows][K/32]. K % 32 == 0. */
int gen_quant_matrix(uint64_t seed, uint32_t wset, uint32_t layer,
                     uint32_t tensor, uint32_t expert, int rows, int K,
                     float sigma, uint8_t* q, uint16_t* s, int nthreads) {
  if (rows <= 0 || K <= 0 || K % 32 != 0 || !q || !s) return -1;
  gen_job j;
  memset(&j, 0, sizeof j);
  j.key = gen_key(seed, wset, layer, tensor, expert);
  j.rows = rows;
  j.K = K;
  j.sigma = sigma;
  j.q = q;
  j.s = s;
  run_rows(quant_rows, j, nthreads);
  return 0;
}

/* Dense matrix [rows][K] of sigma*N(0,1): fp32 (out_f32) and/or bf16 bits
 * (out_bf16, round to nearest even); either may be NULL. */
int gen_dense_matrix(uint64_t seed, uint32_t wset, uint32_t layer,
                     uint32_t tensor, uint32_t expert, int rows, int K,
                     float sigma, float* out_f32, uint16_t* out_bf16,
                     int nthreads) {
  if (rows <= 0 || K <= 0 || (!out_f32 && !out_bf16)) return -1;
  gen_job j;
  memset(&j, 0, sizeof j);
  j.key = gen_key(seed, wset, layer, tensor, expert);
  j.rows = rows;
  j.K = K;
  j.sigma = sigma;
  j.f = out_f32;
  j.bf = out_bf16;
  run_rows(f32_rows, j, nthreads);
  return 0;
}

/* Seeded permutation of 0..n-1 (Fisher-Yates driven by the stream). */
int gen_permutation(uint64_t seed, uint32_t wset, uint32_t layer,
                    uint32_t tensor, int n, int32_t* out) {
  if (n <= 0 || !out) return -1;
  uint64_t key = gen_key(seed, wset, layer, tensor, 0);
  for (int i = 0; i < n; ++i) out[i] = i;
  for (int i = n - 1; i > 0; --i) {
    int j = (int)(gen_u64(key, (uint64_t)i) % (uint64_t)(i + 1));
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
  return 0;
}

/* Zipf(s) prior as a logit bias: b_e = -s * ln(rank_e), where rank_e in
 * 1..E is a seeded permutation (softmax of b is proportional to rank^-s). */
int gen_zipf_bias(uint64_t seed, uint32_t wset, uint32_t layer, int E,
                  float s_exp, float* bias) {
  if (E <= 0 || !bias) return -1;
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  if (!perm) return -2;
  gen_permutation(seed, wset, layer, GEN_T_BIAS_PERM, E, perm);
  for (int e = 0; e < E; ++e) {
    float rank = (float)(perm[e] + 1);
    bias[e] = G_MUL(-s_exp, gen_ln(rank));
  }
  free(perm);
  return 0;
}
