/*
 * Seeded synthetic-input generator shared by the host (gen.c) and the GPU
 * (gen_device.cu) builds of this module.  It holds none of the MoE layer's
 * arithmetic: it only draws random numbers and encodes expert weights into
 * the packed 4-bit form the layer consumes.
 *
 * Everything here is written so that the host and device builds produce
 * bit-identical bytes:
 *   - the random stream is integer-only (SplitMix64 output function used as a
 *     counter-based generator: state_n = key + (n+1)*golden_gamma, output =
 *     mix(state_n); Steele, Lea & Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014);
 *   - the normal sampler is the Box-Muller transform evaluated with single
 *     precision +, -, *, /, sqrt only (each correctly rounded in IEEE 754),
 *     with our own series for ln and sin/cos, and with no fused multiply-add:
 *     the host build uses -ffp-contract=off, the device build the _rn
 *     intrinsics (which are never contracted).
 * The series are written from their Taylor / atanh expansions; the sampler
 * needs reproducibility, not last-ulp accuracy (truncation error < 1e-7).
 */
#ifndef MOE_WORKLOAD_GEN_COMMON_H
#define MOE_WORKLOAD_GEN_COMMON_H

#include <stdint.h>

#if defined(__CUDACC__)
#define GEN_FN __host__ __device__ static inline
#else
#define GEN_FN static inline
#endif

#if defined(__CUDA_ARCH__)
#define G_ADD(a, b) __fadd_rn((a), (b))
#define G_SUB(a, b) __fsub_rn((a), (b))
#define G_MUL(a, b) __fmul_rn((a), (b))
#define G_DIV(a, b) __fdiv_rn((a), (b))
#define G_SQRT(a) __fsqrt_rn(a)
#else
#include <math.h>
#define G_ADD(a, b) ((a) + (b))
#define G_SUB(a, b) ((a) - (b))
#define G_MUL(a, b) ((a) * (b))
#define G_DIV(a, b) ((a) / (b))
#define G_SQRT(a) sqrtf(a)
#endif

/* Tensor ids used to derive independent streams. */
enum {
  GEN_T_ROUTER = 1,
  GEN_T_GATE = 2,
  GEN_T_UP = 3,
  GEN_T_DOWN = 4,
  GEN_T_SH_GATE = 5,
  GEN_T_SH_UP = 6,
  GEN_T_SH_DOWN = 7,
  GEN_T_X = 8,
  GEN_T_BIAS_PERM = 9,
  GEN_T_SLOT_PERM = 10,
  GEN_T_DRAFT = 11
};

GEN_FN uint64_t gen_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

/* n-th output of the SplitMix64 sequence started at `key`. */
GEN_FN uint64_t gen_u64(uint64_t key, uint64_t n) {
  return gen_mix64(key + (n + 1ULL) * 0x9e3779b97f4a7c15ULL);
}

/* Stream key for (seed, weight set, layer, tensor, expert). */
GEN_FN uint64_t gen_key(uint64_t seed, uint32_t wset, uint32_t layer,
                        uint32_t tensor, uint32_t expert) {
  uint64_t k = gen_mix64(seed ^ 0x5eed5eed5eed5eedULL);
  k = gen_mix64(k ^ ((uint64_t)wset << 32) ^ (uint64_t)layer);
  k = gen_mix64(k ^ ((uint64_t)tensor << 40) ^ (uint64_t)expert);
  return k;
}

/* Uniform in (0, 1] with 24 random bits: exact in fp32. */
GEN_FN float gen_uniform(uint64_t key, uint64_t n) {
  uint32_t b = (uint32_t)(gen_u64(key, n) >> 40); /* 24 bits */
  return (float)(b + 1u) * (1.0f / 16777216.0f);
}

GEN_FN uint32_t gen_f32_bits(float f) {
  union {
    float f;
    uint32_t u;
  } v;
  v.f = f;
  return v.u;
}
GEN_FN float gen_bits_f32(uint32_t u) {
  union {
    float f;
    uint32_t u;
  } v;
  v.u = u;
  return v.f;
}

/* Natural log of a positive normal u: u = m * 2^e, m in [sqrt(1/2), sqrt(2)),
 * ln m = 2 atanh(t), t = (m-1)/(m+1), atanh(t) = t + t^3/3 + t^5/5 + ... */
GEN_FN float gen_ln(float u) {
  uint32_t b = gen_f32_bits(u);
  int e = (int)((b >> 23) & 0xff) - 127;
  float m = gen_bits_f32((b & 0x007fffffu) | 0x3f800000u); /* [1, 2) */
  if (m > 1.41421356f) {
    m = G_MUL(m, 0.5f);
    e += 1;
  }
  float t = G_DIV(G_SUB(m, 1.0f), G_ADD(m, 1.0f));
  float t2 = G_MUL(t, t);
  float p = G_ADD(G_MUL(t2, 1.0f / 13.0f), 1.0f / 11.0f);
  p = G_ADD(G_MUL(t2, p), 1.0f / 9.0f);
  p = G_ADD(G_MUL(t2, p), 1.0f / 7.0f);
  p = G_ADD(G_MUL(t2, p), 1.0f / 5.0f);
  p = G_ADD(G_MUL(t2, p), 1.0f / 3.0f);
  p = G_ADD(G_MUL(t2, p), 1.0f);
  float lnm = G_MUL(G_MUL(2.0f, t), p);
  return G_ADD(lnm, G_MUL((float)e, 0.693147180559945f));
}

/* cos and sin of 2*pi*f for f in [0, 1). */
GEN_FN void gen_cossin_2pi(float f, float* c, float* s) {
  float f4 = G_MUL(f, 4.0f); /* exact */
  int q = (int)f4;
  if (q > 3) q = 3;
  float r = G_SUB(f4, (float)q);            /* exact, in [0, 1) */
  float ph = G_MUL(r, 1.57079632679490f);   /* [0, pi/2) */
  float p2 = G_MUL(ph, ph);
  /* sin(ph) = ph * (1 - p2/3! + p2^2/5! - ... ), Horner in p2 */
  float sp = 1.0f / 6227020800.0f;
  sp = G_SUB(G_MUL(p2, sp), 1.0f / 39916800.0f);
  sp = G_ADD(G_MUL(p2, sp), 1.0f / 362880.0f);
  sp = G_SUB(G_MUL(p2, sp), 1.0f / 5040.0f);
  sp = G_ADD(G_MUL(p2, sp), 1.0f / 120.0f);
  sp = G_SUB(G_MUL(p2, sp), 1.0f / 6.0f);
  sp = G_ADD(G_MUL(p2, sp), 1.0f);
  float sn = G_MUL(ph, sp);
  /* cos(ph) = 1 - p2/2! + p2^2/4! - ... */
  float cp = -1.0f / 87178291200.0f;
  cp = G_ADD(G_MUL(p2, cp), 1.0f / 479001600.0f);
  cp = G_SUB(G_MUL(p2, cp), 1.0f / 3628800.0f);
  cp = G_ADD(G_MUL(p2, cp), 1.0f / 40320.0f);
  cp = G_SUB(G_MUL(p2, cp), 1.0f / 720.0f);
  cp = G_ADD(G_MUL(p2, cp), 1.0f / 24.0f);
  cp = G_SUB(G_MUL(p2, cp), 0.5f);
  cp = G_ADD(G_MUL(p2, cp), 1.0f);
  float cs = cp;
  switch (q) {
    case 0: *c = cs; *s = sn; break;
    case 1: *c = -sn; *s = cs; break;
    case 2: *c = -cs; *s = -sn; break;
    default: *c = sn; *s = -cs; break;
  }
}

/* Standard normal number `i` of stream `key` (Box-Muller on the pair
 * i/2: uniforms 2*(i/2) and 2*(i/2)+1; even i takes the cosine branch). */
GEN_FN float gen_normal(uint64_t key, uint64_t i) {
  uint64_t p = i >> 1;
  float u1 = gen_uniform(key, 2 * p);
  float u2 = gen_uniform(key, 2 * p + 1) - (1.0f / 16777216.0f); /* [0,1) */
  float r = G_SQRT(G_MUL(-2.0f, gen_ln(u1)));
  float c, s;
  gen_cossin_2pi(u2, &c, &s);
  return (i & 1) ? G_MUL(r, s) : G_MUL(r, c);
}

/* IEEE binary32 -> binary16, round to nearest even (bit manipulation). */
GEN_FN uint16_t gen_f32_to_f16_rn(float f) {
  uint32_t x = gen_f32_bits(f);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7fffffffu;
  if (ax >= 0x7f800000u) { /* inf or nan */
    return (uint16_t)(sign | 0x7c00u | (ax > 0x7f800000u ? 0x200u : 0u));
  }
  if (ax >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u); /* rounds to inf */
  if (ax < 0x38800000u) { /* result is subnormal or zero in binary16 */
    if (ax < 0x33000000u) return (uint16_t)sign; /* |f| < 2^-25 rounds to 0 */
    /* f = m * 2^(e-150) with m the 24-bit significand; in units of the
     * binary16 subnormal step 2^-24 that is m >> (126 - e), 14 <= shift <= 24 */
    uint32_t e = ax >> 23;
    uint32_t m = (ax & 0x007fffffu) | 0x00800000u;
    uint32_t sh = 126u - e;
    uint32_t q = m >> sh;
    uint32_t rem = m & ((1u << sh) - 1u);
    uint32_t half = 1u << (sh - 1u);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q);
  }
  /* normal */
  uint32_t e = (ax >> 23) - 127u + 15u;
  uint32_t m = ax & 0x007fffffu;
  uint32_t q = (e << 10) | (m >> 13);
  uint32_t rem = m & 0x1fffu;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q += 1u; /* may carry to inf */
  return (uint16_t)(sign | q);
}

/* binary16 -> binary32 (exact). */
GEN_FN float gen_f16_to_f32(uint16_t h) {
  uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
  uint32_t e = ((uint32_t)h >> 10) & 0x1fu;
  uint32_t m = (uint32_t)h & 0x3ffu;
  if (e == 0) {
    if (m == 0) return gen_bits_f32(sign);
    /* subnormal: m * 2^-24, exact in fp32 */
    float v = G_MUL((float)m, 1.0f / 16777216.0f);
    return sign ? -v : v;
  }
  if (e == 31) return gen_bits_f32(sign | 0x7f800000u | (m << 13));
  return gen_bits_f32(sign | ((e - 15u + 127u) << 23) | (m << 13));
}

/* IEEE binary32 -> bfloat16, round to nearest even (finite inputs). */
GEN_FN uint16_t gen_f32_to_bf16_rn(float f) {
  uint32_t x = gen_f32_bits(f);
  if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((x >> 16) | 0x40u);
  uint32_t lsb = (x >> 16) & 1u;
  return (uint16_t)((x + 0x7fffu + lsb) >> 16);
}

/* Encode one block of 32 weights as symmetric 4-bit codes with one binary16
 * scale: d = max|w|/7, s = f16_rn(d), q = clamp(round_half_away(w/s), -8, 7),
 * stored as nibble q+8; byte j holds element 2j (low nibble) and 2j+1 (high).
 * A zero block gets s = 0 and all codes 0. */
GEN_FN uint16_t gen_quant_block32(const float* w, uint8_t* out16) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    float a = w[i] < 0.0f ? -w[i] : w[i];
    amax = a > amax ? a : amax;
  }
  float d = G_DIV(amax, 7.0f);
  uint16_t sbits = gen_f32_to_f16_rn(d);
  float s = gen_f16_to_f32(sbits);
  for (int j = 0; j < 16; ++j) {
    int qq[2];
    for (int h = 0; h < 2; ++h) {
      int q = 0;
      if (s != 0.0f) {
        float r = G_DIV(w[2 * j + h], s);
        /* round half away from zero: exact for |r| < 2^22 */
        float ar = r < 0.0f ? -r : r;
        int qi = 9; /* anything >= 8.5 clamps */
        if (ar < 8.5f) {
          float fl = (float)(int)ar;
          float fr = G_SUB(ar, fl);
          qi = (int)fl + (fr >= 0.5f ? 1 : 0);
        }
        q = r < 0.0f ? -qi : qi;
        if (q < -8) q = -8;
        if (q > 7) q = 7;
      }
      qq[h] = q + 8;
    }
    out16[j] = (uint8_t)(qq[0] | (qq[1] << 4));
  }
  return sbits;
}

#endif
