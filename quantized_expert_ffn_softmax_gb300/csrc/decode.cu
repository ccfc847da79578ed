// Decode / MTP-verify path (1..4 tokens): one persistent cooperative kernel
// (one CTA per SM) runs a whole stack of MoE layers.  Per layer:
//
//   phase R  the layer input: x (first layer) or, in stacks, the residual
//            h = bf16(h + bf16(y)) of the previous layer's output y (fp32,
//            reduced in L2); RMS norm -> u; router GEMV (fp32) over this
//            CTA's experts, whose W_r rows were prefetched into shared
//            memory during the previous layer
//   barrier
//   top-k    ranking, not serial selection: every warp ranks its slice of
//            the logits with warp shuffles, the slices' top-k candidates
//            rank each other in shared memory; softmax over the selection;
//            the expert-unit list.  Computed redundantly by every CTA.
//   units    a work unit is (expert unit, 32-row block of its F); CTA c
//            takes units c, c + grid, ...  Per unit: the block's gate/up
//            rows (two 16-row items copied into a 2-deep stage ring by a
//            dedicated copy warp), fused dequant GEMV + SwiGLU -> 32 values
//            of w*h per token; then the block's 32 columns of the down
//            matrix (one 5-D TMA box for library layers, per-thread async
//            copies for the allocation-free entry point) against all H
//            outputs, added into the layer's fp32 output in L2 with
//            reductions
//   barrier
//
// Only the router logits and the layer output cross between CTAs (through
// L2); every weight byte is read from HBM once.  The output's fp32 sums
// arrive in any order, so the last bit may differ between runs.  Packed
// 4-bit codes become fp16 pairs with a
// magic-exponent OR (0x6400 | n = 1024 + n, minus 1032 = n - 8, exact; a
// nibble one position higher goes into 0x5400 = 64.0 instead).  One token:
// products with the fp16 activations are exact and summed within a
// 32-weight block in fp16, then scaled by the block scale and summed in
// fp32.  Two to four tokens: the biased codes and the activations go
// through mma.sync tiles with fp32 accumulation (see mma_16816).
// Activations are rescaled by a per-token power of two before the fp16
// conversion, so their range never overflows fp16.
#include <math.h>

#include <mutex>
#include <stdlib.h>

#include "device_common.cuh"
#include "moe_internal.cuh"
#include "profile.cuh"

namespace moe {
namespace {

using namespace dev;

constexpr int kWarps = kDecodeThreads / 32;  // compute warps; warp kWarps issues the copies

// Barrier of the compute warps only (named barrier 1): the copy warp runs
// its own schedule and never joins it.
__device__ __forceinline__ void cta_sync() { named_bar_sync(1, kDecodeThreads); }

// Orders this thread's generic-proxy global writes before later async-proxy
// (TMA) accesses, and the reverse.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// out[0..3] += v (fp32) with one vector reduction in L2; out 16-byte aligned.
__device__ __forceinline__ void red_add_v4(float* out, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(out), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// Grid barrier on a counter zeroed before the launch: barrier number `n`
// completes when the counter reaches (n + 1) * gridDim.x.  Waits are bounded
// by a %globaltimer deadline; a recorded error makes every later wait return
// at once, so a failing launch still ends in bounded time.
__device__ __forceinline__ void grid_sync(GridBarrier* b, unsigned& n, int* err,
                                          uint64_t timeout_ns, int extra) {
  cta_sync();
  if (threadIdx.x == 0) {
    const unsigned target = (n + 1) * gridDim.x + (unsigned)extra;
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&b->count) : "memory");
    if (ld_acquire_u32(&b->count) < target) {
      const uint64_t t0 = global_timer();
      unsigned spins = 0;
      while (ld_acquire_u32(&b->count) < target) {
        if ((++spins & 15u) == 0) {
          if (ld_relaxed_i32(err) != 0) break;
          if (global_timer() - t0 > timeout_ns) {
            atomicCAS(err, 0, (int)MOE_ERR_TIMEOUT);
            break;
          }
        }
      }
    }
  }
  ++n;
  cta_sync();
}

// Shift that brings amax into [32, 64).
__device__ __forceinline__ int range_shift(float amax) {
  if (!(amax > 0.0f) || !isfinite(amax)) return 0;
  int e = ((__float_as_int(amax) >> 23) & 0xff) - 127;
  int s = e - 5;
  return s < -100 ? -100 : (s > 100 ? 100 : s);
}

// 32 packed 4-bit codes (one 16-byte block) dotted with one token's 32
// activations, held as 4 x (4 fp16 pairs) in the order the codes unpack:
// word q of the block covers elements 8q..8q+7; pair j of word q is
// (element 8q+j, element 8q+j+4).
// Nibbles in bits 0-3 of a half word are ORed into the mantissa of 1024.0
// (0x6400: unit step), nibbles in bits 4-7 into that of 64.0 (0x5400: step
// 1/16, so n * 16 adds n); one shift by 8 brings nibbles 2 and 3 into those
// positions.  Subtracting 1032 or 72 leaves n - 8 exactly.
__device__ __forceinline__ void unpack_codes(uint32_t w, __half2 (&h)[4]) {
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 k72 = __halves2half2(__ushort_as_half(0x5480), __ushort_as_half(0x5480));
  const uint32_t w8 = w >> 8;
  uint32_t v[4];
  v[0] = (w & 0x000F000Fu) | 0x64006400u;   // (1024 + n0, 1024 + n4)
  v[1] = (w & 0x00F000F0u) | 0x54005400u;   // (64 + n1, 64 + n5)
  v[2] = (w8 & 0x000F000Fu) | 0x64006400u;  // (1024 + n2, 1024 + n6)
  v[3] = (w8 & 0x00F000F0u) | 0x54005400u;  // (64 + n3, 64 + n7)
  h[0] = __hsub2(*reinterpret_cast<__half2*>(&v[0]), k1032);
  h[1] = __hsub2(*reinterpret_cast<__half2*>(&v[1]), k72);
  h[2] = __hsub2(*reinterpret_cast<__half2*>(&v[2]), k1032);
  h[3] = __hsub2(*reinterpret_cast<__half2*>(&v[3]), k72);
}

template <int TT>
__device__ __forceinline__ void dot_block(const uint4 w, const uint4 (&act)[TT][4],
                                          float (&out)[TT]) {
  __half2 c[4][4];
  unpack_codes(w.x, c[0]);
  unpack_codes(w.y, c[1]);
  unpack_codes(w.z, c[2]);
  unpack_codes(w.w, c[3]);
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    const __half2* a0 = reinterpret_cast<const __half2*>(&act[t][0]);
    const __half2* a1 = reinterpret_cast<const __half2*>(&act[t][1]);
    const __half2* a2 = reinterpret_cast<const __half2*>(&act[t][2]);
    const __half2* a3 = reinterpret_cast<const __half2*>(&act[t][3]);
    __half2 s0 = __hmul2(c[0][0], a0[0]);
    __half2 s1 = __hmul2(c[2][0], a2[0]);
#pragma unroll
    for (int j = 1; j < 4; ++j) {
      s0 = __hfma2(c[0][j], a0[j], s0);
      s1 = __hfma2(c[2][j], a2[j], s1);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s0 = __hfma2(c[1][j], a1[j], s0);
      s1 = __hfma2(c[3][j], a3[j], s1);
    }
    // each half of s0 + s1 sums 16 products below 64 * 8 in magnitude
    // (activations scaled below 64, codes in [-8, 7]): at most 8192, far
    // inside the fp16 range
    const float2 f0 = __half22float2(__hadd2(s0, s1));
    out[t] = f0.x + f0.y;
  }
}

// Tensor-core form of the same dot products, for more than one token
// (mma.sync m16n8k16, fp16 operands, fp32 accumulation).  In an MMA the 16
// k of lane c (= lane % 4) are those of word c of a code block: the k slots
// 2c, 2c+1 hold pair j of the word and 2c+8, 2c+9 pair j+1 (j = 0 in the
// first MMA of a block, 2 in the second), and operand B holds the same pairs
// of the activations.  The codes go in still biased, 1024 + n (pairs 0, 2)
// or 64 + n (pairs 1, 3): fp16 products are exact in fp32, and the bias,
// the sum of 1032 or 72 times each activation of the block, is taken off
// through the accumulator's initial value.  That costs about ten of the
// accumulator's 24 bits and saves the fp16 subtractions of the unpack.
__device__ __forceinline__ void unpack_biased(uint32_t w, uint32_t (&v)[4]) {
  const uint32_t w8 = w >> 8;
  v[0] = (w & 0x000F000Fu) | 0x64006400u;   // (1024 + n0, 1024 + n4)
  v[1] = (w & 0x00F000F0u) | 0x54005400u;   // (64 + n1, 64 + n5)
  v[2] = (w8 & 0x000F000Fu) | 0x64006400u;  // (1024 + n2, 1024 + n6)
  v[3] = (w8 & 0x00F000F0u) | 0x54005400u;  // (64 + n3, 64 + n7)
}

// d += A B for one m16n8k16 tile.  Lane (g = lane / 4, c = lane % 4) holds
// A rows g and g + 8 at k 2c, 2c+1 (a0, a1) and 2c+8, 2c+9 (a2, a3), B
// column g at k 2c, 2c+1 (b0) and 2c+8, 2c+9 (b1), and D rows g and g + 8
// at columns 2c and 2c+1 (d0, d1 and d2, d3).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Reduce-scatter of N values (power of two, <= 32) across a warp: returns the
// warp sum of value index (lane >> (5 - log2 N)).
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[N], int lane) {
  constexpr int LOGN = (N >= 32) ? 5 : (N >= 16) ? 4 : (N >= 8) ? 3 : (N >= 4) ? 2 : (N >= 2) ? 1 : 0;
#pragma unroll
  for (int s = 0; s < LOGN; ++s) {
    const int half = N >> (s + 1);
    const int k = 16 >> s;
    const bool upper = (lane & k) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, k);
    }
  }
#pragma unroll
  for (int k = 16 >> LOGN; k >= 1; k >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], k);
  return v[0];
}

// Monotonic 32-bit key of a float (larger float -> larger key, > 0); NaN -> 0;
// -0 and +0 get the same key (they compare equal).
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0u;
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of T tokens' logits by the whole CTA, by ranking instead of serial
// selection rounds.  Level 1: thread (warp w, lane) holds the logits
// e = 32w + lane + 256j, j < NPL, of each token and counts, with 32 warp
// shuffles per j, how many logits of its warp beat each of them (larger
// value, or equal value and lower expert id); a logit of warp rank r < k
// becomes candidate w*k + r.  Level 2: each of the 8k candidates of a token
// counts the candidates that beat it (2 or 4 adjacent lanes share one
// candidate, each scanning a quarter or half of the list); rank r < k is the
// r-th selection.
// A candidate is the 64-bit key (order_key(z) << 32) | ~e (0 = empty), so
// candidates compare as plain integers and never tie.
template <int NPL, int TT>
__device__ __forceinline__ void topk_level1(const float* z, int T, int E, int k,
                                            uint64_t (*cand)[kWarps * kMaxTopK]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the tokens' ranks are independent: one pass over the source lanes ranks
  // G tokens at once (G * NPL <= 4 keeps the keys and ranks in registers;
  // tokens past T rank zeros and are dropped)
  constexpr int G = (TT * NPL <= 4) ? TT : ((4 / NPL) < 1 ? 1 : (4 / NPL));
#pragma unroll
  for (int t0 = 0; t0 < TT; t0 += G) {
    if (t0 >= T) break;
    uint32_t key[G][NPL];
    int rank[G][NPL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        const int t = t0 + g, e = 32 * warp + lane + 256 * j;
        key[g][j] = (t < T && e < E) ? order_key(__ldcg(z + (size_t)t * E + e)) : 0u;
        rank[g][j] = 0;
      }
#pragma unroll 8
    for (int src = 0; src < 32; ++src) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int jj = 0; jj < NPL; ++jj) {
          const uint32_t ks = __shfl_sync(0xffffffffu, key[g][jj], src);
#pragma unroll
          for (int j = 0; j < NPL; ++j) {
            // logit (src, jj) has the lower expert id iff jj < j, or jj == j and src < lane
            const bool lower_id = (jj < j) || (jj == j && src < lane);
            rank[g][j] += (ks > key[g][j] || (ks == key[g][j] && lower_id)) ? 1 : 0;
          }
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int t = t0 + g;
      if (t >= T) break;
#pragma unroll
      for (int j = 0; j < NPL; ++j)
        if (rank[g][j] < k) {
          const uint32_t e = (uint32_t)(32 * warp + lane + 256 * j);
          cand[t][warp * k + rank[g][j]] = key[g][j] ? (((uint64_t)key[g][j] << 32) | (uint64_t)(~e)) : 0ull;
        }
    }
  }
}

// Level 2: the kWarps * k candidates of each token rank one another (the
// number of larger keys is the rank; keys are distinct), P lanes per
// candidate, each scanning 128 / P entries of the candidate list padded to
// 128 / P * P entries with zeros (empty).  P = 4 when the list holds at most
// 64 candidates, else 2.  The P lanes of a candidate sit 32 / P lanes apart
// (lane = candidate-in-warp + (32 / P) * part): a warp's 16-byte shared loads
// are served eight lanes at a time, and eight consecutive lanes then read
// one address (a broadcast) instead of P addresses in the same banks, which
// cost P times as long.
template <int P>
__device__ __forceinline__ void rank_candidates(const uint64_t (*cand)[kWarps * kMaxTopK],
                                                uint64_t (*sel_key)[kMaxTopK], int T, int k, int tid) {
  constexpr int ncp = kDecodeThreads / P;  // padded list length: 64 or 128
  constexpr int per = ncp / P;             // entries each lane scans: 16 or 64
  constexpr int CW = 32 / P;               // candidates per warp
  static_assert(ncp <= kWarps * kMaxTopK, "the padded list fits the candidate array");
  const int nc = kWarps * k;
  const int lane = tid & 31;
  const int c = (tid >> 5) * CW + (lane % CW), part = lane / CW;
  for (int t = 0; t < T; ++t) {
    const uint64_t mine = (c < nc) ? cand[t][c] : 0ull;
    int r = 0;
    const ulonglong2* src = reinterpret_cast<const ulonglong2*>(&cand[t][part * per]);
#pragma unroll
    for (int q = 0; q < per / 2; ++q) {
      const ulonglong2 o = src[q];
      r += (part * per + 2 * q < nc && o.x > mine) ? 1 : 0;
      r += (part * per + 2 * q + 1 < nc && o.y > mine) ? 1 : 0;
    }
#pragma unroll
    for (int o = CW; o < 32; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    if (part == 0 && c < nc && r < k && mine != 0ull) sel_key[t][r] = mine;
  }
}

// The same ranking for several tokens at once, when a token has at most 64
// candidates: one thread per (token, candidate), tokens tid / 64; each
// thread counts the larger keys among its token's candidates (every lane of
// a warp reads the same entry: a broadcast).
__device__ __forceinline__ void rank_candidates_tokens(const uint64_t (*cand)[kWarps * kMaxTopK],
                                                       uint64_t (*sel_key)[kMaxTopK], int T, int k,
                                                       int tid) {
  static_assert(kDecodeThreads >= 64 * kMaxDecodeTokens, "a thread per token and candidate");
  const int t = tid >> 6, c = tid & 63;
  const int nc = kWarps * k;
  if (t >= T) return;
  const uint64_t mine = (c < nc) ? cand[t][c] : 0ull;
  int r = 0;
  const ulonglong2* src = reinterpret_cast<const ulonglong2*>(&cand[t][0]);
#pragma unroll
  for (int q = 0; q < 32; ++q) {
    const ulonglong2 o = src[q];
    r += (2 * q < nc && o.x > mine) ? 1 : 0;
    r += (2 * q + 1 < nc && o.y > mine) ? 1 : 0;
  }
  if (c < nc && r < k && mine != 0ull) sel_key[t][r] = mine;
}

}  // namespace

// Shared-memory carve of the decode kernel (mirrored on the host).
struct DecodeSmem {
  size_t mbar, misc, slots, xb, hres, xp, wr, gbuf, dst, corrx, red, total;
  size_t g_stage;
  int nmy;
  // gu: gate/up items by the tensor-core path (more than one token), which
  // adds the activations' code-bias sums and the items' cross-warp sums
  __host__ __device__ static DecodeSmem make(int H, int E, int TT, int grid, int g_stages, int gu) {
    DecodeSmem s;
    const int C = H / 32;
    s.nmy = (E + 1 + grid - 1) / grid;  // router rows per CTA, with room for the gate row
    s.g_stage = (size_t)16 * H + (size_t)64 * C;  // gate+up rows (2 x 16 x H/2) + scales
    size_t o = 0;
    s.mbar = o;
    o += 128;
    s.misc = o;
    o += 12288;
    s.slots = o;
    o += ((size_t)E * 4 + 15) & ~(size_t)15;
    s.xb = o;
    o += (size_t)TT * H * 2;
    s.hres = o;
    o += (size_t)TT * H * 2;
    s.wr = o;
    o += (size_t)s.nmy * H * 4;
    o = (o + 127) & ~(size_t)127;
    s.xp = o;  // x pair planes
    s.gbuf = (o + (size_t)TT * H * 2 + 127) & ~(size_t)127;
    o = s.gbuf + (size_t)g_stages * s.g_stage;
    o = (o + 127) & ~(size_t)127;
    s.dst = o;  // down block of a work unit: 16 code bytes + a 4-byte scale pair per output row
    o += (size_t)H * 20;
    o = (o + 127) & ~(size_t)127;
    s.corrx = s.red = o;
    if (gu) {
      o += (size_t)C * 16;  // [C][4] fp32: per block and token
      o = (o + 127) & ~(size_t)127;
      s.red = o;            // [2][kWarps][32 rows][TT] fp32, by item parity
      o += (size_t)2 * kWarps * 32 * TT * 4;
    }
    s.total = (o + 127) & ~(size_t)127;
    return s;
  }
};

struct DecodeMisc {
  int x_shift[4];
  int n_routed;
  int n_units;
  int pad0[2];
  int sel_id[kMaxDecodeTokens][kMaxTopK];
  float sel_w[kMaxDecodeTokens][kMaxTopK];
  uint64_t cand[kMaxDecodeTokens][kWarps * kMaxTopK];  // top-k level-1 candidates, w*k + r
  uint64_t sel_key[kMaxDecodeTokens][kMaxTopK];       // top-k level-2 result
  int unit_expert[kMaxUnits];
  int unit_slot[kMaxUnits];
  float unit_w[kMaxUnits][kMaxDecodeTokens];
  unsigned bitmap[kMaxExperts / 32];
  int prefix[kMaxExperts / 32 + 1];
  float red_ss[kWarps][4];
  float red_mx[kWarps][4];
  float red_z[kWarps][4];
  float hst[2][16][4];  // w*h of a gate/up item's 16 rows (double-buffered by item)
  uint4 actD[kMaxDecodeTokens][4];  // w*h of a work unit's 32 rows as fp16 pair planes
  int dsh[kMaxDecodeTokens];        // their power-of-two shifts
  float corrd[kMaxDecodeTokens];    // their code-bias sums (tensor path, more than one token)
  // expert cache of a partially resident layer
  int n_miss;
  int miss_unit[kMaxUnits];         // routed units whose expert has no slot
  unsigned inuse[kMaxExperts / 32];  // slots of this call's resident units
  unsigned long long red_key[kWarps];
};
static_assert(sizeof(DecodeMisc) <= 12288, "misc region too small");

// mbarrier slots: gate/up stages full (G) and empty (E), router rows (R),
// slot table (S), down stage full (D) and empty (DE)
enum { kBarG0 = 0, kBarG1 = 1, kBarE0 = 2, kBarE1 = 3, kBarR = 4, kBarS = 5, kBarD = 6, kBarDE = 7,
       kNumBars = 8 };
// named barriers between the compute warps and the copy warp: the router
// rows buffer is free (compute warps arrive), the unit list is ready (all sync)
enum { kNbRowsFree = 3, kNbUnits = 2 };

// Rows per box of the down-code tensor map: the largest multiple of 32 that
// is at most 256 and divides H/4 (H/4 is a multiple of 32).
__host__ __device__ __forceinline__ int down_qbox(int H) {
  const int hq = H / 4;
  for (int q = 256; q >= 32; q -= 32)
    if (hq % q == 0) return q;
  return 32;
}

// 4-byte async copy global -> shared (the .ca form; .cg takes 16 bytes only)
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Expert-cache misses of one layer, from the host tier into their slots.
// The bytes of all misses form one index space of 16-byte vectors (miss,
// tensor, offset; tensors in the order gate codes, gate scales, up codes, up
// scales, down codes, down scales, block-major down scales, each a multiple
// of 16 bytes); this CTA copies its 1/grid slice with four loads in flight
// per thread, so the layer's misses cost about one host round trip per four
// vectors of a thread, not one per tensor and miss.
__device__ __forceinline__ void copy_misses(const CacheDev* cd, const LayerDev& W, int F, int H,
                                         int n_miss, const int* miss_unit, const int* unit_expert,
                                         const int* unit_slot, int tid) {
  const size_t gqe = (size_t)F * (H / 2), gse = (size_t)F * (H / 32) * 2;
  const size_t dqe = (size_t)H * (F / 2), dse = (size_t)H * (F / 32) * 2;
  const size_t per16 = (2 * (gqe + gse) + dqe + 2 * dse) / 16;  // vectors per expert
  const size_t nvec = per16 * (size_t)n_miss;
  const size_t lo = nvec * blockIdx.x / gridDim.x, hi = nvec * (blockIdx.x + 1) / gridDim.x;
  auto locate = [&](size_t g, bool dst) -> char* {
    const size_t i = g / per16;
    size_t o = (g - i * per16) * 16;
    const int u = miss_unit[i];
    const size_t row = dst ? (size_t)unit_slot[u] : (size_t)__ldg(cd->host_row + unit_expert[u]);
    const char* base;
    size_t n;
    if (o < gqe) {
      base = dst ? (const char*)W.gate_q : (const char*)cd->gate_q, n = gqe;
    } else if ((o -= gqe) < gse) {
      base = dst ? (const char*)W.gate_s : (const char*)cd->gate_s, n = gse;
    } else if ((o -= gse) < gqe) {
      base = dst ? (const char*)W.up_q : (const char*)cd->up_q, n = gqe;
    } else if ((o -= gqe) < gse) {
      base = dst ? (const char*)W.up_s : (const char*)cd->up_s, n = gse;
    } else if ((o -= gse) < dqe) {
      base = dst ? (const char*)W.down_q : (const char*)cd->down_q, n = dqe;
    } else if ((o -= dqe) < dse) {
      base = dst ? (const char*)W.down_s : (const char*)cd->down_s, n = dse;
    } else {
      o -= dse;
      base = dst ? (const char*)W.down_sb : (const char*)cd->down_sb, n = dse;
    }
    return const_cast<char*>(base) + row * n + o;
  };
  constexpr int kInFlight = 4;
  for (size_t g0 = lo + tid; g0 < hi; g0 += (size_t)kInFlight * kDecodeThreads) {
    uint4 val[kInFlight];
#pragma unroll
    for (int q = 0; q < kInFlight; ++q) {
      const size_t g = g0 + (size_t)q * kDecodeThreads;
      if (g < hi) val[q] = *reinterpret_cast<const uint4*>(locate(g, false));
    }
#pragma unroll
    for (int q = 0; q < kInFlight; ++q) {
      const size_t g = g0 + (size_t)q * kDecodeThreads;
      if (g < hi) *reinterpret_cast<uint4*>(locate(g, true)) = val[q];
    }
  }
}

// kVar: some layer of the launch uses a routing variant (routing_flags != 0);
// the default instantiation carries none of their code.
template <int TT, bool kVar>
__global__ void __launch_bounds__(kDecodeBlock, 1)
    moe_decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = p.H, E = p.E, k = p.k, F = p.F, Fs = p.Fs, T = p.T;
  const int C = H / 32;
  const int CF = F / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grid = gridDim.x;
  const DecodeSmem L = DecodeSmem::make(H, E, TT, grid, p.g_stages, p.gu_mma);
  const int NG = p.g_stages;  // 1 or 2
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L.mbar);
  DecodeMisc& M = *reinterpret_cast<DecodeMisc*>(smem + L.misc);
  int* slots = reinterpret_cast<int*>(smem + L.slots);
  uint16_t* xb = reinterpret_cast<uint16_t*>(smem + L.xb);      // layer input (u)
  uint16_t* hres = reinterpret_cast<uint16_t*>(smem + L.hres);  // residual stream (stacks)
  uint4* xp = reinterpret_cast<uint4*>(smem + L.xp);
  float* wr = reinterpret_cast<float*>(smem + L.wr);
  unsigned char* gbuf = smem + L.gbuf;
  unsigned char* dst_s = smem + L.dst;
  float* corrx = reinterpret_cast<float*>(smem + L.corrx);  // tensor path: [C][4]
  float* gred = reinterpret_cast<float*>(smem + L.red);     // tensor path: item sums
  // gate/up items by the tensor cores: more than one token, hidden % 256 == 0
  const bool gu_mma = TT > 1 && p.gu_mma != 0;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(&mbar[i], (i == kBarE0 || i == kBarE1 || i == kBarDE) ? kWarps : 1);
    fence_mbar_init();
  }
  __syncthreads();  // the only barrier of all kDecodeBlock threads
  const uint64_t tmo = p.timeout_ns;
  const bool stack = (p.mode == kModeStack);
  // Router rows of this CTA in layer l: e = blockIdx.x + j * grid, j < rows;
  // with a gated shared expert, row E is the gate vector (its logit g . u
  // goes to p.gz instead of the logits).
  const int rows_e = ((int)blockIdx.x < E) ? (E - (int)blockIdx.x + grid - 1) / grid : 0;
  auto router_rows = [&](int l) {
    if constexpr (!kVar) {
      return rows_e;
    } else {
      const int Er = E + ((p.routing_flags[l] & MOE_ROUTING_SHARED_GATE) ? 1 : 0);
      return ((int)blockIdx.x < Er) ? (Er - (int)blockIdx.x + grid - 1) / grid : 0;
    }
  };
  // The slot table of layer l goes to shared memory by one bulk copy when its
  // size and alignment allow; otherwise the unit list reads it from global.
  auto slots_bulk_of = [&](int l) {
    return (E % 4) == 0 && (reinterpret_cast<uintptr_t>(p.layers[l].slot_of) & 15u) == 0;
  };
  // Work units: a unit is (expert unit, 32-row block of its F); CTA c takes
  // units c, c + grid, ...; each has two 16-row gate/up items.
  const int ipu = F / 16;  // gate/up items per routed unit
  const int bpu = F / 32;  // blocks per routed unit
  const int Hq = H / 4;
  auto my_units = [&](int n_routed) {
    const int n_wu = n_routed * bpu + Fs / 32;
    return ((int)blockIdx.x < n_wu) ? (n_wu - (int)blockIdx.x + grid - 1) / grid : 0;
  };
  auto item_of = [&](int q) { return 2 * ((int)blockIdx.x + (q >> 1) * grid) + (q & 1); };
  // unit and block of this CTA's j-th work unit
  auto wu_of = [&](int j, int n_routed, int& u, int& b) {
    const int w = blockIdx.x + j * grid;
    if (w < n_routed * bpu) {
      u = w / bpu;
      b = w - u * bpu;
    } else {
      u = n_routed;
      b = w - n_routed * bpu;
    }
  };

  // ------------------------------------------------ the copy warp
  // One warp issues every bulk and tensor copy and the compute warps only
  // wait on the mbarriers: per layer, the next layer's router rows once this
  // CTA's router product has read the buffer, then (after the unit list)
  // the first gate/up items, the first down block and the next layer's slot
  // table, and refills as the compute warps release stages.  The warp stays
  // converged; each group of copies is issued by one elected lane
  // (elect.sync): copies issued from lane-divergent code are taken one lane
  // at a time, each at a multiple of the cost.
  if (warp == kWarps) {
    auto issue_rows = [&](int l) {  // all lanes
      const LayerDev& W = p.layers[l];
      const int rows = router_rows(l);
      if (rows && elect_one()) {
        mbar_expect_tx(&mbar[kBarR], (uint32_t)rows * H * 4u);
        for (int j = 0; j < rows; ++j) {
          const int e = blockIdx.x + j * grid;
          bulk_g2s(wr + (size_t)j * H, (!kVar || e < E) ? W.router_w + (size_t)e * H : p.sh_gate_w[l],
                   H * 4u, &mbar[kBarR]);
        }
      }
      __syncwarp();
    };
    auto issue_slots = [&](int l) {  // all lanes
      if (slots_bulk_of(l) && elect_one()) {
        mbar_expect_tx(&mbar[kBarS], (uint32_t)E * 4u);
        bulk_g2s(slots, p.layers[l].slot_of, (uint32_t)E * 4u, &mbar[kBarS]);
      }
      __syncwarp();
    };
    // gate/up item q into stage q % NG: one elected lane arms the stage and
    // issues its four copies
    auto issue_g = [&](int l, int q, int n_routed) {
      const LayerDev& W = p.layers[l];
      const int it = item_of(q);
      const uint8_t* gq;
      const uint16_t* gs;
      const uint8_t* uq;
      const uint16_t* us;
      int row0;  // the item's first row in its tensors
      if (it < n_routed * ipu) {
        const int u = it / ipu;
        const int f0 = (it - u * ipu) * 16;
        const size_t slot = (size_t)M.unit_slot[u];
        row0 = (int)slot * F + f0;
        gq = W.gate_q + (slot * F + f0) * (H / 2);
        uq = W.up_q + (slot * F + f0) * (H / 2);
        gs = W.gate_s + (slot * F + f0) * C;
        us = W.up_s + (slot * F + f0) * C;
      } else {
        const int f0 = (it - n_routed * ipu) * 16;
        row0 = f0;
        gq = W.sh_gate_q + (size_t)f0 * (H / 2);
        uq = W.sh_up_q + (size_t)f0 * (H / 2);
        gs = W.sh_gate_s + (size_t)f0 * C;
        us = W.sh_up_s + (size_t)f0 * C;
      }
      unsigned char* st = gbuf + (size_t)(q % NG) * L.g_stage;
      uint64_t* bar = &mbar[kBarG0 + (q % NG)];
      if (elect_one()) {
        mbar_expect_tx(bar, (uint32_t)L.g_stage);
        if (gu_mma) {
          // the same bytes, block-major: codes [C][16 rows][16 B], scales
          // [C/8][16 rows][8] (the tensor path's conflict-free layout)
          const CUtensorMap* tm = W.tm_gu + (it < n_routed * ipu ? 0 : 2);
          tma_load_3d(st, tm, 0, row0, 0, bar);
          tma_load_3d(st + 16 * (H / 2), tm + 1, 0, row0, 0, bar);
          tma_load_3d(st + 16 * H, tm + 4, 0, row0, 0, bar);
          tma_load_3d(st + 16 * H + 32 * C, tm + 5, 0, row0, 0, bar);
        } else {
          bulk_g2s(st, gq, 16u * (H / 2), bar);
          bulk_g2s(st + 16 * (H / 2), uq, 16u * (H / 2), bar);
          bulk_g2s(st + 16 * H, gs, 16u * C * 2u, bar);
          bulk_g2s(st + 16 * H + 32 * C, us, 16u * C * 2u, bar);
        }
      }
      __syncwarp();
    };
    // Down block of work unit j: codes of every output row, row r at
    // position (r % 4) * H/4 + r / 4 (one 5-D TMA box), and the block's H scales
    // from the block-major copy (one bulk copy); one elected lane.
    auto issue_d = [&](int l, int j, int n_routed) {
      const LayerDev& W = p.layers[l];
      int u, b;
      wu_of(j, n_routed, u, b);
      const bool routed = u < n_routed;
      const size_t slot = routed ? (size_t)M.unit_slot[u] : 0;
      const CUtensorMap* tm = routed ? &p.tm_down[l] : &p.tm_sh_down[l];
      if (elect_one()) {
        mbar_expect_tx(&mbar[kBarD], (uint32_t)H * 18u);
        tma_load_5d(dst_s, tm, 16 * b, 0, 0, 0, (int)slot, &mbar[kBarD]);
        const uint16_t* sb = routed ? W.down_sb + (slot * CF + b) * H : W.sh_down_sb + (size_t)b * H;
        bulk_g2s(dst_s + (size_t)H * 16, sb, (uint32_t)H * 2u, &mbar[kBarD]);
      }
      __syncwarp();
    };
    // waits by lane 0, result shared with the warp (lanes stay converged)
    auto wait0 = [&](uint64_t* bar, uint32_t parity) {
      int r = 1;
      if (lane == 0) r = mbar_wait(bar, parity, p.err, tmo) ? 1 : 0;
      return __shfl_sync(0xffffffffu, r, 0) != 0;
    };
    issue_slots(0);
    issue_rows(0);
    // stage releases seen per gate/up stage (phase parity), as two scalars:
    // an array indexed by the stage would live in local memory
    uint32_t e_done0 = 0u, e_done1 = 0u, d_done = 0u;
    bool ok = true;  // false after a failed wait: keep the barrier schedule, issue nothing
    for (int l = 0; l < p.n_layers; ++l) {
      named_bar_sync(kNbRowsFree, kDecodeBlock);
      if (ok && l + 1 < p.n_layers && p.mode != kModeRoute) issue_rows(l + 1);
      named_bar_sync(kNbUnits, kDecodeBlock);
      if (p.mode == kModeRoute) continue;
      fence_proxy_async_global();  // slots just filled by generic stores (expert-cache misses)
      const int n_routed = M.n_routed;
      const int my_wu = my_units(n_routed), n_items = 2 * my_wu;
      if (ok) {
        for (int q = 0; q < NG && q < n_items; ++q) issue_g(l, q, n_routed);
        if (p.down_tma && my_wu > 0) issue_d(l, 0, n_routed);
        if (l + 1 < p.n_layers) issue_slots(l + 1);
      }
      for (int q = 0; q < n_items; ++q) {
        const int sg = q % NG;
        if (q + NG < n_items) {
          if (ok) ok = wait0(&mbar[kBarE0 + sg], (sg ? e_done1 : e_done0) & 1u);
          if (ok) issue_g(l, q + NG, n_routed);
        }
        if (sg) ++e_done1;
        else ++e_done0;
        if (p.down_tma && (q & 1)) {
          const int j = q >> 1;
          if (j + 1 < my_wu) {
            if (ok) ok = wait0(&mbar[kBarDE], d_done & 1u);
            if (ok) issue_d(l, j + 1, n_routed);
          }
          ++d_done;
        }
      }
    }
    return;
  }

  // ------------------------------------------------ the compute warps
  // items consumed per gate/up stage (phase parity), as two scalars: an
  // array indexed by the stage would live in local memory
  uint32_t gcount0 = 0u, gcount1 = 0u;
  uint32_t ph_r = 0u, ph_s = 0u, ph_d = 0u;  // router rows, slot table, down stage fills waited for
  unsigned nbar = 0;
  // the first layer reduces into accumulator 0: zero it here (the layer's
  // first grid barrier orders this before any reduction; the kernel zeroes
  // the other accumulator for each next layer)
  for (int i = blockIdx.x * kDecodeThreads + tid; i < TT * H; i += grid * kDecodeThreads) p.yacc[i] = 0.0f;

  for (int l = 0; l < p.n_layers; ++l) {
    const LayerDev& W = p.layers[l];
    // slots of this layer's expert table (fewer than E when partially resident)
    const int S_l = W.cache ? __ldg(&W.cache->n_slots) : E;
    // the previous layer's output, reduced in L2 (layers after the first)
    const float* yprev = p.yacc + (size_t)((l + 1) & 1) * kMaxDecodeTokens * H;

    // ------------------------------------------------ phase R: stage x, router
    // pass 1: stage x (8 bf16 per thread and step) and take its sum of
    // squares (stacks) and max |x| from the registers
    uint16_t* stage_dst = stack ? hres : xb;
    {
      float ss[TT], mx[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) ss[t] = mx[t] = 0.0f;
      // steps in batches of TT, each batch's global loads issued before any
      // of them is used: one L2 round trip per batch rather than per step
      const int NI1 = TT * (H / 8);
      for (int i0 = tid; i0 < NI1; i0 += TT * kDecodeThreads) {
        uint4 xin[TT], hv[TT];
        float4 ya[TT], yb[TT];
#pragma unroll
        for (int k = 0; k < TT; ++k) {
          const int i = i0 + k * kDecodeThreads, t = i / (H / 8);
          xin[k] = hv[k] = make_uint4(0, 0, 0, 0);
          ya[k] = yb[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (i < NI1 && t < T) {
            const int g8 = i - t * (H / 8);
            if (l == 0) {
              xin[k] = __ldcg(reinterpret_cast<const uint4*>(p.x_in + (size_t)t * H) + g8);
            } else {
              hv[k] = reinterpret_cast<const uint4*>(hres)[i];
              ya[k] = __ldcg(reinterpret_cast<const float4*>(yprev + (size_t)t * H) + 2 * g8);
              yb[k] = __ldcg(reinterpret_cast<const float4*>(yprev + (size_t)t * H) + 2 * g8 + 1);
            }
          }
        }
#pragma unroll
        for (int k = 0; k < TT; ++k) {
          const int i = i0 + k * kDecodeThreads, t = i / (H / 8);
          if (i >= NI1) break;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (t < T) {
            const int g8 = i - t * (H / 8);
            if (l == 0) {
              v = xin[k];
            } else {
              // residual: h_l = bf16(h_{l-1} + bf16(y_{l-1})); h_{l-1} is still
              // staged here (stacks only: a single layer has no layer 1)
              const float yy[8] = {ya[k].x, ya[k].y, ya[k].z, ya[k].w, yb[k].x, yb[k].y, yb[k].z, yb[k].w};
              const uint32_t hw[4] = {hv[k].x, hv[k].y, hv[k].z, hv[k].w};
              uint32_t o[4], yo[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const __nv_bfloat16 ylo = __float2bfloat16_rn(yy[2 * q]);
                const __nv_bfloat16 yhi = __float2bfloat16_rn(yy[2 * q + 1]);
                const float lo = __uint_as_float(hw[q] << 16) + __bfloat162float(ylo);
                const float hi = __uint_as_float(hw[q] & 0xffff0000u) + __bfloat162float(yhi);
                o[q] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
                       ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
                yo[q] = (uint32_t)__bfloat16_as_ushort(ylo) | ((uint32_t)__bfloat16_as_ushort(yhi) << 16);
              }
              v = make_uint4(o[0], o[1], o[2], o[3]);
              if (blockIdx.x == 0 && p.h_trace)
                reinterpret_cast<uint4*>(p.h_trace + ((size_t)(l - 1) * T + t) * H)[g8] = v;
              if (blockIdx.x == 0 && p.y_trace)
                reinterpret_cast<uint4*>(p.y_trace + ((size_t)(l - 1) * T + t) * H)[g8] =
                    make_uint4(yo[0], yo[1], yo[2], yo[3]);
            }
          }
          reinterpret_cast<uint4*>(stage_dst)[i] = v;
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          float a = 0.0f, m = 0.0f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = __uint_as_float(w[q] << 16), hi = __uint_as_float(w[q] & 0xffff0000u);
            a = fmaf(lo, lo, fmaf(hi, hi, a));
            m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
          }
#pragma unroll
          for (int tt = 0; tt < TT; ++tt)
            if (tt == t) {
              ss[tt] += a;
              mx[tt] = fmaxf(mx[tt], m);
            }
        }
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float a = warp_sum(ss[t]), b = warp_max(mx[t]);
        if (lane == 0) {
          M.red_ss[warp][t] = a;
          M.red_mx[warp][t] = b;
        }
      }
      cta_sync();
      float inv[TT], sc[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        float a = 0.0f, b = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          a += M.red_ss[w][t];
          b = fmaxf(b, M.red_mx[w][t]);
        }
        // pre-norm: u = bf16(h / sqrt(mean(h^2) + eps)), unit gain
        inv[t] = stack ? rsqrtf(a / (float)H + 1e-6f) : 1.0f;
        // max |u| <= max |h| * inv, up to one bf16 rounding
        const int s = range_shift(b * inv[t] * 1.0079f);
        sc[t] = pow2f(-s);
        if (tid == 0) M.x_shift[t] = s;
      }
      // pass 2, one 8-group (32c + 8q .. +7) per step: u (stacks) and the
      // fp16 pair planes xp[(t*4 + q)*C + c] = pairs (x[32c+8q+j], x[32c+8q+j+4])
      const int NI = TT * (H / 8);
      for (int i0 = tid; i0 < NI; i0 += kDecodeThreads) {
        // within a full aligned block of 32 steps, lane L takes step
        // 4 (L % 8) + ((L % 8) / 2 + L / 8) % 4 of the block: every quarter
        // warp's 16-byte accesses of stage_dst / xb (at i) and of the pair
        // planes (at g / 4) then fall in eight different bank groups
        const int L = i0 & 31, base = i0 & ~31;
        const int i = (base + 32 <= NI) ? base + 4 * (L & 7) + ((((L & 7) >> 1) + (L >> 3)) & 3) : i0;
        const int t = i / (H / 8), g = i - t * (H / 8);
        float inv_t = 1.0f, sc_t = 1.0f;
#pragma unroll
        for (int tt = 0; tt < TT; ++tt)
          if (tt == t) {
            inv_t = inv[tt];
            sc_t = sc[tt];
          }
        const uint4 v = reinterpret_cast<const uint4*>(stage_dst)[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float e[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          e[2 * q] = __uint_as_float(w[q] << 16);
          e[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
        }
        if (stack) {
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __nv_bfloat16 lo = __float2bfloat16_rn(e[2 * q] * inv_t);
            const __nv_bfloat16 hi = __float2bfloat16_rn(e[2 * q + 1] * inv_t);
            e[2 * q] = __bfloat162float(lo);
            e[2 * q + 1] = __bfloat162float(hi);
            o[q] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
          }
          const uint4 u = make_uint4(o[0], o[1], o[2], o[3]);
          reinterpret_cast<uint4*>(xb)[i] = u;
          if (blockIdx.x == 0 && p.in_trace && t < T)
            reinterpret_cast<uint4*>(p.in_trace + ((size_t)l * T + t) * H)[g] = u;
        }
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          __half2 hh = __floats2half2_rn(e[j] * sc_t, e[j + 4] * sc_t);
          out[j] = *reinterpret_cast<uint32_t*>(&hh);
        }
        if (gu_mma) {
          // tensor path: planes [t][block][word] (this step's index), and
          // per block and token the bias sum of the unpacked codes, 1032 on
          // pairs 0, 2 and 72 on pairs 1, 3 of every word; the block's four
          // words are in lanes L, L^8, L^16, L^24 (full 32-step groups here)
          xp[i] = make_uint4(out[0], out[1], out[2], out[3]);
          float cbs = 0.0f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&out[j]));
            cbs += ((j & 1) ? 72.0f : 1032.0f) * (f.x + f.y);
          }
          cbs += __shfl_xor_sync(0xffffffffu, cbs, 8);
          cbs += __shfl_xor_sync(0xffffffffu, cbs, 16);
          if (L < 8) corrx[(g >> 2) * 4 + t] = cbs;
        } else {
          xp[(t * 4 + (g & 3)) * C + (g >> 2)] = make_uint4(out[0], out[1], out[2], out[3]);
        }
      }
      cta_sync();
    }
    // router: this CTA's expert rows e = blockIdx + j*grid (W_r rows staged
    // in shared memory by the copy warp); row j is split over the warps w
    // with w % nr == j, each summing one slice of H; the slices meet in
    // shared memory
    const int my_rows = router_rows(l);
    // this thread's router bias (read before the row wait, off the critical path)
    const float bias_mine =
        (tid < min(my_rows, kWarps) * T && (!kVar || (int)blockIdx.x + (tid / T) * grid < E))
            ? __ldg(W.router_b + blockIdx.x + (tid / T) * grid) : 0.0f;
    if (my_rows > 0) {
      mbar_wait(&mbar[kBarR], ph_r, p.err, tmo);
      ph_r ^= 1u;
    }
    for (int j0 = 0; j0 < my_rows; j0 += kWarps) {  // batches of at most kWarps rows
      const int nr = min(kWarps, my_rows - j0);
      const int j = warp % nr, part = warp / nr;
      const int nparts = (kWarps - j + nr - 1) / nr;
      const int n4 = H / 4, chunk = (n4 + nparts - 1) / nparts;
      const int i0 = part * chunk, i1 = min(n4, i0 + chunk);
      const float4* wrow = reinterpret_cast<const float4*>(wr + (size_t)(j0 + j) * H);
      float acc[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) acc[t] = 0.0f;
      for (int idx = i0 + lane; idx < i1; idx += 32) {
        const float4 wv = wrow[idx];
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const uint2 xv = *reinterpret_cast<const uint2*>(xb + t * H + 4 * idx);
          acc[t] = fmaf(wv.x, __uint_as_float(xv.x << 16), acc[t]);
          acc[t] = fmaf(wv.y, __uint_as_float(xv.x & 0xffff0000u), acc[t]);
          acc[t] = fmaf(wv.z, __uint_as_float(xv.y << 16), acc[t]);
          acc[t] = fmaf(wv.w, __uint_as_float(xv.y & 0xffff0000u), acc[t]);
        }
      }
      // this thread is done reading the rows (generic proxy), which the copy
      // warp refills by bulk copies once the batch is summed
      fence_proxy_async_smem();
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float s = warp_sum(acc[t]);
        if (lane == 0) M.red_z[warp][t] = s;
      }
      cta_sync();
      const bool last_batch = j0 + kWarps >= my_rows;
      if (last_batch) named_bar_arrive(kNbRowsFree, kDecodeBlock);  // the copy warp may refill the rows buffer
      if (tid < nr * T) {
        const int jr = tid / T, t = tid - (tid / T) * T;
        float z = 0.0f;
        for (int w = jr; w < kWarps; w += nr) z += M.red_z[w][t];
        const int e = blockIdx.x + (j0 + jr) * grid;
        if (!kVar || e < E)
          p.z[(size_t)t * E + e] = z + (j0 == 0 ? bias_mine : __ldg(W.router_b + e));
        else
          p.gz[t] = z;  // the shared-expert gate logit
      }
      if (!last_batch) cta_sync();  // red_z is reused by the next batch
    }
    if (my_rows <= 0) named_bar_arrive(kNbRowsFree, kDecodeBlock);
    grid_sync(p.bar, nbar, p.err, tmo, p.debug_extra_arrivals);

    // ------------------------------------------------ top-k + softmax + units
    // (every CTA computes it redundantly from the logits in L2)
    if (tid < kMaxDecodeTokens * kMaxTopK) (&M.sel_key[0][0])[tid] = 0ull;
    if (E <= 256) topk_level1<1, TT>(p.z, T, E, k, M.cand);
    else if (E <= 512) topk_level1<2, TT>(p.z, T, E, k, M.cand);
    else topk_level1<4, TT>(p.z, T, E, k, M.cand);
    cta_sync();
    if (TT > 1 && kWarps * k <= 64) rank_candidates_tokens(M.cand, M.sel_key, T, k, tid);
    else if (kWarps * k <= 64) rank_candidates<4>(M.cand, M.sel_key, T, k, tid);
    else rank_candidates<2>(M.cand, M.sel_key, T, k, tid);
    cta_sync();
    // the slot table of this layer (bulk-copied during the previous layer)
    const bool slots_bulk = slots_bulk_of(l);
    if (slots_bulk) {
      mbar_wait(&mbar[kBarS], ph_s, p.err, tmo);
      ph_s ^= 1u;
    }
    auto slot_lookup = [&](int e) { return slots_bulk ? slots[e] : __ldg(W.slot_of + e); };
    // a partially resident layer's table holds -1 for experts without a slot
    const bool partial = W.cache != nullptr && p.mode != kModeRoute;
    auto slot_checked = [&](int e) {
      int s = slot_lookup(e);
      if (s >= S_l || (s < 0 && !partial)) {
        atomicCAS(p.err, 0, (int)MOE_ERR_BOUNDS);
        s = 0;
      }
      return s;
    };
    if (warp < T) {
      const uint64_t sk = (lane < k) ? M.sel_key[warp][lane] : 0ull;
      uint32_t ok2 = (uint32_t)(sk >> 32);
      int oi2 = (sk != 0ull) ? (int)(~(uint32_t)sk) : -1;
      const bool bad = (lane < k) && (ok2 == 0u || oi2 < 0 || oi2 >= E);
      if (__any_sync(0xffffffffu, bad)) {  // only reachable with non-finite logits
        if (lane == 0) atomicCAS(p.err, 0, (int)MOE_ERR_BOUNDS);
        if (lane < k) {
          oi2 = lane;
          ok2 = 0x80000000u;
        }
      }
      const float zv = key_value(ok2);
      float ex, den;
      if constexpr (kVar) {
        // the weights' logits: the selection logit, or without the bias when
        // the bias only selects
        const int rf = p.routing_flags[l];
        const bool sel_only = (rf & MOE_ROUTING_BIAS_SELECT_ONLY) != 0;
        const float base = (sel_only && lane < k) ? zv - __ldg(W.router_b + oi2) : zv;
        float m;
        if (rf & MOE_ROUTING_NO_RENORM) {
          // softmax over all E experts, taken at the selected ones
          const float* zt = p.z + (size_t)warp * E;
          m = -INFINITY;
          for (int e = lane; e < E; e += 32)
            m = fmaxf(m, __ldcg(zt + e) - (sel_only ? __ldg(W.router_b + e) : 0.0f));
          m = warp_max(m);
          float acc = 0.0f;
          for (int e = lane; e < E; e += 32)
            acc += __expf(__ldcg(zt + e) - (sel_only ? __ldg(W.router_b + e) : 0.0f) - m);
          den = warp_sum(acc);
        } else {
          // lane 0 holds the largest selection logit; with the bias removed
          // the order may change, so take the maximum
          m = sel_only ? warp_max(lane < k ? base : -INFINITY) : __shfl_sync(0xffffffffu, zv, 0);
          den = warp_sum(lane < k ? __expf(base - m) : 0.0f);
        }
        ex = (lane < k) ? __expf(base - m) : 0.0f;
      } else {
        const float z0 = __shfl_sync(0xffffffffu, zv, 0);
        ex = (lane < k) ? __expf(zv - z0) : 0.0f;
        den = warp_sum(ex);
      }
      if (lane < k) {
        M.sel_id[warp][lane] = oi2;
        M.sel_w[warp][lane] = ex / den;
        if constexpr (TT == 1) {  // the units: the selection in selection order
          M.unit_w[lane][0] = ex / den;
          M.unit_expert[lane] = oi2;
          M.unit_slot[lane] = slot_checked(oi2);
        }
      }
      if (TT == 1 && lane == 0) {
        M.n_routed = k;
        M.n_units = k + (Fs > 0 ? 1 : 0);
      }
    }
    if constexpr (TT == 1) {
      // one token: the units are the selection itself, in selection order,
      // written by the softmax warp above (only unit_w[u][0] is read)
    } else {
      if (tid < kMaxExperts / 32) M.bitmap[tid] = 0u;
      for (int i = tid; i < kMaxUnits * kMaxDecodeTokens; i += kDecodeThreads)
        (&M.unit_w[0][0])[i] = 0.0f;
      cta_sync();
      if (tid < T * k) atomicOr(&M.bitmap[M.sel_id[tid / k][tid % k] >> 5], 1u << (M.sel_id[tid / k][tid % k] & 31));
      cta_sync();
      if (warp == 0) {  // exclusive prefix of the bitmap's popcounts
        const int c = __popc(M.bitmap[lane]);
        int x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        M.prefix[lane] = x - c;
        if (lane == 31) {
          M.prefix[32] = x;
          M.n_routed = x;
          M.n_units = x + (Fs > 0 ? 1 : 0);
        }
      }
      cta_sync();
      if (tid < T * k) {
        const int t = tid / k, r = tid % k;
        const int e = M.sel_id[t][r];
        const int u = M.prefix[e >> 5] + __popc(M.bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
        M.unit_w[u][t] = M.sel_w[t][r];
        M.unit_expert[u] = e;
        const int s = slot_checked(e);
        M.unit_slot[u] = s;
      }
    }
    if (blockIdx.x == 0 && tid < T * k) {
      const int t = tid / k, r = tid % k;
      if (p.ids_out) p.ids_out[((size_t)l * T + t) * k + r] = M.sel_id[t][r];
      if (p.w_out) p.w_out[((size_t)l * T + t) * k + r] = M.sel_w[t][r];
    }
    {
      // the shared expert is the unit after the routed ones, weight 1
      const int nr = (TT == 1) ? k : M.n_routed;
      if (Fs > 0 && tid < kMaxDecodeTokens) {
        float ws = 1.0f;  // gated: sigmoid of the gate logit a CTA wrote before the barrier
        if (kVar && (p.routing_flags[l] & MOE_ROUTING_SHARED_GATE) && tid < T)
          ws = 1.0f / (1.0f + __expf(-__ldcg(p.gz + tid)));
        M.unit_w[nr][tid] = (tid < T) ? ws : 0.0f;
      }
    }
    if (partial) {
      // ---- expert cache: misses are served before the units run
      const CacheDev* cd = W.cache;
      const int nr_l = (TT == 1) ? k : M.n_routed;
      if (tid < kMaxExperts / 32) M.inuse[tid] = 0u;
      cta_sync();  // the unit list is complete
      if (tid == 0) {
        int n = 0;
        for (int u = 0; u < nr_l; ++u)
          if (M.unit_slot[u] < 0) M.miss_unit[n++] = u;
        M.n_miss = n;
      }
      if (tid < nr_l && M.unit_slot[tid] >= 0)
        atomicOr(&M.inuse[M.unit_slot[tid] >> 5], 1u << (M.unit_slot[tid] & 31));
      cta_sync();
      const int n_miss = M.n_miss;  // the same in every CTA (same tables, same selection)
      if (n_miss > 0) {
        // victims: the least recently used slots this call does not use
        // (ties to the lower slot), one block-wide argmin per miss; every
        // CTA reaches the same choice
        unsigned long long key[kMaxExperts / kDecodeThreads];
#pragma unroll
        for (int j = 0; j < kMaxExperts / kDecodeThreads; ++j) {
          const int sl = tid + j * kDecodeThreads;
          key[j] = (sl < S_l) ? (((unsigned long long)__ldcg(cd->last_use + sl) << 32) | (unsigned)sl)
                              : ~0ull;
        }
        for (int i = 0; i < n_miss; ++i) {
          unsigned long long best = ~0ull;
#pragma unroll
          for (int j = 0; j < kMaxExperts / kDecodeThreads; ++j) {
            const int sl = tid + j * kDecodeThreads;
            if (sl < S_l && !((M.inuse[sl >> 5] >> (sl & 31)) & 1u) && key[j] < best) best = key[j];
          }
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other < best ? other : best;
          }
          if (lane == 0) M.red_key[warp] = best;
          cta_sync();
          if (tid == 0) {
            unsigned long long b = ~0ull;
            for (int w = 0; w < kWarps; ++w) b = M.red_key[w] < b ? M.red_key[w] : b;
            int v = (int)(b & 0xffffffffu);
            if (b == ~0ull) {  // no free slot (n_slots too small): not reachable after validation
              atomicCAS(p.err, 0, (int)MOE_ERR_BOUNDS);
              v = 0;
            }
            M.inuse[v >> 5] |= 1u << (v & 31);
            M.unit_slot[M.miss_unit[i]] = v;
          }
          cta_sync();
        }
        // the missed experts, from the host tier into their new slots
        {
          copy_misses(cd, W, F, H, n_miss, M.miss_unit, M.unit_expert, M.unit_slot, tid);
          fence_proxy_async_global();  // the slots are read next by TMA
        }
        grid_sync(p.bar, nbar, p.err, tmo, p.debug_extra_arrivals);
        // every CTA has its copy of the tables and stamps: CTA 0 records the
        // new residency
        if (blockIdx.x == 0 && tid == 0) {
          int32_t* so = const_cast<int32_t*>(W.slot_of);
          for (int i = 0; i < n_miss; ++i) {
            const int u = M.miss_unit[i], e = M.unit_expert[u], v = M.unit_slot[u];
            const int old = cd->slot_expert[v];
            if (old >= 0 && old < E) so[old] = -1;
            so[e] = v;
            cd->slot_expert[v] = e;
          }
        }
      }
      if (blockIdx.x == 0 && tid < nr_l) cd->last_use[M.unit_slot[tid]] = p.step;
      if (blockIdx.x == 0 && tid == 0) {
        atomicAdd(&cd->stats[0], (unsigned long long)(nr_l - n_miss));
        atomicAdd(&cd->stats[1], (unsigned long long)n_miss);
      }
    }
    // the slot table was read through the generic proxy; the next layer's
    // bulk copy (async proxy) overwrites it.  The unit list is ready: the
    // copy warp starts this layer's weight copies.
    fence_proxy_async_smem();
    named_bar_sync(kNbUnits, kDecodeBlock);
    if (p.mode == kModeRoute) continue;
    const int n_routed = M.n_routed;
    // the other accumulator held the previous layer's output, which every
    // CTA read in phase R: zero it for the next layer (its first reductions
    // come after the next barrier)
    {
      float* ynext = p.yacc + (size_t)((l + 1) & 1) * kMaxDecodeTokens * H;
      for (int i = blockIdx.x * kDecodeThreads + tid; i < TT * H; i += grid * kDecodeThreads) ynext[i] = 0.0f;
    }

    // ------------------------------------------------ work units
    // A work unit is (unit, 32-row block of its F): gate/up rows of the block
    // (two 16-row items through the stage ring), then the block's columns of
    // the down matrix against all H outputs.  The copy warp brings the data.
    const int my_wu = my_units(n_routed);
    const int n_my_items = 2 * my_wu;
    // caller-layout layers (no tensor maps): the down block is copied per
    // thread, 16 code bytes and the 4-byte scale pair holding the block's
    // scale per row, at the same row positions as the TMA path
    auto issue_d_threads = [&](int j) {
      int u, b;
      wu_of(j, n_routed, u, b);
      const uint8_t* cq;
      const uint16_t* cs;
      int Fu;
      if (u < n_routed) {
        const size_t slot = (size_t)M.unit_slot[u];
        cq = W.down_q + slot * H * (size_t)(F / 2);
        cs = W.down_s + slot * H * (size_t)CF;
        Fu = F;
      } else {
        cq = W.sh_down_q;
        cs = W.sh_down_s;
        Fu = Fs;
      }
      const uint32_t s_codes = smem_u32(dst_s), s_scales = smem_u32(dst_s + (size_t)H * 16);
      for (int r = tid; r < H; r += kDecodeThreads) {
        const uint32_t pos = (uint32_t)((r & 3) * Hq + (r >> 2));
        cp_async_16(s_codes + pos * 16u, cq + (size_t)r * (Fu / 2) + 16 * b);
        cp_async_4(s_scales + pos * 4u, cs + (size_t)r * (Fu / 32) + (b & ~1));
      }
      cp_async_commit();
    };
    if (!p.down_tma && my_wu > 0) issue_d_threads(0);

    // ------------------------------------------------ gate/up + SwiGLU, then down per block
    {
      float* ycur = p.yacc + (size_t)(l & 1) * kMaxDecodeTokens * H;
      // warp w owns row pairs 2w, 2w+1 of every item (gate and up rows)
      for (int q = 0; q < n_my_items; ++q) {
        const int it = item_of(q);
        const int u = (it < n_routed * ipu) ? it / ipu : n_routed;
        const int sg = q % NG;
        const uint32_t par = (sg ? gcount1 : gcount0) & 1u;
        if (sg) ++gcount1;
        else ++gcount0;
        const unsigned char* st = gbuf + (size_t)sg * L.g_stage;
        mbar_wait(&mbar[kBarG0 + sg], par, p.err, tmo);
        if (gu_mma) {
          // tensor path: warp w takes blocks w, w + 8, ... of all 32 rows;
          // lane (g, c) ends with rows g, g + 8 of gate and of up for
          // tokens 2c, 2c + 1, summed over its blocks
          const int g = lane >> 2, cq = lane & 3;
          float ag[4] = {0.0f, 0.0f, 0.0f, 0.0f}, au[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          for (int b = warp; b < C; b += kWarps) {
            uint4 bx = make_uint4(0u, 0u, 0u, 0u);
            if (g < T) bx = xp[(g * C + b) * 4 + cq];
            float2 cr = make_float2(0.0f, 0.0f);
            if (2 * cq < TT) cr = *reinterpret_cast<const float2*>(corrx + b * 4 + 2 * cq);
            const unsigned char* cg = st + (size_t)b * 256 + g * 16 + 4 * cq;  // gate codes, row g
            const unsigned char* cu = cg + 16 * (H / 2);                       // up codes, row g
            uint32_t v0[4], v1[4];
            float dg[4] = {-cr.x, -cr.y, -cr.x, -cr.y}, du[4] = {-cr.x, -cr.y, -cr.x, -cr.y};
            unpack_biased(*reinterpret_cast<const uint32_t*>(cg), v0);
            unpack_biased(*reinterpret_cast<const uint32_t*>(cg + 128), v1);
            mma_16816(dg, v0[0], v1[0], v0[1], v1[1], bx.x, bx.y);
            mma_16816(dg, v0[2], v1[2], v0[3], v1[3], bx.z, bx.w);
            unpack_biased(*reinterpret_cast<const uint32_t*>(cu), v0);
            unpack_biased(*reinterpret_cast<const uint32_t*>(cu + 128), v1);
            mma_16816(du, v0[0], v1[0], v0[1], v1[1], bx.x, bx.y);
            mma_16816(du, v0[2], v1[2], v0[3], v1[3], bx.z, bx.w);
            // scales of (row g, block b) and (row g + 8, block b)
            const unsigned char* sc0 = st + 16 * H + ((size_t)(b >> 3) * 16 + g) * 16 + (b & 7) * 2;
            const float sg0 = __half2float(*reinterpret_cast<const __half*>(sc0));
            const float sg1 = __half2float(*reinterpret_cast<const __half*>(sc0 + 128));
            const float su0 = __half2float(*reinterpret_cast<const __half*>(sc0 + 32 * C));
            const float su1 = __half2float(*reinterpret_cast<const __half*>(sc0 + 32 * C + 128));
            ag[0] = fmaf(sg0, dg[0], ag[0]);
            ag[1] = fmaf(sg0, dg[1], ag[1]);
            ag[2] = fmaf(sg1, dg[2], ag[2]);
            ag[3] = fmaf(sg1, dg[3], ag[3]);
            au[0] = fmaf(su0, du[0], au[0]);
            au[1] = fmaf(su0, du[1], au[1]);
            au[2] = fmaf(su1, du[2], au[2]);
            au[3] = fmaf(su1, du[3], au[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&mbar[kBarE0 + sg]);  // this warp is done with the stage
          // this warp's sums of the item's 32 rows (gate 0..15, up 16..31)
          float* rw = gred + (size_t)(q & 1) * (kWarps * 32 * TT) + (size_t)warp * 32 * TT;
          if (2 * cq < TT) {
            rw[g * TT + 2 * cq] = ag[0];
            rw[(g + 8) * TT + 2 * cq] = ag[2];
            rw[(16 + g) * TT + 2 * cq] = au[0];
            rw[(24 + g) * TT + 2 * cq] = au[2];
            if (2 * cq + 1 < TT) {
              rw[g * TT + 2 * cq + 1] = ag[1];
              rw[(g + 8) * TT + 2 * cq + 1] = ag[3];
              rw[(16 + g) * TT + 2 * cq + 1] = au[1];
              rw[(24 + g) * TT + 2 * cq + 1] = au[3];
            }
          }
          cta_sync();  // every warp's sums of the item are in place
          if (tid < 16 * TT) {
            const int r = tid / TT, t = tid - (tid / TT) * TT;
            const float* ri = gred + (size_t)(q & 1) * (kWarps * 32 * TT);
            float gs = 0.0f, us = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
              gs += ri[(w * 32 + r) * TT + t];
              us += ri[(w * 32 + 16 + r) * TT + t];
            }
            const float xs = pow2f(M.x_shift[t]);
            const float gv = gs * xs, uv = us * xs;
            const float h = gv / (1.0f + __expf(-gv)) * uv;
            M.hst[q & 1][r][t] = h * M.unit_w[u][t];
          }
        } else {
          float acc[4][TT];  // rows: gate 2w, gate 2w+1, up 2w, up 2w+1
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < TT; ++t) acc[r][t] = 0.0f;
          for (int c = lane; c < C; c += 32) {
            uint4 act[TT][4];
#pragma unroll
            for (int t = 0; t < TT; ++t)
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) act[t][qq] = xp[(t * 4 + qq) * C + c];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int mat = r >> 1, row = 2 * warp + (r & 1);
              const uint4 wv = *reinterpret_cast<const uint4*>(st + (size_t)mat * 16 * (H / 2) +
                                                               (size_t)row * (H / 2) + c * 16);
              const float s =
                  __half2float(reinterpret_cast<const __half*>(st + 16 * H + mat * 32 * C)[row * C + c]);
              float d[TT];
              dot_block<TT>(wv, act, d);
#pragma unroll
              for (int t = 0; t < TT; ++t) acc[r][t] = fmaf(s, d[t], acc[r][t]);
            }
          }
          // the stage is refilled by bulk copies (async proxy): fence this
          // warp's generic reads of it before handing it back
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&mbar[kBarE0 + sg]);  // this warp is done with the stage
          float v[4 * TT];
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < TT; ++t) v[r * TT + t] = acc[r][t];
          // value idx = r*TT + t ends in lanes [idx*REP, (idx+1)*REP); the up row
          // of the same (row pair, token) is 2*TT indices on: 16 lanes further
          const float s = warp_reduce_scatter<4 * TT>(v, lane);
          const float up = __shfl_down_sync(0xffffffffu, s, 16);
          constexpr int REP = 32 / (4 * TT);
          if (lane < 16 && (lane & (REP - 1)) == 0) {
            const int idx = lane / REP;
            const int rp = idx / TT, t = idx - (idx / TT) * TT;
            const float xs = pow2f(M.x_shift[t]);
            const float g = s * xs, uu = up * xs;
            const float h = g / (1.0f + __expf(-g)) * uu;
            M.hst[q & 1][2 * warp + rp][t] = h * M.unit_w[u][t];
          }
        }
        // the down block after the odd item reads both items' rows: the
        // even item needs no barrier of its own (the next item writes the
        // other half of hst, and the stages are guarded by mbarriers)
        if ((q & 1) == 0) continue;
        cta_sync();  // both items' 16 rows of w*h are staged
        // ---- down block of work unit j: both halves of its 32 rows are staged
        const int j = q >> 1;
        int ub, b;
        wu_of(j, n_routed, ub, b);
        if (tid < TT * 4) {
          // fp16 pair planes of the block's 32 w*h values per token, in the
          // code unpack order, scaled by a power of two that puts the
          // token's max |w h| in [32, 64) (the shift goes beside them)
          const int t = tid >> 2, qw = tid & 3;
          float m = 0.0f;
#pragma unroll
          for (int f = 0; f < 32; ++f) m = fmaxf(m, fabsf(M.hst[f >> 4][f & 15][t]));
          const int sh = range_shift(m);
          const float sc = pow2f(-sh);
          uint32_t o[4];
          float cb = 0.0f;  // bias of this word's codes in the tensor path
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int e0 = 8 * qw + jj, e1 = e0 + 4;
            __half2 hh = __floats2half2_rn(M.hst[e0 >> 4][e0 & 15][t] * sc, M.hst[e1 >> 4][e1 & 15][t] * sc);
            o[jj] = *reinterpret_cast<uint32_t*>(&hh);
            if constexpr (TT > 1) {
              const float2 f = __half22float2(hh);
              cb += ((jj & 1) ? 72.0f : 1032.0f) * (f.x + f.y);
            }
          }
          M.actD[t][qw] = make_uint4(o[0], o[1], o[2], o[3]);
          if (qw == 0) M.dsh[t] = sh;
          if constexpr (TT > 1) {  // the four words of token t sit in lanes 4t .. 4t + 3
            constexpr unsigned mask = (TT * 4 >= 32) ? 0xffffffffu : ((1u << (TT * 4)) - 1u);
            cb += __shfl_xor_sync(mask, cb, 1);
            cb += __shfl_xor_sync(mask, cb, 2);
            if (qw == 0) M.corrd[t] = cb;
          }
        }
        if (p.down_tma) {
          mbar_wait(&mbar[kBarD], ph_d, p.err, tmo);
          ph_d ^= 1u;
        } else {
          cp_async_wait<0>();
        }
        cta_sync();  // the act planes, and every thread's copies of the down block
        const unsigned char* dc = dst_s;
        const unsigned char* dsc = dst_s + (size_t)H * 16;
        if constexpr (TT > 1) {
          // tensor path: tile (q0, jr) holds rows 4 (q0 + i) + jr, i < 16, at
          // positions jr H/4 + q0 + i (16 bytes each: one 32-column block);
          // after the four tiles of a group lane (g, c) holds rows
          // 4 (q0 + g) .. + 3 and 4 (q0 + g + 8) .. + 3 of tokens 2c, 2c + 1
          const int g = lane >> 2, cq = lane & 3;
          const int tA = 2 * cq, tB = 2 * cq + 1;
          uint4 bx = make_uint4(0u, 0u, 0u, 0u);
          if (g < T) bx = M.actD[g][cq];
          const bool liveA = tA < T && M.unit_w[ub][tA] != 0.0f;
          const bool liveB = tB < T && M.unit_w[ub][tB] != 0.0f;
          const float ca = tA < T ? -M.corrd[tA] : 0.0f;
          const float cb = tB < T ? -M.corrd[tB] : 0.0f;
          const float yA = liveA ? pow2f(M.dsh[tA]) : 0.0f;
          const float yB = liveB ? pow2f(M.dsh[tB]) : 0.0f;
          for (int G = warp; G < Hq / 16; G += kWarps) {
            const int q0 = 16 * G;
            float d[4][4];
#pragma unroll
            for (int jr = 0; jr < 4; ++jr) {
              const unsigned char* rb = dc + ((size_t)jr * Hq + q0 + g) * 16 + 4 * cq;
              uint32_t v0[4], v1[4];
              unpack_biased(*reinterpret_cast<const uint32_t*>(rb), v0);
              unpack_biased(*reinterpret_cast<const uint32_t*>(rb + 8 * 16), v1);
              d[jr][0] = ca;
              d[jr][1] = cb;
              d[jr][2] = ca;
              d[jr][3] = cb;
              mma_16816(d[jr], v0[0], v1[0], v0[1], v1[1], bx.x, bx.y);
              mma_16816(d[jr], v0[2], v1[2], v0[3], v1[3], bx.z, bx.w);
            }
            float s0[4], s1[4];  // scales of rows 4 (q0 + g) + jr and 4 (q0 + g + 8) + jr
            if (p.down_tma) {
              const uint2 a = *reinterpret_cast<const uint2*>(dsc + (size_t)(q0 + g) * 8);
              const uint2 e = *reinterpret_cast<const uint2*>(dsc + (size_t)(q0 + g + 8) * 8);
              s0[0] = __half2float(__ushort_as_half((uint16_t)(a.x & 0xffffu)));
              s0[1] = __half2float(__ushort_as_half((uint16_t)(a.x >> 16)));
              s0[2] = __half2float(__ushort_as_half((uint16_t)(a.y & 0xffffu)));
              s0[3] = __half2float(__ushort_as_half((uint16_t)(a.y >> 16)));
              s1[0] = __half2float(__ushort_as_half((uint16_t)(e.x & 0xffffu)));
              s1[1] = __half2float(__ushort_as_half((uint16_t)(e.x >> 16)));
              s1[2] = __half2float(__ushort_as_half((uint16_t)(e.y & 0xffffu)));
              s1[3] = __half2float(__ushort_as_half((uint16_t)(e.y >> 16)));
            } else {
#pragma unroll
              for (int jr = 0; jr < 4; ++jr) {
                const uint32_t sa = *reinterpret_cast<const uint32_t*>(dsc + ((size_t)jr * Hq + q0 + g) * 4);
                const uint32_t se = *reinterpret_cast<const uint32_t*>(dsc + ((size_t)jr * Hq + q0 + g + 8) * 4);
                s0[jr] = __half2float(__ushort_as_half((uint16_t)((b & 1) ? (sa >> 16) : (sa & 0xffffu))));
                s1[jr] = __half2float(__ushort_as_half((uint16_t)((b & 1) ? (se >> 16) : (se & 0xffffu))));
              }
            }
            if (liveA) {
              red_add_v4(ycur + (size_t)tA * H + 4 * (q0 + g), s0[0] * d[0][0] * yA, s0[1] * d[1][0] * yA,
                         s0[2] * d[2][0] * yA, s0[3] * d[3][0] * yA);
              red_add_v4(ycur + (size_t)tA * H + 4 * (q0 + g + 8), s1[0] * d[0][2] * yA,
                         s1[1] * d[1][2] * yA, s1[2] * d[2][2] * yA, s1[3] * d[3][2] * yA);
            }
            if (liveB) {
              red_add_v4(ycur + (size_t)tB * H + 4 * (q0 + g), s0[0] * d[0][1] * yB, s0[1] * d[1][1] * yB,
                         s0[2] * d[2][1] * yB, s0[3] * d[3][1] * yB);
              red_add_v4(ycur + (size_t)tB * H + 4 * (q0 + g + 8), s1[0] * d[0][3] * yB,
                         s1[1] * d[1][3] * yB, s1[2] * d[2][3] * yB, s1[3] * d[3][3] * yB);
            }
          }
        } else {
          uint4 act[TT][4];
          float ysc[TT];
          bool live[TT];
#pragma unroll
          for (int t = 0; t < TT; ++t) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) act[t][qq] = M.actD[t][qq];
            ysc[t] = pow2f(M.dsh[t]);
            live[t] = (t < T) && M.unit_w[ub][t] != 0.0f;
          }
          // four consecutive output rows 4 q4 .. 4 q4 + 3 per thread and step,
          // added into the layer output with one vector reduction per token
          for (int q4 = tid; q4 < Hq; q4 += kDecodeThreads) {
            float d[4][TT], sc4[4];
            if (p.down_tma) {  // rows 4 q4 .. 4 q4 + 3 of the block-major scales
              const uint2 sv = *reinterpret_cast<const uint2*>(dsc + (size_t)q4 * 8);
              sc4[0] = __half2float(__ushort_as_half((uint16_t)(sv.x & 0xffffu)));
              sc4[1] = __half2float(__ushort_as_half((uint16_t)(sv.x >> 16)));
              sc4[2] = __half2float(__ushort_as_half((uint16_t)(sv.y & 0xffffu)));
              sc4[3] = __half2float(__ushort_as_half((uint16_t)(sv.y >> 16)));
            } else {
#pragma unroll
              for (int jr = 0; jr < 4; ++jr) {
                const uint32_t sp = *reinterpret_cast<const uint32_t*>(dsc + ((size_t)jr * Hq + q4) * 4);
                sc4[jr] = __half2float(__ushort_as_half((uint16_t)((b & 1) ? (sp >> 16) : (sp & 0xffffu))));
              }
            }
#pragma unroll
            for (int jr = 0; jr < 4; ++jr) {
              const uint4 wv = *reinterpret_cast<const uint4*>(dc + ((size_t)jr * Hq + q4) * 16);
              dot_block<TT>(wv, act, d[jr]);
            }
#pragma unroll
            for (int t = 0; t < TT; ++t)
              if (live[t])
                red_add_v4(ycur + (size_t)t * H + 4 * q4, sc4[0] * d[0][t] * ysc[t],
                           sc4[1] * d[1][t] * ysc[t], sc4[2] * d[2][t] * ysc[t],
                           sc4[3] * d[3][t] * ysc[t]);
          }
        }
        // the copy warp refills the stage by TMA (async proxy) once every
        // warp has released it
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&mbar[kBarDE]);
        // every thread is done with the down stage and the act planes before
        // the next unit's; after the last unit the grid barrier's own CTA
        // barrier comes first
        if (j + 1 < my_wu) {
          cta_sync();
          if (!p.down_tma) issue_d_threads(j + 1);
        }
      }
    }
    // the next layer's bulk copies land in shared memory this layer read
    // through the generic proxy: order those reads before them
    fence_proxy_async_smem();
    grid_sync(p.bar, nbar, p.err, tmo, p.debug_extra_arrivals);
  }

  // ------------------------------------------------ output: y, or h_L for stacks
  if (p.mode != kModeRoute) {
    const float* yl = p.yacc + (size_t)((p.n_layers - 1) & 1) * kMaxDecodeTokens * H;
    for (int i = blockIdx.x * kDecodeThreads + tid; i < T * H; i += grid * kDecodeThreads) {
      const __nv_bfloat16 yb = __float2bfloat16_rn(__ldcg(yl + i));
      if (p.y_trace) p.y_trace[(size_t)(p.n_layers - 1) * T * H + i] = __bfloat16_as_ushort(yb);
      if (stack) {
        const float xv = __bfloat162float(__ushort_as_bfloat16(hres[i]));
        const uint16_t xn = __bfloat16_as_ushort(__float2bfloat16_rn(xv + __bfloat162float(yb)));
        p.y_out[i] = xn;
        if (p.h_trace) p.h_trace[(size_t)(p.n_layers - 1) * T * H + i] = xn;
      } else {
        p.y_out[i] = __bfloat16_as_ushort(yb);
      }
    }
  }
}

// 5-D map over one matrix of down codes [slots][H][Fd/2] (bytes) in which
// row r = 4 q + j of a slot, q = QB q_hi + q_lo, is addressed as
// (byte, q_lo, q_hi, j, slot): dims {Fd/2, QB, H/(4 QB), 4, slots}, strides
// {2 Fd, 2 Fd QB, Fd/2, H Fd/2} bytes, QB = down_qbox(H).  The box {16, QB,
// H/(4 QB), 4, 1} is one whole 32-column block of a slot in one copy, landing
// with row r at position j * H/4 + q: the four row planes one after another.
static bool encode_down_map(CUtensorMap* m, const void* base, int H, int Fd, int slots) {
  auto enc = tmap_encode_fn();
  if (!enc) return false;
  const int QB = down_qbox(H), nqb = H / 4 / QB;
  cuuint64_t dims[5] = {(cuuint64_t)Fd / 2, (cuuint64_t)QB, (cuuint64_t)nqb, 4, (cuuint64_t)slots};
  cuuint64_t strides[4] = {2 * (cuuint64_t)Fd, 2 * (cuuint64_t)Fd * QB, (cuuint64_t)Fd / 2,
                           (cuuint64_t)H * Fd / 2};
  cuuint32_t box[5] = {16, (cuuint32_t)QB, (cuuint32_t)nqb, 4, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D maps over one gate or up matrix of `rows` rows for the tensor path's
// block-major stage.  Codes [rows][H/2] bytes as (byte, row, block): dims
// {16, rows, H/32}, strides {H/2, 16}, box {16, 16, H/32} lands 16 rows as
// [block][row][16 B].  Scales [rows][H/32] fp16 as (half, row, 8-block
// chunk): dims {8, rows, H/256}, strides {H/16, 16}, box {8, 16, H/256}
// lands them as [chunk][row][8].
static bool encode_gu_maps(CUtensorMap* codes, CUtensorMap* scales, const void* q, const void* sc,
                           int H, int rows) {
  auto enc = tmap_encode_fn();
  if (!enc) return false;
  cuuint64_t dq[3] = {16, (cuuint64_t)rows, (cuuint64_t)H / 32};
  cuuint64_t sq[2] = {(cuuint64_t)H / 2, 16};
  cuuint32_t bq[3] = {16, 16, (cuuint32_t)H / 32};
  cuuint64_t ds[3] = {8, (cuuint64_t)rows, (cuuint64_t)H / 256};
  cuuint64_t ss[2] = {(cuuint64_t)H / 16, 16};
  cuuint32_t bs[3] = {8, 16, (cuuint32_t)H / 256};
  cuuint32_t e1[3] = {1, 1, 1};
  return enc(codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q), dq, sq, bq, e1,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
         enc(scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(sc), ds, ss, bs, e1,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

moe_status decode_prepare(moe_layer* L, const char** why) {
  const moe_layer_config& c = L->cfg;
  const bool sh = c.shared_ffn > 0;
  if (!encode_down_map(&L->tm_dec_down, L->dev.down_q, c.hidden, c.ffn, c.n_slots) ||
      !encode_down_map(&L->tm_dec_sh_down, sh ? L->dev.sh_down_q : L->dev.down_q, c.hidden,
                       sh ? c.shared_ffn : c.ffn, 1)) {
    *why = "cuTensorMapEncodeTiled failed (decode down codes)";
    return MOE_ERR_CUDA;
  }
  L->dev.tm_gu = nullptr;
  if (c.hidden % 256 == 0) {
    // gate, up, shared gate, shared up: codes in maps 0-3, scales in 4-7
    // (without a shared expert, 2, 3, 6, 7 repeat the routed ones unused)
    CUtensorMap m[8];
    const int R = c.n_slots * c.ffn, Rs = sh ? c.shared_ffn : R;
    const LayerDev& D = L->dev;
    if (!encode_gu_maps(&m[0], &m[4], D.gate_q, D.gate_s, c.hidden, R) ||
        !encode_gu_maps(&m[1], &m[5], D.up_q, D.up_s, c.hidden, R) ||
        !encode_gu_maps(&m[2], &m[6], sh ? D.sh_gate_q : D.gate_q, sh ? D.sh_gate_s : D.gate_s,
                        c.hidden, Rs) ||
        !encode_gu_maps(&m[3], &m[7], sh ? D.sh_up_q : D.up_q, sh ? D.sh_up_s : D.up_s, c.hidden, Rs)) {
      *why = "cuTensorMapEncodeTiled failed (decode gate/up codes)";
      return MOE_ERR_CUDA;
    }
    if (cudaMalloc(&L->tm_gu_block, sizeof m) != cudaSuccess) {
      L->tm_gu_block = nullptr;
      cudaGetLastError();
      *why = "device memory for the gate/up tensor maps";
      return MOE_ERR_OOM;
    }
    if (cudaMemcpy(L->tm_gu_block, m, sizeof m, cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      *why = "gate/up tensor maps to device memory";
      return MOE_ERR_CUDA;
    }
    L->dev.tm_gu = static_cast<const CUtensorMap*>(L->tm_gu_block);
  }
  return MOE_OK;
}

size_t decode_smem_bytes(const DecodeParams& p, int num_sms) {
  const int TT = p.T == 1 ? 1 : (p.T == 2 ? 2 : 4);
  return DecodeSmem::make(p.H, p.E, TT, num_sms, 1, 0).total;
}

template <int TT>
static moe_status launch_tt(const DecodeParams& p_in, cudaStream_t stream, int num_sms,
                            const char** why) {
  bool var = false;
  for (int l = 0; l < p_in.n_layers; ++l) var = var || p_in.routing_flags[l] != 0;
  auto kern = var ? moe_decode_kernel<TT, true> : moe_decode_kernel<TT, false>;
  DecodeParams p = p_in;
  const int grid = num_sms;  // one CTA per SM
  // gate/up items by the tensor cores for more than one token when every
  // layer has the block-major maps and two stages still fit; otherwise the
  // fp16 path with two gate/up stages when they fit, else one
  const size_t cap = (size_t)227 * 1024;
  bool gu = TT > 1 && p.H % 256 == 0;
  for (int l = 0; l < p.n_layers; ++l) gu = gu && p.layers[l].tm_gu != nullptr;
  p.g_stages = 2;
  p.gu_mma = 0;
  DecodeSmem sm = DecodeSmem::make(p.H, p.E, TT, grid, 2, 0);
  if (gu) {
    const DecodeSmem sg = DecodeSmem::make(p.H, p.E, TT, grid, 2, 1);
    if (sg.total <= cap) {
      p.gu_mma = 1;
      sm = sg;
    }
  }
  if (sm.total > cap) {
    p.g_stages = 1;
    sm = DecodeSmem::make(p.H, p.E, TT, grid, 1, 0);
  }
  if (sm.total > cap) {
    *why = "decode shared-memory footprint exceeds 227 KB for this shape";
    return MOE_ERR_INVALID;
  }
  const size_t smem = sm.total;
  // the shared-memory limit and the residency check, once per instantiation
  // and footprint (a host-side cost on every call otherwise)
  static std::mutex mu;
  static size_t checked_smem[16][2] = {};  // per device and routing instantiation: largest footprint verified
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) dev = -1;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || smem > checked_smem[dev][var ? 1 : 0]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess) {
        *why = "cudaFuncSetAttribute(max dynamic smem) failed";
        return MOE_ERR_CUDA;
      }
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeBlock, smem) !=
              cudaSuccess ||
          per_sm < 1) {
        *why = "decode kernel cannot be resident (occupancy query)";
        return MOE_ERR_CUDA;
      }
      if (dev >= 0) checked_smem[dev][var ? 1 : 0] = smem;
    }
  }
  if (cudaMemsetAsync(p.bar, 0, sizeof(GridBarrier), stream) != cudaSuccess) {
    *why = "cudaMemsetAsync(barrier) failed";
    return MOE_ERR_CUDA;
  }
  void* args[] = {&p};
  prof::Scope scope("moe_decode_kernel", stream);
  cudaError_t e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kDecodeBlock),
                                              args, smem, stream);
  if (e != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status launch_decode(const DecodeParams& p, cudaStream_t stream, int num_sms,
                         const char** why) {
  if (p.T == 1) return launch_tt<1>(p, stream, num_sms, why);
  if (p.T == 2) return launch_tt<2>(p, stream, num_sms, why);
  return launch_tt<4>(p, stream, num_sms, why);
}

}  // namespace moe
