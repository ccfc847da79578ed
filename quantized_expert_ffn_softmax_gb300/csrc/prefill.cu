// Prefill path (5 or more tokens): bucketed grouped GEMMs on the tcgen05
// tensor cores.
//
//   prep       x (bf16) -> x16: fp16, scaled per token by a power of two so
//              the row maximum lies in [1, 2), K reordered inside every group
//              of 8 to the order in which packed 4-bit codes unpack
//   router     z = W_r x + b as one tcgen05 GEMM with K' = 2H: W_r is split
//              on the fly into two fp16 terms (hi + mid, 22 significant bits)
//              so the logits keep fp32-level accuracy for the exact top-k
//   top-k      one warp per token; softmax over the selected logits
//   bucket     stable counting sort of the (token, slot) assignments by
//              expert; builds the work-unit lists of the two GEMMs
//   gate/up    per unit (expert, 128-token tile, 128-row F tile):
//              D_g, D_u = W_g/u[128 x H] . X[tokens]^T in TMEM, epilogue
//              h = silu(g) * u -> fp16 rows of Hmid (bucket order)
//   down       per unit (expert, token tile, 128-row H tile):
//              D = W_d[128 x F] . Hmid[tokens]^T, epilogue y += w * D
//              scattered to the tokens' rows (fp32 reductions in L2)
//   finalize   y (fp32) -> bf16
//
// GEMM engine: one persistent CTA per SM, warp-specialised.
//   warps 0-3   epilogue (TMEM lanes 0-127 = the 128 rows of the tile)
//   warps 4-11  A producers: dequantise 4-bit codes (or split fp32 router
//               weights) into fp16 128x64 tiles in the 128-byte swizzled
//               K-major layout, straight into the stage's shared memory
//   B loaders   gate/up: warps 12-13 gather the unit's token rows (bucket
//               order) with per-thread 16-byte async copies into the same
//               swizzled layout; down/router: warp 12 loads the unit's
//               contiguous rows as one TMA tile per K step
//   last warp   TMEM allocator and single-thread tcgen05.mma issuer
// A 4-stage shared-memory ring (full/empty mbarriers) feeds the MMA; two
// TMEM accumulators let the epilogue of one unit overlap the next unit's
// MMAs.  Every wait is bounded and gives up once the error word is set.
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "device_common.cuh"
#include "moe_internal.cuh"
#include "profile.cuh"

namespace moe {
namespace {

using namespace dev;

constexpr int kNT = 128;           // token tile = largest MMA N used
constexpr int kStages = 4;
constexpr int kTileA = 128 * 128;  // bytes: 128 rows x 64 fp16
constexpr int kTileB = kNT * 128;  // bytes: kNT rows x 64 fp16
constexpr int kEpiWarps = 4;
constexpr int kProdWarp0 = 4;
constexpr int kProdWarps = 8;
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kBWarp0 = 12;
constexpr int kBucketThreads = 1024;
constexpr int kPrefetch = 4;       // K steps of weight codes each producer keeps in flight
constexpr int kBLag = 2;           // K steps of gathered token rows each B loader keeps in flight

enum GemmMode : int { kSwiglu = 0, kScatter = 1, kRouter = 2 };

// Warp roles after the epilogue and A-producer warps: the gate/up GEMM
// gathers its token rows with two warps of per-thread async copies; the
// down and router GEMMs read contiguous rows with one TMA tile per K step.
// At most 16 warps, so that no SM sub-partition holds more than four and a
// thread may use 128 registers.
template <int MODE>
struct Roles {
  static constexpr int kBWarps = (MODE == kSwiglu) ? 2 : 1;
  static constexpr int kMmaWarp = kBWarp0 + kBWarps;
  static constexpr int kThreads = (kMmaWarp + 1) * 32;
};

struct GemmParams {
  int H, E, k, F, Fs, T, Tk;
  int n_units_router;        // router: number of units (no list)
  const int32_t* n_units;    // gate/up or down: device count
  const int4* units;
  LayerDev W;
  const __half* x16;
  const int32_t* perm_tok;
  const float* perm_w;
  const int32_t* xshift;
  __half* hmid_r;
  __half* hmid_s;
  float* yacc;
  float* z;
  int router_shift;
  int* err;
  unsigned long long timeout_ns;
};

struct UnitInfo {
  int e, p0, n, mt, K;
  bool shared;
};

template <int MODE>
__device__ __forceinline__ UnitInfo unit_info(const GemmParams& p, int u) {
  UnitInfo U;
  if (MODE == kRouter) {
    const int nmt = (p.E + 127) / 128;
    const int tt = u / nmt;
    U.mt = u - tt * nmt;
    U.p0 = tt * kNT;
    U.n = min(kNT, p.T - U.p0);
    U.e = 0;
    U.shared = false;
    U.K = 2 * p.H;
  } else {
    const int4 v = p.units[u];
    U.e = v.x;
    U.p0 = v.y;
    U.n = v.z;
    U.mt = v.w;
    U.shared = (v.x == p.E);
    U.K = (MODE == kSwiglu) ? p.H : (U.shared ? p.Fs : p.F);
  }
  return U;
}

// 8 packed 4-bit codes (one 32-bit word, elements 8j..8j+7) -> 8 fp16
// weights (code - 8) * scale, in the unpack order 0,4,1,5,2,6,3,7.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, __half2 s2) {
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
    __half2 h = __hmul2(__hsub2(*reinterpret_cast<__half2*>(&v), k1032), s2);
    o[j] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Store chunk j (16 B, K elements 8j..8j+7) of row r into a 128-byte
// swizzled K-major tile.
__device__ __forceinline__ void st_tile_chunk(unsigned char* tile, int r, int j, uint4 v) {
  *reinterpret_cast<uint4*>(tile + r * 128 + ((j ^ (r & 7)) << 4)) = v;
}

template <int MODE>
__global__ void __launch_bounds__(Roles<MODE>::kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_hr,
                    const __grid_constant__ CUtensorMap tm_hs) {
  constexpr int NA = (MODE == kSwiglu) ? 2 : 1;
  constexpr int STAGE = NA * kTileA + kTileB;
  constexpr int kMmaWarp = Roles<MODE>::kMmaWarp;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * STAGE);
  uint64_t* full_a = bars;
  uint64_t* full_b = bars + kStages;
  uint64_t* empty = bars + 2 * kStages;
  uint64_t* tfull = bars + 3 * kStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  // per-unit token metadata of the epilogue: two words per token column
  int* meta_i = reinterpret_cast<int*>(smem + kStages * STAGE + 256);
  float* meta_f = reinterpret_cast<float*>(meta_i + kNT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_a[s], kProdThreads);
      mbar_init(&full_b[s], MODE == kSwiglu ? Roles<MODE>::kBWarps * 32 : 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps * 32);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_units = (MODE == kRouter) ? p.n_units_router : __ldcg(p.n_units);
  const uint64_t tmo = p.timeout_ns;

  if (warp < kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    // Thread r owns accumulator row r (TMEM lane r).  The per-token factors
    // of the unit (power-of-two input scales, routing weights, destination
    // rows) are staged in shared memory once per unit, one token per thread.
    const int r = warp * 32 + lane;
    int j = 0;
    float bias_r = 0.0f;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++j) {
      const UnitInfo U = unit_info<MODE>(p, u);
      if (MODE == kRouter) {
        const int e = U.mt * 128 + r;
        bias_r = e < p.E ? __ldg(p.W.router_b + e) : 0.0f;
      }
      named_bar_sync(1, kEpiWarps * 32);  // the previous unit is done with meta
      if (r < U.n) {
        if (MODE == kSwiglu) {
          const int tok = U.shared ? (U.p0 + r) : __ldg(p.perm_tok + U.p0 + r);
          const int sx = __ldg(p.xshift + tok);
          meta_i[r] = sx;  // D * 2^sx = x-scale restored; h stored * 2^-2sx
        } else if (MODE == kScatter) {
          const int tok = U.shared ? (U.p0 + r) : __ldg(p.perm_tok + U.p0 + r);
          const float wgt = U.shared ? 1.0f : __ldg(p.perm_w + U.p0 + r);
          meta_i[r] = tok;
          meta_f[r] = wgt * pow2f(2 * __ldg(p.xshift + tok));
        } else {
          meta_f[r] = pow2f(__ldg(p.xshift + U.p0 + r) - p.router_shift);
        }
      }
      const int b = j & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&tfull[b], (j >> 1) & 1, p.err, tmo);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // meta is ready, and the four warps agree on whether to go on (the
      // break must be uniform: the named barriers wait for all of them)
      if (!named_bar_and(1, kEpiWarps * 32, ok)) break;
      tc_fence_after();
      const int neff = (U.n + 15) & ~15;
      const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * 256);
      int q = 0;
      __half* hrow = nullptr;
      size_t hstride = 0;
      if (MODE == kSwiglu) {
        const int f = U.mt * 128 + r;
        q = (f & ~7) | ((f & 4) ? (((f & 3) << 1) | 1) : ((f & 3) << 1));
        hstride = U.shared ? (size_t)p.Fs : (size_t)p.F;
        hrow = (U.shared ? p.hmid_s : p.hmid_r) + (size_t)U.p0 * hstride + q;
      }
      constexpr int CW = (NA == 2) ? 16 : 32;  // columns per TMEM load
      for (int c0 = 0; c0 < neff; c0 += CW) {
        uint32_t v0[CW], v1[CW];
        tmem_ld(tbase + c0, v0);
        if (NA == 2) tmem_ld(tbase + 128 + c0, v1);
        tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < CW; ++jj) {
          const int t = c0 + jj;
          if (t >= U.n) continue;
          if (MODE == kSwiglu) {
            const int sx = meta_i[t];
            const float g = __uint_as_float(v0[jj]) * pow2f(sx);
            const float uu = __uint_as_float(v1[jj]) * pow2f(sx);
            const float h = __fdividef(g, 1.0f + __expf(-g)) * uu;
            hrow[(size_t)t * hstride] = __float2half_rn(h * pow2f(-2 * sx));
          } else if (MODE == kScatter) {
            atomicAdd(p.yacc + (size_t)meta_i[t] * p.H + U.mt * 128 + r,
                      __uint_as_float(v0[jj]) * meta_f[t]);
          } else {
            const int e = U.mt * 128 + r;
            if (e < p.E)
              p.z[(size_t)(U.p0 + t) * p.E + e] = __uint_as_float(v0[jj]) * meta_f[t] + bias_r;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[b]);
    }
  } else if (warp < kProdWarp0 + kProdWarps) {
    // ------------------------------------------------------------ A producers
    const int pi = threadIdx.x - kProdWarp0 * 32;  // 0..255
    const int r = pi & 127;
    const int part = pi >> 7;  // gate/up: matrix; down/router: which half of the K step
    const LayerDev& Wd = p.W;
    uint32_t it = 0;
    bool alive = true;
    for (int u = blockIdx.x; u < n_units && alive; u += gridDim.x) {
      const UnitInfo U = unit_info<MODE>(p, u);
      const int nks = U.K / 64;
      if (MODE == kSwiglu) {
        const int f = U.mt * 128 + r;
        const int H = p.H;
        const uint8_t* q;
        const uint16_t* sc;
        if (U.shared) {
          q = (part ? Wd.sh_up_q : Wd.sh_gate_q) + (size_t)f * (H / 2);
          sc = (part ? Wd.sh_up_s : Wd.sh_gate_s) + (size_t)f * (H / 32);
        } else {
          const size_t slot = (size_t)__ldg(Wd.slot_of + U.e);
          q = (part ? Wd.up_q : Wd.gate_q) + (slot * p.F + f) * (H / 2);
          sc = (part ? Wd.up_s : Wd.gate_s) + (slot * p.F + f) * (H / 32);
        }
        // a ring of kPrefetch K steps of codes and scales in registers keeps
        // that many global loads in flight per thread
        uint4 ca[kPrefetch], cb[kPrefetch];
        uint32_t cs[kPrefetch];
#pragma unroll
        for (int i = 0; i < kPrefetch; ++i) {
          if (i < nks) {
            ca[i] = ld_stream(q + i * 32);
            cb[i] = ld_stream(q + i * 32 + 16);
            cs[i] = __ldg(reinterpret_cast<const uint32_t*>(sc + 2 * i));
          }
        }
        for (int ks0 = 0; ks0 < nks && alive; ks0 += kPrefetch) {
#pragma unroll
          for (int i = 0; i < kPrefetch; ++i) {
            const int ks = ks0 + i;
            if (ks < nks && alive) {
              const int s = it % kStages;
              bool ok = true;
              if (lane == 0) ok = mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, p.err, tmo);
              ok = __shfl_sync(0xffffffffu, ok, 0);
              if (!ok) {
                alive = false;
              } else {
                unsigned char* tile = smem + s * STAGE + part * kTileA;
                const __half2 slo = __half2half2(__ushort_as_half((uint16_t)(cs[i] & 0xffffu)));
                const __half2 shi = __half2half2(__ushort_as_half((uint16_t)(cs[i] >> 16)));
                st_tile_chunk(tile, r, 0, dequant_word(ca[i].x, slo));
                st_tile_chunk(tile, r, 1, dequant_word(ca[i].y, slo));
                st_tile_chunk(tile, r, 2, dequant_word(ca[i].z, slo));
                st_tile_chunk(tile, r, 3, dequant_word(ca[i].w, slo));
                st_tile_chunk(tile, r, 4, dequant_word(cb[i].x, shi));
                st_tile_chunk(tile, r, 5, dequant_word(cb[i].y, shi));
                st_tile_chunk(tile, r, 6, dequant_word(cb[i].z, shi));
                st_tile_chunk(tile, r, 7, dequant_word(cb[i].w, shi));
                fence_proxy_async_smem();
                mbar_arrive(&full_a[s]);
                ++it;
                if (ks + kPrefetch < nks) {
                  ca[i] = ld_stream(q + (ks + kPrefetch) * 32);
                  cb[i] = ld_stream(q + (ks + kPrefetch) * 32 + 16);
                  cs[i] = __ldg(reinterpret_cast<const uint32_t*>(sc + 2 * (ks + kPrefetch)));
                }
              }
            }
          }
        }
      } else if (MODE == kScatter) {
        const int i = U.mt * 128 + r;  // output row of H
        const int K = U.K;
        const uint8_t* q;
        const uint16_t* sc;
        if (U.shared) {
          q = Wd.sh_down_q + (size_t)i * (K / 2);
          sc = Wd.sh_down_s + (size_t)i * (K / 32);
        } else {
          const size_t slot = (size_t)__ldg(Wd.slot_of + U.e);
          q = Wd.down_q + (slot * p.H + i) * (K / 2);
          sc = Wd.down_s + (slot * p.H + i) * (K / 32);
        }
        uint4 cc[kPrefetch];
        uint16_t cv[kPrefetch];
#pragma unroll
        for (int j = 0; j < kPrefetch; ++j) {
          if (j < nks) {
            cc[j] = ld_stream(q + j * 32 + part * 16);
            cv[j] = __ldg(sc + 2 * j + part);
          }
        }
        for (int ks0 = 0; ks0 < nks && alive; ks0 += kPrefetch) {
#pragma unroll
          for (int j = 0; j < kPrefetch; ++j) {
            const int ks = ks0 + j;
            if (ks < nks && alive) {
              const int s = it % kStages;
              bool ok = true;
              if (lane == 0) ok = mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, p.err, tmo);
              ok = __shfl_sync(0xffffffffu, ok, 0);
              if (!ok) {
                alive = false;
              } else {
                unsigned char* tile = smem + s * STAGE;
                const __half2 s2 = __half2half2(__ushort_as_half(cv[j]));
                st_tile_chunk(tile, r, part * 4 + 0, dequant_word(cc[j].x, s2));
                st_tile_chunk(tile, r, part * 4 + 1, dequant_word(cc[j].y, s2));
                st_tile_chunk(tile, r, part * 4 + 2, dequant_word(cc[j].z, s2));
                st_tile_chunk(tile, r, part * 4 + 3, dequant_word(cc[j].w, s2));
                fence_proxy_async_smem();
                mbar_arrive(&full_a[s]);
                ++it;
                if (ks + kPrefetch < nks) {
                  cc[j] = ld_stream(q + (ks + kPrefetch) * 32 + part * 16);
                  cv[j] = __ldg(sc + 2 * (ks + kPrefetch) + part);
                }
              }
            }
          }
        }
      } else {
        // router: rows are experts; K' = 2H; step ks < H/64 writes the fp16
        // "hi" term of w * 2^router_shift, later steps the "mid" remainder
        const int e = U.mt * 128 + r;
        const bool valid = e < p.E;
        const float* wrow = Wd.router_w + (size_t)(valid ? e : 0) * p.H;
        const float scale = pow2f(p.router_shift);
        const int kpp = p.H / 64;
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int pass = ks / kpp, kk = ks - pass * kpp;
          float4 v[8];
          const float4* src = reinterpret_cast<const float4*>(wrow + kk * 64 + part * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = valid ? __ldg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          const int s = it % kStages;
          bool ok = true;
          if (lane == 0) ok = mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, p.err, tmo);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            alive = false;
            break;
          }
          unsigned char* tile = smem + s * STAGE;
#pragma unroll
          for (int g = 0; g < 4; ++g) {  // 8-element group g of this half
            const float a[8] = {v[2 * g].x, v[2 * g].y, v[2 * g].z, v[2 * g].w,
                                v[2 * g + 1].x, v[2 * g + 1].y, v[2 * g + 1].z, v[2 * g + 1].w};
            uint32_t o[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {  // pair jj = (element jj, element jj + 4)
              const float w0 = a[jj] * scale, w1 = a[jj + 4] * scale;
              const __half h0 = __float2half_rn(w0), h1 = __float2half_rn(w1);
              __half2 hv;
              if (pass == 0)
                hv = __halves2half2(h0, h1);
              else
                hv = __halves2half2(__float2half_rn(w0 - __half2float(h0)),
                                    __float2half_rn(w1 - __half2float(h1)));
              o[jj] = *reinterpret_cast<uint32_t*>(&hv);
            }
            st_tile_chunk(tile, r, part * 4 + g, make_uint4(o[0], o[1], o[2], o[3]));
          }
          fence_proxy_async_smem();
          mbar_arrive(&full_a[s]);
        }
      }
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ B loaders
    uint32_t it = 0;
    bool alive = true;
    if (MODE == kSwiglu) {
      // lane l of B warp bw copies 16-byte chunk (l & 7) of rows
      // bw*RW + 4i + (l >> 3), i < RW/4: every warp instruction moves four
      // whole 128-byte rows.  A thread's copies of K step j form one async
      // group; it retires step j (wait, proxy fence, arrive) kBLag steps later.
      constexpr int RW = kNT / Roles<MODE>::kBWarps;  // rows per warp
      const int bw = warp - kBWarp0;
      const int c = lane & 7;
      for (int u = blockIdx.x; u < n_units && alive; u += gridDim.x) {
        const UnitInfo U = unit_info<MODE>(p, u);
        const int neff = (U.n + 15) & ~15;
        uint32_t src[RW / 4];  // element offset of the chunk in x16
        uint32_t dst[RW / 4];  // byte offset in the B tile, or ~0 if not loaded
#pragma unroll
        for (int i = 0; i < RW / 4; ++i) {
          const int row = bw * RW + 4 * i + (lane >> 3);
          int t = row < U.n ? row : U.n - 1;  // padding rows repeat a valid row
          const int tok = U.shared ? (U.p0 + t) : __ldg(p.perm_tok + U.p0 + t);
          src[i] = (uint32_t)tok * (uint32_t)p.H + (uint32_t)(c * 8);
          dst[i] = (row < neff) ? (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4)) : 0xffffffffu;
        }
        const int nks = U.K / 64;
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % kStages;
          bool ok = true;
          if (lane == 0) ok = mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, p.err, tmo);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            alive = false;
            break;
          }
          const uint32_t tile = smem_u32(smem + s * STAGE + NA * kTileA);
#pragma unroll
          for (int i = 0; i < RW / 4; ++i)
            if (dst[i] != 0xffffffffu) cp_async_16(tile + dst[i], p.x16 + src[i] + ks * 64);
          cp_async_commit();
          if (it >= (uint32_t)kBLag) {
            cp_async_wait<kBLag>();
            fence_proxy_async_smem();
            mbar_arrive(&full_b[(it - kBLag) % kStages]);
          }
        }
      }
      // every copy lands before the CTA can exit; retire the last steps
      cp_async_wait<0>();
      if (alive) {
        fence_proxy_async_smem();
        for (uint32_t q = it > (uint32_t)kBLag ? it - kBLag : 0u; q < it; ++q)
          mbar_arrive(&full_b[q % kStages]);
      }
    } else {
      if (lane == 0) {
        const int kpp = p.H / 64;
        for (int u = blockIdx.x; u < n_units && alive; u += gridDim.x) {
          const UnitInfo U = unit_info<MODE>(p, u);
          const CUtensorMap* tm = (MODE == kScatter) ? (U.shared ? &tm_hs : &tm_hr) : &tm_x;
          const int nks = U.K / 64;
          for (int ks = 0; ks < nks; ++ks, ++it) {
            const int s = it % kStages;
            if (!mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, p.err, tmo)) {
              alive = false;
              break;
            }
            mbar_expect_tx(&full_b[s], (uint32_t)kTileB);
            const int col = ((MODE == kRouter) ? (ks % kpp) : ks) * 64;
            tma_load_2d(smem + s * STAGE + NA * kTileA, tm, col, U.p0, &full_b[s]);
          }
        }
        // let every copy this thread issued land before the CTA can exit
        const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
        for (uint32_t q = first; q < it; ++q)
          mbar_wait(&full_b[q % kStages], (q / kStages) & 1, p.err, tmo);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0;
      int j = 0, committed = -1;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++j) {
        const UnitInfo U = unit_info<MODE>(p, u);
        const int neff = (U.n + 15) & ~15;
        const int b = j & 1;
        if (!mbar_wait(&tempty[b], ((j >> 1) & 1) ^ 1, p.err, tmo)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(b * 256), d1 = d0 + 128;
        const uint32_t idesc = idesc_f16_m128(neff);
        const int nks = U.K / 64;
        bool ok = true;
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&full_a[s], ph, p.err, tmo) || !mbar_wait(&full_b[s], ph, p.err, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * STAGE);
          const uint64_t da0 = smem_desc_sw128(sa);
          const uint64_t da1 = smem_desc_sw128(sa + kTileA);
          const uint64_t db = smem_desc_sw128(sa + NA * kTileA);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (ks | kk) ? 1u : 0u;
            umma_f16(d0, da0 + 2 * kk, db + 2 * kk, idesc, acc);
            if (NA == 2) umma_f16(d1, da1 + 2 * kk, db + 2 * kk, idesc, acc);
          }
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[b]);
        committed = j;
      }
      // Normally the epilogue has consumed every committed accumulator.  On
      // an error path, wait (bounded) for the last commit so that no MMA is
      // still writing TMEM when it is released.
      if (committed >= 0 && ld_relaxed_i32(p.err) != 0) {
        // the sticky error makes mbar_wait return at once: poll directly
        const uint64_t t0 = global_timer();
        while (!mbar_test(&tfull[committed & 1], (committed >> 1) & 1) &&
               global_timer() - t0 < tmo) {
        }
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- SIMT kernels

// x (bf16 [T][H]) -> x16 (fp16, row scaled by 2^-shift so max |x| in [1, 2),
// 8-groups reordered 0,4,1,5,2,6,3,7); one warp per token.
__global__ void prep_x16_kernel(const uint16_t* __restrict__ x, int T, int H,
                                __half* __restrict__ x16, int32_t* __restrict__ xshift) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  float m = 0.0f;
  for (int g = lane; g < H / 8; g += 32) {
    const uint4 v = row[g];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xffff0000u))));
  }
  m = warp_max(m);
  int s = 0;
  if (m > 0.0f && isfinite(m)) s = ((__float_as_int(m) >> 23) & 0xff) - 127;
  s = s < -60 ? -60 : (s > 60 ? 60 : s);
  if (lane == 0) xshift[t] = s;
  const float sc = pow2f(-s);
  uint4* out = reinterpret_cast<uint4*>(x16 + (size_t)t * H);
  for (int g = lane; g < H / 8; g += 32) {
    const uint4 v = row[g];
    float e[8];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e[2 * i] = __uint_as_float(w[i] << 16) * sc;
      e[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u) * sc;
    }
    uint32_t o[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      __half2 h = __floats2half2_rn(e[jj], e[jj + 4]);
      o[jj] = *reinterpret_cast<uint32_t*>(&h);
    }
    out[g] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void topk_kernel(const float* __restrict__ z, int T, int E, int k,
                            int32_t* __restrict__ ids, float* __restrict__ w, int* err) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  int id;
  float wt;
  const bool ok = warp_topk_softmax(z + (size_t)t * E, E, k, &id, &wt);
  if (!ok && lane == 0) atomicCAS(err, 0, (int)MOE_ERR_BOUNDS);
  if (lane < k) {
    ids[(size_t)t * k + lane] = id;
    w[(size_t)t * k + lane] = wt;
  }
}

struct BucketParams {
  const int32_t* ids;
  const float* w;
  int T, k, E, F, Fs, H;
  int32_t* offsets;
  int32_t* perm_tok;
  float* perm_w;
  int4* gu_units;
  int4* dn_units;
  int32_t* n_units;
  int* err;
};

// Exclusive block scan of one int per thread (1024 threads); returns the
// thread's prefix, *total receives the sum.
__device__ __forceinline__ int block_scan_1024(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    scratch[32 + lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  const int before = (warp ? scratch[32 + warp - 1] : 0) + x - v;
  *total = scratch[32 + 31];
  __syncthreads();
  return before;
}

// Stable counting sort of the T*k assignments by expert (then token), and
// the work-unit lists of the gate/up and down GEMMs.  One CTA of 1024
// threads; warp w owns a contiguous range of tokens.
__global__ void __launch_bounds__(kBucketThreads, 1) bucket_kernel(const BucketParams p) {
  extern __shared__ int sm[];
  const int E = p.E, k = p.k, T = p.T;
  int* hist = sm;                  // [32][E]: per-warp counts, then cursors
  int* tot = hist + 32 * E;        // [E]
  int* offs = tot + E;             // [E]
  int* tbase = offs + E;           // [E + 1]
  int* scratch = tbase + E + 1;    // [64]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (T + 31) / 32;
  const int t_begin = warp * per, t_end = min(T, t_begin + per);

  for (int i = tid; i < 32 * E; i += kBucketThreads) hist[i] = 0;
  __syncthreads();
  // per-warp histograms (a token's k ids are distinct: no lane conflicts)
  for (int t0 = t_begin; t0 < t_end; t0 += 16) {
    int col[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      col[i] = (lane < k && t0 + i < t_end) ? __ldg(p.ids + (size_t)(t0 + i) * k + lane) : -1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = col[i];
      if (e >= 0 && e < E) hist[warp * E + e] += 1;
      else if (lane < k && t0 + i < t_end) atomicCAS(p.err, 0, (int)MOE_ERR_BOUNDS);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kBucketThreads) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();
  // offsets and tile bases (E <= 1024: one expert per thread)
  {
    const int c = tid < E ? tot[tid] : 0;
    const int nt = (c + kNT - 1) / kNT;
    int total;
    const int off = block_scan_1024(c, scratch, &total);
    int ntiles;
    const int tb = block_scan_1024(nt, scratch, &ntiles);
    if (tid < E) {
      offs[tid] = off;
      tbase[tid] = tb;
      p.offsets[tid] = off;
    }
    if (tid == 0) {
      p.offsets[E] = total;
      tbase[E] = ntiles;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kBucketThreads)
    for (int w = 0; w < 32; ++w) hist[w * E + e] += offs[e];
  __syncthreads();
  // stable scatter: each warp walks its tokens in order
  for (int t0 = t_begin; t0 < t_end; t0 += 16) {
    int col[16];
    float wc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const bool in = lane < k && t0 + i < t_end;
      col[i] = in ? __ldg(p.ids + (size_t)(t0 + i) * k + lane) : -1;
      wc[i] = in ? __ldg(p.w + (size_t)(t0 + i) * k + lane) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = col[i];
      if (e >= 0 && e < E) {
        const int pos = hist[warp * E + e]++;
        p.perm_tok[pos] = t0 + i;
        p.perm_w[pos] = wc[i];
      }
      __syncwarp();
    }
  }
  // work units: routed tiles g -> (expert, tile) by binary search on tbase
  const int ntiles = tbase[E];
  const int mF = p.F / 128, mH = p.H / 128, mS = p.Fs / 128;
  for (int g = tid; g < ntiles; g += kBucketThreads) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {  // last e with tbase[e] <= g
      const int mid = (lo + hi + 1) >> 1;
      if (tbase[mid] <= g) lo = mid;
      else hi = mid - 1;
    }
    const int e = lo;
    const int i = g - tbase[e];
    const int p0 = offs[e] + i * kNT;
    const int n = min(kNT, tot[e] - i * kNT);
    for (int mt = 0; mt < mF; ++mt) p.gu_units[(size_t)g * mF + mt] = make_int4(e, p0, n, mt);
    for (int mt = 0; mt < mH; ++mt) p.dn_units[(size_t)g * mH + mt] = make_int4(e, p0, n, mt);
  }
  const int stiles = mS > 0 ? (T + kNT - 1) / kNT : 0;
  for (int g = tid; g < stiles; g += kBucketThreads) {
    const int p0 = g * kNT, n = min(kNT, T - p0);
    for (int mt = 0; mt < mS; ++mt)
      p.gu_units[(size_t)ntiles * mF + (size_t)g * mS + mt] = make_int4(E, p0, n, mt);
    for (int mt = 0; mt < mH; ++mt)
      p.dn_units[(size_t)(ntiles + g) * mH + mt] = make_int4(E, p0, n, mt);
  }
  if (tid == 0) {
    p.n_units[0] = ntiles * mF + stiles * mS;
    p.n_units[1] = (ntiles + stiles) * mH;
  }
}

__global__ void finalize_kernel(const float* __restrict__ yacc, size_t n, uint16_t* __restrict__ y) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    y[i] = __bfloat16_as_ushort(__float2bfloat16_rn(yacc[i]));
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct PrefillSizes {
  size_t x16, xshift, zf, ids, w, offsets, perm_tok, perm_w, gu, dn, nunits, hmid_r, hmid_s, yacc;
  int max_gu, max_dn;
  static PrefillSizes make(const moe_layer_config& c) {
    PrefillSizes s;
    const size_t Tm = (size_t)c.max_tokens, H = c.hidden, E = c.n_experts, k = c.top_k;
    const size_t F = c.ffn, Fs = c.shared_ffn;
    const size_t Tk = Tm * k;
    const size_t routed_tiles = (Tk + kNT - 1) / kNT + E;
    const size_t shared_tiles = Fs ? (Tm + kNT - 1) / kNT : 0;
    s.max_gu = (int)(routed_tiles * (F / 128) + shared_tiles * (Fs / 128));
    s.max_dn = (int)((routed_tiles + shared_tiles) * (H / 128));
    s.x16 = Tm * H * 2;
    s.xshift = Tm * 4;
    s.zf = Tm * E * 4;
    s.ids = Tk * 4;
    s.w = Tk * 4;
    s.offsets = (E + 1) * 4;
    s.perm_tok = Tk * 4;
    s.perm_w = Tk * 4;
    s.gu = (size_t)s.max_gu * 16;
    s.dn = (size_t)s.max_dn * 16;
    s.nunits = 16;
    s.hmid_r = Tk * F * 2;
    s.hmid_s = Tm * (Fs ? Fs : 128) * 2;
    s.yacc = Tm * H * 4;
    return s;
  }
  size_t total() const {
    return align256(x16) + align256(xshift) + align256(zf) + align256(ids) + align256(w) +
           align256(offsets) + align256(perm_tok) + align256(perm_w) + align256(gu) + align256(dn) +
           align256(nunits) + align256(hmid_r) + align256(hmid_s) + align256(yacc);
  }
};

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  }
  return fn;
}

// 2-D fp16 map [rows][cols], box {64, 128} (128 rows of 128 bytes: one
// K step of a B tile), 128B swizzle; rows past the end read as zero.
bool encode_rows(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kNT};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
moe_status launch_gemm(const GemmParams& gp, moe_layer* L, int grid, cudaStream_t s,
                       const char** why) {
  constexpr int NA = (MODE == kSwiglu) ? 2 : 1;
  const size_t smem = (size_t)kStages * (NA * kTileA + kTileB) + 1024 + 256 + 8 * kNT;
  auto kern = moe_gemm_kernel<MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    *why = "cudaFuncSetAttribute(gemm smem)";
    return MOE_ERR_CUDA;
  }
  static const char* const names[3] = {"moe_gemm_gateup_swiglu", "moe_gemm_down_scatter",
                                       "moe_gemm_router"};
  prof::Scope scope(names[MODE], s);
  kern<<<grid, Roles<MODE>::kThreads, smem, s>>>(gp, L->tmap_x16, L->tmap_hr, L->tmap_hs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace

size_t prefill_workspace_bytes(const moe_layer_config& c) { return PrefillSizes::make(c).total(); }

moe_status prefill_init(moe_layer* L, void* scratch, const char** why) {
  const moe_layer_config& c = L->cfg;
  const PrefillSizes z = PrefillSizes::make(c);
  char* p = static_cast<char*>(scratch);
  auto take = [&](size_t bytes) {
    char* r = p;
    p += align256(bytes);
    return r;
  };
  Workspace& w = L->ws;
  w.x16 = (__half*)take(z.x16);
  w.xshift = (int32_t*)take(z.xshift);
  w.zf = (float*)take(z.zf);
  w.topk_ids = (int32_t*)take(z.ids);
  w.topk_w = (float*)take(z.w);
  w.offsets = (int32_t*)take(z.offsets);
  w.perm_tok = (int32_t*)take(z.perm_tok);
  w.perm_w = (float*)take(z.perm_w);
  w.gu_units = (int4*)take(z.gu);
  w.dn_units = (int4*)take(z.dn);
  w.n_units = (int32_t*)take(z.nunits);
  w.hmid_r = (__half*)take(z.hmid_r);
  w.hmid_s = (__half*)take(z.hmid_s);
  w.yacc = (float*)take(z.yacc);
  w.max_gu_units = z.max_gu;
  w.max_dn_units = z.max_dn;
  const uint64_t Tm = c.max_tokens;
  const uint64_t Fs = c.shared_ffn ? c.shared_ffn : 128;
  if (!encode_rows(&L->tmap_x16, w.x16, c.hidden, Tm) ||
      !encode_rows(&L->tmap_hr, w.hmid_r, c.ffn, Tm * c.top_k) ||
      !encode_rows(&L->tmap_hs, w.hmid_s, Fs, Tm)) {
    *why = "cuTensorMapEncodeTiled failed (driver entry point unavailable?)";
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status launch_prefill(moe_layer* L, const uint16_t* x, int T, uint16_t* y, int32_t* ids_out,
                          float* w_out, bool route_only, cudaStream_t s, const char** why) {
  const moe_layer_config& c = L->cfg;
  const Workspace& ws = L->ws;
  const int H = c.hidden, E = c.n_experts, k = c.top_k;
  cudaError_t e;

  {
    prof::Scope sc("moe_prep_x16", s);
    prep_x16_kernel<<<(T + 7) / 8, 256, 0, s>>>(x, T, H, ws.x16, ws.xshift);
  }

  GemmParams gp;
  memset(&gp, 0, sizeof gp);
  gp.H = H;
  gp.E = E;
  gp.k = k;
  gp.F = c.ffn;
  gp.Fs = c.shared_ffn;
  gp.T = T;
  gp.Tk = T * k;
  gp.W = L->dev;
  gp.x16 = ws.x16;
  gp.perm_tok = ws.perm_tok;
  gp.perm_w = ws.perm_w;
  gp.xshift = ws.xshift;
  gp.hmid_r = ws.hmid_r;
  gp.hmid_s = ws.hmid_s;
  gp.yacc = ws.yacc;
  gp.z = ws.zf;
  gp.router_shift = L->router_shift;
  gp.err = ws.err;
  gp.timeout_ns = 1000000000ull;
  {
    const char* t = getenv("MOE_WAIT_TIMEOUT_US");
    if (t && *t && atoll(t) > 0) gp.timeout_ns = (unsigned long long)atoll(t) * 1000ull;
  }
  gp.n_units_router = ((T + kNT - 1) / kNT) * ((E + 127) / 128);
  moe_status st = launch_gemm<kRouter>(gp, L, std::min(gp.n_units_router, L->num_sms), s, why);
  if (st != MOE_OK) return st;

  int32_t* ids = (route_only && ids_out) ? ids_out : ws.topk_ids;
  float* wts = (route_only && w_out) ? w_out : ws.topk_w;
  {
    prof::Scope sc("moe_topk", s);
    topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(ws.zf, T, E, k, ids, wts, ws.err);
  }
  if (route_only) {
    if ((e = cudaGetLastError()) != cudaSuccess) {
      *why = cudaGetErrorString(e);
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  if (ids_out &&
      cudaMemcpyAsync(ids_out, ids, sizeof(int32_t) * T * k, cudaMemcpyDeviceToDevice, s) != cudaSuccess) {
    *why = "copy ids";
    return MOE_ERR_CUDA;
  }

  BucketParams bp;
  bp.ids = ids;
  bp.w = wts;
  bp.T = T;
  bp.k = k;
  bp.E = E;
  bp.F = c.ffn;
  bp.Fs = c.shared_ffn;
  bp.H = H;
  bp.offsets = ws.offsets;
  bp.perm_tok = ws.perm_tok;
  bp.perm_w = ws.perm_w;
  bp.gu_units = ws.gu_units;
  bp.dn_units = ws.dn_units;
  bp.n_units = ws.n_units;
  bp.err = ws.err;
  const size_t bsmem = sizeof(int) * (32 * (size_t)E + 3 * (size_t)E + 1 + 64);
  if (cudaFuncSetAttribute(bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bsmem) !=
      cudaSuccess) {
    *why = "cudaFuncSetAttribute(bucket smem)";
    return MOE_ERR_CUDA;
  }
  {
    prof::Scope sc("moe_bucket", s);
    bucket_kernel<<<1, kBucketThreads, bsmem, s>>>(bp);
  }

  gp.units = ws.gu_units;
  gp.n_units = ws.n_units;
  if ((st = launch_gemm<kSwiglu>(gp, L, L->num_sms, s, why)) != MOE_OK) return st;
  if ((e = cudaMemsetAsync(ws.yacc, 0, sizeof(float) * (size_t)T * H, s)) != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  gp.units = ws.dn_units;
  gp.n_units = ws.n_units + 1;
  if ((st = launch_gemm<kScatter>(gp, L, L->num_sms, s, why)) != MOE_OK) return st;
  {
    prof::Scope sc("moe_finalize", s);
    finalize_kernel<<<2 * L->num_sms, 256, 0, s>>>(ws.yacc, (size_t)T * H, y);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
