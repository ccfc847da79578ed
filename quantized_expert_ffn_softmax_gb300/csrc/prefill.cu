// Prefill path (5 or more tokens): bucketed grouped GEMMs on the tcgen05
// tensor cores.
//
//   prep       x (bf16) -> x16: fp16, scaled per token by a power of two so
//              the row maximum lies in [1, 2), K reordered inside every group
//              of 8 to the order in which packed 4-bit codes unpack
//   router     z = W_r x + b as one tcgen05 GEMM with K' = 2H: W_r * 2^shift
//              is split once, at layer creation, into two fp16 terms (hi +
//              mid, about 22 significant bits) so the logits keep
//              fp32-level accuracy for the exact top-k
//   top-k      one warp per token; softmax over the selected logits (or the
//              routing variants), and the gate weight of a gated shared
//              expert
//   bucket     stable counting sort of the (token, slot) assignments by
//              expert in three launches (chunk counts, one-CTA scans and the
//              work-unit lists, chunk scatter)
//   gather     the x16 row of every assignment, copied into bucket order
//              (operand B of the routed gate/up GEMM)
//   gate/up    per unit (expert, 128-token tile, 128-row F tile):
//              D_g, D_u = W_g/u[128 x H] . X[tokens]^T in TMEM, epilogue
//              h = w * silu(g) * u -> fp16 rows of Hmid (bucket order; w the
//              assignment's routing weight or the shared expert's gate)
//   down       per unit (expert, token tile, 256-row H tile as two 128-row
//              A matrices): D = W_d[256 x F] . Hmid[tokens]^T, epilogue
//              D as fp16 rows of a partial-output buffer (bucket order; the
//              shared expert's rows after the routed ones, in token order)
//   combine    per token, the sum of its k + 1 partial rows -> bf16 y (in a
//              prefill-sized stack, inside the layer-boundary kernel)
//
// GEMM engine: one persistent CTA per SM, warp-specialised.
//   warps 0-3   epilogue (TMEM lanes 0-127 = the 128 rows of the tile)
//   warps 4-11  A producers: dequantise 4-bit codes from the raw ring into
//               fp16 128x64 tiles written into tensor memory (tcgen05.st),
//               each thread reading its own row's block scales from global
//               memory four K steps per load; the router's A tiles come
//               ready-made by TMA instead
//   B loader    one warp, one elected lane issuing: the unit's contiguous
//               token rows (bucket order; the shared expert's in token
//               order) as one TMA tile per K step, 128-byte swizzled K-major
//   raw loader  one warp, one elected lane issuing: TMA tiles of packed
//               codes (128 rows x 32 bytes per matrix and K step) into a
//               raw ring
//   MMA warps   one warp per A matrix (gate/up and down: two; router: one),
//               one elected lane issuing tcgen05.mma, A from tensor memory,
//               B from shared memory; the first also allocates TMEM
// Every role runs its loop warp-wide and issues its tcgen05 and TMA
// instructions under elect.sync: issued from inside `if (lane == 0)` an
// MMA costs its thread about three times as long.  A stage ring (two
// stages of two K steps: the A slots in TMEM, two B tiles in shared memory)
// feeds the MMAs, one tcgen05.commit per stage and issuer.  The two
// 128-column accumulators fill TMEM's lower half; the epilogue stages the
// unit's output rows in shared memory and releases them early.
// Every wait is bounded and gives up once the error word is set.
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "device_common.cuh"
#include "moe_internal.cuh"
#include "profile.cuh"

namespace moe {

// cuTensorMapEncodeTiled from the driver (null when unavailable)
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
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

namespace {

using namespace dev;

constexpr int kNT = 128;           // token tile = largest MMA N used
constexpr int kTileA = 128 * 128;  // bytes: 128 rows x 64 fp16
constexpr int kTileB = kNT * 128;  // bytes: kNT rows x 64 fp16
constexpr int kRawTile = 128 * 32; // bytes: 128 rows x 64 packed 4-bit codes
constexpr int kEpiWarps = 4;
constexpr int kProdWarp0 = 4;
constexpr int kProdWarps = 8;
constexpr int kBWarp0 = 12;
constexpr int kBucketThreads = 1024;
constexpr int kMaxBucketChunks = 256;  // chunks of assignments in the bucketing

enum GemmMode : int { kSwiglu = 0, kScatter = 1, kRouter = 2 };

// Shared-memory rings and warp roles of one GEMM kernel.
//   stage ring  S stages, each NA dequantised fp16 128x64 tiles (MMA operand
//               A) and one fp16 kNTx64 token tile (operand B); full_a marks
//               the stage ready (the producer warps' arrivals and the B
//               tile's bytes; the router's A and B tiles both arrive by
//               TMA on full_b instead), one tcgen05.commit per K
//               step releases the whole stage
//   raw ring    SR stages of NA packed-code tiles, filled by TMA; the gate/up
//               and down GEMMs dequantise from it (the router GEMM reads its
//               fp32 weights directly and has no raw ring)
// Warps after the epilogue (0-3) and A producers (4-11): the B loader (one
// TMA tile of contiguous token rows per K step), the raw loader, and the
// MMA issuers.  At most 16 warps, so that no SM sub-partition holds more
// than four and a thread may use 128 registers.
template <int MODE>
struct Gemm {
  // gate/up and down stage their dequantised A tiles in tensor memory (the
  // MMA reads A from TMEM, B from shared memory); the router keeps A in
  // shared memory.  TMEM columns: accumulators from 0, A stages from kACol0.
  static constexpr bool kTmemA = (MODE != kRouter);
  // A matrices per unit: gate and up, or two 128-row tiles of W_d
  static constexpr int NA = (MODE == kRouter) ? 1 : 2;
  // K steps (of 64) per stage: gate/up and down take two, so that each MMA
  // issuer waits and commits once per 8 MMAs (its fixed cost per stage is
  // about as long as four MMAs of 128 tokens)
  static constexpr int KS = (MODE == kRouter) ? 1 : 2;
  static constexpr int S = (MODE == kRouter) ? 6 : 2;
  static constexpr int SR = (MODE == kRouter) ? 0 : (MODE == kScatter ? 11 : 12);
  static constexpr int SRb = SR > 0 ? SR : 1;  // barrier slots
  static constexpr int kAccBufs = (MODE == kRouter) ? 2 : 1;
  static constexpr int kAccCols = NA * 128;  // gate | up, or one accumulator
  static constexpr int kACol0 = 256;
  static constexpr int kACols = KS * NA * 32;  // per stage: 64 fp16 of K per matrix and step = 32 columns
  static_assert(kAccBufs * kAccCols <= kACol0, "accumulators below the A stages");
  static_assert(!kTmemA || kACol0 + S * kACols <= 512, "A stages fit in TMEM");
  static constexpr int kBWarps = 1;
  static constexpr int kRawWarp = kBWarp0 + kBWarps;
  // MMA issuers: one thread per A matrix, each in its own warp.  A thread
  // needs about 50 cycles to issue one tcgen05.mma, and an M128 x N128 x K16
  // MMA keeps the tensor core busy for 64: one thread issuing both the gate
  // and the up MMAs of a K step, plus its waits and commit, leaves the
  // tensor core idle a third of the time.  The first issuer warp also owns
  // the TMEM allocation.
  static constexpr int kMmaWarp = kRawWarp + (SR > 0 ? 1 : 0);
  static constexpr int kThreads = (kMmaWarp + NA) * 32;
  static constexpr int kRawBytes = NA * kRawTile;  // packed codes of the NA matrices
  static constexpr int kBOff = kTmemA ? 0 : NA * kTileA;       // B tile offset in a stage
  static constexpr int kStageBytes = kBOff + KS * kTileB;
  static constexpr int OFF_RAW = S * kStageBytes;
  static constexpr int OFF_BAR = OFF_RAW + SR * kRawBytes;
  static constexpr int kBarBytes = ((8 * (3 * S + 2 * SRb + 6) + 4) + 127) & ~127;
  static constexpr int OFF_META = OFF_BAR + kBarBytes;
  // gate/up and down: the unit's outputs staged as fp16 [128 or 256 rows of
  // the accumulators][kNT tokens] so the accumulators are released as soon
  // as they are read; the write-out transposes to token-major rows.  The
  // 16-byte chunks of a row are XOR-swizzled (stage_off) so that both the
  // drain's row-wise stores and the write-out's column-wise loads are free
  // of bank conflicts.
  static constexpr int kHRows = (MODE == kScatter) ? 256 : 128;
  static constexpr int kHStage = (MODE != kRouter) ? kHRows * kNT * 2 : 0;
  static constexpr int OFF_HST = OFF_META + 8 * kNT;
  static constexpr int kSmem = OFF_HST + kHStage + 1024;  // + slack for 1 KB alignment
  static_assert(kThreads <= 16 * 32, "at most 16 warps");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(OFF_META % 16 == 0, "token factors are read as 16-byte vectors");
  // producers take K steps in pairs (every K/64 is even: K is a multiple
  // of 128), halving the per-step waits and fences
  static constexpr int kGroup = (MODE == kRouter) ? 1 : 2;
  static_assert(MODE == kRouter || (kGroup == KS && SR >= 2 * kGroup), "a producer group fills one stage");
};

// Tensor maps of one GEMM launch.
struct GemmMaps {
  CUtensorMap a_routed[2];  // packed codes of the routed experts (gate, up | down)
  CUtensorMap a_shared[2];  // packed codes of the shared expert
  CUtensorMap b[2];         // B rows, routed | shared: gate/up xg, x16; down hmid_r, hmid_s; router x16
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
  __half* ypart;             // down: weighted partial output rows (routed, then shared)
  float* z;
  const float* gw;           // [T] shared-expert gate weights, or null (weight 1)
  int router_shift;
  int* err;
  unsigned long long timeout_ns;
};

struct UnitInfo {
  int e, p0, n, mt, K;
  bool shared;
};

template <int MODE>
__device__ __forceinline__ UnitInfo unit_from(const GemmParams& p, int4 v) {
  UnitInfo U;
  U.e = v.x;
  U.p0 = v.y;
  U.n = v.z;
  U.mt = v.w;
  U.shared = (v.x == p.E);
  U.K = (MODE == kSwiglu) ? p.H : (U.shared ? p.Fs : p.F);
  return U;
}
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
    U = unit_from<MODE>(p, p.units[u]);
  }
  return U;
}

// 8 packed 4-bit codes (one 32-bit word, elements 8j..8j+7) -> 8 fp16
// weights (code - 8) * scale, in the unpack order 0,4,1,5,2,6,3,7.  A nibble
// in bits 0-3 of a half word ORed into 1024.0 (0x6400) reads 1024 + n; one
// in bits 4-7 ORed into 64.0 (0x5400, mantissa step 1/16) reads 64 + n; a
// single shift by 8 brings the other two nibbles into those positions.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, __half2 s2) {
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 k72 = __halves2half2(__ushort_as_half(0x5480), __ushort_as_half(0x5480));
  const uint32_t w8 = w >> 8;
  uint32_t v[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x54005400u,
                   (w8 & 0x000F000Fu) | 0x64006400u, (w8 & 0x00F000F0u) | 0x54005400u};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __half2 h = __hmul2(__hsub2(*reinterpret_cast<__half2*>(&v[j]), (j & 1) ? k72 : k1032), s2);
    o[j] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// First block scale of weight row r of the A matrix `part` of a unit (gate
// or up of the F tile; the first or second 128 rows of the H tile) whose
// expert sits in `slot`, or null for rows past the matrix.
template <int MODE>
__device__ __forceinline__ const uint16_t* scale_row(const GemmParams& p, const UnitInfo& U, int slot, int part,
                                                     int r) {
  const LayerDev& W = p.W;
  const size_t C = (size_t)(U.K / 32);
  if (MODE == kSwiglu) {
    const size_t row = (U.shared ? 0 : (size_t)slot * p.F) + (size_t)U.mt * 128 + r;
    const uint16_t* base = part ? (U.shared ? W.sh_up_s : W.up_s) : (U.shared ? W.sh_gate_s : W.gate_s);
    return base + row * C;
  }
  const int h = U.mt * 256 + part * 128 + r;  // output row of W_d
  if (h >= p.H) return nullptr;                // second half of the last tile when H % 256 == 128
  const size_t row = (U.shared ? 0 : (size_t)slot * p.H) + h;
  return (U.shared ? W.sh_down_s : W.down_s) + row * C;
}

// The scale words (two fp16 each) of K steps s0..s0+3 of one row: one
// 16-byte load when aligned and whole, else one word per step that exists.
__device__ __forceinline__ uint4 load_scale_quad(const uint16_t* srow, int s0, int nks) {
  if (!srow) return make_uint4(0u, 0u, 0u, 0u);  // rows past the matrix: zero weights
  const uint16_t* q = srow + 2 * s0;
  if (s0 + 4 <= nks && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) return __ldg(reinterpret_cast<const uint4*>(q));
  const uint32_t* w = reinterpret_cast<const uint32_t*>(q);
  uint4 v = make_uint4(__ldg(w), 0u, 0u, 0u);
  if (s0 + 1 < nks) v.y = __ldg(w + 1);
  if (s0 + 2 < nks) v.z = __ldg(w + 2);
  if (s0 + 3 < nks) v.w = __ldg(w + 3);
  return v;
}

// Offset (fp16 elements) of chunk j (tokens 8j..8j+7) of staging row `row`:
// rows of kNT tokens, chunk slots XOR-swizzled by the row and the row's
// 8-group, so 8 consecutive rows writing one chunk, or 8 rows 8 apart
// reading one chunk, touch 8 different 16-byte bank groups.
__device__ __forceinline__ int stage_off(int row, int j) {
  return row * kNT + (((j & ~7) | ((j ^ row ^ (row >> 3)) & 7)) << 3);
}

template <int MODE>
__global__ void __launch_bounds__(Gemm<MODE>::kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ GemmMaps maps) {
  using G = Gemm<MODE>;
  constexpr int NA = G::NA, S = G::S, SR = G::SR;
  constexpr int kMmaWarp = G::kMmaWarp;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* sR = smem + G::OFF_RAW;   // SR stages x NA raw code tiles
  uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* full_b = full_a + S;
  uint64_t* empty = full_b + S;
  uint64_t* raw_full = empty + S;
  uint64_t* raw_empty = raw_full + G::SRb;
  uint64_t* tfull = raw_empty + G::SRb;
  uint64_t* tempty = tfull + 2;
  uint64_t* tdrain = tempty + 2;  // per MMA issuer: its own MMAs are complete (error path)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tdrain + 2);
  // per-unit token metadata of the epilogue: two words per token column
  int* meta_i = reinterpret_cast<int*>(smem + G::OFF_META);
  float* meta_f = reinterpret_cast<float*>(meta_i + kNT);
  __half* hst = reinterpret_cast<__half*>(smem + G::OFF_HST);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_a[s], kProdWarps + 1);  // + the B loader's arrive with the tile's bytes
      mbar_init(&full_b[s], 1);
      mbar_init(&empty[s], NA);  // one commit per MMA issuer
    }
    for (int s = 0; s < SR; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kProdWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], NA);
      mbar_init(&tempty[b], kEpiWarps * 32);
      mbar_init(&tdrain[b], 1);
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
          // D * 2^sx restores x; h is stored * w * 2^-2sx, i.e.
          // silu(g) * (D_u * w * 2^-sx): the routing weight w (or the shared
          // expert's gate) rides on u's factor, exactly (a power of two
          // times w), so that the down GEMM's output needs no factor; the
          // combine restores 2^2sx per token
          const int tok = U.shared ? (U.p0 + r) : __ldg(p.perm_tok + U.p0 + r);
          const int sx = __ldg(p.xshift + tok);
          const float w = U.shared ? (p.gw ? __ldg(p.gw + tok) : 1.0f) : __ldg(p.perm_w + U.p0 + r);
          meta_f[r] = pow2f(sx);
          reinterpret_cast<float*>(meta_i)[r] = pow2f(-sx) * w;
        } else if (MODE == kRouter) {
          meta_f[r] = pow2f(__ldg(p.xshift + U.p0 + r) - p.router_shift);
        }
      }
      const int b = (G::kAccBufs == 2) ? (j & 1) : 0;
      const uint32_t tpar = (G::kAccBufs == 2) ? ((j >> 1) & 1) : (j & 1);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[b], tpar, p.err, tmo));
      // meta is ready, and the four warps agree on whether to go on (the
      // break must be uniform: the named barriers wait for all of them)
      if (!named_bar_and(1, kEpiWarps * 32, ok)) break;
      tc_fence_after();
      const int neff = (U.n + 15) & ~15;
      const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * G::kAccCols);
      constexpr int CW = (NA == 2) ? 16 : 32;  // columns per TMEM load
      if constexpr (MODE == kSwiglu) {
        // drain: the next chunk's TMEM loads are issued before this chunk is
        // processed; per element one scale, SiLU, one product, one store
        const float* sA = meta_f;
        const float* sB = reinterpret_cast<const float*>(meta_i);
        uint32_t g0[CW], u0[CW];
        tmem_ld(tbase, g0);
        tmem_ld(tbase + 128, u0);
        tmem_wait_ld();
        for (int c0 = 0; c0 < neff; c0 += CW) {
          uint32_t g1[CW], u1[CW];
          const bool more = c0 + CW < neff;
          if (more) {
            tmem_ld(tbase + c0 + CW, g1);
            tmem_ld(tbase + 128 + c0 + CW, u1);
          }
          // the chunk's token factors are read into registers before its
          // first store: loads placed between the stores would each wait
          // for the stores before them (the compiler cannot rule out aliasing)
          float fa[CW], fb[CW];
#pragma unroll
          for (int q = 0; q < CW; q += 4) {
            const float4 va = *reinterpret_cast<const float4*>(sA + c0 + q);
            const float4 vb = *reinterpret_cast<const float4*>(sB + c0 + q);
            fa[q] = va.x, fa[q + 1] = va.y, fa[q + 2] = va.z, fa[q + 3] = va.w;
            fb[q] = vb.x, fb[q + 1] = vb.y, fb[q + 2] = vb.z, fb[q + 3] = vb.w;
          }
          __half2 hv[CW / 2];
#pragma unroll
          for (int jj = 0; jj < CW; jj += 2) {  // tokens t, t+1 as one half2
            const __half2 g = __floats2half2_rn(__uint_as_float(g0[jj]) * fa[jj],
                                                __uint_as_float(g0[jj + 1]) * fa[jj + 1]);
            const __half2 u = __floats2half2_rn(__uint_as_float(u0[jj]) * fb[jj],
                                                __uint_as_float(u0[jj + 1]) * fb[jj + 1]);
            hv[jj / 2] = __hmul2(silu_fast2(g), u);
          }
          static_assert(CW == 16, "two 16-byte stores per chunk");
          *reinterpret_cast<uint4*>(hst + stage_off(r, c0 >> 3)) = *reinterpret_cast<const uint4*>(&hv[0]);
          *reinterpret_cast<uint4*>(hst + stage_off(r, (c0 >> 3) + 1)) = *reinterpret_cast<const uint4*>(&hv[4]);
          if (more) {
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < CW; ++jj) {
              g0[jj] = g1[jj];
              u0[jj] = u1[jj];
            }
          }
        }
      } else if constexpr (MODE == kScatter) {
        // drain: D of both 128-row halves (the SwiGLU rows already carry the
        // routing weight) as fp16 into the staging rows [token][256]; the
        // next chunk's TMEM loads are issued before this chunk is processed
        uint32_t v0[CW], v1[CW];
        tmem_ld(tbase, v0);
        tmem_ld(tbase + 128, v1);
        tmem_wait_ld();
        for (int c0 = 0; c0 < neff; c0 += CW) {
          uint32_t n0[CW], n1[CW];
          const bool more = c0 + CW < neff;
          if (more) {
            tmem_ld(tbase + c0 + CW, n0);
            tmem_ld(tbase + 128 + c0 + CW, n1);
          }
          __half2 a[CW / 2], c[CW / 2];
#pragma unroll
          for (int jj = 0; jj < CW; jj += 2) {
            a[jj / 2] = __floats2half2_rn(__uint_as_float(v0[jj]), __uint_as_float(v0[jj + 1]));
            c[jj / 2] = __floats2half2_rn(__uint_as_float(v1[jj]), __uint_as_float(v1[jj + 1]));
          }
          static_assert(CW == 16, "two 16-byte stores per chunk and half");
          *reinterpret_cast<uint4*>(hst + stage_off(r, c0 >> 3)) = *reinterpret_cast<const uint4*>(&a[0]);
          *reinterpret_cast<uint4*>(hst + stage_off(r, (c0 >> 3) + 1)) = *reinterpret_cast<const uint4*>(&a[4]);
          *reinterpret_cast<uint4*>(hst + stage_off(128 + r, c0 >> 3)) = *reinterpret_cast<const uint4*>(&c[0]);
          *reinterpret_cast<uint4*>(hst + stage_off(128 + r, (c0 >> 3) + 1)) = *reinterpret_cast<const uint4*>(&c[4]);
          if (more) {
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < CW; ++jj) {
              v0[jj] = n0[jj];
              v1[jj] = n1[jj];
            }
          }
        }
      } else {
        for (int c0 = 0; c0 < neff; c0 += CW) {
          uint32_t v0[CW];
          tmem_ld(tbase + c0, v0);
          tmem_wait_ld();
          // per 16 tokens: factors into registers first, then the stores (a
          // shared load after a global store through a generic pointer
          // would have to wait for it)
#pragma unroll
          for (int hq = 0; hq < CW; hq += 16) {
            float tf[16];
#pragma unroll
            for (int q = 0; q < 16; q += 4) {
              const float4 vf = *reinterpret_cast<const float4*>(meta_f + c0 + hq + q);
              tf[q] = vf.x, tf[q + 1] = vf.y, tf[q + 2] = vf.z, tf[q + 3] = vf.w;
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int t = c0 + hq + jj;
              const int e = U.mt * 128 + r;
              if (t < U.n && e < p.E)
                p.z[(size_t)(U.p0 + t) * p.E + e] = __uint_as_float(v0[hq + jj]) * tf[jj] + bias_r;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[b]);
      if (MODE != kRouter) {
        // write the staged rows out (16-byte stores) while the MMAs of the
        // next unit already run in the released accumulator
        named_bar_sync(2, kEpiWarps * 32);
        size_t hstride;
        __half* hbase;
        int nch;  // 16-byte chunks of a token's output row
        if (MODE == kSwiglu) {
          hstride = U.shared ? (size_t)p.Fs : (size_t)p.F;
          hbase = (U.shared ? p.hmid_s : p.hmid_r) + (size_t)U.p0 * hstride + U.mt * 128;
          nch = 16;
        } else {
          hstride = (size_t)p.H;
          hbase = p.ypart + ((size_t)(U.shared ? p.Tk : 0) + U.p0) * hstride + U.mt * 256;
          nch = (U.mt * 256 + 256 <= p.H) ? 32 : 16;  // only the first half exists past H
        }
        // 8 x 8 blocks (staging rows 8c..8c+7, tokens 8tb..8tb+7): eight
        // 16-byte shared loads, a transpose in registers, and one 16-byte
        // output chunk per token.  Gate/up: row 8c+i goes to position
        // 8c + (0,2,4,6,1,3,5,7)[i], the unpack order of the down GEMM's K,
        // so output word j pairs rows j and j+4; down: rows 2j and 2j+1.
        // Consecutive lanes take consecutive chunks c of the same tokens, so
        // each warp store writes whole contiguous row segments.
        const int ntb = (U.n + 7) >> 3;
        for (int blk = r; blk < nch * ntb; blk += kEpiWarps * 32) {
          const int c = blk % nch, tb = blk / nch;
          uint4 rows[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            rows[i] = *reinterpret_cast<const uint4*>(hst + stage_off(8 * c + i, tb));
#pragma unroll
          for (int tt = 0; tt < 8; ++tt) {
            const int t = 8 * tb + tt;
            if (t >= U.n) break;
            const uint32_t sel = (tt & 1) ? 0x7632u : 0x5410u;
            uint32_t w[4];
#pragma unroll
            for (int jw = 0; jw < 4; ++jw) {
              const int ra = (MODE == kSwiglu) ? jw : 2 * jw, rb = (MODE == kSwiglu) ? jw + 4 : 2 * jw + 1;
              const uint32_t* pa = reinterpret_cast<const uint32_t*>(&rows[ra]);
              const uint32_t* pb = reinterpret_cast<const uint32_t*>(&rows[rb]);
              w[jw] = __byte_perm(pa[tt >> 1], pb[tt >> 1], sel);
            }
            *reinterpret_cast<uint4*>(hbase + (size_t)t * hstride + c * 8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  } else if (warp < kProdWarp0 + kProdWarps) {
    // ------------------------------------------------------------ A producers
    const int pi = threadIdx.x - kProdWarp0 * 32;  // 0..255
    uint32_t it = 0;
    bool alive = true;
    // (the router GEMM has no A producers: its A tiles arrive by TMA)
    if constexpr (MODE != kRouter) {
      // thread = (part, row r), r = 32*(warp%4) + lane: the TMEM lane it
      // writes (a warp reaches only its own quarter of the 128 lanes)
      // and part = the A matrix (gate or up; the first or second 128 rows of
      // the down GEMM's H tile), all 64 K of the step
      // Codes come from the raw ring (one TMA tile per matrix and step).
      // K steps go in groups of P (nks is even): one set of waits and one
      // round of hand-backs per group.  Per group: the raw stages' words
      // into registers (every lane waits for the stage itself, so that its
      // own reads follow the TMA's completion), the raw stages handed back
      // at once (after a proxy fence), the dequantisation, and only then the
      // wait for free A stages: the dequantisation overlaps the MMAs still
      // reading them.
      const int r = 32 * (warp & 3) + lane;
      const int part = pi >> 7;
      const int h = (r >> 2) & 1;  // the swizzle bit of row r in a raw tile
      constexpr int P = G::kGroup;
      constexpr int OW = 32;  // TMEM columns per thread and step: 64 fp16
      // This row's block scales: one 32-bit word (two fp16) per K step, read
      // four steps at a time, a quad ahead of their use; the next unit's
      // first quad during the current unit's last one.  The next unit's
      // descriptor is read at the start of a unit and its expert's slot one
      // quad later, so that no chain of dependent loads stalls a unit start.
      int nks = 0;
      const uint16_t* srow = nullptr;
      uint4 sq = make_uint4(0u, 0u, 0u, 0u);
      if ((int)blockIdx.x < n_units) {
        const UnitInfo U0 = unit_info<MODE>(p, blockIdx.x);
        nks = U0.K / 64;
        srow = scale_row<MODE>(p, U0, U0.shared ? 0 : __ldg(p.W.slot_of + U0.e), part, r);
        sq = load_scale_quad(srow, 0, nks);
      }
      for (int u = blockIdx.x; u < n_units && alive; u += gridDim.x) {
        const bool has_next = u + (int)gridDim.x < n_units;
        const int4 vn = has_next ? p.units[u + gridDim.x] : make_int4(0, 0, 0, 0);
        int slot_n = 0, nks_n = 0;
        const uint16_t* srow_n = nullptr;
        for (int ks0 = 0; ks0 < nks && alive; ks0 += 4) {
          const bool last = ks0 + 4 >= nks;
          if (has_next && (ks0 == 4 || (last && ks0 < 4)))
            slot_n = (vn.x == p.E) ? 0 : __ldg(p.W.slot_of + vn.x);
          uint4 sn = sq;
          if (!last) {
            sn = load_scale_quad(srow, ks0 + 4, nks);
          } else if (has_next) {
            const UnitInfo Un = unit_from<MODE>(p, vn);
            nks_n = Un.K / 64;
            srow_n = scale_row<MODE>(p, Un, slot_n, part, r);
            sn = load_scale_quad(srow_n, 0, nks_n);
          }
          const uint32_t sqw[4] = {sq.x, sq.y, sq.z, sq.w};
#pragma unroll
          for (int dd = 0; dd < 4; dd += P) {
            if (ks0 + dd >= nks || !alive) break;
            bool ok = true;
            uint4 ca[P], cb[P];
#pragma unroll
            for (int q = 0; q < P; ++q) {
              const uint32_t iq = it + q;
              const int sr = iq % SR;
              if (ok) ok = mbar_wait(&raw_full[sr], (iq / SR) & 1, p.err, tmo);
              ok = __all_sync(0xffffffffu, ok);
              if (ok) {
                // row r's first 16 bytes sit at 16 h, its second at 16 (h ^ 1)
                // (the tile's 32-byte swizzle)
                const unsigned char* rs = sR + sr * G::kRawBytes + part * kRawTile + r * 32;
                ca[q] = *reinterpret_cast<const uint4*>(rs + 16 * h);
                cb[q] = *reinterpret_cast<const uint4*>(rs + 16 * (h ^ 1));
              }
            }
            if (!ok) {
              alive = false;
              break;
            }
            // the stages were read through the generic proxy and are refilled
            // by TMA (async proxy): fence before handing them back
            fence_proxy_async_smem();
            __syncwarp();
            if (elect_one())
#pragma unroll
              for (int q = 0; q < P; ++q) mbar_arrive(&raw_empty[(it + q) % SR]);
            __syncwarp();
            uint32_t o[P][OW];
#pragma unroll
            for (int q = 0; q < P; ++q) {
              const __half2 slo = __half2half2(__ushort_as_half((uint16_t)(sqw[dd + q] & 0xffffu)));
              const __half2 shi = __half2half2(__ushort_as_half((uint16_t)(sqw[dd + q] >> 16)));
              const uint32_t wds[8] = {ca[q].x, ca[q].y, ca[q].z, ca[q].w,
                                       cb[q].x, cb[q].y, cb[q].z, cb[q].w};
#pragma unroll
              for (int w = 0; w < 8; ++w) {
                const uint4 d = dequant_word(wds[w], w < 4 ? slo : shi);
                o[q][4 * w] = d.x;
                o[q][4 * w + 1] = d.y;
                o[q][4 * w + 2] = d.z;
                o[q][4 * w + 3] = d.w;
              }
            }
            const uint32_t bs = it / G::KS;  // the group's stage
            ok = __all_sync(0xffffffffu, mbar_wait(&empty[bs % S], ((bs / S) & 1) ^ 1, p.err, tmo));
            if (!ok) {
              alive = false;
              break;
            }
            tc_fence_after();  // the MMAs that read these A stages are complete
            const uint32_t arow = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)G::kACol0;
#pragma unroll
            for (int q = 0; q < P; ++q) {
              const uint32_t acol = arow + (uint32_t)((bs % S) * G::kACols + q * NA * 32) + (uint32_t)(part * OW);
              tmem_st32(acol, o[q]);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();  // the warp's stores are complete: one arrive for the warp
            if (elect_one()) mbar_arrive(&full_a[bs % S]);
            __syncwarp();
            it += P;
          }
          sq = sn;
        }
        nks = nks_n;
        srow = srow_n;
      }
    }
  } else if (warp < G::kRawWarp) {
    // ------------------------------------------------------------ B loader
    // One TMA tile (kNT rows x 64 fp16) per K step at the unit's first row:
    // gate/up reads the bucket-ordered copy of x16 (routed units) or x16
    // (shared expert), down the SwiGLU rows, the router x16 and, on the
    // same barrier, its A tile.  Rows past a unit's end belong to the next
    // unit (or read as zero past the buffer); their columns are discarded.
    // The warp runs the loop (warp-uniform waits and exits); one elected
    // lane issues the copies.
    uint32_t it = 0;
    bool alive = true;
    uint64_t* fulls = (MODE == kRouter) ? full_b : full_a;  // the stage's ready barriers
    const int kpp = p.H / 64;
    for (int u = blockIdx.x; u < n_units && alive; u += gridDim.x) {
      const UnitInfo U = unit_info<MODE>(p, u);
      const CUtensorMap* tm = (MODE == kRouter) ? &maps.b[0] : &maps.b[U.shared ? 1 : 0];
      const int nks = U.K / 64;
      for (int ks = 0; ks < nks; ++ks, ++it) {
        const uint32_t bs = it / G::KS, sub = it % G::KS;  // stage, K step within it
        const int st = bs % S;
        uint64_t* fullb = &fulls[st];
        if (sub == 0 && !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((bs / S) & 1) ^ 1, p.err, tmo))) {
          alive = false;
          break;
        }
        if (elect_one()) {
          if (sub == 0) {
            if (MODE == kRouter) {
              // router: the A tile (fp16 hi | mid router weights) rides on the same barrier
              mbar_expect_tx(fullb, (uint32_t)(kTileA + kTileB));
              tma_load_2d(smem + st * G::kStageBytes, &maps.a_routed[0], ks * 64, U.mt * 128, fullb);
            } else {
              mbar_expect_tx(fullb, (uint32_t)(G::KS * kTileB));  // the stage's K steps
            }
          }
          const int col = ((MODE == kRouter) ? (ks % kpp) : ks) * 64;
          tma_load_2d(smem + st * G::kStageBytes + G::kBOff + sub * kTileB, tm, col, U.p0, fullb);
        }
        __syncwarp();
      }
    }
    // let every copy this warp issued land before the CTA can exit
    const uint32_t nst = (it + G::KS - 1) / G::KS;
    const uint32_t first = nst > (uint32_t)S ? nst - S : 0u;
    for (uint32_t q = first; q < nst; ++q) drain_wait(&fulls[q % S], (q / S) & 1, tmo);
    __syncwarp();
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ raw loader
    // Per K step: one TMA tile of packed codes (128 rows x 32 bytes) per
    // matrix into the raw ring.  (The block scales are read by the
    // producers themselves, four K steps per load.)  The warp runs the
    // loop; one elected lane issues the copies.
    if constexpr (SR > 0) {
      uint32_t it = 0;
      bool alive = true;
      const LayerDev& Wd = p.W;
      for (int u = blockIdx.x; u < n_units && alive; u += gridDim.x) {
        const UnitInfo U = unit_info<MODE>(p, u);
        const int slot = U.shared ? 0 : __ldg(Wd.slot_of + U.e);
        const int rows_per_slot = (MODE == kSwiglu) ? p.F : p.H;
        // gate/up: both matrices at the F tile's rows; down: the two
        // 128-row halves of the 256-row H tile (past H: the next expert's
        // rows or zero fill, never used)
        const int row = (U.shared ? 0 : slot * rows_per_slot) + U.mt * (MODE == kScatter ? 256 : 128);
        const int row1 = (MODE == kScatter) ? row + 128 : row;
        const CUtensorMap* m0 = U.shared ? &maps.a_shared[0] : &maps.a_routed[0];
        const CUtensorMap* m1 = U.shared ? &maps.a_shared[1] : &maps.a_routed[1];
        const int nks = U.K / 64;
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int sr = it % SR;
          if (!__all_sync(0xffffffffu, mbar_wait(&raw_empty[sr], ((it / SR) & 1) ^ 1, p.err, tmo))) {
            alive = false;
            break;
          }
          if (elect_one()) {
            unsigned char* dst = sR + sr * G::kRawBytes;
            mbar_expect_tx(&raw_full[sr], (uint32_t)(NA * kRawTile));
            tma_load_2d(dst, m0, ks * 32, row, &raw_full[sr]);
            if (NA == 2) tma_load_2d(dst + kRawTile, m1, ks * 32, row1, &raw_full[sr]);
          }
          __syncwarp();
        }
      }
      const uint32_t first = it > (uint32_t)SR ? it - SR : 0u;
      for (uint32_t q = first; q < it; ++q) drain_wait(&raw_full[q % SR], (q / SR) & 1, tmo);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ MMA issuers
    // Issuer m (warp kMmaWarp + m) issues the MMAs of A matrix m (gate or
    // up; the only matrix of down and router) into accumulator column block
    // m.  Both wait for the same stages; a stage is released, and an
    // accumulator published, when every issuer has committed.  The whole
    // warp runs the loop and waits on the barriers (the exits stay
    // warp-uniform); one elected lane issues the MMAs and the commits (the
    // same lane every time: a commit tracks its own thread's MMAs).
    const int m = warp - kMmaWarp;
    uint32_t it = 0;
    int j = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++j) {
      const UnitInfo U = unit_info<MODE>(p, u);
      const int neff = (U.n + 15) & ~15;
      const int b = (G::kAccBufs == 2) ? (j & 1) : 0;
      const uint32_t tpar = (G::kAccBufs == 2) ? ((j >> 1) & 1) : (j & 1);
      if (!__all_sync(0xffffffffu, mbar_wait(&tempty[b], tpar ^ 1, p.err, tmo))) break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(b * G::kAccCols + 128 * m);
      const uint32_t idesc = idesc_f16_m128(neff);
      const int nks = U.K / 64;
      bool ok = true;
      for (int ks = 0; ks < nks; ++ks, ++it) {
        const uint32_t bs = it / G::KS, sub = it % G::KS;  // stage, K step within it
        const int st = bs % S;
        if (sub == 0) {
          if (!__all_sync(0xffffffffu,
                          mbar_wait(MODE == kRouter ? &full_b[st] : &full_a[st], (bs / S) & 1, p.err, tmo))) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const uint32_t s_addr = smem_u32(smem + st * G::kStageBytes);
        const uint64_t db = smem_desc_sw128(s_addr + G::kBOff + sub * kTileB);
        if (elect_one()) {
          if constexpr (G::kTmemA) {
            const uint32_t a0 = tmem + (uint32_t)(G::kACol0 + st * G::kACols + sub * NA * 32 + 32 * m);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 16 K = 8 TMEM columns per MMA
              umma_f16_ts(d, a0 + 8 * kk, db + 2 * kk, idesc, (ks | kk) ? 1u : 0u);
          } else {
            const uint64_t da0 = smem_desc_sw128(s_addr);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_f16(d, da0 + 2 * kk, db + 2 * kk, idesc, (ks | kk) ? 1u : 0u);
          }
          if (sub == G::KS - 1) umma_commit(&empty[st]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) umma_commit(&tfull[b]);
      __syncwarp();
    }
    // Normally the epilogue has consumed every committed accumulator.  On
    // an error path, wait (bounded) until this warp's MMAs are complete, so
    // that none still writes TMEM when it is released.
    if (__any_sync(0xffffffffu, ld_relaxed_i32(p.err) != 0)) {
      if (elect_one()) umma_commit(&tdrain[m]);
      __syncwarp();
      drain_wait(&tdrain[m], 0, tmo);
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

// Top-k of one token's E logits held by one warp (logit e in lane e % 32,
// slot e / 32; NJ = slots per lane, E <= 32 NJ), descending by value, ties
// to the lower expert id; then the softmax weights.  Each lane keeps the
// best logit it has not given away; per round the warp takes the maximum of
// the 32 lane bests and only the winning lane rescans its slots.  Lane r < k
// receives id and weight r.  Returns false if a non-finite logit left no
// valid candidate.  Routing variants: with bsel (the bias, which then only
// selects) the weights use z_e - bsel[e]; with renorm false they are the
// softmax over all E such values, taken at the selection, instead of the
// softmax over the selection.
template <int NJ>
__device__ __forceinline__ bool warp_topk_softmax(const float* z, int E, int k, const float* bsel,
                                                  bool renorm, int* id_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  float v[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? z[e] : -INFINITY;
  }
  uint32_t taken = 0;
  // this lane's best slot not yet taken (ties: lower slot = lower id)
  auto lane_best = [&](float& bv, int& bi) {
    bv = -INFINITY;
    bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < bi))) {
        bv = v[j];
        bi = e;
      }
    }
  };
  float lv;
  int li;
  lane_best(lv, li);
  int my_id = 0;
  float my_z = 0.0f, z0 = 0.0f;
  bool ok = true;
  for (int r = 0; r < k; ++r) {
    float bv = lv;
    int bi = li;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi < 0 || bi >= E) {  // only reachable with non-finite logits
      ok = false;
      bi = r;
    }
    if ((bi & 31) == lane) {
      taken |= 1u << (bi >> 5);
      lane_best(lv, li);
    }
    if (r == 0) z0 = bv;
    if (lane == r) {
      my_id = bi;
      my_z = bv;
    }
  }
  const float base = (bsel && lane < k) ? my_z - __ldg(bsel + my_id) : my_z;
  float m = z0, den;
  if (renorm) {
    if (bsel) m = warp_max(lane < k ? base : -INFINITY);
    den = warp_sum(lane < k ? __expf(base - m) : 0.0f);
  } else {
    float mm = -INFINITY;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < E) mm = fmaxf(mm, v[j] - (bsel ? __ldg(bsel + e) : 0.0f));
    }
    m = warp_max(mm);
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < E) acc += __expf(v[j] - (bsel ? __ldg(bsel + e) : 0.0f) - m);
    }
    den = warp_sum(acc);
  }
  const float ex = (lane < k) ? __expf(base - m) : 0.0f;
  *id_out = my_id;
  *w_out = ex / den;
  return ok;
}

// One warp per token: top-k and routing weights (with the layer's routing
// variants: bsel = the bias when it only selects, renorm), and, for a gated
// shared expert, gw[t] = sigmoid(gate . x_t) over the bf16 input row.
template <int NJ>
__global__ void topk_kernel(const float* __restrict__ z, int T, int E, int k,
                            const float* __restrict__ bsel, int renorm,
                            const float* __restrict__ gate, const uint16_t* __restrict__ x, int H,
                            float* __restrict__ gw, int32_t* __restrict__ ids,
                            float* __restrict__ w, int* err) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  int id;
  float wt;
  const bool ok = warp_topk_softmax<NJ>(z + (size_t)t * E, E, k, bsel, renorm != 0, &id, &wt);
  if (!ok && lane == 0) atomicCAS(err, 0, (int)MOE_ERR_BOUNDS);
  if (lane < k) {
    ids[(size_t)t * k + lane] = id;
    w[(size_t)t * k + lane] = wt;
  }
  if (gate) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const float4* gr = reinterpret_cast<const float4*>(gate);
    float acc = 0.0f;
    for (int g = lane; g < H / 8; g += 32) {
      const uint4 xv = __ldg(xr + g);
      const float4 g0 = __ldg(gr + 2 * g), g1 = __ldg(gr + 2 * g + 1);
      acc = fmaf(g0.x, __uint_as_float(xv.x << 16), acc);
      acc = fmaf(g0.y, __uint_as_float(xv.x & 0xffff0000u), acc);
      acc = fmaf(g0.z, __uint_as_float(xv.y << 16), acc);
      acc = fmaf(g0.w, __uint_as_float(xv.y & 0xffff0000u), acc);
      acc = fmaf(g1.x, __uint_as_float(xv.z << 16), acc);
      acc = fmaf(g1.y, __uint_as_float(xv.z & 0xffff0000u), acc);
      acc = fmaf(g1.z, __uint_as_float(xv.w << 16), acc);
      acc = fmaf(g1.w, __uint_as_float(xv.w & 0xffff0000u), acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) gw[t] = 1.0f / (1.0f + __expf(-acc));
  }
}

struct BucketParams {
  const int32_t* ids;
  const float* w;
  int T, k, E, F, Fs, H;
  int nc;            // chunks of the (token, slot) assignments, in order
  int32_t* ccount;   // [nc][E] per-chunk counts, then per-chunk bases (before offsets)
  int32_t* offsets;
  int32_t* perm_tok;
  float* perm_w;
  int32_t* pos;      // [T*k] bucket position of each assignment, -1 if its id is invalid
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

// Stable counting sort of the T*k assignments (t, j), taken in the order
// t*k + j, by expert; and the work-unit lists of the two GEMMs.  Three
// launches: per-chunk counts (one warp per chunk of consecutive
// assignments), one CTA for the scans and the unit lists, and the stable
// scatter (one warp per chunk; equal experts within a 32-assignment step
// take consecutive positions in lane order).
__device__ __forceinline__ void chunk_range(const BucketParams& p, int c, int* a_begin, int* a_end) {
  const long long n = (long long)p.T * p.k;
  *a_begin = (int)(n * c / p.nc);
  *a_end = (int)(n * (c + 1) / p.nc);
}

__global__ void __launch_bounds__(32) bucket_count_kernel(const BucketParams p) {
  extern __shared__ int h[];  // [E]
  const int E = p.E, lane = threadIdx.x, c = blockIdx.x;
  for (int i = lane; i < E; i += 32) h[i] = 0;
  __syncwarp();
  int a_begin, a_end;
  chunk_range(p, c, &a_begin, &a_end);
  for (int a = a_begin + lane; a < a_end; a += 32) {
    const int e = __ldg(p.ids + a);
    if (e >= 0 && e < E) atomicAdd(&h[e], 1);
    else atomicCAS(p.err, 0, (int)MOE_ERR_BOUNDS);
  }
  __syncwarp();
  for (int i = lane; i < E; i += 32) p.ccount[(size_t)c * E + i] = h[i];
}

__global__ void __launch_bounds__(32) bucket_scatter_kernel(const BucketParams p) {
  extern __shared__ int cur[];  // [E]: next position of each expert in this chunk
  const int E = p.E, k = p.k, lane = threadIdx.x, c = blockIdx.x;
  for (int i = lane; i < E; i += 32) cur[i] = p.ccount[(size_t)c * E + i] + p.offsets[i];
  __syncwarp();
  int a_begin, a_end;
  chunk_range(p, c, &a_begin, &a_end);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int a0 = a_begin; a0 < a_end; a0 += 32) {
    const int a = a0 + lane;
    int e = (a < a_end) ? __ldg(p.ids + a) : -1;
    const float wv = (a < a_end) ? __ldg(p.w + a) : 0.0f;
    if (e >= E) e = -1;
    if (e < 0 && a < a_end) p.pos[a] = -1;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    int base = 0;
    if (e >= 0) base = cur[e];
    __syncwarp();
    if (e >= 0) {
      const int pos = base + __popc(same & lt_mask);
      p.perm_tok[pos] = a / k;
      p.perm_w[pos] = wv;
      p.pos[a] = pos;
      if ((same & lt_mask) == 0) cur[e] = base + __popc(same);
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kBucketThreads, 1) bucket_scan_kernel(const BucketParams p) {
  extern __shared__ int sm[];
  const int E = p.E, T = p.T;
  int* tot = sm;                   // [E]
  int* offs = tot + E;             // [E]
  int* tbase = offs + E;           // [E + 1]
  int* scratch = tbase + E + 1;    // [64]
  const int tid = threadIdx.x;
  // per expert: exclusive scan over the chunks (chunk bases) and the total
  for (int e = tid; e < E; e += kBucketThreads) {
    int run = 0;
    for (int c0 = 0; c0 < p.nc; c0 += 8) {  // 8 loads in flight per step
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (c0 + i < p.nc) ? p.ccount[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (c0 + i < p.nc) p.ccount[(size_t)(c0 + i) * E + e] = run;
        run += v[i];
      }
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
  // work units: routed tiles g -> (expert, tile) by binary search on tbase
  const int ntiles = tbase[E];
  const int mF = p.F / 128, mH = (p.H + 255) / 256, mS = p.Fs / 128;  // down: 256-row H tiles
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

// Operand B of the routed gate/up GEMM: the x16 row of every bucketed
// (token, expert) assignment, copied into bucket order so that a unit's K
// step is one TMA tile.  One warp per row, 16-byte copies.
__global__ void gather_rows_kernel(const __half* __restrict__ x16, const int32_t* __restrict__ perm_tok,
                                   int n_rows, int T, int H, __half* __restrict__ xg) {
  const int lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int chunks = H / 8;  // 16-byte chunks per row
  for (int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < n_rows; p += nwarps) {
    int tok = __ldg(perm_tok + p);
    if ((unsigned)tok >= (unsigned)T) tok = 0;  // cannot happen after a clean bucketing
    const uint4* src = reinterpret_cast<const uint4*>(x16 + (size_t)tok * H);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)p * H);
#pragma unroll 8
    for (int c = lane; c < chunks; c += 32) __stcs(dst + c, __ldg(src + c));  // streaming: keep x16 in L2
  }
}

// The partial output rows of one layer's down GEMM and what the combine
// needs to sum them per token: y[t] = 2^(2 sx_t) * (sum over the token's
// assignments of its row + its shared-expert row).
struct PartsView {
  const __half* rows;     // [T*k routed, bucket order | T shared, token order][H]
  const int32_t* pos;     // [T*k] bucket position of (token, slot), -1 if none
  const int32_t* xshift;  // [T] the inputs' power-of-two shifts
  int T, k, shared;
};

constexpr int kCombChunks = 4;  // 16-byte chunks per lane and pass: 1024 outputs per warp pass
constexpr int kCombRows = 4;    // partial rows loaded at once (in flight) per warp

// The partial row that lane j stands for: j < k, the token's slot j (its
// bucket position, -1 if none); j == k, the token's shared-expert row when
// the layer has one; -1 otherwise.  Every lane must call this.
__device__ __forceinline__ long long combine_row(const PartsView& v, int t, int lane) {
  const int n = v.T * v.k;
  long long r = -1;
  if (lane < v.k) {
    const int p = __ldg(v.pos + (size_t)t * v.k + lane);
    r = (p >= 0 && p < n) ? p : -1;
  } else if (lane == v.k && v.shared) {
    r = (long long)n + t;
  }
  return r;
}

// Outputs of token t in the chunks g = g0 + lane + 32 i (i < kCombChunks,
// g < G) of 8 values: the sum of the token's partial rows (slot order, then
// the shared row) times sc.  `myrow` is this lane's combine_row.  Rows are
// loaded kCombRows at a time, so that a warp keeps that many in flight.
__device__ __forceinline__ void combine_block(const PartsView& v, int t, int g0, int G, int H,
                                              long long myrow, float sc,
                                              float (&y)[kCombChunks][8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < kCombChunks; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) y[i][e] = 0.0f;
  const int nrows = v.k + 1;  // lanes 0..k
  for (int j0 = 0; j0 < nrows; j0 += kCombRows) {
    uint4 q[kCombRows][kCombChunks];
    bool has[kCombRows];
#pragma unroll
    for (int b = 0; b < kCombRows; ++b) {
      const long long row = __shfl_sync(0xffffffffu, myrow, (j0 + b) & 31);
      has[b] = j0 + b < nrows && row >= 0;  // the same in every lane
      const uint4* src = reinterpret_cast<const uint4*>(v.rows + (size_t)(has[b] ? row : 0) * H);
#pragma unroll
      for (int i = 0; i < kCombChunks; ++i) {
        const int g = g0 + lane + 32 * i;
        q[b][i] = (has[b] && g < G) ? __ldcs(src + g) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int b = 0; b < kCombRows; ++b) {
      if (!has[b]) continue;
#pragma unroll
      for (int i = 0; i < kCombChunks; ++i) {
        const uint32_t w[4] = {q[b][i].x, q[b][i].y, q[b][i].z, q[b][i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          y[i][2 * e] += f.x;
          y[i][2 * e + 1] += f.y;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kCombChunks; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) y[i][e] *= sc;
}

// y (bf16 [T][H]) = the combined partial rows; one warp per token.
__global__ void combine_kernel(const PartsView v, int H, uint16_t* __restrict__ y) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= v.T) return;
  const long long myrow = combine_row(v, t, lane);
  const float sc = pow2f(2 * __ldg(v.xshift + t));
  const bool vec = (reinterpret_cast<uintptr_t>(y) & 15u) == 0;
  const int G = H / 8;
  for (int g0 = 0; g0 < G; g0 += 32 * kCombChunks) {
    float yb[kCombChunks][8];
    combine_block(v, t, g0, G, H, myrow, sc, yb);
#pragma unroll
    for (int i = 0; i < kCombChunks; ++i) {
      const int g = g0 + lane + 32 * i;
      if (g >= G) break;
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        o[q] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(yb[i][2 * q])) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(yb[i][2 * q + 1])) << 16);
      uint16_t* dst = y + (size_t)t * H + 8 * g;
      if (vec) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dst[2 * q] = (uint16_t)(o[q] & 0xffffu);
          dst[2 * q + 1] = (uint16_t)(o[q] >> 16);
        }
      }
    }
  }
}

// Router weights for the prefill router GEMM: row e of `out` is the fp16
// "hi" term of W_r[e] * 2^shift (K < H), then the fp16 remainder "mid" of
// the same products (K >= H), each 8-group of K reordered to the unpack
// order 0,4,1,5,2,6,3,7 that the fp16 activations use.
__global__ void router_split_kernel(const float* __restrict__ wr, int E, int H, int shift,
                                    __half* __restrict__ out) {
  const size_t n8 = (size_t)E * H / 8;
  const float sc = pow2f(shift);
  for (size_t g = blockIdx.x * (size_t)blockDim.x + threadIdx.x; g < n8; g += (size_t)gridDim.x * blockDim.x) {
    const size_t e = g / (H / 8), c = g - e * (H / 8);
    const float* src = wr + e * H + 8 * c;
    uint32_t hi[4], mid[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {  // pair jj = (element jj, element jj + 4)
      const float w0 = src[jj] * sc, w1 = src[jj + 4] * sc;
      const __half h0 = __float2half_rn(w0), h1 = __float2half_rn(w1);
      __half2 a = __halves2half2(h0, h1);
      __half2 b = __halves2half2(__float2half_rn(w0 - __half2float(h0)),
                                 __float2half_rn(w1 - __half2float(h1)));
      hi[jj] = *reinterpret_cast<uint32_t*>(&a);
      mid[jj] = *reinterpret_cast<uint32_t*>(&b);
    }
    reinterpret_cast<uint4*>(out + e * 2 * H)[c] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    reinterpret_cast<uint4*>(out + e * 2 * H + H)[c] = make_uint4(mid[0], mid[1], mid[2], mid[3]);
  }
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct PrefillSizes {
  size_t x16, xg, xshift, zf, ids, w, offsets, perm_tok, perm_w, pos, gu, dn, nunits, hmid_r, hmid_s, wr16,
      ccount;
  int max_gu, max_dn;
  static PrefillSizes make(const moe_layer_config& c) {
    PrefillSizes s;
    const size_t Tm = (size_t)c.max_tokens, H = c.hidden, E = c.n_experts, k = c.top_k;
    const size_t F = c.ffn, Fs = c.shared_ffn;
    const size_t Tk = Tm * k;
    const size_t routed_tiles = (Tk + kNT - 1) / kNT + E;
    const size_t shared_tiles = Fs ? (Tm + kNT - 1) / kNT : 0;
    s.max_gu = (int)(routed_tiles * (F / 128) + shared_tiles * (Fs / 128));
    s.max_dn = (int)((routed_tiles + shared_tiles) * ((H + 255) / 256));
    s.x16 = Tm * H * 2;
    s.xg = (Tk + Tm) * H * 2;  // gate/up operand rows, then the down GEMM's output rows
    s.xshift = Tm * 4;
    s.zf = Tm * E * 4;
    s.ids = Tk * 4;
    s.w = Tk * 4;
    s.offsets = (E + 1) * 4;
    s.perm_tok = Tk * 4;
    s.perm_w = Tk * 4;
    s.pos = Tk * 4;
    s.gu = (size_t)s.max_gu * 16;
    s.dn = (size_t)s.max_dn * 16;
    s.nunits = 16;
    s.hmid_r = Tk * F * 2;
    s.hmid_s = Tm * (Fs ? Fs : 128) * 2;
    s.wr16 = E * 2 * H * 2;
    s.ccount = (size_t)kMaxBucketChunks * E * 4;
    return s;
  }
  size_t total() const {
    return align256(x16) + align256(xg) + align256(xshift) + align256(zf) + align256(ids) + align256(w) +
           align256(offsets) + align256(perm_tok) + align256(perm_w) + align256(pos) + align256(gu) + align256(dn) +
           align256(nunits) + align256(hmid_r) + align256(hmid_s) + align256(wr16) +
           align256(ccount);
  }
};

// 2-D fp16 map [rows][cols], box {64, 128} (128 rows of 128 bytes: one
// K step of a B tile), 128B swizzle; rows past the end read as zero.
bool encode_rows(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  auto enc = tmap_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kNT};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over packed 4-bit codes [rows][bytes_per_row], box {32, 128}:
// one K step (64 codes) of 128 weight rows, stored as 32-byte rows with the
// 32-byte swizzle: row r's 16-byte halves swap places when (r >> 2) & 1, so
// that a warp reading one half of 32 consecutive rows meets no bank twice.
bool encode_codes(CUtensorMap* m, const void* base, uint64_t bytes_per_row, uint64_t rows) {
  auto enc = tmap_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {bytes_per_row, rows};
  cuuint64_t strides[1] = {bytes_per_row};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
moe_status launch_gemm(const GemmParams& gp, moe_layer* L, int grid, cudaStream_t s,
                       const char** why) {
  const size_t smem = (size_t)Gemm<MODE>::kSmem;
  auto kern = moe_gemm_kernel<MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    *why = "cudaFuncSetAttribute(gemm smem)";
    return MOE_ERR_CUDA;
  }
  static const char* const names[3] = {"moe_gemm_gateup_swiglu", "moe_gemm_down_scatter",
                                       "moe_gemm_router"};
  prof::Scope scope(names[MODE], s);
  GemmMaps maps;
  if (MODE == kSwiglu) {
    maps.a_routed[0] = L->tmap_gate;
    maps.a_routed[1] = L->tmap_up;
    maps.a_shared[0] = L->tmap_sh_gate;
    maps.a_shared[1] = L->tmap_sh_up;
    maps.b[0] = L->tmap_xg;
    maps.b[1] = L->tmap_x16;
  } else if (MODE == kScatter) {
    maps.a_routed[0] = maps.a_routed[1] = L->tmap_down;
    maps.a_shared[0] = maps.a_shared[1] = L->tmap_sh_down;
    maps.b[0] = L->tmap_hr;
    maps.b[1] = L->tmap_hs;
  } else {
    maps.a_routed[0] = maps.a_routed[1] = maps.a_shared[0] = maps.a_shared[1] = L->tmap_wr16;
    maps.b[0] = maps.b[1] = L->tmap_x16;
  }
  kern<<<grid, Gemm<MODE>::kThreads, smem, s>>>(gp, maps);
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
  w.xg = (__half*)take(z.xg);
  w.xshift = (int32_t*)take(z.xshift);
  w.zf = (float*)take(z.zf);
  w.topk_ids = (int32_t*)take(z.ids);
  w.topk_w = (float*)take(z.w);
  w.offsets = (int32_t*)take(z.offsets);
  w.perm_tok = (int32_t*)take(z.perm_tok);
  w.perm_w = (float*)take(z.perm_w);
  w.pos = (int32_t*)take(z.pos);
  w.gu_units = (int4*)take(z.gu);
  w.dn_units = (int4*)take(z.dn);
  w.n_units = (int32_t*)take(z.nunits);
  w.hmid_r = (__half*)take(z.hmid_r);
  w.hmid_s = (__half*)take(z.hmid_s);
  w.wr16 = (__half*)take(z.wr16);
  w.ccount = (int32_t*)take(z.ccount);
  w.max_gu_units = z.max_gu;
  w.max_dn_units = z.max_dn;
  const uint64_t Tm = c.max_tokens;
  const uint64_t Fs = c.shared_ffn ? c.shared_ffn : 128;
  // packed-code maps; without a shared expert its maps alias the routed ones
  const LayerDev& d = L->dev;
  const uint64_t S = c.n_slots, H = c.hidden, F = c.ffn;
  const bool sh = c.shared_ffn > 0;
  if (!encode_rows(&L->tmap_x16, w.x16, c.hidden, Tm) ||
      !encode_rows(&L->tmap_xg, w.xg, c.hidden, Tm * c.top_k) ||
      !encode_rows(&L->tmap_hr, w.hmid_r, c.ffn, Tm * c.top_k) ||
      !encode_rows(&L->tmap_hs, w.hmid_s, Fs, Tm) ||
      !encode_codes(&L->tmap_gate, d.gate_q, H / 2, S * F) ||
      !encode_codes(&L->tmap_up, d.up_q, H / 2, S * F) ||
      !encode_codes(&L->tmap_down, d.down_q, F / 2, S * H) ||
      !encode_codes(&L->tmap_sh_gate, sh ? d.sh_gate_q : d.gate_q, H / 2, sh ? Fs : F) ||
      !encode_codes(&L->tmap_sh_up, sh ? d.sh_up_q : d.up_q, H / 2, sh ? Fs : F) ||
      !encode_codes(&L->tmap_sh_down, sh ? d.sh_down_q : d.down_q, sh ? Fs / 2 : F / 2, H)) {
    *why = "cuTensorMapEncodeTiled failed (driver entry point unavailable?)";
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status prefill_bind_stream(moe_layer* L, const char** why) {
  const moe_layer_config& c = L->cfg;
  const uint64_t E = c.n_experts, H = c.hidden, F = c.ffn;
  const LayerDev& d = L->pf_dev;
  if (!encode_codes(&L->tmap_gate, d.gate_q, H / 2, E * F) ||
      !encode_codes(&L->tmap_up, d.up_q, H / 2, E * F) ||
      !encode_codes(&L->tmap_down, d.down_q, F / 2, E * H)) {
    *why = "cuTensorMapEncodeTiled failed (staging buffer)";
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status prefill_prepare_router(moe_layer* L, const char** why) {
  const moe_layer_config& c = L->cfg;
  router_split_kernel<<<4 * L->num_sms, 256>>>(L->dev.router_w, c.n_experts, c.hidden, L->router_shift,
                                               L->ws.wr16);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  if (!encode_rows(&L->tmap_wr16, L->ws.wr16, 2 * (uint64_t)c.hidden, (uint64_t)c.n_experts)) {
    *why = "cuTensorMapEncodeTiled failed (router weights)";
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Partially resident layers, before the grouped GEMMs: every expert with a
// nonempty bucket is copied into row e of the staging buffer, from its HBM
// slot or (not resident) from the host tier over the host link.  Block
// (e, tensor t, part) copies one slice of one of the six routed tensors.
__global__ void stream_in_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ slot_of,
                                 const CacheDev* __restrict__ cache, LayerDev slots, LayerDev stage,
                                 int H, int F) {
  const int e = blockIdx.x, t = blockIdx.y;
  if (__ldg(offsets + e + 1) == __ldg(offsets + e)) return;
  const size_t gqe = (size_t)F * (H / 2), gse = (size_t)F * (H / 32) * 2;
  const size_t dqe = (size_t)H * (F / 2), dse = (size_t)H * (F / 32) * 2;
  const size_t per[6] = {gqe, gse, gqe, gse, dqe, dse};
  const int sl = __ldg(slot_of + e);
  const char* src;
  char* dst;
  const size_t n = per[t];
  {
    const char* sp[6] = {(const char*)slots.gate_q, (const char*)slots.gate_s, (const char*)slots.up_q,
                         (const char*)slots.up_s, (const char*)slots.down_q, (const char*)slots.down_s};
    const char* hp[6] = {(const char*)cache->gate_q, (const char*)cache->gate_s,
                         (const char*)cache->up_q, (const char*)cache->up_s,
                         (const char*)cache->down_q, (const char*)cache->down_s};
    char* dp[6] = {(char*)stage.gate_q, (char*)stage.gate_s, (char*)stage.up_q,
                   (char*)stage.up_s, (char*)stage.down_q, (char*)stage.down_s};
    src = (sl >= 0) ? sp[t] + (size_t)sl * n : hp[t] + (size_t)__ldg(cache->host_row + e) * n;
    dst = dp[t] + (size_t)e * n;
  }
  const size_t nv = n / 16;  // every tensor is a multiple of 16 bytes
  const size_t lo = nv * blockIdx.z / gridDim.z, hi = nv * (blockIdx.z + 1) / gridDim.z;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  size_t i = lo + threadIdx.x;
  for (; i + 3 * blockDim.x < hi; i += 4 * blockDim.x) {  // four loads in flight per thread
    const uint4 a = s4[i], b = s4[i + blockDim.x], c = s4[i + 2 * blockDim.x],
                d = s4[i + 3 * blockDim.x];
    d4[i] = a;
    d4[i + blockDim.x] = b;
    d4[i + 2 * blockDim.x] = c;
    d4[i + 3 * blockDim.x] = d;
  }
  for (; i < hi; i += blockDim.x) d4[i] = s4[i];
}

// Layer boundary of a prefill-sized stack, one warp per token:
//   y  = bf16(yacc)              (the previous layer's fp32 output; skipped
//   h' = bf16(h + y)              for the first layer, where h' = h)
//   u  = bf16(h' / sqrt(mean(h'^2) + 1e-6))
// and the next layer's fp16 operand rows of u (per-token power-of-two
// shift, K pairs in the nibble unpack order, as prep_x16_kernel).  With
// norm == 0 (after the last layer) only h' is formed.  Trace pointers may
// be null.
__global__ void stack_boundary_kernel(const uint16_t* __restrict__ h, const PartsView parts,
                                      int T, int H, int norm, uint16_t* __restrict__ h_out,
                                      uint16_t* __restrict__ y_trace, uint16_t* __restrict__ u,
                                      __half* __restrict__ x16, int32_t* __restrict__ xshift) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  const int G = H / 8;
  const uint4* hr = reinterpret_cast<const uint4*>(h + (size_t)t * H);
  uint4* ho = reinterpret_cast<uint4*>(h_out + (size_t)t * H);
  const bool has_y = parts.rows != nullptr;
  long long myrow = -1;
  float ysc = 1.0f;
  if (has_y) {
    myrow = combine_row(parts, t, lane);
    ysc = pow2f(2 * __ldg(parts.xshift + t));
  }
  // pass 1: y (the sum of the layer's partial rows), h', sum of squares
  float ss = 0.0f;
  for (int g0 = 0; g0 < G; g0 += 32 * kCombChunks) {
    float yb[kCombChunks][8];
    if (has_y) combine_block(parts, t, g0, G, H, myrow, ysc, yb);
#pragma unroll
    for (int i = 0; i < kCombChunks; ++i) {
      const int g = g0 + lane + 32 * i;
      if (g >= G) break;
      uint4 v = hr[g];
      if (has_y) {
        const float (&yy)[8] = yb[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4], yo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __nv_bfloat16 ylo = __float2bfloat16_rn(yy[2 * q]);
          const __nv_bfloat16 yhi = __float2bfloat16_rn(yy[2 * q + 1]);
          const float lo = __uint_as_float(w[q] << 16) + __bfloat162float(ylo);
          const float hi = __uint_as_float(w[q] & 0xffff0000u) + __bfloat162float(yhi);
          o[q] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
                 ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
          yo[q] = (uint32_t)__bfloat16_as_ushort(ylo) | ((uint32_t)__bfloat16_as_ushort(yhi) << 16);
        }
        v = make_uint4(o[0], o[1], o[2], o[3]);
        if (y_trace) reinterpret_cast<uint4*>(y_trace + (size_t)t * H)[g] = make_uint4(yo[0], yo[1], yo[2], yo[3]);
      }
      if (has_y || h_out != h) ho[g] = v;
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = __uint_as_float(w[q] << 16), hi = __uint_as_float(w[q] & 0xffff0000u);
        ss = fmaf(lo, lo, fmaf(hi, hi, ss));
      }
    }
  }
  if (!norm) return;
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)H + 1e-6f);
  __syncwarp();
  // pass 2: u and its max |u| (the row is read back from this warp's writes)
  const uint4* hh = reinterpret_cast<const uint4*>(h_out + (size_t)t * H);
  uint4* ur = reinterpret_cast<uint4*>(u + (size_t)t * H);
  float m = 0.0f;
  for (int g = lane; g < G; g += 32) {
    const uint4 v = hh[g];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat16 lo = __float2bfloat16_rn(__uint_as_float(w[q] << 16) * inv);
      const __nv_bfloat16 hi = __float2bfloat16_rn(__uint_as_float(w[q] & 0xffff0000u) * inv);
      m = fmaxf(m, fmaxf(fabsf(__bfloat162float(lo)), fabsf(__bfloat162float(hi))));
      o[q] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
    }
    ur[g] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  m = warp_max(m);
  int sft = 0;
  if (m > 0.0f && isfinite(m)) sft = ((__float_as_int(m) >> 23) & 0xff) - 127;
  sft = sft < -60 ? -60 : (sft > 60 ? 60 : sft);
  if (lane == 0) xshift[t] = sft;
  const float sc = pow2f(-sft);
  __syncwarp();
  // pass 3: the fp16 operand row
  uint4* out = reinterpret_cast<uint4*>(x16 + (size_t)t * H);
  for (int g = lane; g < G; g += 32) {
    const uint4 v = ur[g];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float e[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e[2 * i] = __uint_as_float(w[i] << 16) * sc;
      e[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u) * sc;
    }
    uint32_t o[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      __half2 hv = __floats2half2_rn(e[jj], e[jj + 4]);
      o[jj] = *reinterpret_cast<uint32_t*>(&hv);
    }
    out[g] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

static PartsView parts_of(const moe_layer* L, int T) {
  PartsView v;
  v.rows = L->ws.xg;
  v.pos = L->ws.pos;
  v.xshift = L->ws.xshift;
  v.T = T;
  v.k = L->cfg.top_k;
  v.shared = L->cfg.shared_ffn > 0 ? 1 : 0;
  return v;
}

moe_status launch_stack_boundary(moe_layer* next, const uint16_t* h, const moe_layer* prev, int T,
                                 int H, uint16_t* h_out, uint16_t* y_trace, uint16_t* u,
                                 cudaStream_t s, const char** why) {
  PartsView parts;
  memset(&parts, 0, sizeof parts);
  if (prev) parts = parts_of(prev, T);
  {
    prof::Scope sc("moe_stack_boundary", s);
    stack_boundary_kernel<<<(T + 7) / 8, 256, 0, s>>>(h, parts, T, H, next ? 1 : 0, h_out, y_trace, u,
                                                      next ? next->ws.x16 : nullptr,
                                                      next ? next->ws.xshift : nullptr);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status launch_prefill(moe_layer* L, const uint16_t* x, int T, uint16_t* y, int32_t* ids_out,
                          float* w_out, bool route_only, cudaStream_t s, const char** why,
                          bool prepped, bool keep_parts) {
  const moe_layer_config& c = L->cfg;
  const Workspace& ws = L->ws;
  const int H = c.hidden, E = c.n_experts, k = c.top_k;
  cudaError_t e;

  if (!prepped) {
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
  gp.ypart = ws.xg;  // the gather rows are dead once gate/up is done
  gp.z = ws.zf;
  gp.gw = (c.routing_flags & MOE_ROUTING_SHARED_GATE) ? L->ws.gw : nullptr;
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
    const int rf = c.routing_flags;
    auto kern = (E <= 256) ? topk_kernel<8> : (E <= 512) ? topk_kernel<16> : topk_kernel<kMaxExperts / 32>;
    kern<<<(T + 7) / 8, 256, 0, s>>>(
        ws.zf, T, E, k, (rf & MOE_ROUTING_BIAS_SELECT_ONLY) ? L->dev.router_b : nullptr,
        (rf & MOE_ROUTING_NO_RENORM) ? 0 : 1, (rf & MOE_ROUTING_SHARED_GATE) ? L->sh_gate_w : nullptr,
        x, H, L->ws.gw, ids, wts, ws.err);
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
  bp.pos = ws.pos;
  bp.gu_units = ws.gu_units;
  bp.dn_units = ws.dn_units;
  bp.n_units = ws.n_units;
  bp.err = ws.err;
  bp.nc = std::max(1, std::min(kMaxBucketChunks, (T * k + 1023) / 1024));  // ~1024 per chunk
  bp.ccount = ws.ccount;
  const size_t bsmem = sizeof(int) * (3 * (size_t)E + 1 + 64);
  {
    prof::Scope sc("moe_bucket_count", s);
    bucket_count_kernel<<<bp.nc, 32, sizeof(int) * E, s>>>(bp);
  }
  {
    prof::Scope sc("moe_bucket_scan", s);
    bucket_scan_kernel<<<1, kBucketThreads, bsmem, s>>>(bp);
  }
  {
    prof::Scope sc("moe_bucket_scatter", s);
    bucket_scatter_kernel<<<bp.nc, 32, sizeof(int) * E, s>>>(bp);
  }

  {
    prof::Scope sc("moe_gather_rows", s);
    const int rows = T * k;
    const int blocks = std::max(1, std::min((rows + 7) / 8, 8 * L->num_sms));
    gather_rows_kernel<<<blocks, 256, 0, s>>>(ws.x16, ws.perm_tok, rows, T, H, ws.xg);
  }

  if (L->dev.cache) {
    // partial residency: stage the experts this batch selects, then run the
    // GEMMs on the staging buffer (identity slot table)
    {
      prof::Scope sc("moe_stream_in", s);
      stream_in_kernel<<<dim3(E, 6, 4), 256, 0, s>>>(ws.offsets, L->dev.slot_of, L->dev.cache, L->dev,
                                                       L->pf_dev, H, c.ffn);
    }
    gp.W = L->pf_dev;
  }
  gp.units = ws.gu_units;
  gp.n_units = ws.n_units;
  if ((st = launch_gemm<kSwiglu>(gp, L, L->num_sms, s, why)) != MOE_OK) return st;
  gp.units = ws.dn_units;
  gp.n_units = ws.n_units + 1;
  if ((st = launch_gemm<kScatter>(gp, L, L->num_sms, s, why)) != MOE_OK) return st;
  if (!keep_parts) {
    prof::Scope sc("moe_combine", s);
    combine_kernel<<<(T + 7) / 8, 256, 0, s>>>(parts_of(L, T), H, y);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
