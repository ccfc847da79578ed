// Decode / MTP-verify path (1..4 tokens): one persistent cooperative kernel
// runs a whole stack of MoE layers.  Per layer:
//   phase R  (stacks: RMS-normalise the residual stream h -> u)
//            router GEMV (fp32, one warp per expert row)        -> z
//   barrier
//   top-k + softmax + unit list, computed redundantly by every CTA
//   phase G  fused dequant + gate/up GEMV + SwiGLU              -> h
//   barrier
//   phase D  fused dequant + down GEMV + weighted combine
//            (+ residual h + bf16(y) for stacks)                -> y / h_{l+1}
//   barrier
// The expert weights are streamed once with 128-bit non-allocating loads;
// the per-block binary16 scales of each tile are staged in shared memory by
// the bulk-copy (TMA) engine.  Packed 4-bit codes become fp16 pairs with a
// magic-exponent OR (0x6400 | n = 1024 + n, minus 1032 = n - 8, exact);
// products with the fp16 activations are exact and summed within a 32-weight
// block in fp16, then scaled by the block scale and summed in fp32.
// Activations are rescaled by a per-token power of two before the fp16
// conversion, so their range never overflows fp16.
#include <math.h>

#include "device_common.cuh"
#include "moe_internal.cuh"
#include "profile.cuh"

namespace moe {
namespace {

using namespace dev;

// Bounded wait for a bulk-copy phase; on timeout records the error and
// returns (the caller then computes on whatever is in shared memory).
__device__ __forceinline__ void mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* err,
                                                  uint64_t timeout_ns) {
  if (mbar_test(bar, parity)) return;
  const uint64_t t0 = global_timer();
  while (!mbar_test(bar, parity)) {
    if (global_timer() - t0 > timeout_ns) {
      atomicCAS(err, 0, (int)MOE_ERR_TIMEOUT);
      return;
    }
  }
}

// Grid barrier on a counter zeroed before the launch: barrier number `n`
// completes when the counter reaches (n + 1) * gridDim.x.  Waits are bounded
// by a %globaltimer deadline; a recorded error makes every later wait return
// at once, so a failing launch still ends in bounded time.
__device__ __forceinline__ void grid_sync(GridBarrier* b, unsigned& n, int* err,
                                          uint64_t timeout_ns, int extra) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned target = (n + 1) * gridDim.x + (unsigned)extra;
    __threadfence();
    atomicAdd(&b->count, 1u);
    if (ld_acquire_u32(&b->count) < target) {
      const uint64_t t0 = global_timer();
      while (ld_acquire_u32(&b->count) < target) {
        if (ld_relaxed_i32(err) != 0) break;
        if (global_timer() - t0 > timeout_ns) {
          atomicCAS(err, 0, (int)MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
    __threadfence();
  }
  ++n;
  __syncthreads();
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
__device__ __forceinline__ void unpack_codes(uint32_t w, __half2 (&h)[4]) {
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | 0x64006400u;  // (1024+n_lo, 1024+n_hi)
    h[j] = __hsub2(*reinterpret_cast<__half2*>(&v), k1032);     // exact n - 8
  }
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
    const float2 f0 = __half22float2(s0);
    const float2 f1 = __half22float2(s1);
    out[t] = (f0.x + f0.y) + (f1.x + f1.y);
  }
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

}  // namespace

// Shared-memory carve of the decode kernel (mirrored on the host).
struct DecodeSmem {
  size_t mbar, misc, red, xb, hres, xp, sc, hp, total;
  __host__ __device__ static DecodeSmem make(int H, int F, int Fs, int TT, int max_units) {
    DecodeSmem s;
    const int C = H / 32;
    const int n_routed_max = max_units - 1;
    size_t o = 0;
    s.mbar = o;
    o += 16;
    s.misc = o;
    o += 8192;
    s.red = o;
    o += 8 * 32 * 4;
    s.xb = o;
    o += (size_t)TT * H * 2;
    s.hres = o;
    o += (size_t)TT * H * 2;
    s.xp = o;
    o += (size_t)TT * H * 2;
    s.sc = o;
    size_t sc_gu = (size_t)2 * 16 * C * 2;
    size_t sc_dn = (size_t)n_routed_max * 8 * (F / 32) * 2 + (size_t)8 * (Fs / 32) * 2;
    o += (sc_gu > sc_dn ? sc_gu : sc_dn);
    o = (o + 127) & ~(size_t)127;
    s.hp = o;
    o += ((size_t)n_routed_max * F + Fs) * TT * 2;
    s.total = (o + 127) & ~(size_t)127;
    return s;
  }
};

// misc region layout (ints / floats, each array padded)
struct DecodeMisc {
  int x_shift[4];
  int d_shift[4];
  int n_routed;
  int n_units;
  int pad0[6];
  int sel_id[kMaxDecodeTokens][kMaxTopK];
  float sel_z[kMaxDecodeTokens][kMaxTopK];
  float sel_w[kMaxDecodeTokens][kMaxTopK];
  int unit_expert[kMaxUnits];
  int unit_slot[kMaxUnits];
  float unit_w[kMaxUnits][kMaxDecodeTokens];
  unsigned bitmap[kMaxExperts / 32];
  int prefix[kMaxExperts / 32 + 1];
  float tok_max[8][4];
  float inv_rms[4];
};
static_assert(sizeof(DecodeMisc) <= 8192, "misc region too small");

template <int TT>
__global__ void __launch_bounds__(kDecodeThreads, 1) moe_decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = p.H, E = p.E, k = p.k, F = p.F, Fs = p.Fs, T = p.T;
  const int C = H / 32;
  const int CF = F / 32;
  const int CS = Fs / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const DecodeSmem L = DecodeSmem::make(H, F, Fs, TT, p.max_units);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L.mbar);
  DecodeMisc& M = *reinterpret_cast<DecodeMisc*>(smem + L.misc);
  float* red = reinterpret_cast<float*>(smem + L.red);
  uint16_t* xb = reinterpret_cast<uint16_t*>(smem + L.xb);      // layer input (u)
  uint16_t* hres = reinterpret_cast<uint16_t*>(smem + L.hres);  // residual stream (stacks)
  uint4* xp = reinterpret_cast<uint4*>(smem + L.xp);
  __half* sc = reinterpret_cast<__half*>(smem + L.sc);
  uint4* hp = reinterpret_cast<uint4*>(smem + L.hp);

  if (tid == 0) {
    mbar_init(mbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  uint32_t phase = 0;
  unsigned nbar = 0;
  const uint64_t tmo = p.timeout_ns;

  for (int l = 0; l < p.n_layers; ++l) {
    const LayerDev& W = p.layers[l];
    const uint16_t* xsrc = (l == 0) ? p.x_in : (p.xbuf + (size_t)(l & 1) * kMaxDecodeTokens * H);

    // ------------------------------------------------ phase R: stage x, router
    const bool stack = (p.mode == kModeStack);
    uint16_t* stage_dst = stack ? hres : xb;
    for (int i = tid; i < TT * (H / 8); i += kDecodeThreads) {
      const int t = i / (H / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < T) v = __ldcg(reinterpret_cast<const uint4*>(xsrc + (size_t)t * H) + (i - t * (H / 8)));
      reinterpret_cast<uint4*>(stage_dst)[i] = v;
    }
    __syncthreads();
    if (stack) {
      // pre-norm: u = bf16(h / sqrt(mean(h^2) + eps)), unit gain
      float ss[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) ss[t] = 0.0f;
      for (int i = tid; i < H; i += kDecodeThreads) {
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const float v = __bfloat162float(__ushort_as_bfloat16(hres[t * H + i]));
          ss[t] = fmaf(v, v, ss[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float v = warp_sum(ss[t]);
        if (lane == 0) M.tok_max[warp][t] = v;
      }
      __syncthreads();
      if (tid < TT) {
        float v = 0.0f;
        for (int w = 0; w < kDecodeThreads / 32; ++w) v += M.tok_max[w][tid];
        M.inv_rms[tid] = rsqrtf(v / (float)H + 1e-6f);
      }
      __syncthreads();
      for (int i = tid; i < TT * H; i += kDecodeThreads) {
        const int t = i / H;
        const float v = __bfloat162float(__ushort_as_bfloat16(hres[i])) * M.inv_rms[t];
        xb[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
      __syncthreads();
      if (blockIdx.x == 0 && p.in_trace)
        for (int i = tid; i < T * H; i += kDecodeThreads) p.in_trace[(size_t)l * T * H + i] = xb[i];
    }
    {
      // per-token |x| max -> power-of-two shift for the fp16 activations
      float m[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) m[t] = 0.0f;
      for (int i = tid; i < H; i += kDecodeThreads) {
#pragma unroll
        for (int t = 0; t < TT; ++t)
          m[t] = fmaxf(m[t], fabsf(__bfloat162float(__ushort_as_bfloat16(xb[t * H + i]))));
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        float v = warp_max(m[t]);
        if (lane == 0) M.tok_max[warp][t] = v;
      }
      __syncthreads();
      if (tid < TT) {
        float v = 0.0f;
        for (int w = 0; w < kDecodeThreads / 32; ++w) v = fmaxf(v, M.tok_max[w][tid]);
        M.x_shift[tid] = range_shift(v);
      }
      __syncthreads();
      // fp16 pair planes: xp[(t*4 + q)*C + c] = pairs (x[32c+8q+j], x[32c+8q+j+4]), j < 4
      for (int i = tid; i < TT * C * 4; i += kDecodeThreads) {
        const int t = i / (4 * C);
        const int rem = i - t * 4 * C;
        const int q = rem / C;
        const int c = rem - q * C;
        const float sc_t = pow2f(-M.x_shift[t]);
        const uint16_t* src = xb + t * H + 32 * c + 8 * q;
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float a = __bfloat162float(__ushort_as_bfloat16(src[j])) * sc_t;
          float b = __bfloat162float(__ushort_as_bfloat16(src[j + 4])) * sc_t;
          __half2 hh = __floats2half2_rn(a, b);
          out[j] = *reinterpret_cast<uint32_t*>(&hh);
        }
        xp[(t * 4 + q) * C + c] = make_uint4(out[0], out[1], out[2], out[3]);
      }
    }
    // router: expert e handled by warp (e / gridDim.x) % 8 of CTA e % gridDim.x
    for (int e = blockIdx.x + warp * gridDim.x; e < E; e += 8 * gridDim.x) {
      const float4* wr = reinterpret_cast<const float4*>(W.router_w + (size_t)e * H);
      float acc[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) acc[t] = 0.0f;
      for (int base = 0; base < H / 4; base += 32 * 8) {
        float4 wv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int idx = base + j * 32 + lane;
          wv[j] = (idx < H / 4) ? __ldg(wr + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int idx = base + j * 32 + lane;
          if (idx < H / 4) {
#pragma unroll
            for (int t = 0; t < TT; ++t) {
              const uint2 xv = *reinterpret_cast<const uint2*>(xb + t * H + 4 * idx);
              const float x0 = __uint_as_float(xv.x << 16), x1 = __uint_as_float(xv.x & 0xffff0000u);
              const float x2 = __uint_as_float(xv.y << 16), x3 = __uint_as_float(xv.y & 0xffff0000u);
              acc[t] = fmaf(wv[j].x, x0, acc[t]);
              acc[t] = fmaf(wv[j].y, x1, acc[t]);
              acc[t] = fmaf(wv[j].z, x2, acc[t]);
              acc[t] = fmaf(wv[j].w, x3, acc[t]);
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float s = warp_sum(acc[t]);
        if (lane == 0 && t < T) p.z[(size_t)t * E + e] = s + W.router_b[e];
      }
    }
    grid_sync(p.bar, nbar, p.err, tmo, p.debug_extra_arrivals);

    // ------------------------------------------------ top-k + softmax + units
    if (warp < T) {
      const int t = warp;
      int id;
      float wt;
      // z was written by other CTAs before the barrier: read it through L2
      if (!warp_topk_softmax_ldcg(p.z + (size_t)t * E, E, k, &id, &wt) && lane == 0)
        atomicCAS(p.err, 0, (int)MOE_ERR_BOUNDS);
      if (lane < k) {
        M.sel_id[t][lane] = id;
        M.sel_w[t][lane] = wt;
      }
    }
    if (tid < kMaxExperts / 32) M.bitmap[tid] = 0u;
    for (int i = tid; i < kMaxUnits * kMaxDecodeTokens; i += kDecodeThreads)
      (&M.unit_w[0][0])[i] = 0.0f;
    __syncthreads();
    if (tid < T * k) atomicOr(&M.bitmap[M.sel_id[tid / k][tid % k] >> 5], 1u << (M.sel_id[tid / k][tid % k] & 31));
    __syncthreads();
    if (tid == 0) {
      int s = 0;
      for (int i = 0; i < kMaxExperts / 32; ++i) {
        M.prefix[i] = s;
        s += __popc(M.bitmap[i]);
      }
      M.prefix[kMaxExperts / 32] = s;
      M.n_routed = s;
      M.n_units = s + (Fs > 0 ? 1 : 0);
    }
    __syncthreads();
    if (tid < T * k) {
      const int t = tid / k, r = tid % k;
      const int e = M.sel_id[t][r];
      const int u = M.prefix[e >> 5] + __popc(M.bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
      M.unit_w[u][t] = M.sel_w[t][r];
      M.unit_expert[u] = e;
    }
    __syncthreads();
    const int n_routed = M.n_routed;
    if (tid < n_routed) {
      int s = W.slot_of[M.unit_expert[tid]];
      if (s < 0 || s >= E) {
        atomicCAS(p.err, 0, (int)MOE_ERR_BOUNDS);
        s = 0;
      }
      M.unit_slot[tid] = s;
    }
    if (Fs > 0 && tid < kMaxDecodeTokens) M.unit_w[n_routed][tid] = (tid < T) ? 1.0f : 0.0f;
    if (blockIdx.x == 0 && tid < T * k) {
      const int t = tid / k, r = tid % k;
      if (p.ids_out) p.ids_out[((size_t)l * T + t) * k + r] = M.sel_id[t][r];
      if (p.w_out) p.w_out[((size_t)l * T + t) * k + r] = M.sel_w[t][r];
    }
    __syncthreads();
    if (p.mode == kModeRoute) continue;

    // ------------------------------------------------ phase G: gate/up + SwiGLU
    {
      const int ipu = F / 16;  // items per routed unit
      const int n_items = n_routed * ipu + Fs / 16;
      const int rg = tid >> 6, cl = tid & 63;
      const int mat = rg >> 1, rb = rg & 1;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const uint8_t* gq;
        const uint16_t* gs;
        const uint8_t* uq;
        const uint16_t* us;
        int f0, Fu;
        size_t hoff;
        if (it < n_routed * ipu) {
          const int u = it / ipu;
          f0 = (it - u * ipu) * 16;
          const size_t slot = (size_t)M.unit_slot[u];
          gq = W.gate_q + slot * F * (H / 2);
          uq = W.up_q + slot * F * (H / 2);
          gs = W.gate_s + slot * F * C;
          us = W.up_s + slot * F * C;
          Fu = F;
          hoff = (size_t)u * kMaxDecodeTokens * F;
        } else {
          f0 = (it - n_routed * ipu) * 16;
          gq = W.sh_gate_q;
          uq = W.sh_up_q;
          gs = W.sh_gate_s;
          us = W.sh_up_s;
          Fu = Fs;
          hoff = (size_t)(p.max_units - 1) * kMaxDecodeTokens * F;
        }
        if (tid == 0) {
          mbar_expect_tx(mbar, 2u * 16u * C * 2u);
          bulk_g2s(sc, gs + (size_t)f0 * C, 16u * C * 2u, mbar);
          bulk_g2s(sc + 16 * C, us + (size_t)f0 * C, 16u * C * 2u, mbar);
        }
        const uint8_t* qrow = (mat ? uq : gq) + (size_t)(f0 + rb * 8) * (H / 2);
        float acc[8][TT];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int t = 0; t < TT; ++t) acc[r][t] = 0.0f;
        bool waited = false;
        for (int c = cl; c < C; c += 64) {
          uint4 wv[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) wv[r] = ld_stream(qrow + (size_t)r * (H / 2) + c * 16);
          if (!waited) {
            mbar_wait_bounded(mbar, phase, p.err, tmo);
            waited = true;
          }
          uint4 act[TT][4];
#pragma unroll
          for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int q = 0; q < 4; ++q) act[t][q] = xp[(t * 4 + q) * C + c];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            float d[TT];
            dot_block<TT>(wv[r], act, d);
            const float s = __half2float(sc[(mat * 16 + rb * 8 + r) * C + c]);
#pragma unroll
            for (int t = 0; t < TT; ++t) acc[r][t] = fmaf(s, d[t], acc[r][t]);
          }
        }
        // reduce the 8*TT sums of this 64-thread row group
        {
          float v[8 * TT];
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int t = 0; t < TT; ++t) v[r * TT + t] = acc[r][t];
          const float s = warp_reduce_scatter<8 * TT>(v, lane);
          constexpr int REP = 32 / (8 * TT);
          constexpr int SH = (REP == 8) ? 3 : (REP == 4) ? 2 : (REP == 2) ? 1 : 0;
          if ((lane & (REP - 1)) == 0) red[warp * 32 + (lane >> SH)] = s;
        }
        __syncthreads();
        if (tid < 16 * TT) {
          const int f = tid / TT, t = tid - (tid / TT) * TT;
          const int rbf = f >> 3, r = f & 7;
          const int ig = r * TT + t;
          const int wg = 2 * (0 * 2 + rbf), wu = 2 * (1 * 2 + rbf);
          const float xs = pow2f(M.x_shift[t]);
          const float g = (red[wg * 32 + ig] + red[(wg + 1) * 32 + ig]) * xs;
          const float uu = (red[wu * 32 + ig] + red[(wu + 1) * 32 + ig]) * xs;
          const float h = g / (1.0f + __expf(-g)) * uu;
          p.hbuf[hoff + (size_t)t * Fu + f0 + f] = h;
        }
        if (!waited && tid == 0) mbar_wait_bounded(mbar, phase, p.err, tmo);
        phase ^= 1u;
        __syncthreads();
      }
    }
    grid_sync(p.bar, nbar, p.err, tmo, p.debug_extra_arrivals);

    // ------------------------------------------------ phase D: down + combine
    {
      const int n_units = M.n_units;
      const size_t sh_hoff = (size_t)(p.max_units - 1) * kMaxDecodeTokens * F;
      // per-token max of |w * h| -> shift
      float m[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) m[t] = 0.0f;
      for (int u = 0; u < n_units; ++u) {
        const int Fu = (u < n_routed) ? F : Fs;
        const size_t ho = (u < n_routed) ? (size_t)u * kMaxDecodeTokens * F : sh_hoff;
        for (int f = tid; f < Fu; f += kDecodeThreads) {
#pragma unroll
          for (int t = 0; t < TT; ++t)
            m[t] = fmaxf(m[t], fabsf(M.unit_w[u][t] * __ldcg(p.hbuf + ho + (size_t)t * Fu + f)));
        }
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        float v = warp_max(m[t]);
        if (lane == 0) M.tok_max[warp][t] = v;
      }
      __syncthreads();
      if (tid < TT) {
        float v = 0.0f;
        for (int w = 0; w < kDecodeThreads / 32; ++w) v = fmaxf(v, M.tok_max[w][tid]);
        M.d_shift[tid] = range_shift(v);
      }
      __syncthreads();
      // stage w*h as fp16 pair planes: unit u base = u*TT*4*CF (shared: n_routed*TT*4*CF)
      {
        const int n_chunks = n_routed * CF + CS;
        for (int i = tid; i < n_chunks * TT; i += kDecodeThreads) {
          const int t = i / n_chunks;
          const int pc = i - t * n_chunks;
          int u, c, Cu;
          size_t ho;
          if (pc < n_routed * CF) {
            u = pc / CF;
            c = pc - u * CF;
            Cu = CF;
            ho = (size_t)u * kMaxDecodeTokens * F;
          } else {
            u = n_routed;
            c = pc - n_routed * CF;
            Cu = CS;
            ho = sh_hoff;
          }
          const float wt = M.unit_w[u][t] * pow2f(-M.d_shift[t]);
          const float4* src = reinterpret_cast<const float4*>(p.hbuf + ho + (size_t)t * (Cu * 32) + c * 32);
          float vv[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 f4 = __ldcg(src + j);
            vv[4 * j] = f4.x * wt;
            vv[4 * j + 1] = f4.y * wt;
            vv[4 * j + 2] = f4.z * wt;
            vv[4 * j + 3] = f4.w * wt;
          }
          uint4* dst = hp + (size_t)u * TT * 4 * CF + (size_t)t * 4 * Cu + c;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              __half2 hh = __floats2half2_rn(vv[8 * q + j], vv[8 * q + j + 4]);
              o[j] = *reinterpret_cast<uint32_t*>(&hh);
            }
            dst[q * Cu] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      __syncthreads();
      const int P = n_routed * CF + CS;
      const uint32_t sc_bytes = (uint32_t)(n_routed * 8 * CF * 2 + 8 * CS * 2);
      for (int it = blockIdx.x; it < H / 8; it += gridDim.x) {
        const int i0 = it * 8;
        if (tid == 0) {
          mbar_expect_tx(mbar, sc_bytes);
          for (int u = 0; u < n_routed; ++u)
            bulk_g2s(sc + u * 8 * CF, W.down_s + ((size_t)M.unit_slot[u] * H + i0) * CF, 8u * CF * 2u,
                     mbar);
          if (CS) bulk_g2s(sc + n_routed * 8 * CF, W.sh_down_s + (size_t)i0 * CS, 8u * CS * 2u, mbar);
        }
        float acc[8][TT];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int t = 0; t < TT; ++t) acc[r][t] = 0.0f;
        bool waited = false;
        for (int pp = tid; pp < P; pp += kDecodeThreads) {
          int u, c, Cu;
          const uint8_t* base;
          if (pp < n_routed * CF) {
            u = pp / CF;
            c = pp - u * CF;
            Cu = CF;
            base = W.down_q + (size_t)M.unit_slot[u] * H * (F / 2);
          } else {
            u = n_routed;
            c = pp - n_routed * CF;
            Cu = CS;
            base = W.sh_down_q;
          }
          uint4 wv[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) wv[r] = ld_stream(base + (size_t)(i0 + r) * (Cu * 16) + c * 16);
          if (!waited) {
            mbar_wait_bounded(mbar, phase, p.err, tmo);
            waited = true;
          }
          uint4 act[TT][4];
          const uint4* ap = hp + (size_t)u * TT * 4 * CF + c;
#pragma unroll
          for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int q = 0; q < 4; ++q) act[t][q] = ap[(t * 4 + q) * Cu];
          const __half* scu = sc + u * 8 * CF;
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            float d[TT];
            dot_block<TT>(wv[r], act, d);
            const float s = __half2float(scu[r * Cu + c]);
#pragma unroll
            for (int t = 0; t < TT; ++t) acc[r][t] = fmaf(s, d[t], acc[r][t]);
          }
        }
        {
          float v[8 * TT];
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int t = 0; t < TT; ++t) v[r * TT + t] = acc[r][t];
          const float s = warp_reduce_scatter<8 * TT>(v, lane);
          constexpr int REP = 32 / (8 * TT);
          constexpr int SH = (REP == 8) ? 3 : (REP == 4) ? 2 : (REP == 2) ? 1 : 0;
          if ((lane & (REP - 1)) == 0) red[warp * 32 + (lane >> SH)] = s;
        }
        if (!waited) mbar_wait_bounded(mbar, phase, p.err, tmo);
        phase ^= 1u;
        __syncthreads();
        if (tid < 8 * TT) {
          const int r = tid / TT, t = tid - (tid / TT) * TT;
          float y = 0.0f;
#pragma unroll
          for (int w = 0; w < kDecodeThreads / 32; ++w) y += red[w * 32 + tid];
          y *= pow2f(M.d_shift[t]);
          const int i = i0 + r;
          if (t < T) {
            const __nv_bfloat16 yb = __float2bfloat16_rn(y);
            if (p.mode == kModeForward) {
              p.y_out[(size_t)t * H + i] = __bfloat16_as_ushort(yb);
            } else {
              const float xv = __bfloat162float(__ushort_as_bfloat16(hres[t * H + i]));
              const uint16_t xn = __bfloat16_as_ushort(__float2bfloat16_rn(xv + __bfloat162float(yb)));
              uint16_t* dst = (l == p.n_layers - 1)
                                  ? p.y_out
                                  : p.xbuf + (size_t)((l + 1) & 1) * kMaxDecodeTokens * H;
              dst[(size_t)t * H + i] = xn;
              if (p.h_trace) p.h_trace[((size_t)l * T + t) * H + i] = xn;
            }
          }
        }
        __syncthreads();
      }
    }
    if (l + 1 < p.n_layers) grid_sync(p.bar, nbar, p.err, tmo, p.debug_extra_arrivals);
  }
}

size_t decode_smem_bytes(const DecodeParams& p) {
  const int TT = p.T == 1 ? 1 : (p.T == 2 ? 2 : 4);
  return DecodeSmem::make(p.H, p.F, p.Fs, TT, p.max_units).total;
}

template <int TT>
static moe_status launch_tt(const DecodeParams& p, cudaStream_t stream, int num_sms,
                            const char** why) {
  auto kern = moe_decode_kernel<TT>;
  const size_t smem = DecodeSmem::make(p.H, p.F, p.Fs, TT, p.max_units).total;
  if (smem > 227 * 1024) {
    *why = "decode shared-memory footprint exceeds 227 KB for this shape";
    return MOE_ERR_INVALID;
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    *why = "cudaFuncSetAttribute(max dynamic smem) failed";
    return MOE_ERR_CUDA;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeThreads, smem) !=
          cudaSuccess ||
      per_sm < 1) {
    *why = "decode kernel cannot be resident (occupancy query)";
    return MOE_ERR_CUDA;
  }
  int grid = num_sms * (per_sm > 2 ? 2 : per_sm);
  if (cudaMemsetAsync(&p.bar->count, 0, sizeof(unsigned), stream) != cudaSuccess) {
    *why = "cudaMemsetAsync(barrier) failed";
    return MOE_ERR_CUDA;
  }
  void* args[] = {const_cast<DecodeParams*>(&p)};
  prof::Scope scope("moe_decode_kernel", stream);
  cudaError_t e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kDecodeThreads),
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
