// C ABI of the routed MoE FFN layer: validation, HBM ownership, staging of
// host buffers, and dispatch to the decode (1..4 tokens) and prefill paths.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "moe_internal.cuh"
#include "profile.cuh"

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  cudaGetLastError();
  return fail(e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA, "%s: %s", what,
              cudaGetErrorString(e));
}

#define CUDA_TRY(call, what)                  \
  do {                                        \
    cudaError_t e_ = (call);                  \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool is_device_ptr(const void* p) {
  if (!p) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Where a caller's activation buffer lives: device (or managed) memory,
// pinned host memory mapped into the device's address space (`dev` receives
// the device address), or pageable host memory.
enum class PtrKind { Device, PinnedHost, Pageable };
PtrKind ptr_kind(const void* p, void** dev) {
  *dev = nullptr;
  cudaPointerAttributes a;
  if (!p || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return PtrKind::Pageable;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return PtrKind::Device;
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    *dev = a.devicePointer;
    return PtrKind::PinnedHost;
  }
  return PtrKind::Pageable;
}

// dst [S][CB][H] = src [S][H][CB] (binary16 bits): the down scales of each
// slot with the 32-column block index outermost
__global__ void scales_block_major(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                   int S, int H, int CB) {
  const size_t n = (size_t)S * H * CB;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t s = i / ((size_t)H * CB), rem = i - s * H * CB;
    const size_t r = rem / CB, b = rem - r * CB;
    dst[(s * CB + b) * H + r] = src[i];
  }
}

// ------------------------------------------------------------ partial residency

// Staging buffer of the prefill path for partially resident layers: one
// layer's routed experts (every expert e in row e), shared by the layers of
// one shape on one device; the last layer to release it frees it.
}  // namespace
struct StreamBuf {
  int device = 0, H = 0, F = 0, E = 0;
  int refs = 0;
  void* base = nullptr;
  uint8_t* gate_q = nullptr;
  uint16_t* gate_s = nullptr;
  uint8_t* up_q = nullptr;
  uint16_t* up_s = nullptr;
  uint8_t* down_q = nullptr;
  uint16_t* down_s = nullptr;
  int32_t* ident = nullptr;  // [E] identity slot table
};
namespace {
std::mutex g_stream_mu;
std::vector<StreamBuf*> g_streams;

moe_status stream_acquire(moe_layer* L) {
  const moe_layer_config& c = L->cfg;
  std::lock_guard<std::mutex> lk(g_stream_mu);
  for (StreamBuf* b : g_streams)
    if (b->device == L->device && b->H == c.hidden && b->F == c.ffn && b->E == c.n_experts) {
      ++b->refs;
      L->stream = b;
      return MOE_OK;
    }
  StreamBuf* b = new StreamBuf();
  b->device = L->device;
  b->H = c.hidden;
  b->F = c.ffn;
  b->E = c.n_experts;
  const size_t E = c.n_experts, H = c.hidden, F = c.ffn;
  const size_t gq = E * F * (H / 2), gs = E * F * (H / 32) * 2, dq = E * H * (F / 2),
               ds = E * H * (F / 32) * 2, id = E * 4;
  size_t o[8], off = 0;
  const size_t sz[7] = {gq, gs, gq, gs, dq, ds, id};
  for (int i = 0; i < 7; ++i) {
    o[i] = off;
    off = align_up(off + sz[i], 256);
  }
  cudaError_t e = cudaMalloc(&b->base, off);
  if (e != cudaSuccess) {
    delete b;
    return cuda_fail(e, "cudaMalloc(prefill staging buffer)");
  }
  char* p = static_cast<char*>(b->base);
  b->gate_q = (uint8_t*)(p + o[0]);
  b->gate_s = (uint16_t*)(p + o[1]);
  b->up_q = (uint8_t*)(p + o[2]);
  b->up_s = (uint16_t*)(p + o[3]);
  b->down_q = (uint8_t*)(p + o[4]);
  b->down_s = (uint16_t*)(p + o[5]);
  b->ident = (int32_t*)(p + o[6]);
  std::vector<int32_t> ident(E);
  for (size_t i = 0; i < E; ++i) ident[i] = (int32_t)i;
  e = cudaMemset(b->base, 0, off);
  if (e == cudaSuccess) e = cudaMemcpy(b->ident, ident.data(), id, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(b->base);
    delete b;
    return cuda_fail(e, "initialise prefill staging buffer");
  }
  b->refs = 1;
  g_streams.push_back(b);
  L->stream = b;
  return MOE_OK;
}

void stream_release(moe_layer* L) {
  if (!L->stream) return;
  std::lock_guard<std::mutex> lk(g_stream_mu);
  StreamBuf* b = L->stream;
  L->stream = nullptr;
  if (--b->refs > 0) return;
  for (size_t i = 0; i < g_streams.size(); ++i)
    if (g_streams[i] == b) {
      g_streams.erase(g_streams.begin() + i);
      break;
    }
  cudaFree(b->base);
  delete b;
}

// The slots and host tier of a partially resident layer (its weights block
// is allocated; slot i must receive expert resident[i]).  rows[e] is the
// caller's row of expert e.
moe_status fill_partial(moe_layer* L, const moe_layer_weights* w, cudaMemcpyKind kind,
                        const std::vector<int32_t>& rows, const std::vector<int32_t>& resident,
                        const std::vector<int32_t>& res_slot) {
  const moe_layer_config& c = L->cfg;
  const size_t E = c.n_experts, S = c.n_slots, H = c.hidden, F = c.ffn;
  const size_t gqe = F * (H / 2), gse = F * (H / 32) * 2, dqe = H * (F / 2), dse = H * (F / 32) * 2;
  // the resident experts into their slots
  const void* src[6] = {w->gate_q, w->gate_s, w->up_q, w->up_s, w->down_q, w->down_s};
  void* dst[6] = {(void*)L->dev.gate_q, (void*)L->dev.gate_s, (void*)L->dev.up_q,
                  (void*)L->dev.up_s,   (void*)L->dev.down_q, (void*)L->dev.down_s};
  const size_t per[6] = {gqe, gse, gqe, gse, dqe, dse};
  for (size_t i = 0; i < S; ++i) {
    const size_t row = (size_t)rows[resident[i]];
    for (int t = 0; t < 6; ++t)
      CUDA_TRY(cudaMemcpy(static_cast<char*>(dst[t]) + i * per[t],
                          static_cast<const char*>(src[t]) + row * per[t], per[t], kind),
               "copy a resident expert");
  }
  CUDA_TRY(cudaMemcpy((void*)L->dev.slot_of, res_slot.data(), sizeof(int32_t) * E,
                      cudaMemcpyHostToDevice),
           "write the slot table");
  // host tier: every expert in the caller's row order, plus block-major down scales
  size_t o[8], off = 0;
  const size_t sz[7] = {E * gqe, E * gse, E * gqe, E * gse, E * dqe, E * dse, E * dse};
  for (int i = 0; i < 7; ++i) {
    o[i] = off;
    off = align_up(off + sz[i], 256);
  }
  CUDA_TRY(cudaHostAlloc(&L->host_tier, off, cudaHostAllocMapped | cudaHostAllocPortable),
           "cudaHostAlloc(host tier)");
  L->host_tier_bytes = off;
  char* hb = static_cast<char*>(L->host_tier);
  const cudaMemcpyKind to_host =
      (kind == cudaMemcpyDeviceToDevice) ? cudaMemcpyDeviceToHost : cudaMemcpyHostToHost;
  for (int t = 0; t < 6; ++t)
    CUDA_TRY(cudaMemcpy(hb + o[t], src[t], sz[t], to_host), "fill the host tier");
  {
    const size_t CB = F / 32;
    const uint16_t* rs = reinterpret_cast<const uint16_t*>(hb + o[5]);
    uint16_t* bs = reinterpret_cast<uint16_t*>(hb + o[6]);
    for (size_t r = 0; r < E; ++r)
      for (size_t h = 0; h < H; ++h)
        for (size_t b = 0; b < CB; ++b) bs[(r * CB + b) * H + h] = rs[(r * H + h) * CB + b];
  }
  void* hd = nullptr;
  CUDA_TRY(cudaHostGetDevicePointer(&hd, L->host_tier, 0), "map the host tier");
  char* hdb = static_cast<char*>(hd);
  // cache state on the device: CacheDev | host_row [E] | slot_expert [S] |
  // last_use [S] | stats [2]
  size_t co[5], coff = 0;
  const size_t csz[5] = {sizeof(moe::CacheDev), 4 * E, 4 * S, 4 * S, 16};
  for (int i = 0; i < 5; ++i) {
    co[i] = coff;
    coff = align_up(coff + csz[i], 256);
  }
  void* cb = nullptr;
  CUDA_TRY(cudaMalloc(&cb, coff), "cudaMalloc(expert cache state)");
  L->cache_dev = static_cast<moe::CacheDev*>(cb);
  char* cbb = static_cast<char*>(cb);
  moe::CacheDev& C = L->cache_host;
  C.n_slots = (int)S;
  C.host_row = (const int32_t*)(cbb + co[1]);
  C.slot_expert = (int32_t*)(cbb + co[2]);
  C.last_use = (uint32_t*)(cbb + co[3]);
  C.stats = (unsigned long long*)(cbb + co[4]);
  C.gate_q = (const uint8_t*)(hdb + o[0]);
  C.gate_s = (const uint16_t*)(hdb + o[1]);
  C.up_q = (const uint8_t*)(hdb + o[2]);
  C.up_s = (const uint16_t*)(hdb + o[3]);
  C.down_q = (const uint8_t*)(hdb + o[4]);
  C.down_s = (const uint16_t*)(hdb + o[5]);
  C.down_sb = (const uint16_t*)(hdb + o[6]);
  CUDA_TRY(cudaMemset(cb, 0, coff), "clear expert cache state");
  CUDA_TRY(cudaMemcpy(cb, &C, sizeof C, cudaMemcpyHostToDevice), "write expert cache state");
  CUDA_TRY(cudaMemcpy((void*)C.host_row, rows.data(), 4 * E, cudaMemcpyHostToDevice),
           "write host rows");
  CUDA_TRY(cudaMemcpy(C.slot_expert, resident.data(), 4 * S, cudaMemcpyHostToDevice),
           "write slot experts");
  L->dev.cache = L->cache_dev;
  return MOE_OK;
}

struct Stage {
  const uint16_t* x = nullptr;
  uint16_t* y = nullptr;
  bool y_host = false;  // y is copied back from the staging buffer, then the stream synchronised
  bool y_sync = false;  // y is pinned host memory written in place: synchronise before returning
};

}  // namespace

namespace moe {
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }

unsigned next_step() {
  static std::atomic<unsigned> step{0u};
  return ++step;
}

unsigned long long wait_timeout_ns() {
  const char* s = getenv("MOE_WAIT_TIMEOUT_US");
  if (s && *s) {
    long long us = atoll(s);
    if (us > 0) return (uint64_t)us * 1000ull;
  }
  return 1000000000ull;  // 1 s
}

moe_status validate_config(const moe_layer_config* c, int num_sms) {
  if (!c) return fail(MOE_ERR_INVALID, "config is NULL");
  if (c->hidden < 128 || c->hidden > 8192 || c->hidden % 128)
    return fail(MOE_ERR_INVALID, "hidden=%d: need a multiple of 128 in [128, 8192]", c->hidden);
  if (c->n_experts < 1 || c->n_experts > moe::kMaxExperts)
    return fail(MOE_ERR_INVALID, "n_experts=%d: need 1..%d", c->n_experts, moe::kMaxExperts);
  if (c->top_k < 1 || c->top_k > moe::kMaxTopK || c->top_k > c->n_experts)
    return fail(MOE_ERR_INVALID, "top_k=%d: need 1..min(16, n_experts)", c->top_k);
  if (c->ffn < 128 || c->ffn > 4096 || c->ffn % 128)
    return fail(MOE_ERR_INVALID, "ffn=%d: need a multiple of 128 in [128, 4096]", c->ffn);
  if (c->shared_ffn < 0 || c->shared_ffn > 4096 || c->shared_ffn % 128)
    return fail(MOE_ERR_INVALID, "shared_ffn=%d: need 0 or a multiple of 128 up to 4096",
                c->shared_ffn);
  {
    const int smin = std::min(c->n_experts, kMaxDecodeTokens * c->top_k);
    if (c->n_slots < smin || c->n_slots > c->n_experts)
      return fail(MOE_ERR_INVALID, "n_slots=%d: need %d..n_experts=%d (a 4-token batch's experts fit)",
                  c->n_slots, smin, c->n_experts);
  }
  if (c->max_tokens < 1 || c->max_tokens > 65536)
    return fail(MOE_ERR_INVALID, "max_tokens=%d: need 1..65536", c->max_tokens);
  const int known = MOE_ROUTING_NO_RENORM | MOE_ROUTING_BIAS_SELECT_ONLY | MOE_ROUTING_SHARED_GATE;
  if (c->routing_flags & ~known)
    return fail(MOE_ERR_INVALID, "routing_flags=0x%x has unknown bits", c->routing_flags);
  if ((c->routing_flags & MOE_ROUTING_SHARED_GATE) && c->shared_ffn == 0)
    return fail(MOE_ERR_INVALID, "MOE_ROUTING_SHARED_GATE needs a shared expert (shared_ffn > 0)");
  // single-token decode must fit the decode kernel's smallest shared-memory
  // layout: one gate/up stage (16 rows of H), the CTA's router rows, the
  // token planes and the w*h staging of k + 1 units (with routing variants,
  // also the router bias).  Batches of 2..4 tokens need more; a batch that
  // does not fit is refused by the call (MOE_ERR_INVALID).
  {
    moe::DecodeParams p{};  // host-side sizing only
    p.H = c->hidden;
    p.E = c->n_experts;
    p.F = c->ffn;
    p.Fs = c->shared_ffn;
    p.T = 1;
    p.max_units = std::min(c->top_k, c->n_experts) + 1;
    const size_t bias = c->routing_flags ? (((size_t)c->n_experts * 4 + 127) & ~(size_t)127) : 0;
    // num_sms <= 0: no device yet; the grid that gives the smallest
    // footprint (one router row per CTA) refuses only what fits no GPU
    const size_t need = moe::decode_smem_bytes(p, num_sms > 0 ? num_sms : c->n_experts + 1) + bias;
    if (need > (size_t)227 * 1024)
      return fail(MOE_ERR_INVALID,
                  "hidden=%d, n_experts=%d: the decode kernel needs %zu KB of shared memory (> 227 KB)",
                  c->hidden, c->n_experts, (need + 1023) / 1024);
  }
  return MOE_OK;
}
}  // namespace moe

extern "C" {

int moe_version(void) { return 300; }

const char* moe_last_error(void) { return g_last_error.c_str(); }

moe_status moe_layer_create(const moe_layer_config* cfg, const moe_layer_weights* w,
                            int weights_on_device, moe_layer** out) {
  if (!out) return fail(MOE_ERR_INVALID, "out is NULL");
  *out = nullptr;
  // shape limits first (no device needed), the exact decode footprint for
  // this device's SM count once the weights are known to be there
  moe_status st = moe::validate_config(cfg, 0);
  if (st != MOE_OK) return st;
  if (!w || !w->router_w || !w->slot_of_expert || !w->gate_q || !w->gate_s || !w->up_q ||
      !w->up_s || !w->down_q || !w->down_s)
    return fail(MOE_ERR_INVALID, "a required weight pointer is NULL");
  if (cfg->shared_ffn > 0 && (!w->sh_gate_q || !w->sh_gate_s || !w->sh_up_q || !w->sh_up_s ||
                              !w->sh_down_q || !w->sh_down_s))
    return fail(MOE_ERR_INVALID, "shared_ffn > 0 but a shared-expert pointer is NULL");
  if ((cfg->routing_flags & MOE_ROUTING_SHARED_GATE) && !w->sh_gate_w)
    return fail(MOE_ERR_INVALID, "MOE_ROUTING_SHARED_GATE but sh_gate_w is NULL");
  int device = 0, num_sms = 0;
  CUDA_TRY(cudaGetDevice(&device), "cudaGetDevice");
  CUDA_TRY(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device),
           "query the SM count");
  if ((st = moe::validate_config(cfg, num_sms)) != MOE_OK) return st;
  const char* fault = getenv("MOE_FAULT_ALLOC");
  if (fault && atoi(fault) == 1) return fail(MOE_ERR_OOM, "allocation failure injected by MOE_FAULT_ALLOC");

  const int H = cfg->hidden, E = cfg->n_experts, F = cfg->ffn, Fs = cfg->shared_ffn;
  const int S = cfg->n_slots, k = cfg->top_k, Tm = cfg->max_tokens;
  const cudaMemcpyKind kind = weights_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;

  // slot table: the caller's row of every expert, a permutation of 0..E-1
  std::vector<int32_t> slots(E);
  CUDA_TRY(cudaMemcpy(slots.data(), w->slot_of_expert, sizeof(int32_t) * E,
                      weights_on_device ? cudaMemcpyDeviceToHost : cudaMemcpyHostToHost),
           "read slot table");
  {
    std::vector<char> seen(E, 0);
    for (int e = 0; e < E; ++e) {
      const int s = slots[e];
      if (s < 0 || s >= E || seen[s])
        return fail(MOE_ERR_INVALID, "slot_of_expert is not a permutation (expert %d -> %d)", e, s);
      seen[s] = 1;
    }
  }
  const bool partial = S < E;
  // partial residency: the experts first placed in HBM (largest profile
  // value first, ties to the lower id), slot i holding resident[i]
  std::vector<int32_t> resident, res_slot(E, -1);
  if (partial) {
    std::vector<float> prof(E, 0.0f);
    if (w->expert_profile)
      CUDA_TRY(cudaMemcpy(prof.data(), w->expert_profile, sizeof(float) * E,
                          weights_on_device ? cudaMemcpyDeviceToHost : cudaMemcpyHostToHost),
               "read expert profile");
    std::vector<int32_t> order(E);
    for (int e = 0; e < E; ++e) order[e] = e;
    if (w->expert_profile)
      std::stable_sort(order.begin(), order.end(),
                       [&](int a, int b) { return prof[a] > prof[b]; });
    resident.assign(order.begin(), order.begin() + S);
    for (int i = 0; i < S; ++i) res_slot[resident[i]] = i;
  }

  moe_layer* L = new moe_layer();
  L->cfg = *cfg;
  L->device = device;
  L->num_sms = num_sms;

  // ---- weights: one allocation, 256-B aligned sub-buffers
  struct Piece {
    const void* src;
    size_t bytes;
    size_t off;
  };
  std::vector<Piece> pieces;
  size_t off = 0;
  auto add = [&](const void* src, size_t bytes) {
    off = align_up(off, 256);
    pieces.push_back({src, bytes, off});
    off += bytes;
    return pieces.size() - 1;
  };
  const size_t gq = (size_t)S * F * (H / 2), gs = (size_t)S * F * (H / 32) * 2;
  const size_t dq = (size_t)S * H * (F / 2), ds = (size_t)S * H * (F / 32) * 2;
  // fully resident: the caller's arrays are copied whole (slot = caller row);
  // partial: the slots are filled expert by expert below
  size_t i_rw = add(w->router_w, sizeof(float) * E * H);
  size_t i_rb = add(w->router_bias, sizeof(float) * E);
  size_t i_sl = add(partial ? nullptr : w->slot_of_expert, sizeof(int32_t) * E);
  size_t i_gq = add(partial ? nullptr : w->gate_q, gq), i_gs = add(partial ? nullptr : w->gate_s, gs);
  size_t i_uq = add(partial ? nullptr : w->up_q, gq), i_us = add(partial ? nullptr : w->up_s, gs);
  size_t i_dq = add(partial ? nullptr : w->down_q, dq), i_ds = add(partial ? nullptr : w->down_s, ds);
  size_t i_sgq = 0, i_sgs = 0, i_suq = 0, i_sus = 0, i_sdq = 0, i_sds = 0;
  if (Fs > 0) {
    i_sgq = add(w->sh_gate_q, (size_t)Fs * (H / 2));
    i_sgs = add(w->sh_gate_s, (size_t)Fs * (H / 32) * 2);
    i_suq = add(w->sh_up_q, (size_t)Fs * (H / 2));
    i_sus = add(w->sh_up_s, (size_t)Fs * (H / 32) * 2);
    i_sdq = add(w->sh_down_q, (size_t)H * (Fs / 2));
    i_sds = add(w->sh_down_s, (size_t)H * (Fs / 32) * 2);
  }
  const bool gated = (cfg->routing_flags & MOE_ROUTING_SHARED_GATE) != 0;
  size_t i_sgw = 0;
  if (gated) i_sgw = add(w->sh_gate_w, sizeof(float) * H);
  // block-major copies of the down scales for the decode kernel (filled
  // from the row-major ones below)
  const size_t i_dsb = add(nullptr, ds);
  const size_t i_sdsb = Fs > 0 ? add(nullptr, (size_t)H * (Fs / 32) * 2) : 0;
  L->weights_bytes = align_up(off, 256);
  cudaError_t e = cudaMalloc(&L->weights_block, L->weights_bytes);
  if (e != cudaSuccess) {
    delete L;
    return cuda_fail(e, "cudaMalloc(weights)");
  }
  char* base = static_cast<char*>(L->weights_block);
  for (const Piece& p : pieces) {
    if (p.src)
      e = cudaMemcpy(base + p.off, p.src, p.bytes, kind);
    else
      e = cudaMemset(base + p.off, 0, p.bytes);  // router bias omitted: zero (or filled below)
    if (e != cudaSuccess) {
      moe_layer_destroy(L);
      return cuda_fail(e, "copy weights");
    }
  }
  auto at = [&](size_t i) { return static_cast<const void*>(base + pieces[i].off); };
  L->dev.router_w = (const float*)at(i_rw);
  L->dev.router_b = (const float*)at(i_rb);
  L->dev.slot_of = (const int32_t*)at(i_sl);
  L->dev.gate_q = (const uint8_t*)at(i_gq);
  L->dev.gate_s = (const uint16_t*)at(i_gs);
  L->dev.up_q = (const uint8_t*)at(i_uq);
  L->dev.up_s = (const uint16_t*)at(i_us);
  L->dev.down_q = (const uint8_t*)at(i_dq);
  L->dev.down_s = (const uint16_t*)at(i_ds);
  if (Fs > 0) {
    L->dev.sh_gate_q = (const uint8_t*)at(i_sgq);
    L->dev.sh_gate_s = (const uint16_t*)at(i_sgs);
    L->dev.sh_up_q = (const uint8_t*)at(i_suq);
    L->dev.sh_up_s = (const uint16_t*)at(i_sus);
    L->dev.sh_down_q = (const uint8_t*)at(i_sdq);
    L->dev.sh_down_s = (const uint16_t*)at(i_sds);
  }
  L->sh_gate_w = gated ? (const float*)at(i_sgw) : nullptr;
  if (partial && (st = fill_partial(L, w, kind, slots, resident, res_slot)) != MOE_OK) {
    moe_layer_destroy(L);
    return st;
  }
  L->dev.down_sb = (const uint16_t*)at(i_dsb);
  L->dev.sh_down_sb = Fs > 0 ? (const uint16_t*)at(i_sdsb) : nullptr;
  {
    const size_t n = (size_t)S * H * (F / 32);
    scales_block_major<<<(unsigned)((n + 255) / 256), 256>>>(L->dev.down_s, (uint16_t*)L->dev.down_sb,
                                                            S, H, F / 32);
    if (Fs > 0) {
      const size_t ns = (size_t)H * (Fs / 32);
      scales_block_major<<<(unsigned)((ns + 255) / 256), 256>>>(
          L->dev.sh_down_s, (uint16_t*)L->dev.sh_down_sb, 1, H, Fs / 32);
    }
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      moe_layer_destroy(L);
      return cuda_fail(e, "block-major down scales");
    }
    const char* why = "";
    if ((st = moe::decode_prepare(L, &why)) != MOE_OK) {
      moe_layer_destroy(L);
      return fail(st, "decode tensor maps: %s", why);
    }
  }

  // ---- workspace
  size_t wo = 0;
  auto wadd = [&](size_t bytes) {
    wo = align_up(wo, 256);
    size_t r = wo;
    wo += bytes;
    return r;
  };
  size_t o_z = wadd(sizeof(float) * moe::kMaxDecodeTokens * E);
  size_t o_bar = wadd(sizeof(moe::GridBarrier));
  size_t o_err = wadd(sizeof(int) * 4);
  size_t o_xs = wadd(sizeof(uint16_t) * (size_t)Tm * H);
  size_t o_ys = wadd(sizeof(uint16_t) * (size_t)Tm * H);
  size_t o_ul = wadd(sizeof(uint16_t) * (size_t)Tm * H);
  size_t o_is = wadd(sizeof(int32_t) * (size_t)Tm * k);
  size_t o_ws = wadd(sizeof(float) * (size_t)Tm * k);
  size_t o_gz = wadd(sizeof(float) * moe::kMaxDecodeTokens);
  size_t o_ya = wadd(sizeof(float) * 2 * moe::kMaxDecodeTokens * H);
  size_t o_gw = wadd(sizeof(float) * (size_t)Tm);
  size_t o_pf = wadd(moe::prefill_workspace_bytes(*cfg));
  L->ws.bytes = align_up(wo, 256);
  e = cudaMalloc(&L->ws_block, L->ws.bytes);
  if (e != cudaSuccess) {
    moe_layer_destroy(L);
    return cuda_fail(e, "cudaMalloc(workspace)");
  }
  char* wb = static_cast<char*>(L->ws_block);
  L->ws.z = (float*)(wb + o_z);
  L->ws.bar = (moe::GridBarrier*)(wb + o_bar);
  L->ws.err = (int*)(wb + o_err);
  L->ws.x_stage = (uint16_t*)(wb + o_xs);
  L->ws.y_stage = (uint16_t*)(wb + o_ys);
  L->ws.u_layer = (uint16_t*)(wb + o_ul);
  L->ws.ids_stage = (int32_t*)(wb + o_is);
  L->ws.w_stage = (float*)(wb + o_ws);
  L->ws.gz = (float*)(wb + o_gz);
  L->ws.dyacc = (float*)(wb + o_ya);
  L->ws.gw = (float*)(wb + o_gw);
  L->ws.scratch = wb + o_pf;
  e = cudaMemset(L->ws_block, 0, L->ws.bytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    moe_layer_destroy(L);
    return cuda_fail(e, "initialise workspace");
  }
  {
    const char* why = "";
    if ((st = moe::prefill_init(L, L->ws.scratch, &why)) != MOE_OK) {
      moe_layer_destroy(L);
      return fail(st, "prefill workspace: %s", why);
    }
  }
  // The prefill router splits W_r * 2^shift into two fp16 terms; the shift
  // puts max |W_r| in [16, 32) so neither term overflows or underflows.
  {
    std::vector<float> wr((size_t)E * H);
    e = cudaMemcpy(wr.data(), L->dev.router_w, sizeof(float) * wr.size(), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
      moe_layer_destroy(L);
      return cuda_fail(e, "read router weights");
    }
    float m = 0.0f;
    for (float v : wr) m = fabsf(v) > m ? fabsf(v) : m;
    int ex = 0;
    if (m > 0.0f && isfinite(m)) frexpf(m, &ex);  // m = f * 2^ex, f in [0.5, 1)
    int sh = 5 - ex;                             // m * 2^sh in [16, 32)
    L->router_shift = sh < -60 ? -60 : (sh > 60 ? 60 : sh);
  }
  {
    const char* why = "";
    if ((st = moe::prefill_prepare_router(L, &why)) != MOE_OK) {
      moe_layer_destroy(L);
      return fail(st, "prefill router weights: %s", why);
    }
  }
  if (partial) {
    // prefill view: the routed experts of a call are staged, expert e in row
    // e of the shared buffer, under an identity slot table
    if ((st = stream_acquire(L)) != MOE_OK) {
      moe_layer_destroy(L);
      return st;
    }
    L->pf_dev = L->dev;
    L->pf_dev.slot_of = L->stream->ident;
    L->pf_dev.gate_q = L->stream->gate_q;
    L->pf_dev.gate_s = L->stream->gate_s;
    L->pf_dev.up_q = L->stream->up_q;
    L->pf_dev.up_s = L->stream->up_s;
    L->pf_dev.down_q = L->stream->down_q;
    L->pf_dev.down_s = L->stream->down_s;
    L->pf_dev.cache = nullptr;
    const char* why = "";
    if ((st = moe::prefill_bind_stream(L, &why)) != MOE_OK) {
      moe_layer_destroy(L);
      return fail(st, "prefill staging maps: %s", why);
    }
  }
  *out = L;
  return MOE_OK;
}

void moe_layer_destroy(moe_layer* layer) {
  if (!layer) return;
  cudaDeviceSynchronize();
  if (layer->weights_block) cudaFree(layer->weights_block);
  if (layer->ws_block) cudaFree(layer->ws_block);
  if (layer->cache_dev) cudaFree(layer->cache_dev);
  if (layer->tm_gu_block) cudaFree(layer->tm_gu_block);
  if (layer->host_tier) cudaFreeHost(layer->host_tier);
  stream_release(layer);
  cudaGetLastError();
  delete layer;
}

moe_status moe_cache_stats(moe_layer* layer, uint64_t* hits, uint64_t* misses,
                           int32_t* slot_of_expert, int reset, void* stream) {
  if (!layer) return fail(MOE_ERR_INVALID, "layer is NULL");
  CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream), "cudaStreamSynchronize");
  unsigned long long st[2] = {0ull, 0ull};
  if (layer->cache_dev) {
    CUDA_TRY(cudaMemcpy(st, layer->cache_host.stats, sizeof st, cudaMemcpyDeviceToHost),
             "read cache statistics");
    if (reset)
      CUDA_TRY(cudaMemset(layer->cache_host.stats, 0, sizeof st), "reset cache statistics");
  }
  if (hits) *hits = st[0];
  if (misses) *misses = st[1];
  if (slot_of_expert)
    CUDA_TRY(cudaMemcpy(slot_of_expert, layer->dev.slot_of, sizeof(int32_t) * layer->cfg.n_experts,
                        cudaMemcpyDeviceToHost),
             "read the slot table");
  return MOE_OK;
}

moe_status moe_status_sync(moe_layer* layer, void* stream) {
  if (!layer) return fail(MOE_ERR_INVALID, "layer is NULL");
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  int err = 0;
  CUDA_TRY(cudaMemcpy(&err, layer->ws.err, sizeof(int), cudaMemcpyDeviceToHost), "read error word");
  if (err != 0) {
    CUDA_TRY(cudaMemset(layer->ws.err, 0, sizeof(int)), "clear error word");
    return fail((moe_status)err, "a kernel recorded error %d", err);
  }
  return MOE_OK;
}

}  // extern "C"

namespace {

moe::DecodeParams decode_params(moe_layer* L0, int T, int mode) {
  moe::DecodeParams p;
  memset(&p, 0, sizeof p);
  const moe_layer_config& c = L0->cfg;
  p.H = c.hidden;
  p.E = c.n_experts;
  p.k = c.top_k;
  p.F = c.ffn;
  p.Fs = c.shared_ffn;
  p.T = T;
  p.mode = mode;
  p.max_units = ((T * c.top_k < c.n_experts) ? T * c.top_k : c.n_experts) + 1;
  p.z = L0->ws.z;
  p.gz = L0->ws.gz;
  p.yacc = L0->ws.dyacc;
  p.bar = L0->ws.bar;
  p.err = L0->ws.err;
  p.timeout_ns = moe::wait_timeout_ns();
  const char* dbg = getenv("MOE_DEBUG_UNREACHABLE_BARRIER");
  p.debug_extra_arrivals = (dbg && atoi(dbg) == 1) ? 1 : 0;
  return p;
}

// Runs `n_layers` layers on <= 4 tokens with the decode kernel (chunks of
// kMaxLayersPerLaunch layers per launch).
moe_status run_decode(moe_layer* const* layers, int n_layers, const uint16_t* x, int T,
                      uint16_t* y, uint16_t* h_trace, uint16_t* in_trace, uint16_t* y_trace,
                      int32_t* ids_trace, float* w_out, int mode, cudaStream_t stream) {
  moe_layer* L0 = layers[0];
  const int H = L0->cfg.hidden;
  const uint16_t* cur = x;
  for (int l0 = 0; l0 < n_layers; l0 += moe::kMaxLayersPerLaunch) {
    const int nl = (n_layers - l0 < moe::kMaxLayersPerLaunch) ? n_layers - l0 : moe::kMaxLayersPerLaunch;
    moe::DecodeParams p = decode_params(L0, T, mode);
    p.n_layers = nl;
    p.x_in = cur;
    p.y_out = y;
    p.h_trace = h_trace ? h_trace + (size_t)l0 * T * H : nullptr;
    p.in_trace = in_trace ? in_trace + (size_t)l0 * T * H : nullptr;
    p.y_trace = y_trace ? y_trace + (size_t)l0 * T * H : nullptr;
    p.ids_out = ids_trace ? ids_trace + (size_t)l0 * T * L0->cfg.top_k : nullptr;
    p.w_out = w_out;
    p.down_tma = 1;
    p.step = moe::next_step();
    for (int l = 0; l < nl; ++l) {
      p.layers[l] = layers[l0 + l]->dev;
      p.tm_down[l] = layers[l0 + l]->tm_dec_down;
      p.tm_sh_down[l] = layers[l0 + l]->tm_dec_sh_down;
      p.routing_flags[l] = layers[l0 + l]->cfg.routing_flags;
      p.sh_gate_w[l] = layers[l0 + l]->sh_gate_w;
    }
    const char* why = "";
    moe_status st = moe::launch_decode(p, stream, L0->num_sms, &why);
    if (st != MOE_OK) return fail(st, "decode launch: %s", why);
    cur = y;
  }
  return MOE_OK;
}

// One layer on any token count: decode kernel for <= 4 tokens, the prefill
// path above that.
moe_status forward_device(moe_layer* L, const uint16_t* x, int T, uint16_t* y, cudaStream_t s) {
  if (T <= moe::kMaxDecodeTokens) {
    moe_layer* one[1] = {L};
    return run_decode(one, 1, x, T, y, nullptr, nullptr, nullptr, nullptr, nullptr,
                      moe::kModeForward, s);
  }
  const char* why = "";
  moe_status st = moe::launch_prefill(L, x, T, y, nullptr, nullptr, false, s, &why);
  if (st != MOE_OK) return fail(st, "prefill: %s", why);
  return MOE_OK;
}

moe_status check_common(moe_layer* L, const void* x, int T) {
  if (!L) return fail(MOE_ERR_INVALID, "layer is NULL");
  if (!x) return fail(MOE_ERR_INVALID, "x is NULL");
  if (T < 1 || T > L->cfg.max_tokens)
    return fail(MOE_ERR_CAPACITY, "n_tokens=%d outside [1, %d]", T, L->cfg.max_tokens);
  return MOE_OK;
}

// Brings x to the device (staging host input) and picks the y target.
// Decode-sized calls (`in_place`) read a pinned host x and write a pinned
// host y through their device addresses: 4 KB per token each way, which the
// kernel moves faster than two extra stream operations would.  Such an x,
// like the source of a stream-ordered copy, must stay unchanged until the
// stream reaches the call.
moe_status stage_in(moe_layer* L, const void* x, int T, void* y, Stage* st, cudaStream_t s,
                    bool in_place = false) {
  const size_t bytes = sizeof(uint16_t) * (size_t)T * L->cfg.hidden;
  void* xd = nullptr;
  const PtrKind xk = ptr_kind(x, &xd);
  if (xk == PtrKind::Device) {
    if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
      st->x = static_cast<const uint16_t*>(x);
    } else {  // the kernels read x with 16-byte loads: realign through the staging buffer
      CUDA_TRY(cudaMemcpyAsync(L->ws.x_stage, x, bytes, cudaMemcpyDeviceToDevice, s), "realign x");
      st->x = L->ws.x_stage;
    }
  } else if (in_place && xk == PtrKind::PinnedHost && (reinterpret_cast<uintptr_t>(xd) & 15u) == 0) {
    st->x = static_cast<const uint16_t*>(xd);
  } else {
    CUDA_TRY(cudaMemcpyAsync(L->ws.x_stage, x, bytes, cudaMemcpyHostToDevice, s), "copy x to device");
    st->x = L->ws.x_stage;
  }
  if (y) {
    void* yd = nullptr;
    const PtrKind yk = ptr_kind(y, &yd);
    if (yk == PtrKind::Device) {
      st->y = static_cast<uint16_t*>(y);
    } else if (in_place && yk == PtrKind::PinnedHost) {
      st->y = static_cast<uint16_t*>(yd);
      st->y_sync = true;
    } else {
      st->y = L->ws.y_stage;
      st->y_host = true;
    }
  }
  return MOE_OK;
}

moe_status stage_out(moe_layer* L, int T, void* y, const Stage& st, cudaStream_t s) {
  if (st.y_host) {
    const size_t bytes = sizeof(uint16_t) * (size_t)T * L->cfg.hidden;
    CUDA_TRY(cudaMemcpyAsync(y, st.y, bytes, cudaMemcpyDeviceToHost, s), "copy y to host");
  }
  if (st.y_host || st.y_sync) CUDA_TRY(cudaStreamSynchronize(s), "synchronise after writing y");
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_route(moe_layer* layer, const void* x_bf16, int n_tokens, int32_t* topk_ids,
                     float* topk_w, void* stream) {
  moe_status st = check_common(layer, x_bf16, n_tokens);
  if (st != MOE_OK) return st;
  if (!topk_ids || !topk_w) return fail(MOE_ERR_INVALID, "topk_ids / topk_w is NULL");
  cudaStream_t s = (cudaStream_t)stream;
  Stage sg;
  if ((st = stage_in(layer, x_bf16, n_tokens, nullptr, &sg, s)) != MOE_OK) return st;
  const int k = layer->cfg.top_k;
  const bool ids_host = !is_device_ptr(topk_ids), w_host = !is_device_ptr(topk_w);
  int32_t* ids = ids_host ? layer->ws.ids_stage : topk_ids;
  float* w = w_host ? layer->ws.w_stage : topk_w;
  if (n_tokens <= moe::kMaxDecodeTokens) {
    moe_layer* one[1] = {layer};
    st = run_decode(one, 1, sg.x, n_tokens, nullptr, nullptr, nullptr, nullptr, ids, w,
                    moe::kModeRoute, s);
  } else {
    const char* why = "";
    st = moe::launch_prefill(layer, sg.x, n_tokens, nullptr, ids, w, true, s, &why);
    if (st != MOE_OK) st = fail(st, "prefill route: %s", why);
  }
  if (st != MOE_OK) return st;
  if (ids_host)
    CUDA_TRY(cudaMemcpyAsync(topk_ids, ids, sizeof(int32_t) * n_tokens * k, cudaMemcpyDeviceToHost, s),
             "copy ids to host");
  if (w_host)
    CUDA_TRY(cudaMemcpyAsync(topk_w, w, sizeof(float) * n_tokens * k, cudaMemcpyDeviceToHost, s),
             "copy weights to host");
  if (ids_host || w_host) CUDA_TRY(cudaStreamSynchronize(s), "synchronise after route");
  return MOE_OK;
}

moe_status moe_forward(moe_layer* layer, const void* x_bf16, int n_tokens, void* y_bf16,
                       void* stream) {
  moe_status st = check_common(layer, x_bf16, n_tokens);
  if (st != MOE_OK) return st;
  if (!y_bf16) return fail(MOE_ERR_INVALID, "y is NULL");
  if (x_bf16 == y_bf16) return fail(MOE_ERR_INVALID, "x and y must not overlap");
  cudaStream_t s = (cudaStream_t)stream;
  Stage sg;
  if ((st = stage_in(layer, x_bf16, n_tokens, y_bf16, &sg, s, n_tokens <= moe::kMaxDecodeTokens)) != MOE_OK)
    return st;
  if ((st = forward_device(layer, sg.x, n_tokens, sg.y, s)) != MOE_OK) return st;
  return stage_out(layer, n_tokens, y_bf16, sg, s);
}

moe_status moe_stack_forward_traced(moe_layer* const* layers, int n_layers, const void* x_bf16,
                                    int n_tokens, void* y_bf16, void* h_trace_bf16,
                                    void* in_trace_bf16, void* y_trace_bf16, int32_t* ids_trace,
                                    void* stream) {
  if (!layers || n_layers < 1) return fail(MOE_ERR_INVALID, "need at least one layer");
  moe_status st = check_common(layers[0], x_bf16, n_tokens);
  if (st != MOE_OK) return st;
  if (!y_bf16) return fail(MOE_ERR_INVALID, "y is NULL");
  const moe_layer_config& c0 = layers[0]->cfg;
  for (int l = 0; l < n_layers; ++l) {
    if (!layers[l]) return fail(MOE_ERR_INVALID, "layer %d is NULL", l);
    const moe_layer_config& c = layers[l]->cfg;
    if (c.hidden != c0.hidden || c.n_experts != c0.n_experts || c.top_k != c0.top_k ||
        c.ffn != c0.ffn || c.shared_ffn != c0.shared_ffn)
      return fail(MOE_ERR_INVALID, "layer %d has a different shape from layer 0", l);
  }
  if ((h_trace_bf16 && !is_device_ptr(h_trace_bf16)) || (ids_trace && !is_device_ptr(ids_trace)) ||
      (in_trace_bf16 && !is_device_ptr(in_trace_bf16)) ||
      (y_trace_bf16 && !is_device_ptr(y_trace_bf16)))
    return fail(MOE_ERR_INVALID, "trace buffers must be device memory");
  cudaStream_t s = (cudaStream_t)stream;
  Stage sg;
  if ((st = stage_in(layers[0], x_bf16, n_tokens, y_bf16, &sg, s, n_tokens <= moe::kMaxDecodeTokens)) !=
      MOE_OK)
    return st;
  const int H = c0.hidden, k = c0.top_k;
  if (n_tokens <= moe::kMaxDecodeTokens) {
    st = run_decode(layers, n_layers, sg.x, n_tokens, sg.y, (uint16_t*)h_trace_bf16,
                    (uint16_t*)in_trace_bf16, (uint16_t*)y_trace_bf16, ids_trace, nullptr,
                    moe::kModeStack, s);
    if (st != MOE_OK) return st;
  } else {
    // prefill-sized stack, layer by layer.  Each layer boundary is one
    // kernel: the sum of the previous layer's partial output rows, y_l,
    // becomes the residual
    // h_{l+1} = bf16(h_l + bf16(y_l)), then u_{l+1} = rmsnorm(h_{l+1}) and its
    // fp16 operand rows go straight into the next layer's workspace.  h
    // ping-pongs between two staging buffers (or lands in the h trace).
    moe_layer* L0 = layers[0];
    const size_t n = (size_t)n_tokens * H;
    uint16_t* P = L0->ws.x_stage;
    uint16_t* Q = L0->ws.y_stage;
    uint16_t* U = L0->ws.u_layer;
    uint16_t* ht = (uint16_t*)h_trace_bf16;
    uint16_t* it = (uint16_t*)in_trace_bf16;
    uint16_t* yt = (uint16_t*)y_trace_bf16;
    const uint16_t* cur = sg.x;
    const char* why = "";
    st = moe::launch_stack_boundary(layers[0], cur, nullptr, n_tokens, H, const_cast<uint16_t*>(cur),
                                    nullptr, it ? it : U, s, &why);
    if (st != MOE_OK) return fail(st, "stack input: %s", why);
    for (int l = 0; l < n_layers; ++l) {
      const uint16_t* u_l = it ? it + (size_t)l * n : U;
      st = moe::launch_prefill(layers[l], u_l, n_tokens, nullptr,
                               ids_trace ? ids_trace + (size_t)l * n_tokens * k : nullptr, nullptr,
                               false, s, &why, /*prepped=*/true, /*keep_parts=*/true);
      if (st != MOE_OK) return fail(st, "prefill layer %d: %s", l, why);
      const bool last = l == n_layers - 1;
      moe_layer* next = last ? nullptr : layers[l + 1];
      uint16_t* dst = ht ? ht + (size_t)l * n : (last ? sg.y : (cur == P ? Q : P));
      st = moe::launch_stack_boundary(next, cur, layers[l], n_tokens, H, dst,
                                      yt ? yt + (size_t)l * n : nullptr,
                                      next ? (it ? it + (size_t)(l + 1) * n : U) : nullptr, s, &why);
      if (st != MOE_OK) return fail(st, "layer %d boundary: %s", l, why);
      cur = dst;
    }
    if (ht)
      CUDA_TRY(cudaMemcpyAsync(sg.y, cur, n * 2, cudaMemcpyDeviceToDevice, s), "stack output");
  }
  return stage_out(layers[0], n_tokens, y_bf16, sg, s);
}

moe_status moe_last_buckets(moe_layer* layer, int n_tokens, int32_t* offsets, int32_t* perm_token,
                            void* stream) {
  if (!layer || !offsets || !perm_token) return fail(MOE_ERR_INVALID, "NULL argument");
  if (n_tokens <= moe::kMaxDecodeTokens || n_tokens > layer->cfg.max_tokens)
    return fail(MOE_ERR_CAPACITY, "n_tokens=%d is not a prefill-path batch", n_tokens);
  cudaStream_t s = (cudaStream_t)stream;
  const size_t nE = (size_t)layer->cfg.n_experts + 1;
  const size_t nP = (size_t)n_tokens * layer->cfg.top_k;
  const cudaMemcpyKind ko = is_device_ptr(offsets) ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost;
  const cudaMemcpyKind kp = is_device_ptr(perm_token) ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost;
  CUDA_TRY(cudaMemcpyAsync(offsets, layer->ws.offsets, sizeof(int32_t) * nE, ko, s), "copy offsets");
  CUDA_TRY(cudaMemcpyAsync(perm_token, layer->ws.perm_tok, sizeof(int32_t) * nP, kp, s), "copy perm");
  CUDA_TRY(cudaStreamSynchronize(s), "synchronise");
  return MOE_OK;
}

moe_status moe_stack_forward(moe_layer* const* layers, int n_layers, const void* x_bf16,
                             int n_tokens, void* y_bf16, void* stream) {
  return moe_stack_forward_traced(layers, n_layers, x_bf16, n_tokens, y_bf16, nullptr, nullptr,
                                  nullptr, nullptr, stream);
}

}  // extern "C"
