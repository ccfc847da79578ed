// Allocation-free decode entry point.
//
// Some callers cannot allocate device memory at the point where they need a
// layer evaluated: code running while a CUDA graph is being captured into a
// pool they do not own, plug-ins inside a host framework whose allocator is
// the only one allowed to call cudaMalloc, or processes that must keep a
// fixed device-memory budget after start-up.  moe_forward_noalloc serves
// them: the caller passes device pointers to the packed weights, the input
// and the output, and every piece of scratch memory the decode kernel needs
// (router logits, expert intermediates, grid-barrier counter, error word)
// comes from one file-scope __device__ array of fixed size, below.
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "moe_internal.cuh"

namespace {

// Scratch of the allocation-free entry point: 4 MiB per GPU that loads the
// library, held until the process exits.  Every call uses it.
constexpr size_t kNoAllocScratchBytes = 4u << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

moe_status fail(moe_status s, const char* m) {
  moe::set_last_error(m);
  return s;
}

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

bool device_accessible(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace

extern "C" {

moe_status moe_forward_noalloc(const moe_layer_config* cfg, const moe_layer_weights* w,
                               const void* x_bf16, int n_tokens, void* y_bf16,
                               int32_t* status_out, void* stream) {
  if (!cfg || !w || !x_bf16 || !y_bf16) return fail(MOE_ERR_INVALID, "NULL argument");
  const int H = cfg->hidden, E = cfg->n_experts, k = cfg->top_k, F = cfg->ffn,
            Fs = cfg->shared_ffn;
  if (H < 128 || H > 8192 || H % 128 || E < 1 || E > moe::kMaxExperts || k < 1 ||
      k > moe::kMaxTopK || k > E || F < 128 || F > 4096 || F % 128 || Fs < 0 || Fs > 4096 ||
      Fs % 128 || cfg->n_slots != E)
    return fail(MOE_ERR_INVALID, "layer shape outside the library's limits");
  const int known = MOE_ROUTING_NO_RENORM | MOE_ROUTING_BIAS_SELECT_ONLY | MOE_ROUTING_SHARED_GATE;
  const bool gated = (cfg->routing_flags & MOE_ROUTING_SHARED_GATE) != 0;
  if ((cfg->routing_flags & ~known) || (gated && (Fs == 0 || !w->sh_gate_w)))
    return fail(MOE_ERR_INVALID, "routing_flags unknown, or a shared gate without shared expert or sh_gate_w");
  if (n_tokens < 1 || n_tokens > moe::kMaxDecodeTokens)
    return fail(MOE_ERR_CAPACITY, "n_tokens must be 1..4 for the allocation-free entry point");
  if (!w->router_w || !w->router_bias || !w->slot_of_expert || !w->gate_q || !w->gate_s ||
      !w->up_q || !w->up_s || !w->down_q || !w->down_s ||
      (Fs > 0 && (!w->sh_gate_q || !w->sh_gate_s || !w->sh_up_q || !w->sh_up_s ||
                  !w->sh_down_q || !w->sh_down_s)))
    return fail(MOE_ERR_INVALID, "a weight pointer is NULL (router_bias is required here)");
  if ((reinterpret_cast<uintptr_t>(x_bf16) & 15u) != 0)
    return fail(MOE_ERR_INVALID, "x must be 16-byte aligned");
  if (!device_accessible(x_bf16) || !device_accessible(y_bf16) ||
      !device_accessible(w->gate_q) || (status_out && !device_accessible(status_out)))
    return fail(MOE_ERR_INVALID, "x, y, weights and status_out must be device memory");

  // scratch carve: barrier | error word | xbuf | z | hbuf
  const int routed_max = (n_tokens * k < E) ? n_tokens * k : E;
  const size_t o_bar = 0;
  const size_t o_err = up256(o_bar + sizeof(moe::GridBarrier));
  const size_t o_xbuf = up256(o_err + 16);
  const size_t o_z = up256(o_xbuf + sizeof(uint16_t) * 2 * moe::kMaxDecodeTokens * H);
  const size_t o_gz = up256(o_z + sizeof(float) * moe::kMaxDecodeTokens * E);
  const size_t o_ya = up256(o_gz + sizeof(float) * moe::kMaxDecodeTokens);
  const size_t o_h = up256(o_ya + sizeof(float) * 2 * moe::kMaxDecodeTokens * H);
  const size_t need = o_h + sizeof(float) * moe::kMaxDecodeTokens * ((size_t)routed_max * F + Fs);
  if (need > kNoAllocScratchBytes)
    return fail(MOE_ERR_CAPACITY,
                "shape needs more than the 4 MiB static scratch of the allocation-free path");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(MOE_ERR_CUDA, "no current CUDA device");
  }
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
      // once per device, with that device current: the device address of the
      // static array (its name in host code is only a host-side stand-in)
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return fail(MOE_ERR_CUDA, "cudaGetSymbolAddress(static scratch) failed");
      }
      g_scratch_ptr[dev] = p;
    }
    base = g_scratch_ptr[dev];
  }
  char* sb = static_cast<char*>(base);
  cudaStream_t s = (cudaStream_t)stream;
  int* err = status_out ? status_out : reinterpret_cast<int*>(sb + o_err);
  if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) {
    cudaGetLastError();
    return fail(MOE_ERR_CUDA, "clear status word");
  }

  moe::DecodeParams p;
  memset(&p, 0, sizeof p);
  p.H = H;
  p.E = E;
  p.k = k;
  p.F = F;
  p.Fs = Fs;
  p.T = n_tokens;
  p.n_layers = 1;
  p.mode = moe::kModeForward;
  p.max_units = routed_max + 1;
  p.x_in = static_cast<const uint16_t*>(x_bf16);
  p.y_out = static_cast<uint16_t*>(y_bf16);
  p.xbuf = reinterpret_cast<uint16_t*>(sb + o_xbuf);
  p.z = reinterpret_cast<float*>(sb + o_z);
  p.gz = reinterpret_cast<float*>(sb + o_gz);
  p.yacc = reinterpret_cast<float*>(sb + o_ya);
  p.hbuf = reinterpret_cast<float*>(sb + o_h);
  p.bar = reinterpret_cast<moe::GridBarrier*>(sb + o_bar);
  p.err = err;
  p.timeout_ns = 1000000000ull;
  p.layers[0].router_w = w->router_w;
  p.layers[0].router_b = w->router_bias;
  p.layers[0].slot_of = w->slot_of_expert;
  p.layers[0].gate_q = w->gate_q;
  p.layers[0].gate_s = w->gate_s;
  p.layers[0].up_q = w->up_q;
  p.layers[0].up_s = w->up_s;
  p.layers[0].down_q = w->down_q;
  p.layers[0].down_s = w->down_s;
  p.layers[0].sh_gate_q = w->sh_gate_q;
  p.layers[0].sh_gate_s = w->sh_gate_s;
  p.layers[0].sh_up_q = w->sh_up_q;
  p.layers[0].sh_up_s = w->sh_up_s;
  p.layers[0].sh_down_q = w->sh_down_q;
  p.layers[0].sh_down_s = w->sh_down_s;
  p.sh_gate_w[0] = gated ? w->sh_gate_w : nullptr;
  p.routing_flags[0] = cfg->routing_flags;
  int num_sms = 0;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(MOE_ERR_CUDA, "query SM count");
  }
  const char* why = "";
  moe_status st = moe::launch_decode(p, s, num_sms, &why);
  if (st != MOE_OK) return fail(st, why);
  return MOE_OK;
}

}  // extern "C"
