// Allocation-free decode entry point.
//
// Some callers cannot allocate device memory at the point where they need a
// layer evaluated: code running while a CUDA graph is being captured into a
// pool they do not own, plug-ins inside a host framework whose allocator is
// the only one allowed to call cudaMalloc, or processes that must keep a
// fixed device-memory budget after start-up.  moe_forward_noalloc serves
// them: the caller passes device pointers to the packed weights, the input
// and the output, and every piece of scratch memory the decode kernel needs
// (router logits, the fp32 layer-output accumulators, grid-barrier counter,
// error word) comes from one file-scope __device__ array of fixed size,
// below.
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "moe_internal.cuh"

namespace {

// Scratch of the allocation-free entry point: 128 KiB per GPU that loads the
// library, held until the process exits.  Every call uses it.  Carve:
// grid-barrier counter | error word | router logits [4][E] | shared-gate
// logits [4] | two fp32 layer-output accumulators [2][4][H].  The largest
// shape that fits has H = 2048 with any E, or H = 3072 with E <= 1024;
// H = 4096 needs 129 KiB and more and is refused.
constexpr size_t kNoAllocScratchBytes = 128u << 10;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

moe_status fail(moe_status s, const char* m) {
  moe::set_last_error(m);
  return s;
}

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

// p is device (or managed) memory of device `dev`, aligned to `align` bytes
bool usable_on(const void* p, int dev, size_t align) {
  if (!p || (reinterpret_cast<uintptr_t>(p) & (align - 1)) != 0) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

}  // namespace

extern "C" {

moe_status moe_forward_noalloc(const moe_layer_config* cfg, const moe_layer_weights* w,
                               const void* x_bf16, int n_tokens, void* y_bf16,
                               int32_t* status_out, void* stream) {
  if (!cfg || !w || !x_bf16 || !y_bf16) return fail(MOE_ERR_INVALID, "NULL argument");
  int dev = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(MOE_ERR_CUDA, "no usable current CUDA device");
  }
  // the same limits as moe_layer_create, including the decode kernel's
  // shared-memory footprint (checked before anything is queued)
  moe_status vst = moe::validate_config(cfg, num_sms);
  if (vst != MOE_OK) return vst;
  const int H = cfg->hidden, E = cfg->n_experts, k = cfg->top_k, F = cfg->ffn,
            Fs = cfg->shared_ffn;
  if (cfg->n_slots != E)
    return fail(MOE_ERR_INVALID, "the allocation-free entry point needs n_slots == n_experts");
  const bool gated = (cfg->routing_flags & MOE_ROUTING_SHARED_GATE) != 0;
  if (n_tokens < 1 || n_tokens > moe::kMaxDecodeTokens)
    return fail(MOE_ERR_CAPACITY, "n_tokens must be 1..4 for the allocation-free entry point");
  // every buffer the kernel reads or writes: device memory of this device.
  // The weights are read by bulk and 16-byte async copies, x by 16-byte
  // loads: 16-byte alignment; y, the status word and the bias take 2 and 4.
  const void* const weights16[] = {w->router_w, w->slot_of_expert, w->gate_q, w->gate_s,
                                   w->up_q,     w->up_s,           w->down_q, w->down_s};
  for (const void* q : weights16)
    if (!usable_on(q, dev, 16))
      return fail(MOE_ERR_INVALID,
                  "router_w, slot_of_expert and the routed weights must be 16-byte aligned "
                  "device memory of the current device");
  if (Fs > 0) {
    const void* const shared16[] = {w->sh_gate_q, w->sh_gate_s, w->sh_up_q,
                                    w->sh_up_s,   w->sh_down_q, w->sh_down_s};
    for (const void* q : shared16)
      if (!usable_on(q, dev, 16))
        return fail(MOE_ERR_INVALID,
                    "the shared-expert weights must be 16-byte aligned device memory of the "
                    "current device");
  }
  if (gated && !usable_on(w->sh_gate_w, dev, 16))
    return fail(MOE_ERR_INVALID,
                "MOE_ROUTING_SHARED_GATE: sh_gate_w must be 16-byte aligned device memory");
  if (!usable_on(w->router_bias, dev, 4))
    return fail(MOE_ERR_INVALID, "router_bias is required: 4-byte aligned device memory");
  if (!usable_on(x_bf16, dev, 16))
    return fail(MOE_ERR_INVALID, "x must be 16-byte aligned device memory of the current device");
  if (!usable_on(y_bf16, dev, 2))
    return fail(MOE_ERR_INVALID, "y must be device memory of the current device");
  if (status_out && !usable_on(status_out, dev, 4))
    return fail(MOE_ERR_INVALID, "status_out must be device memory of the current device");

  // scratch carve: barrier | error word | z | gz | yacc
  const size_t o_bar = 0;
  const size_t o_err = up256(o_bar + sizeof(moe::GridBarrier));
  const size_t o_z = up256(o_err + 16);
  const size_t o_gz = up256(o_z + sizeof(float) * moe::kMaxDecodeTokens * E);
  const size_t o_ya = up256(o_gz + sizeof(float) * moe::kMaxDecodeTokens);
  const size_t need = o_ya + sizeof(float) * 2 * moe::kMaxDecodeTokens * H;
  if (need > kNoAllocScratchBytes)
    return fail(MOE_ERR_CAPACITY,
                "shape needs more than the 128 KiB static scratch of the allocation-free path");

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
  p.max_units = ((n_tokens * k < E) ? n_tokens * k : E) + 1;
  p.x_in = static_cast<const uint16_t*>(x_bf16);
  p.y_out = static_cast<uint16_t*>(y_bf16);
  p.z = reinterpret_cast<float*>(sb + o_z);
  p.gz = reinterpret_cast<float*>(sb + o_gz);
  p.yacc = reinterpret_cast<float*>(sb + o_ya);
  p.bar = reinterpret_cast<moe::GridBarrier*>(sb + o_bar);
  p.err = err;
  p.timeout_ns = moe::wait_timeout_ns();
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
  const char* why = "";
  moe_status st = moe::launch_decode(p, s, num_sms, &why);
  if (st != MOE_OK) return fail(st, why);
  return MOE_OK;
}

}  // extern "C"
