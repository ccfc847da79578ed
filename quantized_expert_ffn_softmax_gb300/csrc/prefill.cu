// Prefill path (more than 4 tokens).  Interim version: tokens are processed
// in groups of up to 4 by the decode kernel.
#include <string.h>

#include "moe_internal.cuh"

namespace moe {

size_t prefill_workspace_bytes(const moe_layer_config& c) {
  (void)c;
  return 256;
}

moe_status launch_prefill(moe_layer* L, const uint16_t* x, int T, uint16_t* y, int32_t* ids_out,
                          float* w_out, bool route_only, cudaStream_t stream, const char** why) {
  const moe_layer_config& c = L->cfg;
  for (int t0 = 0; t0 < T; t0 += kMaxDecodeTokens) {
    const int n = (T - t0 < kMaxDecodeTokens) ? T - t0 : kMaxDecodeTokens;
    DecodeParams p;
    memset(&p, 0, sizeof p);
    p.H = c.hidden;
    p.E = c.n_experts;
    p.k = c.top_k;
    p.F = c.ffn;
    p.Fs = c.shared_ffn;
    p.T = n;
    p.n_layers = 1;
    p.mode = route_only ? kModeRoute : kModeForward;
    p.max_units = ((n * c.top_k < c.n_experts) ? n * c.top_k : c.n_experts) + 1;
    p.x_in = x + (size_t)t0 * c.hidden;
    p.y_out = y ? y + (size_t)t0 * c.hidden : nullptr;
    p.ids_out = ids_out ? ids_out + (size_t)t0 * c.top_k : nullptr;
    p.w_out = w_out ? w_out + (size_t)t0 * c.top_k : nullptr;
    p.xbuf = L->ws.xbuf;
    p.z = L->ws.z;
    p.hbuf = L->ws.hbuf;
    p.bar = L->ws.bar;
    p.err = L->ws.err;
    p.timeout_ns = 1000000000ull;
    p.layers[0] = L->dev;
    moe_status st = launch_decode(p, stream, L->num_sms, why);
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

}  // namespace moe
