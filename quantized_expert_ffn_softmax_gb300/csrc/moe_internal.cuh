// Internal definitions shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxLayersPerLaunch = 64;
constexpr int kMaxDecodeTokens = 4;
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kDecodeThreads = 256;                 // compute threads of a decode CTA
constexpr int kDecodeBlock = kDecodeThreads + 32;   // + the copy warp
constexpr int kMaxUnits = kMaxDecodeTokens * kMaxTopK + 1;  // routed + shared

// Expert cache of a partially resident layer (n_slots < n_experts), in
// device memory: the host tier holds every expert (caller row order) in
// pinned memory the GPU reads over the host link.
struct CacheDev {
  int n_slots;
  const int32_t* host_row;        // [E] row of expert e in the host tier
  int32_t* slot_expert;           // [S] expert held by each slot, -1 = none
  uint32_t* last_use;             // [S] launch number of the slot's last use
  unsigned long long* stats;      // [2] hits, misses (decode lookups)
  const uint8_t* gate_q;          // host tier [E][F][H/2] (device-accessible)
  const uint16_t* gate_s;         // [E][F][H/32]
  const uint8_t* up_q;
  const uint16_t* up_s;
  const uint8_t* down_q;          // [E][H][F/2]
  const uint16_t* down_s;         // [E][H][F/32]
  const uint16_t* down_sb;        // [E][F/32][H] block-major down scales
};

// Device pointers of one layer's weights (library-owned copies).
struct LayerDev {
  const float* router_w;  // [E][H]
  const float* router_b;  // [E]
  const int32_t* slot_of; // [E]
  const uint8_t* gate_q;  // [S][F][H/2]
  const uint16_t* gate_s; // [S][F][H/32]
  const uint8_t* up_q;
  const uint16_t* up_s;
  const uint8_t* down_q;  // [S][H][F/2]
  const uint16_t* down_s; // [S][H][F/32]
  const uint8_t* sh_gate_q;
  const uint16_t* sh_gate_s;
  const uint8_t* sh_up_q;
  const uint16_t* sh_up_s;
  const uint8_t* sh_down_q;
  const uint16_t* sh_down_s;
  // library layers only: the down scales again, block-major, for the decode
  // kernel's one-copy-per-block loads: [S][F/32][H] and [Fs/32][H]
  const uint16_t* down_sb;
  const uint16_t* sh_down_sb;
  // partially resident layers: the cache (device memory); slot_of then holds
  // each expert's slot or -1 and is rewritten by the decode kernel
  const CacheDev* cache;
  // library layers with hidden % 256 == 0: eight 3-D tensor maps (device
  // memory) that land a gate/up item block-major for the decode kernel's
  // tensor-core path: codes of gate, up, shared gate, shared up as
  // [H/32 blocks][16 rows][16 B], then their scales as [H/256][16 rows][8];
  // null otherwise
  const CUtensorMap* tm_gu;
};

// Generation-counting grid barrier state (one per workspace, 128-B aligned).
struct GridBarrier {
  unsigned int count;
  unsigned int gen;
  unsigned int pad[30];
};

enum DecodeMode : int { kModeForward = 0, kModeStack = 1, kModeRoute = 2 };

struct DecodeParams {
  // library layers: 4-D tensor maps over each layer's down codes (routed
  // [S][H][F/2], shared [H][Fs/2]) that fetch one 32-column block of every
  // output row in four row planes (row r to position (r % 4) * H/4 + r / 4)
  CUtensorMap tm_down[kMaxLayersPerLaunch];
  CUtensorMap tm_sh_down[kMaxLayersPerLaunch];
  int down_tma;  // 1: down blocks by TMA + block-major scales; 0: per-thread copies
  unsigned step;  // launch number (least-recently-used stamps of the expert caches)
  int H, E, k, F, Fs;
  int T;          // real tokens (1..4)
  int n_layers;
  int mode;       // DecodeMode
  int max_units;  // min(T*k, E) routed units + shared
  const uint16_t* x_in;  // [T][H] bf16 (device)
  uint16_t* y_out;       // forward: y [T][H]; stack: h_L [T][H]
  uint16_t* h_trace;     // [L][T][H] or null
  uint16_t* in_trace;    // [L][T][H] or null: each layer's normalised input
  uint16_t* y_trace;     // [L][T][H] or null: each layer's output bf16(y_l)
  int32_t* ids_out;      // [L][T][k] or null
  float* w_out;          // [L][T][k] or null
  float* z;              // [4][E]
  float* gz;             // [4] shared-expert gate logits g . u (MOE_ROUTING_SHARED_GATE)
  float* yacc;           // [2][4][H] layer outputs, reduced in L2 (fp32)
  GridBarrier* bar;
  int* err;
  unsigned long long timeout_ns;
  // Test hook: every grid barrier waits for this many arrivals more than the
  // grid has, so the bounded wait runs out and records MOE_ERR_TIMEOUT.
  int debug_extra_arrivals;
  int g_stages;        // set by the launcher: gate/up shared-memory stages (1 or 2)
  int gu_mma;          // set by the launcher: gate/up items by the tensor-core path (T > 1)
  LayerDev layers[kMaxLayersPerLaunch];
  // per layer: MOE_ROUTING_* bits and the shared-expert gate vector [H]
  // (MOE_ROUTING_SHARED_GATE), kept apart from the weight pointers
  int routing_flags[kMaxLayersPerLaunch];
  const float* sh_gate_w[kMaxLayersPerLaunch];
};

// Workspace of one layer object.
struct Workspace {
  float* z = nullptr;
  GridBarrier* bar = nullptr;
  int* err = nullptr;
  uint16_t* x_stage = nullptr;  // [max_tokens][H] staging for host inputs
  uint16_t* y_stage = nullptr;  // [max_tokens][H] staging for host outputs
  uint16_t* u_layer = nullptr;  // [max_tokens][H] per-layer normalised input in prefill-sized stacks
  int32_t* ids_stage = nullptr; // [max_tokens][k]
  float* w_stage = nullptr;     // [max_tokens][k]
  float* gz = nullptr;          // [4] decode: shared-expert gate logits
  float* dyacc = nullptr;       // [2][4][H] decode: layer outputs, reduced in L2
  float* gw = nullptr;          // [max_tokens] prefill: shared-expert gate weights
  // prefill
  __half* x16 = nullptr;        // [max_tokens][H] fp16, per-token scaled, K-permuted
  // [max_tokens*(k+1)][H]: x16 rows in bucket order (operand B of the routed
  // gate/up GEMM); after it, the down GEMM's weighted output rows (routed in
  // bucket order, then the shared expert's in token order)
  __half* xg = nullptr;
  int32_t* xshift = nullptr;    // [max_tokens] per-token power-of-two shift
  float* zf = nullptr;          // [max_tokens][E] router logits
  int32_t* topk_ids = nullptr;  // [max_tokens][k]
  float* topk_w = nullptr;      // [max_tokens][k]
  int32_t* offsets = nullptr;   // [E+1] bucket offsets
  int32_t* perm_tok = nullptr;  // [max_tokens*k] token of each bucketed row
  float* perm_w = nullptr;      // [max_tokens*k] routing weight of each bucketed row
  int32_t* pos = nullptr;       // [max_tokens*k] bucket position of each (token, slot), -1 if none
  int4* gu_units = nullptr;     // gate/up work units
  int4* dn_units = nullptr;     // down work units
  int32_t* n_units = nullptr;   // [2] counts of the two lists
  __half* hmid_r = nullptr;     // [max_tokens*k][F] routed SwiGLU output (bucket order)
  __half* hmid_s = nullptr;     // [max_tokens][Fs] shared-expert SwiGLU output
  __half* wr16 = nullptr;       // [E][2H] router weights * 2^shift as fp16 hi | mid terms
  int32_t* ccount = nullptr;    // [chunks][E] bucketing counts / chunk bases
  int max_gu_units = 0, max_dn_units = 0;
  void* scratch = nullptr;
  size_t bytes = 0;
};

}  // namespace moe

struct moe_layer {
  moe_layer_config cfg;
  moe::LayerDev dev;
  CUtensorMap tmap_x16;      // x16 rows, box {64, 128}, 128B swizzle
  CUtensorMap tmap_xg;       // xg rows, same box
  CUtensorMap tmap_hr;       // hmid_r rows, same box
  CUtensorMap tmap_hs;       // hmid_s rows, same box
  CUtensorMap tmap_wr16;     // wr16 rows [E][2H], box {64, 128}, 128B swizzle
  CUtensorMap tmap_gate;     // packed codes [slots*F][H/2], box {32 B, 128 rows}
  CUtensorMap tmap_up;       // packed codes [slots*F][H/2]
  CUtensorMap tmap_down;     // packed codes [slots*H][F/2]
  CUtensorMap tmap_sh_gate;  // shared expert [Fs][H/2]
  CUtensorMap tmap_sh_up;    // shared expert [Fs][H/2]
  CUtensorMap tmap_sh_down;  // shared expert [H][Fs/2]
  CUtensorMap tm_dec_down;     // decode: 4-D view of down codes (see DecodeParams::tm_down)
  CUtensorMap tm_dec_sh_down;  // decode: the same over the shared expert's down codes
  void* tm_gu_block = nullptr;  // device copy of the decode gate/up maps (LayerDev::tm_gu)
  int router_shift = 0;               // router weights are scaled by 2^router_shift
  const float* sh_gate_w = nullptr;   // [H] device copy of the shared-expert gate vector, or null
  void* weights_block = nullptr;  // one allocation holding all weight copies
  size_t weights_bytes = 0;
  void* ws_block = nullptr;       // one allocation holding the workspace
  moe::Workspace ws;
  int device = 0;
  int num_sms = 0;
  // partial residency (cfg.n_slots < cfg.n_experts)
  void* host_tier = nullptr;        // pinned, mapped: every expert (caller row order)
  size_t host_tier_bytes = 0;
  moe::CacheDev cache_host{};       // host copy of the device CacheDev
  moe::CacheDev* cache_dev = nullptr;  // in ws_block
  moe::LayerDev pf_dev{};           // prefill view: routed experts in the staging buffer
  struct StreamBuf* stream = nullptr;  // staging buffer shared by partial layers
};

namespace moe {
// moe_api.cu: message returned by moe_last_error() on this thread
void set_last_error(const char* msg);
// moe_api.cu: checks a layer shape against the library's limits and the
// decode kernel's shared memory on a grid of num_sms CTAs (num_sms <= 0:
// on the grid that needs the least); sets the thread's error message and
// returns MOE_ERR_INVALID when it fails
moe_status validate_config(const moe_layer_config* c, int num_sms);
// moe_api.cu: limit of every bounded device-side wait (MOE_WAIT_TIMEOUT_US
// in the environment, else 1 s)
unsigned long long wait_timeout_ns();
// decode.cu
moe_status launch_decode(const DecodeParams& p, cudaStream_t stream, int num_sms,
                         const char** why);
// shared memory of the decode kernel for p's shape on a grid of num_sms CTAs
size_t decode_smem_bytes(const DecodeParams& p, int num_sms);
// moe_api.cu: next launch number (expert-cache stamps)
unsigned next_step();
// prefill.cu: re-encodes the routed-code tensor maps over the staging buffer
// of a partially resident layer (L->pf_dev)
moe_status prefill_bind_stream(moe_layer* L, const char** why);
// prefill.cu: cuTensorMapEncodeTiled from the driver (null when unavailable)
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn();
// decode.cu: the decode tensor maps of a layer (after its weights are in place)
moe_status decode_prepare(moe_layer* L, const char** why);
// prefill.cu
// prepped: the layer's fp16 operand rows (ws.x16/xshift) already hold x;
// keep_parts: leave the output as the down GEMM's weighted partial rows (y
// unused), for launch_stack_boundary to sum
moe_status launch_prefill(moe_layer* L, const uint16_t* x, int T, uint16_t* y, int32_t* ids_out,
                          float* w_out, bool route_only, cudaStream_t stream, const char** why,
                          bool prepped = false, bool keep_parts = false);
// Layer boundary of a prefill-sized stack: y = the sum of prev's partial
// output rows (launch_prefill with keep_parts), h_out = bf16(h + bf16(y))
// (h_out = h when prev is null), and for the next layer (null after the
// last) u = rmsnorm(h_out) and its fp16 operand rows in next's workspace.
moe_status launch_stack_boundary(moe_layer* next, const uint16_t* h, const moe_layer* prev, int T,
                                 int H, uint16_t* h_out, uint16_t* y_trace, uint16_t* u,
                                 cudaStream_t s, const char** why);
size_t prefill_workspace_bytes(const moe_layer_config& c);
// Carves the prefill workspace out of `scratch` and encodes the tensor maps.
moe_status prefill_init(moe_layer* L, void* scratch, const char** why);
// after router_shift is known: the fp16 hi/mid split of the router weights
moe_status prefill_prepare_router(moe_layer* L, const char** why);
}  // namespace moe
