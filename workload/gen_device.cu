// Device build of the seeded synthetic-input generator (see gen_common.h).
// Every float operation goes through an _rn intrinsic, so the bytes equal the
// host build's.  Used to fill multi-gigabyte expert banks directly in HBM.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gen_common.h"

namespace {

__global__ void quant_experts_kernel(uint64_t seed, uint32_t wset, uint32_t layer,
                                     uint32_t tensor, int n_experts,
                                     const int32_t* __restrict__ slot_of, int rows,
                                     int K, float sigma, uint8_t* __restrict__ q,
                                     uint16_t* __restrict__ s) {
  const int nb = K / 32;
  const int64_t blocks_per_expert = (int64_t)rows * nb;
  const int64_t total = blocks_per_expert * n_experts;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(idx / blocks_per_expert);
    const int64_t rb = idx - (int64_t)e * blocks_per_expert;
    const int r = (int)(rb / nb);
    const int b = (int)(rb - (int64_t)r * nb);
    const uint64_t key = gen_key(seed, wset, layer, tensor, (uint32_t)e);
    const int slot = slot_of ? slot_of[e] : e;
    float w[32];
    const uint64_t base = (uint64_t)r * (uint64_t)K + (uint64_t)b * 32u;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) w[i] = G_MUL(sigma, gen_normal(key, base + (uint64_t)i));
    uint8_t out[16];
    uint16_t sb = gen_quant_block32(w, out);
    const size_t qoff = (size_t)slot * rows * (K / 2) + (size_t)r * (K / 2) + (size_t)b * 16;
    uint4 v;
    v.x = (uint32_t)out[0] | ((uint32_t)out[1] << 8) | ((uint32_t)out[2] << 16) | ((uint32_t)out[3] << 24);
    v.y = (uint32_t)out[4] | ((uint32_t)out[5] << 8) | ((uint32_t)out[6] << 16) | ((uint32_t)out[7] << 24);
    v.z = (uint32_t)out[8] | ((uint32_t)out[9] << 8) | ((uint32_t)out[10] << 16) | ((uint32_t)out[11] << 24);
    v.w = (uint32_t)out[12] | ((uint32_t)out[13] << 8) | ((uint32_t)out[14] << 16) | ((uint32_t)out[15] << 24);
    *reinterpret_cast<uint4*>(q + qoff) = v;
    s[(size_t)slot * rows * nb + (size_t)r * nb + b] = sb;
  }
}

__global__ void dense_kernel(uint64_t key, int64_t n, float sigma, float* __restrict__ out_f32,
                             uint16_t* __restrict__ out_bf16) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v = G_MUL(sigma, gen_normal(key, (uint64_t)i));
    if (out_f32) out_f32[i] = v;
    if (out_bf16) out_bf16[i] = gen_f32_to_bf16_rn(v);
  }
}

}  // namespace

extern "C" {

// Fills the quantized matrices of experts 0..n_experts-1 for one (layer,
// tensor): expert e is written at slot slot_of[e] (slot_of is a device array
// or NULL for the identity) of q [n_slots][rows][K/2] and s [n_slots][rows][K/32].
int gen_dev_quant_experts(uint64_t seed, uint32_t wset, uint32_t layer, uint32_t tensor,
                          int n_experts, const int32_t* slot_of, int rows, int K, float sigma,
                          uint8_t* q, uint16_t* s, void* stream) {
  if (n_experts <= 0 || rows <= 0 || K <= 0 || K % 32 || !q || !s) return -1;
  const int64_t total = (int64_t)n_experts * rows * (K / 32);
  int64_t grid = (total + 255) / 256;
  if (grid > 152 * 64) grid = 152 * 64;
  quant_experts_kernel<<<(int)grid, 256, 0, (cudaStream_t)stream>>>(
      seed, wset, layer, tensor, n_experts, slot_of, rows, K, sigma, q, s);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

// Dense sigma*N(0,1) array of n elements for stream (seed, wset, layer, tensor,
// expert): fp32 and/or bf16 bits (either pointer may be NULL).
int gen_dev_dense(uint64_t seed, uint32_t wset, uint32_t layer, uint32_t tensor,
                  uint32_t expert, int64_t n, float sigma, float* out_f32, uint16_t* out_bf16,
                  void* stream) {
  if (n <= 0 || (!out_f32 && !out_bf16)) return -1;
  const uint64_t key = gen_key(seed, wset, layer, tensor, expert);
  int64_t grid = (n + 255) / 256;
  if (grid > 152 * 64) grid = 152 * 64;
  dense_kernel<<<(int)grid, 256, 0, (cudaStream_t)stream>>>(key, n, sigma, out_f32, out_bf16);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // extern "C"
