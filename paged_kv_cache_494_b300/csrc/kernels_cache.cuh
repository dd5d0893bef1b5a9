// K1 reshape_and_cache and K2 copy_blocks: bit copies in 16-byte vectors.
//
// K1: new K/V of arriving tokens are stored in the block the allocator handed out, at the slot's
// offset ("¿Cómo gestiona Paged Attention la caché KV...?", "PagedAttention divide el estado KV en
// bloques de tamaño fijo": the runtime allocates further physical blocks as tokens arrive).
// K2: copy-on-write copies only the page where a request diverges ("Paged Attention optimiza el uso
// de memoria en LLMs", copy-on-write paragraph; "PagedAttention e vLLM", "Approfondimento tecnico").
// Both are HBM-bound; neither converts values.
#pragma once

#include "pkv_device.cuh"

namespace pkv_dev {

// One thread per 16-byte piece of one (token, KV head) row, for K and V together.
// k, v: [n_tokens][Hkv][PPR] pieces; caches: [NB][Hkv][B][PPR] pieces.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const uint4* __restrict__ k,
                                                                const uint4* __restrict__ v,
                                                                const int64_t* __restrict__ slots, int32_t n_tokens,
                                                                int32_t Hkv, int32_t PPR, int32_t B, int64_t n_slots,
                                                                uint4* __restrict__ k_cache,
                                                                uint4* __restrict__ v_cache) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t total = static_cast<int64_t>(n_tokens) * Hkv * PPR;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t row = idx / PPR;
    const int32_t piece = static_cast<int32_t>(idx - row * PPR);
    const int32_t i = static_cast<int32_t>(row / Hkv);
    const int32_t h = static_cast<int32_t>(row - static_cast<int64_t>(i) * Hkv);
    const int64_t s = __ldg(slots + i);
    if (s < 0) continue;
    if (s >= n_slots) {
      record_error(ERRBIT_BOUNDS);
      continue;
    }
    const int64_t blk = s / B;
    const int64_t off = s - blk * B;
    const int64_t dst = ((blk * Hkv + h) * B + off) * PPR + piece;
    k_cache[dst] = __ldg(k + idx);
    v_cache[dst] = __ldg(v + idx);
  }
}

constexpr int kMaxLayers = 128;

struct LayerCaches {
  uint4* k[kMaxLayers];
  uint4* v[kMaxLayers];
};

// grid.x = n_pairs * num_layers; each CTA copies one K block and one V block (PPB pieces each).
__global__ void __launch_bounds__(256) copy_blocks_kernel(LayerCaches caches, const int32_t* __restrict__ pairs,
                                                          int32_t num_layers, int64_t PPB, int32_t num_blocks) {
  pdl_wait();
  pdl_launch_dependents();
  const int32_t pair = blockIdx.x / num_layers;
  const int32_t layer = blockIdx.x - pair * num_layers;
  const int32_t src = __ldg(pairs + 2 * pair);
  const int32_t dst = __ldg(pairs + 2 * pair + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0) record_error(ERRBIT_BOUNDS);
    return;
  }
  const uint4* ks = caches.k[layer] + static_cast<int64_t>(src) * PPB;
  const uint4* vs = caches.v[layer] + static_cast<int64_t>(src) * PPB;
  uint4* kd = caches.k[layer] + static_cast<int64_t>(dst) * PPB;
  uint4* vd = caches.v[layer] + static_cast<int64_t>(dst) * PPB;
  for (int64_t i = threadIdx.x; i < PPB; i += blockDim.x) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

}  // namespace pkv_dev
