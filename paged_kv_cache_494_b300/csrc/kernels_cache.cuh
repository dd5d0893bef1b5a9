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
                                                                uint4* __restrict__ v_cache, unsigned int* err) {
  set_error_word(err);
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
                                                          int32_t num_layers, int64_t PPB, int32_t num_blocks,
                                                          unsigned int* err) {
  set_error_word(err);
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

// FP8 E4M3 cache write: one warp per (token, KV head) row of D bf16 values, for K and V.
// Per row: amax = max |x|, scale = amax / 448 (IEEE division; 1 when amax == 0), codes =
// e4m3(x / scale) rounded to nearest even with saturation. K rows are stored token-major
// (k8[blk][h][off][:]), V rows dim-major within the page (v8t[blk][h][d][off]); the scales go to
// ks / vs [blk][h][off] (V codes of a 16-token group in the order 0,1,8,9,2,3,10,11,... so that
// the decode's fragments line up). Quantising the cache is one of the pages' cache strategies ("¿Cuánta memoria
// reservar para la caché KV?", "Adaptar el presupuesto a la estrategia de caché").
template <int D>
__device__ __forceinline__ float quantize_lane(const __nv_bfloat16* row, int lane, uint32_t* codes_out) {
  constexpr int E = D / 32;  // values per lane
  float x[E];
  if constexpr (E == 4) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(row) + lane);
    x[0] = bf16_lo(raw.x); x[1] = bf16_hi(raw.x); x[2] = bf16_lo(raw.y); x[3] = bf16_hi(raw.y);
  } else {
    const uint32_t raw = __ldg(reinterpret_cast<const uint32_t*>(row) + lane);
    x[0] = bf16_lo(raw); x[1] = bf16_hi(raw);
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint32_t word = 0;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    word |= f32x2_to_e4m3x2(__fdiv_rn(x[e], scale), __fdiv_rn(x[e + 1], scale)) << (8 * e);
  *codes_out = word;
  return scale;
}

template <int D>
__global__ void __launch_bounds__(256) reshape_and_cache_fp8_kernel(
    const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v, const int64_t* __restrict__ slots,
    int32_t n_tokens, int32_t Hkv, int32_t B, int64_t n_slots, uint8_t* __restrict__ k8, uint8_t* __restrict__ v8t,
    float* __restrict__ ks, float* __restrict__ vs, unsigned int* err) {
  set_error_word(err);
  pdl_wait();
  pdl_launch_dependents();
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t total = static_cast<int64_t>(n_tokens) * Hkv;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < total;
       r += warps) {
    const int32_t i = static_cast<int32_t>(r / Hkv);
    const int32_t h = static_cast<int32_t>(r - static_cast<int64_t>(i) * Hkv);
    const int64_t s = __ldg(slots + i);
    if (s < 0) continue;
    if (s >= n_slots) {
      if (lane == 0) record_error(ERRBIT_BOUNDS);
      continue;
    }
    const int64_t blk = s / B, off = s - (s / B) * B;
    const int64_t page = blk * Hkv + h;
    uint32_t kw, vw;
    const float kscale = quantize_lane<D>(k + r * D, lane, &kw);
    const float vscale = quantize_lane<D>(v + r * D, lane, &vw);
    uint8_t* kdst = k8 + (page * B + off) * D + E * lane;
    if constexpr (E == 4) {
      *reinterpret_cast<uint32_t*>(kdst) = kw;
    } else {
      *reinterpret_cast<uint16_t*>(kdst) = static_cast<uint16_t>(kw);
    }
    // V: dim-major page; within each 16-token group the byte order of tokens is
    // (0,1,8,9, 2,3,10,11, 4,5,12,13, 6,7,14,15)
    const int64_t j = off & 15;
    const int64_t pos = (off - j) + (j < 8 ? 4 * (j >> 1) + (j & 1) : 4 * ((j - 8) >> 1) + 2 + (j & 1));
#pragma unroll
    for (int e = 0; e < E; ++e) v8t[(page * D + E * lane + e) * B + pos] = static_cast<uint8_t>(vw >> (8 * e));
    if (lane == 0) {
      ks[page * B + off] = kscale;
      vs[page * B + off] = vscale;
    }
  }
}

}  // namespace pkv_dev
