// Device primitives for libpagedkv kernels (sm_103a): error word, mbarriers with bounded waits,
// 1-D TMA bulk copies global -> shared, bf16 unpacking. Included by pkv_ops.cu only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "pagedkv.h"

namespace pkv_dev {

// Error bits recorded by kernels, read and cleared by pkv_last_error.
enum : unsigned int { ERRBIT_BOUNDS = 1u, ERRBIT_TIMEOUT = 2u };

// Kernel error word of the process. This header is included by exactly one translation unit
// (pkv_ops.cu).
__device__ unsigned int g_error_bits = 0;

// Error word of the running kernel: the word of the pool the call belongs to (set with
// pkv_pool_set_error_word), or null for the process-wide word. Every kernel stores it here first
// thing (all threads store the same value), so code deep inside a kernel (bounded waits included)
// records into the right word without carrying the pointer.
__shared__ unsigned int* s_err_word;

__device__ __forceinline__ void set_error_word(unsigned int* w) { s_err_word = w; }

__device__ __forceinline__ void record_error(unsigned int bit) {
  unsigned int* w = s_err_word;
  atomicOr(w ? w : &g_error_bits, bit);
}

// Makes a tagged task counter ((low 32 bits of the tag) << 32 | count) belong to this call: a value
// with another tag (an
// earlier call's, or fresh memory) is replaced by (tag << 32) | 0; a value with this tag is left as it
// is (takers may already have counted on it). Bounded: gives up quietly, and takers then install the
// tag themselves.
__device__ __forceinline__ void install_task_tag(unsigned long long* ctr, unsigned long long tag) {
  const unsigned long long tg = tag & 0xffffffffull;
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(ctr);
  for (int it = 0; it < 64 && (cur >> 32) != tg; ++it) {
    const unsigned long long prev = atomicCAS(ctr, cur, tg << 32);
    if (prev == cur) return;
    cur = prev;
  }
}

// Upper bound on mbarrier polls before a wait gives up. Each try_wait may itself suspend the thread
// for a hardware-chosen interval (measured on B300: ~4 us per unsatisfied poll), so a stuck wait
// gives up after about a second of running; a copy in flight completes in microseconds.
constexpr uint32_t kMaxPolls = 1u << 18;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA) before first use.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete. Returns false (and records
// ERRBIT_TIMEOUT) if it did not complete within kMaxPolls polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kMaxPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  record_error(ERRBIT_TIMEOUT);
  return false;
}

// Programmatic dependent launch. Every libpagedkv kernel calls pdl_wait() before its first global
// memory access, so launching with programmatic stream serialisation keeps plain stream order for
// data while the launch itself overlaps the tail of the previous kernel in the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy (TMA engine) of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory, with an L2 eviction-priority hint (policy from
// createpolicy); completion is signalled on `bar` as tx bytes.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t smem_dst, const void* gmem_src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_dst),
      "l"(gmem_src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D tiled tensor copy (TMA) global -> shared through a tensor map, completion on `bar`.
// x (innermost, elements) must keep x * sizeof(elem) a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 3-D tiled tensor copy (TMA) global -> shared with an L2 cache hint; x as for tma_load_2d.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 int32_t z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// Four 8x8 b16 matrices from shared memory (lane i gives the row address of row i%8 of matrix i/8).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Same, each matrix transposed on the way into registers.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Transpose of an 8x8 matrix of 16-bit elements spread over the warp in mma fragment order (lane
// 4r + c holds row r, columns 2c and 2c + 1): afterwards lane 4r + c holds row r of the transpose.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D = A(16x16, bf16, row) * B(16x8, bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> packed bf16 pair (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// D = A(16x16, f16, row) * B(16x8, f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> packed f16 pair (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Halves of a packed f16 pair -> floats (exact).
__device__ __forceinline__ float f16_lo(uint32_t w) {
  float f;
  asm("{ .reg .f16 a, b; mov.b32 {a, b}, %1; cvt.f32.f16 %0, a; }" : "=f"(f) : "r"(w));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  float f;
  asm("{ .reg .f16 a, b; mov.b32 {a, b}, %1; cvt.f32.f16 %0, b; }" : "=f"(f) : "r"(w));
  return f;
}

// Two FP8 E4M3 codes (low byte first) -> packed f16 pair (exact: every E4M3 value is an f16).
// Four E4M3 codes (bytes 0..3 of w) -> two f16x2: lo = codes 0, 1; hi = codes 2, 3 (exact).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two floats -> two FP8 E4M3 codes (round to nearest even, saturated to +-448); `lo` in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// bf16 pair packed in a 32-bit word -> two floats (exact: bf16 is the top half of a float).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Loads 16 bytes of stored elements from shared memory and widens them to floats.
template <typename T>
struct Widen;

template <>
struct Widen<float> {
  static constexpr int kPer16 = 4;  // elements per 16 bytes
  __device__ __forceinline__ static void load(const unsigned char* p, float* f) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};

template <>
struct Widen<__nv_bfloat16> {
  static constexpr int kPer16 = 8;
  __device__ __forceinline__ static void load(const unsigned char* p, float* f) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  }
};

}  // namespace pkv_dev
