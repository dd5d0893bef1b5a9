// Encoders of the two descriptors a 5th-generation tensor-core MMA (tcgen05.mma, kind::f16) reads:
// the 64-bit shared-memory matrix descriptor and the 32-bit instruction descriptor. Plain C++
// (constexpr, no CUDA types) so that the host-side unit test compiles them with g++ and checks them
// against encodings worked out by hand from the field tables below.
//
// Shared-memory matrix descriptor (one per operand in shared memory):
//   bits  0-13  start address >> 4 (shared-window byte address, 16-byte aligned)
//   bits 16-29  leading-dimension byte offset >> 4 (LBO)
//   bits 32-45  stride-dimension byte offset >> 4 (SBO)
//   bits 46-47  descriptor version, 1 for tcgen05
//   bits 49-51  base offset (0: every swizzle atom starts on its natural alignment)
//   bit  52     LBO mode (0: relative byte offset)
//   bits 61-63  layout / swizzle: 0 none, 2 = 128-byte swizzle, 4 = 64-byte, 6 = 32-byte
// With the 128-byte swizzle an atom is 8 rows x 128 bytes (1024 bytes, 1024-aligned):
//   K-major operand (K contiguous in a row): SBO = distance between 8-row groups along M/N; a
//     16-element K step inside the 128-byte row is addressed by advancing the start address by
//     32 bytes (the swizzle is a function of the address, so the hardware finds the right chunk);
//     LBO is not used.
//   MN-major operand (M/N contiguous in a row, K = rows): LBO = distance between 64-element atoms
//     along M/N, SBO = distance between 8-row groups along K.
//
// Instruction descriptor, kind::f16 (A and B 16-bit, the same type):
//   bits  4-5   accumulator format (1 = f32)
//   bits  7-9   A format (0 = f16, 1 = bf16)
//   bits 10-12  B format (0 = f16, 1 = bf16)
//   bit  13/14  negate A / B (0)
//   bit  15     A major (0 = K-major, 1 = MN-major)
//   bit  16     B major (0 = K-major, 1 = MN-major)
//   bits 17-22  N >> 3
//   bits 24-28  M >> 4
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define PKV_HD __host__ __device__
#else
#define PKV_HD
#endif

namespace pkv_umma {

enum : uint32_t { kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6 };

PKV_HD constexpr uint64_t smem_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes, uint32_t swizzle) {
  return static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(swizzle & 7u) << 61);
}

// f32 accumulate, bf16 A and B.
PKV_HD constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shapes one CTA of kind::f16 with cta_group::1 may issue: M 64 or 128, N a multiple of 8 (M 64)
// or 16 (M 128) between 8/16 and 256.
PKV_HD constexpr bool valid_f16_shape(int M, int N) {
  return (M == 64 && N >= 8 && N <= 256 && N % 8 == 0) || (M == 128 && N >= 16 && N <= 256 && N % 16 == 0);
}

}  // namespace pkv_umma
