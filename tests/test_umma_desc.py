"""The tensor-core descriptor encoders (paged_kv_cache_494_b300/csrc/umma_desc.hpp) against encodings
worked out by hand from the field tables in that header, for the exact operand shapes the tcgen05
prefill kernel issues (CPU only: the header is plain C++ compiled here with g++).

Hand-worked values:
* S = Q K^T, M 128, N 32 keys, A and B K-major, bf16 in, f32 out:
    f32 accumulate (1 << 4) = 0x10, A bf16 (1 << 7) = 0x80, B bf16 (1 << 10) = 0x400,
    N >> 3 = 4 at bit 17 = 0x80000, M >> 4 = 8 at bit 24 = 0x8000000      -> 0x08080490
* O += P V, M 128, N = D = 128, A K-major, B (V, dims contiguous) MN-major (1 << 16) = 0x10000,
    N >> 3 = 16 at bit 17 = 0x200000                                        -> 0x08210490
  and with D = 64: N >> 3 = 8 at bit 17 = 0x100000                         -> 0x08110490
* K-major operand at shared address 0x400, 128-byte swizzle, SBO 1024 (8 rows of 128 bytes), LBO 16:
    address >> 4 = 0x40, LBO >> 4 = 1 at bit 16 = 0x10000, SBO >> 4 = 0x40 at bit 32,
    version 1 at bit 46 = 0x4000_0000_0000, swizzle 2 at bit 61 = 0x4000_0000_0000_0000
                                                                            -> 0x4000404000010040
* MN-major V operand at 0x9000, LBO 4096 (next 64-dim half), SBO 1024      -> 0x4000404001000900
"""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_cache_494_b300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "umma_desc.hpp"
using namespace pkv_umma;
int main() {
  std::printf("%08x\n", idesc_bf16_f32(128, 32, false, false));
  std::printf("%08x\n", idesc_bf16_f32(128, 128, false, true));
  std::printf("%08x\n", idesc_bf16_f32(128, 64, false, true));
  std::printf("%016llx\n", (unsigned long long)smem_desc(0x400, 16, 1024, kSwizzle128B));
  std::printf("%016llx\n", (unsigned long long)smem_desc(0x9000, 4096, 1024, kSwizzle128B));
  std::printf("%016llx\n", (unsigned long long)smem_desc(0x12340, 16, 1024, kSwizzleNone));
  std::printf("%d %d %d %d %d\n", (int)valid_f16_shape(128, 32), (int)valid_f16_shape(128, 128),
              (int)valid_f16_shape(128, 24), (int)valid_f16_shape(256, 64), (int)valid_f16_shape(64, 8));
  return 0;
}
"""


@pytest.fixture(scope="module")
def encodings(tmp_path_factory):
    d = tmp_path_factory.mktemp("umma")
    src = d / "enc.cpp"
    src.write_text(PROGRAM)
    exe = d / "enc"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, "-o", str(exe), str(src)], check=True)
    return subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")


def test_instruction_descriptors(encodings):
    assert encodings[0] == "08080490"      # S = Q K^T: M 128, N 32
    assert encodings[1] == "08210490"      # O += P V: M 128, N 128, B MN-major
    assert encodings[2] == "08110490"      # O += P V: M 128, N 64, B MN-major


def test_shared_memory_descriptors(encodings):
    assert encodings[3] == "4000404000010040"
    assert encodings[4] == "4000404001000900"
    # no swizzle: layout field 0; the start address keeps bits 4..17 of 0x12340 -> 0x1234
    assert encodings[5] == "0000404000011234"


def test_shape_rules(encodings):
    assert encodings[6] == "1 1 0 0 1"
