// Internal pool state shared by the host allocator and the device-op entry points.
#pragma once

#include <cstdint>
#include <set>
#include <vector>

#include "pagedkv.h"

struct pkv_pool {
  pkv_pool_desc desc{};                       // copy; desc.initial_free_list is cleared
  std::vector<int32_t> free_stack;            // back() is handed out next
  std::vector<int32_t> refcount;              // [num_blocks]
  std::vector<std::vector<int32_t>> tables;   // [max_seqs] logical -> physical block
  std::vector<int32_t> lens;                  // [max_seqs]
  std::vector<uint8_t> live;                  // [max_seqs]
  std::set<int32_t> free_ids;                 // unused sequence ids, smallest first
  int64_t n_cow = 0;
  int64_t n_allocs_ok = 0;                    // successful pkv_alloc / pkv_append calls
  int64_t n_tokens = 0;
  int32_t n_used = 0;                         // blocks with refcount > 0
  int32_t n_shared = 0;                       // blocks with refcount > 1
};

namespace pkv {
inline int elem_bytes(int32_t dtype) { return dtype == PKV_F32 ? 4 : 2; }
}  // namespace pkv
