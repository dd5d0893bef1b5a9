// Internal pool state shared by the host allocator and the device-op entry points.
#pragma once

#include <cstdint>
#include <list>
#include <set>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

// Key of a cached prompt block: cache namespace, the entry id of the previous block of the prompt
// (-1 for the first block) and the block's token ids.
struct PrefixKey {
  uint64_t ns = 0;
  int64_t parent = -1;
  std::vector<int32_t> tokens;
  bool operator==(const PrefixKey& o) const { return ns == o.ns && parent == o.parent && tokens == o.tokens; }
};

struct PrefixKeyHash {
  size_t operator()(const PrefixKey& k) const {
    uint64_t h = 1469598103934665603ull;  // FNV-1a over the key's words
    auto mix = [&h](uint64_t v) {
      for (int i = 0; i < 8; ++i) {
        h ^= (v >> (8 * i)) & 0xffu;
        h *= 1099511628211ull;
      }
    };
    mix(k.ns);
    mix(static_cast<uint64_t>(k.parent));
    for (int32_t t : k.tokens) mix(static_cast<uint32_t>(t));
    return static_cast<size_t>(h);
  }
};

struct PrefixEntry {
  int64_t id;
  int32_t block;
};

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
  // prefix cache (pkv_alloc_prefix): the cache holds one reference on every cached block
  std::unordered_map<PrefixKey, PrefixEntry, PrefixKeyHash> prefix_entries;
  std::unordered_map<int32_t, PrefixKey> prefix_key_of_block;
  int64_t next_entry_id = 0;
  std::list<int32_t> evictable;               // cached blocks held only by the cache, oldest first
  std::unordered_map<int32_t, std::list<int32_t>::iterator> evictable_pos;
  // device error word the pool's kernels record into (pkv_pool_set_error_word); null: process-wide
  unsigned int* d_err_word = nullptr;
};

namespace pkv {
inline int elem_bytes(int32_t dtype) { return dtype == PKV_F32 ? 4 : (dtype == PKV_FP8 ? 1 : 2); }
}  // namespace pkv
