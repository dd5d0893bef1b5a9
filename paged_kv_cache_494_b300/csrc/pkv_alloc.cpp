// Host block allocator of libpagedkv: pool of fixed-size blocks, per-sequence block tables,
// reference counts, fork (prefix sharing) and copy-on-write of the partially filled last block.
//
// Mechanism from the pages: blocks drawn from a shared pool as tokens arrive and a block table
// per request ("¿Cómo gestiona Paged Attention la caché KV...?", "PagedAttention divide el estado
// KV en bloques de tamaño fijo"); unshared blocks return to the pool when a request ends ("Los
// bloques liberados regresan a un conjunto compartido"); reference counts ("La gestión de bloques
// tiene sus propios costes"); sharing of identical prefixes with copy-on-write of the page where a
// request diverges ("PagedAttention e vLLM", "Approfondimento tecnico"; "Paged Attention optimiza
// el uso de memoria en LLMs", copy-on-write paragraph); release of references without freeing
// pages in use ("Servicio de modelos de lenguaje con un presupuesto de memoria" §8).
// The orderings the pages leave open (free-list order, id choice, when a copy fires) are fixed in
// include/pagedkv.h.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>

#include "pkv_pool.hpp"

namespace {

int32_t ceil_div(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }

void add_ref(pkv_pool* p, int32_t b) {
  int32_t& r = p->refcount[b];
  if (r == 0) p->n_used++;
  if (r == 1) p->n_shared++;
  r++;
}

// Returns true when the block became free. A cached block left with only the cache's reference
// becomes evictable.
bool drop_ref(pkv_pool* p, int32_t b) {
  int32_t& r = p->refcount[b];
  r--;
  if (r == 1) {
    p->n_shared--;
    if (!p->prefix_key_of_block.empty() && p->prefix_key_of_block.count(b)) {
      p->evictable.push_back(b);
      p->evictable_pos[b] = std::prev(p->evictable.end());
    }
  }
  if (r == 0) {
    p->n_used--;
    return true;
  }
  return false;
}

int32_t take_block(pkv_pool* p) {
  int32_t b = p->free_stack.back();
  p->free_stack.pop_back();
  add_ref(p, b);
  return b;
}

// Blocks one more position costs a sequence of length len whose last block has refcount rc_last.
int32_t cost_of_one(int32_t len, int32_t B, int32_t rc_last) {
  if (len % B == 0) return 1;
  return rc_last > 1 ? 1 : 0;
}

// Appends one position to a live sequence; returns its slot. Emits at most one CoW pair.
int64_t append_one(pkv_pool* p, int32_t seq, int32_t* pair_out, int32_t* n_pair) {
  const int32_t B = p->desc.block_size;
  std::vector<int32_t>& t = p->tables[seq];
  int32_t& len = p->lens[seq];
  if (len % B == 0) {
    t.push_back(take_block(p));
  } else if (p->refcount[t.back()] > 1) {
    const int32_t old = t.back();
    const int32_t dst = take_block(p);
    pair_out[0] = old;
    pair_out[1] = dst;
    (*n_pair)++;
    drop_ref(p, old);   // still referenced by the other holders
    t.back() = dst;
    p->n_cow++;
  }
  const int64_t slot = static_cast<int64_t>(t[len / B]) * B + len % B;
  len++;
  p->n_tokens++;
  return slot;
}

bool injected_failure(const pkv_pool* p) {
  return p->desc.fail_after_n_allocs >= 0 && p->n_allocs_ok >= p->desc.fail_after_n_allocs;
}

}  // namespace

extern "C" {

int pkv_version(void) { return PKV_VERSION; }

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID: return "invalid argument";
    case PKV_ERR_NO_BLOCKS: return "not enough free blocks";
    case PKV_ERR_NO_SEQ: return "sequence is not live";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_DEVICE_BOUNDS: return "kernel met a block id or slot outside the pool";
    case PKV_ERR_CAPACITY: return "sequence or block-table capacity exceeded";
    case PKV_ERR_DEVICE_TIMEOUT: return "kernel timed out waiting for its own copy";
    case PKV_ERR_SCRATCH_TOO_SMALL: return "call needs more scratch than the library's built-in array holds";
  }
  return "unknown status";
}

pkv_status pkv_pool_create(const pkv_pool_desc* d, pkv_pool** out) {
  if (!d || !out) return PKV_ERR_INVALID;
  *out = nullptr;
  if (d->num_layers < 1 || d->num_kv_heads < 1 || d->head_dim < 1 || d->block_size < 1 || d->num_blocks < 1 ||
      d->max_seqs < 1 || d->max_blocks_per_seq < 1 ||
      (d->dtype != PKV_F32 && d->dtype != PKV_BF16 && d->dtype != PKV_FP8))
    return PKV_ERR_INVALID;
  pkv_pool* p = new (std::nothrow) pkv_pool();
  if (!p) return PKV_ERR_INVALID;
  p->desc = *d;
  p->desc.initial_free_list = nullptr;
  const int32_t NB = d->num_blocks;
  std::vector<int32_t> order(NB);
  if (d->initial_free_list) {
    std::vector<uint8_t> seen(NB, 0);
    for (int32_t i = 0; i < NB; ++i) {
      const int32_t b = d->initial_free_list[i];
      if (b < 0 || b >= NB || seen[b]) {
        delete p;
        return PKV_ERR_INVALID;
      }
      seen[b] = 1;
      order[i] = b;
    }
  } else {
    for (int32_t i = 0; i < NB; ++i) order[i] = i;
  }
  p->free_stack.assign(order.rbegin(), order.rend());   // order[0] on top
  p->refcount.assign(NB, 0);
  p->tables.resize(d->max_seqs);
  p->lens.assign(d->max_seqs, 0);
  p->live.assign(d->max_seqs, 0);
  for (int32_t s = 0; s < d->max_seqs; ++s) p->free_ids.insert(p->free_ids.end(), s);
  *out = p;
  return PKV_OK;
}

void pkv_pool_destroy(pkv_pool* p) { delete p; }

int64_t pkv_bytes_per_token(const pkv_pool* p) {
  if (!p) return 0;
  const int64_t codes = 2LL * p->desc.num_layers * p->desc.num_kv_heads * p->desc.head_dim * pkv::elem_bytes(p->desc.dtype);
  const int64_t scales = p->desc.dtype == PKV_FP8 ? 2LL * p->desc.num_layers * p->desc.num_kv_heads * 4 : 0;
  return codes + scales;
}

int64_t pkv_layer_scale_bytes(const pkv_pool* p) {
  if (!p || p->desc.dtype != PKV_FP8) return 0;
  return static_cast<int64_t>(p->desc.num_blocks) * p->desc.num_kv_heads * p->desc.block_size * 4;
}

int64_t pkv_layer_cache_bytes(const pkv_pool* p) {
  if (!p) return 0;
  return static_cast<int64_t>(p->desc.num_blocks) * p->desc.num_kv_heads * p->desc.block_size * p->desc.head_dim *
         pkv::elem_bytes(p->desc.dtype);
}

pkv_status pkv_alloc(pkv_pool* p, int32_t seq, int32_t n_tokens, int32_t* seq_out, int64_t* slots_out,
                     int32_t* cow_pairs_out, int32_t* n_cow_out) {
  if (!p || !seq_out || !cow_pairs_out || !n_cow_out || n_tokens < 0 || (n_tokens > 0 && !slots_out))
    return PKV_ERR_INVALID;
  const int32_t B = p->desc.block_size;
  int32_t len = 0, rc_last = 0;
  if (seq == -1) {
    if (p->free_ids.empty()) return PKV_ERR_CAPACITY;
  } else {
    if (seq < 0 || seq >= p->desc.max_seqs || !p->live[seq]) return PKV_ERR_NO_SEQ;
    len = p->lens[seq];
    if (!p->tables[seq].empty() && p->tables[seq].back() >= 0) rc_last = p->refcount[p->tables[seq].back()];
  }
  const int64_t new_len = static_cast<int64_t>(len) + n_tokens;
  if (ceil_div(new_len, B) > p->desc.max_blocks_per_seq) return PKV_ERR_CAPACITY;
  if (injected_failure(p)) return PKV_ERR_NO_BLOCKS;
  int64_t need = ceil_div(new_len, B) - ceil_div(len, B);
  if (n_tokens > 0 && len % B != 0 && rc_last > 1) need++;
  if (need > static_cast<int64_t>(p->free_stack.size())) return PKV_ERR_NO_BLOCKS;
  // commit
  if (seq == -1) {
    seq = *p->free_ids.begin();
    p->free_ids.erase(p->free_ids.begin());
    p->live[seq] = 1;
    p->lens[seq] = 0;
    p->tables[seq].clear();
  }
  int32_t n_pair = 0;
  for (int32_t i = 0; i < n_tokens; ++i) slots_out[i] = append_one(p, seq, cow_pairs_out, &n_pair);
  *seq_out = seq;
  *n_cow_out = n_pair;
  p->n_allocs_ok++;
  return PKV_OK;
}

pkv_status pkv_append(pkv_pool* p, const int32_t* seqs, int32_t n, int64_t* slots_out, int32_t* cow_pairs_out,
                      int32_t* n_cow_out) {
  if (!p || n < 0 || !n_cow_out || (n > 0 && (!seqs || !slots_out || !cow_pairs_out))) return PKV_ERR_INVALID;
  const int32_t B = p->desc.block_size;
  {
    std::vector<int32_t> sorted(seqs, seqs + n);
    std::sort(sorted.begin(), sorted.end());
    if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return PKV_ERR_INVALID;
  }
  for (int32_t i = 0; i < n; ++i)
    if (seqs[i] < 0 || seqs[i] >= p->desc.max_seqs || !p->live[seqs[i]]) return PKV_ERR_NO_SEQ;
  for (int32_t i = 0; i < n; ++i)
    if (ceil_div(static_cast<int64_t>(p->lens[seqs[i]]) + 1, B) > p->desc.max_blocks_per_seq) return PKV_ERR_CAPACITY;
  if (injected_failure(p)) return PKV_ERR_NO_BLOCKS;
  // dry run in order: a copy-on-write lowers the shared block's count seen by later sequences
  std::unordered_map<int32_t, int32_t> rc_delta;
  int64_t need = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = seqs[i];
    const int32_t len = p->lens[s];
    int32_t rc_last = 0, last = -1;
    if (!p->tables[s].empty() && p->tables[s].back() >= 0) {   // a released last block is a hole (-1)
      last = p->tables[s].back();
      rc_last = p->refcount[last] + rc_delta[last];
    }
    const int32_t c = cost_of_one(len, B, rc_last);
    if (len % B != 0 && c == 1) rc_delta[last]--;
    need += c;
  }
  if (need > static_cast<int64_t>(p->free_stack.size())) return PKV_ERR_NO_BLOCKS;
  int32_t n_pair = 0;
  for (int32_t i = 0; i < n; ++i) slots_out[i] = append_one(p, seqs[i], cow_pairs_out + 2 * n_pair, &n_pair);
  *n_cow_out = n_pair;
  p->n_allocs_ok++;
  return PKV_OK;
}

pkv_status pkv_fork(pkv_pool* p, int32_t parent, int32_t* child_out) {
  if (!p || !child_out) return PKV_ERR_INVALID;
  if (parent < 0 || parent >= p->desc.max_seqs || !p->live[parent]) return PKV_ERR_NO_SEQ;
  if (p->free_ids.empty()) return PKV_ERR_CAPACITY;
  const int32_t c = *p->free_ids.begin();
  p->free_ids.erase(p->free_ids.begin());
  p->live[c] = 1;
  p->tables[c] = p->tables[parent];
  p->lens[c] = p->lens[parent];
  for (int32_t b : p->tables[c])
    if (b >= 0) add_ref(p, b);   // released (sliding-window) entries stay holes
  p->n_tokens += p->lens[c];
  *child_out = c;
  return PKV_OK;
}

pkv_status pkv_free(pkv_pool* p, int32_t seq) {
  if (!p) return PKV_ERR_INVALID;
  if (seq < 0 || seq >= p->desc.max_seqs || !p->live[seq]) return PKV_ERR_NO_SEQ;
  for (int32_t b : p->tables[seq])
    if (b >= 0 && drop_ref(p, b)) p->free_stack.push_back(b);
  p->n_tokens -= p->lens[seq];
  p->tables[seq].clear();
  p->lens[seq] = 0;
  p->live[seq] = 0;
  p->free_ids.insert(seq);
  return PKV_OK;
}

pkv_status pkv_release_before(pkv_pool* p, int32_t seq, int32_t position, int32_t* n_released_out) {
  if (!p) return PKV_ERR_INVALID;
  if (seq < 0 || seq >= p->desc.max_seqs || !p->live[seq]) return PKV_ERR_NO_SEQ;
  if (position < 0 || position > p->lens[seq]) return PKV_ERR_INVALID;
  const int32_t B = p->desc.block_size;
  std::vector<int32_t>& t = p->tables[seq];
  int32_t released = 0;
  for (int32_t i = 0; i < static_cast<int32_t>(t.size()) && static_cast<int64_t>(i + 1) * B <= position; ++i) {
    if (t[i] < 0) continue;
    if (drop_ref(p, t[i])) p->free_stack.push_back(t[i]);
    t[i] = -1;
    ++released;
  }
  if (n_released_out) *n_released_out = released;
  return PKV_OK;
}

pkv_status pkv_alloc_prefix(pkv_pool* p, uint64_t ns, const int32_t* tokens, int32_t n_tokens, int32_t* seq_out,
                            int64_t* slots_out, int32_t* n_cached_out) {
  if (!p || !seq_out || !n_cached_out || n_tokens < 0 || (n_tokens > 0 && (!tokens || !slots_out)))
    return PKV_ERR_INVALID;
  const int32_t B = p->desc.block_size;
  if (p->free_ids.empty()) return PKV_ERR_CAPACITY;
  const int32_t nblk = ceil_div(n_tokens, B);
  if (nblk > p->desc.max_blocks_per_seq) return PKV_ERR_CAPACITY;
  if (injected_failure(p)) return PKV_ERR_NO_BLOCKS;
  // leading full blocks found in the cache
  std::vector<int32_t> hits;
  int64_t parent = -1;
  PrefixKey key;
  key.ns = ns;
  for (int32_t i = 0; i < n_tokens / B; ++i) {
    key.parent = parent;
    key.tokens.assign(tokens + static_cast<int64_t>(i) * B, tokens + static_cast<int64_t>(i + 1) * B);
    auto it = p->prefix_entries.find(key);
    if (it == p->prefix_entries.end()) break;
    hits.push_back(it->second.block);
    parent = it->second.id;
  }
  const int64_t need = nblk - static_cast<int64_t>(hits.size());
  if (need > static_cast<int64_t>(p->free_stack.size())) return PKV_ERR_NO_BLOCKS;
  // commit
  const int32_t seq = *p->free_ids.begin();
  p->free_ids.erase(p->free_ids.begin());
  p->live[seq] = 1;
  std::vector<int32_t>& t = p->tables[seq];
  t.clear();
  for (int32_t blk : hits) {
    if (p->refcount[blk] == 1) {  // was held by the cache alone: no longer evictable
      p->evictable.erase(p->evictable_pos[blk]);
      p->evictable_pos.erase(blk);
    }
    add_ref(p, blk);
    t.push_back(blk);
  }
  for (int32_t i = static_cast<int32_t>(hits.size()); i < nblk; ++i) {
    const int32_t blk = take_block(p);
    t.push_back(blk);
    if (static_cast<int64_t>(i + 1) * B <= n_tokens) {  // full block: register it
      key.parent = parent;
      key.tokens.assign(tokens + static_cast<int64_t>(i) * B, tokens + static_cast<int64_t>(i + 1) * B);
      const int64_t id = p->next_entry_id++;
      p->prefix_entries[key] = PrefixEntry{id, blk};
      p->prefix_key_of_block[blk] = key;
      add_ref(p, blk);  // the cache's own reference
      parent = id;
    }
  }
  p->lens[seq] = n_tokens;
  p->n_tokens += n_tokens;
  for (int32_t pos = 0; pos < n_tokens; ++pos) slots_out[pos] = static_cast<int64_t>(t[pos / B]) * B + pos % B;
  *seq_out = seq;
  *n_cached_out = static_cast<int32_t>(hits.size()) * B;
  p->n_allocs_ok++;
  return PKV_OK;
}

pkv_status pkv_prefix_evict(pkv_pool* p, int32_t max_blocks, int32_t* n_evicted_out) {
  if (!p || max_blocks < 0) return PKV_ERR_INVALID;
  int32_t n = 0;
  while (n < max_blocks && !p->evictable.empty()) {
    const int32_t blk = p->evictable.front();
    p->evictable.pop_front();
    p->evictable_pos.erase(blk);
    auto kit = p->prefix_key_of_block.find(blk);
    p->prefix_entries.erase(kit->second);
    p->prefix_key_of_block.erase(kit);
    if (drop_ref(p, blk)) p->free_stack.push_back(blk);
    ++n;
  }
  if (n_evicted_out) *n_evicted_out = n;
  return PKV_OK;
}

pkv_status pkv_prefix_stats(const pkv_pool* p, int32_t* n_cached_blocks, int32_t* n_evictable) {
  if (!p) return PKV_ERR_INVALID;
  if (n_cached_blocks) *n_cached_blocks = static_cast<int32_t>(p->prefix_entries.size());
  if (n_evictable) *n_evictable = static_cast<int32_t>(p->evictable.size());
  return PKV_OK;
}

pkv_status pkv_block_table(const pkv_pool* p, const int32_t* seqs, int32_t n, int32_t* table_out,
                           int32_t* lens_out) {
  if (!p || n < 0 || (n > 0 && !seqs)) return PKV_ERR_INVALID;
  for (int32_t i = 0; i < n; ++i)
    if (seqs[i] < 0 || seqs[i] >= p->desc.max_seqs || !p->live[seqs[i]]) return PKV_ERR_NO_SEQ;
  const int32_t MB = p->desc.max_blocks_per_seq;
  for (int32_t i = 0; i < n; ++i) {
    const std::vector<int32_t>& t = p->tables[seqs[i]];
    if (table_out) {
      int32_t* row = table_out + static_cast<int64_t>(i) * MB;
      std::copy(t.begin(), t.end(), row);
      std::fill(row + t.size(), row + MB, -1);
    }
    if (lens_out) lens_out[i] = p->lens[seqs[i]];
  }
  return PKV_OK;
}

pkv_status pkv_shared_prefix_blocks(const pkv_pool* p, const int32_t* seqs, int32_t n, int32_t* out_blocks) {
  if (!p || n <= 0 || !seqs || !out_blocks) return PKV_ERR_INVALID;
  for (int32_t i = 0; i < n; ++i)
    if (seqs[i] < 0 || seqs[i] >= p->desc.max_seqs || !p->live[seqs[i]]) return PKV_ERR_NO_SEQ;
  // full blocks of the shortest sequence bound the count; then the first logical block whose
  // physical id differs between any two sequences ends it
  int64_t k_max = INT64_MAX;
  for (int32_t i = 0; i < n; ++i) k_max = std::min<int64_t>(k_max, p->lens[seqs[i]] / p->desc.block_size);
  const std::vector<int32_t>& t0 = p->tables[seqs[0]];
  int64_t k = 0;
  for (; k < k_max; ++k) {
    bool same = true;
    for (int32_t i = 1; i < n && same; ++i) same = p->tables[seqs[i]][k] == t0[k];
    if (!same) break;
  }
  *out_blocks = static_cast<int32_t>(k);
  return PKV_OK;
}

pkv_status pkv_pool_stats(const pkv_pool* p, pkv_stats* out) {
  if (!p || !out) return PKV_ERR_INVALID;
  out->num_free = static_cast<int32_t>(p->free_stack.size());
  out->num_used = p->n_used;
  out->num_shared = p->n_shared;
  out->num_seqs = p->desc.max_seqs - static_cast<int32_t>(p->free_ids.size());
  out->num_cow = p->n_cow;
  out->num_tokens = p->n_tokens;
  return PKV_OK;
}

pkv_status pkv_export_state(const pkv_pool* p, int32_t* refcounts, int32_t* free_list, int32_t* n_free) {
  if (!p) return PKV_ERR_INVALID;
  if (refcounts) std::copy(p->refcount.begin(), p->refcount.end(), refcounts);
  if (free_list) std::copy(p->free_stack.begin(), p->free_stack.end(), free_list);
  if (n_free) *n_free = static_cast<int32_t>(p->free_stack.size());
  return PKV_OK;
}

}  // extern "C"
