/*
 * libpagedkv — paged KV cache and paged decode attention for NVIDIA B300 (sm_103a).
 *
 * C ABI. Every entry point returns a pkv_status (nothing throws across the boundary).
 * Plain pointers and sizes only. "host" pointers are ordinary CPU memory; "device"
 * pointers are CUDA global memory on the current device, owned by the caller. The
 * library allocates no device memory: caches, q, outputs, tables and workspaces all
 * belong to the caller. Device operations are enqueued on the caller's stream
 * (a cudaStream_t passed as void*; NULL = legacy default stream) and never synchronise,
 * except pkv_last_error. Kernels are launched with programmatic dependent launch (unless
 * PKV_PDL=0): a decode kernel may start while the kernel before it on the stream is still
 * running, once that kernel allows it (griddepcontrol.launch_dependents; library kernels do so),
 * and reads context_lens and block_tables before it waits for that kernel to finish; it reads
 * the caches, q and the workspace, and writes its outputs, only after the wait (only a bad length
 * may be recorded in the error word before it). A kernel of the caller that allows its dependents
 * to launch early must not write context_lens or block_tables after doing so.
 *
 * Method (sources are the pages this library implements):
 *  - KV state of a request lives in fixed-size physical blocks of B token positions
 *    drawn from a shared pool as tokens arrive; a per-request block table maps logical
 *    order to physical blocks ("¿Cómo gestiona Paged Attention la caché KV cuando hay
 *    solicitudes simultáneas de IA local?", section "PagedAttention divide el estado KV
 *    en bloques de tamaño fijo"; "Paged Attention optimiza el uso de memoria en LLMs",
 *    16-token pages and the page table).
 *  - Finished requests return their unshared blocks to the pool at once ("¿Cómo gestiona
 *    Paged Attention la caché KV...?", "Los bloques liberados regresan a un conjunto
 *    compartido"); the runtime keeps
 *    block tables and reference counts ("La gestión de bloques tiene sus propios costes").
 *  - Identical prefixes share physical pages; only the page where a request diverges is
 *    copied ("PagedAttention e vLLM", "Approfondimento tecnico"; "Paged Attention optimiza
 *    el uso de memoria en LLMs", copy-on-write paragraph). Cancellation releases references without freeing pages
 *    still in use ("Servicio de modelos de lenguaje con un presupuesto de memoria" §8).
 *  - Decode attention is exact softmax(scale * q.K^T) V, computed blockwise with running
 *    max/sum statistics (same page §6); GQA query heads share a KV head in contiguous
 *    groups ("¿Cuánta memoria reservar para la caché KV?", "Emplear las cabezas KV").
 *
 * Cache layout (one K and one V tensor per layer, same for every layer):
 *     cache[num_blocks][num_kv_heads][block_size][head_dim]   (dtype of the pool)
 * Token slot s (from pkv_alloc) lives at block s / block_size, offset s % block_size.
 * Block ids are shared by all layers: one block table serves every layer, since every
 * layer stores every token (per-token budget 2*L*Hkv*D*bytes, "Servicio de modelos de
 * lenguaje con un presupuesto de memoria" §3).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_VERSION 1

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef struct pkv_pool pkv_pool; /* opaque; the library owns all host metadata */

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID = -1,        /* bad argument (null pointer, size, alignment, dtype, unsupported shape) */
  PKV_ERR_NO_BLOCKS = -2,      /* pool has too few free blocks for the whole call (or injected failure) */
  PKV_ERR_NO_SEQ = -3,         /* sequence id is not live */
  PKV_ERR_CUDA = -4,           /* a CUDA runtime call failed (launch, attribute, device query) */
  PKV_ERR_DEVICE_BOUNDS = -5,  /* a kernel met a block id or slot outside the pool and skipped it */
  PKV_ERR_CAPACITY = -6,       /* max_seqs or max_blocks_per_seq would be exceeded */
  PKV_ERR_DEVICE_TIMEOUT = -7, /* a kernel gave up waiting for a copy it issued (bounded wait) */
  PKV_ERR_SCRATCH_TOO_SMALL = -8 /* pkv_paged_decode_static: the call needs more than the built-in scratch */
} pkv_status;

/* Storage type of a pool. PKV_FP8: K and V as FP8 E4M3 codes with one float32 scale per (token,
 * KV head) for K and one for V; q stays bf16. FP8 layouts: k_cache [NB][Hkv][B][D] codes (token-major
 * like the others), v_cache [NB][Hkv][D][B] codes (dim-major within a page; each 16-token group of
 * a dim row in the token order 0,1,8,9,2,3,10,11,4,5,12,13,6,7,14,15), k_scale / v_scale
 * [NB][Hkv][B] float32. Quantising the cache is one of the cache strategies ("¿Cuánta memoria reservar
 * para la caché KV?", "Adaptar el presupuesto a la estrategia de caché"); it changes the numerics, so
 * fp8 pools use the *_fp8 entry points and their own contract. */
typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_FP8 = 2 } pkv_dtype;

typedef struct {
  int32_t num_layers;          /* layers sharing the block table (>= 1) */
  int32_t num_kv_heads;        /* Hkv (>= 1) */
  int32_t head_dim;            /* D; device ops support 64 and 128 */
  int32_t block_size;          /* B tokens per block (>= 1; device ops need a multiple of 16) */
  int32_t num_blocks;          /* NB physical blocks in the pool */
  int32_t max_seqs;            /* sequence ids are 0 .. max_seqs-1 */
  int32_t max_blocks_per_seq;  /* MB: row length of block tables */
  int32_t dtype;               /* pkv_dtype of q, K and V */
  const int32_t* initial_free_list; /* host, optional: permutation of [0, NB) giving the order in
                                       which blocks are first handed out; NULL = 0, 1, ..., NB-1.
                                       Copied at create time. */
  int32_t fail_after_n_allocs; /* host fault injection: once this many pkv_alloc/pkv_append calls
                                  have succeeded, later ones fail with PKV_ERR_NO_BLOCKS and change
                                  nothing. -1 = off. */
} pkv_pool_desc;

typedef struct {
  int32_t num_free;    /* blocks on the free list */
  int32_t num_used;    /* blocks with refcount > 0 */
  int32_t num_shared;  /* blocks with refcount > 1 */
  int32_t num_seqs;    /* live sequences */
  int64_t num_cow;     /* copy-on-write pairs emitted since creation */
  int64_t num_tokens;  /* sum of live sequence lengths */
} pkv_stats;

/* ---- library info ----------------------------------------------------------------------- */

PKV_API int pkv_version(void);
PKV_API const char* pkv_status_string(pkv_status status);

/* ---- pool (host) -------------------------------------------------------------------------- */

/* Create a pool. desc is read and copied (host). On success *out owns the pool. Errors:
 * PKV_ERR_INVALID for non-positive sizes, an unknown dtype or a list that is not a permutation. */
PKV_API pkv_status pkv_pool_create(const pkv_pool_desc* desc, pkv_pool** out);
PKV_API void pkv_pool_destroy(pkv_pool* pool);

/* Bytes of K plus V per token across all layers: 2 * L * Hkv * D * sizeof(dtype)
 * ("Servicio de modelos de lenguaje con un presupuesto de memoria" §3); fp8 pools add their scales,
 * 2 * L * Hkv * 4 bytes. */
PKV_API int64_t pkv_bytes_per_token(const pkv_pool* pool);
/* Bytes of ONE cache tensor (K or V) of ONE layer: NB * Hkv * B * D * sizeof(dtype). */
PKV_API int64_t pkv_layer_cache_bytes(const pkv_pool* pool);
/* fp8 pools: bytes of ONE scale tensor (k_scale or v_scale) of ONE layer, NB * Hkv * B * 4; else 0. */
PKV_API int64_t pkv_layer_scale_bytes(const pkv_pool* pool);

/* ---- allocator (host only, no device work, all-or-nothing) ---------------------------------- */

/* Append n_tokens >= 0 positions to sequence seq (seq = -1: create a new sequence, which takes
 * the lowest unused id). For every appended position, in order: if the sequence length is a
 * multiple of B a free block is taken (free list order, LIFO reuse); otherwise, if the partially
 * filled last block has refcount > 1, it is copied on write: a free block dst is taken, the pair
 * (last, dst) is reported, the old block loses a reference and the table points at dst. The slot
 * of position t is table[t / B] * B + t % B.
 * Outputs (host): *seq_out; slots_out[n_tokens] (int64); cow_pairs_out[2] receives (src, dst) when
 * *n_cow_out == 1 (at most one copy per call). slots_out may be NULL when n_tokens == 0.
 * Check order: n_tokens < 0 -> INVALID; new id unavailable -> CAPACITY; seq not live -> NO_SEQ;
 * ceil((len + n) / B) > max_blocks_per_seq -> CAPACITY; injected failure -> NO_BLOCKS;
 * free blocks < blocks needed -> NO_BLOCKS. On error nothing changes. */
PKV_API pkv_status pkv_alloc(pkv_pool* pool, int32_t seq, int32_t n_tokens, int32_t* seq_out, int64_t* slots_out,
                     int32_t* cow_pairs_out, int32_t* n_cow_out);

/* One decode step: append ONE position to each of n distinct live sequences seqs[0..n), in that
 * order, with the pkv_alloc rules. Host outputs: slots_out[n] (int64), cow_pairs_out[2 * n] holding
 * *n_cow_out (src, dst) pairs in emission order. All-or-nothing for the whole batch (duplicate ids:
 * PKV_ERR_INVALID). Counts as one call for fail_after_n_allocs. */
PKV_API pkv_status pkv_append(pkv_pool* pool, const int32_t* seqs, int32_t n, int64_t* slots_out,
                      int32_t* cow_pairs_out, int32_t* n_cow_out);

/* New sequence sharing every block of parent (each block's refcount + 1); takes the lowest
 * unused id. Errors: NO_SEQ, CAPACITY. */
PKV_API pkv_status pkv_fork(pkv_pool* pool, int32_t parent, int32_t* child_out);

/* Release seq: every block of its table, in table order, loses one reference; a block that
 * reaches zero goes on top of the free list. Blocks still referenced elsewhere stay in use. */
PKV_API pkv_status pkv_free(pkv_pool* pool, int32_t seq);

/* Sliding-window release: drop this sequence's reference to every block whose positions all lie
 * before `position` (0 <= position <= length), in table order; a block reaching refcount 0 goes on
 * top of the free list. Released table entries become -1 (a hole); the sequence length is unchanged,
 * so later appends and the slots of remaining positions do not move. Decode with a window that starts
 * at or after `position` never reads the holes ("Adaptar el presupuesto a la estrategia de caché":
 * a window bounds the history a sequence keeps). *n_released_out (may be NULL) = references dropped.
 * Errors: NO_SEQ, INVALID (position out of range). */
PKV_API pkv_status pkv_release_before(pkv_pool* pool, int32_t seq, int32_t position, int32_t* n_released_out);

/* ---- prefix cache (host only) ------------------------------------------------------------- */
/* Prompt blocks are shared by content ("Servicio de modelos de lenguaje con un presupuesto de
 * memoria" §8: the key must cover every input that affects the state, reused pages must never
 * expose another request's continuation, eviction must not free pages in use; "PagedAttention e
 * vLLM", "Implementazione nel mondo reale": a shared system prompt is processed once).
 * The key of prompt block i is (cache_namespace, the cache entry of block i-1, the B token ids of
 * block i); the caller folds the model version and every configuration value that changes K/V into
 * cache_namespace. Only full blocks are cached; a lookup stops at the first miss. Entry ids are never
 * reused, so entries whose parent was evicted can no longer be reached. The cache holds one reference
 * on each cached block; a cached block held by nothing else is evictable. */

/* New sequence for the prompt tokens[0..n_tokens): the leading full blocks found in the cache are
 * shared (refcount + 1); the rest are taken from the free list and the full ones are registered.
 * Outputs: *seq_out; slots_out[n_tokens]; *n_cached_out = number of leading positions whose K/V is
 * already in the cache (a multiple of B) — the caller writes K/V only for positions >= that (and must
 * order those writes before any read of the newly registered blocks, e.g. on one stream).
 * Check order: CAPACITY (no id, or too many blocks), injected failure, NO_BLOCKS (free list too short;
 * the cache is not evicted implicitly). All-or-nothing. */
PKV_API pkv_status pkv_alloc_prefix(pkv_pool* pool, uint64_t cache_namespace, const int32_t* tokens,
                                    int32_t n_tokens, int32_t* seq_out, int64_t* slots_out, int32_t* n_cached_out);

/* Evict up to max_blocks evictable cached blocks, in the order they became evictable (oldest first):
 * each leaves the cache and goes on top of the free list. Blocks any sequence still holds are never
 * evicted. *n_evicted_out (may be NULL) = blocks evicted. */
PKV_API pkv_status pkv_prefix_evict(pkv_pool* pool, int32_t max_blocks, int32_t* n_evicted_out);

/* Number of cached blocks and of evictable ones (either output may be NULL). */
PKV_API pkv_status pkv_prefix_stats(const pkv_pool* pool, int32_t* n_cached_blocks, int32_t* n_evictable);

/* Sharing structure for pkv_paged_decode_shared_prefix: *out_blocks = the number of leading logical
 * blocks k that every one of the n live sequences maps to the same physical block (a prompt forked
 * into children, whose full blocks stay shared until copy-on-write), counting only blocks that are
 * full in every sequence (k < len / block_size for the shortest one). n >= 1. */
PKV_API pkv_status pkv_shared_prefix_blocks(const pkv_pool* pool, const int32_t* seqs, int32_t n,
                                            int32_t* out_blocks);

/* Host copies of the block tables of n live sequences: table_out[n][max_blocks_per_seq]
 * (int32, unused entries -1) and lens_out[n]. Either output may be NULL. */
PKV_API pkv_status pkv_block_table(const pkv_pool* pool, const int32_t* seqs, int32_t n, int32_t* table_out,
                           int32_t* lens_out);

PKV_API pkv_status pkv_pool_stats(const pkv_pool* pool, pkv_stats* out);

/* Allocator state for checking: refcounts[NB]; free_list[NB] from the bottom of the stack to its
 * top (the top is handed out next), first *n_free entries valid. */
PKV_API pkv_status pkv_export_state(const pkv_pool* pool, int32_t* refcounts, int32_t* free_list, int32_t* n_free);

/* ---- device operations -------------------------------------------------------------------- */
/* All pointers below are device pointers unless marked host; they must be 16-byte aligned.
 * Host-side argument errors return PKV_ERR_INVALID before anything is enqueued; a failed launch
 * returns PKV_ERR_CUDA. Kernels never fault on bad block ids or slots: they skip the access and
 * record PKV_ERR_DEVICE_BOUNDS for pkv_last_error. */

/* Slot-mapped append of new K/V (bit copy, no conversion): for each token i with slot s = slots[i]
 * (s < 0: skipped), for every KV head h: k_cache[s/B][h][s%B][:] = k[i][h][:], same for V.
 * k, v: [n_tokens][Hkv][D] in the pool dtype; slots: int64 [n_tokens]; caches: one layer. */
PKV_API pkv_status pkv_reshape_and_cache(const pkv_pool* pool, const void* k, const void* v, const int64_t* slots,
                                 int32_t n_tokens, void* k_cache, void* v_cache, void* stream);

/* Copy-on-write block copies for every layer: for l < num_layers and each pair i (in order),
 * k_caches[l][dst_i] = k_caches[l][src_i] and the same for V (a whole block: Hkv * B * D values).
 * k_caches, v_caches: HOST arrays of num_layers device pointers; pairs: device int32 [n_pairs][2]
 * (src, dst). A dst must not also be a src in the same call (the allocator never emits that). */
PKV_API pkv_status pkv_copy_blocks(const pkv_pool* pool, void* const* k_caches, void* const* v_caches,
                           const int32_t* pairs, int32_t n_pairs, void* stream);

/* Paged decode attention for one layer. For each sequence b < n_seqs and query head j < num_q_heads
 * (num_q_heads a multiple of Hkv; KV head h = j / (num_q_heads / Hkv)):
 *     out[b][j][:] = sum_{t < len_b} softmax_t(scale * q[b][j] . K_b[t]) V_b[t]
 * where K_b[t] = k_cache[block_tables[b][t / B]][h][t % B][:] and len_b = context_lens[b] (the
 * length includes the token appended in this step; len_b == 0 gives a zero row).
 * q: [n_seqs][num_q_heads][D] pool dtype; out: float32 [n_seqs][num_q_heads][D];
 * block_tables: int32 [n_seqs][max_blocks_per_seq]; context_lens: int32 [n_seqs], each at most
 * max_blocks_per_seq * B.
 * partition_tokens = 0: the library splits the total work evenly over the GPU (whole 16-token
 * chunks) and merges the parts of split sequences by log-sum-exp inside the same kernel.
 * partition_tokens > 0 (a multiple of 16): every sequence is cut into partitions of that many
 * tokens, each computed separately and merged the same way. The result never depends on where
 * blocks are placed physically (it may depend, to rounding, on a sequence's batch position).
 * workspace: device scratch of at least pkv_decode_workspace_bytes(...) bytes (may be NULL if that
 * is 0); its contents need no initialisation. Concurrent calls must not share a workspace.
 * Batch size: n_seqs <= 16384. Every CTA also keeps 4 bytes per sequence of prefix sums in shared
 * memory beside its copy ring (8 with partition_tokens > 0 or a window, 12 with both); a batch whose
 * arrays do not fit the device's per-block shared memory is rejected with PKV_ERR_INVALID (on B300
 * with bf16 D = 128 that happens only with both partitions and a window, above 13,796 sequences).
 * Large batches lower the number of resident CTAs per SM.
 * CUDA graphs: a call may be captured in a graph and the graph replayed any number of times (the
 * device pointers and sizes of the call are baked into the graph); every replay computes what a
 * direct call would. Make one direct call of the same shape before capturing: the first call of a
 * shape sets the kernel's shared-memory limit and looks up its occupancy. */
PKV_API pkv_status pkv_paged_decode(const pkv_pool* pool, float* out, const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                            int32_t n_seqs, int32_t num_q_heads, float scale, int32_t partition_tokens,
                            void* workspace, size_t workspace_bytes, void* stream);

/* ---- fp8 pools ------------------------------------------------------------------------------- */

/* Quantising slot-mapped append into an fp8 pool: for each token i with slot s >= 0 and each KV head,
 * the row x = k[i][h][:] (bf16) is stored as codes e4m3(x / scale), rounded to nearest even and
 * saturated to +-448, with scale = amax|x| / 448 (float32 IEEE division; 1 if amax == 0) written to
 * k_scale[s/B][h][s%B]; the same for V into the dim-major v_cache. Deterministic and bit-reproducible. */
PKV_API pkv_status pkv_reshape_and_cache_fp8(const pkv_pool* pool, const void* k, const void* v,
                                             const int64_t* slots, int32_t n_tokens, void* k_cache, void* v_cache,
                                             float* k_scale, float* v_scale, void* stream);

/* Copy-on-write for fp8 pools: as pkv_copy_blocks, also copying the blocks' scales
 * (k_scales / v_scales: HOST arrays of num_layers device pointers). */
PKV_API pkv_status pkv_copy_blocks_fp8(const pkv_pool* pool, void* const* k_caches, void* const* v_caches,
                                       void* const* k_scales, void* const* v_scales, const int32_t* pairs,
                                       int32_t n_pairs, void* stream);

/* Paged decode over an fp8 pool (head_dim 128, num_q_heads / Hkv <= 8): the attention of
 * pkv_paged_decode_window over the dequantised values code * scale (q bf16, out float32), with the
 * same split modes, window and workspace size. Contract: max abs error <= 2e-3 against the exact
 * attention over the dequantised cache; |V| entries must stay below ~7000 (f16 range of the scaled
 * softmax weights). */
PKV_API pkv_status pkv_paged_decode_fp8(const pkv_pool* pool, float* out, const void* q, const void* k_cache,
                                        const void* v_cache, const float* k_scale, const float* v_scale,
                                        const int32_t* block_tables, const int32_t* context_lens, int32_t n_seqs,
                                        int32_t num_q_heads, float scale, int32_t window, int32_t partition_tokens,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* Sliding-window variant: as pkv_paged_decode, but each query attends only to the last `window`
 * positions of its sequence, t in [max(0, len_b - window), len_b) ("¿Cuánta memoria reservar para la
 * caché KV?", "Adaptar el presupuesto a la estrategia de caché": a sliding-window layer keeps a
 * bounded history). window = 0 means no window (identical to pkv_paged_decode). Blocks entirely
 * before the window are never read, so they may have been released with pkv_release_before (their
 * table entries are then -1). Uses the same workspace size as pkv_paged_decode. */
PKV_API pkv_status pkv_paged_decode_window(const pkv_pool* pool, float* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           const int32_t* context_lens, int32_t n_seqs, int32_t num_q_heads,
                                           float scale, int32_t window, int32_t partition_tokens, void* workspace,
                                           size_t workspace_bytes, void* stream);

/* Causal paged prefill / multi-token append attention. Sequence b has final length len_b =
 * context_lens[b] (its new positions included) and its last q_len_b = cu_q[b+1] - cu_q[b] positions
 * are queries: row cu_q[b] + i of q is position p = len_b - q_len_b + i, and for each query head j
 *     out[row][j][:] = sum_{t in T(p)} softmax_t(scale * q[row][j] . K_b[t]) V_b[t]
 * with T(p) = [0, p], or [max(0, p - window + 1), p] when window > 0 (prefill and generation are
 * separate phases of one request: "¿Cuánta memoria reservar para la caché KV?", "Verificar una carga
 * representativa por etapas"; exact attention: "Servicio de modelos…" §6). The K/V of the new
 * positions must already be in the cache (pkv_reshape_and_cache, same stream). q_len_b = 1 for all b
 * is a decode step. q: [total_q][num_q_heads][D] bf16, out: float32 same shape; cu_q: device int32
 * [n_seqs + 1], cu_q[0] = 0, cu_q[n_seqs] = total_q, q_len_b <= len_b. Needs a bf16 pool (D 64 or 128,
 * block size a multiple of 16, max_blocks_per_seq <= 8192) and num_q_heads / Hkv <= 8. No workspace. */
PKV_API pkv_status pkv_paged_prefill(const pkv_pool* pool, float* out, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                                     const int32_t* cu_q, int32_t n_seqs, int32_t total_q, int32_t num_q_heads,
                                     float scale, int32_t window, void* stream);

/* Shared-prefix (cascade) decode: pkv_paged_decode's result for a batch whose sequences all begin with
 * the same prefix_blocks physical blocks (a forked prompt whose children share its full blocks by
 * reference count until one of them writes: "Paged Attention optimiza el uso de memoria en LLMs",
 * copy-on-write paragraph; "PagedAttention e vLLM", "Implementazione nel mondo reale").
 * The shared blocks are read once for the whole batch instead of once per sequence: every query row
 * of the batch attends to them in one tensor-core pass (the rows of all sequences stacked as the M
 * side of each matrix product, split over the keys to fill the GPU), each sequence's private suffix
 * t in [prefix_blocks * B, len_b) is attended by the decode kernel, and the two parts are combined by
 * their log-sum-exp ("Servicio de modelos de lenguaje con un presupuesto de memoria" §6), so `out`
 * is the exact attention over [0, len_b) to rounding.
 * Arguments as pkv_paged_decode (partition_tokens fixed to 0), plus prefix_blocks: how many leading
 * table entries every sequence shares. Requires block_tables[b][k] == block_tables[0][k] for every
 * b < n_seqs and k < prefix_blocks (a mismatch is recorded as PKV_ERR_DEVICE_BOUNDS, and the rows
 * are then attended over sequence 0's prefix) and context_lens[b] >= prefix_blocks * B (a shorter
 * sequence records PKV_ERR_DEVICE_BOUNDS). prefix_blocks = 0 is pkv_paged_decode.
 * Needs a bf16 pool with D 64 or 128, block size a multiple of 16 and num_q_heads / Hkv <= 8;
 * otherwise PKV_ERR_INVALID. workspace: at least pkv_decode_shared_prefix_workspace_bytes(...)
 * bytes, no initialisation needed; concurrent calls must not share one. Launches three kernels on
 * `stream`. */
PKV_API pkv_status pkv_paged_decode_shared_prefix(const pkv_pool* pool, float* out, const void* q,
                                                  const void* k_cache, const void* v_cache,
                                                  const int32_t* block_tables, const int32_t* context_lens,
                                                  int32_t n_seqs, int32_t num_q_heads, float scale,
                                                  int32_t prefix_blocks, void* workspace, size_t workspace_bytes,
                                                  void* stream);

/* Workspace bytes pkv_paged_decode_shared_prefix needs (prefix_blocks = 0: those of pkv_paged_decode
 * without partitions; 0 for unsupported arguments). */
PKV_API size_t pkv_decode_shared_prefix_workspace_bytes(const pkv_pool* pool, int32_t n_seqs, int32_t num_q_heads,
                                                        int32_t prefix_blocks);

/* Workspace bytes pkv_paged_decode needs for these arguments on the current device. */
PKV_API size_t pkv_decode_workspace_bytes(const pkv_pool* pool, int32_t n_seqs, int32_t num_q_heads,
                                  int32_t partition_tokens);

/* Paged decode for callers that may not allocate device memory at all.
 *
 * No counterpart on the source pages: this is a deployment convenience of this library. Some
 * callers cannot call cudaMalloc or hand out scratch buffers: a plugin inside a host application
 * that owns every device byte through its own fixed arena, a latency-critical serving loop where
 * an allocation (and the device synchronisation it implies) is not acceptable, or a process with a
 * memory budget fixed at start-up. This entry point takes the same arguments as pkv_paged_decode
 * minus the workspace and instead uses a scratch array compiled into the library:
 * PKV_STATIC_SCRATCH_BYTES (16 MiB) of device memory that every GPU which loads the library keeps
 * until the process exits. It calls no allocator (no cudaMalloc, no cudaFree, no library routine
 * that allocates).
 *  - The first call on each device looks up the array's device address (cudaGetSymbolAddress with
 *    that device current) and remembers it with the id of the device's context; make that first
 *    call before any stream capture. A call that finds another context current (the device was
 *    reset, e.g. by cudaDeviceReset, and its context re-created) looks the address up again, since
 *    the array then lives at a new address; that call, too, should come before any capture.
 *  - Every call on a device uses the same array. Its contents need no initialisation (each call
 *    writes every scratch entry it later reads), but calls whose kernels overlap on the GPU (other
 *    streams, other threads) race on it: serialise them, e.g. on one stream.
 *  - A problem whose workspace (pkv_decode_workspace_bytes) exceeds PKV_STATIC_SCRATCH_BYTES is
 *    rejected with PKV_ERR_SCRATCH_TOO_SMALL before anything is enqueued. */
#define PKV_STATIC_SCRATCH_BYTES (16u << 20)
PKV_API pkv_status pkv_paged_decode_static(const pkv_pool* pool, float* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           const int32_t* context_lens, int32_t n_seqs, int32_t num_q_heads,
                                           float scale, int32_t partition_tokens, void* stream);

/* Synchronise the current device, then return and clear the error recorded by kernels
 * (PKV_ERR_DEVICE_BOUNDS / PKV_ERR_DEVICE_TIMEOUT), PKV_ERR_CUDA if the device reports an error,
 * else PKV_OK. Reads the process-wide error word and, when pool is not NULL and has one, the pool's
 * own word (pkv_pool_set_error_word). pool may be NULL. */
PKV_API pkv_status pkv_last_error(const pkv_pool* pool);

/* Per-pool error reporting (no counterpart on the pages: it serves this library's failure
 * detection). By default every kernel records a bad block id or slot (PKV_ERR_DEVICE_BOUNDS) or a
 * bounded wait that gave up (PKV_ERR_DEVICE_TIMEOUT) in one process-wide word, which only
 * pkv_last_error reads, after synchronising the whole device. A caller that serves several streams
 * or pools gives each pool its own word instead: d_word is a device pointer to one uint32_t owned
 * by the caller (4-byte aligned, zeroed by the caller before first use; NULL returns the pool to
 * the process-wide word). From then on the pool's device operations record into d_word with
 * atomicOr. The library allocates nothing. Calls that overlap on the GPU share the word. */
PKV_API pkv_status pkv_pool_set_error_word(pkv_pool* pool, uint32_t* d_word);

/* Reads and clears the pool's error word in stream order on `stream`, then waits for that stream
 * only (no device-wide synchronisation): PKV_ERR_DEVICE_BOUNDS / PKV_ERR_DEVICE_TIMEOUT if a kernel
 * of this pool recorded one before this point of the stream, PKV_ERR_CUDA if a CUDA call failed,
 * PKV_ERR_INVALID if the pool has no error word, else PKV_OK. */
PKV_API pkv_status pkv_stream_error(const pkv_pool* pool, void* stream);

/* ---- diagnostics -------------------------------------------------------------------------- */
/* Self-test of the bounded waits of the pipelined kernels (no counterpart on the pages: it checks
 * this library's failure detection). Enqueues one warp on `stream` that waits, with the same
 * bounded wait the decode and prefill kernels use, on a shared-memory barrier that nothing
 * signals. The wait gives up after its poll limit (about a second), records
 * PKV_ERR_DEVICE_TIMEOUT for pkv_last_error and the kernel returns normally, leaving the CUDA
 * context usable. gave_up: device int32 (may be NULL), set to 1 when the wait gave up.
 * Returns PKV_ERR_CUDA if the launch fails. */
PKV_API pkv_status pkv_selftest_wait_timeout(int32_t* gave_up, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
