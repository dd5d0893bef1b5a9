// Paged decode attention (K3) and the log-sum-exp merge of split sequences (K4), in one kernel.
//
// What is computed ("Servicio de modelos de lenguaje con un presupuesto de memoria" §6): for each
// sequence b and query head j, out = softmax(scale * q K^T) V over the sequence's first len_b
// positions, processed block by block with running max / sum statistics. Keys and values are
// found through the block table ("¿Cómo gestiona Paged Attention la caché KV...?", "PagedAttention
// divide el estado KV en bloques de tamaño fijo"). Query head j reads KV head j / G, G = Hq / Hkv
// ("¿Cuánta memoria reservar para la caché KV?", "Emplear las cabezas KV, en particular con GQA").
//
// Work decomposition (B300 design, not from the pages):
//  * A "unit" is one (sequence, KV head); its positions are cut into 16-token chunks. A chunk of one
//    KV head is one contiguous run of 16*D elements inside a physical block (block_size % 16 == 0).
//  * All units' chunks form one flat list (sequence-major, then head). Each warp of a persistent grid
//    takes an equal contiguous share of that list (balanced mode), or an equal share of whole
//    partitions of `part_chunks` chunks (fixed-partition mode). A warp therefore serves one GQA group
//    per chunk: all G query heads of the KV head use each staged K/V chunk once.
//  * Per warp, a ring of `stages` shared-memory slots is filled by TMA copies that complete on an
//    mbarrier; lane 0 issues them `stages` chunks ahead of the compute. The bf16 path uses 2-D
//    tensor copies with 128-byte swizzle (16 rows x 128 bytes per box) so that ldmatrix reads are
//    free of bank conflicts, and computes S^T = K q^T and O^T = V^T P^T with mma.sync (m16n8k16,
//    fp32 accumulate); the fp32 path uses 1-D bulk copies and CUDA-core dot products.
//  * A segment is the part of a unit one warp processes. A segment that is a whole unit writes the
//    output directly; otherwise it writes (m, l, o/l) to the workspace and arrives on the unit's
//    counter; the warp that arrives last merges the unit's segments: M = max m_k,
//    w_k = l_k 2^(m_k - M), o = sum w_k o_k / sum w_k. m is kept in log2 units (scores
//    pre-multiplied by scale * log2 e), which changes no result. Units whose segments all lie in
//    one CTA count arrivals in shared memory under CTA-scope fences; the others use global
//    counters under GPU-scope fences. Global counters carry a tag unique to the call in their high
//    48 bits, so they never need clearing: a count left by an earlier call (or never written)
//    carries another tag and restarts at 1. The warp that merges a unit (all its parts have
//    arrived, nothing else touches the counter in this launch) also sets the counter back to 0, so
//    a launch replayed with the same tag (a captured CUDA graph) starts from zero too.
//  * The split depends only on the context lengths, never on physical block ids, so results are
//    bitwise invariant under any placement of the blocks.
#pragma once

#include <cmath>

#include "pkv_device.cuh"

namespace pkv_dev {

constexpr int kChunk = 16;  // tokens per staged chunk

// Tensor maps of the K and V caches viewed as 2-D [rows = NB*Hkv*B][D] bf16 arrays.
struct TmaMaps {  // CUtensorMap is itself 64-byte aligned
  CUtensorMap k;
  CUtensorMap v;
};

struct DecodeArgs {
  float* out;                    // [n_seqs][Hq][D]
  const void* q;                 // [n_seqs][Hq][D]
  const void* k_cache;           // [NB][Hkv][B][D]
  const void* v_cache;
  const int32_t* block_tables;   // [n_seqs][MB]
  const int32_t* context_lens;   // [n_seqs]
  float* ws_ml;                  // [n_slots][G][2]  (m in log2 units, l)
  float* ws_o;                   // [n_slots][G][D]  (o already divided by l)
  unsigned long long* ws_count;  // [n_units] arrival counters: (call tag << 16) | segments arrived
  int32_t n_seqs, Hq, Hkv, B, NB, MB;
  int32_t part_chunks;           // 0: balanced split; > 0: chunks per partition
  int32_t max_parts;             // fixed mode: partition slots per unit
  int32_t stages;                // ring depth per warp
  int32_t total_warps;           // warps of the decode grid (balanced-mode slot count / 2)
  int32_t window;                // > 0: attend only to the last `window` positions (sliding window)
  int32_t min_chunks;            // balanced mode: at least this many chunks per warp (fewer, longer ranges)
  float scale_log2;              // scale * log2(e)
  const float* k_scale;          // fp8 pools: [NB][Hkv][B] per-(token, head) scales (else unused)
  const float* v_scale;
  unsigned long long tag;        // 48-bit tag of this call for ws_count
  unsigned int* err;             // error word of the call's pool (null: the process-wide word)
  int32_t start;                 // > 0 (a multiple of 16): attend only to positions >= start
  float* lse_out;                // optional [n_seqs][Hq]: log2 of the softmax denominator of each row, in
                                 // log2 units of the scaled scores (m + log2 l); -inf for an empty row
  int32_t* defer_meta;           // balanced mode, non-null: dynamic tasks and no merging here (no fences, no
                                 // arrivals): each segment of a unit cut by task boundaries leaves its
                                 // partial in its slot, and block 0 writes [T, pref[0..n]] here for the
                                 // later kernel that merges them
  int32_t max_tasks;             // deferred mode: slots for at most this many tasks (2 per task)
  int32_t late_wait;             // non-zero: this kernel reads nothing the previous kernel writes (that one let
                                 // it launch once its own inputs were complete); it waits for the previous
                                 // kernel only before it completes
};


// Arrival of one segment of a split unit. Returns true for the warp that completes the unit.
// Lock-free: the CAS only fails when another segment arrived in between.
__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void fence_acq_rel_cta() { asm volatile("fence.acq_rel.cta;" ::: "memory"); }

__device__ __forceinline__ bool arrive_last(unsigned long long* ctr, unsigned long long tag, int64_t n_parts) {
  unsigned long long old = ld_relaxed_gpu(ctr), assumed, next;
  do {
    assumed = old;
    next = ((assumed >> 16) == tag) ? assumed + 1 : ((tag << 16) | 1ull);
    old = atomicCAS(ctr, assumed, next);
  } while (old != assumed);
  return static_cast<int64_t>(next & 0xffffull) == n_parts;
}

// Take k consecutive dynamic tasks of a deferred-mode decode; returns the first index. The counter
// holds (low 32 bits of the call tag << 32) | count. A value left by an earlier call (another tag, or
// fresh memory) is replaced by this call's tag with count k by whichever taker gets there first,
// which takes index 0. Returns `none` (and records PKV_ERR_DEVICE_TIMEOUT) if the counter could not
// be taken in a bounded number of tries.
__device__ __forceinline__ int64_t grab_tasks(unsigned long long* ctr, unsigned long long tag, unsigned int k,
                                              int64_t none) {
  const unsigned long long tg = tag & 0xffffffffull;   // odd, so never the zero of fresh memory
  unsigned long long cur = ld_relaxed_gpu(ctr);
  for (int it = 0; it < 256; ++it) {
    if ((cur >> 32) == tg) {
      const unsigned long long v = atomicAdd(ctr, static_cast<unsigned long long>(k));
      if ((v >> 32) == tg) return static_cast<int64_t>(v & 0xffffffffull);
      cur = v + k;   // (cannot happen once installed: the tag is only ever replaced by a later call)
    }
    const unsigned long long prev = atomicCAS(ctr, cur, (tg << 32) | k);
    if (prev == cur) return 0;
    cur = prev;
  }
  record_error(ERRBIT_TIMEOUT);
  return none;
}

// Log-sum-exp merge of one unit's n_parts segments by one warp. Segment k's slot is
// 2 * (wf + k) + (k == 0 ? first_kind : 0) in balanced mode (part_chunks == 0), else
// u * max_parts + k. kWide loads all of a segment's values before combining them (more registers,
// one memory latency per segment); the narrow form works through them one float4 at a time.
// Loads of published partials: from L2 when other SMs wrote them (their stores do not update this
// SM's L1), through L1 when this CTA's own warps did (CTA-scope ordering).
template <bool kCta, class T>
__device__ __forceinline__ T ld_part(const T* p) {
  if constexpr (kCta) return *p;
  else return __ldcg(p);
}

template <int D, int G, bool kWide, bool kCta>
__device__ __noinline__ void merge_unit(const DecodeArgs& a, int32_t b, int32_t h, int64_t n_parts, int64_t wf,
                                        int first_kind, int lane) {
  const int64_t u = static_cast<int64_t>(b) * a.Hkv + h;
  auto slot_of = [&](int64_t k) -> int64_t {
    return a.part_chunks != 0 ? u * a.max_parts + k : 2 * (wf + k) + (k == 0 ? first_kind : 0);
  };
  constexpr int V4 = G * D / 4;  // float4 values per unit
  constexpr int R = kWide ? (V4 + 31) / 32 : 1;
  if constexpr (!kWide) {
#pragma unroll 1
    for (int idx = lane; idx < V4; idx += 32) {
      const int j = idx / (D / 4);
      float M = -INFINITY, wsum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
      for (int64_t k = 0; k < n_parts; ++k) {
        const int64_t sl = slot_of(k);
        const float2 ml = ld_part<kCta>(reinterpret_cast<const float2*>(a.ws_ml + (sl * G + j) * 2));
        const float4 o = ld_part<kCta>(reinterpret_cast<const float4*>(a.ws_o + (sl * G + j) * D) + (idx - j * (D / 4)));
        const float Mn = fmaxf(M, ml.x);
        const float c = exp2f(M - Mn);
        const float wk = ml.y * exp2f(ml.x - Mn);
        acc.x = fmaf(wk, o.x, acc.x * c);
        acc.y = fmaf(wk, o.y, acc.y * c);
        acc.z = fmaf(wk, o.z, acc.z * c);
        acc.w = fmaf(wk, o.w, acc.w * c);
        wsum = fmaf(wsum, c, wk);
        M = Mn;
      }
      const float inv = 1.f / wsum;
      reinterpret_cast<float4*>(a.out + (static_cast<int64_t>(b) * a.Hq + h * G + j) * D)[idx - j * (D / 4)] =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      if (a.lse_out != nullptr && idx == j * (D / 4)) a.lse_out[static_cast<int64_t>(b) * a.Hq + h * G + j] = M + log2f(wsum);
    }
  } else {
    float M[R], wsum[R];
    float4 acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      M[r] = -INFINITY;
      wsum[r] = 0.f;
      acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 2
    for (int64_t k = 0; k < n_parts; ++k) {
      const int64_t s = slot_of(k);
      float2 ml[R];
      float4 o[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {  // all of this segment's loads first (L2: written by other warps)
        const int idx = lane + 32 * r;
        if (idx < V4) {
          const int j = idx / (D / 4);
          ml[r] = ld_part<kCta>(reinterpret_cast<const float2*>(a.ws_ml + (s * G + j) * 2));
          o[r] = ld_part<kCta>(reinterpret_cast<const float4*>(a.ws_o + (s * G + j) * D) + (idx - j * (D / 4)));
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (lane + 32 * r < V4) {
          const float Mn = fmaxf(M[r], ml[r].x);
          const float c = exp2f(M[r] - Mn);  // rescales what was accumulated so far (0 at the start)
          const float wk = ml[r].y * exp2f(ml[r].x - Mn);
          acc[r].x = fmaf(wk, o[r].x, acc[r].x * c);
          acc[r].y = fmaf(wk, o[r].y, acc[r].y * c);
          acc[r].z = fmaf(wk, o[r].z, acc[r].z * c);
          acc[r].w = fmaf(wk, o[r].w, acc[r].w * c);
          wsum[r] = fmaf(wsum[r], c, wk);
          M[r] = Mn;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int idx = lane + 32 * r;
      if (idx < V4) {
        const int j = idx / (D / 4);
        const float inv = 1.f / wsum[r];
        reinterpret_cast<float4*>(a.out + (static_cast<int64_t>(b) * a.Hq + h * G + j) * D)[idx - j * (D / 4)] =
            make_float4(acc[r].x * inv, acc[r].y * inv, acc[r].z * inv, acc[r].w * inv);
        if (a.lse_out != nullptr && idx == j * (D / 4))
          a.lse_out[static_cast<int64_t>(b) * a.Hq + h * G + j] = M[r] + log2f(wsum[r]);
      }
    }
  }
}

__device__ __forceinline__ int32_t clamped_len(const DecodeArgs& a, int32_t b) {
  int32_t len = __ldg(a.context_lens + b);
  const int32_t cap = a.MB * a.B;
  if (len < 0 || len > cap) {
    record_error(ERRBIT_BOUNDS);
    len = len < 0 ? 0 : cap;
  }
  return len;
}

// Position of one warp in the flat chunk list.
struct Cursor {
  int32_t b, h, c, nch;  // chunk c of unit (b, h); nch = chunks of sequence b
};

// Largest b in [0, n) with Hkv * pref[b] <= x (sequences with no chunks are skipped naturally).
__device__ __forceinline__ int32_t find_seq(const int32_t* pref, int32_t n, int32_t Hkv, int64_t x) {
  int32_t lo = 0, hi = n - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(pref[mid]) * Hkv <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Cursor locate(const int32_t* pref, int32_t n, int32_t Hkv, int64_t x) {
  Cursor cu;
  cu.b = find_seq(pref, n, Hkv, x);
  cu.nch = pref[cu.b + 1] - pref[cu.b];
  const int64_t r = x - static_cast<int64_t>(pref[cu.b]) * Hkv;
  cu.h = static_cast<int32_t>(r / cu.nch);
  cu.c = static_cast<int32_t>(r - static_cast<int64_t>(cu.h) * cu.nch);
  return cu;
}

__device__ __forceinline__ void advance(Cursor& cu, const int32_t* pref, int32_t n, int32_t Hkv) {
  if (++cu.c < cu.nch) return;
  cu.c = 0;
  if (++cu.h < Hkv) return;
  cu.h = 0;
  do {
    ++cu.b;
    cu.nch = cu.b < n ? pref[cu.b + 1] - pref[cu.b] : 1;
  } while (cu.nch == 0);
}

// Chunk index where item i (fixed-partition mode) starts; items are (unit, partition) pairs.
__device__ __forceinline__ int64_t item_start(const int32_t* pref, const int32_t* ipref, int32_t n, int32_t Hkv,
                                              int32_t PC, int64_t i) {
  if (i >= static_cast<int64_t>(ipref[n]) * Hkv) return static_cast<int64_t>(pref[n]) * Hkv;
  const int32_t b = find_seq(ipref, n, Hkv, i);
  const int32_t np = ipref[b + 1] - ipref[b];
  const int64_t r = i - static_cast<int64_t>(ipref[b]) * Hkv;
  const int32_t h = static_cast<int32_t>(r / np);
  const int32_t p = static_cast<int32_t>(r - static_cast<int64_t>(h) * np);
  const int32_t nch = pref[b + 1] - pref[b];
  return static_cast<int64_t>(pref[b]) * Hkv + static_cast<int64_t>(h) * nch + static_cast<int64_t>(p) * PC;
}

// Shared-memory carve-up of the decode kernel: [1 KB alignment slack][ring: per warp `stages` stages]
// [mbarriers][64-int scan scratch][pref][ipref (fixed partitions only)][cfirst (window only)].
// Stages start on 1024-byte boundaries (128-byte swizzle atoms).
__host__ __device__ inline size_t decode_ring_bytes(int nw, int stages, int stage_bytes) {
  return static_cast<size_t>(nw) * stages * stage_bytes;
}
__host__ __device__ inline size_t decode_smem_bytes(int nw, int stages, int stage_bytes, int n_seqs, bool parts,
                                                    bool window) {
  return 1024 + decode_ring_bytes(nw, stages, stage_bytes) + static_cast<size_t>(nw) * stages * 8 + 256 +
         (1 + (parts ? 1 : 0) + (window ? 1 : 0)) * static_cast<size_t>(n_seqs + 1) * 4;
}

// Block-wide exclusive prefix sums over sequences of chunk counts (pref) and partition counts
// (ipref, fixed-partition mode only, else null); pref[n] / ipref[n] hold the totals; cfirst[b]
// (window only, else null) is the first chunk of sequence b that the attention reads (0, or the
// chunk holding position len - window). Every thread of the CTA
// takes part. Lengths are loaded kPrefixBatch tiles at a time so that their latencies overlap.
// wsum: 64 ints of smem.
constexpr int kPrefixBatch = 8;

__device__ __forceinline__ void build_prefix(const DecodeArgs& a, int32_t* pref, int32_t* ipref, int32_t* cfirst,
                                             int32_t* wsum) {
  const int32_t n = a.n_seqs;
  const int32_t PC = a.part_chunks > 0 ? a.part_chunks : 1;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int32_t cap = a.MB * a.B;
  int32_t carry_c = 0, carry_i = 0;  // running totals, identical in every thread
  for (int32_t base = 0; base < n; base += nt * kPrefixBatch) {
    int32_t raw[kPrefixBatch];
#pragma unroll
    for (int k = 0; k < kPrefixBatch; ++k) {
      const int32_t b = base + k * nt + tid;
      raw[k] = b < n ? __ldg(a.context_lens + b) : 0;
    }
#pragma unroll
    for (int k = 0; k < kPrefixBatch; ++k) {
      if (base + k * nt >= n) break;  // uniform across the CTA
      const int32_t b = base + k * nt + tid;
      int32_t len = raw[k];
      if (len < 0 || len > cap) {
        record_error(ERRBIT_BOUNDS);
        len = len < 0 ? 0 : cap;
      }
      int32_t c0 = (a.window > 0 && len > a.window) ? (len - a.window) / kChunk : 0;
      if (a.start > 0) {   // positions before `start` belong to another call (a shared prefix)
        if (len < a.start) {   // (threads past the last sequence hold 0: no chunks, no error)
          if (b < n) record_error(ERRBIT_BOUNDS);
          len = a.start;
        }
        c0 = max(c0, a.start / kChunk);
      }
      const int32_t c = (len + kChunk - 1) / kChunk - c0;
      const int32_t ci = (c + PC - 1) / PC;
      int32_t ic = c, ii = ci;  // inclusive warp scan
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t tc = __shfl_up_sync(0xffffffffu, ic, off);
        const int32_t ti = __shfl_up_sync(0xffffffffu, ii, off);
        if (lane >= off) {
          ic += tc;
          ii += ti;
        }
      }
      if (lane == 31) {
        wsum[warp] = ic;
        wsum[32 + warp] = ii;
      }
      __syncthreads();
      int32_t pc = 0, pi = 0, tc = 0, ti = 0;
      for (int w2 = 0; w2 < nw; ++w2) {
        const int32_t sc = wsum[w2], si = wsum[32 + w2];
        if (w2 < warp) {
          pc += sc;
          pi += si;
        }
        tc += sc;
        ti += si;
      }
      if (b < n) {
        pref[b] = carry_c + pc + ic - c;
        if (ipref) ipref[b] = carry_i + pi + ii - ci;
        if (cfirst) cfirst[b] = c0;
      }
      carry_c += tc;
      carry_i += ti;
      __syncthreads();  // wsum is reused by the next tile
    }
  }
  if (tid == 0) {
    pref[n] = carry_c;
    if (ipref) ipref[n] = carry_i;
  }
}

// ------------------------------------------------------------------------------------------------
// SIMT math: CUDA-core dot products with warp shuffles (fp32 caches, and bf16 when G > 8).
// Lane layout: LPT lanes per token, each holding EPL elements of the head dimension (PIECES
// 16-byte pieces spaced LPT pieces apart, so a quarter-warp reads 128 contiguous bytes);
// TPP tokens per pass. Scores are pre-scaled into log2 units through q.
// ------------------------------------------------------------------------------------------------
template <typename T, int D, int G>
struct SimtMath {
  static constexpr int es = sizeof(T);
  static constexpr int PER16 = Widen<T>::kPer16;
  static constexpr int EPL = (G <= 5) ? 16 : 8;
  static constexpr int LPT = D / EPL;
  static constexpr int TPP = 32 / LPT;
  static constexpr int PASSES = kChunk / TPP;
  static constexpr int PIECES = EPL / PER16;
  static constexpr int CB = kChunk * D * es;  // bytes of one K (or V) chunk
  static constexpr int kStageBytes = 2 * CB;
  static constexpr int kMinCtasPerSm = 1;     // register-heavy: let the compiler use up to 255
  static constexpr int kQElem = es;
  static constexpr bool kMaskVariants = false;  // one chunk routine checks the token range itself
  static_assert(LPT * EPL == D && TPP * LPT == 32 && PASSES * TPP == kChunk, "lane layout");
  static_assert(PIECES * PER16 == EPL, "pieces");

  struct Regs {
    float q[G][EPL];
    float o[G][EPL];
    float m[G], l[G];
  };

  // lane 0: stage the chunk starting at cache row `row0` (= (blk*Hkv + h)*B + offset)
  __device__ static void issue(const DecodeArgs& a, const TmaMaps&, uint32_t dst, uint32_t bar, int64_t row0,
                               uint64_t policy) {
    mbar_arrive_expect_tx(bar, 2 * CB);
    const int64_t byte0 = row0 * D * es;
    bulk_g2s_hint(dst, static_cast<const unsigned char*>(a.k_cache) + byte0, CB, bar, policy);
    bulk_g2s_hint(dst + CB, static_cast<const unsigned char*>(a.v_cache) + byte0, CB, bar, policy);
  }

  __device__ static void load_q(Regs& r, const DecodeArgs& a, int32_t b, int32_t h, int lane) {
    const int cl = lane % LPT;
    const T* qbase = static_cast<const T*>(a.q) + (static_cast<int64_t>(b) * a.Hq + h * G) * D;
#pragma unroll
    for (int j = 0; j < G; ++j) {
#pragma unroll
      for (int i = 0; i < PIECES; ++i) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qbase + j * D + (cl + i * LPT) * PER16));
        Widen<T>::load(reinterpret_cast<const unsigned char*>(&raw), &r.q[j][i * PER16]);
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) r.q[j][e] *= a.scale_log2;
    }
  }

  __device__ static void reset(Regs& r) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      r.m[j] = -INFINITY;
      r.l[j] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) r.o[j][e] = 0.f;
    }
  }

  // Tokens vlo <= tok < vhi of the chunk are inside the attention range; the rest are masked.
  template <bool kMask>
  __device__ static void chunk(Regs& r, const unsigned char* kb, int vlo, int vhi, float, int lane) {
    const unsigned char* vb = kb + CB;
    const int tg = lane / LPT;
    const int cl = lane % LPT;
    float sc[PASSES][G];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int tok = p * TPP + tg;
      float kf[EPL];
#pragma unroll
      for (int pc = 0; pc < PIECES; ++pc)
        Widen<T>::load(kb + (tok * D + (cl + pc * LPT) * PER16) * es, kf + pc * PER16);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) s = fmaf(r.q[j][e], kf[e], s);
#pragma unroll
        for (int off = LPT / 2; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        sc[p][j] = (tok >= vlo && tok < vhi) ? s : -INFINITY;
      }
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
      float mx = sc[0][j];
#pragma unroll
      for (int p = 1; p < PASSES; ++p) mx = fmaxf(mx, sc[p][j]);
#pragma unroll
      for (int off = LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mnew = fmaxf(r.m[j], mx);
      const float alpha = exp2f(r.m[j] - mnew);
      r.m[j] = mnew;
      if (alpha != 1.f) {
        r.l[j] *= alpha;
#pragma unroll
        for (int e = 0; e < EPL; ++e) r.o[j][e] *= alpha;
      }
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        sc[p][j] = exp2f(sc[p][j] - mnew);
        r.l[j] += sc[p][j];
      }
    }
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int tok = p * TPP + tg;
      if (tok >= vlo && tok < vhi) {   // values outside the range may be garbage (even NaN)
        float vf[EPL];
#pragma unroll
        for (int pc = 0; pc < PIECES; ++pc)
          Widen<T>::load(vb + (tok * D + (cl + pc * LPT) * PER16) * es, vf + pc * PER16);
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
          for (int e = 0; e < EPL; ++e) r.o[j][e] = fmaf(sc[p][j], vf[e], r.o[j][e]);
      }
    }
  }

  // Writes o / l for the G heads to dst[G][D]; if ml != nullptr also (m, l) to ml[G][2].
  __device__ static void finish(Regs& r, float* dst, float* ml, float* lse, int lane) {
    const int tg = lane / LPT;
    const int cl = lane % LPT;
#pragma unroll
    for (int j = 0; j < G; ++j) {
      float lt = r.l[j];
#pragma unroll
      for (int off = LPT; off < 32; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        float t = r.o[j][e];
#pragma unroll
        for (int off = LPT; off < 32; off <<= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        r.o[j][e] = t;
      }
      if (j % TPP != tg) continue;
      const float inv = 1.f / lt;
#pragma unroll
      for (int pc = 0; pc < PIECES; ++pc) {
        float4* d4 = reinterpret_cast<float4*>(dst + j * D + (cl + pc * LPT) * PER16);
#pragma unroll
        for (int k4 = 0; k4 < PER16 / 4; ++k4) {
          const float* src = &r.o[j][pc * PER16 + 4 * k4];
          d4[k4] = make_float4(src[0] * inv, src[1] * inv, src[2] * inv, src[3] * inv);
        }
      }
      if (ml != nullptr && cl == 0) {
        ml[2 * j] = r.m[j];
        ml[2 * j + 1] = lt;
      }
      if (lse != nullptr && cl == 0) lse[j] = r.m[j] + log2f(lt);
    }
  }
};

// ------------------------------------------------------------------------------------------------
// Tensor-core math for bf16 caches, G <= 8 query heads per KV head, in transposed form: the 16-row
// side of m16n8k16 is filled by 16 tokens (scores) or 16 dims (output) and the heads sit on the
// 8-wide side, so no mma row is padding.
//
// S^T = K q^T per 16-token chunk: A = the K chunk (rows = tokens) read with ldmatrix from the
// swizzled boxes, B = q^T (column n = a head), fp32 accumulate: D/16 mma. O^T += V^T P^T: A = V^T
// read with ldmatrix.trans (16 dims per m-tile), B = P^T, which movmatrix.trans makes from the
// score fragment: D/16 m-tiles. P is carried as bf16 hi + lo (lo = bf16(P - hi)), ~2^-17 relative.
// With G <= 4 the 8 columns hold every head twice: the lanes of columns 0..3 pass hi, those of
// columns 4..7 (same scores, same maxima) pass lo, so one mma per m-tile accumulates both and the
// halves are added at the end; with G > 4 each m-tile takes a second mma for lo.
// Lane (g = lane/4, t = lane%4) owns columns {2t, 2t+1}: the scores of tokens {g, g+8} and the
// output dims {16i + g, 16i + g + 8}; its running max and sum belong to those two columns.
// The running max is raised only when a chunk's max exceeds it by more than kRescaleLog2 (the
// exponentials then stay below 2^kRescaleLog2), which skips most rescales of O without changing
// the result: numerator and denominator always use the same max.
// ------------------------------------------------------------------------------------------------
template <int D, int G>
struct MmaMath {
  static_assert(G >= 1 && G <= 8, "G <= 8");
  static_assert(D == 64 || D == 128, "D");
  static constexpr int KB = D / 64;          // 128-byte boxes per row
  static constexpr int BOX = kChunk * 128;   // one box: 16 rows x 128 bytes
  static constexpr int CB = KB * BOX;        // K (or V) chunk bytes
  static constexpr int kStageBytes = 2 * CB;
  static constexpr int kMinCtasPerSm = 3;    // 12 warps per SM: the register budget is 168 per thread
  static constexpr int KS = D / 16;          // k-steps of q.K and m-tiles of p.V
  static constexpr bool kPaired = G <= 4;    // columns 4..7 repeat heads 0..3 and carry lo
  static constexpr float kRescaleLog2 = 8.f;
  static constexpr int kQElem = 2;
  static constexpr bool kMaskVariants = true;   // full chunks skip the masking work

  struct Regs {
    uint32_t qb[KS][2];  // B fragment of q^T: head of column g, dims 16ks + {2t, 2t+1} and {+8, +9}
    float o[KS][4];      // O^T: dims 16i + g ([0], [1]) and 16i + g + 8 ([2], [3]); columns 2t, 2t+1
    float m[2], l[2];    // running max (log2 units) and this lane's share of the sum, per column
  };

  // Head carried by column n, or -1 for a padding column.
  __device__ static __forceinline__ int head_of(int n) {
    const int hd = kPaired ? (n & 3) : n;
    return hd < G ? hd : -1;
  }

  __device__ static void issue(const DecodeArgs&, const TmaMaps& maps, uint32_t dst, uint32_t bar, int64_t row0,
                               uint64_t policy) {
    mbar_arrive_expect_tx(bar, 2 * CB);
    const int32_t y = static_cast<int32_t>(row0);
    if constexpr (KB == 2) {
      // 3-D maps (64 dims, rows, the row's two halves): one copy per operand lands as the two
      // 16-row x 128-byte boxes, half after half, with the same swizzle
      tma_load_3d_hint(dst, &maps.k, 0, y, 0, bar, policy);
      tma_load_3d_hint(dst + CB, &maps.v, 0, y, 0, bar, policy);
    } else {
#pragma unroll
      for (int kb = 0; kb < KB; ++kb) {
        tma_load_2d(dst + kb * BOX, &maps.k, 64 * kb, y, bar, policy);
        tma_load_2d(dst + CB + kb * BOX, &maps.v, 64 * kb, y, bar, policy);
      }
    }
  }

  __device__ static void load_q(Regs& r, const DecodeArgs& a, int32_t b, int32_t h, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int hd = head_of(g);
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                             (static_cast<int64_t>(b) * a.Hq + h * G + max(hd, 0)) * D);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      r.qb[ks][0] = hd >= 0 ? __ldg(qrow + 8 * ks + t) : 0u;
      r.qb[ks][1] = hd >= 0 ? __ldg(qrow + 8 * ks + 4 + t) : 0u;
    }
  }

  __device__ static void reset(Regs& r) {
    r.m[0] = r.m[1] = -INFINITY;
    r.l[0] = r.l[1] = 0.f;
#pragma unroll
    for (int i = 0; i < KS; ++i) r.o[i][0] = r.o[i][1] = r.o[i][2] = r.o[i][3] = 0.f;
  }

  // Byte offset of 16-byte block `cb` (0..7) of row `row` inside a 128B-swizzled box.
  __device__ static __forceinline__ uint32_t swz(int row, int cb) {
    return static_cast<uint32_t>(row * 128 + ((cb ^ (row & 7)) << 4));
  }

  // Tokens vlo <= tok < vhi of the chunk are inside the attention range; the rest are masked.
  template <bool kMask>  // kMask: some tokens of the chunk lie outside [vlo, vhi)
  __device__ static void chunk(Regs& r, const unsigned char* kbase, int vlo, int vhi, float scale_log2, int lane) {
    const uint32_t kb = smem_addr(kbase);
    const uint32_t vb = kb + CB;
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: matrix index and row of this lane's address
    // ---- S^T = K q^T (two accumulators: half-length dependency chains)
    float se[4] = {0.f, 0.f, 0.f, 0.f}, so[4] = {0.f, 0.f, 0.f, 0.f};
    const int ktok = mr + 8 * (mi & 1);       // matrices 0, 2: tokens 0..7; 1, 3: tokens 8..15
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int db = 2 * ks + (mi >> 1);      // matrices 0, 1: dims 16ks..+7; 2, 3: dims 16ks+8..+15
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kb + (db >> 3) * BOX + swz(ktok, db & 7), a0, a1, a2, a3);
      if (ks & 1)
        mma_bf16_16816(so, a0, a1, a2, a3, r.qb[ks][0], r.qb[ks][1]);
      else
        mma_bf16_16816(se, a0, a1, a2, a3, r.qb[ks][0], r.qb[ks][1]);
    }
    // ---- online softmax per column over tokens {g, g+8} of every lane
    const bool okg = !kMask || (g >= vlo && g < vhi), okg8 = !kMask || (g + 8 >= vlo && g + 8 < vhi);
    float x[4];
    x[0] = okg ? (se[0] + so[0]) * scale_log2 : -INFINITY;
    x[1] = okg ? (se[1] + so[1]) * scale_log2 : -INFINITY;
    x[2] = okg8 ? (se[2] + so[2]) * scale_log2 : -INFINITY;
    x[3] = okg8 ? (se[3] + so[3]) * scale_log2 : -INFINITY;
    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const bool raise0 = mx0 > r.m[0] + kRescaleLog2, raise1 = mx1 > r.m[1] + kRescaleLog2;
    if (__any_sync(0xffffffffu, raise0 || raise1)) {
      const float m0 = raise0 ? mx0 : r.m[0], m1 = raise1 ? mx1 : r.m[1];
      const float al0 = exp2f(r.m[0] - m0), al1 = exp2f(r.m[1] - m1);  // 0 on the first chunk, 1 if unchanged
      r.m[0] = m0;
      r.m[1] = m1;
      r.l[0] *= al0;
      r.l[1] *= al1;
#pragma unroll
      for (int i = 0; i < KS; ++i) {
        r.o[i][0] *= al0;
        r.o[i][2] *= al0;
        r.o[i][1] *= al1;
        r.o[i][3] *= al1;
      }
    }
    float pr[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pr[e] = exp2f(x[e] - r.m[e & 1]);
    r.l[0] += pr[0] + pr[2];
    r.l[1] += pr[1] + pr[3];
    // ---- P^T fragments: pack [token][column] as bf16 pairs, transpose with movmatrix
    const uint32_t h0 = pack_bf16x2(pr[0], pr[1]);  // token g
    const uint32_t h1 = pack_bf16x2(pr[2], pr[3]);  // token g + 8
    const uint32_t l0 = pack_bf16x2(pr[0] - bf16_lo(h0), pr[1] - bf16_hi(h0));
    const uint32_t l1 = pack_bf16x2(pr[2] - bf16_lo(h1), pr[3] - bf16_hi(h1));
    uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
    if constexpr (kPaired) {
      const bool lo_lane = t >= 2;             // columns 4..7
      bh0 = movmatrix_t(lo_lane ? l0 : h0);
      bh1 = movmatrix_t(lo_lane ? l1 : h1);
    } else {
      bh0 = movmatrix_t(h0);
      bh1 = movmatrix_t(h1);
      bl0 = movmatrix_t(l0);
      bl1 = movmatrix_t(l1);
    }
    // ---- O^T += V^T P^T; V entries of masked tokens are zeroed (they may hold NaN)
    uint32_t mk01 = 0xffffffffu, mk23 = 0xffffffffu;  // A registers 0/1: tokens 2t, 2t+1; 2/3: 2t+8, 2t+9
    if constexpr (kMask) {
      const int k0 = 2 * t;
      mk01 = (k0 >= vlo && k0 < vhi ? 0x0000ffffu : 0u) | (k0 + 1 >= vlo && k0 + 1 < vhi ? 0xffff0000u : 0u);
      mk23 = (k0 + 8 >= vlo && k0 + 8 < vhi ? 0x0000ffffu : 0u) | (k0 + 9 >= vlo && k0 + 9 < vhi ? 0xffff0000u : 0u);
    }
    const int vtok = mr + 8 * (mi >> 1);       // matrices 0, 1: tokens 0..7; 2, 3: tokens 8..15
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      const int db = 2 * i + (mi & 1);         // matrices 0, 2: dims 16i..+7; 1, 3: dims 16i+8..+15
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vb + (db >> 3) * BOX + swz(vtok, db & 7), a0, a1, a2, a3);
      if constexpr (kMask) {
        a0 &= mk01;
        a1 &= mk01;
        a2 &= mk23;
        a3 &= mk23;
      }
      mma_bf16_16816(r.o[i], a0, a1, a2, a3, bh0, bh1);
      if constexpr (!kPaired) mma_bf16_16816(r.o[i], a0, a1, a2, a3, bl0, bl1);
    }
  }

  __device__ static void finish(Regs& r, float* dst, float* ml, float* lse, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float lt0 = r.l[0], lt1 = r.l[1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
    }
    if constexpr (kPaired) {  // lane t < 2 holds hi of heads 2t, 2t+1, lane t + 2 their lo
#pragma unroll
      for (int i = 0; i < KS; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) r.o[i][e] += __shfl_xor_sync(0xffffffffu, r.o[i][e], 2);
    }
    const int hd0 = 2 * t, hd1 = 2 * t + 1;
    const bool w0 = (!kPaired || t < 2) && hd0 < G;
    const bool w1 = (!kPaired || t < 2) && hd1 < G;
    const float inv0 = 1.f / lt0, inv1 = 1.f / lt1;
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      const int d0 = 16 * i + g;
      if (w0) {
        dst[hd0 * D + d0] = r.o[i][0] * inv0;
        dst[hd0 * D + d0 + 8] = r.o[i][2] * inv0;
      }
      if (w1) {
        dst[hd1 * D + d0] = r.o[i][1] * inv1;
        dst[hd1 * D + d0 + 8] = r.o[i][3] * inv1;
      }
    }
    if (ml != nullptr && g == 0) {
      if (w0) {
        ml[2 * hd0] = r.m[0];
        ml[2 * hd0 + 1] = lt0;
      }
      if (w1) {
        ml[2 * hd1] = r.m[1];
        ml[2 * hd1 + 1] = lt1;
      }
    }
    if (lse != nullptr && g == 0) {
      if (w0) lse[hd0] = r.m[0] + log2f(lt0);
      if (w1) lse[hd1] = r.m[1] + log2f(lt1);
    }
  }
};

// ------------------------------------------------------------------------------------------------
// FP8 E4M3 caches (D = 128), G <= 8: f16 tensor-core math on exactly converted codes, in the same
// transposed form as the bf16 path (tokens or dims on the 16-row side, heads on the 8-wide side).
//
// Stage: [K box: 16 rows x 128 B, 128-byte swizzle][V box: 128 dims x 16 tokens (V is stored
// dim-major in fp8 pools)][16 K scales][16 V scales], padded to 5120 bytes.
// S^T = K q^T: the contraction over d is order-free, so within each 16-dim k-step the fragment's
// k indices {2t, 2t+1} and {2t+8, 2t+9} stand for dims {4t, 4t+1} and {4t+2, 4t+3}: ldmatrix on the
// fp8 rows hands lane t the 4 consecutive codes 4t..4t+3, which cvt turns into its two f16 A pairs;
// q^T is loaded in the same dim order. O^T += V^T P^T: ldmatrix on the dim-major V rows hands lane t
// stored bytes 4t..4t+3, and the fp8 V page stores each 16-token group in the order
// (0,1,8,9, 2,3,10,11, 4,5,12,13, 6,7,14,15), so those bytes are tokens {2t, 2t+1} and {2t+8, 2t+9}:
// exactly the k indices of the A fragment. Per-token scales: S *= k_scale; P' = p * v_scale * 1024
// is carried as f16 hi + lo (paired columns as in the bf16 path); the running max is raised when a
// chunk exceeds it by 2^2, so p <= 4 and P' stays inside the f16 normal range for |V| < ~7000.
// ------------------------------------------------------------------------------------------------
template <int G, int kCtas = 3>
struct Fp8Math {
  static_assert(G >= 1 && G <= 8, "G <= 8");
  static constexpr int D = 128;
  static constexpr int KBOX = kChunk * 128;
  static constexpr int VBOX = D * kChunk;
  static constexpr int kScaleOff = KBOX + VBOX;
  static constexpr int kTxBytes = KBOX + VBOX + 2 * kChunk * 4;
  static constexpr int kStageBytes = 5120;
  static constexpr int kMinCtasPerSm = kCtas;   // resident CTAs per SM the register budget is cut for
  static constexpr int KS = D / 16;          // k-steps of q.K and m-tiles of p.V
  static constexpr bool kPaired = G <= 4;
  static constexpr float kRescaleLog2 = 2.f;
  static constexpr int kQElem = 2;
  static constexpr bool kMaskVariants = true;
  static constexpr float kPScale = 1024.f;

  struct Regs {
    uint32_t qb[KS][2];  // B fragment of q^T (f16): dims 16ks + {4t, 4t+1} and {4t+2, 4t+3}
    float o[KS][4];      // O^T: dims 16i + g ([0], [1]) and 16i + g + 8 ([2], [3]); columns 2t, 2t+1
    float m[2], l[2];
  };

  __device__ static __forceinline__ int head_of(int n) {
    const int hd = kPaired ? (n & 3) : n;
    return hd < G ? hd : -1;
  }

  __device__ static void issue(const DecodeArgs& a, const TmaMaps& maps, uint32_t dst, uint32_t bar, int64_t row0,
                               uint64_t policy) {
    const int64_t page = row0 / a.B;
    const int32_t off = static_cast<int32_t>(row0 - page * a.B);
    mbar_arrive_expect_tx(bar, kTxBytes);
    tma_load_2d(dst, &maps.k, 0, static_cast<int32_t>(row0), bar, policy);
    if (a.B == kChunk)   // the chunk is the whole V page of this (block, head): one contiguous 2 KB run
      bulk_g2s_hint(dst + KBOX, static_cast<const unsigned char*>(a.v_cache) + page * VBOX, VBOX, bar, policy);
    else                 // a 16-token column slice of a wider page: 2-D box
      tma_load_2d(dst + KBOX, &maps.v, off, static_cast<int32_t>(page * D), bar, policy);
    bulk_g2s_hint(dst + kScaleOff, a.k_scale + row0, kChunk * 4, bar, policy);
    bulk_g2s_hint(dst + kScaleOff + kChunk * 4, a.v_scale + row0, kChunk * 4, bar, policy);
  }

  __device__ static void load_q(Regs& r, const DecodeArgs& a, int32_t b, int32_t h, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int hd = head_of(g);
    const uint2* qrow = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                       (static_cast<int64_t>(b) * a.Hq + h * G + max(hd, 0)) * D);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (hd >= 0) {
        const uint2 w = __ldg(qrow + 4 * ks + t);   // dims 16ks + 4t .. +3
        r.qb[ks][0] = pack_f16x2(bf16_lo(w.x), bf16_hi(w.x));
        r.qb[ks][1] = pack_f16x2(bf16_lo(w.y), bf16_hi(w.y));
      } else {
        r.qb[ks][0] = r.qb[ks][1] = 0u;
      }
    }
  }

  __device__ static void reset(Regs& r) {
    r.m[0] = r.m[1] = -INFINITY;
    r.l[0] = r.l[1] = 0.f;
#pragma unroll
    for (int i = 0; i < KS; ++i) r.o[i][0] = r.o[i][1] = r.o[i][2] = r.o[i][3] = 0.f;
  }

  template <bool kMask>  // kMask: some tokens of the chunk lie outside [vlo, vhi)
  __device__ static void chunk(Regs& r, const unsigned char* stage, int vlo, int vhi, float scale_log2, int lane) {
    const uint32_t kb = smem_addr(stage);
    const uint32_t vb = kb + KBOX;
    const float* scl = reinterpret_cast<const float*>(stage + kScaleOff);
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, mr = lane & 7;
    // ---- S^T = K q^T
    float se[4] = {0.f, 0.f, 0.f, 0.f}, so[4] = {0.f, 0.f, 0.f, 0.f};
    const int ktok = mr + 8 * (mi & 1);       // matrices 0, 2: tokens 0..7; 1, 3: tokens 8..15
#pragma unroll
    for (int p = 0; p < KS / 2; ++p) {
      const int db = 2 * p + (mi >> 1);       // matrices 0, 1: k-step 2p; 2, 3: k-step 2p + 1
      uint32_t w0, w1, w2, w3;
      ldsm_x4(kb + ktok * 128 + ((db ^ (ktok & 7)) << 4), w0, w1, w2, w3);
      uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
      e4m3x4_to_f16x2x2(w0, a0, a2);
      e4m3x4_to_f16x2x2(w1, a1, a3);
      e4m3x4_to_f16x2x2(w2, c0, c2);
      e4m3x4_to_f16x2x2(w3, c1, c3);
      mma_f16_16816(se, a0, a1, a2, a3, r.qb[2 * p][0], r.qb[2 * p][1]);
      mma_f16_16816(so, c0, c1, c2, c3, r.qb[2 * p + 1][0], r.qb[2 * p + 1][1]);
    }
    // ---- online softmax per column over tokens {g, g+8}
    const bool okg = !kMask || (g >= vlo && g < vhi), okg8 = !kMask || (g + 8 >= vlo && g + 8 < vhi);
    const float ks0 = scl[g] * scale_log2, ks8 = scl[g + 8] * scale_log2;
    float x[4];
    x[0] = okg ? (se[0] + so[0]) * ks0 : -INFINITY;
    x[1] = okg ? (se[1] + so[1]) * ks0 : -INFINITY;
    x[2] = okg8 ? (se[2] + so[2]) * ks8 : -INFINITY;
    x[3] = okg8 ? (se[3] + so[3]) * ks8 : -INFINITY;
    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const bool raise0 = mx0 > r.m[0] + kRescaleLog2, raise1 = mx1 > r.m[1] + kRescaleLog2;
    if (__any_sync(0xffffffffu, raise0 || raise1)) {
      const float m0 = raise0 ? mx0 : r.m[0], m1 = raise1 ? mx1 : r.m[1];
      const float al0 = exp2f(r.m[0] - m0), al1 = exp2f(r.m[1] - m1);
      r.m[0] = m0;
      r.m[1] = m1;
      r.l[0] *= al0;
      r.l[1] *= al1;
#pragma unroll
      for (int i = 0; i < KS; ++i) {
        r.o[i][0] *= al0;
        r.o[i][2] *= al0;
        r.o[i][1] *= al1;
        r.o[i][3] *= al1;
      }
    }
    float pr[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pr[e] = exp2f(x[e] - r.m[e & 1]);
    r.l[0] += pr[0] + pr[2];
    r.l[1] += pr[1] + pr[3];
    // a masked token's scale may be garbage (even NaN): select 0 rather than multiply
    const float vs0 = scl[kChunk + g] * kPScale, vs8 = scl[kChunk + g + 8] * kPScale;
    const float p0 = okg ? pr[0] * vs0 : 0.f, p1 = okg ? pr[1] * vs0 : 0.f;
    const float p2 = okg8 ? pr[2] * vs8 : 0.f, p3 = okg8 ? pr[3] * vs8 : 0.f;
    const uint32_t h0 = pack_f16x2(p0, p1), h1 = pack_f16x2(p2, p3);
    const uint32_t l0 = pack_f16x2(p0 - f16_lo(h0), p1 - f16_hi(h0));
    const uint32_t l1 = pack_f16x2(p2 - f16_lo(h1), p3 - f16_hi(h1));
    uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
    if constexpr (kPaired) {
      const bool lo_lane = t >= 2;
      bh0 = movmatrix_t(lo_lane ? l0 : h0);
      bh1 = movmatrix_t(lo_lane ? l1 : h1);
    } else {
      bh0 = movmatrix_t(h0);
      bh1 = movmatrix_t(h1);
      bl0 = movmatrix_t(l0);
      bl1 = movmatrix_t(l1);
    }
    // ---- O^T += V^T P^T; V entries of masked tokens are zeroed (they may hold NaN)
    uint32_t mk01 = 0xffffffffu, mk23 = 0xffffffffu;  // A registers 0/1: tokens 2t, 2t+1; 2/3: 2t+8, 2t+9
    if constexpr (kMask) {
      const int k0 = 2 * t;
      mk01 = (k0 >= vlo && k0 < vhi ? 0x0000ffffu : 0u) | (k0 + 1 >= vlo && k0 + 1 < vhi ? 0xffff0000u : 0u);
      mk23 = (k0 + 8 >= vlo && k0 + 8 < vhi ? 0x0000ffffu : 0u) | (k0 + 9 >= vlo && k0 + 9 < vhi ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int q = 0; q < KS / 2; ++q) {             // 32 dims: m-tiles 2q and 2q + 1
      uint32_t v0, v1, v2, v3;
      ldsm_x4(vb + (32 * q + 8 * mi + mr) * kChunk, v0, v1, v2, v3);
      uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
      e4m3x4_to_f16x2x2(v0, a0, a2);
      e4m3x4_to_f16x2x2(v1, a1, a3);
      e4m3x4_to_f16x2x2(v2, c0, c2);
      e4m3x4_to_f16x2x2(v3, c1, c3);
      if constexpr (kMask) {
        a0 &= mk01;
        a1 &= mk01;
        c0 &= mk01;
        c1 &= mk01;
        a2 &= mk23;
        a3 &= mk23;
        c2 &= mk23;
        c3 &= mk23;
      }
      mma_f16_16816(r.o[2 * q], a0, a1, a2, a3, bh0, bh1);
      mma_f16_16816(r.o[2 * q + 1], c0, c1, c2, c3, bh0, bh1);
      if constexpr (!kPaired) {
        mma_f16_16816(r.o[2 * q], a0, a1, a2, a3, bl0, bl1);
        mma_f16_16816(r.o[2 * q + 1], c0, c1, c2, c3, bl0, bl1);
      }
    }
  }

  __device__ static void finish(Regs& r, float* dst, float* ml, float* lse, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float lt0 = r.l[0], lt1 = r.l[1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
    }
    if constexpr (kPaired) {
#pragma unroll
      for (int i = 0; i < KS; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) r.o[i][e] += __shfl_xor_sync(0xffffffffu, r.o[i][e], 2);
    }
    const int hd0 = 2 * t, hd1 = 2 * t + 1;
    const bool w0 = (!kPaired || t < 2) && hd0 < G;
    const bool w1 = (!kPaired || t < 2) && hd1 < G;
    const float inv0 = 1.f / (lt0 * kPScale), inv1 = 1.f / (lt1 * kPScale);
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      const int d0 = 16 * i + g;
      if (w0) {
        dst[hd0 * D + d0] = r.o[i][0] * inv0;
        dst[hd0 * D + d0 + 8] = r.o[i][2] * inv0;
      }
      if (w1) {
        dst[hd1 * D + d0] = r.o[i][1] * inv1;
        dst[hd1 * D + d0 + 8] = r.o[i][3] * inv1;
      }
    }
    if (ml != nullptr && g == 0) {
      if (w0) {
        ml[2 * hd0] = r.m[0];
        ml[2 * hd0 + 1] = lt0;
      }
      if (w1) {
        ml[2 * hd1] = r.m[1];
        ml[2 * hd1 + 1] = lt1;
      }
    }
    if (lse != nullptr && g == 0) {
      if (w0) lse[hd0] = r.m[0] + log2f(lt0);
      if (w1) lse[hd1] = r.m[1] + log2f(lt1);
    }
  }
};


// Tasks of a deferred-mode decode, at fixed boundaries: the first 3/4 of the NP chunks in tasks of
// about `big` = max(min_chunks, S + 1) chunks, the last quarter in tasks of about big / 4 (at least
// S + 1: the producer then runs at most one task ahead of the consumer), at most max_tasks in all.
// Warps take them in order, so the small ones fill the end, where warps finish at different times.
struct TaskMap {
  int64_t NP, NP1, T1, T2;   // chunks, chunks in the big tasks, big tasks, small tasks
  __device__ __forceinline__ int64_t count() const { return T1 + T2; }
  __device__ __forceinline__ int64_t lo(int64_t t) const {   // first chunk of task t (t <= T1 + T2)
    if (t < T1) return NP1 * t / T1;
    if (t >= T1 + T2) return NP;   // (one region: T2 = 0, NP1 = NP)
    return NP1 + (NP - NP1) * (t - T1) / T2;
  }
  __device__ __forceinline__ int64_t of(int64_t p) const {   // task holding chunk p < NP
    return p < NP1 ? ((p + 1) * T1 - 1) / NP1 : T1 + ((p - NP1 + 1) * T2 - 1) / (NP - NP1);
  }
};

__device__ __forceinline__ TaskMap defer_task_map(int64_t NP, int32_t min_chunks, int S, int32_t max_tasks) {
  TaskMap m;
  m.NP = NP;
  const int64_t big = min_chunks > S + 1 ? min_chunks : S + 1;
  const int64_t small = big / 4 > S + 1 ? big / 4 : S + 1;
  if (NP < 4 * big || max_tasks < 2) {   // one region
    m.NP1 = NP;
    m.T1 = NP / big < 1 ? 1 : (NP / big > max_tasks ? max_tasks : NP / big);
    m.T2 = 0;
    return m;
  }
  m.NP1 = NP * 3 / 4;
  m.T1 = m.NP1 / big;
  m.T2 = (NP - m.NP1) / small;
  if (m.T1 + m.T2 > max_tasks) {   // keep the proportions within the slot budget (fewer, longer tasks)
    const int64_t t1 = m.T1 * max_tasks / (m.T1 + m.T2);
    const int64_t t2 = max_tasks - (t1 < 1 ? 1 : t1);
    m.T1 = t1 < 1 ? 1 : t1;
    m.T2 = t2 < 1 ? 1 : (t2 < m.T2 ? t2 : m.T2);
  }
  return m;
}

// ------------------------------------------------------------------------------------------------
// Deferred-merge decode of one warp (defer_meta set): dynamic tasks, no merging here.
// Tasks have fixed chunk ranges, so a task's segments and their slots do not depend on which warp
// runs it: in balanced mode the TaskMap boundaries (slots 2 t for the task's first segment, 2 t + 1
// for its last), in fixed-partition mode one task per (unit, partition) item (slot u * max_parts + k,
// as in the in-kernel merge). Every task is taken from the call's counter (a CTA's first tasks, one
// per warp, by one atomic at kernel entry), so CTAs that start late (their SM was still busy) or
// warps that get slower memory service take fewer, and CTAs that start after the last task was
// taken do nothing. A unit one task holds whole is final: its rows go to `out` (and lse_out). Every
// other segment leaves its partial in its slot for the merging kernel that follows, which finds
// them from defer_meta (written by block 0). The producer runs on into the next task without
// draining the ring and records each stage's task in stage_task, from which the consumer switches.
// ------------------------------------------------------------------------------------------------
template <class Math, int D, int G>
__device__ __forceinline__ void decode_deferred(const DecodeArgs& a, const TmaMaps& maps, unsigned char* ring,
                                                uint64_t* bars, const int32_t* pref, const int32_t* ipref,
                                                const int32_t* cfirst, int64_t NP, int64_t first_task,
                                                int32_t* stage_task, int lane) {
  constexpr int SB = Math::kStageBytes;
  const int S = a.stages;
  const int32_t n = a.n_seqs, Hkv = a.Hkv, PC = a.part_chunks;
  const TaskMap tm = defer_task_map(NP, a.min_chunks, S, a.max_tasks);
  const int64_t T = PC > 0 ? static_cast<int64_t>(ipref[n]) * Hkv : tm.count();
  if (NP == 0) return;
  auto t_lo = [&](int64_t t) { return PC > 0 ? item_start(pref, ipref, n, Hkv, PC, t) : tm.lo(t); };
  auto next_task = [&]() -> int64_t {
    long long t = 0;
    if (lane == 0) t = grab_tasks(a.ws_count, a.tag, 1u, T);
    return __shfl_sync(0xffffffffu, t, 0);
  };
  auto bad_range = [&](int64_t t) {   // a task's chunks lie in [0, NP) and are not empty
    const int64_t l0 = t_lo(t), l1 = t_lo(t + 1);
    return l0 < 0 || l1 > NP || l1 <= l0;
  };
  int64_t ptk = first_task;   // the producer's task
  if (ptk >= T) return;
  if (bad_range(ptk)) {
    if (lane == 0) record_error(ERRBIT_BOUNDS);
    return;
  }

  // --- producer: (p_pg, p_sub) = page and chunk within the page of pf ---
  const int32_t cpb = a.B / kChunk;
  Cursor pf = locate(pref, n, Hkv, t_lo(ptk));
  int64_t p_left = t_lo(ptk + 1) - t_lo(ptk);
  bool p_done = false;
  int32_t p_pg = 0, p_sub = 0;
  auto p_unit_start = [&]() {
    const int32_t ch = (cfirst ? cfirst[pf.b] : 0) + pf.c;
    p_pg = ch / cpb;
    p_sub = ch - p_pg * cpb;
    constexpr int kQLines = (G * D * Math::kQElem + 127) / 128;
    if (lane < kQLines)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const unsigned char*>(a.q) +
                                                    ((static_cast<int64_t>(pf.b) * a.Hq + pf.h * G) * D) * Math::kQElem +
                                                    128 * lane));
  };
  p_unit_start();
  int32_t win_b = -1, win_base = 0, win_val = -1;
  const uint64_t policy = policy_evict_first();
  int64_t issued = 0;
  auto issue = [&](int stage) {
    if (pf.b != win_b || p_pg < win_base || p_pg >= win_base + 32) {
      win_b = pf.b;
      win_base = p_pg;
      const int32_t idx = win_base + lane;
      win_val = idx < a.MB ? __ldg(a.block_tables + static_cast<int64_t>(pf.b) * a.MB + idx) : -1;
    }
    const int32_t blk = __shfl_sync(0xffffffffu, win_val, p_pg - win_base);
    if (lane == 0) {
      stage_task[stage] = static_cast<int32_t>(ptk);
      const uint32_t bar = smem_addr(bars + stage);
      if (blk >= 0 && blk < a.NB) {
        const int64_t row0 = (static_cast<int64_t>(blk) * Hkv + pf.h) * a.B + p_sub * kChunk;
        fence_proxy_async_smem();
        Math::issue(a, maps, smem_addr(ring + static_cast<size_t>(stage) * SB), bar, row0, policy);
      } else {
        record_error(ERRBIT_BOUNDS);
        mbar_arrive(bar);  // completes the phase with no data; the chunk's result is garbage
      }
    }
    ++issued;
    if (--p_left > 0) {
      if (pf.c + 1 < pf.nch) {
        ++pf.c;
        if (++p_sub == cpb) {
          p_sub = 0;
          ++p_pg;
        }
      } else {
        advance(pf, pref, n, Hkv);
        p_unit_start();
      }
    } else {   // this task is issued: take the next one
      ptk = next_task();
      if (ptk < T && bad_range(ptk)) {
        if (lane == 0) record_error(ERRBIT_BOUNDS);
        ptk = T;
      }
      if (ptk < T) {
        pf = locate(pref, n, Hkv, t_lo(ptk));
        p_left = t_lo(ptk + 1) - t_lo(ptk);
        p_unit_start();
      } else {
        p_done = true;
      }
    }
  };
  for (int s = 0; s < S && !p_done; ++s) issue(s);
  __syncwarp();

  // --- consumer: switches task when the current one is used up (stage_task names the next) ---
  int64_t ctk = -1, c_left = 0;
  Cursor cc;
  typename Math::Regs r;
  int32_t seg_c0 = 0, len_b = 0;
  int seg_idx = 0;
  int stage = 0;
  uint32_t phase = 0;
  int64_t consumed = 0;
  bool aborted = false;
  while (consumed < issued) {
    if (c_left == 0) {   // the chunk at this stage begins the next task
      ctk = stage_task[stage];
      cc = locate(pref, n, Hkv, t_lo(ctk));
      c_left = t_lo(ctk + 1) - t_lo(ctk);
      seg_c0 = cc.c;
      seg_idx = 0;
      len_b = clamped_len(a, cc.b);
      Math::load_q(r, a, cc.b, cc.h, lane);
      Math::reset(r);
    }
    if (!mbar_wait_bounded(smem_addr(bars + stage), phase)) {
      aborted = true;
      break;
    }
    const int32_t tok_abs = ((cfirst ? cfirst[cc.b] : 0) + cc.c) * kChunk;
    const int32_t vhi = min(kChunk, len_b - tok_abs);
    const int32_t vlo = a.window > 0 ? max(0, len_b - a.window - tok_abs) : 0;
    if (!Math::kMaskVariants || vlo > 0 || vhi < kChunk)
      Math::template chunk<true>(r, ring + static_cast<size_t>(stage) * SB, vlo, vhi, a.scale_log2, lane);
    else
      Math::template chunk<false>(r, ring + static_cast<size_t>(stage) * SB, vlo, vhi, a.scale_log2, lane);
    __syncwarp();
    ++consumed;
    if (!p_done) issue(stage);
    __syncwarp();   // stage_task written by lane 0 before any lane reads it
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
    const bool unit_end = (cc.c + 1 == cc.nch);
    const bool task_end = (c_left == 1);
    if (unit_end || task_end) {
      if (seg_c0 == 0 && unit_end) {   // the task holds the whole unit: final rows
        Math::finish(r, a.out + (static_cast<int64_t>(cc.b) * a.Hq + cc.h * G) * D, nullptr,
                     a.lse_out ? a.lse_out + static_cast<int64_t>(cc.b) * a.Hq + cc.h * G : nullptr, lane);
      } else {
        const int64_t slot = PC > 0 ? (static_cast<int64_t>(cc.b) * Hkv + cc.h) * a.max_parts + cc.c / PC
                                    : 2 * ctk + (seg_idx == 0 ? 0 : 1);
        Math::finish(r, a.ws_o + slot * G * D, a.ws_ml + slot * G * 2, nullptr, lane);
      }
      ++seg_idx;
    }
    if (--c_left > 0) {
      const int32_t prev_b = cc.b;
      advance(cc, pref, n, Hkv);
      if (unit_end) {
        if (cc.b != prev_b) len_b = clamped_len(a, cc.b);
        Math::load_q(r, a, cc.b, cc.h, lane);
        Math::reset(r);
        seg_c0 = cc.c;
      }
    }
  }
  if (aborted) {   // drain the copies still in flight, each with one more bounded wait
    for (int64_t k = consumed; k < issued; ++k)
      mbar_wait_bounded(smem_addr(bars + static_cast<int>(k % S)), static_cast<uint32_t>((k / S) & 1));
  }
}

// ------------------------------------------------------------------------------------------------
// The decode kernel: prefix of chunk counts, even split of the flat chunk list over warps, a
// per-warp TMA ring, segment bookkeeping and output / partial writes. Math is a policy.
// ------------------------------------------------------------------------------------------------
// kDefer: the deferred-merge instantiation (defer_meta set); the regular one does not contain that
// path (measured: its code in the regular kernel cost ~0.8% of the serving decode).
template <class Math, int D, int G, bool kDefer>
__global__ void __launch_bounds__(128, Math::kMinCtasPerSm) paged_decode_kernel(const __grid_constant__ DecodeArgs a,
                                                           const __grid_constant__ TmaMaps maps) {
  constexpr int SB = Math::kStageBytes;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int NW = blockDim.x >> 5;
  const int S = a.stages;
  const int32_t n = a.n_seqs, Hkv = a.Hkv;
  const int32_t PC = a.part_chunks;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  unsigned char* ring = smem + static_cast<size_t>(warp) * S * SB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + decode_ring_bytes(NW, S, SB)) + warp * S;
  int32_t* wsum = reinterpret_cast<int32_t*>(smem + decode_ring_bytes(NW, S, SB) + static_cast<size_t>(NW) * S * 8);
  int32_t* pref = wsum + 64;
  int32_t* ipref = PC > 0 ? pref + (n + 1) : nullptr;
  int32_t* cfirst = (a.window > 0 || a.start > 0) ? pref + (PC > 0 ? 2 : 1) * (n + 1) : nullptr;

  // Arrival counters of split units whose segments all belong to this CTA, indexed by the unit's
  // first warp within the CTA (a warp is the first warp of at most one split unit). wsum[16..24) is
  // not used by the prefix build; the barrier after it orders the zeroing before any arrival.
  int32_t* cta_cnt = wsum + 16;
  if (threadIdx.x < NW) cta_cnt[threadIdx.x] = 0;
  set_error_word(a.err);
  // deferred mode: the CTA's first tasks, one per warp, taken at once, while the prefix is built
  // (wsum[8] is not used by the prefix build); it uses the workspace, so it waits first
  if constexpr (kDefer) {
    if (!a.late_wait) pdl_wait();
    if (threadIdx.x == 0)
      wsum[8] = static_cast<int32_t>(grab_tasks(a.ws_count, a.tag, static_cast<unsigned int>(NW), 0x7fffffff));
  }
  build_prefix(a, pref, ipref, cfirst, wsum);
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_addr(bars + s), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int W = gridDim.x * NW;
  const int w = blockIdx.x * NW + warp;
  const int64_t NP = static_cast<int64_t>(pref[n]) * Hkv;

  // Empty sequences: zero rows (and a log-sum-exp of -inf: no weight in a later merge). Outputs are
  // written only after the dependency wait.
  auto zero_empty = [&]() {
    for (int32_t b = w; b < n; b += W) {
      if (pref[b + 1] != pref[b]) continue;
      float4* o = reinterpret_cast<float4*>(a.out + static_cast<int64_t>(b) * a.Hq * D);
      for (int i = lane; i < a.Hq * D / 4; i += 32) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (a.lse_out != nullptr)
        for (int i = lane; i < a.Hq; i += 32) a.lse_out[static_cast<int64_t>(b) * a.Hq + i] = -INFINITY;
    }
  };

  // Balanced mode splits the chunks over Weff = min(W, max(1, NP / mc)) warps, mc = min_chunks (half
  // of it below 8192 chunks in all): every range is non-empty (the merge relies on it) and problems
  // are not cut into slivers whose fixed costs (first copy latency, partial writes, merges of many
  // parts) outweigh their work.
  // Ranges of at least half an average unit (capped at twice min_chunks), so that a unit is cut about
  // twice: each cut costs a partial write and, across CTAs, a GPU-scope fence (~6 us of one warp under
  // load). Measured on B300 (64 sequences of ~1,000 tokens, G 5: 32,360 chunks, units of ~63): 1,011
  // warps with 32-chunk ranges 66 us against 1,776 warps with 18-chunk ranges 74 us; larger batches
  // (serving: 90,664 chunks) still use every warp.
  int64_t mc = a.min_chunks;
  const int64_t units = static_cast<int64_t>(n) * Hkv;
  const int64_t half_unit = units > 0 ? NP / units / 2 : 0;
  if (half_unit > mc) mc = half_unit < 2 * mc ? half_unit : 2 * mc;
  if (NP < 8192) mc = (mc + 1) / 2;  // small problems: shorter ranges
  const int64_t Wmax = NP / mc > 0 ? NP / mc : 1;
  const int64_t Weff = Wmax < W ? Wmax : W;
  if constexpr (kDefer) {
    zero_empty();
    const TaskMap tm = defer_task_map(NP, a.min_chunks, S, a.max_tasks);
    if (blockIdx.x == 0) {   // where the merging kernel finds each unit's parts
      for (int32_t i = threadIdx.x; i <= n; i += blockDim.x) {
        a.defer_meta[5 + i] = pref[i];
        if (PC > 0) a.defer_meta[5 + (n + 1) + i] = ipref[i];
      }
      if (threadIdx.x == 0) {
        a.defer_meta[0] = PC;
        a.defer_meta[1] = static_cast<int32_t>(tm.T1);
        a.defer_meta[2] = static_cast<int32_t>(tm.T2);
        a.defer_meta[3] = static_cast<int32_t>(tm.NP1 & 0xffffffffll);
        a.defer_meta[4] = static_cast<int32_t>(tm.NP1 >> 32);
      }
    }
    // stage_task of this warp: wsum[40 + 4 warp + stage] (S <= 4; not used by the prefix build)
    decode_deferred<Math, D, G>(a, maps, ring, bars, pref, ipref, cfirst, NP, static_cast<int64_t>(wsum[8]) + warp,
                                wsum + 40 + 4 * warp, lane);
    if (a.late_wait) pdl_wait();
    pdl_launch_dependents();
    return;
  }
  int64_t lo = 0, hi = 0;
  if (PC == 0) {
    if (w < Weff) {
      lo = NP * w / Weff;
      hi = NP * (w + 1) / Weff;
    }
  } else {
    const int64_t NI = static_cast<int64_t>(ipref[n]) * Hkv;
    lo = item_start(pref, ipref, n, Hkv, PC, NI * w / W);
    hi = item_start(pref, ipref, n, Hkv, PC, NI * (w + 1) / W);
  }
  const int64_t n_chunks = hi - lo;

  // --- producer (lane 0 issues; the block-table window is spread over the lanes) ---
  // pf walks the chunks ahead of the consumer; (p_pg, p_sub) = its page in the block table and
  // chunk within that page, stepped without divisions except at unit changes.
  const int32_t cpb = a.B / kChunk;
  Cursor pf = n_chunks > 0 ? locate(pref, n, Hkv, lo) : Cursor{0, 0, 0, 1};   // idle warps: unused
  int32_t p_pg = 0, p_sub = 0;
  auto p_unit_start = [&]() {
    const int32_t ch = (cfirst ? cfirst[pf.b] : 0) + pf.c;
    p_pg = ch / cpb;
    p_sub = ch - p_pg * cpb;
    // warm L2 with the unit's queries: load_q reads them when the consumer gets here
    constexpr int kQLines = (G * D * Math::kQElem + 127) / 128;
    if (lane < kQLines)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const unsigned char*>(a.q) +
                                                    ((static_cast<int64_t>(pf.b) * a.Hq + pf.h * G) * D) * Math::kQElem +
                                                    128 * lane));
  };
  int32_t win_b = -1, win_base = 0, win_val = -1;
  if (n_chunks > 0) {
    p_unit_start();
    // the first block-table window (an input, like context_lens)
    win_b = pf.b;
    win_base = p_pg;
    const int32_t idx = win_base + lane;
    win_val = idx < a.MB ? __ldg(a.block_tables + static_cast<int64_t>(pf.b) * a.MB + idx) : -1;
  }
  // The prefix build and the first block-table window above read only context_lens and block_tables;
  // the caches, q and the workspace are read, and outputs written, only after this wait, so that work
  // overlaps the tail of the kernel before (measured with the build alone: serving step 4.297 -> 4.247
  // ms).
  if (!a.late_wait) pdl_wait();
  zero_empty();
  if (n_chunks <= 0) return;
  const uint64_t policy = policy_evict_first();
  int64_t issued = 0;

  auto issue = [&](int stage) {
    if (pf.b != win_b || p_pg < win_base || p_pg >= win_base + 32) {
      win_b = pf.b;
      win_base = p_pg;
      const int32_t idx = win_base + lane;
      win_val = idx < a.MB ? __ldg(a.block_tables + static_cast<int64_t>(pf.b) * a.MB + idx) : -1;
    }
    const int32_t blk = __shfl_sync(0xffffffffu, win_val, p_pg - win_base);
    if (lane == 0) {
      const uint32_t bar = smem_addr(bars + stage);
      if (blk >= 0 && blk < a.NB) {
        const int64_t row0 = (static_cast<int64_t>(blk) * Hkv + pf.h) * a.B + p_sub * kChunk;
        fence_proxy_async_smem();
        Math::issue(a, maps, smem_addr(ring + static_cast<size_t>(stage) * SB), bar, row0, policy);
      } else {
        record_error(ERRBIT_BOUNDS);
        mbar_arrive(bar);  // completes the phase with no data; the chunk's result is garbage
      }
    }
    ++issued;
    if (pf.c + 1 < pf.nch) {
      ++pf.c;
      if (++p_sub == cpb) {
        p_sub = 0;
        ++p_pg;
      }
    } else {
      advance(pf, pref, n, Hkv);
      if (issued < n_chunks) p_unit_start();
    }
  };

  for (int s = 0; s < S && issued < n_chunks; ++s) issue(s);

  // --- consumer ---
  Cursor cc = locate(pref, n, Hkv, lo);
  typename Math::Regs r;
  int32_t seg_c0 = cc.c;
  int seg_idx = 0;
  int stage = 0;
  uint32_t phase = 0;

  int32_t len_b = clamped_len(a, cc.b);
  Math::load_q(r, a, cc.b, cc.h, lane);
  Math::reset(r);

  // Split units. A segment that ends inside this warp's range (the tail of a unit begun by the
  // previous warp) is published a few chunks later: its partial is stored at once, and the release
  // fence and arrival wait until those stores have drained, so the fence costs little. The segment
  // that ends the range (usually the unit's last one to finish) first checks whether all other
  // segments are already published; if so it merges at once from its own partial and theirs,
  // without a release or arrival of its own. Otherwise it publishes and the last arrival merges.
  constexpr int kPubDelay = 2;
  bool pub = false;
  int pub_wait = 0;
  int32_t pub_b = 0, pub_h = 0, pub_kind = 0;
  int64_t pub_parts = 0, pub_wf = 0;
  // Release / acquire around an arrival (memory-model order): every lane's partial stores, then the
  // warp barrier, then the release fence and lane 0's atomic; on the last arrival, the acquire fence
  // and a warp barrier before any lane reads the other segments' partials.
  auto publish = [&]() {
    __syncwarp();
    fence_acq_rel_gpu();  // this warp's partial stores are visible before the arrival
    int last = 0;
    if (lane == 0)
      last = arrive_last(a.ws_count + static_cast<int64_t>(pub_b) * Hkv + pub_h, a.tag, pub_parts) ? 1 : 0;
    if (__shfl_sync(0xffffffffu, last, 0)) {
      fence_acq_rel_gpu();
      __syncwarp();
      merge_unit<D, G, false, false>(a, pub_b, pub_h, pub_parts, pub_wf, pub_kind, lane);
      if (lane == 0) a.ws_count[static_cast<int64_t>(pub_b) * Hkv + pub_h] = 0ull;   // every part has arrived
    }
    pub = false;
  };
  bool pend = false;  // this warp merges a unit after the loop (its registers are free then)
  bool pend_cta = false;  // ... whose segments all belong to this CTA
  int32_t pend_b = 0, pend_h = 0, pend_kind = 0;
  int64_t pend_parts = 0, pend_wf = 0;

  bool aborted = false;
  int64_t i = 0;
  for (; i < n_chunks; ++i) {
    if (!mbar_wait_bounded(smem_addr(bars + stage), phase)) {
      aborted = true;
      break;
    }
    const int32_t tok_abs = ((cfirst ? cfirst[cc.b] : 0) + cc.c) * kChunk;
    const int32_t vhi = min(kChunk, len_b - tok_abs);
    const int32_t vlo = a.window > 0 ? max(0, len_b - a.window - tok_abs) : 0;
    if (!Math::kMaskVariants || vlo > 0 || vhi < kChunk)
      Math::template chunk<true>(r, ring + static_cast<size_t>(stage) * SB, vlo, vhi, a.scale_log2, lane);
    else
      Math::template chunk<false>(r, ring + static_cast<size_t>(stage) * SB, vlo, vhi, a.scale_log2, lane);
    __syncwarp();
    if (issued < n_chunks) issue(stage);
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
    if (pub && --pub_wait == 0) publish();

    // segment end: write the whole-unit result or a partial
    const bool unit_end = (cc.c + 1 == cc.nch);
    const bool part_end = (PC != 0) && ((cc.c + 1) % PC == 0);
    const bool range_end = (i + 1 == n_chunks);
    if (unit_end || part_end || range_end) {
      const bool complete = (seg_c0 == 0) && unit_end;
      if (complete) {
        Math::finish(r, a.out + (static_cast<int64_t>(cc.b) * a.Hq + cc.h * G) * D, nullptr,
                     a.lse_out ? a.lse_out + static_cast<int64_t>(cc.b) * a.Hq + cc.h * G : nullptr, lane);
      } else {
        const int64_t u = static_cast<int64_t>(cc.b) * Hkv + cc.h;
        const int64_t slot = (PC == 0) ? (2 * static_cast<int64_t>(w) + (seg_idx == 0 ? 0 : 1))
                                       : (u * a.max_parts + cc.c / PC);
        // Segments of this unit: balanced mode, warps warp_of(s_u) .. warp_of(e_u - 1) where
        // warp_of(p) = floor(((p + 1) * Weff - 1) / NP); fixed mode, its partitions.
        int64_t n_parts, wf = 0;
        int first_kind = 0;
        if (PC == 0) {
          const int64_t s_u = static_cast<int64_t>(pref[cc.b]) * Hkv + static_cast<int64_t>(cc.h) * cc.nch;
          const int64_t e_u = s_u + cc.nch;
          wf = ((s_u + 1) * Weff - 1) / NP;
          n_parts = (e_u * Weff - 1) / NP - wf + 1;
          first_kind = (s_u == NP * wf / Weff) ? 0 : 1;
        } else {
          n_parts = (cc.nch + PC - 1) / PC;
        }
        const bool intra = (PC == 0) && (wf / NW == (wf + n_parts - 1) / NW);
        if (pub) publish();
        if (a.defer_meta != nullptr) {   // merged by a later kernel
          Math::finish(r, a.ws_o + slot * G * D, a.ws_ml + slot * G * 2, nullptr, lane);
        } else if (intra) {
          // all segments in this CTA: CTA-scope release / acquire around a shared-memory count
          Math::finish(r, a.ws_o + slot * G * D, a.ws_ml + slot * G * 2, nullptr, lane);
          __syncwarp();
          fence_acq_rel_cta();
          int last = 0;
          if (lane == 0) last = (atomicAdd(cta_cnt + (wf % NW), 1) + 1 == n_parts) ? 1 : 0;
          if (__shfl_sync(0xffffffffu, last, 0)) {
            fence_acq_rel_cta();
            __syncwarp();
            if (range_end) {
              pend = true;
              pend_cta = true;
              pend_b = cc.b;
              pend_h = cc.h;
              pend_parts = n_parts;
              pend_wf = wf;
              pend_kind = first_kind;
            } else {
              merge_unit<D, G, false, true>(a, cc.b, cc.h, n_parts, wf, first_kind, lane);
            }
          }
        } else if (range_end) {
          int others = 0;
          if (lane == 0) {
            const unsigned long long v = ld_acquire_gpu(a.ws_count + u);
            others = ((v >> 16) == a.tag && static_cast<int64_t>(v & 0xffffull) == n_parts - 1) ? 1 : 0;
          }
          others = __shfl_sync(0xffffffffu, others, 0);
          if (others) fence_acq_rel_gpu();  // the other segments' partials are read after this point
          Math::finish(r, a.ws_o + slot * G * D, a.ws_ml + slot * G * 2, nullptr, lane);
          int mine = others;
          if (!others) {
            __syncwarp();
            fence_acq_rel_gpu();
            if (lane == 0) mine = arrive_last(a.ws_count + u, a.tag, n_parts) ? 1 : 0;
            mine = __shfl_sync(0xffffffffu, mine, 0);
            if (mine) fence_acq_rel_gpu();
          }
          __syncwarp();  // this warp's own partial is visible to all its lanes
          if (mine) {
            pend = true;
            pend_b = cc.b;
            pend_h = cc.h;
            pend_parts = n_parts;
            pend_wf = wf;
            pend_kind = first_kind;
          }
        } else {
          Math::finish(r, a.ws_o + slot * G * D, a.ws_ml + slot * G * 2, nullptr, lane);
          pub = true;
          pub_wait = kPubDelay;
          pub_b = cc.b;
          pub_h = cc.h;
          pub_parts = n_parts;
          pub_wf = wf;
          pub_kind = first_kind;
        }
      }
      ++seg_idx;
    }
    if (i + 1 < n_chunks) {
      const int32_t prev_b = cc.b;
      advance(cc, pref, n, Hkv);
      if (unit_end || part_end) {
        if (unit_end) {
          if (cc.b != prev_b) len_b = clamped_len(a, cc.b);
          Math::load_q(r, a, cc.b, cc.h, lane);
        }
        Math::reset(r);
        seg_c0 = cc.c;
      }
    }
  }
  if (aborted) {
    // Drain the copies this warp still has in flight, the one whose wait gave up included (it may
    // only have been slow), each with one more bounded wait, then leave.
    for (int64_t k = i; k < issued; ++k)
      mbar_wait_bounded(smem_addr(bars + static_cast<int>(k % S)), static_cast<uint32_t>((k / S) & 1));
  }
  if (pub) publish();
  if (a.late_wait) pdl_wait();
  pdl_launch_dependents();
  if (pend) {
    if (pend_cta) {
      merge_unit<D, G, true, true>(a, pend_b, pend_h, pend_parts, pend_wf, pend_kind, lane);
    } else {
      merge_unit<D, G, true, false>(a, pend_b, pend_h, pend_parts, pend_wf, pend_kind, lane);
      if (lane == 0) a.ws_count[static_cast<int64_t>(pend_b) * Hkv + pend_h] = 0ull;   // every part has arrived
    }
  }
}

// Merge after a deferred-mode decode. The decode left, for each (sequence, KV head) unit, either the
// final rows in `out` (with their log-sum-exp in lse_s when one is wanted: a unit one task held
// whole) or one normalised partial per task of a unit cut by task boundaries. For a shared-prefix
// (cascade) call the decode covered only each sequence's private suffix, and the tensor-core prefill
// kernel in shared-prefix mode attended the shared prefix once for all rows (n_split key splits,
// part_o / part_lse). The exact attention over the whole context is the log-sum-exp combination of
// all of a row's parts ("Servicio de modelos de lenguaje con un presupuesto de memoria" §6:
// blockwise exact attention with running statistics):
//     M = max_k lse_k, w_k = 2^(lse_k - M), out = sum_k w_k o_k / sum_k w_k   (each o_k normalised).
// One warp per (sequence, query head) row, the loads of 4 parts in flight at a time; a final row
// with no prefix parts is left as it is. With prefix_blocks > 0 the kernel also checks that every
// table of the call begins with sequence 0's first prefix_blocks entries (else PKV_ERR_DEVICE_BOUNDS).
struct CascadeMergeArgs {
  float* out;
  const float* lse_s;       // [n_rows] suffix log-sum-exp of rows whose unit was not split
  const float* part_o;      // [n_split][n_rows][D] prefix partials (normalised)
  const float* part_lse;    // [n_split][n_rows]
  const float* dec_o;       // decode slots [2 W][G][D] (normalised)
  const float* dec_ml;      // decode slots [2 W][G][2] (m, l)
  const int32_t* meta;      // [part_chunks, T1, T2, NP1 low, NP1 high, pref[0..n], ipref[0..n] (partitions)]
  int32_t max_parts;        // fixed-partition mode: slots per unit
  unsigned long long* task_ctr;   // the decode's task counter: zeroed here (CUDA-graph replays reuse the call tag)
  const int32_t* tables;
  int64_t n_rows;
  int32_t D, G, Hkv, n_split, MB, n_seqs, prefix_blocks;
  unsigned int* err;
};

__global__ void __launch_bounds__(256, 4) merge_prefix_kernel(const __grid_constant__ CascadeMergeArgs a) {
  set_error_word(a.err);
  pdl_wait();
  const int64_t gthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gtid == 0 && a.task_ctr != nullptr) *a.task_ctr = 0ull;   // the decode has completed
  for (int64_t i = gtid; i < static_cast<int64_t>(a.n_seqs) * a.prefix_blocks; i += gthreads) {
    const int64_t b = i / a.prefix_blocks, k = i - b * a.prefix_blocks;
    if (__ldg(a.tables + b * a.MB + k) != __ldg(a.tables + k)) record_error(ERRBIT_BOUNDS);
  }
  const int lane = threadIdx.x & 31;
  const int D = a.D, Hq = a.Hkv * a.G;
  const bool has_c = lane < D / 4;                 // this lane's float4 of the row
  const int32_t PC = __ldg(a.meta);
  const int32_t* pref = a.meta + 5;
  TaskMap tm;   // the decode's task boundaries (balanced mode)
  tm.NP = static_cast<int64_t>(__ldg(pref + a.n_seqs)) * a.Hkv;
  tm.T1 = __ldg(a.meta + 1);
  tm.T2 = __ldg(a.meta + 2);
  tm.NP1 = static_cast<int64_t>(static_cast<uint32_t>(__ldg(a.meta + 3))) | (static_cast<int64_t>(__ldg(a.meta + 4)) << 32);
  constexpr int kBatch = 4;
  for (int64_t row = gtid >> 5; row < a.n_rows; row += gthreads >> 5) {
    const int32_t b = static_cast<int32_t>(row / Hq), j = static_cast<int32_t>(row - static_cast<int64_t>(b) * Hq);
    const int32_t h = j / a.G, jj = j - h * a.G;
    // the suffix parts of the row: none (empty suffix), the final row (unit of one task), or one
    // partial per task of a cut unit
    const int64_t nch = __ldg(pref + b + 1) - __ldg(pref + b);
    int64_t wf = 0, n_suf = 0;
    int first_kind = 0;
    if (nch > 0 && PC > 0) {   // fixed partitions: one task per partition, slot u * max_parts + k
      n_suf = (nch + PC - 1) / PC;
    } else if (nch > 0) {      // balanced: the tasks holding the unit's first and last chunks
      const int64_t s_u = static_cast<int64_t>(__ldg(pref + b)) * a.Hkv + h * nch, e_u = s_u + nch;
      wf = tm.of(s_u);
      n_suf = tm.of(e_u - 1) - wf + 1;
      first_kind = (s_u == tm.lo(wf)) ? 0 : 1;
    }
    const bool whole = n_suf == 1;
    const int64_t n_parts = (n_suf > 1 ? n_suf : 0) + a.n_split;
    if ((whole || n_parts == 0) && a.n_split == 0) continue;   // final already (or an empty row's zeros)
    const int64_t u = static_cast<int64_t>(b) * a.Hkv + h;
    auto slot_of = [&](int64_t p) -> int64_t {
      return PC > 0 ? u * a.max_parts + p : 2 * (wf + p) + (p == 0 ? first_kind : 0);
    };
    // part p < n_suf: decode slot of the cut unit's p-th segment; then the prefix splits
    auto part_lse = [&](int64_t p) -> float {
      if (p < n_parts - a.n_split) {
        const int64_t slot = slot_of(p);
        const float2 ml = __ldg(reinterpret_cast<const float2*>(a.dec_ml) + slot * a.G + jj);
        return ml.x + log2f(ml.y);
      }
      return __ldg(a.part_lse + (p - (n_parts - a.n_split)) * a.n_rows + row);
    };
    auto part_o = [&](int64_t p) -> const float4* {
      if (p < n_parts - a.n_split) {
        const int64_t slot = slot_of(p);
        return reinterpret_cast<const float4*>(a.dec_o + (slot * a.G + jj) * D);
      }
      return reinterpret_cast<const float4*>(a.part_o + ((p - (n_parts - a.n_split)) * a.n_rows + row) * D);
    };
    const float ls = whole ? __ldg(a.lse_s + row) : -INFINITY;
    float M = ls;
    for (int64_t k0 = 0; k0 < n_parts; k0 += 32) {
      float v = k0 + lane < n_parts ? part_lse(k0 + lane) : -INFINITY;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
      M = fmaxf(M, v);
    }
    const float ws = whole ? exp2f(ls - M) : 0.f;
    float wsum = ws;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (whole && has_c) {
      const float4 so = reinterpret_cast<const float4*>(a.out + row * D)[lane];
      acc = make_float4(ws * so.x, ws * so.y, ws * so.z, ws * so.w);
    }
    for (int64_t k0 = 0; k0 < n_parts; k0 += 32) {
      const int nk = static_cast<int>(n_parts - k0 < 32 ? n_parts - k0 : 32);
      const float wl = lane < nk ? exp2f(part_lse(k0 + lane) - M) : 0.f;
      float t = wl;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
      wsum += t;
      for (int jb = 0; jb < nk; jb += kBatch) {
        float4 v[kBatch];
        float wj[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          wj[u] = __shfl_sync(0xffffffffu, wl, (jb + u) & 31);
          v[u] = (has_c && jb + u < nk) ? __ldg(part_o(k0 + jb + u) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          acc.x = fmaf(wj[u], v[u].x, acc.x);
          acc.y = fmaf(wj[u], v[u].y, acc.y);
          acc.z = fmaf(wj[u], v[u].z, acc.z);
          acc.w = fmaf(wj[u], v[u].w, acc.w);
        }
      }
    }
    if (has_c) {
      const float inv = 1.f / wsum;
      reinterpret_cast<float4*>(a.out + row * D)[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
  }
  pdl_launch_dependents();
}

}  // namespace pkv_dev
