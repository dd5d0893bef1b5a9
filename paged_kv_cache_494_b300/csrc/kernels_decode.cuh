// Paged decode attention (K3) and its log-sum-exp merge (K4 reduce).
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
//  * Per warp, a ring of `stages` shared-memory slots is filled by 1-D TMA bulk copies (one for K,
//    one for V, 16*D*sizeof(T) bytes each) that complete on an mbarrier; lane 0 issues them
//    `stages` chunks ahead of the compute.
//  * A segment is the part of a unit one warp processes. A segment that is a whole unit writes the
//    output directly; otherwise it writes (m, l, o/l) to the workspace and the reduce kernel merges
//    the segments of the unit: M = max m_k, w_k = l_k 2^(m_k - M), o = sum w_k o_k / sum w_k.
//    m is kept in log2 units (scores pre-multiplied by scale * log2 e), which changes no result.
//  * The split depends only on the context lengths, never on physical block ids, so results are
//    bitwise invariant under any placement of the blocks.
#pragma once

#include <cmath>

#include "pkv_device.cuh"

namespace pkv_dev {

constexpr int kChunk = 16;  // tokens per staged chunk

struct DecodeArgs {
  float* out;                    // [n_seqs][Hq][D]
  const void* q;                 // [n_seqs][Hq][D]
  const void* k_cache;           // [NB][Hkv][B][D]
  const void* v_cache;
  const int32_t* block_tables;   // [n_seqs][MB]
  const int32_t* context_lens;   // [n_seqs]
  float* ws_ml;                  // [n_slots][G][2]  (m in log2 units, l)
  float* ws_o;                   // [n_slots][G][D]  (o already divided by l)
  int32_t* ws_desc;              // balanced mode: [n_units][2]
  int32_t n_seqs, Hq, Hkv, B, NB, MB;
  int32_t part_chunks;           // 0: balanced split; > 0: chunks per partition
  int32_t max_parts;             // fixed mode: partition slots per unit
  int32_t stages;                // ring depth per warp
  int32_t total_warps;           // warps of the decode grid (balanced-mode slot count / 2)
  float scale_log2;              // scale * log2(e)
};

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

// Shared-memory carve-up of the decode kernel. Ring first (each stage: K chunk then V chunk).
__host__ __device__ inline size_t decode_ring_bytes(int nw, int stages, int chunk_bytes) {
  return static_cast<size_t>(nw) * stages * 2 * chunk_bytes;
}
__host__ __device__ inline size_t decode_smem_bytes(int nw, int stages, int chunk_bytes, int n_seqs) {
  return decode_ring_bytes(nw, stages, chunk_bytes) + static_cast<size_t>(nw) * stages * 8 +
         2 * static_cast<size_t>(n_seqs + 1) * 4;
}

// Prefix sums over sequences of chunk counts (pref) and partition counts (ipref), by warp 0.
__device__ __forceinline__ void build_prefix(const DecodeArgs& a, int32_t* pref, int32_t* ipref, int lane) {
  const int32_t n = a.n_seqs;
  const int32_t PC = a.part_chunks > 0 ? a.part_chunks : 1;
  const int32_t per = (n + 31) / 32;
  const int32_t lo = min(lane * per, n), hi = min(lo + per, n);
  int32_t sc = 0, si = 0;
  for (int32_t b = lo; b < hi; ++b) {
    const int32_t nch = (clamped_len(a, b) + kChunk - 1) / kChunk;
    sc += nch;
    si += (nch + PC - 1) / PC;
  }
  int32_t ec = sc, ei = si;  // inclusive scan, then make exclusive
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t tc = __shfl_up_sync(0xffffffffu, ec, off);
    const int32_t ti = __shfl_up_sync(0xffffffffu, ei, off);
    if (lane >= off) {
      ec += tc;
      ei += ti;
    }
  }
  ec -= sc;
  ei -= si;
  for (int32_t b = lo; b < hi; ++b) {
    pref[b] = ec;
    ipref[b] = ei;
    const int32_t nch = (clamped_len(a, b) + kChunk - 1) / kChunk;
    ec += nch;
    ei += (nch + PC - 1) / PC;
  }
  if (lane == 31) {
    pref[n] = ec;
    ipref[n] = ei;
  }
}

// ------------------------------------------------------------------------------------------------
// SIMT decode: CUDA-core dot products with warp shuffles. Lane layout: LPT lanes per token, each
// holding EPL consecutive-by-piece elements of the head dimension; TPP tokens per pass.
// ------------------------------------------------------------------------------------------------
template <typename T, int D, int G>
struct SimtShape {
  static constexpr int es = sizeof(T);
  static constexpr int PER16 = Widen<T>::kPer16;
  static constexpr int EPL = (G <= 5) ? 16 : 8;
  static constexpr int LPT = D / EPL;
  static constexpr int TPP = 32 / LPT;
  static constexpr int PASSES = kChunk / TPP;
  static constexpr int PIECES = EPL / PER16;
  static constexpr int CB = kChunk * D * es;  // bytes of one K (or V) chunk
  static_assert(LPT * EPL == D && TPP * LPT == 32 && PASSES * TPP == kChunk, "lane layout");
  static_assert(PIECES * PER16 == EPL, "pieces");
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(128) paged_decode_simt_kernel(DecodeArgs a) {
  using Sh = SimtShape<T, D, G>;
  constexpr int es = Sh::es, PER16 = Sh::PER16, EPL = Sh::EPL, LPT = Sh::LPT, TPP = Sh::TPP;
  constexpr int PASSES = Sh::PASSES, PIECES = Sh::PIECES, CB = Sh::CB;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int NW = blockDim.x >> 5;
  const int S = a.stages;
  const int32_t n = a.n_seqs, Hkv = a.Hkv;
  const int32_t PC = a.part_chunks;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem + static_cast<size_t>(warp) * S * 2 * CB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + decode_ring_bytes(NW, S, CB)) + warp * S;
  int32_t* pref = reinterpret_cast<int32_t*>(smem + decode_ring_bytes(NW, S, CB) + static_cast<size_t>(NW) * S * 8);
  int32_t* ipref = pref + (n + 1);

  if (warp == 0) build_prefix(a, pref, ipref, lane);
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_addr(bars + s), 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int W = gridDim.x * NW;
  const int w = blockIdx.x * NW + warp;
  const int64_t NP = static_cast<int64_t>(pref[n]) * Hkv;

  // Empty sequences: zero rows (and mark their units complete for the reduce).
  for (int32_t b = w; b < n; b += W) {
    if (clamped_len(a, b) != 0) continue;
    float4* o = reinterpret_cast<float4*>(a.out + static_cast<int64_t>(b) * a.Hq * D);
    for (int i = lane; i < a.Hq * D / 4; i += 32) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (PC == 0)
      for (int32_t h = lane; h < Hkv; h += 32) a.ws_desc[2 * (static_cast<int64_t>(b) * Hkv + h)] = -1;
  }

  // Balanced mode splits the chunks over Weff = min(W, NP) warps so that every range between a
  // unit's first and last warp is non-empty (the reduce relies on it).
  const int64_t Weff = NP < W ? NP : W;
  int64_t lo, hi;
  if (PC == 0) {
    if (w >= Weff) return;
    lo = NP * w / Weff;
    hi = NP * (w + 1) / Weff;
  } else {
    const int64_t NI = static_cast<int64_t>(ipref[n]) * Hkv;
    lo = item_start(pref, ipref, n, Hkv, PC, NI * w / W);
    hi = item_start(pref, ipref, n, Hkv, PC, NI * (w + 1) / W);
  }
  const int64_t n_chunks = hi - lo;
  if (n_chunks <= 0) return;

  const int tg = lane / LPT;  // token group
  const int cl = lane % LPT;  // piece column

  // --- producer state (lane-uniform except the table window register) ---
  Cursor pf = locate(pref, n, Hkv, lo);
  int32_t win_b = -1, win_base = 0, win_val = -1;
  const uint64_t policy = policy_evict_first();
  int64_t issued = 0;

  auto issue = [&](int stage) {
    const int32_t tok0 = pf.c * kChunk;
    const int32_t pg = tok0 / a.B;
    if (pf.b != win_b || pg < win_base || pg >= win_base + 32) {
      win_b = pf.b;
      win_base = pg;
      const int32_t idx = win_base + lane;
      win_val = idx < a.MB ? __ldg(a.block_tables + static_cast<int64_t>(pf.b) * a.MB + idx) : -1;
    }
    const int32_t blk = __shfl_sync(0xffffffffu, win_val, pg - win_base);
    if (lane == 0) {
      const uint32_t bar = smem_addr(bars + stage);
      if (blk >= 0 && blk < a.NB) {
        const int64_t e0 = ((static_cast<int64_t>(blk) * Hkv + pf.h) * a.B + (tok0 - pg * a.B)) * D;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, 2 * CB);
        const uint32_t dst = smem_addr(ring + static_cast<size_t>(stage) * 2 * CB);
        bulk_g2s_hint(dst, static_cast<const unsigned char*>(a.k_cache) + e0 * es, CB, bar, policy);
        bulk_g2s_hint(dst + CB, static_cast<const unsigned char*>(a.v_cache) + e0 * es, CB, bar, policy);
      } else {
        record_error(ERRBIT_BOUNDS);
        mbar_arrive(bar);  // completes the phase with no data; the chunk's result is garbage
      }
    }
    advance(pf, pref, n, Hkv);
    ++issued;
  };

  for (int s = 0; s < S && issued < n_chunks; ++s) issue(s);

  // --- consumer state ---
  Cursor cc = locate(pref, n, Hkv, lo);
  float qf[G][EPL];
  float of[G][EPL];
  float m[G], l[G];
  int32_t len_b = 0;
  int32_t seg_c0 = cc.c;
  int seg_idx = 0;

  auto load_q = [&]() {
    const T* qbase = static_cast<const T*>(a.q) + (static_cast<int64_t>(cc.b) * a.Hq + cc.h * G) * D;
#pragma unroll
    for (int j = 0; j < G; ++j) {
#pragma unroll
      for (int i = 0; i < PIECES; ++i) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qbase + j * D + (cl + i * LPT) * PER16));
        Widen<T>::load(reinterpret_cast<const unsigned char*>(&raw), &qf[j][i * PER16]);
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) qf[j][e] *= a.scale_log2;
    }
  };
  auto reset_state = [&]() {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) of[j][e] = 0.f;
    }
  };
  auto write_desc = [&](int64_t x) {  // balanced mode, at the first chunk of a unit
    if (PC != 0 || lane != 0) return;
    const int64_t e_u = x + cc.nch;
    const int64_t u = static_cast<int64_t>(cc.b) * Hkv + cc.h;
    if (e_u <= hi) {
      a.ws_desc[2 * u] = -1;
    } else {
      const int64_t w_last = (e_u * Weff - 1) / NP;
      a.ws_desc[2 * u] = (w << 1) | (seg_idx == 0 ? 0 : 1);
      a.ws_desc[2 * u + 1] = static_cast<int32_t>(w_last);
    }
  };

  len_b = clamped_len(a, cc.b);
  load_q();
  reset_state();
  if (cc.c == 0) write_desc(lo);

  bool aborted = false;
  int64_t i = 0;
  for (; i < n_chunks; ++i) {
    const int stage = static_cast<int>(i % S);
    const uint32_t parity = static_cast<uint32_t>((i / S) & 1);
    if (!mbar_wait_bounded(smem_addr(bars + stage), parity)) {
      aborted = true;
      break;
    }
    const unsigned char* kb = ring + static_cast<size_t>(stage) * 2 * CB;
    const unsigned char* vb = kb + CB;
    const int32_t nvalid = min(kChunk, len_b - cc.c * kChunk);

    // scores for this lane's tokens (log2 units), masked beyond the context length
    float sc[PASSES][G];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int tok = p * TPP + tg;
      float kf[EPL];
#pragma unroll
      for (int pc = 0; pc < PIECES; ++pc) Widen<T>::load(kb + (tok * D + (cl + pc * LPT) * PER16) * es, kf + pc * PER16);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) s = fmaf(qf[j][e], kf[e], s);
#pragma unroll
        for (int off = LPT / 2; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        sc[p][j] = tok < nvalid ? s : -INFINITY;
      }
    }
    // online softmax update
#pragma unroll
    for (int j = 0; j < G; ++j) {
      float mx = sc[0][j];
#pragma unroll
      for (int p = 1; p < PASSES; ++p) mx = fmaxf(mx, sc[p][j]);
#pragma unroll
      for (int off = LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mnew = fmaxf(m[j], mx);
      const float alpha = exp2f(m[j] - mnew);
      m[j] = mnew;
      if (alpha != 1.f) {
        l[j] *= alpha;
#pragma unroll
        for (int e = 0; e < EPL; ++e) of[j][e] *= alpha;
      }
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        sc[p][j] = exp2f(sc[p][j] - mnew);
        l[j] += sc[p][j];
      }
    }
    // weighted values
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int tok = p * TPP + tg;
      if (tok < nvalid) {
        float vf[EPL];
#pragma unroll
        for (int pc = 0; pc < PIECES; ++pc)
          Widen<T>::load(vb + (tok * D + (cl + pc * LPT) * PER16) * es, vf + pc * PER16);
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
          for (int e = 0; e < EPL; ++e) of[j][e] = fmaf(sc[p][j], vf[e], of[j][e]);
      }
    }
    __syncwarp();
    if (issued < n_chunks) issue(stage);

    // segment end: write the whole-unit result or a partial
    const bool unit_end = (cc.c + 1 == cc.nch);
    const bool part_end = (PC != 0) && ((cc.c + 1) % PC == 0);
    const bool range_end = (i + 1 == n_chunks);
    if (unit_end || part_end || range_end) {
      float lt[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        lt[j] = l[j];
#pragma unroll
        for (int off = LPT; off < 32; off <<= 1) lt[j] += __shfl_xor_sync(0xffffffffu, lt[j], off);
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          float t = of[j][e];
#pragma unroll
          for (int off = LPT; off < 32; off <<= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
          of[j][e] = t;
        }
      }
      const bool complete = (seg_c0 == 0) && unit_end;
      const int64_t u = static_cast<int64_t>(cc.b) * Hkv + cc.h;
      int64_t slot = 0;
      if (!complete) slot = (PC == 0) ? (2 * static_cast<int64_t>(w) + (seg_idx == 0 ? 0 : 1))
                                      : (u * a.max_parts + cc.c / PC);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        if (j % TPP != tg) continue;
        const float inv = 1.f / lt[j];
        float* dst = complete ? a.out + (static_cast<int64_t>(cc.b) * a.Hq + cc.h * G + j) * D
                              : a.ws_o + (slot * G + j) * D;
#pragma unroll
        for (int pc = 0; pc < PIECES; ++pc) {
          float4* d4 = reinterpret_cast<float4*>(dst + (cl + pc * LPT) * PER16);
#pragma unroll
          for (int k4 = 0; k4 < PER16 / 4; ++k4) {
            const float* src = &of[j][pc * PER16 + 4 * k4];
            d4[k4] = make_float4(src[0] * inv, src[1] * inv, src[2] * inv, src[3] * inv);
          }
        }
        if (!complete && cl == 0) {
          a.ws_ml[(slot * G + j) * 2] = m[j];
          a.ws_ml[(slot * G + j) * 2 + 1] = lt[j];
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
          load_q();
          if (cc.c == 0) write_desc(lo + i + 1);
        }
        reset_state();
        seg_c0 = cc.c;
      }
    }
  }
  if (aborted) {
    // Drain the copies this warp still has in flight (bounded), then leave.
    for (int64_t k = i + 1; k < issued; ++k)
      mbar_wait_bounded(smem_addr(bars + static_cast<int>(k % S)), static_cast<uint32_t>((k / S) & 1));
  }
}

// ------------------------------------------------------------------------------------------------
// Log-sum-exp merge of the segments of split units. One CTA per unit (b, h).
// ------------------------------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(128) decode_reduce_kernel(DecodeArgs a) {
  const int64_t u = blockIdx.x;
  const int32_t b = static_cast<int32_t>(u / a.Hkv);
  const int32_t h = static_cast<int32_t>(u - static_cast<int64_t>(b) * a.Hkv);
  int64_t first_slot, n_parts;
  int32_t first_kind = 0;
  if (a.part_chunks == 0) {
    const int32_t d0 = a.ws_desc[2 * u];
    if (d0 < 0) return;
    first_slot = d0 >> 1;          // warp id of the first segment
    first_kind = d0 & 1;
    const int32_t w_last = a.ws_desc[2 * u + 1];
    if (w_last < first_slot || w_last >= a.total_warps) {   // never written by a finished decode
      if (threadIdx.x == 0) record_error(ERRBIT_BOUNDS);
      return;
    }
    n_parts = w_last - first_slot + 1;
  } else {
    const int32_t nch = (clamped_len(a, b) + kChunk - 1) / kChunk;
    n_parts = (nch + a.part_chunks - 1) / a.part_chunks;
    if (n_parts <= 1) return;
    if (n_parts > a.max_parts) {
      if (threadIdx.x == 0) record_error(ERRBIT_BOUNDS);
      return;
    }
    first_slot = u * a.max_parts;
  }
  auto slot_of = [&](int64_t k) -> int64_t {
    if (a.part_chunks != 0) return first_slot + k;
    return 2 * (first_slot + k) + (k == 0 ? first_kind : 0);
  };
  for (int idx = threadIdx.x; idx < G * D / 4; idx += blockDim.x) {
    const int j = idx / (D / 4);
    const int d4 = idx - j * (D / 4);
    float M = -INFINITY;
    for (int64_t k = 0; k < n_parts; ++k) M = fmaxf(M, a.ws_ml[(slot_of(k) * G + j) * 2]);
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t k = 0; k < n_parts; ++k) {
      const int64_t s = slot_of(k);
      const float wk = a.ws_ml[(s * G + j) * 2 + 1] * exp2f(a.ws_ml[(s * G + j) * 2] - M);
      const float4 o = reinterpret_cast<const float4*>(a.ws_o + (s * G + j) * D)[d4];
      acc.x = fmaf(wk, o.x, acc.x);
      acc.y = fmaf(wk, o.y, acc.y);
      acc.z = fmaf(wk, o.z, acc.z);
      acc.w = fmaf(wk, o.w, acc.w);
      wsum += wk;
    }
    const float inv = 1.f / wsum;
    reinterpret_cast<float4*>(a.out + (static_cast<int64_t>(b) * a.Hq + h * G + j) * D)[d4] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
}

}  // namespace pkv_dev
