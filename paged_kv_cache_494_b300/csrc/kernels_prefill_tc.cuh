// Paged prefill / multi-token append attention (causal) on the 5th-generation tensor cores:
// tcgen05.mma with operands in shared memory (filled by TMA) and accumulators in tensor memory.
//
// What is computed is exactly what kernels_prefill.cuh computes (the attention of "Servicio de
// modelos de lenguaje con un presupuesto de memoria" §6 for the prefill phase named in "¿Cuánta
// memoria reservar para la caché KV?", "Verificar una carga representativa por etapas"): query i of
// sequence b sits at position p = len_b - q_len_b + i and attends causally to [0, p] (or the last
// `window` positions) through the block table.
//
// Decomposition (B300 design):
//  * One CTA per 128-row tile of one KV head: row r = (query token r / G, query head r % G of the
//    GQA group), 128 / G query tokens per CTA, so every staged K/V byte feeds 128 rows. Tiles of a
//    sequence are dispatched from its last (longest causal range) to its first.
//  * 6 warps. Warp 4 (one lane) issues TMA copies: the Q tile once (3-D tensor map over
//    [token][head][dim], 128-byte swizzle), then 32-key K and V tiles through a ring of 3 stages,
//    16 keys (one block piece) per copy, chunks outside the causal range filled with zeros by
//    out-of-range coordinates. Warp 5 allocates tensor memory and one lane issues the MMAs.
//    Warps 0-3 own one row each per thread (tensor-memory lane = row): softmax and the epilogue.
//  * Per 32-key tile j: S_j = Q K_j^T (M 128, N 32, K = D; into one of two S buffers in tensor
//    memory, so S_{j+1} is computed while S_j is in softmax); the softmax threads load their row of
//    S_j, apply the causal / window mask and the running max (raised only when a tile exceeds it by
//    2^8, so rescales of O are rare), and write P_j to shared memory as bf16 hi and the bf16 rounding
//    of the remainder lo, side by side in one 128-byte row ([hi keys 0..31][lo keys 0..31]); then
//    O += P V_j is one MMA chain over K = 64 (hi against V, then lo against the same V), so P keeps
//    ~17 bits and the O accumulator (f32, tensor memory) sees the exact-attention weights.
//  * Every wait is bounded (pkv_device.cuh); a role that gives up sets a shared abort flag, every
//    role stops, the producer waits for its copies in flight, the MMA lane for its MMAs, and the
//    tensor memory is freed before the CTA leaves.
#pragma once

#include "kernels_prefill.cuh"
#include "umma_desc.hpp"

namespace pkv_dev {

constexpr int kTcRows = 128;   // M of every MMA: rows of one CTA
constexpr int kTcKeys = 32;    // keys per tile: N of S = Q K^T, half the K of O += P V
constexpr int kTcStages = 3;   // K/V ring depth
constexpr int kTcThreads = 192;

template <int D, int G>
struct TcShape {
  static constexpr int TQ = kTcRows / G;            // query tokens per CTA
  static constexpr int ROWS = TQ * G;               // real rows (128 or slightly fewer)
  static constexpr int DH = D / 64;                 // 128-byte halves of a D-wide row
  static constexpr int Q_REGION = kTcRows * 128;    // one D half of the Q tile (16 KB)
  static constexpr int Q_BYTES = DH * Q_REGION;
  static constexpr int KV_REGION = kTcKeys * 128;   // one D half of a K (or V) tile (4 KB)
  static constexpr int K_BYTES = DH * KV_REGION;
  static constexpr int STAGE_BYTES = 2 * K_BYTES;   // K tile, then V tile
  static constexpr int P_BYTES = kTcRows * 128;     // [row][hi keys 0..31 | lo keys 0..31] bf16
  static constexpr int S_COL = D;                   // tensor-memory columns: O at 0..D-1, S at D, D+32
  static constexpr uint32_t TMEM_COLS = (D + 2 * kTcKeys) <= 128 ? 128u : 256u;
  static constexpr int KSTEPS = D / 16;             // k-steps of S = Q K^T
  static constexpr int RING_OFF = Q_BYTES;
  static constexpr int P_OFF = RING_OFF + kTcStages * STAGE_BYTES;
  static constexpr int BAR_OFF = P_OFF + P_BYTES;
  static constexpr int N_BARS = 1 + 2 * kTcStages + 2 + 2 + 1 + 1 + 1;
  static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;   // tmem base, abort flag, scan scratch, prefix
  static_assert(D == 64 || D == 128, "D");
  static_assert(G >= 1 && G <= 8, "G");
};

// [1 KB alignment slack][Q][ring][P][barriers][tmem base, abort][64-int scan scratch][tile prefix]
template <int D, int G>
__host__ __device__ inline size_t prefill_tc_smem_bytes(int n_seqs) {
  return 1024 + TcShape<D, G>::MISC_OFF + 16 + 256 + static_cast<size_t>(n_seqs + 1) * 4;
}

// ---- tcgen05 primitives (one instruction each; syntax of the PTX ISA) ----------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// The mbarrier gets one arrival once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16 in, f32 accumulate), shapes from the descriptor.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 consecutive f32 columns of this thread's tensor-memory lane (warp w reads lanes 32(w%4)..+31).
// The wait for the load is part of the same statement, so no use of the registers can be scheduled
// before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 3-D tiled TMA load (coordinates innermost first), completion on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            int32_t z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Tensor maps of one prefill call: K and V caches as 2-D [rows = NB*Hkv*B][D] (boxes 16 x 64, 128-byte
// swizzle) and q as 3-D [total_q][Hq][D] (boxes of (128 / G) tokens x G heads x 64 dims, 128-byte
// swizzle).
struct TcMaps {
  CUtensorMap k;
  CUtensorMap v;
  CUtensorMap q;
};

template <int D, int G>
__global__ void __launch_bounds__(kTcThreads, 2) paged_prefill_tc_kernel(const __grid_constant__ PrefillArgs a,
                                                                        const __grid_constant__ TcMaps maps) {
  using Sh = TcShape<D, G>;
  constexpr int TQ = Sh::TQ, ROWS = Sh::ROWS, DH = Sh::DH;
  constexpr float kRescaleLog2 = 8.f;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t n = a.n_seqs;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t q_s = sbase, ring_s = sbase + Sh::RING_OFF, p_s = sbase + Sh::P_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + kTcStages;
  uint64_t* s_full = kv_empty + kTcStages;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* drain = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Sh::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Sh::MISC_OFF + 4);
  int32_t* wsum = reinterpret_cast<int32_t*>(smem + Sh::MISC_OFF + 16);
  int32_t* tpref = wsum + 64;

  pdl_wait();   // before any global access, and before holding tensor memory

  // ---- query-tile prefix over sequences (block-wide scan)
  {
    const int nw = kTcThreads / 32;
    int32_t carry = 0;
    for (int32_t base = 0; base < n; base += kTcThreads) {
      const int32_t b = base + tid;
      int32_t c = 0;
      if (b < n) {
        int32_t ql = __ldg(a.cu_q + b + 1) - __ldg(a.cu_q + b);
        if (ql < 0) {
          record_error(ERRBIT_BOUNDS);
          ql = 0;
        }
        c = (ql + TQ - 1) / TQ;
      }
      int32_t ic = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, ic, off);
        if (lane >= off) ic += t;
      }
      if (lane == 31) wsum[warp] = ic;
      __syncthreads();
      int32_t pc = 0, tc = 0;
      for (int w2 = 0; w2 < nw; ++w2) {
        if (w2 < warp) pc += wsum[w2];
        tc += wsum[w2];
      }
      if (b < n) tpref[b] = carry + pc + ic - c;
      carry += tc;
      __syncthreads();
    }
    if (tid == 0) tpref[n] = carry;
    __syncthreads();
  }
  const int32_t tile = blockIdx.x;
  if (tile >= tpref[n]) {
    pdl_launch_dependents();
    return;
  }
  int32_t b = 0;
  {
    int32_t lo = 0, hi = n - 1;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if (tpref[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  const int32_t h = blockIdx.y;
  const int32_t n_qt = tpref[b + 1] - tpref[b];
  const int32_t qt = n_qt - 1 - (tile - tpref[b]);          // longest causal ranges first
  int32_t len = __ldg(a.context_lens + b);
  const int32_t cap = a.MB * a.B;
  if (len < 0 || len > cap) {
    if (tid == 0) record_error(ERRBIT_BOUNDS);
    len = len < 0 ? 0 : cap;
  }
  const int32_t q0 = __ldg(a.cu_q + b);
  int32_t ql = __ldg(a.cu_q + b + 1) - q0;
  if (ql > len) {
    if (tid == 0) record_error(ERRBIT_BOUNDS);
    ql = len;
  }
  const int32_t t_begin = qt * TQ;
  const int32_t t_end = min(t_begin + TQ, ql);
  if (t_begin >= t_end) {
    pdl_launch_dependents();
    return;
  }
  const int32_t pos0 = len - ql;
  const int32_t p_lo = pos0 + t_begin, p_hi = pos0 + t_end - 1;
  const int32_t c_lo = (a.window > 0 && p_lo - a.window + 1 > 0) ? (p_lo - a.window + 1) / kChunk : 0;
  const int32_t c_hi = p_hi / kChunk;
  const int32_t kt_lo = c_lo / 2, kt_hi = c_hi / 2;          // 32-key tiles = 2 chunks of 16
  const int32_t n_tiles = kt_hi - kt_lo + 1;
  const int32_t ws_max = a.window > 0 ? p_hi - a.window + 1 : 0;   // latest window start in the CTA

  // ---- barriers, tensor memory, padding rows of Q
  if (tid == 32 * 4) {
    mbar_init(smem_addr(q_full), 1);
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(smem_addr(kv_full + s), 1);
      mbar_init(smem_addr(kv_empty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(s_full + s), 1);
      mbar_init(smem_addr(s_free + s), 4);
    }
    mbar_init(smem_addr(p_full), 4);
    mbar_init(smem_addr(pv_done), 1);
    mbar_init(smem_addr(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_addr(tmem_slot), Sh::TMEM_COLS);
    tmem_relinquish();
  }
  if constexpr (ROWS < kTcRows) {   // rows the Q copy does not write: zeros (their results are dropped)
    for (int i = tid; i < (kTcRows - ROWS) * 8 * DH; i += kTcThreads) {
      const int dh = i / ((kTcRows - ROWS) * 8), rem = i % ((kTcRows - ROWS) * 8);
      *reinterpret_cast<uint4*>(smem + dh * Sh::Q_REGION + (ROWS + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ================= producer: TMA copies (one lane) =================
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      mbar_arrive_expect_tx(smem_addr(q_full), DH * ROWS * 128);
#pragma unroll
      for (int dh = 0; dh < DH; ++dh)
        tma_load_3d(q_s + dh * Sh::Q_REGION, &maps.q, 64 * dh, h * G, q0 + t_begin, smem_addr(q_full));
      int32_t issued = 0;
      for (int32_t j = 0; j < n_tiles; ++j) {
        const int s = j % kTcStages;
        if (j >= kTcStages &&
            !mbar_wait_bounded(smem_addr(kv_empty + s), static_cast<uint32_t>(((j / kTcStages) - 1) & 1))) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        const uint32_t kst = ring_s + s * Sh::STAGE_BYTES, vst = kst + Sh::K_BYTES;
        const uint32_t bar = smem_addr(kv_full + s);
        mbar_arrive_expect_tx(bar, Sh::STAGE_BYTES);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int32_t ci = (kt_lo + j) * 2 + c;            // 16-key chunk of the sequence
          int32_t y = -kChunk;                               // fully out of range: zero fill
          if (ci >= c_lo && ci <= c_hi) {
            const int32_t tok0 = ci * kChunk;
            const int32_t pg = tok0 / a.B;
            const int32_t blk = __ldg(a.block_tables + static_cast<int64_t>(b) * a.MB + pg);
            if (blk >= 0 && blk < a.NB)
              y = static_cast<int32_t>((static_cast<int64_t>(blk) * a.Hkv + h) * a.B + (tok0 - pg * a.B));
            else
              record_error(ERRBIT_BOUNDS);
          }
#pragma unroll
          for (int dh = 0; dh < DH; ++dh) {
            tma_load_2d(kst + dh * Sh::KV_REGION + c * (kChunk * 128), &maps.k, 64 * dh, y, bar, policy);
            tma_load_2d(vst + dh * Sh::KV_REGION + c * (kChunk * 128), &maps.v, 64 * dh, y, bar, policy);
          }
        }
        issued = j + 1;
      }
      // drain: the last copy issued into each stage (and Q) has landed before the CTA may leave
      mbar_wait_bounded(smem_addr(q_full), 0u);
      for (int s = 0; s < kTcStages; ++s) {
        const int32_t cnt = issued > s ? (issued - 1 - s) / kTcStages + 1 : 0;   // copies into stage s
        if (cnt > 0) mbar_wait_bounded(smem_addr(kv_full + s), static_cast<uint32_t>((cnt - 1) & 1));
      }
    }
  } else if (warp == 5) {
    // ================= MMA issue (one lane) =================
    if (lane == 0) {
      constexpr uint32_t idesc_s = pkv_umma::idesc_bf16_f32(kTcRows, kTcKeys, false, false);
      constexpr uint32_t idesc_pv = pkv_umma::idesc_bf16_f32(kTcRows, D, false, true);
      static_assert(pkv_umma::valid_f16_shape(kTcRows, kTcKeys) && pkv_umma::valid_f16_shape(kTcRows, D), "shape");
      bool ok = mbar_wait_bounded(smem_addr(q_full), 0u);
      auto pv = [&](int32_t i) -> bool {   // O += P_i V_i
        if (!mbar_wait_bounded(smem_addr(p_full), static_cast<uint32_t>(i & 1))) return false;
        tc_fence_after();
        const uint32_t vst = ring_s + (i % kTcStages) * Sh::STAGE_BYTES + Sh::K_BYTES;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // keys 0-15, 16-31 of hi, then of lo
          const uint64_t ad = pkv_umma::smem_desc(p_s + kk * 32, 16, 1024, pkv_umma::kSwizzle128B);
          const uint64_t bd =
              pkv_umma::smem_desc(vst + (kk & 1) * (16 * 128), Sh::KV_REGION, 1024, pkv_umma::kSwizzle128B);
          umma_f16(tmem, ad, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_addr(kv_empty + (i % kTcStages)));
        tc_commit(smem_addr(pv_done));
        return true;
      };
      int32_t j = 0;
      for (; ok && j < n_tiles; ++j) {
        const int s = j % kTcStages, sb = j & 1;
        if (!mbar_wait_bounded(smem_addr(kv_full + s), static_cast<uint32_t>((j / kTcStages) & 1)) ||
            (j >= 2 && !mbar_wait_bounded(smem_addr(s_free + sb), static_cast<uint32_t>(((j >> 1) - 1) & 1))) ||
            *abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kst = ring_s + s * Sh::STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < Sh::KSTEPS; ++kk) {
          const uint32_t off = (kk >> 2), col = (kk & 3) * 32;
          const uint64_t ad = pkv_umma::smem_desc(q_s + off * Sh::Q_REGION + col, 16, 1024, pkv_umma::kSwizzle128B);
          const uint64_t bd = pkv_umma::smem_desc(kst + off * Sh::KV_REGION + col, 16, 1024, pkv_umma::kSwizzle128B);
          umma_f16(tmem + Sh::S_COL + kTcKeys * sb, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(smem_addr(s_full + sb));
        if (j >= 1 && !pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && !pv(n_tiles - 1)) ok = false;
      if (!ok) *abort_flag = 1;
      // every MMA issued has completed before tensor memory is read for the last time or freed
      tc_commit(smem_addr(drain));
      mbar_wait_bounded(smem_addr(drain), 0u);
    }
  } else {
    // ================= softmax and epilogue: thread tid owns row tid =================
    const int r = tid;
    const int32_t tok = min(t_begin + r / G, t_end - 1);      // padding rows repeat a real token
    const bool row_real = r < ROWS && t_begin + r / G < t_end;
    const int32_t p_r = pos0 + tok;
    const int32_t ws_r = a.window > 0 ? p_r - a.window + 1 : 0;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * warp) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int32_t j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      if (!mbar_wait_bounded(smem_addr(s_full + sb), static_cast<uint32_t>((j >> 1) & 1)) || *abort_flag) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[32];
      tmem_ld32(tmem + lane_addr + Sh::S_COL + kTcKeys * sb, s);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(s_free + sb));
      const int32_t kbase = (kt_lo + j) * kTcKeys;
      const bool full = kbase >= ws_max && kbase + kTcKeys - 1 <= p_lo;   // no key of the tile is masked
      float mx = -INFINITY;
      if (full) {
#pragma unroll
        for (int k = 0; k < 32; ++k) mx = fmaxf(mx, s[k]);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int32_t key = kbase + k;
          if (!(key <= p_r && key >= ws_r)) s[k] = -INFINITY;   // select, never multiply: s may be NaN
          mx = fmaxf(mx, s[k]);
        }
      }
      mx *= a.scale_log2;
      const bool raise = mx > m + kRescaleLog2;
      const float mnew = raise ? mx : m;
      const float alpha = raise ? exp2f(m - mnew) : 1.f;         // 0 while m is still -inf
      m = mnew;
      const float msafe = m == -INFINITY ? 0.f : m;               // a row with no key yet: weights 0
      float sum = 0.f;
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const float p0 = exp2f(fmaf(s[k], a.scale_log2, -msafe));
        const float p1 = exp2f(fmaf(s[k + 1], a.scale_log2, -msafe));
        sum += p0 + p1;
        const uint32_t hw = pack_bf16x2(p0, p1);
        hi[k / 2] = hw;
        lo[k / 2] = pack_bf16x2(p0 - bf16_lo(hw), p1 - bf16_hi(hw));
      }
      l = l * alpha + sum;
      // P_j may overwrite P_{j-1} and O may be rescaled only once O += P_{j-1} V_{j-1} has completed
      if (j > 0) {
        if (!mbar_wait_bounded(smem_addr(pv_done), static_cast<uint32_t>((j - 1) & 1))) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, raise)) {
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            float o[32];
            tmem_ld32(tmem + lane_addr + c, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= alpha;
            tmem_st32(tmem + lane_addr + c, o);
          }
          tmem_wait_st();
        }
      }
      // P row: 16-byte chunk c (c < 4: hi keys 8c..8c+7; c >= 4: lo keys 8(c-4)..) at c ^ (r & 7)
      unsigned char* prow = smem + Sh::P_OFF + r * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) =
            make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
        *reinterpret_cast<uint4*>(prow + (((c + 4) ^ (r & 7)) << 4)) =
            make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
      }
      // keys at or past the context end may hold anything (even NaN) in the staged V: zero them
      if (kbase + kTcKeys > len) {
        const int s = j % kTcStages;
        mbar_wait_bounded(smem_addr(kv_full + s), static_cast<uint32_t>((j / kTcStages) & 1));   // landed
        const int z0 = max(0, len - kbase);
        unsigned char* vst = smem + Sh::RING_OFF + s * Sh::STAGE_BYTES + Sh::K_BYTES;
        for (int i = tid; i < (kTcKeys - z0) * 8 * DH; i += 128) {
          const int dh = i / ((kTcKeys - z0) * 8), rem = i % ((kTcKeys - z0) * 8);
          *reinterpret_cast<uint4*>(vst + dh * Sh::KV_REGION + (z0 + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();   // generic-proxy writes of P (and V zeros) before the MMA reads them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(p_full));
    }
    // ---- epilogue: O / l for the real rows
    if (ok && !*abort_flag) {
      if (mbar_wait_bounded(smem_addr(pv_done), static_cast<uint32_t>((n_tiles - 1) & 1))) {
        tc_fence_after();
        const float inv = 1.f / l;
        float* dst = a.out + ((static_cast<int64_t>(q0) + tok) * a.Hq + h * G + (r % G)) * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tmem + lane_addr + c, o);
          if (row_real) {
#pragma unroll
            for (int k = 0; k < 32; k += 4)
              *reinterpret_cast<float4*>(dst + c + k) =
                  make_float4(o[k] * inv, o[k + 1] * inv, o[k + 2] * inv, o[k + 3] * inv);
          }
        }
      } else {
        *abort_flag = 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, Sh::TMEM_COLS);
  }
  pdl_launch_dependents();
}

}  // namespace pkv_dev
