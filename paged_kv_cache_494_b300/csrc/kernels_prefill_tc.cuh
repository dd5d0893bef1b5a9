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
//  * A Q tile is 128 rows of one KV head: row r = (query token r / G, query head r % G of the GQA
//    group), 128 / G query tokens. A work item is NT consecutive Q tiles of one (sequence, KV head)
//    (NT = 2: every staged K/V byte then feeds 256 rows, and the two tiles' softmax and MMA chains
//    interleave on the tensor core). The kernel is persistent, one CTA per SM: each CTA walks the
//    work items heaviest first (level-major: every sequence's last item, then the ones before), and
//    every role keeps its barrier phases running across items, so the next item's Q and K/V copies
//    and first S MMAs overlap the current item's last steps and epilogue.
//  * Warps 0 .. 4NT-1: softmax and epilogue, one row per thread (warp w serves tile w / 4, tensor-
//    memory lanes 32 (w % 4) ..). Warp 4NT issues TMA copies (one lane; the warp reads block-table
//    entries 32 at a time and hands them over by shuffle): the Q tiles once (3-D tensor map over
//    [token][head][dim], 128-byte swizzle), then 64-key K and V steps of the union of the tiles'
//    causal ranges through a ring of STAGES stages, 16 keys (one block piece) per copy, chunks
//    outside the range filled with zeros by out-of-range coordinates; the copies of a step are issued
//    by 16 lanes at once (a tensor copy costs ~100 cycles to issue). Per tile, one lane of one warp
//    issues the S MMAs and one lane of another the O += P V MMAs, so no chain waits on another's
//    inputs (a tcgen05.mma costs tens of cycles to issue). The first S warp allocates tensor memory.
//  * Per tile and 64-key step i: S_i = Q K_i^T (M 128, N 64, K = D) into one of two S buffers of the
//    tile in tensor memory, so S_{i+1} is computed while S_i is in softmax; the softmax threads load
//    their row of S_i, apply the causal / window mask and the running max (raised only when a step
//    exceeds it by 2^8, so rescales of O are rare), and write P_i back over S_i in tensor memory as
//    bf16 pairs: hi (keys 0..63, 32 columns) and the bf16 rounding of the remainder lo (the next 32
//    columns). O += P V_i is one MMA chain over K = 128 (hi against V, then lo against the same V)
//    with the A operand read from tensor memory, so P keeps ~17 bits and the O accumulator (f32,
//    tensor memory) sees the exact-attention weights; shared memory holds only Q and the K/V ring.
//  * Every wait is bounded (pkv_device.cuh); a role that gives up sets a shared abort flag, every
//    role stops, the producer waits for its copies in flight, the MMA lane for its MMAs, and the
//    tensor memory is freed before the CTA leaves.
#pragma once

#include "kernels_prefill.cuh"
#include "umma_desc.hpp"

namespace pkv_dev {

constexpr int kTcRows = 128;   // M of every MMA: rows of one Q tile
constexpr int kTcKeys = 64;    // keys per step: N of S = Q K^T, half the K of O += P V
constexpr int kTcChunks = kTcKeys / kChunk;   // 16-key block pieces per step

template <int D, int G, int NT, int STAGES>
struct TcShape {
  static constexpr int TQ = kTcRows / G;            // query tokens per Q tile
  static constexpr int ROWS = TQ * G;               // real rows (128 or slightly fewer)
  // warps: 4NT softmax, 1 producer, then per tile one S-issuing and one PV-issuing warp
  static constexpr int THREADS = 128 * NT + 32 * (1 + 2 * NT);
  static constexpr int PRODUCER = 4 * NT;
  static constexpr int MMA = 4 * NT + 1;            // S MMAs of tile 0 (warp MMA + t: tile t); allocates tensor memory
  static constexpr int MMA_PV = 4 * NT + 1 + NT;    // O += P V MMAs of tile 0 (MMA_PV + t: tile t)
  static constexpr int DH = D / 64;                 // 128-byte halves of a D-wide row
  static constexpr int Q_REGION = kTcRows * 128;    // one D half of a Q tile (16 KB)
  static constexpr int Q_TILE = DH * Q_REGION;
  static constexpr int KV_REGION = kTcKeys * 128;   // one D half of a K (or V) step (8 KB)
  static constexpr int K_BYTES = DH * KV_REGION;
  static constexpr int STAGE_BYTES = 2 * K_BYTES;   // K step, then V step
  static constexpr int TCOLS = D + 2 * kTcKeys;     // tensor-memory columns of a tile: O, then 2 S buffers
  static constexpr uint32_t TMEM_COLS = NT * TCOLS <= 128 ? 128u : NT * TCOLS <= 256 ? 256u : 512u;
  static constexpr int KSTEPS = D / 16;             // k-steps of S = Q K^T
  static constexpr int RING_OFF = NT * Q_TILE;
  static constexpr int BAR_OFF = RING_OFF + STAGES * STAGE_BYTES;
  // q_full, q_empty, kv_full/empty[STAGES], per tile: s_full[2], p_full[2], p_free[2], o_free; drain
  static constexpr int NTB = 7;                     // barriers per tile
  static constexpr int N_BARS = 2 + 2 * STAGES + NTB * NT + 1;
  static constexpr int SOFTMAX_THREADS = 128 * NT;
  // epilogue staging, per softmax warp: 32 rows x 16 floats (2 KB), 16-byte slots XOR-swizzled
  static constexpr int EPI_WARP_BYTES = 32 * 16 * 4;
  static constexpr int EPI_OFF = BAR_OFF + (N_BARS * 8 + 127) / 128 * 128;
  static constexpr int MISC_OFF = EPI_OFF + 4 * NT * EPI_WARP_BYTES;   // tmem base, abort flag, scan scratch, prefix
  static_assert(D == 64 || D == 128, "D");
  static_assert(G >= 1 && G <= 8, "G");
  static_assert(NT == 1 || NT == 2, "NT");
  static_assert(NT * TCOLS <= 512, "tensor memory");
};

// [1 KB alignment slack][Q tiles][ring][barriers][epilogue staging][tmem base, abort][64-int scan scratch][prefix]
template <class Sh>
__host__ __device__ inline size_t prefill_tc_smem_bytes(int n_seqs) {
  return 1024 + Sh::MISC_OFF + 16 + 256 + static_cast<size_t>(n_seqs + 1) * 4;
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
// D[tmem] (+)= A[tmem] * B[smem], kind::f16: A (M x K, 16-bit) in tensor memory, row m in lane m,
// elements k and k + 1 packed in one 32-bit column (K = 16 per instruction: 8 columns).
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
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
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
  tmem_st32(taddr, f);
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Packed pairs of f32 (sm_100 and later execute one instruction per pair): low half = first value.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

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

// One work item of the persistent loop: NT consecutive Q tiles of one (sequence, KV head).
struct TcItem {
  int32_t b, h, q0, len, pos0, t_begin, t_end, n_act, c_lo, c_hi, kt_lo, n_steps;
  int32_t fixed_pos;   // shared-prefix mode: the position of every row (shared_len - 1); else -1
  int32_t split;       // shared-prefix mode: key split of the item
};

template <int D, int G, int NT, int STAGES>
__global__ void __launch_bounds__(TcShape<D, G, NT, STAGES>::THREADS, 1)
    paged_prefill_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ TcMaps maps) {
  using Sh = TcShape<D, G, NT, STAGES>;
  constexpr int TQ = Sh::TQ, ROWS = Sh::ROWS, DH = Sh::DH, NTHR = Sh::THREADS, NTB = Sh::NTB;
  constexpr int ITEM = NT * TQ;             // query tokens per work item
  constexpr float kRescaleLog2 = 8.f;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t n = a.n_seqs;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t q_s = sbase, ring_s = sbase + Sh::RING_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::BAR_OFF);
  uint64_t* q_full = bars;                 // Q tiles of the current item landed
  uint64_t* q_empty = bars + 1;            // every S MMA of the previous item completed (Q may be reloaded)
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_empty = kv_full + STAGES;
  uint64_t* tbar = kv_empty + STAGES;      // per tile t, tbar + NTB t: s_full[2], p_full[2], p_free[2], o_free
  uint64_t* drain = tbar + NTB * NT;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Sh::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Sh::MISC_OFF + 4);
  int32_t* max_items = reinterpret_cast<int32_t*>(smem + Sh::MISC_OFF + 8);
  int32_t* wsum = reinterpret_cast<int32_t*>(smem + Sh::MISC_OFF + 16);
  int32_t* tpref = wsum + 64;

  set_error_word(a.err);
  pdl_wait();   // before any global access, and before holding tensor memory
  if (a.early_trigger) pdl_launch_dependents();
  if (a.task_ctr != nullptr && blockIdx.x == 0 && tid == 0) install_task_tag(a.task_ctr, a.task_tag);

  // ---- items per sequence (prefix over sequences) and the largest count; shared-prefix mode: one
  // virtual sequence whose queries are all total_q rows
  const bool shared = a.shared_len > 0;
  if (tid == 0) *max_items = 0;
  if (shared) {
    if (tid == 0) {
      tpref[0] = 0;
      tpref[1] = (a.total_q + ITEM - 1) / ITEM;
      *max_items = tpref[1];
    }
    __syncthreads();
  } else {
    constexpr int nw = NTHR / 32;
    int32_t carry = 0;
    for (int32_t base = 0; base < n; base += NTHR) {
      const int32_t b = base + tid;
      int32_t c = 0;
      if (b < n) {
        int32_t ql = __ldg(a.cu_q + b + 1) - __ldg(a.cu_q + b);
        if (ql < 0) {
          record_error(ERRBIT_BOUNDS);
          ql = 0;
        }
        c = (ql + ITEM - 1) / ITEM;
      }
      int32_t ic = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, ic, off);
        if (lane >= off) ic += t;
      }
      if (lane == 31) wsum[warp] = ic;
      __syncthreads();
      if (c > 0) atomicMax(max_items, c);
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
  // Work slots, heaviest first: slot x = (level L, sequence b, KV head h), level-major; level L of
  // sequence b is its item counted from the end (the longest causal range first). CTA c takes slots
  // c, c + gridDim.x, ...; slots past a sequence's item count are empty.
  const int64_t per_level = shared ? static_cast<int64_t>(*max_items) * a.Hkv : static_cast<int64_t>(n) * a.Hkv;
  const int32_t n_split = shared ? (a.shared_len + a.split_keys - 1) / a.split_keys : 1;
  const int64_t n_slots = shared ? static_cast<int64_t>(n_split) * per_level : static_cast<int64_t>(*max_items) * per_level;
  if (static_cast<int64_t>(blockIdx.x) >= n_slots) {
    pdl_launch_dependents();
    return;
  }
  auto get_item = [&](int64_t x, TcItem& it) -> bool {
    if (shared) {   // slot = (split, item, KV head): every item of a split has the same key range
      it.split = static_cast<int32_t>(x / per_level);
      const int64_t r2 = x - static_cast<int64_t>(it.split) * per_level;
      const int32_t item = static_cast<int32_t>(r2 / a.Hkv);
      it.h = static_cast<int32_t>(r2 - static_cast<int64_t>(item) * a.Hkv);
      it.b = 0;
      it.q0 = 0;
      it.len = a.shared_len;
      it.pos0 = 0;
      it.fixed_pos = a.shared_len - 1;
      it.t_begin = item * ITEM;
      it.t_end = min(it.t_begin + ITEM, a.total_q);
      it.n_act = (it.t_end - it.t_begin + TQ - 1) / TQ;
      const int32_t k0 = it.split * a.split_keys, k1 = min(k0 + a.split_keys, a.shared_len);
      it.c_lo = k0 / kChunk;
      it.c_hi = (k1 - 1) / kChunk;
      it.kt_lo = it.c_lo / kTcChunks;
      it.n_steps = it.c_hi / kTcChunks - it.kt_lo + 1;
      return true;
    }
    it.fixed_pos = -1;
    it.split = 0;
    const int32_t L = static_cast<int32_t>(x / per_level);
    const int64_t r = x - static_cast<int64_t>(L) * per_level;
    it.b = static_cast<int32_t>(r / a.Hkv);
    it.h = static_cast<int32_t>(r - static_cast<int64_t>(it.b) * a.Hkv);
    const int32_t nb = tpref[it.b + 1] - tpref[it.b];
    if (L >= nb) return false;
    const int32_t qt = nb - 1 - L;
    int32_t len = __ldg(a.context_lens + it.b);
    const int32_t cap = a.MB * a.B;
    if (len < 0 || len > cap) {
      if (tid == 0) record_error(ERRBIT_BOUNDS);
      len = len < 0 ? 0 : cap;
    }
    it.q0 = __ldg(a.cu_q + it.b);
    int32_t ql = __ldg(a.cu_q + it.b + 1) - it.q0;
    if (ql > len) {
      if (tid == 0) record_error(ERRBIT_BOUNDS);
      ql = len;
    }
    it.len = len;
    it.t_begin = qt * ITEM;
    it.t_end = min(it.t_begin + ITEM, ql);
    if (it.t_begin >= it.t_end) return false;
    it.pos0 = len - ql;
    it.n_act = (it.t_end - it.t_begin + TQ - 1) / TQ;
    const int32_t p_first = it.pos0 + it.t_begin;
    it.c_lo = (a.window > 0 && p_first - a.window + 1 > 0) ? (p_first - a.window + 1) / kChunk : 0;
    it.c_hi = (it.pos0 + it.t_end - 1) / kChunk;
    it.kt_lo = it.c_lo / kTcChunks;
    it.n_steps = it.c_hi / kTcChunks - it.kt_lo + 1;
    return true;
  };
  auto tile_first_tok = [&](const TcItem& it, int t) { return it.t_begin + t * TQ; };
  auto tile_last_tok = [&](const TcItem& it, int t) { return min(it.t_begin + (t + 1) * TQ, it.t_end) - 1; };
  // step range of tile t within the item's ring steps: [off, off + cnt)
  auto tile_off = [&](const TcItem& it, int t) -> int32_t {
    if (it.fixed_pos >= 0) return 0;
    const int32_t p = it.pos0 + tile_first_tok(it, t);
    const int32_t c = (a.window > 0 && p - a.window + 1 > 0) ? (p - a.window + 1) / kChunk : 0;
    return c / kTcChunks - it.kt_lo;
  };
  auto tile_cnt = [&](const TcItem& it, int t) -> int32_t {
    if (it.fixed_pos >= 0) return it.n_steps;
    return (it.pos0 + tile_last_tok(it, t)) / kChunk / kTcChunks - it.kt_lo - tile_off(it, t) + 1;
  };

  // ---- barriers, tensor memory, padding rows of Q
  if (tid == 32 * Sh::PRODUCER) {
    mbar_init(smem_addr(q_full), 1);
    mbar_init(smem_addr(q_empty), NT);      // one commit from each S-issuing lane per item
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(kv_full + s), 1);
      mbar_init(smem_addr(kv_empty + s), NT);   // one arrival per PV-issuing lane per step
    }
    for (int t = 0; t < NT; ++t) {
      uint64_t* tb = tbar + NTB * t;
      mbar_init(smem_addr(tb + 0), 1);   // s_full[0..1]: one commit (S of the buffer is ready)
      mbar_init(smem_addr(tb + 1), 1);
      mbar_init(smem_addr(tb + 2), 4);   // p_full[0..1]: one arrival per softmax warp (P written)
      mbar_init(smem_addr(tb + 3), 4);
      mbar_init(smem_addr(tb + 4), 1);   // p_free[0..1]: one commit per O += P V reading the buffer
      mbar_init(smem_addr(tb + 5), 1);   //   (it completes once that MMA and every earlier one of the lane has)
      mbar_init(smem_addr(tb + 6), 4);   // o_free: one arrival per softmax warp per item (O read out)
    }
    mbar_init(smem_addr(drain), 2 * NT);   // one commit from each MMA-issuing lane
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == Sh::MMA) {
    tmem_alloc(smem_addr(tmem_slot), Sh::TMEM_COLS);
    tmem_relinquish();
  }
  if constexpr (ROWS < kTcRows) {   // rows the Q copies never write: zeros (their results are dropped)
    constexpr int PER = (kTcRows - ROWS) * 8;   // 16-byte pieces per D half
    for (int i = tid; i < NT * DH * PER; i += NTHR) {
      const int reg = i / PER, rem = i % PER;   // reg = tile * DH + dh
      *reinterpret_cast<uint4*>(smem + reg * Sh::Q_REGION + (ROWS + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == Sh::PRODUCER) {
    // ================= producer: TMA copies (lane 0 waits; the warp reads the block table) ==========
    const uint64_t policy = policy_evict_first();
    constexpr int BOXES = kTcChunks * 2 * DH;           // copies of one step: chunk x (K, V) x D half
    const int my_c = lane / (2 * DH), my_kv = (lane / DH) & 1, my_dh = lane % DH;   // lane < BOXES
    int32_t J = 0, k = 0;                               // ring steps and items of this CTA so far
    bool stop = false;
    for (int64_t x = blockIdx.x; !stop && x < n_slots; x += gridDim.x) {
      TcItem it;
      if (!get_item(x, it)) continue;
      int st = 0;
      if (lane == 0) {   // Q of this item once every S MMA of the previous item has completed
        if (k > 0 && !mbar_wait_bounded(smem_addr(q_empty), static_cast<uint32_t>((k - 1) & 1))) *abort_flag = 1;
        st = *abort_flag;
        if (!st) mbar_arrive_expect_tx(smem_addr(q_full), it.n_act * DH * ROWS * 128);
      }
      if (__shfl_sync(0xffffffffu, st, 0)) break;
      __syncwarp();
      if (lane < it.n_act * DH) {   // one Q box per lane: tile lane / DH, D half lane % DH
        const int t = lane / DH, dh = lane % DH;
        tma_load_3d(q_s + (t * DH + dh) * Sh::Q_REGION, &maps.q, 64 * dh, it.h * G,
                    it.q0 + tile_first_tok(it, t), smem_addr(q_full));
      }
      ++k;
      const int32_t* table = a.block_tables + static_cast<int64_t>(it.b) * a.MB;
      int32_t win_base = -1 << 30, win_val = -1;
      for (int32_t j = 0; j < it.n_steps; ++j, ++J) {
        const int s = J % STAGES;
        if (lane == 0) {
          if (J >= STAGES &&
              !mbar_wait_bounded(smem_addr(kv_empty + s), static_cast<uint32_t>(((J / STAGES) - 1) & 1)))
            *abort_flag = 1;
          st = *abort_flag;
        }
        if (__shfl_sync(0xffffffffu, st, 0)) {
          stop = true;
          break;
        }
        const uint32_t bar = smem_addr(kv_full + s);
        // block-table entries of the step's chunks: window of 32 pages, one per lane
        const int32_t pg0 = (it.kt_lo + j) * kTcKeys / a.B;
        const int32_t pg_last = ((it.kt_lo + j) * kTcKeys + kTcKeys - 1) / a.B;
        if (pg0 < win_base || pg_last >= win_base + 32) {
          win_base = pg0;
          win_val = pg0 + lane < a.MB ? __ldg(table + pg0 + lane) : -1;
        }
        const int32_t ci = (it.kt_lo + j) * kTcChunks + my_c;   // this lane's 16-key chunk
        const int32_t pg = ci * kChunk / a.B;
        const int32_t blk = __shfl_sync(0xffffffffu, win_val, min(max(pg - win_base, 0), 31));
        if (lane == 0) mbar_arrive_expect_tx(bar, Sh::STAGE_BYTES);
        __syncwarp();
        if (lane < BOXES) {
          int32_t y = -kChunk;                                  // fully out of range: zero fill
          if (ci >= it.c_lo && ci <= it.c_hi) {
            if (blk >= 0 && blk < a.NB)
              y = static_cast<int32_t>((static_cast<int64_t>(blk) * a.Hkv + it.h) * a.B + (ci * kChunk - pg * a.B));
            else if (my_kv == 0 && my_dh == 0)
              record_error(ERRBIT_BOUNDS);
          }
          const uint32_t dst = ring_s + s * Sh::STAGE_BYTES + my_kv * Sh::K_BYTES + my_dh * Sh::KV_REGION +
                               my_c * (kChunk * 128);
          tma_load_2d(dst, my_kv ? &maps.v : &maps.k, 64 * my_dh, y, bar, policy);
        }
      }
    }
    if (lane == 0) {
      // drain: the last Q and the last copy issued into each stage have landed before the CTA may leave
      if (k > 0) mbar_wait_bounded(smem_addr(q_full), static_cast<uint32_t>((k - 1) & 1));
      for (int s = 0; s < STAGES; ++s) {
        const int32_t c = J > s ? (J - 1 - s) / STAGES + 1 : 0;   // copies into stage s
        if (c > 0) mbar_wait_bounded(smem_addr(kv_full + s), static_cast<uint32_t>((c - 1) & 1));
      }
    }
  } else if (warp >= Sh::MMA) {
    // ================= MMA issue: S of tile t on warp MMA + t, O += P V on warp MMA_PV + t =========
    if (lane == 0) {
      constexpr uint32_t idesc_s = pkv_umma::idesc_bf16_f32(kTcRows, kTcKeys, false, false);
      constexpr uint32_t idesc_pv = pkv_umma::idesc_bf16_f32(kTcRows, D, false, true);
      static_assert(pkv_umma::valid_f16_shape(kTcRows, kTcKeys) && pkv_umma::valid_f16_shape(kTcRows, D), "shape");
      const bool is_s = warp < Sh::MMA_PV;
      const int t = is_s ? warp - Sh::MMA : warp - Sh::MMA_PV;
      uint64_t* tb = tbar + NTB * t;
      const uint32_t qt_s = q_s + t * Sh::Q_TILE;
      bool ok = true;
      int32_t J0 = 0, I = 0, k = 0;   // ring steps before this item, steps of tile t, items so far
      for (int64_t x = blockIdx.x; ok && x < n_slots; x += gridDim.x) {
        TcItem it;
        if (!get_item(x, it)) continue;
        const bool act = t < it.n_act;
        const int32_t off = act ? tile_off(it, t) : 0, cnt = act ? tile_cnt(it, t) : 0;
        if (is_s) {
          if (!mbar_wait_bounded(smem_addr(q_full), static_cast<uint32_t>(k & 1)) || *abort_flag) {
            ok = false;
            break;
          }
          for (int32_t i = 0; i < cnt; ++i, ++I) {   // S of the tile's step i (ring step J0 + off + i)
            const int32_t J = J0 + off + i;
            const int sb = I & 1;
            if (!mbar_wait_bounded(smem_addr(kv_full + J % STAGES), static_cast<uint32_t>((J / STAGES) & 1)) ||
                (I >= 2 && !mbar_wait_bounded(smem_addr(tb + 4 + sb), static_cast<uint32_t>(((I >> 1) - 1) & 1))) ||
                *abort_flag) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t kst = ring_s + (J % STAGES) * Sh::STAGE_BYTES;
#pragma unroll
            for (int kk = 0; kk < Sh::KSTEPS; ++kk) {
              const uint32_t dh = (kk >> 2), col = (kk & 3) * 32;
              const uint64_t ad =
                  pkv_umma::smem_desc(qt_s + dh * Sh::Q_REGION + col, 16, 1024, pkv_umma::kSwizzle128B);
              const uint64_t bd =
                  pkv_umma::smem_desc(kst + dh * Sh::KV_REGION + col, 16, 1024, pkv_umma::kSwizzle128B);
              umma_f16(tmem + t * Sh::TCOLS + D + kTcKeys * sb, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(smem_addr(tb + sb));
          }
          if (!ok) break;
          tc_commit(smem_addr(q_empty));   // Q of this item is no longer read once these S MMAs complete
        } else {
          // every ring step of the item gets one arrival from this lane on kv_empty: after its MMAs when
          // the tile uses the step, otherwise a plain arrival once the stage's previous phase is over
          for (int32_t j = 0; ok && j < it.n_steps; ++j) {
            const int32_t J = J0 + j, i = j - off;
            if (i >= 0 && i < cnt) {
              const int sb = I & 1;
              if (!mbar_wait_bounded(smem_addr(tb + 2 + sb), static_cast<uint32_t>((I >> 1) & 1)) ||
                  (i == 0 && k > 0 && !mbar_wait_bounded(smem_addr(tb + 6), static_cast<uint32_t>((k - 1) & 1))) ||
                  *abort_flag) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t vst = ring_s + (J % STAGES) * Sh::STAGE_BYTES + Sh::K_BYTES;
              const uint32_t pt = tmem + t * Sh::TCOLS + D + kTcKeys * sb;   // P of buffer sb (lane 0)
#pragma unroll
              for (int kk = 0; kk < 2 * kTcKeys / 16; ++kk) {   // keys 16q..16q+15 of hi (kk < 4), then of lo
                const int q = kk & 3;
                const uint64_t bd =
                    pkv_umma::smem_desc(vst + q * (16 * 128), Sh::KV_REGION, 1024, pkv_umma::kSwizzle128B);
                umma_f16_ta(tmem + t * Sh::TCOLS, pt + kk * 8, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
              }
              tc_commit(smem_addr(tb + 4 + sb));
              tc_commit(smem_addr(kv_empty + J % STAGES));
              ++I;
            } else {
              if (J >= STAGES &&
                  !mbar_wait_bounded(smem_addr(kv_empty + J % STAGES), static_cast<uint32_t>(((J / STAGES) - 1) & 1))) {
                ok = false;
                break;
              }
              mbar_arrive(smem_addr(kv_empty + J % STAGES));
            }
          }
        }
        J0 += it.n_steps;
        ++k;
      }
      if (!ok) *abort_flag = 1;
      // every MMA this lane issued has completed before tensor memory is read for the last time or freed
      tc_commit(smem_addr(drain));
      mbar_wait_bounded(smem_addr(drain), 0u);
    }
  } else {
    // ================= softmax and epilogue: thread owns row r of tile t =================
    const int t = warp >> 2, r = tid & 127;
    uint64_t* tb = tbar + NTB * t;
    const uint32_t tm = tmem + t * Sh::TCOLS + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    int32_t J0 = 0, I = 0;   // ring steps before this item, steps of tile t so far
    bool ok = true;
    for (int64_t x = blockIdx.x; ok && x < n_slots; x += gridDim.x) {
      TcItem it;
      if (!get_item(x, it)) continue;
      const bool active = t < it.n_act;
      if (active) {
        const int32_t first = tile_first_tok(it, t), last = tile_last_tok(it, t);
        const int32_t tok = min(first + r / G, last);               // padding rows repeat a real token
        const bool row_real = r < ROWS && first + r / G <= last;
        const int32_t p_r = it.fixed_pos >= 0 ? it.fixed_pos : it.pos0 + tok;
        const int32_t ws_r = a.window > 0 ? p_r - a.window + 1 : 0;
        const int32_t p_min = it.fixed_pos >= 0 ? it.fixed_pos : it.pos0 + first;   // smallest position of the tile
        const int32_t ws_max = a.window > 0 ? it.pos0 + last - a.window + 1 : 0;
        const int32_t t_off = tile_off(it, t), t_cnt = tile_cnt(it, t);
        float m = -INFINITY, l = 0.f;
        for (int32_t i = 0; i < t_cnt; ++i, ++I) {
          const int sb = I & 1;
          if (!mbar_wait_bounded(smem_addr(tb + sb), static_cast<uint32_t>((I >> 1) & 1)) || *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          float s[kTcKeys];
          {
            float h0[32], h1[32];
            tmem_ld32(tm + D + kTcKeys * sb, h0);
            tmem_ld32(tm + D + kTcKeys * sb + 32, h1);
#pragma unroll
            for (int k2 = 0; k2 < 32; ++k2) {
              s[k2] = h0[k2];
              s[32 + k2] = h1[k2];
            }
          }
          const int32_t step = t_off + i;                            // step index within the item
          const int32_t kbase = (it.kt_lo + step) * kTcKeys;
          const bool full = kbase >= ws_max && kbase + kTcKeys - 1 <= p_min;   // no key of the step is masked
          if (!full) {
#pragma unroll
            for (int k2 = 0; k2 < kTcKeys; ++k2) {
              const int32_t key = kbase + k2;
              if (!(key <= p_r && key >= ws_r)) s[k2] = -INFINITY;   // select, never multiply: s may be NaN
            }
          }
          // row maximum as a tree (short dependency chains)
          float mt[kTcKeys / 2];
#pragma unroll
          for (int k2 = 0; k2 < kTcKeys / 2; ++k2) mt[k2] = fmaxf(s[2 * k2], s[2 * k2 + 1]);
#pragma unroll
          for (int w = kTcKeys / 4; w >= 1; w >>= 1)
#pragma unroll
            for (int k2 = 0; k2 < w; ++k2) mt[k2] = fmaxf(mt[k2], mt[k2 + w]);
          const float mx = mt[0] * a.scale_log2;
          const bool raise = mx > m + kRescaleLog2;
          const float mnew = raise ? mx : m;
          const float alpha = raise ? exp2f(m - mnew) : 1.f;         // 0 while m is still -inf
          m = mnew;
          const float msafe = m == -INFINITY ? 0.f : m;               // a row with no key yet: weights 0
          // p = 2^(s * scale_log2 - m) in pairs; hi = bf16(p), lo = bf16(p - hi); sum in 4 packed partials
          uint32_t hi[kTcKeys / 2], lo[kTcKeys / 2];
          unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
          const unsigned long long c2 = f2_pack(a.scale_log2, a.scale_log2), nm2 = f2_pack(-msafe, -msafe);
#pragma unroll
          for (int k2 = 0; k2 < kTcKeys; k2 += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[k2], s[k2 + 1]), c2, nm2), x0, x1);
            const float p0 = exp2f(x0), p1 = exp2f(x1);
            const unsigned long long pp = f2_pack(p0, p1);
            acc[(k2 >> 1) & 3] = f2_add(acc[(k2 >> 1) & 3], pp);
            const uint32_t hw = pack_bf16x2(p0, p1);
            hi[k2 / 2] = hw;
            float r0, r1;
            f2_unpack(f2_sub(pp, f2_pack(bf16_lo(hw), bf16_hi(hw))), r0, r1);
            lo[k2 / 2] = pack_bf16x2(r0, r1);
          }
          float sa, sb2;
          f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), sa, sb2);
          l = l * alpha + (sa + sb2);
          // O may be rescaled only once O += P V of the tile's previous step (I - 1) has completed: the
          // buffer of that step sees its ((I - 1) >> 1)-th completion then. A parity wait tells only the
          // current phase from the previous one, so it is made on a barrier known to be within one
          // phase of the target: the use of the buffer before (step I - 3) completed before S of step
          // I - 1 was issued, and its next use (step I + 1) cannot complete before P of step I exists.
          if (i > 0 && __any_sync(0xffffffffu, raise)) {
            if (!mbar_wait_bounded(smem_addr(tb + 4 + ((I - 1) & 1)), static_cast<uint32_t>(((I - 1) >> 1) & 1))) {
              ok = false;
              *abort_flag = 1;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              float o[32];
              tmem_ld32(tm + c, o);
#pragma unroll
              for (int k2 = 0; k2 < 32; ++k2) o[k2] *= alpha;
              tmem_st32(tm + c, o);
            }
            tmem_wait_st();
          }
          // P over S in tensor memory: hi pairs in the buffer's first 32 columns, lo in the next 32
          tmem_st32u(tm + D + kTcKeys * sb, hi);
          tmem_st32u(tm + D + kTcKeys * sb + 32, lo);
          tmem_wait_st();
          // keys at or past the context end may hold anything (even NaN) in the staged V: zero them
          // (every tile using the step writes the same zeros before its own O += P V)
          if (kbase + kTcKeys > it.len) {
            const int32_t J = J0 + step;
            const int s_ = J % STAGES;
            mbar_wait_bounded(smem_addr(kv_full + s_), static_cast<uint32_t>((J / STAGES) & 1));   // landed
            const int z0 = max(0, it.len - kbase);
            unsigned char* vst = smem + Sh::RING_OFF + s_ * Sh::STAGE_BYTES + Sh::K_BYTES;
            for (int q = r; q < (kTcKeys - z0) * 8 * DH; q += 128) {
              const int dh = q / ((kTcKeys - z0) * 8), rem = q % ((kTcKeys - z0) * 8);
              *reinterpret_cast<uint4*>(vst + dh * Sh::KV_REGION + (z0 + rem / 8) * 128 + (rem % 8) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();   // generic-proxy writes of V zeros before the MMA reads them
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(tb + 2 + sb));
        }
        if (!ok || *abort_flag) {
          ok = false;
          break;
        }
        // ---- epilogue: O / l for the real rows (once O += P V of the last step I - 1, and with it every
        // earlier one, has completed: the same one-phase argument), then O is free for the next item
        if (!mbar_wait_bounded(smem_addr(tb + 4 + ((I - 1) & 1)), static_cast<uint32_t>(((I - 1) >> 1) & 1))) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const float inv = 1.f / l;
        const int64_t orow = (static_cast<int64_t>(it.q0) + tok) * a.Hq + it.h * G + (r % G);
        float* dst = shared ? a.part_o + (static_cast<int64_t>(it.split) * a.total_q * a.Hq + orow) * D
                            : a.out + orow * D;
        if (shared && row_real) a.part_lse[static_cast<int64_t>(it.split) * a.total_q * a.Hq + orow] = m + log2f(l);
        // Coalesced stores: each 32 x 16 block of the warp's rows goes through shared memory, so that
        // a store instruction writes 64 contiguous bytes of each of 8 rows (4 lanes per row) instead
        // of 16 bytes of each of 32 rows. Slot s of row j sits at slot s ^ ((j >> 1) & 3) of that row:
        // both the row-wise writes and the column-wise reads hit 8 distinct 16-byte bank groups per
        // quarter warp. rd[i]: destination of row 8 i + lane / 4 (null for a padding row).
        float4* stg = reinterpret_cast<float4*>(smem + Sh::EPI_OFF + warp * Sh::EPI_WARP_BYTES);
        float* rd[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          rd[i] = reinterpret_cast<float*>(__shfl_sync(
              0xffffffffu, reinterpret_cast<unsigned long long>(row_real ? dst : nullptr), 8 * i + (lane >> 2)));
        const int sl = lane & 3;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tm + c, o);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              const float* v = o + 16 * hf + 4 * s4;
              stg[lane * 4 + (s4 ^ ((lane >> 1) & 3))] = make_float4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int row = 8 * i + (lane >> 2);
              const float4 v = stg[row * 4 + (sl ^ ((row >> 1) & 3))];
              if (rd[i] != nullptr) *reinterpret_cast<float4*>(rd[i] + c + 16 * hf + 4 * sl) = v;
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(tb + 6));   // O of this tile is free for the next item
      J0 += it.n_steps;
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == Sh::MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, Sh::TMEM_COLS);
  }
  pdl_launch_dependents();
}

}  // namespace pkv_dev
