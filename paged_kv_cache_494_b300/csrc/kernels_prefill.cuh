// Paged prefill / multi-token append attention (causal), bf16 K/V on tensor cores.
//
// What is computed: a prefill (or a multi-token append) adds q_len_b positions to sequence b, whose
// final length is len_b; query i sits at position p = len_b - q_len_b + i and attends causally to
// positions [0, p] (or the last `window` of them) through the block table. Prefill and generation
// are separate phases of one request ("¿Cuánta memoria reservar para la caché KV?", "Verificar una
// carga representativa por etapas"; "Servicio de modelos de lenguaje..." §7); the attention itself is
// the exact softmax attention of §6 of that page, computed blockwise with running statistics.
//
// Decomposition (B300 design): one CTA per (query tile, KV head). A CTA's 4 warps each own up to 16
// mma rows, a row being one (query token, query head of the GQA group): 16 / G tokens per warp,
// 4 * (16 / G) per CTA, so the whole group shares each K/V chunk. The CTA streams the chunks of its
// tile's causal range through one ring of `stages` shared-memory slots, filled by 2-D tensor TMA
// (128-byte swizzle; thread 0 issues) with a `full` mbarrier (TMA bytes) and an `empty` mbarrier
// (one arrival per warp) per slot. S = Q K^T and O += P V use mma.sync m16n8k16 with fp32
// accumulation; P goes through two mmas, its bf16 rounding (hi) and the bf16 rounding of the remainder
// (lo), so the weights keep ~17 bits. No split of the context: prefill tiles give enough CTAs.
#pragma once

#include "kernels_decode.cuh"

namespace pkv_dev {

struct PrefillArgs {
  float* out;                    // [total_q][Hq][D]
  const void* q;                 // [total_q][Hq][D] bf16
  const int32_t* block_tables;   // [n_seqs][MB]
  const int32_t* context_lens;   // [n_seqs] final lengths (the new positions included)
  const int32_t* cu_q;           // [n_seqs + 1] query rows of sequence b: cu_q[b] .. cu_q[b+1]
  int32_t n_seqs, Hq, Hkv, B, NB, MB, window, stages;
  float scale_log2;
  unsigned int* err;             // error word of the call's pool (null: the process-wide word)
  // Shared-prefix mode (tcgen05 kernel only; shared_len > 0): the keys are positions [0, shared_len)
  // of sequence 0's table, every one of the total_q rows of q attends to all of them (no causal
  // mask), and the keys are cut into splits of split_keys (a multiple of 64); split s writes its
  // normalised partial output to part_o[s][row][head][:] and m + log2 l to part_lse[s][row][head].
  // cu_q and context_lens are not read.
  int32_t total_q, shared_len, split_keys;
  float* part_o;
  float* part_lse;
  int32_t early_trigger;   // tcgen05 kernel: the next kernel may launch once this one passed its own wait
  unsigned long long* task_ctr;   // optional: the following decode's task counter, set to its call tag
  unsigned long long task_tag;    //   here so that its first takers find it installed
};

template <int D, int G>
struct PrefillShape {
  static constexpr int NW = 4;                 // warps per CTA
  static constexpr int TQW = 16 / G;           // query tokens per warp (rows = TQW * G <= 16)
  static constexpr int TQ = NW * TQW;          // query tokens per CTA
  static constexpr int BOX = kChunk * 128;     // 16 rows x 128 bytes
  static constexpr int KB = D / 64;
  static constexpr int CB = KB * BOX;          // K (or V) chunk bytes
  static constexpr int kStageBytes = 2 * CB;
  static constexpr int KS = D / 16;
  static constexpr int NT = D / 8;
  static constexpr int kQBytes = NW * 16 * D * 2;  // each warp's 16 query rows, staged for ldmatrix
};

// [1 KB alignment slack][ring: stages x stage][query rows][full / empty mbarriers][scan scratch]
// [query-tile prefix][block-table entries]
__host__ __device__ inline size_t prefill_smem_bytes(int stages, int stage_bytes, int q_bytes, int n_seqs,
                                                     int max_blocks) {
  return 1024 + static_cast<size_t>(stages) * stage_bytes + q_bytes + static_cast<size_t>(stages) * 16 + 256 +
         static_cast<size_t>(n_seqs + 1) * 4 + static_cast<size_t>(max_blocks) * 4;
}

__device__ __forceinline__ uint32_t prefill_swz(int row, int cb) {
  return static_cast<uint32_t>(row * 128 + ((cb ^ (row & 7)) << 4));
}

template <int D, int G>
__global__ void __launch_bounds__(128, 4) paged_prefill_kernel(const __grid_constant__ PrefillArgs a,
                                                            const __grid_constant__ TmaMaps maps) {
  using Sh = PrefillShape<D, G>;
  constexpr int NW = Sh::NW, TQW = Sh::TQW, TQ = Sh::TQ, BOX = Sh::BOX, CB = Sh::CB, SB = Sh::kStageBytes;
  constexpr int KS = Sh::KS, NT = Sh::NT;
  constexpr float kRescaleLog2 = 8.f;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int S = a.stages;
  const int32_t n = a.n_seqs;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  unsigned char* ring = smem;
  unsigned char* qsm = smem + static_cast<size_t>(S) * SB;   // [NW][16 rows][D] bf16, 16-byte blocks swizzled
  uint64_t* full = reinterpret_cast<uint64_t*>(qsm + Sh::kQBytes);
  uint64_t* empty = full + S;
  int32_t* wsum = reinterpret_cast<int32_t*>(empty + S);
  int32_t* tpref = wsum + 64;          // [n + 1] query-tile prefix over sequences
  int32_t* tab = tpref + (n + 1);      // block-table entries of this CTA's chunk range

  set_error_word(a.err);
  pdl_wait();

  // ---- query-tile prefix over sequences (block-wide scan)
  {
    int32_t carry = 0;
    for (int32_t base = 0; base < n; base += blockDim.x) {
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
      for (int w2 = 0; w2 < NW; ++w2) {
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
  const int32_t qt = tile - tpref[b];
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
  const int32_t t_begin = qt * TQ;                         // first query token of this CTA
  const int32_t t_end = min(t_begin + TQ, ql);             // one past the last
  if (t_begin >= t_end) {
    pdl_launch_dependents();
    return;
  }
  const int32_t pos0 = len - ql;                           // position of query token 0
  const int32_t p_lo = pos0 + t_begin, p_hi = pos0 + t_end - 1;
  const int32_t c_lo = (a.window > 0 && p_lo - a.window + 1 > 0) ? (p_lo - a.window + 1) / kChunk : 0;
  const int32_t c_hi = p_hi / kChunk;
  const int32_t n_chunks = c_hi - c_lo + 1;

  // ---- block-table entries of the range, and barriers
  const int32_t pg_lo = c_lo * kChunk / a.B, pg_hi = c_hi * kChunk / a.B;
  for (int32_t i = tid; i <= pg_hi - pg_lo; i += blockDim.x)
    tab[i] = __ldg(a.block_tables + static_cast<int64_t>(b) * a.MB + pg_lo + i);
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(full + s), 1);
      mbar_init(smem_addr(empty + s), NW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t policy = policy_evict_first();
  auto issue = [&](int32_t i) {  // thread 0 only: chunk i of the range into stage i % S
    const int stage = i % S;
    const int32_t tok0 = (c_lo + i) * kChunk;
    const int32_t pg = tok0 / a.B;
    const int32_t blk = tab[pg - pg_lo];
    const uint32_t bar = smem_addr(full + stage);
    if (blk >= 0 && blk < a.NB) {
      const int32_t y = static_cast<int32_t>((static_cast<int64_t>(blk) * a.Hkv + h) * a.B + (tok0 - pg * a.B));
      const uint32_t dst = smem_addr(ring + static_cast<size_t>(stage) * SB);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, 2 * CB);
#pragma unroll
      for (int kb = 0; kb < Sh::KB; ++kb) {
        tma_load_2d(dst + kb * BOX, &maps.k, 64 * kb, y, bar, policy);
        tma_load_2d(dst + CB + kb * BOX, &maps.v, 64 * kb, y, bar, policy);
      }
    } else {
      record_error(ERRBIT_BOUNDS);
      mbar_arrive(bar);
    }
  };
  if (tid == 0)
    for (int32_t i = 0; i < S && i < n_chunks; ++i) issue(i);

  // ---- per-warp rows: row r = (token r / G, head r % G); lane owns rows g and g + 8
  const int g = lane >> 2, t = lane & 3;
  const int32_t wt_begin = t_begin + warp * TQW;            // this warp's first token
  const int32_t wt_last = min(wt_begin + TQW, t_end) - 1;   // its last real token (< begin: none)
  const bool warp_has_rows = wt_last >= wt_begin;
  int32_t row_tok[2], row_head[2];
  bool row_real[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int r = g + 8 * k;
    const int32_t tk = wt_begin + r / G;
    row_real[k] = warp_has_rows && r < TQW * G && tk <= wt_last;
    row_tok[k] = warp_has_rows ? min(tk, wt_last) : t_begin;   // padding rows repeat a real token
    row_head[k] = r < TQW * G ? r % G : 0;
  }
  const int32_t row_pos[2] = {pos0 + row_tok[0], pos0 + row_tok[1]};
  const int32_t row_ws[2] = {a.window > 0 ? row_pos[0] - a.window + 1 : 0,
                             a.window > 0 ? row_pos[1] - a.window + 1 : 0};

  // This warp's 16 query rows (row r = token r / G, head r % G; padding rows repeat a real token)
  // into shared memory: 16-byte block c of row r at ((c & 7) ^ (r & 7)) + (c & ~7), so that the
  // ldmatrix reads of the A fragments below are free of bank conflicts. Reading q from shared memory
  // for every chunk instead of holding it in registers keeps the kernel within 128 registers.
  const uint32_t qw = smem_addr(qsm + static_cast<size_t>(warp) * 16 * D * 2);
  {
    const uint4* qb = static_cast<const uint4*>(a.q);
    constexpr int NBK = D / 8;   // 16-byte blocks per row
    unsigned char* qrow_base = qsm + static_cast<size_t>(warp) * 16 * D * 2;
    for (int idx = lane; idx < 16 * NBK; idx += 32) {
      const int rr = idx / NBK, c = idx % NBK;
      const int32_t tk = wt_begin + rr / G;
      const int32_t tok = warp_has_rows ? min(tk, wt_last) : t_begin;
      const int hd = rr < TQW * G ? rr % G : 0;
      const uint4 v = __ldg(qb + ((static_cast<int64_t>(q0) + tok) * a.Hq + h * G + hd) * NBK + c);
      *reinterpret_cast<uint4*>(qrow_base + rr * D * 2 + ((((c & 7) ^ (rr & 7)) + (c & ~7)) << 4)) = v;
    }
    __syncwarp();
  }
  // A fragment of k-step ks: lanes 0..15 address rows 0..15 at dims 16ks.., lanes 16..31 at 16ks+8..
  const int qrow = lane & 15;
  auto q_frag = [&](int ks, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    const int c = 2 * ks + (lane >> 4);
    ldsm_x4(qw + qrow * D * 2 + ((((c & 7) ^ (qrow & 7)) + (c & ~7)) << 4), a0, a1, a2, a3);
  };
  float o[NT][4];
#pragma unroll
  for (int nn = 0; nn < NT; ++nn) o[nn][0] = o[nn][1] = o[nn][2] = o[nn][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const int mi = lane >> 3, mr = lane & 7;
  bool aborted = false;
  int32_t i = 0;
  for (; i < n_chunks; ++i) {
    const int stage = i % S;
    if (!mbar_wait_bounded(smem_addr(full + stage), static_cast<uint32_t>((i / S) & 1))) {
      aborted = true;
      break;
    }
    const int32_t cpos = (c_lo + i) * kChunk;   // position of the chunk's first key
    if (warp_has_rows) {
      const uint32_t kb = smem_addr(ring + static_cast<size_t>(stage) * SB);
      const uint32_t vb = kb + CB;
      // four independent accumulation chains: (n-tile, even / odd k-step)
      float se[2][4], so[2][4], s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) se[nt][e] = so[nt][e] = 0.f;
#pragma unroll
      for (int p = 0; p < KS / 2; ++p) {
        uint32_t qe[4], qo[4];
        q_frag(2 * p, qe[0], qe[1], qe[2], qe[3]);
        q_frag(2 * p + 1, qo[0], qo[1], qo[2], qo[3]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int tok = 8 * nt + mr;
          const int db = 4 * p + mi;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + (db >> 3) * BOX + prefill_swz(tok, db & 7), b0, b1, b2, b3);
          mma_bf16_16816(se[nt], qe[0], qe[1], qe[2], qe[3], b0, b1);
          mma_bf16_16816(so[nt], qo[0], qo[1], qo[2], qo[3], b2, b3);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = se[nt][e] + so[nt][e];
      // keys of this lane: cpos + {2t, 2t+1, 8+2t, 9+2t}; rows g (k = 0, accum [0..1]) and g+8 ([2..3])
      const int kk[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
      float pr[2][4];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int32_t key = cpos + kk[e];
          const bool ok = key <= row_pos[k] && key >= row_ws[k];
          x[e] = ok ? s[e >> 1][2 * k + (e & 1)] * a.scale_log2 : -INFINITY;
        }
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const bool raise = mx > m[k] + kRescaleLog2;
        if (__any_sync(0xffffffffu, raise)) {
          const float mnew = raise ? mx : m[k];
          const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(m[k] - mnew);
          m[k] = mnew;
          l[k] *= alpha;
#pragma unroll
          for (int nn = 0; nn < NT; ++nn) {
            o[nn][2 * k] *= alpha;
            o[nn][2 * k + 1] *= alpha;
          }
        }
        const float msafe = m[k] == -INFINITY ? 0.f : m[k];   // a row with no key yet gets weight 0
#pragma unroll
        for (int e = 0; e < 4; ++e) pr[k][e] = exp2f(x[e] - msafe);
        l[k] += (pr[k][0] + pr[k][1]) + (pr[k][2] + pr[k][3]);
      }
      // A operand: R0 = row g keys 2t.., R1 = row g+8 keys 2t.., R2 = row g keys 8+2t.., R3 = row g+8 keys 8+2t..
      const uint32_t h0 = pack_bf16x2(pr[0][0], pr[0][1]), h1 = pack_bf16x2(pr[1][0], pr[1][1]);
      const uint32_t h2 = pack_bf16x2(pr[0][2], pr[0][3]), h3 = pack_bf16x2(pr[1][2], pr[1][3]);
      const uint32_t l0 = pack_bf16x2(pr[0][0] - bf16_lo(h0), pr[0][1] - bf16_hi(h0));
      const uint32_t l1 = pack_bf16x2(pr[1][0] - bf16_lo(h1), pr[1][1] - bf16_hi(h1));
      const uint32_t l2 = pack_bf16x2(pr[0][2] - bf16_lo(h2), pr[0][3] - bf16_hi(h2));
      const uint32_t l3 = pack_bf16x2(pr[1][2] - bf16_lo(h3), pr[1][3] - bf16_hi(h3));
      // keys at or past the context end may hold garbage (even NaN): zero their V entries
      const bool tail = cpos + kChunk > len;
      uint32_t mask01 = 0xffffffffu, mask23 = 0xffffffffu;
      if (tail) {
        mask01 = ((cpos + 2 * t < len) ? 0x0000ffffu : 0u) | ((cpos + 2 * t + 1 < len) ? 0xffff0000u : 0u);
        mask23 = ((cpos + 8 + 2 * t < len) ? 0x0000ffffu : 0u) | ((cpos + 9 + 2 * t < len) ? 0xffff0000u : 0u);
      }
      const int vtok = mr + 8 * (mi & 1);
#pragma unroll
      for (int pair = 0; pair < NT / 2; ++pair) {
        const int db = 2 * pair + (mi >> 1);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vb + (db >> 3) * BOX + prefill_swz(vtok, db & 7), v0, v1, v2, v3);
        if (tail) {
          v0 &= mask01;
          v1 &= mask23;
          v2 &= mask01;
          v3 &= mask23;
        }
        mma_bf16_16816(o[2 * pair], h0, h1, h2, h3, v0, v1);
        mma_bf16_16816(o[2 * pair], l0, l1, l2, l3, v0, v1);
        mma_bf16_16816(o[2 * pair + 1], h0, h1, h2, h3, v2, v3);
        mma_bf16_16816(o[2 * pair + 1], l0, l1, l2, l3, v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(empty + stage));
    if (tid == 0 && i + S < n_chunks) {
      if (!mbar_wait_bounded(smem_addr(empty + stage), static_cast<uint32_t>((i / S) & 1))) {
        aborted = true;
      } else {
        issue(i + S);
      }
    }
    if (__shfl_sync(0xffffffffu, aborted ? 1 : 0, 0)) break;
  }
  if (aborted) {
    // Thread 0 drains the copies it issued (bounded) so none lands after the CTA exits.
    if (tid == 0)
      for (int32_t k = i; k < n_chunks && k < i + S; ++k)
        mbar_wait_bounded(smem_addr(full + (k % S)), static_cast<uint32_t>((k / S) & 1));
    pdl_launch_dependents();
    return;
  }
  // ---- write the real rows: o / l
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    float lt = l[k];
    lt += __shfl_xor_sync(0xffffffffu, lt, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    if (!row_real[k]) continue;
    const float inv = 1.f / lt;
    float* dst = a.out + ((static_cast<int64_t>(q0) + row_tok[k]) * a.Hq + h * G + row_head[k]) * D;
#pragma unroll
    for (int nn = 0; nn < NT; ++nn)
      *reinterpret_cast<float2*>(dst + 8 * nn + 2 * t) = make_float2(o[nn][2 * k] * inv, o[nn][2 * k + 1] * inv);
  }
  pdl_launch_dependents();
}

}  // namespace pkv_dev
