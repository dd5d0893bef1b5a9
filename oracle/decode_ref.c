/*
 * Paged decode oracle in binary64 (plain C, OpenMP over (sequence, query head)).
 *
 * TEST INFRASTRUCTURE ONLY: called by tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py. Shares no code with the library.
 *
 * Definition ("Servicio de modelos de lenguaje con un presupuesto de memoria" §6):
 * scores = scale * q . k_t, softmax over t, output = sum_t softmax_t * v_t.
 * Paging ("¿Cómo gestiona Paged Attention la caché KV...?", "PagedAttention divide el
 * estado KV en bloques de tamaño fijo"): logical position t of a sequence lives in
 * physical block table[t / B] at offset t % B. The oracle rebuilds the contiguous K and
 * V of the sequence first and then does dense attention; it never splits the context.
 * GQA ("¿Cuánta memoria reservar para la caché KV?", "Emplear las cabezas KV"): query
 * head j reads KV head j / (Hq / Hkv).
 *
 * Sliding window ("¿Cuánta memoria reservar para la caché KV?", "Adaptar el presupuesto a la
 * estrategia de caché"): with window > 0 only positions [max(0, len - window), len) are attended to.
 *
 * Storage types: 0 = float32, 1 = bfloat16 bit patterns (decoded exactly), 3 = binary64 (e.g. a
 * dequantised fp8 pool).
 * Cache layout: cache[block][kv_head][offset][dim].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

static double load_value(const void* base, int dtype, size_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  if (dtype == 3) return ((const double*)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* out: [n_rows][D] binary64, where row r is the flat (b * Hq + j) id rows[r] (rows == NULL: all).
 * Returns the number of OpenMP threads used, or -1 on invalid arguments. */
int oracle_decode(double* out, const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                  int kv_dtype, const int32_t* tables, const int32_t* lens, int n_seqs, int num_q_heads,
                  int num_kv_heads, int head_dim, int block_size, int max_blocks, double scale, int window,
                  const int32_t* rows, int n_rows, int n_threads) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0) return -1;
  const int g = num_q_heads / num_kv_heads;
  const int D = head_dim;
  const long total = rows ? (long)n_rows : (long)n_seqs * num_q_heads;
  if (n_threads <= 0) n_threads = omp_get_max_threads();
  int used = 1;
#pragma omp parallel num_threads(n_threads)
  {
#pragma omp single
    used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 1)
    for (long r = 0; r < total; ++r) {
      const long flat = rows ? (long)rows[r] : r;
      const int b = (int)(flat / num_q_heads);
      const int j = (int)(flat % num_q_heads);
      const int h = j / g;
      const int len = lens[b];
      double* o = out + r * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (len <= 0) continue;
      const int t0 = (window > 0 && len > window) ? len - window : 0;   /* first attended position */
      const int L = len - t0;
      double* K = (double*)malloc(sizeof(double) * (size_t)L * D);
      double* V = (double*)malloc(sizeof(double) * (size_t)L * D);
      double* s = (double*)malloc(sizeof(double) * (size_t)L);
      double* qv = (double*)malloc(sizeof(double) * (size_t)D);
      /* rebuild the contiguous sequence through the block table */
      for (int t = 0; t < L; ++t) {
        const int pos = t0 + t;
        const long blk = tables[(long)b * max_blocks + pos / block_size];
        const size_t base = (((size_t)blk * num_kv_heads + h) * block_size + (pos % block_size)) * D;
        for (int d = 0; d < D; ++d) {
          K[(size_t)t * D + d] = load_value(k_cache, kv_dtype, base + d);
          V[(size_t)t * D + d] = load_value(v_cache, kv_dtype, base + d);
        }
      }
      for (int d = 0; d < D; ++d) qv[d] = load_value(q, q_dtype, ((size_t)b * num_q_heads + j) * D + d);
      /* scores, max, exponentials, weighted sum */
      double m = -INFINITY;
      for (int t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += K[(size_t)t * D + d] * qv[d];
        s[t] = scale * acc;
        if (s[t] > m) m = s[t];
      }
      double l = 0.0;
      for (int t = 0; t < L; ++t) {
        s[t] = exp(s[t] - m);
        l += s[t];
      }
      for (int t = 0; t < L; ++t)
        for (int d = 0; d < D; ++d) o[d] += s[t] * V[(size_t)t * D + d];
      for (int d = 0; d < D; ++d) o[d] /= l;
      free(K);
      free(V);
      free(s);
      free(qv);
    }
  }
  return used;
}

/* Causal prefill / multi-token append (same definition, one query row per new position):
 * sequence b has final length lens[b] and its last q_len_b = cu_q[b+1] - cu_q[b] positions are
 * queries; query i (row cu_q[b] + i of q, position p = lens[b] - q_len_b + i) attends to positions
 * [max(0, p - window + 1), p] (window <= 0: [0, p]). q: [total_q][Hq][D]; out: [total_q][Hq][D].
 * Reading of the pages: prefill and generation are separate phases of one request ("¿Cuánta memoria
 * reservar para la caché KV?", "Verificar una carga representativa por etapas"). */
int oracle_prefill(double* out, const void* q, int q_dtype, const void* k_cache, const void* v_cache, int kv_dtype,
                   const int32_t* tables, const int32_t* lens, const int32_t* cu_q, int n_seqs, int num_q_heads,
                   int num_kv_heads, int head_dim, int block_size, int max_blocks, double scale, int window,
                   int n_threads) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0) return -1;
  const int g = num_q_heads / num_kv_heads;
  const int D = head_dim;
  const long total = (long)cu_q[n_seqs] * num_q_heads;
  if (n_threads <= 0) n_threads = omp_get_max_threads();
  int used = 1;
#pragma omp parallel num_threads(n_threads)
  {
#pragma omp single
    used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 4)
    for (long r = 0; r < total; ++r) {
      const long row = r / num_q_heads;
      const int j = (int)(r % num_q_heads);
      const int h = j / g;
      int b = 0;
      while (cu_q[b + 1] <= row) ++b;
      const int qlen = cu_q[b + 1] - cu_q[b];
      const int p = lens[b] - qlen + (int)(row - cu_q[b]);
      const int t0 = (window > 0 && p - window + 1 > 0) ? p - window + 1 : 0;
      const int L = p + 1 - t0;
      double* o = out + r * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (L <= 0) continue;
      double* s = (double*)malloc(sizeof(double) * (size_t)L);
      double* qv = (double*)malloc(sizeof(double) * (size_t)D);
      for (int d = 0; d < D; ++d) qv[d] = load_value(q, q_dtype, ((size_t)row * num_q_heads + j) * D + d);
      double m = -INFINITY;
      for (int t = 0; t < L; ++t) {
        const int pos = t0 + t;
        const long blk = tables[(long)b * max_blocks + pos / block_size];
        const size_t base = (((size_t)blk * num_kv_heads + h) * block_size + (pos % block_size)) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += load_value(k_cache, kv_dtype, base + d) * qv[d];
        s[t] = scale * acc;
        if (s[t] > m) m = s[t];
      }
      double l = 0.0;
      for (int t = 0; t < L; ++t) {
        s[t] = exp(s[t] - m);
        l += s[t];
      }
      for (int t = 0; t < L; ++t) {
        const int pos = t0 + t;
        const long blk = tables[(long)b * max_blocks + pos / block_size];
        const size_t base = (((size_t)blk * num_kv_heads + h) * block_size + (pos % block_size)) * D;
        for (int d = 0; d < D; ++d) o[d] += s[t] * load_value(v_cache, kv_dtype, base + d);
      }
      for (int d = 0; d < D; ++d) o[d] /= l;
      free(s);
      free(qv);
    }
  }
  return used;
}
