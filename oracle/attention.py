"""Exact attention over paged K/V in binary64 (NumPy), plus the online recurrence and merge.

Test infrastructure only (see ``oracle/__init__``).

Definition followed ("Servicio de modelos de lenguaje con un presupuesto de memoria" §6):
dense attention forms scaled query-key scores, applies softmax and multiplies by the
values; an IO-aware implementation processes blocks while keeping running
normalisation statistics and computes the same operation, not the same bits.

Paging ("¿Cómo gestiona Paged Attention la caché KV...?", "PagedAttention divide el
estado KV..."; "PagedAttention e vLLM", "Approfondimento tecnico"): a block table maps
logical token order to physical blocks; the indirection changes where K/V live, never
the order the model attends in. So the oracle first rebuilds each sequence's
contiguous K and V from its table, then does plain dense attention.

GQA ("¿Cuánta memoria reservar para la caché KV?", "Emplear las cabezas KV, en
particular con GQA"): 40 query heads over 8 KV heads form groups of 5. Reading: query
head j uses KV head j // (Hq / Hkv) (contiguous groups).

Readings where the pages are silent: the context length counts the token appended in
the same step (append, then attend); an empty context gives a zero output row; the
output is binary64 here and float32 on the device.

Cache layout: ``cache[block][kv_head][offset][dim]`` stored as float32, or as bfloat16
bit patterns in uint16 arrays (decoded exactly to binary64 below).
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np


def to_f64(x: np.ndarray) -> np.ndarray:
    """Stored values -> binary64: float32 as is, uint16 as bfloat16 bit patterns (exact)."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def gather_sequence(cache: np.ndarray, table: Sequence[int], length: int, kv_head: int) -> np.ndarray:
    """Contiguous [length, D] binary64 copy of one sequence's K (or V) for one KV head.

    Logical position t lives in physical block table[t // B] at offset t % B.
    """
    B = cache.shape[2]
    rows = [cache[int(table[t // B]), kv_head, t % B, :] if int(table[t // B]) >= 0
            else np.full(cache.shape[3], np.nan, dtype=cache.dtype) for t in range(length)]
    if not rows:
        return np.zeros((0, cache.shape[3]), dtype=np.float64)
    return to_f64(np.stack(rows))


def dense_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * K q) V for one query vector, binary64, max-subtracted."""
    s = scale * (K @ q)
    p = np.exp(s - s.max())
    return (p @ V) / p.sum()


def window_start(length: int, window: int) -> int:
    """First attended position under a sliding window (0 when window == 0 means no window).

    Reading of "¿Cuánta memoria reservar para la caché KV?", "Adaptar el presupuesto a la estrategia
    de caché": a sliding-window layer keeps only its most recent positions; here the last ``window``.
    """
    return max(0, length - window) if window > 0 else 0


def paged_decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, tables: np.ndarray,
                 lens: Sequence[int], scale: float, window: int = 0) -> np.ndarray:
    """Decode attention for every (sequence, query head): out[b, j] in binary64.

    q: [n_seqs, Hq, D] stored values; caches: [NB, Hkv, B, D]; tables: [n_seqs, MB] int.
    With window > 0 only positions [max(0, len - window), len) are attended to.
    """
    n, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    qd = to_f64(q)
    out = np.zeros((n, Hq, D), dtype=np.float64)
    for b in range(n):
        L = int(lens[b])
        if L == 0:
            continue
        t0 = window_start(L, window)
        for h in range(Hkv):
            K = gather_sequence(k_cache, tables[b], L, h)[t0:]
            V = gather_sequence(v_cache, tables[b], L, h)[t0:]
            for j in range(h * g, (h + 1) * g):
                out[b, j] = dense_attention(qd[b, j], K, V, scale)
    return out


def paged_prefill(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, tables: np.ndarray,
                  lens: Sequence[int], cu_q: Sequence[int], scale: float, window: int = 0) -> np.ndarray:
    """Causal attention of the last q_len_b positions of each sequence over its paged context.

    Reading of the pages: prefill and generation are separate phases of the same request
    ("¿Cuánta memoria reservar para la caché KV?", "Verificar una carga representativa por
    etapas"; "Servicio de modelos..." §7: prefill work and decode steps have different shapes).
    A prefill (or multi-token append) adds q_len_b positions to a sequence of final length len_b;
    query i (rows cu_q[b] + i of q) sits at position p = len_b - q_len_b + i and, as in any causal
    decoder, attends to positions [0, p] (or [max(0, p - window + 1), p] with a sliding window).
    q: [total_q, Hq, D]; returns [total_q, Hq, D] binary64. With q_len_b = 1 this is decode.
    """
    total, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    qd = to_f64(q)
    out = np.zeros((total, Hq, D), dtype=np.float64)
    for b in range(len(lens)):
        L = int(lens[b])
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        if q1 == q0:
            continue
        for h in range(Hkv):
            K = gather_sequence(k_cache, tables[b], L, h)
            V = gather_sequence(v_cache, tables[b], L, h)
            for i in range(q1 - q0):
                p = L - (q1 - q0) + i
                t0 = max(0, p - window + 1) if window > 0 else 0
                for j in range(h * g, (h + 1) * g):
                    out[q0 + i, j] = dense_attention(qd[q0 + i, j], K[t0:p + 1], V[t0:p + 1], scale)
    return out


def online_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, block: int) -> np.ndarray:
    """The same operation as ``dense_attention`` via the running max/sum recurrence over blocks.

    For each block: m' = max(m, max s_blk); acc = acc * e^(m - m') + sum_t e^(s_t - m') v_t;
    l = l * e^(m - m') + sum_t e^(s_t - m'); result acc / l.
    """
    m, l = -math.inf, 0.0
    acc = np.zeros(V.shape[1], dtype=np.float64)
    for start in range(0, K.shape[0], block):
        s = scale * (K[start:start + block] @ q)
        m_new = max(m, float(s.max()))
        c = math.exp(m - m_new) if m != -math.inf else 0.0
        p = np.exp(s - m_new)
        acc = acc * c + p @ V[start:start + block]
        l = l * c + float(p.sum())
        m = m_new
    return acc / l


def partial_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> Tuple[float, float, np.ndarray]:
    """(m, l, o) of one partition: max score, sum of e^(s - m), and the l-normalised output."""
    s = scale * (K @ q)
    m = float(s.max())
    p = np.exp(s - m)
    l = float(p.sum())
    return m, l, (p @ V) / l


def merge_partials(parts: List[Tuple[float, float, np.ndarray]]) -> np.ndarray:
    """Log-sum-exp merge of partition results: w_p = l_p e^(m_p - M), o = sum w_p o_p / sum w_p."""
    M = max(m for m, _, _ in parts)
    w = [l * math.exp(m - M) for m, l, _ in parts]
    return sum(wi * o for wi, (_, _, o) in zip(w, parts)) / sum(w)


def brute_force_decode(q: Sequence[Sequence[Sequence[float]]], k_cache, v_cache, tables, lens,
                       scale: float) -> List[List[List[float]]]:
    """Pure-Python loops with ``math.exp`` (tiny inputs only); no NumPy arithmetic.

    Accepts float-valued nested sequences (already decoded) for q and the caches.
    """
    n = len(q)
    Hq = len(q[0])
    D = len(q[0][0])
    Hkv = len(k_cache[0])
    B = len(k_cache[0][0])
    g = Hq // Hkv
    out = []
    for b in range(n):
        rows = []
        for j in range(Hq):
            h = j // g
            L = int(lens[b])
            if L == 0:
                rows.append([0.0] * D)
                continue
            scores = []
            for t in range(L):
                blk = int(tables[b][t // B])
                krow = k_cache[blk][h][t % B]
                scores.append(scale * sum(float(q[b][j][d]) * float(krow[d]) for d in range(D)))
            mx = max(scores)
            ws = [math.exp(x - mx) for x in scores]
            tot = sum(ws)
            o = [0.0] * D
            for t in range(L):
                blk = int(tables[b][t // B])
                vrow = v_cache[blk][h][t % B]
                for d in range(D):
                    o[d] += ws[t] * float(vrow[d])
            rows.append([x / tot for x in o])
        out.append(rows)
    return out
