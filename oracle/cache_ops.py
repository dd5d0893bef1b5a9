"""Slot-mapped cache write and block copy on host arrays (bit copies, NumPy).

Test infrastructure only (see ``oracle/__init__``).

Cache layout per layer (a reading: the pages do not fix one): ``cache[block][kv_head][offset][dim]``,
i.e. the positions of one KV head inside one physical block are contiguous.

* ``reshape_and_cache``: as tokens arrive the runtime stores their K and V in the
  block the allocator gave them ("¿Cómo gestiona Paged Attention la caché KV...?",
  "PagedAttention divide el estado KV en bloques de tamaño fijo"); token i goes to
  slot s_i = block * B + offset; a negative slot means "skip this token".
* ``copy_blocks``: copy-on-write duplicates only the page where a request diverges
  ("Paged Attention optimiza el uso de memoria en LLMs", copy-on-write paragraph;
  "PagedAttention e vLLM", "Approfondimento tecnico"). Applied to every layer, K and V.
"""
from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np


def reshape_and_cache(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
                      slots: Sequence[int]) -> None:
    """In place: cache[s // B, h, s % B, :] = new[i, h, :] for every token i with s = slots[i] >= 0.

    ``k_cache``/``v_cache``: [NB, Hkv, B, D]; ``k``/``v``: [n_tokens, Hkv, D]; any dtype (bit copy).
    """
    B = k_cache.shape[2]
    for i, s in enumerate(slots):
        s = int(s)
        if s < 0:
            continue
        k_cache[s // B, :, s % B, :] = k[i]
        v_cache[s // B, :, s % B, :] = v[i]


def copy_blocks(caches: Sequence[Tuple[np.ndarray, np.ndarray]], pairs: Sequence[Tuple[int, int]]) -> None:
    """In place, for each layer's (K, V) cache and each (src, dst) pair in order: cache[dst] = cache[src]."""
    for kc, vc in caches:
        for src, dst in pairs:
            kc[int(dst)] = kc[int(src)]
            vc[int(dst)] = vc[int(src)]
