"""Closed forms of the KV-cache byte budget and of paging tail waste (integers, exact).

Test infrastructure only (see ``oracle/__init__``).

Sources:
* "Servicio de modelos de lenguaje con un presupuesto de memoria" §3 (bytes per
  retained token = 2 x layers x KV heads x head dim x bytes per scalar, times the
  sum of retained lengths) and §5 (a length-T request on B-slot pages holds
  B*ceil(T/B) slots; its unused tail lies in [0, B-1]).
* "¿Cuánta memoria reservar para la caché KV?", "Plantear la fórmula y sus
  unidades" (same formula with the sum of stored positions for ragged batches)
  and "Ejemplo trabajado: seis secuencias" (40-layer worked example).
* "Paged Attention optimiza el uso de memoria en LLMs", paragraphs on the 2,048-
  token reservation, 16-token pages and the utilisation comparison.

Parity unpinned: the six-request example of "Servicio de modelos..." §9 prints
``page_tail_slots: 32`` but not the six lengths, so no function reproduces it.
"""
from __future__ import annotations

from fractions import Fraction
from typing import Iterable


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_scalar: int) -> int:
    """Bytes of uncompressed K and V state per retained token: 2 (K and V) x L x H x d x b."""
    return 2 * layers * kv_heads * head_dim * bytes_per_scalar


def kv_bytes(lengths: Iterable[int], layers: int, kv_heads: int, head_dim: int,
             bytes_per_scalar: int) -> int:
    """KV bytes of a batch: per-token bytes times the sum of retained lengths (ragged, unpadded)."""
    return kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_scalar) * sum(int(t) for t in lengths)


def pages(T: int, B: int) -> int:
    """Number of B-token pages a length-T request occupies: ceil(T / B)."""
    if T < 0 or B <= 0:
        raise ValueError("T >= 0 and B > 0 required")
    return -(-T // B)


def allocated_slots(T: int, B: int) -> int:
    """Token slots held by a length-T request on B-token pages: B * ceil(T / B)."""
    return B * pages(T, B)


def tail_slots(T: int, B: int) -> int:
    """Unused slots in the last page: allocated capacity minus T."""
    return allocated_slots(T, B) - T


def mean_tail_uniform(n_max: int, B: int) -> Fraction:
    """Mean tail waste over lengths uniform on 1..n_max, by enumeration (exact rational)."""
    return Fraction(sum(tail_slots(T, B) for T in range(1, n_max + 1)), n_max)


def mean_reservation_waste(n_max: int, reserved: int) -> Fraction:
    """Mean unused slots when every request reserves ``reserved`` slots, T uniform on 1..n_max."""
    return Fraction(sum(reserved - T for T in range(1, n_max + 1)), n_max)


def utilisation_paged(lengths: Iterable[int], B: int) -> Fraction:
    """Stored tokens over allocated page slots."""
    ls = [int(t) for t in lengths]
    return Fraction(sum(ls), sum(allocated_slots(T, B) for T in ls))


def utilisation_reserved(lengths: Iterable[int], reserved: int) -> Fraction:
    """Stored tokens over fixed per-request reservations."""
    ls = [int(t) for t in lengths]
    return Fraction(sum(ls), reserved * len(ls))
