"""Seeded synthetic inputs for the paged-decode workloads.

This module is shared by the tests, ``__graft_entry__.smoke()`` and ``bench.py``.
It draws random numbers and encodes them in the storage dtype; it holds none of
the method's arithmetic (no block allocation, no slot mapping, no attention), so
the oracle and the CUDA path can both consume it without sharing any logic.

Workload shapes follow the pages' statement of the problem:

* block/page size of 16 tokens and a page table per request
  ("Paged Attention optimiza el uso de memoria en LLMs", the 16-token example);
* 40 query heads over 8 KV heads, i.e. groups of 5
  ("¿Cuánta memoria reservar para la caché KV?", section on KV heads and GQA);
* 32 layers, 8 KV heads, head dim 128, 2-byte scalars = 128 KiB per token
  ("Servicio de modelos de lenguaje con un presupuesto de memoria", section 3);
* ~500-token average responses ("Paged Attention optimiza...", opening example);
* a shared system prompt forked into many requests with copy-on-write
  ("PagedAttention e vLLM", technical deep dive; "Paged Attention optimiza...").

Nothing here reads the pages at run time.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "lengths", "free_list", "normal_f32",
    "to_bf16_bits", "bf16_bits_to_f32", "encode", "suffix_lengths",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload (sizes only; values are drawn on demand)."""

    name: str
    description: str
    n_layers: int
    n_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str                      # "f32" or "bf16" (storage type of q, K, V)
    length_kind: str                # "fixed" | "uniform" | "lognormal" | "prefix"
    length_args: tuple
    pool_rule: str                  # how the pool size follows from the lengths
    partition_tokens: int = 0       # 0 = balanced split chosen by the library
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS: Dict[str, Workload] = {
    "tiny_f32": Workload(
        name="tiny_f32",
        description="tiny paged decode, 1 layer, fp32: lengths {1,17,100,500}, 8 q / 2 kv heads, "
                    "head_dim 64, block 16, pool of 64 blocks in seeded random order",
        n_layers=1, n_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
        dtype="f32", length_kind="fixed", length_args=(1, 17, 100, 500), pool_rule="fixed:64"),
    "gqa5_bf16": Workload(
        name="gqa5_bf16",
        description="GQA decode, 1 layer, bf16: batch 64, lengths U[100,2048], 40 q / 8 kv heads, "
                    "head_dim 128, block 16, pool = pages + 10%, shuffled free list",
        n_layers=1, n_seqs=64, num_q_heads=40, num_kv_heads=8, head_dim=128, block_size=16,
        dtype="bf16", length_kind="uniform", length_args=(100, 2048), pool_rule="pages*1.1"),
    "serve256_bf16": Workload(
        name="serve256_bf16",
        description="serving-shaped decode, 32 layers, bf16: batch 256, lengths lognormal "
                    "(median 500, sigma 0.8) clipped to [16,4096], 32 q / 8 kv heads, head_dim 128, "
                    "block 16, one appended token per sequence per layer",
        n_layers=32, n_seqs=256, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
        dtype="bf16", length_kind="lognormal", length_args=(500.0, 0.8, 16, 4096),
        pool_rule="(pages+seqs)*1.1"),
    "prefix_cow_bf16": Workload(
        name="prefix_cow_bf16",
        description="shared-prefix copy-on-write, bf16: 128 sequences forked from one 1,024-token "
                    "prompt (64 shared blocks), suffixes U[0,512], 32 q / 8 kv heads, head_dim 128, "
                    "block 16",
        n_layers=1, n_seqs=128, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
        dtype="bf16", length_kind="prefix", length_args=(1024, 0, 512), pool_rule="(pages)*1.1"),
    "prefix_cow_partial_bf16": Workload(
        name="prefix_cow_partial_bf16",
        description="as prefix_cow_bf16 but a 1,016-token prompt (63 full blocks + one half-full "
                    "block), so the first append of each child copies the shared partial block",
        n_layers=1, n_seqs=128, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
        dtype="bf16", length_kind="prefix", length_args=(1016, 0, 512), pool_rule="(pages)*1.1"),
    "prefill_bf16": Workload(
        name="prefill_bf16",
        description="paged prefill (causal), bf16: 16 prompts of 2,048 tokens written to the pool, every "
                    "position a query, 32 q / 8 kv heads, head_dim 128, block 16",
        n_layers=1, n_seqs=16, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
        dtype="bf16", length_kind="fixed", length_args=(2048,) * 16, pool_rule="pages*1.1"),
    "long_split_bf16": Workload(
        name="long_split_bf16",
        description="long-context split-KV decode, bf16: batch 8 x 32,768 tokens, 32 q / 8 kv heads, "
                    "head_dim 128, block 32, 512-token partitions merged by log-sum-exp, blocks "
                    "scattered by seeded permutation across an 80 GB-scale pool",
        n_layers=1, n_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
        dtype="bf16", length_kind="fixed", length_args=(32768,) * 8, pool_rule="bytes:80e9",
        partition_tokens=512),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def _rng(seed: int, stream: int) -> np.random.Generator:
    # independent streams per purpose so that changing one draw never shifts another
    return np.random.default_rng([int(seed), int(stream)])


def lengths(w: Workload, seed: Optional[int] = None) -> np.ndarray:
    """Per-sequence context lengths (int64), drawn with the workload's recipe.

    For the "prefix" kind this returns the final lengths prompt + suffix_b.
    """
    seed = w.seed if seed is None else seed
    r = _rng(seed, 1)
    if w.length_kind == "fixed":
        out = np.asarray(w.length_args, dtype=np.int64)
        assert out.size == w.n_seqs
        return out
    if w.length_kind == "uniform":
        lo, hi = w.length_args
        return r.integers(lo, hi + 1, size=w.n_seqs, dtype=np.int64)
    if w.length_kind == "lognormal":
        median, sigma, lo, hi = w.length_args
        z = r.standard_normal(w.n_seqs)
        return np.clip(np.rint(np.exp(math.log(median) + sigma * z)), lo, hi).astype(np.int64)
    if w.length_kind == "prefix":
        prompt = w.length_args[0]
        return prompt + suffix_lengths(w, seed)
    raise ValueError(w.length_kind)


def suffix_lengths(w: Workload, seed: Optional[int] = None) -> np.ndarray:
    """Unique suffix length of each forked child (prefix workloads only)."""
    seed = w.seed if seed is None else seed
    assert w.length_kind == "prefix"
    _, lo, hi = w.length_args
    return _rng(seed, 2).integers(lo, hi + 1, size=w.n_seqs, dtype=np.int64)


def pool_blocks(w: Workload, lens: np.ndarray) -> int:
    """Number of physical blocks in the pool for this workload's lengths."""
    B = w.block_size
    pages = int(sum((int(t) + B - 1) // B for t in lens))
    rule = w.pool_rule
    if rule.startswith("fixed:"):
        return int(rule.split(":")[1])
    if rule == "pages*1.1":
        return int(math.ceil(1.1 * pages))
    if rule == "(pages+seqs)*1.1":
        return int(math.ceil(1.1 * (pages + w.n_seqs)))
    if rule == "(pages)*1.1":
        # prefix workloads: the prompt's blocks are shared, each child owns its suffix blocks
        prompt = w.length_args[0]
        shared = (prompt + B - 1) // B
        private = sum((int(t) - prompt + B) // B + 1 for t in lens)
        return int(math.ceil(1.1 * (shared + private)))
    if rule.startswith("bytes:"):
        per_block = 2 * w.num_kv_heads * B * w.head_dim * w.elem_bytes * w.n_layers
        return int(float(rule.split(":")[1]) // per_block)
    raise ValueError(rule)


def free_list(num_blocks: int, seed: int) -> np.ndarray:
    """A seeded permutation of [0, num_blocks): the order in which blocks are handed out."""
    return _rng(seed, 3).permutation(num_blocks).astype(np.int32)


def normal_f32(shape, seed: int, stream: int) -> np.ndarray:
    """Standard-normal float32 draws."""
    return _rng(seed, 100 + stream).standard_normal(size=shape, dtype=np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Encode float32 values as bfloat16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    rounded = (u + (0x7FFF + ((u >> 16) & 1))) >> 16
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Decode bfloat16 bit patterns (uint16) into float32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def encode(x_f32: np.ndarray, dtype: str) -> np.ndarray:
    """Store float32 draws in the workload dtype: float32 array, or uint16 bf16 bits."""
    if dtype == "f32":
        return np.ascontiguousarray(x_f32, dtype=np.float32)
    if dtype == "bf16":
        return to_bf16_bits(x_f32)
    raise ValueError(dtype)


def nan_bits(dtype: str):
    """The stored bit pattern used to poison unowned cache memory."""
    return np.float32(np.nan) if dtype == "f32" else np.uint16(0x7FC0)


def prefix_trace(w: Workload, seed: Optional[int] = None) -> List[tuple]:
    """Operation trace of a shared-prefix workload, as plain tuples.

    ("new", prompt_tokens) creates the prompt sequence; ("fork", 0) x n_seqs forks it;
    ("free", 0) releases the prompt; ("append", child_index, n) appends each child's suffix
    in child order.
    """
    seed = w.seed if seed is None else seed
    prompt = w.length_args[0]
    suf = suffix_lengths(w, seed)
    ops: List[tuple] = [("new", prompt)]
    ops += [("fork", 0)] * w.n_seqs
    ops.append(("free", 0))
    ops += [("append", i, int(s)) for i, s in enumerate(suf)]
    return ops
