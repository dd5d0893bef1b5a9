"""Builds paged-decode cases twice from the same seeded inputs: once through libpagedkv (host
allocator + CUDA kernels on the device) and once through the oracle (allocator model + NumPy
scatter on the host). Nothing computed by the library is fed to the oracle.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import numpy as np
import torch

import paged_kv_cache_494_b300 as pkv
import synth
from oracle import alloc_model as am
from oracle import cache_ops as ocache
from oracle import native
from oracle import fp8 as _ofp8  # noqa: F401

TOL = {"f32": 1e-5, "bf16": 2e-3}


def to_device(stored: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(stored)).cuda()
    return torch.from_numpy(np.ascontiguousarray(stored).view(np.int16)).view(torch.bfloat16).cuda()


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def torch_dtype(dtype: str):
    return torch.float32 if dtype == "f32" else torch.bfloat16


class Case:
    """A pool, its sequences and cache contents, built independently on both sides."""

    def __init__(self, *, lengths: Sequence[int], Hq: int, Hkv: int, D: int, B: int, dtype: str,
                 num_blocks: Optional[int] = None, seed: int = 0, free_list: Optional[np.ndarray] = None,
                 max_blocks: Optional[int] = None, host_cache: bool = True, prefix_trace=None,
                 compact_host: bool = False):
        self.Hq, self.Hkv, self.D, self.B, self.dtype = Hq, Hkv, D, B, dtype
        self.seed = seed
        lengths = [int(x) for x in lengths]
        pages = sum(-(-L // B) for L in lengths)
        # headroom for decode-step appends: a few blocks per sequence
        self.NB = num_blocks or max(pages + 4 * len(lengths) + 8, 16)
        self.MB = max_blocks or max(max(-(-L // B) for L in lengths), 1) + 4
        self.scale = 1.0 / math.sqrt(D)
        fl = free_list if free_list is not None else synth.free_list(self.NB, seed)
        n_ids = len(lengths) + 1
        self.pool = pkv.Pool(1, Hkv, D, B, self.NB, n_ids, self.MB, pkv.F32 if dtype == "f32" else pkv.BF16,
                             initial_free_list=fl)
        self.model = am.PoolModel(self.NB, B, n_ids, self.MB, initial_free_list=fl)
        tdt = torch_dtype(dtype)
        shape = (self.NB, Hkv, B, D)
        self.k_cache = torch.full(shape, float("nan"), dtype=tdt, device="cuda")
        self.v_cache = torch.full(shape, float("nan"), dtype=tdt, device="cuda")
        self.host_cache = host_cache
        self.compact = compact_host
        self._recorded = []
        store = np.float32 if dtype == "f32" else np.uint16
        if host_cache and not compact_host:
            self.hk = np.full(shape, synth.nan_bits(dtype), dtype=store)
            self.hv = np.full(shape, synth.nan_bits(dtype), dtype=store)
        self._stream = 0
        if prefix_trace is None:
            self.seqs = []
            for L in lengths:
                self.seqs.append(self._append(-1, L))
        else:
            self._run_prefix(prefix_trace)
        assert sorted(self.seqs) == sorted(self.model.tables) if prefix_trace is None else True
        self.n = len(self.seqs)
        self.q_stored = synth.encode(synth.normal_f32((self.n, Hq, D), seed, 7), dtype)
        self.q = to_device(self.q_stored, dtype)
        tables, lens = self.pool.block_table(self.seqs)
        mtab, mlens = self.model.block_table(self.seqs)
        assert tables.tolist() == mtab and lens.tolist() == mlens      # allocator parity (bit-exact)
        self.tables = torch.from_numpy(tables).cuda()
        self.lens = torch.from_numpy(lens).cuda()
        self.oracle_tables = np.asarray(mtab, dtype=np.int32)
        self.oracle_lens = np.asarray(mlens, dtype=np.int32)
        if self.compact:
            self._build_compact_host()

    def _build_compact_host(self):
        """Host caches holding only the blocks the oracle's tables use, renumbered in order of use."""
        used = [int(b) for b in np.unique(self.oracle_tables[self.oracle_tables >= 0])]
        remap = {b: i for i, b in enumerate(used)}
        store = np.float32 if self.dtype == "f32" else np.uint16
        shape = (len(used), self.Hkv, self.B, self.D)
        self.hk = np.full(shape, synth.nan_bits(self.dtype), dtype=store)
        self.hv = np.full(shape, synth.nan_bits(self.dtype), dtype=store)
        for slots, k, v in self._recorded:
            blk = np.asarray(slots) // self.B
            off = np.asarray(slots) % self.B
            keep = np.array([b in remap for b in blk.tolist()], dtype=bool)
            cslots = [remap[int(b)] * self.B + int(o) for b, o in zip(blk[keep], off[keep])]
            ocache.reshape_and_cache(self.hk, self.hv, k[keep], v[keep], cslots)
        self._recorded = []
        self.oracle_tables = np.where(self.oracle_tables >= 0,
                                      np.vectorize(lambda b: remap.get(int(b), -1))(self.oracle_tables),
                                      -1).astype(np.int32)

    # -- building ----------------------------------------------------------------------------
    def _values(self, n_tokens: int):
        self._stream += 1
        kv = synth.normal_f32((2, n_tokens, self.Hkv, self.D), self.seed, 1000 + self._stream)
        return synth.encode(kv[0], self.dtype), synth.encode(kv[1], self.dtype)

    def _write(self, slots_lib, slots_model, pairs_lib, pairs_model, n_tokens):
        assert slots_lib.tolist() == list(slots_model)
        assert [tuple(p) for p in pairs_lib] == [tuple(p) for p in pairs_model]
        k, v = self._values(n_tokens)
        if len(pairs_lib):
            assert not self.compact, "compact host caches support traces without copy-on-write"
            d_pairs = torch.tensor(np.asarray(pairs_lib, dtype=np.int32).reshape(-1, 2), device="cuda")
            self.pool.copy_blocks([self.k_cache], [self.v_cache], d_pairs)
            if self.host_cache:
                ocache.copy_blocks([(self.hk, self.hv)], pairs_model)
        if n_tokens:
            self.pool.reshape_and_cache(to_device(k, self.dtype), to_device(v, self.dtype),
                                        torch.from_numpy(np.asarray(slots_lib, dtype=np.int64)).cuda(),
                                        self.k_cache, self.v_cache)
            if self.compact:
                self._recorded.append((list(slots_model), k, v))
            elif self.host_cache:
                ocache.reshape_and_cache(self.hk, self.hv, k, v, slots_model)

    def _append(self, seq: int, n_tokens: int) -> int:
        sid, slots, pairs = self.pool.alloc(seq, n_tokens)
        st, msid, mslots, mpairs = self.model.alloc(seq, n_tokens)
        assert st == am.OK and msid == sid
        self._write(slots, mslots, pairs, mpairs, n_tokens)
        return sid

    def _run_prefix(self, trace):
        children = {}
        root = None
        for op in trace:
            if op[0] == "new":
                root = self._append(-1, op[1])
            elif op[0] == "fork":
                c = self.pool.fork(root)
                st, mc = self.model.fork(root)
                assert st == am.OK and mc == c
                children[len(children)] = c
            elif op[0] == "free":
                self.pool.free(root)
                assert self.model.free_seq(root) == am.OK
            else:
                self._append(children[op[1]], op[2])
        self.seqs = [children[i] for i in range(len(children))]

    def decode_step_append(self):
        """Append one token to every sequence (a decode step's a1 + K2 + K1)."""
        slots, pairs = self.pool.append(self.seqs)
        st, mslots, mpairs = self.model.append(self.seqs)
        assert st == am.OK
        self._write(slots, mslots, pairs.tolist(), mpairs, len(self.seqs))
        tables, lens = self.pool.block_table(self.seqs)
        mtab, mlens = self.model.block_table(self.seqs)
        assert tables.tolist() == mtab and lens.tolist() == mlens
        self.tables = torch.from_numpy(tables).cuda()
        self.lens = torch.from_numpy(lens).cuda()
        self.oracle_tables = np.asarray(mtab, dtype=np.int32)
        self.oracle_lens = np.asarray(mlens, dtype=np.int32)

    # -- running -----------------------------------------------------------------------------
    def refresh_tables(self):
        """Re-export both sides' block tables (after releases); they must agree bit-exactly."""
        tables, lens = self.pool.block_table(self.seqs)
        mtab, mlens = self.model.block_table(self.seqs)
        assert tables.tolist() == mtab and lens.tolist() == mlens
        self.tables = torch.from_numpy(tables).cuda()
        self.lens = torch.from_numpy(lens).cuda()
        self.oracle_tables = np.asarray(mtab, dtype=np.int32)
        self.oracle_lens = np.asarray(mlens, dtype=np.int32)

    def gpu_decode(self, partition_tokens: int = 0, q: Optional[torch.Tensor] = None,
                   tables: Optional[torch.Tensor] = None, lens: Optional[torch.Tensor] = None,
                   k_cache=None, v_cache=None, window: int = 0) -> torch.Tensor:
        q = self.q if q is None else q
        out = torch.full((self.n, self.Hq, self.D), float("nan"), dtype=torch.float32, device="cuda")
        nbytes = self.pool.decode_workspace_bytes(self.n, self.Hq, partition_tokens)
        ws = torch.full((max(nbytes, 16) // 4 + 4,), float("nan"), dtype=torch.float32, device="cuda")
        self.pool.paged_decode(out, q, self.k_cache if k_cache is None else k_cache,
                               self.v_cache if v_cache is None else v_cache,
                               self.tables if tables is None else tables, self.lens if lens is None else lens,
                               self.scale, partition_tokens=partition_tokens, workspace=ws, window=window)
        torch.cuda.synchronize()
        return out

    def oracle_decode(self, rows: Optional[List[int]] = None, window: int = 0) -> np.ndarray:
        assert self.host_cache
        return native.decode(self.q_stored, self.hk, self.hv, self.oracle_tables, self.oracle_lens, self.scale,
                             rows=rows, window=window)


def case_from_workload(name: str, seed: Optional[int] = None, host_cache: bool = True,
                       compact_host: bool = False) -> Case:
    w = synth.workload(name)
    seed = w.seed if seed is None else seed
    lens = synth.lengths(w, seed)
    NB = synth.pool_blocks(w, lens)
    kw = dict(lengths=lens, Hq=w.num_q_heads, Hkv=w.num_kv_heads, D=w.head_dim, B=w.block_size, dtype=w.dtype,
              num_blocks=NB, seed=seed, free_list=synth.free_list(NB, seed), host_cache=host_cache,
              compact_host=compact_host)
    if w.length_kind == "prefix":
        kw["prefix_trace"] = synth.prefix_trace(w, seed)
        kw["max_blocks"] = -(-int(lens.max()) // w.block_size) + 1
    return Case(**kw)


class Fp8Case:
    """An fp8 pool built on both sides: the library quantises bf16 K/V on the device; the oracle
    quantises the same decoded values on the host (oracle/fp8.py). Unwritten memory is poisoned
    (NaN codes and scales) on both sides."""

    def __init__(self, *, lengths, Hq, Hkv, B=16, D=128, seed=0, num_blocks=None, prefix_trace=None):
        from oracle import fp8 as ofp8
        self.ofp8 = ofp8
        self.Hq, self.Hkv, self.D, self.B, self.seed = Hq, Hkv, D, B, seed
        lengths = [int(x) for x in lengths]
        pages = sum(-(-L // B) for L in lengths)
        self.NB = num_blocks or max(pages + 4 * len(lengths) + 8, 16)
        self.MB = max(max(-(-L // B) for L in lengths), 1) + 4
        self.scale = 1.0 / math.sqrt(D)
        fl = synth.free_list(self.NB, seed)
        n_ids = len(lengths) + 1
        self.pool = pkv.Pool(1, Hkv, D, B, self.NB, n_ids, self.MB, pkv.FP8, initial_free_list=fl)
        self.model = am.PoolModel(self.NB, B, n_ids, self.MB, initial_free_list=fl)
        ks, vs, ss = self.pool.fp8_shapes()
        self.k8 = torch.full(ks, 0x7F, dtype=torch.uint8, device="cuda")
        self.v8 = torch.full(vs, 0x7F, dtype=torch.uint8, device="cuda")
        self.ksc = torch.full(ss, float("nan"), device="cuda")
        self.vsc = torch.full(ss, float("nan"), device="cuda")
        self.hk8 = np.full(ks, 0x7F, np.uint8)
        self.hv8 = np.full(vs, 0x7F, np.uint8)
        self.hks = np.full(ss, np.nan, np.float32)
        self.hvs = np.full(ss, np.nan, np.float32)
        self._stream = 0
        if prefix_trace is None:
            self.seqs = [self._append(-1, L) for L in lengths]
        else:
            children, root = {}, None
            for op in prefix_trace:
                if op[0] == "new":
                    root = self._append(-1, op[1])
                elif op[0] == "fork":
                    c = self.pool.fork(root)
                    assert self.model.fork(root) == (am.OK, c)
                    children[len(children)] = c
                elif op[0] == "free":
                    self.pool.free(root)
                    self.model.free_seq(root)
                else:
                    self._append(children[op[1]], op[2])
            self.seqs = [children[i] for i in range(len(children))]
        self.n = len(self.seqs)
        self.q_stored = synth.encode(synth.normal_f32((self.n, Hq, D), seed, 7), "bf16")
        self.q = to_device(self.q_stored, "bf16")
        self.refresh_tables()

    def refresh_tables(self):
        tables, lens = self.pool.block_table(self.seqs)
        mtab, mlens = self.model.block_table(self.seqs)
        assert tables.tolist() == mtab and lens.tolist() == mlens
        self.tables = torch.from_numpy(tables).cuda()
        self.lens = torch.from_numpy(lens).cuda()
        self.oracle_tables = np.asarray(mtab, dtype=np.int32)
        self.oracle_lens = np.asarray(mlens, dtype=np.int32)

    def _append(self, seq, n_tokens, magnitude=None):
        sid, slots, pairs = self.pool.alloc(seq, n_tokens)
        st, msid, mslots, mpairs = self.model.alloc(seq, n_tokens)
        assert st == am.OK and msid == sid and slots.tolist() == mslots and pairs == mpairs
        self._stream += 1
        kv = synth.normal_f32((2, n_tokens, self.Hkv, self.D), self.seed, 2000 + self._stream)
        # a spread of row magnitudes, and an all-zero row, exercise the per-row scales
        kv *= np.exp(synth.normal_f32((2, n_tokens, self.Hkv, 1), self.seed, 3000 + self._stream))
        if n_tokens > 3:
            kv[:, 3] = 0.0
        k, v = synth.encode(kv[0], "bf16"), synth.encode(kv[1], "bf16")
        if pairs:
            d_pairs = torch.tensor(np.asarray(pairs, dtype=np.int32).reshape(-1, 2), device="cuda")
            self.pool.copy_blocks_fp8([self.k8], [self.v8], [self.ksc], [self.vsc], d_pairs)
            for src, dst in mpairs:
                for arr in (self.hk8, self.hv8, self.hks, self.hvs):
                    arr[dst] = arr[src]
        if n_tokens:
            self.pool.reshape_and_cache_fp8(to_device(k, "bf16"), to_device(v, "bf16"),
                                            torch.from_numpy(slots.copy()).cuda(), self.k8, self.v8, self.ksc,
                                            self.vsc)
            self.ofp8.reshape_and_cache_fp8(self.hk8, self.hks, self.hv8, self.hvs, synth.bf16_bits_to_f32(k),
                                            synth.bf16_bits_to_f32(v), mslots)
        return sid

    def decode_step_append(self):
        slots, pairs = self.pool.append(self.seqs)
        st, mslots, mpairs = self.model.append(self.seqs)
        assert st == am.OK and slots.tolist() == mslots
        self._stream += 1
        kv = synth.normal_f32((2, self.n, self.Hkv, self.D), self.seed, 5000 + self._stream)
        k, v = synth.encode(kv[0], "bf16"), synth.encode(kv[1], "bf16")
        if len(pairs):
            self.pool.copy_blocks_fp8([self.k8], [self.v8], [self.ksc], [self.vsc],
                                      torch.from_numpy(np.ascontiguousarray(pairs, dtype=np.int32)).cuda())
            for src, dst in mpairs:
                for arr in (self.hk8, self.hv8, self.hks, self.hvs):
                    arr[dst] = arr[src]
        self.pool.reshape_and_cache_fp8(to_device(k, "bf16"), to_device(v, "bf16"), torch.from_numpy(slots).cuda(),
                                        self.k8, self.v8, self.ksc, self.vsc)
        self.ofp8.reshape_and_cache_fp8(self.hk8, self.hks, self.hv8, self.hvs, synth.bf16_bits_to_f32(k),
                                        synth.bf16_bits_to_f32(v), mslots)
        self.refresh_tables()

    def gpu_decode(self, partition_tokens=0, window=0):
        out = torch.full((self.n, self.Hq, self.D), float("nan"), device="cuda")
        nbytes = self.pool.decode_workspace_bytes(self.n, self.Hq, partition_tokens)
        ws = torch.empty(max(nbytes, 16) // 4 + 4, device="cuda")
        self.pool.paged_decode_fp8(out, self.q, self.k8, self.v8, self.ksc, self.vsc, self.tables, self.lens,
                                   self.scale, window=window, partition_tokens=partition_tokens, workspace=ws)
        torch.cuda.synchronize()
        return out

    def oracle_decode(self, window=0):
        K, V = self.ofp8.dequantize_pool(self.hk8, self.hks, self.hv8, self.hvs)
        return native.decode(self.q_stored, K, V, self.oracle_tables, self.oracle_lens, self.scale, window=window)
