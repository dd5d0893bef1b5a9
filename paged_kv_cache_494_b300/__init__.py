"""Python binding of libpagedkv: argument marshalling over the C ABI in include/pagedkv.h.

Every step of the paged-KV hot path (slot assignment, cache write, block copy, paged decode)
runs inside ``libpagedkv.so``: the host allocator in C++, the rest in sm_103a CUDA kernels.
This module only converts Python/NumPy/torch arguments into pointers and sizes. Importing
it fails loudly when the library has not been built; there is no fallback implementation.

torch is used for device memory and streams only: device arguments are CUDA tensors (or raw
device addresses as ints) and operations are enqueued on ``torch.cuda.current_stream()``
unless a stream is given.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

__all__ = ["Pool", "PagedKVError", "lib", "LIB_PATH", "F32", "BF16", "FP8", "status_string", "last_error",
           "EXPORTED_SYMBOLS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python paged_kv_cache_494_b300/build.py` "
                      "(the CUDA library is required; there is no fallback)")

lib = ctypes.CDLL(LIB_PATH)

F32, BF16, FP8 = 0, 1, 2
OK, ERR_INVALID, ERR_NO_BLOCKS, ERR_NO_SEQ, ERR_CUDA, ERR_DEVICE_BOUNDS, ERR_CAPACITY, ERR_DEVICE_TIMEOUT = (
    0, -1, -2, -3, -4, -5, -6, -7)
ERR_SCRATCH_TOO_SMALL = -8
STATIC_SCRATCH_BYTES = 16 << 20

_i32, _i64, _vp, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
_pi32, _pi64 = ctypes.POINTER(_i32), ctypes.POINTER(_i64)


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_layers", _i32), ("num_kv_heads", _i32), ("head_dim", _i32), ("block_size", _i32),
                ("num_blocks", _i32), ("max_seqs", _i32), ("max_blocks_per_seq", _i32), ("dtype", _i32),
                ("initial_free_list", _pi32), ("fail_after_n_allocs", _i32)]


class Stats(ctypes.Structure):
    _fields_ = [("num_free", _i32), ("num_used", _i32), ("num_shared", _i32), ("num_seqs", _i32),
                ("num_cow", _i64), ("num_tokens", _i64)]


_SIGS = {
    "pkv_version": (ctypes.c_int, []),
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_pool_create": (ctypes.c_int, [ctypes.POINTER(PoolDesc), ctypes.POINTER(_vp)]),
    "pkv_pool_destroy": (None, [_vp]),
    "pkv_bytes_per_token": (_i64, [_vp]),
    "pkv_layer_cache_bytes": (_i64, [_vp]),
    "pkv_layer_scale_bytes": (_i64, [_vp]),
    "pkv_alloc": (ctypes.c_int, [_vp, _i32, _i32, _pi32, _pi64, _pi32, _pi32]),
    "pkv_append": (ctypes.c_int, [_vp, _pi32, _i32, _pi64, _pi32, _pi32]),
    "pkv_fork": (ctypes.c_int, [_vp, _i32, _pi32]),
    "pkv_free": (ctypes.c_int, [_vp, _i32]),
    "pkv_block_table": (ctypes.c_int, [_vp, _pi32, _i32, _pi32, _pi32]),
    "pkv_release_before": (ctypes.c_int, [_vp, _i32, _i32, _pi32]),
    "pkv_alloc_prefix": (ctypes.c_int, [_vp, ctypes.c_uint64, _pi32, _i32, _pi32, _pi64, _pi32]),
    "pkv_prefix_evict": (ctypes.c_int, [_vp, _i32, _pi32]),
    "pkv_prefix_stats": (ctypes.c_int, [_vp, _pi32, _pi32]),
    "pkv_pool_stats": (ctypes.c_int, [_vp, ctypes.POINTER(Stats)]),
    "pkv_shared_prefix_blocks": (ctypes.c_int, [_vp, _pi32, _i32, _pi32]),
    "pkv_export_state": (ctypes.c_int, [_vp, _pi32, _pi32, _pi32]),
    "pkv_reshape_and_cache": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp]),
    "pkv_copy_blocks": (ctypes.c_int, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, _i32, _vp]),
    "pkv_paged_decode": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float, _i32, _vp,
                                        _sz, _vp]),
    "pkv_paged_decode_window": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float,
                                               _i32, _i32, _vp, _sz, _vp]),
    "pkv_decode_workspace_bytes": (_sz, [_vp, _i32, _i32, _i32]),
    "pkv_paged_decode_shared_prefix": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float,
                                                      _i32, _vp, _sz, _vp]),
    "pkv_decode_shared_prefix_workspace_bytes": (_sz, [_vp, _i32, _i32, _i32]),
    "pkv_reshape_and_cache_fp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp]),
    "pkv_copy_blocks_fp8": (ctypes.c_int, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                           ctypes.POINTER(_vp), _vp, _i32, _vp]),
    "pkv_paged_decode_fp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float,
                                            _i32, _i32, _vp, _sz, _vp]),
    "pkv_paged_prefill": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, ctypes.c_float,
                                         _i32, _vp]),
    "pkv_paged_decode_static": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float, _i32,
                                               _vp]),
    "pkv_last_error": (ctypes.c_int, [_vp]),
    "pkv_pool_set_error_word": (ctypes.c_int, [_vp, _vp]),
    "pkv_stream_error": (ctypes.c_int, [_vp, _vp]),
    "pkv_selftest_wait_timeout": (ctypes.c_int, [_vp, _vp]),
}
EXPORTED_SYMBOLS = tuple(_SIGS)
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class PagedKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


def status_string(status: int) -> str:
    return lib.pkv_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise PagedKVError(status, where)


def _i32p(a: np.ndarray):
    return a.ctypes.data_as(_pi32)


def _i64p(a: np.ndarray):
    return a.ctypes.data_as(_pi64)


def _dev(x) -> int:
    """Device address of a CUDA tensor (or an int address)."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def last_error() -> int:
    """Synchronise the device and return (and clear) the status recorded by kernels."""
    return lib.pkv_last_error(None)


class Pool:
    """A block pool: host allocator state plus the layout of the caller's device caches."""

    def __init__(self, num_layers: int, num_kv_heads: int, head_dim: int, block_size: int, num_blocks: int,
                 max_seqs: int, max_blocks_per_seq: int, dtype: int = BF16,
                 initial_free_list: Optional[Sequence[int]] = None, fail_after_n_allocs: int = -1):
        self._free_list = None
        fl = None
        if initial_free_list is not None:
            self._free_list = np.ascontiguousarray(initial_free_list, dtype=np.int32)
            if self._free_list.size != num_blocks:
                raise ValueError("initial_free_list must hold num_blocks entries")
            fl = _i32p(self._free_list)
        self.desc = PoolDesc(num_layers, num_kv_heads, head_dim, block_size, num_blocks, max_seqs,
                             max_blocks_per_seq, dtype, fl, fail_after_n_allocs)
        h = _vp()
        _check(lib.pkv_pool_create(ctypes.byref(self.desc), ctypes.byref(h)), "pkv_pool_create")
        self._h = h
        self.num_layers, self.num_kv_heads, self.head_dim = num_layers, num_kv_heads, head_dim
        self.block_size, self.num_blocks, self.max_seqs = block_size, num_blocks, max_seqs
        self.max_blocks_per_seq, self.dtype = max_blocks_per_seq, dtype

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib.pkv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    # -- sizes ---------------------------------------------------------------------------------
    @property
    def bytes_per_token(self) -> int:
        return lib.pkv_bytes_per_token(self._h)

    @property
    def layer_cache_bytes(self) -> int:
        return lib.pkv_layer_cache_bytes(self._h)

    @property
    def layer_scale_bytes(self) -> int:
        return lib.pkv_layer_scale_bytes(self._h)

    def cache_shape(self) -> Tuple[int, int, int, int]:
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    def fp8_shapes(self):
        """fp8 pools: (k_cache [NB][Hkv][B][D], v_cache [NB][Hkv][D][B], scales [NB][Hkv][B]) shapes."""
        NB, H, B, D = self.cache_shape()
        return (NB, H, B, D), (NB, H, D, B), (NB, H, B)

    # -- allocator -----------------------------------------------------------------------------
    def alloc_raw(self, seq: int, n_tokens: int) -> Tuple[int, int, np.ndarray, List[Tuple[int, int]]]:
        """pkv_alloc without raising: (status, seq_id, slots, cow_pairs)."""
        sid = _i32(-1)
        slots = np.zeros(max(int(n_tokens), 1), dtype=np.int64)
        pair = np.zeros(2, dtype=np.int32)
        ncow = _i32(0)
        st = lib.pkv_alloc(self._h, int(seq), int(n_tokens), ctypes.byref(sid), _i64p(slots), _i32p(pair),
                           ctypes.byref(ncow))
        if st != OK:
            return st, -1, np.zeros(0, dtype=np.int64), []
        pairs = [(int(pair[0]), int(pair[1]))] if ncow.value else []
        return st, sid.value, slots[:max(int(n_tokens), 0)], pairs

    def alloc(self, seq: int, n_tokens: int) -> Tuple[int, np.ndarray, List[Tuple[int, int]]]:
        st, sid, slots, pairs = self.alloc_raw(seq, n_tokens)
        _check(st, "pkv_alloc")
        return sid, slots, pairs

    def append_raw(self, seqs: Iterable[int]) -> Tuple[int, np.ndarray, np.ndarray]:
        s = np.ascontiguousarray(list(seqs), dtype=np.int32)
        n = s.size
        slots = np.zeros(max(n, 1), dtype=np.int64)
        pairs = np.zeros(max(2 * n, 2), dtype=np.int32)
        ncow = _i32(0)
        st = lib.pkv_append(self._h, _i32p(s), n, _i64p(slots), _i32p(pairs), ctypes.byref(ncow))
        if st != OK:
            return st, np.zeros(0, dtype=np.int64), np.zeros((0, 2), dtype=np.int32)
        return st, slots[:n], pairs[:2 * ncow.value].reshape(-1, 2)

    def append(self, seqs: Iterable[int]) -> Tuple[np.ndarray, np.ndarray]:
        st, slots, pairs = self.append_raw(seqs)
        _check(st, "pkv_append")
        return slots, pairs

    def fork_raw(self, parent: int) -> Tuple[int, int]:
        c = _i32(-1)
        st = lib.pkv_fork(self._h, int(parent), ctypes.byref(c))
        return st, (c.value if st == OK else -1)

    def fork(self, parent: int) -> int:
        st, c = self.fork_raw(parent)
        _check(st, "pkv_fork")
        return c

    def free_raw(self, seq: int) -> int:
        return lib.pkv_free(self._h, int(seq))

    def free(self, seq: int) -> None:
        _check(self.free_raw(seq), "pkv_free")

    def release_before_raw(self, seq: int, position: int) -> Tuple[int, int]:
        n = _i32(0)
        st = lib.pkv_release_before(self._h, int(seq), int(position), ctypes.byref(n))
        return st, n.value

    def release_before(self, seq: int, position: int) -> int:
        """Sliding window: release the blocks of ``seq`` that lie entirely before ``position``."""
        st, n = self.release_before_raw(seq, position)
        _check(st, "pkv_release_before")
        return n

    def alloc_prefix_raw(self, namespace: int, tokens: Sequence[int]) -> Tuple[int, int, np.ndarray, int]:
        """pkv_alloc_prefix without raising: (status, seq, slots, n_cached_tokens)."""
        tok = np.ascontiguousarray(list(tokens), dtype=np.int32)
        slots = np.zeros(max(tok.size, 1), dtype=np.int64)
        sid, ncached = _i32(-1), _i32(0)
        st = lib.pkv_alloc_prefix(self._h, ctypes.c_uint64(int(namespace) & 0xFFFFFFFFFFFFFFFF),
                                  _i32p(tok) if tok.size else None, tok.size, ctypes.byref(sid), _i64p(slots),
                                  ctypes.byref(ncached))
        if st != OK:
            return st, -1, np.zeros(0, dtype=np.int64), 0
        return st, sid.value, slots[:tok.size], ncached.value

    def alloc_prefix(self, namespace: int, tokens: Sequence[int]) -> Tuple[int, np.ndarray, int]:
        st, sid, slots, ncached = self.alloc_prefix_raw(namespace, tokens)
        _check(st, "pkv_alloc_prefix")
        return sid, slots, ncached

    def prefix_evict(self, max_blocks: int) -> int:
        n = _i32(0)
        _check(lib.pkv_prefix_evict(self._h, int(max_blocks), ctypes.byref(n)), "pkv_prefix_evict")
        return n.value

    def prefix_stats(self) -> Tuple[int, int]:
        a, b = _i32(0), _i32(0)
        _check(lib.pkv_prefix_stats(self._h, ctypes.byref(a), ctypes.byref(b)), "pkv_prefix_stats")
        return a.value, b.value

    def block_table(self, seqs: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
        s = np.ascontiguousarray(list(seqs), dtype=np.int32)
        tables = np.zeros((max(s.size, 1), self.max_blocks_per_seq), dtype=np.int32)
        lens = np.zeros(max(s.size, 1), dtype=np.int32)
        _check(lib.pkv_block_table(self._h, _i32p(s), s.size, _i32p(tables), _i32p(lens)), "pkv_block_table")
        return tables[:s.size], lens[:s.size]

    def shared_prefix_blocks(self, seqs: Sequence[int]) -> int:
        """pkv_shared_prefix_blocks: leading full blocks that all of `seqs` share physically."""
        s = np.ascontiguousarray(list(seqs), dtype=np.int32)
        out = _i32(0)
        _check(lib.pkv_shared_prefix_blocks(self._h, _i32p(s), s.size, ctypes.byref(out)),
               "pkv_shared_prefix_blocks")
        return out.value

    def stats(self) -> dict:
        st = Stats()
        _check(lib.pkv_pool_stats(self._h, ctypes.byref(st)), "pkv_pool_stats")
        return {k: getattr(st, k) for k, _ in Stats._fields_}

    def export_state(self) -> Tuple[List[int], List[int]]:
        rc = np.zeros(self.num_blocks, dtype=np.int32)
        fl = np.zeros(self.num_blocks, dtype=np.int32)
        nf = _i32(0)
        _check(lib.pkv_export_state(self._h, _i32p(rc), _i32p(fl), ctypes.byref(nf)), "pkv_export_state")
        return rc.tolist(), fl[:nf.value].tolist()

    # -- device operations -------------------------------------------------------------------------
    def reshape_and_cache(self, k, v, slots, k_cache, v_cache, stream=None) -> None:
        n = int(slots.shape[0])
        _check(lib.pkv_reshape_and_cache(self._h, _dev(k), _dev(v), _dev(slots), n, _dev(k_cache), _dev(v_cache),
                                         _stream(stream)), "pkv_reshape_and_cache")

    def copy_blocks(self, k_caches: Sequence, v_caches: Sequence, pairs, stream=None) -> None:
        L = self.num_layers
        if len(k_caches) != L or len(v_caches) != L:
            raise ValueError("one K and one V cache per layer")
        kp = (_vp * L)(*[_dev(t) for t in k_caches])
        vp = (_vp * L)(*[_dev(t) for t in v_caches])
        n = int(pairs.shape[0]) if pairs is not None else 0
        _check(lib.pkv_copy_blocks(self._h, kp, vp, _dev(pairs) if n else 0, n, _stream(stream)), "pkv_copy_blocks")

    def decode_workspace_bytes(self, n_seqs: int, num_q_heads: int, partition_tokens: int = 0) -> int:
        return int(lib.pkv_decode_workspace_bytes(self._h, int(n_seqs), int(num_q_heads), int(partition_tokens)))

    def paged_decode(self, out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                     partition_tokens: int = 0, workspace=None, stream=None, window: int = 0) -> None:
        """pkv_paged_decode, or pkv_paged_decode_window when window > 0."""
        n_seqs, num_q_heads = int(q.shape[0]), int(q.shape[1])
        ws_bytes = 0 if workspace is None else int(workspace.numel() * workspace.element_size())
        if window > 0:
            _check(lib.pkv_paged_decode_window(self._h, _dev(out), _dev(q), _dev(k_cache), _dev(v_cache),
                                               _dev(block_tables), _dev(context_lens), n_seqs, num_q_heads,
                                               float(scale), int(window), int(partition_tokens), _dev(workspace),
                                               ws_bytes, _stream(stream)), "pkv_paged_decode_window")
            return
        _check(lib.pkv_paged_decode(self._h, _dev(out), _dev(q), _dev(k_cache), _dev(v_cache), _dev(block_tables),
                                    _dev(context_lens), n_seqs, num_q_heads, float(scale), int(partition_tokens),
                                    _dev(workspace), ws_bytes, _stream(stream)), "pkv_paged_decode")

    def shared_prefix_workspace_bytes(self, n_seqs: int, num_q_heads: int, prefix_blocks: int) -> int:
        return int(lib.pkv_decode_shared_prefix_workspace_bytes(self._h, int(n_seqs), int(num_q_heads),
                                                                int(prefix_blocks)))

    def paged_decode_shared_prefix(self, out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                                   prefix_blocks: int, workspace=None, stream=None) -> None:
        """pkv_paged_decode_shared_prefix: decode for a batch whose tables all start with the same
        prefix_blocks blocks; the shared part is read once for the batch."""
        n_seqs, num_q_heads = int(q.shape[0]), int(q.shape[1])
        ws_bytes = 0 if workspace is None else int(workspace.numel() * workspace.element_size())
        _check(lib.pkv_paged_decode_shared_prefix(self._h, _dev(out), _dev(q), _dev(k_cache), _dev(v_cache),
                                                  _dev(block_tables), _dev(context_lens), n_seqs, num_q_heads,
                                                  float(scale), int(prefix_blocks), _dev(workspace), ws_bytes,
                                                  _stream(stream)), "pkv_paged_decode_shared_prefix")

    def reshape_and_cache_fp8(self, k, v, slots, k_cache, v_cache, k_scale, v_scale, stream=None) -> None:
        n = int(slots.shape[0])
        _check(lib.pkv_reshape_and_cache_fp8(self._h, _dev(k), _dev(v), _dev(slots), n, _dev(k_cache), _dev(v_cache),
                                             _dev(k_scale), _dev(v_scale), _stream(stream)),
               "pkv_reshape_and_cache_fp8")

    def copy_blocks_fp8(self, k_caches, v_caches, k_scales, v_scales, pairs, stream=None) -> None:
        L = self.num_layers
        arr = lambda ts: (_vp * L)(*[_dev(t) for t in ts])
        n = int(pairs.shape[0]) if pairs is not None else 0
        _check(lib.pkv_copy_blocks_fp8(self._h, arr(k_caches), arr(v_caches), arr(k_scales), arr(v_scales),
                                       _dev(pairs) if n else 0, n, _stream(stream)), "pkv_copy_blocks_fp8")

    def paged_decode_fp8(self, out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale: float,
                         window: int = 0, partition_tokens: int = 0, workspace=None, stream=None) -> None:
        n_seqs, num_q_heads = int(q.shape[0]), int(q.shape[1])
        ws_bytes = 0 if workspace is None else int(workspace.numel() * workspace.element_size())
        _check(lib.pkv_paged_decode_fp8(self._h, _dev(out), _dev(q), _dev(k_cache), _dev(v_cache), _dev(k_scale),
                                        _dev(v_scale), _dev(block_tables), _dev(context_lens), n_seqs, num_q_heads,
                                        float(scale), int(window), int(partition_tokens), _dev(workspace), ws_bytes,
                                        _stream(stream)), "pkv_paged_decode_fp8")

    def paged_prefill(self, out, q, k_cache, v_cache, block_tables, context_lens, cu_q, scale: float,
                      window: int = 0, stream=None) -> None:
        """pkv_paged_prefill: causal attention of the last q_len_b positions of each sequence."""
        n_seqs = int(context_lens.shape[0])
        total_q, num_q_heads = int(q.shape[0]), int(q.shape[1])
        _check(lib.pkv_paged_prefill(self._h, _dev(out), _dev(q), _dev(k_cache), _dev(v_cache), _dev(block_tables),
                                     _dev(context_lens), _dev(cu_q), n_seqs, total_q, num_q_heads, float(scale),
                                     int(window), _stream(stream)), "pkv_paged_prefill")

    def paged_decode_static(self, out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                            partition_tokens: int = 0, stream=None) -> None:
        """pkv_paged_decode_static: like paged_decode, with the library's built-in scratch instead of a
        caller workspace (for callers that must not allocate device memory). Calls that overlap on the
        GPU share that scratch and race; keep them on one stream."""
        n_seqs, num_q_heads = int(q.shape[0]), int(q.shape[1])
        _check(lib.pkv_paged_decode_static(self._h, _dev(out), _dev(q), _dev(k_cache), _dev(v_cache),
                                           _dev(block_tables), _dev(context_lens), n_seqs, num_q_heads,
                                           float(scale), int(partition_tokens), _stream(stream)),
               "pkv_paged_decode_static")

    def last_error(self) -> int:
        return lib.pkv_last_error(self._h)

    def set_error_word(self, word) -> None:
        """pkv_pool_set_error_word: the pool's kernels record errors into `word` (a one-element
        device int32 / uint32 tensor the caller zeroes), or the process-wide word again for None."""
        _check(lib.pkv_pool_set_error_word(self._h, _dev(word)), "pkv_pool_set_error_word")

    def stream_error(self, stream=None) -> int:
        """pkv_stream_error: read and clear the pool's error word in stream order; waits for that
        stream only."""
        return lib.pkv_stream_error(self._h, _stream(stream))
