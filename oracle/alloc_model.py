"""Block-pool allocator model: integers only, one Python statement per rule.

Test infrastructure only (see ``oracle/__init__``).

What the pages fix:
* the KV state of a request is a logical sequence of fixed-size blocks drawn from
  a shared pool as tokens arrive; a per-request block table maps logical order to
  physical blocks ("¿Cómo gestiona Paged Attention la caché KV...?", section
  "PagedAttention divide el estado KV en bloques de tamaño fijo"; "PagedAttention
  e vLLM", "Approfondimento tecnico"; "Paged Attention optimiza el uso de memoria
  en LLMs", paragraph on 16-token pages and the page table);
* when a request ends its unshared blocks return to the shared pool at once
  ("¿Cómo gestiona Paged Attention la caché KV...?", "Los bloques liberados regresan a
  un conjunto compartido");
* the runtime keeps reference counts ("La gestión de bloques tiene sus propios
  costes"); cancellation releases references without freeing pages still in use
  ("Servicio de modelos de lenguaje con un presupuesto de memoria" §8);
* identical prefixes (parallel samples, beams, a shared system prompt) point at the
  same physical pages and only the page where a request diverges is copied
  ("PagedAttention e vLLM", "Approfondimento tecnico"; "Paged Attention optimiza...",
  copy-on-write paragraph).

Readings where the pages are silent (the same rules are the library's ABI):
* free list order: blocks are handed out in the order of ``initial_free_list``
  (default 0..NB-1); a freed block goes on top and is handed out next (LIFO);
* a new or forked sequence takes the lowest unused id in [0, max_seqs);
* copy-on-write fires on an append to a sequence whose *partially filled* last
  block has refcount > 1: a fresh block is taken, the pair (old, new) is reported
  for the device copy, the old block loses one reference and the table points at
  the new block. Full shared blocks are never copied; the last holder (refcount 1)
  writes in place;
* slot of logical position t = table[t // B] * B + t % B;
* every call is all-or-nothing: if the free blocks cannot cover the whole call,
  nothing changes.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

OK = 0
ERR_INVALID = -1
ERR_NO_BLOCKS = -2
ERR_NO_SEQ = -3
ERR_CAPACITY = -6


class PoolModel:
    def __init__(self, num_blocks: int, block_size: int, max_seqs: int, max_blocks_per_seq: int,
                 initial_free_list: Optional[Sequence[int]] = None, fail_after_n_allocs: int = -1):
        self.NB = int(num_blocks)
        self.B = int(block_size)
        self.max_seqs = int(max_seqs)
        self.MB = int(max_blocks_per_seq)
        order = list(range(self.NB)) if initial_free_list is None else [int(b) for b in initial_free_list]
        if sorted(order) != list(range(self.NB)):
            raise ValueError("initial_free_list must be a permutation of [0, num_blocks)")
        # stack whose top (end of the list) is the next block handed out
        self.free: List[int] = list(reversed(order))
        self.refcount: List[int] = [0] * self.NB
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self.n_cow = 0
        self.fail_after = int(fail_after_n_allocs)
        self.n_allocs = 0

    # -- helpers -----------------------------------------------------------------
    def _new_id(self) -> int:
        for s in range(self.max_seqs):
            if s not in self.tables:
                return s
        return -1

    def _pop(self) -> int:
        b = self.free.pop()
        self.refcount[b] = 1
        return b

    # -- operations --------------------------------------------------------------
    def alloc(self, seq: int, n_tokens: int) -> Tuple[int, int, List[int], List[Tuple[int, int]]]:
        """Append n_tokens positions to ``seq`` (-1: a new sequence).

        Returns (status, seq_id, slots, cow_pairs)."""
        if n_tokens < 0:
            return ERR_INVALID, -1, [], []
        if seq == -1:
            sid = self._new_id()
            if sid < 0:
                return ERR_CAPACITY, -1, [], []
            table, length = [], 0
        else:
            if seq not in self.tables:
                return ERR_NO_SEQ, -1, [], []
            sid, table, length = seq, self.tables[seq], self.lens[seq]
        B = self.B
        new_blocks = -(-(length + n_tokens) // B) - (-(-length // B))
        if -(-(length + n_tokens) // B) > self.MB:
            return ERR_CAPACITY, -1, [], []
        cow = 1 if (n_tokens > 0 and length % B != 0 and self.refcount[table[-1]] > 1) else 0
        if self.fail_after >= 0 and self.n_allocs >= self.fail_after:
            return ERR_NO_BLOCKS, -1, [], []
        if new_blocks + cow > len(self.free):
            return ERR_NO_BLOCKS, -1, [], []
        # commit
        if seq == -1:
            self.tables[sid] = table = []
            self.lens[sid] = 0
        slots: List[int] = []
        pairs: List[Tuple[int, int]] = []
        for _ in range(n_tokens):
            if length % B == 0:
                table.append(self._pop())
            elif self.refcount[table[-1]] > 1:
                old = table[-1]
                dst = self._pop()
                pairs.append((old, dst))
                self.refcount[old] -= 1
                table[-1] = dst
            slots.append(table[length // B] * B + length % B)
            length += 1
        self.lens[sid] = length
        self.n_cow += len(pairs)
        self.n_allocs += 1
        return OK, sid, slots, pairs

    def append(self, seqs: Sequence[int]) -> Tuple[int, List[int], List[Tuple[int, int]]]:
        """One decode step: one position for each listed sequence, in order, all or nothing.

        Returns (status, slots, cow_pairs). Duplicate ids are invalid."""
        seqs = [int(s) for s in seqs]
        if len(set(seqs)) != len(seqs):
            return ERR_INVALID, [], []
        if any(s not in self.tables for s in seqs):
            return ERR_NO_SEQ, [], []
        if any(-(-(self.lens[s] + 1) // self.B) > self.MB for s in seqs):
            return ERR_CAPACITY, [], []
        if self.fail_after >= 0 and self.n_allocs >= self.fail_after:
            return ERR_NO_BLOCKS, [], []
        # count the blocks the step needs by replaying it on a scratch copy of the refcounts
        rc = list(self.refcount)
        need = 0
        for s in seqs:
            if self.lens[s] % self.B == 0:
                need += 1
            elif rc[self.tables[s][-1]] > 1:
                rc[self.tables[s][-1]] -= 1
                need += 1
        if need > len(self.free):
            return ERR_NO_BLOCKS, [], []
        slots, pairs = [], []
        for s in seqs:
            st, _, sl, pr = self.alloc(s, 1)
            assert st == OK
            self.n_allocs -= 1
            slots += sl
            pairs += pr
        self.n_allocs += 1
        return OK, slots, pairs

    def fork(self, parent: int) -> Tuple[int, int]:
        """New sequence sharing every block of ``parent`` (refcount + 1 each). Returns (status, child)."""
        if parent not in self.tables:
            return ERR_NO_SEQ, -1
        child = self._new_id()
        if child < 0:
            return ERR_CAPACITY, -1
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            if b >= 0:
                self.refcount[b] += 1
        return OK, child

    def release_before(self, seq: int, position: int) -> Tuple[int, int]:
        """Drop the sequence's reference to every block whose positions all lie before ``position``.

        Reading of the pages ("¿Cuánta memoria reservar para la caché KV?", "Adaptar el presupuesto a
        la estrategia de caché": a sliding window bounds the history a sequence keeps): those blocks
        are no longer attended to, so they are released in table order and their entries become -1;
        the length (and every remaining slot) is unchanged. Returns (status, references dropped)."""
        if seq not in self.tables:
            return ERR_NO_SEQ, 0
        if position < 0 or position > self.lens[seq]:
            return ERR_INVALID, 0
        t = self.tables[seq]
        released = 0
        for i in range(len(t)):
            if (i + 1) * self.B > position:
                break
            if t[i] < 0:
                continue
            self.refcount[t[i]] -= 1
            if self.refcount[t[i]] == 0:
                self.free.append(t[i])
            t[i] = -1
            released += 1
        return OK, released

    def free_seq(self, seq: int) -> int:
        """Drop one reference to every block of ``seq`` in table order; a block at zero is freed."""
        if seq not in self.tables:
            return ERR_NO_SEQ
        for b in self.tables.pop(seq):
            if b < 0:
                continue
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
        del self.lens[seq]
        return OK

    # -- views -------------------------------------------------------------------
    def block_table(self, seqs: Sequence[int]) -> Tuple[List[List[int]], List[int]]:
        rows, lens = [], []
        for s in seqs:
            t = self.tables[s]
            rows.append(t + [-1] * (self.MB - len(t)))
            lens.append(self.lens[s])
        return rows, lens

    def export_state(self) -> Tuple[List[int], List[int]]:
        """(refcounts, free blocks from the bottom of the stack to its top)."""
        return list(self.refcount), list(self.free)

    def stats(self) -> Dict[str, int]:
        return {
            "num_free": len(self.free),
            "num_used": sum(1 for r in self.refcount if r > 0),
            "num_shared": sum(1 for r in self.refcount if r > 1),
            "num_cow": self.n_cow,
            "num_seqs": len(self.tables),
            "num_tokens": sum(self.lens.values()),
        }


class PrefixCacheModel(PoolModel):
    """The pool plus a cache of full prompt blocks keyed by their content (integers, dictionaries).

    What the pages fix: "Servicio de modelos de lenguaje con un presupuesto de memoria" §8 — a cache
    key must identify every input that affects the state (model version, relevant configuration);
    reused pages must not expose another request's private continuation nor let it modify shared
    state; cancellation and eviction release references without freeing pages in use. "PagedAttention
    e vLLM", "Implementazione nel mondo reale" — a long system prompt shared by many requests is
    processed once. "Paged Attention optimiza el uso de memoria en LLMs" — requests that start from
    the same point use the same physical pages until they diverge.

    Readings (the library's ABI follows them):
    * key of prompt block i = (namespace, key entry of block i-1 (None for i = 0), the B token ids);
      only full blocks are cached; a lookup stops at the first miss;
    * each cache entry gets an id that is never reused; children refer to their parent by that id, so
      an entry whose parent was evicted can never be hit again;
    * the cache holds one reference on each cached block; when that is the last reference the block
      becomes evictable (queue order = the order in which blocks became evictable; a hit removes it);
    * evict(n) removes up to n evictable blocks, oldest first, and frees them.
    """

    def __init__(self, *args, **kwargs):
        super().__init__(*args, **kwargs)
        self.entries = {}          # (ns, parent_entry_id, tokens) -> (entry_id, block)
        self.entry_of_block = {}   # block -> key
        self.next_entry = 0
        self.evictable = []        # blocks whose only reference is the cache, oldest first

    def _drop(self, b: int):
        """One reference fewer on block b (shared by free_seq / release_before when caching)."""
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self.free.append(b)
        elif self.refcount[b] == 1 and b in self.entry_of_block:
            self.evictable.append(b)

    def free_seq(self, seq: int) -> int:
        if seq not in self.tables:
            return ERR_NO_SEQ
        for b in self.tables.pop(seq):
            if b >= 0:
                self._drop(b)
        del self.lens[seq]
        return OK

    def release_before(self, seq: int, position: int):
        if seq not in self.tables:
            return ERR_NO_SEQ, 0
        if position < 0 or position > self.lens[seq]:
            return ERR_INVALID, 0
        t = self.tables[seq]
        released = 0
        for i in range(len(t)):
            if (i + 1) * self.B > position:
                break
            if t[i] < 0:
                continue
            self._drop(t[i])
            t[i] = -1
            released += 1
        return OK, released

    def alloc_prefix(self, ns: int, tokens):
        """New sequence holding the prompt ``tokens``. Returns (status, seq, slots, n_cached_tokens):
        the K/V of positions < n_cached_tokens are already in cached blocks; the caller writes the rest."""
        tokens = [int(x) for x in tokens]
        n, B = len(tokens), self.B
        sid = self._new_id()
        if sid < 0:
            return ERR_CAPACITY, -1, [], 0
        if -(-n // B) > self.MB:
            return ERR_CAPACITY, -1, [], 0
        if self.fail_after >= 0 and self.n_allocs >= self.fail_after:
            return ERR_NO_BLOCKS, -1, [], 0
        # walk the cache: the leading full blocks that hit
        hits, parent = [], None
        for i in range(n // B):
            key = (ns, parent, tuple(tokens[i * B:(i + 1) * B]))
            if key not in self.entries:
                break
            eid, blk = self.entries[key]
            hits.append(blk)
            parent = eid
        need = -(-n // B) - len(hits)
        if need > len(self.free):
            return ERR_NO_BLOCKS, -1, [], 0
        # commit: shared blocks first, then fresh blocks (full ones are registered)
        table = []
        for blk in hits:
            if self.refcount[blk] == 1:
                self.evictable.remove(blk)
            self.refcount[blk] += 1
            table.append(blk)
        for i in range(len(hits), -(-n // B)):
            blk = self._pop()
            table.append(blk)
            if (i + 1) * B <= n:
                key = (ns, parent, tuple(tokens[i * B:(i + 1) * B]))
                self.entries[key] = (self.next_entry, blk)
                self.entry_of_block[blk] = key
                parent = self.next_entry
                self.next_entry += 1
                self.refcount[blk] += 1          # the cache's own reference
        self.tables[sid] = table
        self.lens[sid] = n
        self.n_allocs += 1
        slots = [table[t // B] * B + t % B for t in range(n)]
        return OK, sid, slots, len(hits) * B

    def evict(self, max_blocks: int) -> int:
        """Remove up to max_blocks evictable blocks from the cache (oldest first) and free them."""
        n = 0
        while n < max_blocks and self.evictable:
            blk = self.evictable.pop(0)
            key = self.entry_of_block.pop(blk)
            del self.entries[key]
            self.refcount[blk] -= 1
            self.free.append(blk)
            n += 1
        return n

    def prefix_stats(self):
        return len(self.entries), len(self.evictable)
