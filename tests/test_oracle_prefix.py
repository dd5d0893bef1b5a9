"""Pins of the prefix-cache model (oracle/alloc_model.PrefixCacheModel).

The key property the pages demand ("Servicio de modelos de lenguaje..." §8): a reused page never
exposes another request's continuation. Checked by simulating memory: the caller writes token ids
only for positions the cache did not already hold; every live sequence must read back exactly its
own tokens through its table, whatever was shared, evicted or freed in between.
"""
import json
import os

import numpy as np
import pytest

from oracle import alloc_model as am
from oracle import budget

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def check(p: am.PrefixCacheModel):
    counts = [0] * p.NB
    for t in p.tables.values():
        for b in t:
            if b >= 0:
                counts[b] += 1
    for b in p.entry_of_block:
        counts[b] += 1                       # the cache's own reference
    assert counts == p.refcount
    assert len(p.free) + sum(1 for r in p.refcount if r > 0) == p.NB
    assert all(p.refcount[b] == 1 for b in p.evictable)
    assert set(p.evictable) == {b for b in p.entry_of_block if p.refcount[b] == 1}
    assert len(p.entries) == len(p.entry_of_block)


def prompt(rng, vocab=3, max_len=60, base=None):
    n = int(rng.integers(0, max_len))
    toks = [int(x) for x in rng.integers(0, vocab, size=n)]
    return toks if base is None else base[:int(rng.integers(0, len(base) + 1))] + toks


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("B", [1, 4, 16])
def test_isolation_through_sharing_and_eviction(seed, B):
    rng = np.random.default_rng(seed)
    p = am.PrefixCacheModel(160, B, 24, 64, initial_free_list=rng.permutation(160))
    mem, mine = {}, {}
    system = [int(x) for x in rng.integers(0, 3, size=40)]     # a common "system prompt"
    for _ in range(300):
        r = rng.random()
        live = sorted(p.tables)
        if r < 0.45 or not live:
            ns = int(rng.integers(0, 2))
            toks = prompt(rng, base=system if rng.random() < 0.7 else None)
            st, sid, slots, ncached = p.alloc_prefix(ns, toks)
            if st != am.OK:
                assert p.evict(4) >= 0
                continue
            assert ncached % B == 0 and ncached <= len(toks)
            for i in range(ncached):                              # cached positions already hold K/V
                assert mem[slots[i]] == (ns, toks[i])
            for i in range(ncached, len(toks)):                   # the caller writes the rest
                mem[slots[i]] = (ns, toks[i])
            mine[sid] = [(ns, t) for t in toks]
        elif r < 0.6:
            s = int(rng.choice(live))
            st, _, slots, pairs = p.alloc(s, 3)
            if st != am.OK:
                continue
            for src, dst in pairs:
                for o in range(B):
                    if src * B + o in mem:
                        mem[dst * B + o] = mem[src * B + o]
            for sl in slots:
                mem[sl] = ("gen", s, len(mine[s]))
                mine[s].append(("gen", s, len(mine[s])))
        elif r < 0.7:
            s = int(rng.choice(live))
            st, c = p.fork(s)
            if st == am.OK:
                mine[c] = list(mine[s])
        elif r < 0.85:
            s = int(rng.choice(live))
            assert p.free_seq(s) == am.OK
            del mine[s]
        else:
            p.evict(int(rng.integers(0, 5)))
        check(p)
        for s, t in p.tables.items():
            got = [mem.get(t[i // B] * B + i % B) for i in range(p.lens[s])]
            assert got == mine[s]


def test_namespace_and_partial_blocks_never_shared():
    p = am.PrefixCacheModel(64, 4, 8, 16)
    toks = list(range(10))                                        # 2 full blocks + 2 tokens
    _, a, sa, na = p.alloc_prefix(1, toks)
    _, b, sb, nb = p.alloc_prefix(1, toks)
    _, c, sc, nc = p.alloc_prefix(2, toks)                        # other model/config identity
    assert (na, nb, nc) == (0, 8, 0)
    assert p.tables[a][:2] == p.tables[b][:2] and p.tables[a][2] != p.tables[b][2]
    assert not set(p.tables[c]) & set(p.tables[a])
    _, d, _, nd = p.alloc_prefix(1, [0, 1, 2, 3, 9, 9, 9, 9])     # diverges in block 1
    assert nd == 4 and p.tables[d][0] == p.tables[a][0] and p.tables[d][1] != p.tables[a][1]


def test_eviction_order_and_in_use_blocks():
    p = am.PrefixCacheModel(64, 4, 8, 16)
    _, a, _, _ = p.alloc_prefix(0, list(range(8)))                # blocks A0 A1 cached
    _, b, _, _ = p.alloc_prefix(0, [7] * 8)                       # blocks B0 B1 cached
    assert p.evict(10) == 0                                       # everything is in use
    p.free_seq(b)
    p.free_seq(a)
    assert p.prefix_stats() == (4, 4)
    order = list(p.evictable)
    assert p.evict(1) == 1 and p.free[-1] == order[0]             # oldest first, onto the free list
    _, c, _, nc = p.alloc_prefix(0, list(range(8)))               # its parent entry was evicted?
    # `order` starts with B's blocks (b was freed first): A's entries are intact and hit
    assert nc == 8
    p.free_seq(c)
    assert p.evict(100) == 3 and p.prefix_stats() == (0, 0)
    check(p)


def test_orphaned_entries_are_unreachable():
    p = am.PrefixCacheModel(64, 4, 8, 16)
    _, a, _, _ = p.alloc_prefix(0, list(range(8)))
    first = p.tables[a][0]
    p.free_seq(a)
    # evict the first block only (it became evictable first)
    assert p.evictable[0] == first and p.evict(1) == 1
    _, b, _, nb = p.alloc_prefix(0, list(range(8)))
    assert nb == 0                                                # the child entry is not reachable
    check(p)


def test_shared_system_prompt_stored_once():
    """200-token prompt, 100 users (the copy-on-write paragraph's example): one copy of its full
    pages; each user holds only the partial last page privately."""
    g = GOLD["shared_prompt"]
    B = 16
    p = am.PrefixCacheModel(2000, B, 128, 64)
    sys_prompt = list(range(g["prompt_tokens"]))
    hits = [p.alloc_prefix(0, sys_prompt)[3] for _ in range(g["users"])]
    full = g["prompt_tokens"] // B
    assert hits[0] == 0 and all(h == full * B for h in hits[1:])
    assert p.stats()["num_used"] == full + g["users"]             # 12 shared + 100 partial pages
    classic = g["users"] * budget.pages(g["prompt_tokens"], B)
    assert classic == 1300 and p.stats()["num_used"] < classic / 10
