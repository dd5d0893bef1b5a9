"""C++ host allocator (libpagedkv) vs the oracle allocator model: bit-exact on seeded traces.

Compares, after every operation: status codes, sequence ids, slots, copy-on-write pairs,
refcounts, the free list (bottom to top), every live block table and length, and the stats.
Host only: runs without a GPU.
"""
import numpy as np
import pytest

import paged_kv_cache_494_b300 as pkv
import synth
from oracle import alloc_model as am


def same_state(lib: pkv.Pool, m: am.PoolModel):
    assert lib.export_state() == m.export_state()
    live = sorted(m.tables)
    if live:
        t, l = lib.block_table(live)
        mt, ml = m.block_table(live)
        assert t.tolist() == mt and l.tolist() == ml
    if isinstance(m, am.PrefixCacheModel):
        assert lib.prefix_stats() == m.prefix_stats()
    s = lib.stats()
    ms = m.stats()
    for k in ("num_free", "num_used", "num_shared", "num_cow", "num_seqs", "num_tokens"):
        assert s[k] == ms[k], k


def drive(seed, NB, B, max_seqs, MB, n_ops, fail_after=-1, max_append=40):
    rng = np.random.default_rng(seed)
    perm = rng.permutation(NB)
    lib = pkv.Pool(1, 2, 64, B, NB, max_seqs, MB, pkv.F32, initial_free_list=perm, fail_after_n_allocs=fail_after)
    m = am.PrefixCacheModel(NB, B, max_seqs, MB, initial_free_list=perm, fail_after_n_allocs=fail_after)
    for _ in range(n_ops):
        live = sorted(m.tables)
        r = rng.random()
        if r < 0.08:
            ns = int(rng.integers(0, 2))
            toks = [int(x) for x in rng.integers(0, 2, size=int(rng.integers(0, 3 * B + 5)))]
            a = lib.alloc_prefix_raw(ns, toks)
            b = m.alloc_prefix(ns, toks)
            assert a[0] == b[0] and a[1] == b[1] and a[2].tolist() == b[2] and a[3] == b[3]
        elif r < 0.1:
            k = int(rng.integers(0, 4))
            assert lib.prefix_evict(k) == m.evict(k)
        elif r < 0.2 or not live:
            n = int(rng.integers(0, max_append))
            a = lib.alloc_raw(-1, n)
            b = m.alloc(-1, n)
            assert a[0] == b[0] and a[1] == b[1] and a[2].tolist() == b[2] and a[3] == b[3]
        elif r < 0.45:
            s = int(rng.choice(live)) if rng.random() < 0.95 else int(rng.integers(0, max_seqs + 2))
            n = int(rng.integers(0, max_append))
            a = lib.alloc_raw(s, n)
            b = m.alloc(s, n)
            assert a[0] == b[0] and a[1] == b[1] and a[2].tolist() == b[2] and a[3] == b[3]
        elif r < 0.6:
            k = int(rng.integers(1, len(live) + 1))
            seqs = [int(x) for x in rng.choice(live, size=k, replace=False)]
            if rng.random() < 0.05:
                seqs.append(seqs[0])            # duplicate id: invalid
            a = lib.append_raw(seqs)
            b = m.append(seqs)
            assert a[0] == b[0] and a[1].tolist() == b[1] and [tuple(p) for p in a[2].tolist()] == b[2]
        elif r < 0.75:
            s = int(rng.choice(live))
            assert lib.fork_raw(s) == m.fork(s)
        elif r < 0.8:
            s = int(rng.choice(live))
            pos = int(rng.integers(0, m.lens[s] + 2))
            assert lib.release_before_raw(s, pos) == m.release_before(s, pos)
        else:
            s = int(rng.choice(live)) if rng.random() < 0.97 else int(rng.integers(0, max_seqs + 2))
            assert lib.free_raw(s) == m.free_seq(s)
        same_state(lib, m)


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("B", [1, 3, 16, 32])
def test_random_traces(seed, B):
    drive(seed, NB=150, B=B, max_seqs=20, MB=40, n_ops=300)


@pytest.mark.parametrize("seed", range(4))
def test_tight_pool_and_fault_injection(seed):
    drive(100 + seed, NB=24, B=4, max_seqs=6, MB=10, n_ops=300, fail_after=150, max_append=12)


def test_prefix_workload_trace():
    """The shared-prefix workload's own trace (one prompt, 128 forks, prompt freed, suffixes)."""
    for name in ("prefix_cow_bf16", "prefix_cow_partial_bf16"):
        w = synth.workload(name)
        lens = synth.lengths(w)
        NB = synth.pool_blocks(w, lens)
        perm = synth.free_list(NB, w.seed)
        MB = -(-int(lens.max()) // w.block_size)
        lib = pkv.Pool(1, w.num_kv_heads, w.head_dim, w.block_size, NB, w.n_seqs + 1, MB, pkv.BF16,
                       initial_free_list=perm)
        m = am.PoolModel(NB, w.block_size, w.n_seqs + 1, MB, initial_free_list=perm)
        ids = {}
        for op in synth.prefix_trace(w):
            if op[0] == "new":
                a, b = lib.alloc_raw(-1, op[1]), m.alloc(-1, op[1])
                assert a[0] == b[0] == 0 and a[2].tolist() == b[2]
                root = b[1]
            elif op[0] == "fork":
                a, b = lib.fork_raw(root), m.fork(root)
                assert a == b
                ids[len(ids)] = b[1]
            elif op[0] == "free":
                assert lib.free_raw(root) == m.free_seq(root) == 0
            else:
                s = ids[op[1]]
                a, b = lib.alloc_raw(s, op[2]), m.alloc(s, op[2])
                assert a[0] == b[0] == 0 and a[2].tolist() == b[2] and a[3] == b[3]
        same_state(lib, m)
        # sharing structure: the prompt's full blocks, shared by all children (closed form), and the
        # brute-force count over the model's tables
        kids = [ids[i] for i in range(len(ids))]
        assert lib.shared_prefix_blocks(kids) == w.length_args[0] // w.block_size
        mt, ml = m.block_table(kids)
        k = 0
        while k < min(ml) // w.block_size and len({row[k] for row in mt}) == 1:
            k += 1
        assert lib.shared_prefix_blocks(kids) == k
        assert lib.shared_prefix_blocks(kids[:1]) == ml[0] // w.block_size


def test_shared_prefix_blocks_hand_worked():
    """Block 4: a 10-token prompt (2 full blocks + 2 tokens), two forks; child 0 appends 7 tokens (its
    first append copies the partial block), child 1 appends nothing. Shared full blocks: 2. Child 1
    alone: 10 // 4 = 2 full blocks. A fresh unrelated sequence shares none."""
    lib = pkv.Pool(1, 1, 8, 4, 32, 8, 8, pkv.BF16)
    root, _, _ = lib.alloc(-1, 10)
    c0, c1 = lib.fork(root), lib.fork(root)
    lib.alloc(c0, 7)
    assert lib.shared_prefix_blocks([c0, c1]) == 2
    assert lib.shared_prefix_blocks([c1]) == 2
    assert lib.shared_prefix_blocks([c0]) == 17 // 4
    other, _, _ = lib.alloc(-1, 12)
    assert lib.shared_prefix_blocks([c0, other]) == 0
    with pytest.raises(pkv.PagedKVError):
        lib.shared_prefix_blocks([])
    lib.free(other)
    with pytest.raises(pkv.PagedKVError) as e:              # a freed sequence id
        lib.shared_prefix_blocks([c0, other])
    assert e.value.status == pkv.ERR_NO_SEQ


def test_large_pool_constructs_fast():
    """An 80 GB-scale pool (610k blocks) with a seeded permutation."""
    perm = synth.free_list(610_000, 0)
    lib = pkv.Pool(1, 8, 128, 32, 610_000, 8, 1024, pkv.BF16, initial_free_list=perm)
    sid, slots, _ = lib.alloc(-1, 32768)
    t, l = lib.block_table([sid])
    assert l[0] == 32768 and t[0, 0] == perm[0] and t[0, 1023] == perm[1023]
