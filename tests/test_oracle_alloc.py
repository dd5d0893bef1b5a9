"""Pins of oracle/alloc_model.py: isolation semantics, conservation, the pages' figures."""
import json
import os

import numpy as np
import pytest

from oracle import alloc_model as am
from oracle import budget

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def check_invariants(p: am.PoolModel):
    """Conservation and reference counting, recomputed from scratch."""
    counts = [0] * p.NB
    for t in p.tables.values():
        for b in t:
            if b >= 0:
                counts[b] += 1
    assert counts == p.refcount
    assert len(set(p.free)) == len(p.free)
    assert all(p.refcount[b] == 0 for b in p.free)
    assert len(p.free) + sum(1 for r in p.refcount if r > 0) == p.NB
    for s, t in p.tables.items():
        assert len(t) == -(-p.lens[s] // p.B)


class Memory:
    """Simulated slot contents: applies the device side effects the allocator asks for."""

    def __init__(self, p: am.PoolModel):
        self.p = p
        self.slot = {}

    def apply(self, slots, pairs, values):
        B = self.p.B
        for src, dst in pairs:          # copy-on-write copies run before the writes
            for o in range(B):
                if src * B + o in self.slot:
                    self.slot[dst * B + o] = self.slot[src * B + o]
                else:
                    self.slot.pop(dst * B + o, None)
        for s, v in zip(slots, values):
            self.slot[s] = v

    def read(self, seq):
        t, L, B = self.p.tables[seq], self.p.lens[seq], self.p.B
        return [self.slot.get(t[i // B] * B + i % B) if t[i // B] >= 0 else "released" for i in range(L)]


def random_ops(seed, p: am.PoolModel, n_ops, max_append=40):
    """Drive the model with seeded random operations; yields (op, result)."""
    rng = np.random.default_rng(seed)
    for _ in range(n_ops):
        live = sorted(p.tables)
        r = rng.random()
        if r < 0.25 or not live:
            n = int(rng.integers(0, max_append))
            yield ("alloc", -1, n), p.alloc(-1, n)
        elif r < 0.6:
            s = int(rng.choice(live))
            n = int(rng.integers(0, max_append))
            yield ("alloc", s, n), p.alloc(s, n)
        elif r < 0.75:
            s = int(rng.choice(live))
            yield ("fork", s), p.fork(s)
        elif r < 0.8:
            s = int(rng.choice(live))
            pos = int(rng.integers(0, p.lens[s] + 1))
            yield ("release", s, pos), p.release_before(s, pos)
        else:
            s = int(rng.choice(live))
            yield ("free", s), p.free_seq(s)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("B", [1, 3, 16])
def test_isolation_and_order(seed, B):
    """Every live sequence reads back exactly its own logical history through its table.

    Pins the semantics the pages demand: the indirection changes where tokens live but not
    their order, and a reused or shared page never exposes another request's continuation.
    """
    p = am.PoolModel(num_blocks=120, block_size=B, max_seqs=24, max_blocks_per_seq=64,
                     initial_free_list=np.random.default_rng(seed).permutation(120))
    mem = Memory(p)
    history = {}
    counter = [0]
    for op, res in random_ops(seed, p, 400):
        if op[0] == "alloc":
            st, sid, slots, pairs = res
            if st != am.OK:
                continue
            vals = list(range(counter[0], counter[0] + op[2]))
            counter[0] += op[2]
            mem.apply(slots, pairs, vals)
            history.setdefault(sid, []).extend(vals) if op[1] != -1 else history.__setitem__(sid, vals)
            assert len(set(slots)) == len(slots)
        elif op[0] == "fork":
            st, child = res
            if st == am.OK:
                history[child] = list(history[op[1]])
        elif op[0] == "release":
            assert res[0] == am.OK
            B_ = p.B
            history[op[1]] = ["released" if (i // B_ + 1) * B_ <= op[2] or h == "released" else h
                              for i, h in enumerate(history[op[1]])]
        else:
            assert res == am.OK
            history.pop(op[1])
        check_invariants(p)
        for s in p.tables:
            assert mem.read(s) == history[s], (op, s)


def test_free_everything_returns_permutation():
    p = am.PoolModel(90, 16, 16, 32, initial_free_list=np.random.default_rng(1).permutation(90))
    for _ in random_ops(3, p, 300):
        pass
    for s in sorted(p.tables):
        assert p.free_seq(s) == am.OK
    assert sorted(p.free) == list(range(90))
    assert p.refcount == [0] * 90


def test_fork_then_free_restores_state():
    p = am.PoolModel(64, 16, 8, 16)
    st, a, _, _ = p.alloc(-1, 37)
    before = (list(p.refcount), list(p.free))
    st, c = p.fork(a)
    assert st == am.OK and p.refcount[p.tables[a][0]] == 2
    assert p.free_seq(c) == am.OK
    assert (list(p.refcount), list(p.free)) == before


def test_cancel_child_keeps_parent_pages():
    """Cancelling a request releases its references without freeing pages still in use."""
    p = am.PoolModel(64, 16, 8, 16)
    _, a, _, _ = p.alloc(-1, 40)
    _, c = p.fork(a)
    _, _, _, pairs = p.alloc(c, 5)          # child diverges: copies only the partial page
    assert len(pairs) == 1 and pairs[0][0] == p.tables[a][-1]
    assert p.free_seq(c) == am.OK
    assert all(p.refcount[b] == 1 for b in p.tables[a])
    assert not set(p.tables[a]) & set(p.free)


def test_500_tokens_on_16_token_pages():
    g = GOLD["pages_for_500"]
    p = am.PoolModel(64, g["page_tokens"], 4, 64)
    st, s, slots, _ = p.alloc(-1, g["tokens"])
    assert st == am.OK and len(p.tables[s]) == g["pages"]
    assert p.stats()["num_used"] * 16 - g["tokens"] == budget.tail_slots(500, 16) == 12


def test_mean_tail_through_allocator():
    """Allocating every length 1..512 on 16-token pages wastes (16-1)/2 = 7.5 slots on average."""
    waste = 0
    for T in range(1, 513):
        p = am.PoolModel(40, 16, 1, 40)
        p.alloc(-1, T)
        waste += p.stats()["num_used"] * 16 - T
    assert waste / 512 == 7.5


def test_shared_prompt_one_copy():
    """200-token prompt shared by 100 users: one copy of its pages instead of 100."""
    g = GOLD["shared_prompt"]
    B = 16
    p = am.PoolModel(2000, B, 128, 64)
    _, root, _, _ = p.alloc(-1, g["prompt_tokens"])
    kids = [p.fork(root)[1] for _ in range(g["users"])]
    prompt_pages = budget.pages(g["prompt_tokens"], B)
    assert p.stats()["num_used"] == prompt_pages                 # one copy shared by everyone
    classic = g["classic_copies"] * prompt_pages
    assert classic == 100 * 13
    # each user's first divergent token copies only the affected (partial) page
    for k in kids:
        _, _, _, pairs = p.alloc(k, 1)
        assert len(pairs) == 1
    full_shared = g["prompt_tokens"] // B
    assert p.stats()["num_used"] == full_shared + 1 + g["users"]
    assert p.stats()["num_shared"] == full_shared


@pytest.mark.parametrize("prompt,expect_cow", [(1024, False), (1016, True)])
def test_prefix_workload_cow_count(prompt, expect_cow):
    """128 children of one prompt, prompt released, suffixes U[0,512] appended in child order.

    With a partial last prompt block every child with a suffix copies it, except the last
    remaining holder which writes in place: A - 1 copies when all A = 128 children append,
    else A. A block-aligned prompt never copies.
    """
    rng = np.random.default_rng(0)
    suf = rng.integers(0, 513, size=128)
    p = am.PoolModel(7000, 16, 256, 128)
    _, root, _, _ = p.alloc(-1, prompt)
    kids = [p.fork(root)[1] for _ in range(128)]
    assert all(p.refcount[b] == 129 for b in p.tables[root])
    p.free_seq(root)
    assert all(p.refcount[b] == 128 for b in p.tables[kids[0]])
    total = 0
    for k, s in zip(kids, suf):
        st, _, _, pairs = p.alloc(k, int(s))
        assert st == am.OK
        total += len(pairs)
    A = int((suf > 0).sum())
    if expect_cow:
        assert total == (A - 1 if A == 128 else A)
    else:
        assert total == 0
    check_invariants(p)


def test_all_or_nothing_errors():
    p = am.PoolModel(4, 16, 2, 3, fail_after_n_allocs=-1)
    _, a, _, _ = p.alloc(-1, 40)            # 3 blocks
    snap = (list(p.refcount), list(p.free), dict(p.lens), {k: list(v) for k, v in p.tables.items()})
    assert p.alloc(a, 20)[0] == am.ERR_CAPACITY       # would need 4 blocks > max_blocks_per_seq
    assert p.alloc(-1, 17)[0] == am.ERR_NO_BLOCKS     # needs 2 blocks, 1 free
    _, b = p.fork(a)
    assert p.fork(a)[0] == am.ERR_CAPACITY           # no sequence id left
    assert p.alloc(7, 1)[0] == am.ERR_NO_SEQ
    assert p.free_seq(7) == am.ERR_NO_SEQ
    p.free_seq(b)
    assert (list(p.refcount), list(p.free), dict(p.lens), {k: list(v) for k, v in p.tables.items()}) == snap


def test_fault_injection_after_n_allocs():
    p = am.PoolModel(32, 16, 8, 8, fail_after_n_allocs=2)
    assert p.alloc(-1, 3)[0] == am.OK
    assert p.alloc(0, 3)[0] == am.OK
    snap = p.export_state()
    assert p.alloc(0, 3)[0] == am.ERR_NO_BLOCKS
    assert p.alloc(-1, 0)[0] == am.ERR_NO_BLOCKS
    assert p.export_state() == snap


def test_handout_order_and_lifo_reuse():
    order = [5, 2, 7, 0, 1, 3, 4, 6]
    p = am.PoolModel(8, 4, 4, 8, initial_free_list=order)
    _, a, slots, _ = p.alloc(-1, 9)
    assert p.tables[a] == [5, 2, 7]
    assert slots[:5] == [20, 21, 22, 23, 8]
    _, b, _, _ = p.alloc(-1, 1)
    assert p.tables[b] == [0]
    p.free_seq(a)
    _, c, _, _ = p.alloc(-1, 1)
    assert p.tables[c] == [7]               # the last block freed is handed out first


def test_release_before_frees_only_unshared_blocks():
    p = am.PoolModel(64, 16, 8, 16)
    _, a, _, _ = p.alloc(-1, 100)              # 7 blocks
    _, c = p.fork(a)
    st, n = p.release_before(a, 50)             # blocks 0..2 lie entirely before position 50
    assert st == am.OK and n == 3 and p.tables[a][:3] == [-1, -1, -1]
    assert all(p.refcount[b] == 1 for b in p.tables[c][:3])   # still held by the fork
    assert p.stats()["num_free"] == 64 - 7
    p.free_seq(c)
    assert p.stats()["num_free"] == 64 - 4     # the released blocks are free once nobody holds them
    assert p.release_before(a, 101) == (am.ERR_INVALID, 0)
    check_invariants(p)
    # appends continue at the same slots after a release
    st, _, slots, _ = p.alloc(a, 1)
    assert st == am.OK and slots == [p.tables[a][6] * 16 + 100 % 16]


# ---- the batched decode-step append (PoolModel.append) ---------------------------------------------
# A decode step appends one position to each of several sequences at once, all or nothing. What fixes
# its result is the single-sequence rule above, pinned by the isolation tests: the step must succeed
# exactly when appending one position to each sequence in turn would, and then leave the same state
# and report the same slots and copy-on-write pairs; otherwise it must fail and change nothing
# ("Servicio de modelos de lenguaje con un presupuesto de memoria" §8: shared pages, copied only where
# a request diverges; "PagedAttention e vLLM", "Approfondimento tecnico").

def _snapshot(p: am.PoolModel):
    return (list(p.refcount), list(p.free), dict(p.lens), {k: list(v) for k, v in p.tables.items()}, p.n_cow)


def sequential_append(p: am.PoolModel, seqs):
    """One position per sequence through single-sequence appends, on a copy of the model (no fault
    injection). Returns (status, slots, pairs, copy)."""
    import copy
    q = copy.deepcopy(p)
    q.fail_after = -1
    slots, pairs = [], []
    for s in seqs:
        st, _, sl, pr = q.alloc(s, 1)
        if st != am.OK:
            return st, [], [], q
        slots += sl
        pairs += pr
    return am.OK, slots, pairs, q


def tight_states(seed, B, n_states, model_cls=am.PoolModel):
    """Seeded pool states with shared partially filled blocks and almost no free blocks: a few
    prompts forked several times, some parents freed, the free list then filled down to 0-3 blocks
    by a filler sequence. Yields (model, sequences to append)."""
    rng = np.random.default_rng(seed)
    for _ in range(n_states):
        NB = int(rng.integers(30, 60))
        p = model_cls(NB, B, 40, 64, initial_free_list=rng.permutation(NB))
        roots = []
        for _ in range(int(rng.integers(1, 4))):
            st, r, _, _ = p.alloc(-1, int(rng.integers(1, 3 * B)))
            if st == am.OK:
                roots.append(r)
        for r in roots:
            for _ in range(int(rng.integers(1, 5))):
                p.fork(r)
        for r in roots:
            if rng.random() < 0.5:
                p.free_seq(r)
        keep = int(rng.integers(0, 4))
        if len(p.free) > keep:
            p.alloc(-1, (len(p.free) - keep) * B)       # filler: takes all but `keep` free blocks
        live = sorted(p.tables)
        k = int(rng.integers(1, len(live) + 1))
        yield p, [int(s) for s in rng.permutation(live)[:k]]


def append_pin_failures(model_cls):
    """Run the append pins against a model class; return the names of those that fail."""
    failed = []
    # hand-worked: a parent whose only block is partial (8 of 16), 3 forks, the parent freed -> the
    # children hold the block 3 times. Appending to all three copies twice (refcount 3 -> 2 -> 1) and
    # the last holder writes in place, so exactly 2 free blocks suffice; with 1 the step must fail.
    for nb_free, expect in ((2, am.OK), (1, am.ERR_NO_BLOCKS)):
        p = model_cls(1 + nb_free, 16, 8, 4)
        _, par, _, _ = p.alloc(-1, 8)
        kids = [p.fork(par)[1] for _ in range(3)]
        p.free_seq(par)
        before = _snapshot(p)
        st, slots, pairs = p.append(kids)
        if st != expect:
            failed.append(f"tight_{nb_free}")
            continue
        if expect == am.OK:
            blk = before[3][kids[0]][0]
            if not (len(pairs) == 2 and all(src == blk for src, _ in pairs)
                    and p.tables[kids[2]] == [blk] and slots[2] == blk * 16 + 8
                    and p.refcount[blk] == 1 and len(p.free) == 0):
                failed.append(f"tight_{nb_free}_result")
        elif _snapshot(p) != before:
            failed.append("tight_unchanged")
    # equivalence with single-sequence appends on seeded tight pools
    for seed in range(3):
        for B in (1, 4, 16):
            for p, seqs in tight_states(seed, B, 25, model_cls):
                before = _snapshot(p)
                exp_st, exp_slots, exp_pairs, q = sequential_append(p, seqs)
                try:
                    st, slots, pairs = p.append(seqs)
                except AssertionError:
                    st, slots, pairs = "raised", [], []
                if exp_st == am.OK:
                    ok = st == am.OK and list(slots) == exp_slots and list(pairs) == exp_pairs and \
                        _snapshot(p) == _snapshot(q)
                else:
                    ok = st == exp_st and _snapshot(p) == before
                if not ok:
                    failed.append("sequential")
                    break
            if "sequential" in failed:
                break
        if "sequential" in failed:
            break
    # duplicate ids are invalid and change nothing
    p = model_cls(16, 4, 4, 8)
    _, a, _, _ = p.alloc(-1, 3)
    before = _snapshot(p)
    try:
        st = p.append([a, a])[0]
    except AssertionError:
        st = "raised"
    if st != am.ERR_INVALID or _snapshot(p) != before:
        failed.append("duplicates")
    # fault injection counts one decode step as one call, however many sequences it appends to
    p = model_cls(32, 4, 4, 8, fail_after_n_allocs=4)
    _, a, _, _ = p.alloc(-1, 3)
    _, b, _, _ = p.alloc(-1, 5)                     # 2 calls
    if p.append([a, b])[0] != am.OK:                # the 3rd call
        failed.append("inject_step")
    elif p.alloc(a, 1)[0] != am.OK:                 # the 4th call is still allowed
        failed.append("inject_count")
    elif p.append([a, b])[0] != am.ERR_NO_BLOCKS:   # the 5th is refused
        failed.append("inject_refuse")
    return failed


def test_append_pins_hold_for_the_oracle():
    assert append_pin_failures(am.PoolModel) == []


def test_append_hand_worked_tight_pool():
    """The worked case on its own: 3 holders of one partial block, 2 free blocks -> 2 copies."""
    p = am.PoolModel(3, 16, 8, 4)
    _, par, _, _ = p.alloc(-1, 8)
    kids = [p.fork(par)[1] for _ in range(3)]
    blk = p.tables[par][0]
    p.free_seq(par)
    assert p.refcount[blk] == 3 and len(p.free) == 2
    st, slots, pairs = p.append(kids)
    assert st == am.OK
    assert [src for src, _ in pairs] == [blk, blk]
    assert sorted(dst for _, dst in pairs) == sorted({0, 1, 2} - {blk})
    assert p.tables[kids[2]] == [blk] and slots[2] == blk * 16 + 8
    assert p.stats()["num_cow"] == 2 and p.stats()["num_free"] == 0
    check_invariants(p)
