"""Paged decode on the GPU against the binary64 oracle on the same seeded inputs.

Tolerances (max abs error): 2e-3 for bf16 K/V with fp32 accumulation, 1e-5 for fp32.
Each side built its own block tables and caches (see gpu_cases.Case).
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
import synth
from oracle import native
from tests.gpu_cases import TOL, Case, case_from_workload, to_device

pytestmark = pytest.mark.gpu


def check(c: Case, out: torch.Tensor, ref=None):
    ref = c.oracle_decode() if ref is None else ref
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert err <= TOL[c.dtype], err
    return err


@pytest.fixture(params=["mma", "simt"])
def path(request, monkeypatch):
    """bf16 decode runs on tensor cores by default; PKV_DECODE_PATH=simt selects the CUDA-core path."""
    if request.param == "simt":
        monkeypatch.setenv("PKV_DECODE_PATH", "simt")
    else:
        monkeypatch.delenv("PKV_DECODE_PATH", raising=False)
    return request.param


@pytest.mark.parametrize("name", ["tiny_f32", "gqa5_bf16", "prefix_cow_bf16", "prefix_cow_partial_bf16"])
@pytest.mark.parametrize("partition_tokens", [0, 512, 64])
def test_workload_parity(name, partition_tokens, path):
    c = case_from_workload(name)
    check(c, c.gpu_decode(partition_tokens))
    assert pkv.last_error() == pkv.OK


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
def test_shapes_and_ragged_tails(dtype, D, G, path):
    if dtype == "f32" and (G == 7 or path == "simt"):
        pytest.skip("fp32 always runs on the CUDA-core path; G = 7 is bf16 only")
    lens = [0, 1, 2, 15, 16, 17, 33, 100, 257, 700]
    c = Case(lengths=lens, Hq=2 * G, Hkv=2, D=D, B=32 if G % 2 else 16, dtype=dtype, seed=G)
    for pt in (0, 32):
        out = c.gpu_decode(pt)
        check(c, out)
        assert torch.all(out[0] == 0)             # empty context gives a zero row
    assert pkv.last_error() == pkv.OK


def test_single_token_returns_v_row():
    c = Case(lengths=[1, 1, 1], Hq=8, Hkv=2, D=128, B=16, dtype="bf16", seed=5)
    out = c.gpu_decode()
    for b in range(3):
        blk = int(c.oracle_tables[b, 0])
        for j in range(8):
            v = c.hv[blk, j // 4, 0].astype(np.uint32) << 16
            assert np.array_equal(out[b, j].cpu().numpy(), v.view(np.float32))


def test_extreme_logits_stay_finite(path):
    c = Case(lengths=[300, 7, 1000], Hq=8, Hkv=2, D=128, B=16, dtype="bf16", seed=13)
    q = (torch.from_numpy(synth.bf16_bits_to_f32(c.q_stored)) * 100.0)
    q_stored = synth.to_bf16_bits(q.numpy())
    c.q_stored = q_stored
    out = c.gpu_decode(q=to_device(q_stored, "bf16"))
    check(c, out)


def test_permutation_invariance_bitwise(path):
    lens = [5, 300, 1, 77, 1024, 16]
    c1 = Case(lengths=lens, Hq=32, Hkv=8, D=128, B=16, dtype="bf16", seed=21, num_blocks=200)
    c2 = Case(lengths=lens, Hq=32, Hkv=8, D=128, B=16, dtype="bf16", seed=21, num_blocks=200,
              free_list=synth.free_list(200, 999))
    assert not np.array_equal(c1.oracle_tables, c2.oracle_tables)
    for pt in (0, 128):
        assert torch.equal(c1.gpu_decode(pt), c2.gpu_decode(pt))


def test_workspace_reused_by_consecutive_calls_bitwise(path):
    """One workspace serves many calls in a row, alternating split modes and problem sizes.

    Each call's arrival counters must ignore the counts its predecessors left behind, so every call
    returns exactly what it returns on a fresh NaN-filled workspace.
    """
    c = case_from_workload("gqa5_bf16", host_cache=False)
    nbytes = max(c.pool.decode_workspace_bytes(c.n, c.Hq, pt) for pt in (0, 512, 64))

    def run(pt, n, ws):
        out = torch.full((n, c.Hq, c.D), float("nan"), dtype=torch.float32, device="cuda")
        c.pool.paged_decode(out, c.q[:n], c.k_cache, c.v_cache, c.tables[:n], c.lens[:n], c.scale,
                            partition_tokens=pt, workspace=ws)
        torch.cuda.synchronize()
        return out

    def nan_ws():
        return torch.full((nbytes // 4 + 4,), float("nan"), dtype=torch.float32, device="cuda")

    sizes = (c.n, c.n // 2)                         # a shorter batch leaves stale counters behind
    fresh = {(pt, n): run(pt, n, nan_ws()) for pt in (0, 512, 64) for n in sizes}
    ws = nan_ws()
    for it in range(12):
        pt, n = (0, 512, 64)[it % 3], sizes[it % 2]
        assert torch.equal(run(pt, n, ws), fresh[(pt, n)]), (it, pt, n)


@pytest.mark.parametrize("name", ["tiny_f32", "gqa5_bf16", "prefix_cow_partial_bf16"])
def test_many_way_splits(name, monkeypatch):
    """One chunk per warp at least (PKV_DECODE_MIN_CHUNKS=1): units cut into dozens of parts."""
    monkeypatch.setenv("PKV_DECODE_MIN_CHUNKS", "1")
    c = case_from_workload(name)
    check(c, c.gpu_decode(0))


def test_shared_prefix_equals_duplicated_bitwise():
    """Same logical data: prefix pages shared through forks vs private copies written separately."""
    B, H, D = 16, 8, 128
    shared = Case(lengths=[48], Hq=32, Hkv=H, D=D, B=B, dtype="bf16", seed=31, num_blocks=64, max_blocks=8)
    child = shared.pool.fork(shared.seqs[0])
    st, mchild = shared.model.fork(shared.seqs[0])
    assert mchild == child
    tables, lens = shared.pool.block_table([shared.seqs[0], child])
    assert tables[0, :3].tolist() == tables[1, :3].tolist()
    spare = [b for b in range(64) if b not in set(tables[0].tolist())][:3]
    dup_tables = tables.copy()
    dup_tables[1, :3] = spare
    for i, dst in enumerate(spare):                      # private copies of the same pages
        shared.k_cache[dst] = shared.k_cache[int(tables[0, i])]
        shared.v_cache[dst] = shared.v_cache[int(tables[0, i])]
    q = torch.cat([shared.q, shared.q])
    shared.n = 2
    lens_d = torch.from_numpy(lens).cuda()
    a = shared.gpu_decode(q=q, tables=torch.from_numpy(tables).cuda(), lens=lens_d)
    b = shared.gpu_decode(q=q, tables=torch.from_numpy(dup_tables).cuda(), lens=lens_d)
    assert torch.equal(a, b)
    # the two rows hold the same data at different batch positions; the balanced split may cut their
    # units differently, so they agree to rounding, not bitwise
    assert float((a[0] - a[1]).abs().max()) <= 1e-5


def test_decode_steps_append_then_attend(path):
    c = Case(lengths=[1, 15, 16, 200, 0, 33], Hq=32, Hkv=8, D=128, B=16, dtype="bf16", seed=41, num_blocks=80)
    for step in range(18):
        c.decode_step_append()
        if step % 6 == 5:
            check(c, c.gpu_decode())
    assert pkv.last_error() == pkv.OK


def test_bad_block_id_reported_not_faulted():
    c = Case(lengths=[40, 40], Hq=8, Hkv=2, D=128, B=16, dtype="bf16", seed=51)
    bad = c.tables.clone()
    bad[1, 1] = c.NB + 5
    out = c.gpu_decode(tables=bad)
    assert pkv.last_error() == pkv.ERR_DEVICE_BOUNDS
    ref = c.oracle_decode()
    assert np.max(np.abs(out[0].double().cpu().numpy() - ref[0])) <= 2e-3   # untouched sequence is right
    too_long = c.lens.clone()
    too_long[0] = c.MB * c.B + 100
    c.gpu_decode(lens=too_long)
    assert pkv.last_error() == pkv.ERR_DEVICE_BOUNDS
    assert pkv.last_error() == pkv.OK


def test_host_argument_checks():
    c = Case(lengths=[40], Hq=8, Hkv=2, D=128, B=16, dtype="bf16", seed=61)
    out = torch.zeros(1, 8, 128, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:           # workspace too small
        c.pool.paged_decode(out, c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale,
                            workspace=torch.zeros(4, device="cuda"))
    assert e.value.status == pkv.ERR_INVALID
    q7 = torch.zeros(1, 7, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(pkv.PagedKVError):                # 7 query heads over 2 KV heads
        c.pool.paged_decode(out, q7, c.k_cache, c.v_cache, c.tables, c.lens, c.scale)
    with pytest.raises(pkv.PagedKVError):                # partition not a multiple of 16
        c.pool.paged_decode(out, c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale, partition_tokens=24)
    odd = pkv.Pool(1, 2, 128, 8, 16, 2, 8, pkv.BF16)     # block size 8 is not supported by the kernels
    assert odd.decode_workspace_bytes(1, 8) == 0


@pytest.mark.parametrize("window", [1, 16, 37, 100, 5000])
@pytest.mark.parametrize("partition_tokens", [0, 64])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_sliding_window_parity(window, partition_tokens, dtype, path):
    if dtype == "f32" and path == "simt":
        pytest.skip("fp32 always runs on the CUDA-core path")
    c = Case(lengths=[0, 1, 15, 16, 17, 100, 257, 700, 1500], Hq=32, Hkv=8, D=128, B=16, dtype=dtype, seed=71)
    out = c.gpu_decode(partition_tokens, window=window)
    check(c, out, c.oracle_decode(window=window))
    assert pkv.last_error() == pkv.OK


def test_window_with_released_blocks(path):
    """Blocks wholly before the window are released (holes in the tables) and never read."""
    W = 128
    c = Case(lengths=[300, 1000, 40, 129, 16 * 9], Hq=32, Hkv=8, D=128, B=16, dtype="bf16", seed=73)
    before = c.pool.stats()["num_free"]
    released = 0
    for sid, L in zip(c.seqs, c.oracle_lens.tolist()):
        released += c.pool.release_before(sid, max(0, L - W))
        st, n = c.model.release_before(sid, max(0, L - W))
        assert st == 0
    c.refresh_tables()
    assert released > 0 and c.pool.stats()["num_free"] == before + released
    assert (c.oracle_tables == -1).any()
    for pt in (0, 32):
        check(c, c.gpu_decode(pt, window=W), c.oracle_decode(window=W))
    assert pkv.last_error() == pkv.OK
    # appends keep working after a release, and the window keeps sliding
    for _ in range(20):
        c.decode_step_append()
    check(c, c.gpu_decode(0, window=W), c.oracle_decode(window=W))
    assert pkv.last_error() == pkv.OK


def test_prefix_cache_requests_decode(path):
    """Requests built through the prefix cache share a 200-token system prompt's full blocks. Each
    caller writes K/V only for positions the cache did not already hold; decode must match the oracle
    (which built its own tables with the cache model and scattered the same values on the host)."""
    from oracle import alloc_model as am
    from oracle import cache_ops as ocache
    from tests.gpu_cases import to_device
    B, Hkv, Hq, D, NB = 16, 8, 32, 128, 300
    fl = synth.free_list(NB, 9)
    pool = pkv.Pool(1, Hkv, D, B, NB, 16, 64, pkv.BF16, initial_free_list=fl)
    model = am.PrefixCacheModel(NB, B, 16, 64, initial_free_list=fl)
    kc = torch.full((NB, Hkv, B, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    hk = np.full((NB, Hkv, B, D), synth.nan_bits("bf16"), dtype=np.uint16)
    hv = np.full_like(hk, synth.nan_bits("bf16"))
    system = list(range(200))
    sys_kv = synth.normal_f32((2, 200, Hkv, D), 9, 1)       # K/V of the shared prompt positions
    seqs = []
    for r in range(6):
        suffix_len = [0, 3, 40, 1, 77, 120][r]
        toks = system + [1000 + 10 * r + i for i in range(suffix_len)]
        suf_kv = synth.normal_f32((2, suffix_len, Hkv, D), 9, 10 + r)
        kv = np.concatenate([sys_kv, suf_kv], axis=1)
        sid, slots, ncached = pool.alloc_prefix(3, toks)
        st, msid, mslots, mncached = model.alloc_prefix(3, toks)
        assert st == 0 and (msid, mslots, mncached) == (sid, slots.tolist(), ncached)
        assert ncached == (0 if r == 0 else 192)
        k = synth.encode(kv[0, ncached:], "bf16")
        v = synth.encode(kv[1, ncached:], "bf16")
        w_slots = torch.from_numpy(slots[ncached:].copy()).cuda()
        pool.reshape_and_cache(to_device(k, "bf16"), to_device(v, "bf16"), w_slots, kc, vc)
        ocache.reshape_and_cache(hk, hv, k, v, mslots[ncached:])
        seqs.append(sid)
    assert pool.prefix_stats() == model.prefix_stats()
    tables, lens = pool.block_table(seqs)
    mtab, mlens = model.block_table(seqs)
    assert tables.tolist() == mtab
    q_stored = synth.encode(synth.normal_f32((6, Hq, D), 9, 99), "bf16")
    out = torch.empty(6, Hq, D, device="cuda")
    ws = torch.empty(pool.decode_workspace_bytes(6, Hq) // 4 + 4, device="cuda")
    pool.paged_decode(out, to_device(q_stored, "bf16"), kc, vc, torch.from_numpy(tables).cuda(),
                      torch.from_numpy(lens).cuda(), 1 / math.sqrt(D), workspace=ws)
    ref = native.decode(q_stored, hk, hv, np.asarray(mtab, dtype=np.int32), np.asarray(mlens, dtype=np.int32),
                        1 / math.sqrt(D))
    err = float(np.max(np.abs(out.double().cpu().numpy() - ref)))
    assert err <= 2e-3, err
    assert pkv.last_error() == pkv.OK


def test_largest_batch_and_the_shared_memory_limit():
    """16,384 sequences (the largest batch the entry point takes) decode correctly; where the
    per-sequence prefix arrays of a call (12 bytes per sequence with partitions and a window) no
    longer fit beside a CTA's copy ring, the call is refused before anything is enqueued."""
    rng = np.random.default_rng(91)
    c = Case(lengths=rng.integers(1, 41, size=16384).tolist(), Hq=8, Hkv=1, D=128, B=16, dtype="bf16", seed=91)
    check(c, c.gpu_decode(0), c.oracle_decode())
    check(c, c.gpu_decode(64), c.oracle_decode())
    check(c, c.gpu_decode(0, window=24), c.oracle_decode(window=24))
    with pytest.raises(pkv.PagedKVError) as e:
        c.gpu_decode(64, window=24)
    assert e.value.status == pkv.ERR_INVALID
    assert pkv.last_error() == pkv.OK


@pytest.mark.parametrize("pt", [0, 512, 64])
def test_cuda_graph_replays_match_direct_calls_bitwise(pt, path):
    """A decode captured in a CUDA graph and replayed several times returns exactly what a direct
    call returns: a replay launches with the captured call's arguments (the same arrival-counter
    tag included), so the counters must start from zero again on every replay."""
    c = case_from_workload("gqa5_bf16", host_cache=False)
    ref = c.gpu_decode(pt)
    nbytes = c.pool.decode_workspace_bytes(c.n, c.Hq, pt)
    ws = torch.full((max(nbytes, 16) // 4 + 4,), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.full_like(ref, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                      # a direct call of the same shape first
        c.pool.paged_decode(out, c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale,
                            partition_tokens=pt, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.pool.paged_decode(out, c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale,
                            partition_tokens=pt, workspace=ws)
    for _ in range(4):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert pkv.last_error() == pkv.OK


@pytest.mark.parametrize("name,pt,window", [("gqa5_bf16", 0, 0), ("gqa5_bf16", 512, 0), ("tiny_f32", 64, 0),
                                            ("prefix_cow_partial_bf16", 0, 300), ("gqa5_bf16", 32, 100)])
def test_deferred_merge_mode(name, pt, window, monkeypatch):
    """PKV_DECODE_DEFER=1: dynamic tasks in the decode, cut units merged by a second kernel (bf16
    pools; an fp32 pool has no deferred instantiation and keeps the in-kernel merge). Same results as
    the oracle for both split modes and a window; repeated calls agree bit for bit (a task's chunks,
    and so its result, do not depend on which warp takes it)."""
    monkeypatch.setenv("PKV_DECODE_DEFER", "1")
    c = case_from_workload(name)
    out = c.gpu_decode(pt, window=window)
    check(c, out, c.oracle_decode(window=window))
    assert torch.equal(c.gpu_decode(pt, window=window), out)
    assert pkv.last_error() == pkv.OK
