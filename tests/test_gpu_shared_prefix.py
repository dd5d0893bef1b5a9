"""Shared-prefix (cascade) decode on the GPU against the binary64 oracle.

A prompt is forked into children that share its full blocks physically (copy-on-write: "Paged
Attention optimiza el uso de memoria en LLMs"; "PagedAttention e vLLM", "Implementazione nel mondo
reale"). pkv_paged_decode_shared_prefix attends the shared blocks once for all children and merges
with each child's private suffix by log-sum-exp; the result must be the ordinary decode attention,
which the oracle computes per sequence over the whole context. Tolerance: 2e-3 max abs (bf16 K/V,
fp32 accumulation), the decode contract.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
import synth
from tests.gpu_cases import TOL, Case, case_from_workload, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["mma", "simt"])
def path(request, monkeypatch):
    """The suffix part runs on the tensor-core decode kernel by default, or the CUDA-core one."""
    if request.param == "simt":
        monkeypatch.setenv("PKV_DECODE_PATH", "simt")
    else:
        monkeypatch.delenv("PKV_DECODE_PATH", raising=False)
    return request.param


def shared_decode(c: Case, prefix_blocks: int, q=None, tables=None, lens=None) -> torch.Tensor:
    q = c.q if q is None else q
    out = torch.full((c.n, c.Hq, c.D), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = c.pool.shared_prefix_workspace_bytes(c.n, c.Hq, prefix_blocks)
    assert nbytes > 0 or prefix_blocks == 0
    ws = torch.full((max(nbytes, 16) // 4 + 4,), float("nan"), dtype=torch.float32, device="cuda")
    c.pool.paged_decode_shared_prefix(out, q, c.k_cache, c.v_cache, c.tables if tables is None else tables,
                                      c.lens if lens is None else lens, c.scale, prefix_blocks, workspace=ws)
    torch.cuda.synchronize()
    return out


def max_err(out: torch.Tensor, ref: np.ndarray) -> float:
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


def forked(prompt: int, suffixes, *, Hq: int, Hkv: int, D: int, B: int, seed: int) -> Case:
    """One prompt, len(suffixes) forks, prompt freed, each child appends its suffix."""
    trace = [("new", prompt)] + [("fork", 0)] * len(suffixes) + [("free", 0)]
    trace += [("append", i, int(s)) for i, s in enumerate(suffixes)]
    lens = [prompt + int(s) for s in suffixes]
    pages = -(-prompt // B) + sum(-(-(prompt % B + int(s)) // B) + 1 for s in suffixes)
    return Case(lengths=lens, Hq=Hq, Hkv=Hkv, D=D, B=B, dtype="bf16", seed=seed, prefix_trace=trace,
                num_blocks=pages + 16, max_blocks=-(-max(lens) // B) + 2)


@pytest.mark.parametrize("name", ["prefix_cow_bf16", "prefix_cow_partial_bf16"])
def test_workload_parity(name, path):
    c = case_from_workload(name)
    pb = c.pool.shared_prefix_blocks(c.seqs)
    assert pb == (1024 if name == "prefix_cow_bf16" else 1016) // 16
    out = shared_decode(c, pb)
    assert max_err(out, c.oracle_decode()) <= TOL["bf16"]
    assert float((out - c.gpu_decode(0)).abs().max()) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK
    # one decode step later (every child appends a token; the partial-prompt children copy-on-write
    # the shared partial block): the shared full blocks are unchanged
    c.decode_step_append()
    assert c.pool.shared_prefix_blocks(c.seqs) == pb
    out = shared_decode(c, pb)
    assert max_err(out, c.oracle_decode()) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
def test_group_sizes_and_ragged_suffixes(D, G):
    """Suffixes of 0 (context = the shared prefix alone), 1 and ragged lengths; a prompt that is not a
    whole number of blocks (its partial block is private after the first append)."""
    c = forked(328, [0, 1, 15, 16, 17, 100, 333, 2, 40], Hq=2 * G, Hkv=2, D=D, B=16, seed=G)
    pb = c.pool.shared_prefix_blocks(c.seqs)
    assert pb == 328 // 16
    out = shared_decode(c, pb)
    assert max_err(out, c.oracle_decode()) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK


@pytest.mark.parametrize("n_children", [1, 2, 255, 257, 600])
def test_batch_sizes_across_work_items(n_children):
    """Batches around the tensor-core kernel's work-item size (256 query rows per item at G = 1), a
    single sequence, and a short prefix split over few keys (64-key split granularity)."""
    rng = np.random.default_rng(n_children)
    suf = rng.integers(0, 80, size=n_children)
    c = forked(96, suf, Hq=8, Hkv=8, D=128, B=32, seed=n_children)
    pb = c.pool.shared_prefix_blocks(c.seqs)
    # the prompt's 3 blocks; a lone sequence shares all its own full blocks with itself
    assert pb == (3 if n_children > 1 else int(c.oracle_lens[0]) // 32)
    out = shared_decode(c, pb)
    assert max_err(out, c.oracle_decode()) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK


def test_long_prefix_and_extreme_logits():
    """A 16k-token shared prefix (many key splits) with logits in the hundreds: the log-sum-exp
    merge of the split parts and the suffix must stay exact."""
    c = forked(16384, [0, 5, 700, 64, 1], Hq=32, Hkv=8, D=128, B=16, seed=31)
    c.q_stored = synth.encode(synth.normal_f32((c.n, c.Hq, c.D), 31, 9) * 30.0, "bf16")
    c.q = to_device(c.q_stored, "bf16")
    pb = c.pool.shared_prefix_blocks(c.seqs)
    out = shared_decode(c, pb)
    assert max_err(out, c.oracle_decode()) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK


def test_shorter_prefix_than_shared_is_exact():
    """Any prefix_blocks up to the shared count is exact (fewer shared blocks only move keys from the
    shared part to the suffix part); 0 is the plain decode, bit for bit, with the workspace size the
    shared-prefix query reports."""
    c = forked(200, [3, 50, 0, 130], Hq=16, Hkv=4, D=128, B=16, seed=5)
    ref = c.oracle_decode()
    for pb in (1, 5, 12):
        assert max_err(shared_decode(c, pb), ref) <= TOL["bf16"]
    assert torch.equal(shared_decode(c, 0), c.gpu_decode(0))
    assert pkv.last_error() == pkv.OK


def test_mismatched_tables_and_lengths_are_reported():
    """Tables that do not share the claimed prefix, or a sequence shorter than it, are recorded as
    PKV_ERR_DEVICE_BOUNDS (no fault); unsupported arguments are rejected on the host."""
    c = forked(64, [10, 20], Hq=8, Hkv=2, D=128, B=16, seed=7)
    t = c.tables.clone()
    t[1, 0] = t[1, 1]                                   # sequence 1 no longer starts with block 0's id
    shared_decode(c, 4, tables=t)
    assert pkv.last_error() == pkv.ERR_DEVICE_BOUNDS
    short = c.lens.clone()
    short[0] = 40                                       # shorter than 4 shared blocks of 16
    shared_decode(c, 4, lens=short)
    assert pkv.last_error() == pkv.ERR_DEVICE_BOUNDS
    shared_decode(c, 4)
    assert pkv.last_error() == pkv.OK
    with pytest.raises(pkv.PagedKVError):               # too small a workspace
        out = torch.empty(c.n, c.Hq, c.D, device="cuda")
        ws = torch.empty(16, dtype=torch.uint8, device="cuda")
        c.pool.paged_decode_shared_prefix(out, c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale, 4,
                                          workspace=ws)
    with pytest.raises(pkv.PagedKVError):               # more shared blocks than a table holds
        c.pool.paged_decode_shared_prefix(out, c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale,
                                          c.MB + 1, workspace=ws)
    f = Case(lengths=[32, 32], Hq=2, Hkv=2, D=64, B=16, dtype="f32", seed=1)
    assert f.pool.shared_prefix_workspace_bytes(2, 2, 1) == 0   # fp32 pools: decode only


def test_repeat_calls_and_cuda_graph_replays_are_bitwise_equal():
    """The suffix decode takes its tasks dynamically, but each task's chunks, and so its result, are
    fixed: repeated calls agree bit for bit. A captured call replayed several times does too (a
    replay reuses the captured call's tag, so the task counter must start from zero again)."""
    c = case_from_workload("prefix_cow_partial_bf16", host_cache=False)
    pb = c.pool.shared_prefix_blocks(c.seqs)
    ref = shared_decode(c, pb)
    assert torch.equal(shared_decode(c, pb), ref)
    nbytes = c.pool.shared_prefix_workspace_bytes(c.n, c.Hq, pb)
    ws = torch.full((nbytes // 4 + 4,), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.full_like(ref, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                      # a direct call of the same shape first
        c.pool.paged_decode_shared_prefix(out, c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale, pb,
                                          workspace=ws, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.pool.paged_decode_shared_prefix(out, c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale, pb,
                                          workspace=ws, stream=s)
    for _ in range(4):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert pkv.last_error() == pkv.OK


def test_one_workspace_across_shapes_bitwise(monkeypatch):
    """One workspace serves shared-prefix calls of different batch sizes and prefix lengths in turn,
    with deferred plain decodes in between (another user of the same task counter): every call returns
    exactly what it returns on a fresh NaN-filled workspace, so stale counters, tags and partials left
    by earlier calls are never taken for its own."""
    monkeypatch.setenv("PKV_DECODE_DEFER", "1")
    c = forked(512, list(range(0, 400, 7)), Hq=16, Hkv=4, D=128, B=16, seed=9)
    pb_full = c.pool.shared_prefix_blocks(c.seqs)
    shapes = [(c.n, pb_full), (c.n // 2, pb_full), (c.n, 7), (c.n // 3, 20)]
    nbytes = max(max(c.pool.shared_prefix_workspace_bytes(n, c.Hq, pb) for n, pb in shapes),
                 c.pool.decode_workspace_bytes(c.n, c.Hq, 0))

    def run(n, pb, ws):
        out = torch.full((n, c.Hq, c.D), float("nan"), dtype=torch.float32, device="cuda")
        c.pool.paged_decode_shared_prefix(out, c.q[:n], c.k_cache, c.v_cache, c.tables[:n], c.lens[:n], c.scale,
                                          pb, workspace=ws)
        torch.cuda.synchronize()
        return out

    def nan_ws():
        return torch.full((nbytes // 4 + 4,), float("nan"), dtype=torch.float32, device="cuda")

    fresh = {s: run(*s, nan_ws()) for s in shapes}
    ref = c.oracle_decode()
    for (n, pb), out in fresh.items():
        assert max_err(out, ref[:n]) <= TOL["bf16"]
    ws = nan_ws()
    plain = torch.empty(c.n, c.Hq, c.D, device="cuda")
    for it in range(12):
        s = shapes[it % len(shapes)]
        assert torch.equal(run(*s, ws), fresh[s]), (it, s)
        if it % 3 == 2:   # a deferred plain decode on the same workspace
            c.pool.paged_decode(plain, c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale, workspace=ws)
    assert pkv.last_error() == pkv.OK
