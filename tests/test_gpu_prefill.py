"""Causal paged prefill / multi-token append on the GPU against the binary64 oracle.

The context of each sequence (including the new positions) is written through the library's
allocator and cache-write kernel on the device, and by the oracle model and NumPy scatter on the
host (gpu_cases.Case); the last q_len_b positions are the queries. Tolerance: 2e-3 max abs (bf16
K/V, fp32 accumulation), the decode contract.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
import synth
from oracle import native
from tests.gpu_cases import Case, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["tc", "mma"], autouse=True)
def path(request, monkeypatch):
    """Every prefill test runs on both kernels: tcgen05 (the default) and mma.sync."""
    if request.param == "mma":
        monkeypatch.setenv("PKV_PREFILL_PATH", "mma")
    else:
        monkeypatch.delenv("PKV_PREFILL_PATH", raising=False)
    return request.param


def test_single_tile_one_kv_head():
    """The smallest case: one CTA (32 query tokens x 4 heads = 128 rows), one 32-key tile."""
    c = Case(lengths=[32], Hq=4, Hkv=1, D=128, B=16, dtype="bf16", seed=3)
    out, ref, _, _ = run_prefill(c, [32])
    assert max_err(out, ref) <= 2e-3
    assert pkv.last_error() == pkv.OK


def run_prefill(c: Case, qlens, window=0, seed=1):
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q_stored = synth.encode(synth.normal_f32((int(cu[-1]), c.Hq, c.D), seed, 55), "bf16")
    out = torch.full((int(cu[-1]), c.Hq, c.D), float("nan"), device="cuda")
    c.pool.paged_prefill(out, to_device(q_stored, "bf16"), c.k_cache, c.v_cache, c.tables, c.lens,
                         torch.from_numpy(cu).cuda(), c.scale, window=window)
    torch.cuda.synchronize()
    ref = native.prefill(q_stored, c.hk, c.hv, c.oracle_tables, c.oracle_lens, cu, c.scale, window=window)
    return out, ref, q_stored, cu


def max_err(out, ref):
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
def test_prefill_shapes(D, G):
    lens = [1, 17, 100, 333, 64, 700, 40]
    qlens = [1, 17, 37, 333, 0, 5, 16]           # full prefill, partial chunks, empty, one token
    c = Case(lengths=lens, Hq=2 * G, Hkv=2, D=D, B=32 if G % 2 else 16, dtype="bf16", seed=G)
    out, ref, _, _ = run_prefill(c, qlens)
    assert max_err(out, ref) <= 2e-3
    assert pkv.last_error() == pkv.OK


@pytest.mark.parametrize("window", [1, 16, 50, 10_000])
def test_prefill_sliding_window(window):
    c = Case(lengths=[300, 90, 1000], Hq=32, Hkv=8, D=128, B=16, dtype="bf16", seed=11)
    out, ref, _, _ = run_prefill(c, [300, 45, 128], window=window)
    assert max_err(out, ref) <= 2e-3
    assert pkv.last_error() == pkv.OK


def test_one_token_per_sequence_matches_decode():
    c = Case(lengths=[1, 15, 16, 17, 500, 2000], Hq=40, Hkv=8, D=128, B=16, dtype="bf16", seed=13)
    out, ref, q_stored, _ = run_prefill(c, [1] * 6)
    assert max_err(out, ref) <= 2e-3
    dec = c.gpu_decode(0, q=to_device(q_stored, "bf16"))
    assert float((dec - out).abs().max()) <= 2e-3


def test_extreme_logits_and_long_prompt():
    c = Case(lengths=[2048, 513], Hq=32, Hkv=8, D=128, B=16, dtype="bf16", seed=17)
    cu = np.array([0, 2048, 2048 + 200], dtype=np.int32)
    q = synth.normal_f32((2248, 32, 128), 17, 9) * 30.0           # logits in the hundreds
    q_stored = synth.encode(q, "bf16")
    out = torch.empty(2248, 32, 128, device="cuda")
    c.pool.paged_prefill(out, to_device(q_stored, "bf16"), c.k_cache, c.v_cache, c.tables, c.lens,
                         torch.from_numpy(cu).cuda(), c.scale)
    torch.cuda.synchronize()
    ref = native.prefill(q_stored, c.hk, c.hv, c.oracle_tables, c.oracle_lens, cu, c.scale)
    assert max_err(out, ref) <= 2e-3


def test_bad_query_counts_reported_not_faulted():
    c = Case(lengths=[40, 40], Hq=8, Hkv=2, D=128, B=16, dtype="bf16", seed=19)
    cu = torch.tensor([0, 50, 60], dtype=torch.int32, device="cuda")    # 50 queries for 40 positions
    q = torch.zeros(60, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(60, 8, 128, device="cuda")
    c.pool.paged_prefill(out, q, c.k_cache, c.v_cache, c.tables, c.lens, cu, c.scale)
    assert pkv.last_error() == pkv.ERR_DEVICE_BOUNDS
    with pytest.raises(pkv.PagedKVError):                                 # fp32 pools are decode-only
        f = Case(lengths=[4], Hq=2, Hkv=2, D=64, B=16, dtype="f32", seed=1)
        f.pool.paged_prefill(torch.zeros(1, 2, 64, device="cuda"), torch.zeros(1, 2, 64, device="cuda"),
                             f.k_cache, f.v_cache, f.tables, f.lens, torch.tensor([0, 1], dtype=torch.int32,
                                                                                  device="cuda"), f.scale)


def test_tensor_core_paths_agree(path, monkeypatch):
    """The tcgen05 and mma.sync kernels on one problem with every tile shape at once: ragged query
    tiles, keys past the context end in the last tile, many sequences."""
    if path != "tc":
        pytest.skip("compares both kernels once")
    rng = np.random.default_rng(23)
    lens = rng.integers(1, 600, size=40).tolist()
    qlens = [int(rng.integers(0, L + 1)) for L in lens]
    c = Case(lengths=lens, Hq=32, Hkv=8, D=128, B=16, dtype="bf16", seed=23)
    out_tc, ref, _, _ = run_prefill(c, qlens)
    monkeypatch.setenv("PKV_PREFILL_PATH", "mma")
    out_mma, _, _, _ = run_prefill(c, qlens)
    assert max_err(out_tc, ref) <= 2e-3 and max_err(out_mma, ref) <= 2e-3
    assert float((out_tc - out_mma).abs().max()) <= 2e-3
