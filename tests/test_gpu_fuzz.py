"""Seeded random problems on the GPU against the binary64 oracle.

Decode: each case draws the head counts (group sizes 1..8), head dim, block size, a length mix
(empty, single-token, ragged, long), a split mode (balanced or fixed partitions), an optional sliding
window, the storage dtype and the minimum chunks per warp (down to one-chunk slivers), then builds the
pool through the library's allocator on the device and the oracle model on the host
(gpu_cases.Case) and compares every output; a few decode steps (append, then attend) follow on the
same pool. The same for fp8 pools (against attention over the dequantised pool), and for prefill /
multi-token append with random query counts (0..len) per sequence.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
import synth
from oracle import native
from tests.gpu_cases import TOL, Case, Fp8Case, to_device

pytestmark = pytest.mark.gpu


def draw(seed: int) -> dict:
    r = np.random.default_rng([seed, 4242])
    hkv = int(r.choice([1, 2, 4, 8]))
    g = int(r.integers(1, 9))
    dtype = "f32" if r.random() < 0.25 else "bf16"
    if dtype == "f32" and g == 7:
        g = 6                                       # fp32 pools support groups 1..6 and 8
    D = int(r.choice([64, 128]))
    B = int(r.choice([16, 32, 64]))
    n = int(r.integers(1, 40))
    kinds = r.random(n)
    lens = np.where(kinds < 0.08, 0, np.where(kinds < 0.16, 1, np.where(
        kinds < 0.9, r.integers(2, 700, size=n), r.integers(700, 3000, size=n))))
    if lens.max() == 0:
        lens[0] = 5
    pt = int(r.choice([0, 0, 16, 64, 512]))
    window = int(r.choice([0, 0, 0, 37, 256]))
    min_chunks = int(r.choice([1, 4, 16]))
    return dict(Hkv=hkv, Hq=hkv * g, dtype=dtype, D=D, B=B, lens=[int(x) for x in lens], pt=pt,
                window=window, min_chunks=min_chunks)


@pytest.mark.parametrize("seed", range(48))
def test_random_decode_problems(seed, monkeypatch):
    p = draw(seed)
    monkeypatch.setenv("PKV_DECODE_MIN_CHUNKS", str(p["min_chunks"]))
    c = Case(lengths=p["lens"], Hq=p["Hq"], Hkv=p["Hkv"], D=p["D"], B=p["B"], dtype=p["dtype"], seed=seed)
    for step in range(3):
        out = c.gpu_decode(p["pt"], window=p["window"])
        got = out.double().cpu().numpy()
        assert np.isfinite(got).all(), (p, step)
        err = float(np.max(np.abs(got - c.oracle_decode(window=p["window"]))))
        assert err <= TOL[p["dtype"]], (p, step, err)
        c.decode_step_append()
    assert pkv.last_error() == pkv.OK


@pytest.mark.parametrize("seed", range(12))
def test_random_fp8_decode_problems(seed):
    p = draw(1000 + seed)
    g = p["Hq"] // p["Hkv"]
    c = Fp8Case(lengths=p["lens"], Hq=p["Hkv"] * g, Hkv=p["Hkv"], B=p["B"], seed=seed)
    for step in range(2):
        out = c.gpu_decode(p["pt"], p["window"])
        got = out.double().cpu().numpy()
        assert np.isfinite(got).all(), (p, step)
        err = float(np.max(np.abs(got - c.oracle_decode(p["window"]))))
        assert err <= 2e-3, (p, step, err)
        c.decode_step_append()
    assert pkv.last_error() == pkv.OK


@pytest.mark.parametrize("seed", range(16))
def test_random_prefill_problems(seed):
    r = np.random.default_rng([seed, 777])
    hkv = int(r.choice([1, 2, 8]))
    g = int(r.integers(1, 9))
    D = int(r.choice([64, 128]))
    B = int(r.choice([16, 32]))
    n = int(r.integers(1, 8))
    lens = [int(x) for x in r.integers(1, 1500, size=n)]
    qlens = [int(r.integers(0, L + 1)) if r.random() < 0.7 else L for L in lens]
    window = int(r.choice([0, 0, 1, 40, 300]))
    c = Case(lengths=lens, Hq=hkv * g, Hkv=hkv, D=D, B=B, dtype="bf16", seed=seed)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    if cu[-1] == 0:
        return
    q_stored = synth.encode(synth.normal_f32((int(cu[-1]), c.Hq, c.D), seed, 56), "bf16")
    out = torch.full((int(cu[-1]), c.Hq, c.D), float("nan"), device="cuda")
    c.pool.paged_prefill(out, to_device(q_stored, "bf16"), c.k_cache, c.v_cache, c.tables, c.lens,
                         torch.from_numpy(cu).cuda(), c.scale, window=window)
    torch.cuda.synchronize()
    ref = native.prefill(q_stored, c.hk, c.hv, c.oracle_tables, c.oracle_lens, cu, c.scale, window=window)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert float(np.max(np.abs(got - ref))) <= 2e-3, (lens, qlens, window, hkv, g, D, B)
    assert pkv.last_error() == pkv.OK
