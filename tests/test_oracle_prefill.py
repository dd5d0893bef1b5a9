"""Pins of the causal prefill oracle (NumPy attention.paged_prefill and C native.prefill)."""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

from oracle import attention as att
from oracle import native
from tests.test_oracle_attention import make_problem

IMPLS = {
    "numpy": lambda *a, **k: att.paged_prefill(*a, **k),
    "c": lambda *a, **k: native.prefill(*a, **k),
}
IMPLS_DECODE = {"numpy": att.paged_decode, "c": native.decode}


def problem(seed, lens, qlens, Hq=8, Hkv=2, D=32, B=16, dtype="bf16"):
    P = make_problem(seed, lens, Hq, Hkv, D, B, dtype)
    rng = np.random.default_rng(seed + 1000)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    from synth import encode
    P["qp"] = encode(rng.standard_normal((int(cu[-1]), Hq, D)).astype(np.float32), dtype)
    P["cu"] = cu
    P["qlens"] = list(qlens)
    return P


def sdpa_causal(P, window=0):
    """torch SDPA (float64) on the contiguous logical K/V with an explicit offset-causal mask."""
    q = torch.from_numpy(att.to_f64(P["qp"]))
    out = torch.zeros(q.shape, dtype=torch.float64)
    for b, (L, ql) in enumerate(zip(P["lens"], P["qlens"])):
        if ql == 0:
            continue
        K = torch.from_numpy(att.to_f64(P["logical"][b][0])).permute(1, 0, 2)[None]
        V = torch.from_numpy(att.to_f64(P["logical"][b][1])).permute(1, 0, 2)[None]
        pos = torch.arange(L - ql, L)[:, None]
        t = torch.arange(L)[None, :]
        mask = t <= pos
        if window > 0:
            mask &= t > pos - window
        qb = q[P["cu"][b]:P["cu"][b + 1]].permute(1, 0, 2)[None]
        o = torch.nn.functional.scaled_dot_product_attention(qb, K, V, attn_mask=mask, scale=P["scale"], enable_gqa=True)
        out[P["cu"][b]:P["cu"][b + 1]] = o[0].permute(1, 0, 2)
    return out.numpy()


def run(impl, P, window=0, **kw):
    return IMPLS[impl](P["qp"], P["kc"], P["vc"], P["tables"], P["lens"], P["cu"], P["scale"], window=window, **kw)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("window", [0, 1, 20])
def test_matches_sdpa_with_offset_causal_mask(impl, window):
    P = problem(3, [40, 17, 5, 100], [40, 3, 1, 64])
    np.testing.assert_allclose(run(impl, P, window), sdpa_causal(P, window), rtol=0, atol=1e-12)


@pytest.mark.parametrize("impl", IMPLS)
def test_one_query_per_sequence_is_decode(impl):
    P = problem(5, [40, 17, 1, 100], [1, 1, 1, 1], Hq=8, Hkv=2)
    dec = IMPLS_DECODE[impl](P["qp"], P["kc"], P["vc"], P["tables"], P["lens"], P["scale"])
    assert np.array_equal(run(impl, P), dec) if impl == "numpy" else np.allclose(run(impl, P), dec, rtol=0,
                                                                                   atol=1e-14)


@pytest.mark.parametrize("impl", IMPLS)
def test_chunked_prefill_equals_one_shot(impl):
    """Positions computed in one prefill call equal the same positions computed chunk by chunk."""
    P = problem(7, [90], [90])
    full = run(impl, P)
    parts = []
    for a, b in [(0, 30), (30, 31), (31, 90)]:
        Q = dict(P)
        Q["qp"] = P["qp"][a:b]
        Q["lens"] = np.array([b], dtype=np.int32)
        Q["cu"] = np.array([0, b - a], dtype=np.int32)
        parts.append(run(impl, Q))
    assert np.array_equal(np.concatenate(parts), full)


@pytest.mark.parametrize("impl", IMPLS)
def test_future_keys_do_not_matter(impl):
    P = problem(9, [50], [20])
    base = run(impl, P)
    logical = [(k.copy(), v.copy()) for k, v in P["logical"]]
    P2 = make_problem(9, [50], 8, 2, 32, 16, "bf16", logical=logical)
    P2.update(qp=P["qp"], cu=P["cu"], qlens=P["qlens"], tables=P["tables"])
    B = 16
    for t in range(45, 50):                       # keys after the position of query 44 - 30 = 14
        blk = P["tables"][0, t // B]
        P2["kc"][blk, :, t % B] = P["kc"][blk, :, t % B] ^ np.uint16(0x1234)
    out = run(impl, P2)
    np.testing.assert_array_equal(out[:15], base[:15])
    assert not np.array_equal(out[15:], base[15:])


def test_c_prefill_mutant_is_caught(tmp_path):
    src = open(os.path.join(os.path.dirname(native.__file__), "decode_ref.c")).read()
    old = "const int p = lens[b] - qlen + (int)(row - cu_q[b]);"
    assert src.count(old) == 1
    (tmp_path / "m.c").write_text(src.replace(old, "const int p = lens[b] - qlen + (int)(row - cu_q[b]) - 1;"))
    so = tmp_path / "libm.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(so), str(tmp_path / "m.c"), "-lm"],
                   check=True)
    import ctypes
    lib = ctypes.CDLL(str(so))
    f = lib.oracle_prefill
    f.restype = ctypes.c_int
    f.argtypes = native._load().oracle_prefill.argtypes
    P = problem(3, [40, 17], [40, 3])
    out = np.zeros(P["qp"].shape, dtype=np.float64)
    f(out.ctypes.data, P["qp"].ctypes.data, 1, P["kc"].ctypes.data, P["vc"].ctypes.data, 1,
      np.ascontiguousarray(P["tables"]).ctypes.data, np.ascontiguousarray(P["lens"], dtype=np.int32).ctypes.data,
      P["cu"].ctypes.data, 2, 8, 2, 32, 16, P["tables"].shape[1], P["scale"], 0, 1)
    assert not np.allclose(out, sdpa_causal(P), rtol=0, atol=1e-12)
