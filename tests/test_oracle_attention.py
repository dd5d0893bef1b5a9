"""Pins of the decode oracle (NumPy and C binary64) against things other than itself.

* torch's scaled_dot_product_attention in float64 on the contiguous logical K/V (a library
  routine the oracle does not use; its enable_gqa convention pins the head grouping);
* closed-form special cases: one token returns its V row, equal keys or a zero query
  give the mean of V, a dominant logit selects its V row;
* extreme logits stay finite ("Servicio de modelos de lenguaje..." §6);
* the online recurrence equals dense attention to binary64 rounding over 8 cases and
  several block sizes (§9 of the same page prints 2.22e-16 over 8 cases);
* invariance under block placement, shared vs duplicated prefix pages, NaN-poisoned
  unowned memory, and the GQA head mapping.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as att
from oracle import native

IMPLS = {
    "numpy": lambda *a, **k: att.paged_decode(*a, **k),
    "c": lambda *a, **k: native.decode(*a, **k),
}


def make_problem(seed, lens, Hq, Hkv, D, B, dtype="f32", NB=None, poison=True, logical=None):
    """Random logical K/V per sequence, scattered into a paged pool by a random placement.

    The scatter here uses NumPy fancy indexing (not the oracle's gather loop).
    Returns dict with stored q, caches, tables, lens and the logical (stored) K/V.
    """
    rng = np.random.default_rng(seed)
    n = len(lens)
    pages = [-(-L // B) for L in lens]
    NB = NB or sum(pages) + 5
    MB = max(max(pages), 1)
    perm = rng.permutation(NB)
    tables = np.full((n, MB), -1, dtype=np.int32)
    pos = 0
    for b, P in enumerate(pages):
        tables[b, :P] = perm[pos:pos + P]
        pos += P
    enc = (lambda x: synth.encode(x, dtype))
    store_dt = np.float32 if dtype == "f32" else np.uint16
    fill = synth.nan_bits(dtype) if poison else store_dt(0)
    kc = np.full((NB, Hkv, B, D), fill, dtype=store_dt)
    vc = np.full((NB, Hkv, B, D), fill, dtype=store_dt)
    if logical is None:
        logical = [(enc(rng.standard_normal((L, Hkv, D)).astype(np.float32)),
                    enc(rng.standard_normal((L, Hkv, D)).astype(np.float32))) for L in lens]
    for b, L in enumerate(lens):
        t = np.arange(L)
        blk = tables[b, t // B]
        kc[blk, :, t % B, :] = logical[b][0]
        vc[blk, :, t % B, :] = logical[b][1]
    q = enc(rng.standard_normal((n, Hq, D)).astype(np.float32))
    return dict(q=q, kc=kc, vc=vc, tables=tables, lens=np.asarray(lens, dtype=np.int32), logical=logical,
                scale=1.0 / math.sqrt(D))


def run(impl, P):
    return IMPLS[impl](P["q"], P["kc"], P["vc"], P["tables"], P["lens"], P["scale"])


def sdpa(P):
    q = torch.from_numpy(att.to_f64(P["q"]))
    out = []
    for b, L in enumerate(P["lens"]):
        if L == 0:
            out.append(torch.zeros(q.shape[1], q.shape[2], dtype=torch.float64))
            continue
        K = torch.from_numpy(att.to_f64(P["logical"][b][0])).permute(1, 0, 2)[None]   # [1, Hkv, L, D]
        V = torch.from_numpy(att.to_f64(P["logical"][b][1])).permute(1, 0, 2)[None]
        o = torch.nn.functional.scaled_dot_product_attention(q[b][None, :, None, :], K, V, scale=P["scale"],
                                                             enable_gqa=True)
        out.append(o[0, :, 0, :])
    return torch.stack(out).numpy()


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(8, 2, 64, 16), (10, 2, 32, 3), (4, 4, 16, 1), (6, 1, 128, 32)])
def test_matches_sdpa(impl, dtype, shape):
    Hq, Hkv, D, B = shape
    P = make_problem(7, [1, 17, 100, 53, 0, 250], Hq, Hkv, D, B, dtype)
    np.testing.assert_allclose(run(impl, P), sdpa(P), rtol=0, atol=1e-12)


@pytest.mark.parametrize("impl", IMPLS)
def test_brute_force_tiny(impl):
    P = make_problem(3, [1, 5, 9], 4, 2, 8, 4, "bf16")
    dec = lambda a: att.to_f64(a).tolist()
    ref = att.brute_force_decode(dec(P["q"]), dec(P["kc"]), dec(P["vc"]), P["tables"].tolist(),
                                 P["lens"].tolist(), P["scale"])
    np.testing.assert_allclose(run(impl, P), np.array(ref), rtol=0, atol=1e-13)


@pytest.mark.parametrize("impl", IMPLS)
def test_single_token_returns_v_row(impl):
    P = make_problem(5, [1, 1], 8, 2, 64, 16, "bf16")
    out = run(impl, P)
    for b in range(2):
        for j in range(8):
            assert np.array_equal(out[b, j], att.to_f64(P["logical"][b][1][0, j // 4]))


@pytest.mark.parametrize("impl", IMPLS)
def test_equal_keys_or_zero_query_give_mean_of_v(impl):
    rng = np.random.default_rng(11)
    L, Hkv, D = 37, 2, 16
    krow = rng.standard_normal((1, Hkv, D)).astype(np.float32)
    K = np.repeat(krow, L, axis=0)
    V = rng.standard_normal((L, Hkv, D)).astype(np.float32)
    P = make_problem(11, [L], 4, Hkv, D, 8, "f32", logical=[(K, V)])
    out = run(impl, P)
    for j in range(4):
        np.testing.assert_allclose(out[0, j], V[:, j // 2, :].astype(np.float64).mean(axis=0), rtol=0, atol=1e-14)
    P["q"][:] = 0
    out = run(impl, P)
    np.testing.assert_allclose(out[0, 0], V[:, 0, :].astype(np.float64).mean(axis=0), rtol=0, atol=1e-14)


@pytest.mark.parametrize("impl", IMPLS)
def test_dominant_logit_selects_row(impl):
    rng = np.random.default_rng(12)
    L, D = 50, 64
    K = (0.01 * rng.standard_normal((L, 1, D))).astype(np.float32)
    V = rng.standard_normal((L, 1, D)).astype(np.float32)
    q = np.zeros((1, 1, D), dtype=np.float32)
    q[0, 0, 0] = 1.0
    K[23, 0, 0] = 8.0 * 70.0               # scaled logit margin > 60 (scale 1/8)
    P = make_problem(12, [L], 1, 1, D, 16, "f32", logical=[(K, V)])
    P["q"] = q
    np.testing.assert_allclose(run(impl, P)[0, 0], V[23, 0].astype(np.float64), rtol=0, atol=1e-20)


@pytest.mark.parametrize("impl", IMPLS)
def test_extreme_logits_finite(impl):
    P = make_problem(13, [300, 7], 8, 2, 64, 16, "f32")
    P["q"] = (P["q"] * 100.0).astype(np.float32)      # logits ~ 1e3
    out = run(impl, P)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, sdpa(P), rtol=0, atol=1e-11)


def test_online_recurrence_equals_dense():
    """8 cases, several block sizes, fixed seed: binary64 agreement as in the page's companion."""
    rng = np.random.default_rng(2024)
    worst = 0.0
    for case in range(8):
        L = int(rng.integers(1, 400))
        D = int(rng.choice([16, 64, 128]))
        q = rng.standard_normal(D)
        K = rng.standard_normal((L, D))
        V = rng.standard_normal((L, D))
        if case >= 6:                       # large-logit cases test the normalisation
            q *= 60.0
        dense = att.dense_attention(q, K, V, 1 / math.sqrt(D))
        for blk in (1, 3, 16, 32):
            err = float(np.max(np.abs(att.online_attention(q, K, V, 1 / math.sqrt(D), blk) - dense)))
            worst = max(worst, err)
    assert worst <= 1e-15


def test_partition_merge_equals_dense():
    rng = np.random.default_rng(99)
    for L, cuts in [(1000, [512]), (2048, [512, 1024, 1536]), (700, [1, 2, 699]), (33, [10, 11, 20])]:
        q, K, V = rng.standard_normal(64), rng.standard_normal((L, 64)), rng.standard_normal((L, 64))
        q *= 5.0
        edges = [0] + cuts + [L]
        parts = [att.partial_attention(q, K[a:b], V[a:b], 0.125) for a, b in zip(edges[:-1], edges[1:])]
        # a few binary64 roundings more than the dense path (normalise, then re-weight)
        np.testing.assert_allclose(att.merge_partials(parts), att.dense_attention(q, K, V, 0.125), rtol=0, atol=1e-14)


@pytest.mark.parametrize("impl", IMPLS)
def test_permutation_invariance(impl):
    lens = [33, 1, 160, 77]
    P1 = make_problem(21, lens, 8, 2, 64, 16, "bf16")
    P2 = make_problem(22, lens, 8, 2, 64, 16, "bf16", logical=P1["logical"])
    P2["q"] = P1["q"]
    assert not np.array_equal(P1["tables"], P2["tables"])
    assert np.array_equal(run(impl, P1), run(impl, P2))


@pytest.mark.parametrize("impl", IMPLS)
def test_shared_prefix_equals_duplicated(impl):
    """Two sequences with the same 48-token prefix: shared physical pages vs private copies."""
    P = make_problem(31, [60, 70], 8, 2, 64, 16, "f32", poison=True)
    pre_k = P["logical"][0][0][:48]
    pre_v = P["logical"][0][1][:48]
    logical = [(np.concatenate([pre_k, P["logical"][b][0][48:]]), np.concatenate([pre_v, P["logical"][b][1][48:]]))
               for b in range(2)]
    dup = make_problem(31, [60, 70], 8, 2, 64, 16, "f32", logical=logical)
    shared = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in dup.items()}
    shared["tables"][1, :3] = shared["tables"][0, :3]     # point sequence 1 at sequence 0's prefix pages
    np.testing.assert_array_equal(run(impl, shared), run(impl, dup))


@pytest.mark.parametrize("impl", IMPLS)
def test_poisoned_pool_is_never_read(impl):
    lens = [5, 16, 31, 100]
    Pn = make_problem(41, lens, 8, 2, 64, 16, "bf16", poison=True, NB=40)
    Pz = make_problem(41, lens, 8, 2, 64, 16, "bf16", poison=False, NB=40, logical=Pn["logical"])
    Pz["q"], Pz["tables"] = Pn["q"], Pn["tables"]
    Pz["kc"][Pz["kc"] != Pz["kc"]] = 0
    out = run(impl, Pn)
    assert np.isfinite(out).all()
    assert np.array_equal(out, run(impl, Pz))


@pytest.mark.parametrize("impl", IMPLS)
def test_empty_context_gives_zero_row(impl):
    P = make_problem(51, [0, 3, 0], 4, 2, 16, 4, "f32")
    out = run(impl, P)
    assert (out[0] == 0).all() and (out[2] == 0).all() and np.isfinite(out).all()


@pytest.mark.parametrize("impl", IMPLS)
def test_gqa_head_grouping(impl):
    """Query head j reads only KV head j // (Hq / Hkv): perturbing another KV head leaves it unchanged."""
    P = make_problem(61, [40, 9], 10, 2, 32, 8, "f32")
    base = run(impl, P)
    logical = [(k.copy(), v.copy()) for k, v in P["logical"]]
    for k, v in logical:
        k[:, 1] += 1.0
        v[:, 1] *= -1.0
    P2 = make_problem(61, [40, 9], 10, 2, 32, 8, "f32", logical=logical)
    P2["q"] = P["q"]
    out = run(impl, P2)
    assert np.array_equal(out[:, :5], base[:, :5])
    assert not np.allclose(out[:, 5:], base[:, 5:])


def test_c_oracle_sampled_rows_and_threads():
    P = make_problem(71, [100, 7, 300], 8, 2, 64, 16, "bf16")
    full, used = native.decode(P["q"], P["kc"], P["vc"], P["tables"], P["lens"], P["scale"], return_threads=True)
    assert used >= 1
    rows = [0, 9, 23, 17]
    part = native.decode(P["q"], P["kc"], P["vc"], P["tables"], P["lens"], P["scale"], rows=rows)
    for r, flat in enumerate(rows):
        assert np.array_equal(part[r], full[flat // 8, flat % 8])


@pytest.mark.parametrize("impl", IMPLS)
def test_sliding_window(impl):
    """Window W: the last W positions only. W >= len is full attention; W = 1 returns the last V
    row; otherwise it equals SDPA on the sliced logical K/V."""
    P = make_problem(81, [300, 40, 1, 17], 8, 2, 64, 16, "bf16")
    full = run(impl, P)
    run_w = lambda W: IMPLS[impl](P["q"], P["kc"], P["vc"], P["tables"], P["lens"], P["scale"], window=W)
    assert np.array_equal(run_w(300), full) and np.array_equal(run_w(10_000), full)
    one = run_w(1)
    for b, L in enumerate(P["lens"]):
        for j in range(8):
            assert np.array_equal(one[b, j], att.to_f64(P["logical"][b][1][L - 1, j // 4]))
    for W in (16, 33, 100):
        sl = dict(P)
        sl["logical"] = [(k[-W:], v[-W:]) for k, v in P["logical"]]
        np.testing.assert_allclose(run_w(W), sdpa(sl), rtol=0, atol=1e-12)


@pytest.mark.parametrize("impl", IMPLS)
def test_window_ignores_released_blocks(impl):
    """Blocks entirely before the window may be released (table entry -1): never read."""
    P = make_problem(83, [300, 100], 8, 2, 64, 16, "f32")
    ref = IMPLS[impl](P["q"], P["kc"], P["vc"], P["tables"], P["lens"], P["scale"], window=64)
    holes = P["tables"].copy()
    holes[0, :(300 - 64) // 16] = -1
    holes[1, :(100 - 64) // 16] = -1
    out = IMPLS[impl](P["q"], P["kc"], P["vc"], holes, P["lens"], P["scale"], window=64)
    assert np.array_equal(out, ref)
