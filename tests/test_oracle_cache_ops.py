"""Pins of oracle/cache_ops.py: scatter by slot and block copy, checked element by element."""
import numpy as np

from oracle import cache_ops


def test_reshape_and_cache_writes_exact_positions():
    rng = np.random.default_rng(0)
    NB, H, B, D = 9, 3, 4, 5
    kc = rng.standard_normal((NB, H, B, D)).astype(np.float32)
    vc = rng.standard_normal((NB, H, B, D)).astype(np.float32)
    k0, v0 = kc.copy(), vc.copy()
    slots = [7, -1, 0, 35, 18]
    k = rng.standard_normal((5, H, D)).astype(np.float32)
    v = rng.standard_normal((5, H, D)).astype(np.float32)
    cache_ops.reshape_and_cache(kc, vc, k, v, slots)
    # position (block, offset) of slot s, independently enumerated
    where = {s: (blk, off) for blk in range(NB) for off in range(B) for s in [blk * B + off]}
    touched = set()
    for i, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = where[s]
        assert np.array_equal(kc[blk, :, off, :], k[i]) and np.array_equal(vc[blk, :, off, :], v[i])
        touched.add((blk, off))
    for blk in range(NB):
        for off in range(B):
            if (blk, off) not in touched:
                assert np.array_equal(kc[blk, :, off], k0[blk, :, off])
                assert np.array_equal(vc[blk, :, off], v0[blk, :, off])


def test_bf16_bits_copied_verbatim():
    kc = np.zeros((2, 1, 2, 3), dtype=np.uint16)
    vc = np.zeros_like(kc)
    k = np.array([[[0x7FC0, 0x8000, 0x0001]]], dtype=np.uint16)    # NaN, -0, denormal
    cache_ops.reshape_and_cache(kc, vc, k, k, [3])
    assert kc[1, 0, 1].tolist() == [0x7FC0, 0x8000, 0x0001]


def test_copy_blocks_all_layers_in_order():
    rng = np.random.default_rng(1)
    layers = [(rng.standard_normal((6, 2, 4, 3)), rng.standard_normal((6, 2, 4, 3))) for _ in range(3)]
    before = [(k.copy(), v.copy()) for k, v in layers]
    cache_ops.copy_blocks(layers, [(1, 4), (2, 0)])
    for (k, v), (k0, v0) in zip(layers, before):
        assert np.array_equal(k[4], k0[1]) and np.array_equal(v[4], v0[1])
        assert np.array_equal(k[0], k0[2]) and np.array_equal(v[0], v0[2])
        for b in (1, 2, 3, 5):
            assert np.array_equal(k[b], k0[b]) and np.array_equal(v[b], v0[b])
