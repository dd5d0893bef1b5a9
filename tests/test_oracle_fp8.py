"""Pins of oracle/fp8.py: the E4M3 codec against torch's float8_e4m3fn and its own definition."""
import numpy as np
import pytest
import torch

from oracle import fp8


def test_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = fp8.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])


def test_known_codes():
    v = fp8.decode_e4m3(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x7E, 0xFE, 0x80], dtype=np.uint8))
    assert v.tolist()[:6] == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 448.0]
    assert v[6] == -448.0 and np.signbit(v[7])
    assert np.isnan(fp8.decode_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.encode_e4m3(fp8.decode_e4m3(codes)), codes)


def test_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.1, 1.0, 30.0, 200.0)]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode_e4m3(x), ref)


def test_ties_go_to_even_and_saturation():
    # 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39): even code 0x38
    assert fp8.encode_e4m3(np.array([1.0625, 1.1875, -1.0625]))[:].tolist() == [0x38, 0x3A, 0xB8]
    assert fp8.encode_e4m3(np.array([464.0, 1e30, -1e9])).tolist() == [0x7E, 0x7E, 0xFE]


def test_quantize_rows_error_bound():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((500, 128)) * rng.uniform(0.01, 50, size=(500, 1))).astype(np.float32)
    x[7] = 0.0
    codes, scale = fp8.quantize_rows(x)
    assert scale[7] == 1.0 and (codes[7] == 0).all()
    deq = fp8.dequantize(codes, scale)
    # each value within half a step of its binade (relative 2^-4 for normals, 2^-10 * scale below)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scale[:, None]) * 1.0001
    assert (np.abs(deq - x) <= bound).all()
    # the largest magnitude of each row maps to +-448 (up to the rounding of scale)
    amax_codes = codes[np.arange(500), np.argmax(np.abs(x), axis=1)] & 0x7F
    assert ((amax_codes == 0x7E) | (amax_codes == 0x7D))[np.abs(x).max(axis=1) > 0].all()


def test_quantising_scatter_and_dequantised_attention():
    """A token written into the fp8 pool reads back as its quantised value, through the
    dim-major V layout; attention over the dequantised pool equals attention over those values."""
    import math
    from oracle import attention as att
    from oracle import native
    rng = np.random.default_rng(2)
    NB, H, B, D = 6, 2, 16, 128
    k8 = np.zeros((NB, H, B, D), np.uint8)
    v8t = np.zeros((NB, H, D, B), np.uint8)
    ks = np.ones((NB, H, B), np.float32)
    vs = np.ones((NB, H, B), np.float32)
    k = rng.standard_normal((20, H, D)).astype(np.float32)
    v = (rng.standard_normal((20, H, D)) * 3).astype(np.float32)
    slots = [5 * B + i for i in range(16)] + [2 * B + i for i in range(4)]
    fp8.reshape_and_cache_fp8(k8, ks, v8t, vs, k, v, slots)
    K, V = fp8.dequantize_pool(k8, ks, v8t, vs)
    kq, ksc = fp8.quantize_rows(k)
    vq, vsc = fp8.quantize_rows(v)
    for i, sl in enumerate(slots):
        assert np.array_equal(K[sl // B, :, sl % B], fp8.dequantize(kq[i], ksc[i]))
        assert np.array_equal(V[sl // B, :, sl % B], fp8.dequantize(vq[i], vsc[i]))
        assert np.array_equal(v8t[sl // B, :, :, fp8.v_byte_offset(sl % B)], vq[i])
    tables = np.array([[5, 2]], np.int32)
    q = rng.standard_normal((1, 4, D)).astype(np.float32)
    a = att.paged_decode(q, K, V, tables, [20], 1 / math.sqrt(D))
    c = native.decode(q, K, V, tables, np.array([20], np.int32), 1 / math.sqrt(D))
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-13)
    Kc = np.concatenate([K[5], K[2, :, :4]], axis=1)          # [H, 20, D] logical order
    Vc = np.concatenate([V[5], V[2, :, :4]], axis=1)
    for j in range(4):
        np.testing.assert_allclose(a[0, j], att.dense_attention(q[0, j].astype(np.float64), Kc[j // 2], Vc[j // 2],
                                                                1 / math.sqrt(D)), rtol=0, atol=1e-14)


def test_v_group_order_is_a_permutation():
    assert sorted(fp8.V_GROUP_ORDER) == list(range(16))
    assert [fp8.v_byte_offset(j) for j in range(32)][16:] == [16 + p for p in fp8.V_POSITION]
    # lane t of a dim row reads bytes 4t..4t+3: tokens (2t, 2t+1, 8+2t, 9+2t)
    for t in range(4):
        assert fp8.V_GROUP_ORDER[4 * t:4 * t + 4] == [2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t]
