"""FP8 E4M3 KV pools on the GPU against the oracle.

Cache writes (codes in both layouts and the per-(token, head) scales) and copy-on-write copies are
bit-exact: both sides quantise in float32 with IEEE division and round to nearest even. Decode is
compared with binary64 attention over the dequantised pool, max abs error <= 2e-3.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
import synth
from tests.gpu_cases import Fp8Case

pytestmark = pytest.mark.gpu


def bits_equal(dev: torch.Tensor, host: np.ndarray) -> bool:
    d = dev.cpu().numpy()
    if host.dtype == np.float32:
        return np.array_equal(d.view(np.uint32), host.view(np.uint32))
    return np.array_equal(d, host)


def assert_pool_equal(c: Fp8Case):
    assert bits_equal(c.k8, c.hk8)
    assert bits_equal(c.v8, c.hv8)
    assert bits_equal(c.ksc, c.hks)
    assert bits_equal(c.vsc, c.hvs)


def test_quantising_write_bit_exact():
    c = Fp8Case(lengths=[1, 17, 100, 333, 5], Hq=8, Hkv=2, seed=1)
    assert_pool_equal(c)
    for _ in range(5):
        c.decode_step_append()
    assert_pool_equal(c)
    assert pkv.last_error() == pkv.OK


def test_copy_on_write_bit_exact_and_decode():
    w = synth.workload("prefix_cow_partial_bf16")
    trace = [("new", 1016)] + [("fork", 0)] * 12 + [("free", 0)] + [("append", i, s) for i, s in
                                                                      enumerate([0, 1, 7, 8, 9, 40, 3, 0, 100, 2, 5, 16])]
    c = Fp8Case(lengths=[1016 + 120] * 12, Hq=32, Hkv=8, seed=2, prefix_trace=trace)
    assert c.pool.stats()["num_cow"] >= 9
    assert_pool_equal(c)
    err = float(np.max(np.abs(c.gpu_decode().double().cpu().numpy() - c.oracle_decode())))
    assert err <= 2e-3, err


@pytest.mark.parametrize("G", [1, 4, 5, 8])
@pytest.mark.parametrize("partition_tokens", [0, 64])
@pytest.mark.parametrize("window", [0, 37])
def test_fp8_decode_parity(G, partition_tokens, window):
    c = Fp8Case(lengths=[1, 2, 15, 16, 17, 100, 257, 700, 2000], Hq=2 * G, Hkv=2, seed=3 + G, B=32 if G % 2 else 16)
    out = c.gpu_decode(partition_tokens, window)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = float(np.max(np.abs(got - c.oracle_decode(window))))
    assert err <= 2e-3, err
    assert pkv.last_error() == pkv.OK


def test_fp8_entry_points_reject_other_pools():
    bf = pkv.Pool(1, 2, 128, 16, 8, 2, 4, pkv.BF16)
    z = torch.zeros(1, device="cuda")
    with pytest.raises(pkv.PagedKVError):
        bf.paged_decode_fp8(torch.zeros(1, 4, 128, device="cuda"), torch.zeros(1, 4, 128, dtype=torch.bfloat16,
                                                                                device="cuda"),
                            z, z, z, z, torch.zeros(1, 4, dtype=torch.int32, device="cuda"),
                            torch.ones(1, dtype=torch.int32, device="cuda"), 0.1)
    f8 = pkv.Pool(1, 2, 128, 16, 8, 2, 4, pkv.FP8)
    with pytest.raises(pkv.PagedKVError):                    # bf16/fp32 write path refuses fp8 pools
        f8.reshape_and_cache(torch.zeros(1, 2, 128, dtype=torch.bfloat16, device="cuda"),
                             torch.zeros(1, 2, 128, dtype=torch.bfloat16, device="cuda"),
                             torch.zeros(1, dtype=torch.int64, device="cuda"),
                             torch.zeros(8, 2, 16, 128, dtype=torch.uint8, device="cuda"),
                             torch.zeros(8, 2, 128, 16, dtype=torch.uint8, device="cuda"))
