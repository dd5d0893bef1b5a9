"""K1 (slot-mapped cache write) and K2 (copy-on-write block copy) against the oracle: bit-exact,
including every byte of blocks nobody wrote (NaN-poisoned on both sides)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
from tests.gpu_cases import Case, case_from_workload, to_device, to_host

pytestmark = pytest.mark.gpu


def bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)


def assert_caches_equal(c: Case):
    assert np.array_equal(bits(to_host(c.k_cache, c.dtype)), bits(c.hk))
    assert np.array_equal(bits(to_host(c.v_cache, c.dtype)), bits(c.hv))


@pytest.mark.parametrize("name", ["tiny_f32", "gqa5_bf16"])
def test_prefill_writes_bit_exact(name):
    assert_caches_equal(case_from_workload(name))


@pytest.mark.parametrize("name", ["prefix_cow_bf16", "prefix_cow_partial_bf16"])
def test_fork_and_copy_on_write_bit_exact(name):
    c = case_from_workload(name)
    assert_caches_equal(c)
    st = c.pool.stats()
    if name.endswith("partial_bf16"):
        assert st["num_cow"] > 100          # every child with a suffix copied the partial block
    else:
        assert st["num_cow"] == 0


def test_decode_step_appends_bit_exact():
    c = Case(lengths=[1, 15, 16, 17, 31, 32, 100, 0], Hq=8, Hkv=2, D=128, B=16, dtype="bf16", seed=3)
    for _ in range(20):
        c.decode_step_append()
    assert_caches_equal(c)
    assert pkv.last_error() == pkv.OK


def test_copy_blocks_many_layers():
    L, NB, H, B, D = 5, 12, 2, 16, 64
    pool = pkv.Pool(L, H, D, B, NB, 2, 4, pkv.BF16)
    g = torch.Generator(device="cuda").manual_seed(0)
    ks = [torch.randn(NB, H, B, D, generator=g, device="cuda").to(torch.bfloat16) for _ in range(L)]
    vs = [torch.randn(NB, H, B, D, generator=g, device="cuda").to(torch.bfloat16) for _ in range(L)]
    k0 = [k.clone() for k in ks]
    v0 = [v.clone() for v in vs]
    pairs = torch.tensor([[3, 7], [0, 11], [5, 1]], dtype=torch.int32, device="cuda")
    pool.copy_blocks(ks, vs, pairs)
    torch.cuda.synchronize()
    for l in range(L):
        exp_k, exp_v = k0[l].clone(), v0[l].clone()
        for s, d in pairs.tolist():
            exp_k[d] = k0[l][s]
            exp_v[d] = v0[l][s]
        assert torch.equal(ks[l].view(torch.int16), exp_k.view(torch.int16))
        assert torch.equal(vs[l].view(torch.int16), exp_v.view(torch.int16))


def test_negative_slots_skipped_and_out_of_range_reported():
    pool = pkv.Pool(1, 2, 64, 16, 4, 2, 4, pkv.F32)
    kc = torch.zeros(4, 2, 16, 64, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones(3, 2, 64, device="cuda")
    v = torch.full((3, 2, 64), 2.0, device="cuda")
    slots = torch.tensor([-1, 5, 4 * 16], dtype=torch.int64, device="cuda")   # skip, write, out of range
    assert pkv.last_error() == pkv.OK
    pool.reshape_and_cache(k, v, slots, kc, vc)
    assert pkv.last_error() == pkv.ERR_DEVICE_BOUNDS
    assert pkv.last_error() == pkv.OK                                       # the error word was cleared
    assert torch.equal(kc[0, :, 5], torch.ones(2, 64, device="cuda"))
    assert float(kc.sum()) == 2 * 64 and float(vc.sum()) == 2 * 2 * 64


def test_bad_copy_pair_reported_not_faulted():
    pool = pkv.Pool(1, 2, 64, 16, 4, 2, 4, pkv.F32)
    kc = torch.zeros(4, 2, 16, 64, device="cuda")
    vc = torch.zeros_like(kc)
    pool.copy_blocks([kc], [vc], torch.tensor([[1, 9]], dtype=torch.int32, device="cuda"))
    assert pkv.last_error() == pkv.ERR_DEVICE_BOUNDS


def test_host_argument_checks():
    pool = pkv.Pool(1, 2, 64, 16, 4, 2, 4, pkv.BF16)
    kc = torch.zeros(4, 2, 16, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(2, 2, 64, device="cuda", dtype=torch.bfloat16)
    slots = torch.zeros(2, dtype=torch.int64, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pool.reshape_and_cache(k.data_ptr() + 2, k, slots, kc, kc)          # misaligned
    assert e.value.status == pkv.ERR_INVALID
