"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every pipelined kernel waits on mbarriers with a poll limit; when it runs out the warp records
PKV_ERR_DEVICE_TIMEOUT, drains its own copies and returns. pkv_selftest_wait_timeout runs that same
wait on a barrier nothing signals (no copy in flight). The test checks the reported status, that the
kernel returned (the host sees its flag), and that the context still serves an ordinary decode.
"""
import time

import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
from tests.gpu_cases import TOL, Case

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_survives():
    assert pkv.last_error() == pkv.OK
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    st = pkv.lib.pkv_selftest_wait_timeout(flag.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == pkv.OK
    assert pkv.last_error() == pkv.ERR_DEVICE_TIMEOUT      # synchronises, then reports and clears
    elapsed = time.perf_counter() - t0
    assert int(flag.item()) == 1
    assert elapsed < 5.0, elapsed                          # the poll limit is about a second
    assert pkv.last_error() == pkv.OK                      # cleared
    c = Case(lengths=[1, 17, 300], Hq=8, Hkv=2, D=128, B=16, dtype="bf16", seed=5)
    got = c.gpu_decode(0).double().cpu().numpy()
    assert float(np.max(np.abs(got - c.oracle_decode()))) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK
    print(f"bounded wait gave up after {elapsed:.3f} s")
