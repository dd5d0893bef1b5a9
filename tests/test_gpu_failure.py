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


def test_per_pool_error_words_on_two_streams():
    """Two pools, each with its own error word, decoding on two streams: a bad block id in one
    pool's table is reported by that pool's stream only; the other pool's word stays clear, the
    process-wide word is untouched, and neither read synchronises the device."""
    assert pkv.last_error() == pkv.OK
    ca = Case(lengths=[40, 300], Hq=8, Hkv=2, D=128, B=16, dtype="bf16", seed=81)
    cb = Case(lengths=[70, 20], Hq=8, Hkv=2, D=128, B=16, dtype="bf16", seed=82)
    wa = torch.zeros(1, dtype=torch.int32, device="cuda")
    wb = torch.zeros(1, dtype=torch.int32, device="cuda")
    ca.pool.set_error_word(wa)
    cb.pool.set_error_word(wb)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    bad = ca.tables.clone()
    bad[1, 2] = ca.NB + 7                                   # out of the pool
    torch.cuda.synchronize()
    outs = []
    for c, s, tables in ((ca, sa, bad), (cb, sb, cb.tables)):
        out = torch.zeros(c.n, c.Hq, c.D, device="cuda")
        ws = torch.empty(c.pool.decode_workspace_bytes(c.n, c.Hq, 0) // 4 + 4, device="cuda")
        with torch.cuda.stream(s):
            c.pool.paged_decode(out, c.q, c.k_cache, c.v_cache, tables, c.lens, c.scale, workspace=ws, stream=s)
        outs.append(out)
    assert cb.pool.stream_error(sb) == pkv.OK
    assert ca.pool.stream_error(sa) == pkv.ERR_DEVICE_BOUNDS
    assert ca.pool.stream_error(sa) == pkv.OK                # read and cleared
    assert int(wa.item()) == 0 and int(wb.item()) == 0
    torch.cuda.synchronize()
    ref_b = cb.oracle_decode()
    assert float(np.max(np.abs(outs[1].double().cpu().numpy() - ref_b))) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK                         # nothing reached the process-wide word
    # every kind of kernel of the pool records into its word: a cache write with a slot past the pool
    slots = torch.tensor([ca.NB * ca.B + 3], dtype=torch.int64, device="cuda")
    k1 = torch.zeros(1, ca.Hkv, ca.D, dtype=torch.bfloat16, device="cuda")
    ca.pool.reshape_and_cache(k1, k1, slots, ca.k_cache, ca.v_cache, stream=sa)
    assert ca.pool.stream_error(sa) == pkv.ERR_DEVICE_BOUNDS
    ca.pool.set_error_word(None)                              # back to the process-wide word
    ca.pool.reshape_and_cache(k1, k1, slots, ca.k_cache, ca.v_cache, stream=sa)
    assert ca.pool.stream_error(sa) == pkv.ERR_INVALID        # no word any more
    assert pkv.last_error() == pkv.ERR_DEVICE_BOUNDS
    cb.pool.set_error_word(None)
