"""pkv_paged_decode_static: paged decode without any caller-provided or allocated scratch.

Callers such as a plugin living inside an application that owns all device memory, or a serving
loop that must never allocate (an allocation can synchronise the device), cannot hand the library
a workspace. For them the library keeps a fixed 16 MiB scratch array of its own on every device.
These tests call that entry point through the C ABI and compare it with the ordinary entry point
(caller workspace) on the same inputs, twice in a row, so that a second call which finds the
previous call's leftovers in the shared scratch is covered too. The file sorts last so that a run
stopping at the first failure has run every other test already.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
from tests.gpu_cases import TOL, Case, case_from_workload

pytestmark = pytest.mark.gpu


def call_static(c: Case, out: torch.Tensor, partition_tokens: int) -> int:
    """The raw C-ABI call (no binding helpers), on the current torch stream."""
    return pkv.lib.pkv_paged_decode_static(
        c.pool._h, out.data_ptr(), c.q.data_ptr(), c.k_cache.data_ptr(), c.v_cache.data_ptr(),
        c.tables.data_ptr(), c.lens.data_ptr(), c.n, c.Hq, ctypes.c_float(c.scale), int(partition_tokens),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,partition_tokens", [
    ("gqa5_bf16", 0), ("gqa5_bf16", 512), ("tiny_f32", 0), ("tiny_f32", 512),
    ("prefix_cow_partial_bf16", 0), ("prefix_cow_partial_bf16", 512), ("serve256_bf16", 0)])
def test_static_scratch_matches_caller_workspace(name, partition_tokens):
    c = case_from_workload(name, host_cache=False)
    ref = c.gpu_decode(partition_tokens)        # ordinary entry point, caller-provided workspace
    assert pkv.last_error() == pkv.OK
    for _ in range(2):                           # two calls in a row share (and reuse) the scratch
        out = torch.full_like(ref, float("nan"))
        assert call_static(c, out, partition_tokens) == pkv.OK
        torch.cuda.synchronize()
        err = float((out.double() - ref.double()).abs().max())
        assert np.isfinite(out.cpu().numpy()).all()
        assert err <= TOL[c.dtype], err
        # the same kernel with the same split: a scratch slot read at the wrong place would change
        # a partial slightly without leaving the tolerance, so the results must agree bit for bit
        assert torch.equal(out, ref)
    assert pkv.last_error() == pkv.OK


def test_static_scratch_rejects_problems_that_do_not_fit():
    # 16-token partitions over a 1024-block table need far more than 16 MiB of partial results
    c = Case(lengths=[40, 3000], Hq=32, Hkv=8, D=128, B=32, dtype="bf16", seed=3, max_blocks=1024)
    need = c.pool.decode_workspace_bytes(c.n, c.Hq, 16)
    assert need > pkv.STATIC_SCRATCH_BYTES
    out = torch.zeros(c.n, c.Hq, c.D, device="cuda")
    assert call_static(c, out, 16) == pkv.ERR_SCRATCH_TOO_SMALL
    assert pkv.status_string(pkv.ERR_SCRATCH_TOO_SMALL).startswith("call needs more scratch")
    assert call_static(c, out, 0) == pkv.OK      # the same problem with the balanced split fits
    torch.cuda.synchronize()
    assert pkv.last_error() == pkv.OK
    # 256 sequences cut into 512-token partitions keep 2048 units x 9 partition slots: too big
    big = case_from_workload("serve256_bf16", host_cache=False)
    assert big.pool.decode_workspace_bytes(big.n, big.Hq, 512) > pkv.STATIC_SCRATCH_BYTES
    out = torch.zeros(big.n, big.Hq, big.D, device="cuda")
    assert call_static(big, out, 512) == pkv.ERR_SCRATCH_TOO_SMALL
