"""Full-size workloads in the launch configuration the benchmark times, checked against the oracle.

serve256_bf16 (one layer of the 32-layer step; the layers are identical launches) and
long_split_bf16 (8 x 32,768 tokens, 512-token partitions, an 80 GB-scale pool) are checked on
every output; the oracle runs in C with OpenMP.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
from tests.gpu_cases import TOL, case_from_workload

pytestmark = pytest.mark.gpu


def max_err(c, out):
    return float(np.max(np.abs(out.double().cpu().numpy() - c.oracle_decode())))


def test_serve256_one_layer_full():
    c = case_from_workload("serve256_bf16")
    out = c.gpu_decode(0)
    assert np.isfinite(out.cpu().numpy()).all()
    assert max_err(c, out) <= TOL["bf16"]
    c.decode_step_append()                     # the step the benchmark times: append, then attend
    assert max_err(c, c.gpu_decode(0)) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK


def test_serve256_one_layer_sliding_window():
    c = case_from_workload("serve256_bf16")
    out = c.gpu_decode(0, window=256)
    err = float(np.max(np.abs(out.double().cpu().numpy() - c.oracle_decode(window=256))))
    assert err <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK


def test_long_split_full():
    c = case_from_workload("long_split_bf16", compact_host=True)
    assert c.NB > 600_000
    for pt in (512, 0):
        out = c.gpu_decode(pt)
        assert max_err(c, out) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK
    del c
    torch.cuda.empty_cache()
