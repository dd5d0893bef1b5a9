"""Full-size workloads in the launch configuration the benchmark times, checked against the oracle.

serve256_bf16 (one layer of the 32-layer step; the layers are identical launches), the same layer on
an fp8 pool, long_split_bf16 (8 x 32,768 tokens, 512-token partitions, an 80 GB-scale pool) and
prefill_bf16 (16 x 2,048-token causal prefill) are checked on every output; the oracle runs in C
with OpenMP.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_494_b300 as pkv
import synth
from oracle import native
from tests.gpu_cases import TOL, Case, Fp8Case, case_from_workload, to_device

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


def test_serve256_fp8_one_layer_full():
    """The fp8 bench line's launch: serving batch on an fp8 pool, balanced split, no window."""
    w = synth.workload("serve256_bf16")
    c = Fp8Case(lengths=synth.lengths(w, 0), Hq=w.num_q_heads, Hkv=w.num_kv_heads, seed=0)
    out = c.gpu_decode(0)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert float(np.max(np.abs(got - c.oracle_decode()))) <= 2e-3
    assert pkv.last_error() == pkv.OK


def test_prefill_bf16_full():
    """The prefill bench line's launch: 16 x 2,048-token prompts, every position a query."""
    w = synth.workload("prefill_bf16")
    lens = synth.lengths(w, 0)
    c = Case(lengths=lens, Hq=w.num_q_heads, Hkv=w.num_kv_heads, D=w.head_dim, B=w.block_size, dtype="bf16",
             seed=0)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q_stored = synth.encode(synth.normal_f32((int(cu[-1]), c.Hq, c.D), 0, 55), "bf16")
    out = torch.empty((int(cu[-1]), c.Hq, c.D), device="cuda")
    c.pool.paged_prefill(out, to_device(q_stored, "bf16"), c.k_cache, c.v_cache, c.tables, c.lens,
                         torch.from_numpy(cu).cuda(), c.scale)
    torch.cuda.synchronize()
    ref = native.prefill(q_stored, c.hk, c.hv, c.oracle_tables, c.oracle_lens, cu, c.scale)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert float(np.max(np.abs(got - ref))) <= TOL["bf16"]
    assert pkv.last_error() == pkv.OK
