"""The C-ABI library loads without a GPU and exports every entry point include/pagedkv.h declares."""
import os
import re
import subprocess

import paged_kv_cache_494_b300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src))
    return names


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ["pkv_pool_create", "pkv_alloc", "pkv_free", "pkv_fork", "pkv_reshape_and_cache",
                 "pkv_copy_blocks", "pkv_paged_decode"]:
        assert must in names


def test_library_exports_every_declared_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\b(pkv_[a-z0-9_]+)\b", out))
    missing = declared_symbols() - exported
    assert not missing, missing
    # the binding wraps exactly the declared entry points
    assert set(pkv.EXPORTED_SYMBOLS) == declared_symbols()


def test_no_torch_types_in_the_boundary():
    src = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    assert "torch" not in src.lower().replace("torch tensors", "")
    assert 'extern "C"' in src


def test_version_and_status_strings():
    assert pkv.lib.pkv_version() == 1
    assert pkv.status_string(pkv.ERR_NO_BLOCKS) == "not enough free blocks"
    assert pkv.status_string(0) == "ok"


def test_sizes_follow_the_budget_formula():
    p = pkv.Pool(32, 8, 128, 16, 100, 4, 8, pkv.BF16)
    assert p.bytes_per_token == 131072
    assert p.layer_cache_bytes == 100 * 8 * 16 * 128 * 2
    # a pool's K+V bytes over all layers equal NB * B * bytes_per_token
    assert 2 * p.num_layers * p.layer_cache_bytes == 100 * 16 * p.bytes_per_token


def test_fp8_sizes():
    p = pkv.Pool(32, 8, 128, 16, 100, 4, 8, pkv.FP8)
    assert p.layer_cache_bytes == 100 * 8 * 16 * 128
    assert p.layer_scale_bytes == 100 * 8 * 16 * 4
    assert p.bytes_per_token == 2 * 32 * 8 * (128 + 4)          # codes + one scale per token and head
    assert pkv.Pool(1, 2, 64, 16, 4, 1, 1, pkv.BF16).layer_scale_bytes == 0


def test_invalid_descriptors_rejected():
    import pytest
    with pytest.raises(pkv.PagedKVError):
        pkv.Pool(1, 0, 64, 16, 10, 2, 2)
    with pytest.raises(pkv.PagedKVError):
        pkv.Pool(1, 2, 64, 16, 4, 2, 2, initial_free_list=[0, 1, 1, 3])
