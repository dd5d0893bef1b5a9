"""bench.py's kernel-source hash ignores comments but not code (it keys the committed ncu traffic)."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_for_sha", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def test_comments_do_not_count_but_code_and_strings_do():
    a = 'int x = 1;  // one\n/* block\n comment */ asm("mov.u32 %0, 1; // kept");\n'
    b = 'int x = 1;\nasm("mov.u32 %0, 1; // kept");   // another note\n'
    c = 'int x = 2;\nasm("mov.u32 %0, 1; // kept");\n'
    assert bench._strip_comments(a) == bench._strip_comments(b)
    assert bench._strip_comments(a) != bench._strip_comments(c)
    assert "// kept" in bench._strip_comments(a)


def test_traffic_record_when_current():
    """bench.py reports ncu traffic only while the capture's source hash matches (else null)."""
    rec = bench.decode_traffic_record("serve256_bf16")
    if rec is None:
        pytest.skip("kernel sources changed since the committed ncu capture: bench.py reports traffic null")
    assert rec["bytes_per_launch_profile"] > rec["algorithmic_bytes_profile"]
