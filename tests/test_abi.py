"""The C ABI library loads on a machine without a GPU and exports exactly the
symbols include/idx.h declares; host-only entry points behave as documented.
No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "idx.h")


@pytest.fixture(scope="module")
def libpath():
    from sparse_attention_indexer_quant_gb300 import build_lib
    return build_lib.build()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^IDX_API\s+[\w\s\*]*?\b(idx_\w+)\s*\(", text, re.M)))


def test_header_lists_the_entry_points():
    names = header_functions()
    for n in ["idx_quant_insert", "idx_quant_q", "idx_mqa_logits", "idx_paged_mqa_logits",
              "idx_topk_rows", "idx_paged_logits_topk", "idx_gather_k"]:
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    for n in header_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(set(re.findall(r"\sT\s(idx_\w+)$", out, re.M)))
    assert exported == header_functions()


def test_binding_signatures_cover_header(libpath):
    from sparse_attention_indexer_quant_gb300 import binding
    assert sorted(binding.SIGNATURES) == header_functions()


def test_arch_gate_is_fail_closed(libpath):
    from sparse_attention_indexer_quant_gb300 import binding
    assert binding.arch_supported(10, 3)
    for major, minor in [(10, 0), (10, 1), (9, 0), (8, 6), (12, 0), (11, 0), (10, 4), (0, 0)]:
        assert not binding.arch_supported(major, minor), (major, minor)


def test_status_strings(libpath):
    from sparse_attention_indexer_quant_gb300 import binding
    lib = binding.lib
    assert lib.idx_version() >= 100
    for s in range(5):
        assert lib.idx_status_string(s)
    assert b"unknown" in lib.idx_status_string(99)


def test_argument_errors_without_gpu(libpath):
    """Shape errors are reported before any device work."""
    from sparse_attention_indexer_quant_gb300 import binding
    lib = binding.lib
    assert lib.idx_quant_insert(None, -1, 128, None, None, 1, 64, None, None) == 1
    assert lib.idx_quant_insert(None, 1, 100, None, None, 1, 64, None, None) == 1
    assert lib.idx_quant_insert(None, 1, 128, None, None, 1, 32, None, None) == 1
    assert lib.idx_topk_rows(None, 1, 10, None, None, 0, None, None) == 1
    assert lib.idx_topk_rows(None, 1, 10, None, None, 4096, None, None) == 1
    args = [None, None, 1, 3, 32, None, 1, 64, None, 1, None, None, None, 64, 0, None, None]
    assert lib.idx_paged_mqa_logits(*args) == 1          # next_n = 3
    args[3], args[4] = 1, 48
    assert lib.idx_paged_mqa_logits(*args) == 1          # H = 48
    assert b"H=48" in lib.idx_last_error_detail()
    assert lib.idx_gather_k(None, 1, 64, None, 1, None, None, -1, None, None, 0, None, None) == 1


def test_workspace_query_is_host_only(libpath):
    from sparse_attention_indexer_quant_gb300 import binding
    n1 = binding.paged_logits_topk_workspace_bytes(64, 1, 512, 2048)
    n2 = binding.paged_logits_topk_workspace_bytes(128, 1, 512, 2048)
    assert n2 >= n1 >= 0
