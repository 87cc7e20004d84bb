"""The C ABI library builds for sm_103a, loads, and exports every symbol that
include/maxsim.h declares. Host-side argument checks are exercised with
arguments that are rejected before any CUDA call, so no GPU is needed."""
import ctypes
import os
import re

import pytest

import maxsim_scoring_02_gb300 as m
from maxsim_scoring_02_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return m.load_library()


def _header_functions():
    src = open(os.path.join(ROOT, "include", "maxsim.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(maxsim_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert _header_functions() == sorted(m.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in m.STATUS_NAMES.items():
        assert lib.maxsim_status_string(code).decode().startswith(name)
    assert lib.maxsim_version() >= 100


def test_host_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)          # 16-byte aligned, never dereferenced: rejected earlier
    # NULL inputs
    assert lib.maxsim_score(None, 1, 32, 128, fake, 10, 128, None, 0, fake, None, None) == 1
    # misaligned D
    assert lib.maxsim_score(fake, 1, 32, 128, P(0x1001), 10, 128, None, 0, fake, None, None) == 1
    # negative sizes / bad dtype
    assert lib.maxsim_score(fake, 1, 0, 128, fake, 10, 128, None, 0, fake, None, None) == 1
    assert lib.maxsim_score(fake, 1, 32, 128, fake, -1, 128, None, 0, fake, None, None) == 1
    assert lib.maxsim_score(fake, 1, 32, 128, fake, 10, 128, None, 7, fake, None, None) == 1
    # tensor-core path needs d % 64 == 0
    assert lib.maxsim_score(fake, 1, 32, 96, fake, 10, 128, None, 0, fake, None, None) == 2
    # varlen: NULL offsets
    assert lib.maxsim_score_varlen(fake, 1, 32, 128, fake, None, 10, 100, 0, fake, None, None) == 1


def test_workspace_size_queries(lib):
    assert m.maxsim_score_pq_workspace_size(32, 16, 256) >= 32 * 16 * 256 * 4
    assert m.maxsim_score_pq_workspace_size(0, 16, 256) == 0


def test_streamed_workspace_size(lib):
    """Two document buffers and two length buffers of one chunk, plus score
    and argmax scratch when several queries need the strided scatter (each
    part rounded up to 16 bytes)."""
    import torch
    r16 = lambda x: (x + 15) // 16 * 16
    nQ, nq, nd, d, chunk = 3, 40, 100, 64, 10
    want = 2 * (r16(chunk * nd * d * 2) + r16(chunk * 4)) + r16(nQ * chunk * 4) + r16(nQ * chunk * nq * 4)
    assert m.maxsim_score_streamed_workspace_size(nQ, nq, nd, d, torch.float16, chunk) == want
    one = 2 * (r16(chunk * nd * d * 4) + r16(chunk * 4))        # one query: outputs written in place
    assert m.maxsim_score_streamed_workspace_size(1, nq, nd, d, torch.float32, chunk) == one
    assert m.maxsim_score_streamed_workspace_size(1, nq, nd, d, torch.float32, 0) == 0
    # a missing workspace is rejected before any CUDA call
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert lib.maxsim_score_streamed(fake, 1, 32, 128, fake, 10, 128, None, 0, fake, None, None, 0, 4, None) == 5
    assert lib.maxsim_score_streamed(fake, 1, 32, 128, None, 10, 128, None, 0, fake, None, fake, 1 << 20, 4, None) == 1


def test_product_path_has_no_oracle_or_cpu_fallback():
    """The package and its C sources never import or link the oracle."""
    pkg = os.path.join(ROOT, "maxsim_scoring_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "maxsim_oracle" not in text, f


def test_backward_halves_validate_before_launch(lib):
    """dQ-only and dD-only backward entry points: missing inputs or outputs,
    fp32 inputs and a missing dQ workspace are rejected on the host."""
    P = ctypes.c_void_p
    fake = P(0x1000)
    # dD only: Q missing / dD missing / fp32 unsupported
    assert lib.maxsim_backward_dd(None, 1, 32, 128, 10, 64, None, 0, fake, fake, fake, None) == 1
    assert lib.maxsim_backward_dd(fake, 1, 32, 128, 10, 64, None, 0, fake, fake, None, None) == 1
    assert lib.maxsim_backward_dd(fake, 1, 32, 128, 10, 64, None, 2, fake, fake, fake, None) == 2
    # dQ only: D missing / dQ missing / workspace missing when the range split needs one
    assert lib.maxsim_backward_dq(1, 32, 128, None, 10, 64, None, 0, fake, fake, fake, None, 0, None) == 1
    assert lib.maxsim_backward_dq(1, 32, 128, fake, 10, 64, None, 0, fake, fake, None, None, 0, None) == 1
    assert m.maxsim_backward_workspace_size(1, 32, 128, 5000, 64) > 0
    assert lib.maxsim_backward_dq(1, 32, 128, fake, 5000, 64, None, 0, fake, fake, fake, None, 0, None) == 5


def test_debug_fault_switch_validates_flags(lib):
    """The test-only fault switch rejects unknown bits before touching a device."""
    assert lib.maxsim_debug_set_faults(0x80, 0) == 1


def test_length_order_validates_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # both layouts at once / missing workspace / missing output
    assert lib.maxsim_length_order(fake, fake, 10, 64, fake, fake, 1 << 20, None) == 1
    assert lib.maxsim_length_order(fake, None, 10, 64, fake, None, 0, None) == 5
    assert lib.maxsim_length_order(fake, None, 10, 64, None, fake, 1 << 20, None) == 1
    assert m.maxsim_length_order_workspace_size(10, 64, 0) > 0
    # ordered scoring: fp32 unsupported, missing order rejected
    assert lib.maxsim_score_ordered(fake, 1, 32, 128, fake, 10, 128, None, fake, 2, fake, None, None) == 2
    assert lib.maxsim_score_ordered(fake, 1, 32, 128, fake, 10, 128, None, None, 0, fake, None, None) == 1
