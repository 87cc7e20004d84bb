"""GPU: failure detection of the bounded pipeline waits, without a GPU fault.

Every wait of the library's pipelined kernels is bounded: when it runs out,
the kernel records MAXSIM_DEVERR_TIMEOUT in the device status word, raises
its abort flag, and every role drains what it has in flight and exits, so
the CUDA context stays usable. This test makes a wait run out on purpose
through the test-only switch maxsim_debug_set_faults: the tensor-core
forward kernel's loader issues nothing, so the other roles wait on barriers
that no one completes. With a 50 ms bound the call must report
MAXSIM_ERR_TIMEOUT through maxsim_device_status, and the next normal call on
the same stream must score exactly as before and match the fp64 oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu
m = pytest.importorskip("maxsim_scoring_02_gb300")
DEV = "cuda"
TIMEOUT_STATUS = 4


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = m.load_library()
    yield lib
    assert lib.maxsim_debug_set_faults(0, 0) == 0


@pytest.mark.parametrize("layout", ["padded", "csr"])
def test_wait_timeout_is_reported_and_the_next_call_is_correct(lib, layout):
    B, nd, d = 300, 128, 128
    Q = workloads.normalized_tokens((32, d), seed=901, dtype="bf16")
    D = workloads.normalized_tokens((B, nd, d), seed=902, dtype="bf16")
    L = workloads.uniform_lengths(B, 0, nd, seed=903)
    off = workloads.csr_offsets(L)
    Dp = torch.cat([D[b, :L[b]] for b in range(B)])
    Qd, Dd, Ld, Dpd, offd = Q.to(DEV), D.to(DEV), L.to(DEV), Dp.to(DEV), off.to(DEV)

    def score():
        if layout == "padded":
            return m.maxsim_score(Qd, Dd, Ld, want_argmax=True)
        return m.maxsim_score_varlen(Qd, Dpd, offd, want_argmax=True)

    ref_out, ref_am = score()
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)

    assert lib.maxsim_debug_set_faults(m.DEBUG_STALL_FWD_LOADER, 50_000_000) == 0
    try:
        score()                                   # the loader stalls: the waits run out
        st, flags = m.maxsim_device_status()      # synchronises the stream: the kernel has exited
        assert st == TIMEOUT_STATUS and flags & m.DEVERR_TIMEOUT, (st, flags)
    finally:
        assert lib.maxsim_debug_set_faults(0, 0) == 0

    out, am = score()
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    assert torch.equal(out, ref_out) and torch.equal(am, ref_am)
    ref, ref_amo, gap = oracle.maxsim(Q[None].double().numpy(), D.double().numpy(), L.numpy(), want_gap=True)
    P.check_scores(out.cpu().numpy(), ref, P.TOL_LOWP)
    eps = P.eps_rows(Q[None].double().numpy(), np.ones(B), d)
    P.check_argmax(am.cpu().numpy(), ref_amo, gap, eps)


def test_unknown_fault_flags_are_rejected(lib):
    assert lib.maxsim_debug_set_faults(0x80, 0) == 1


@pytest.mark.parametrize("kind", ["bf16_scores_only", "fp32_split", "i8_scores_only"])
def test_wait_timeout_in_the_other_tensor_core_kernels(lib, kind):
    """The same stall in the other pipelined kernels' loaders: the two-group
    bf16 launch (scores only), the fp32 three-part kernel and the scores-only
    INT8 kernel. Each reports MAXSIM_ERR_TIMEOUT and then scores exactly as
    before."""
    B, d = 300, 128
    L = workloads.uniform_lengths(B, 0, 128, seed=911)
    off = workloads.csr_offsets(L)
    if kind == "i8_scores_only":
        Qi, sq = workloads.quantize_int8(workloads.normalized_tokens((32, d), seed=912, dtype="fp32"))
        Di, sd = workloads.quantize_int8(workloads.normalized_tokens((int(off[-1]), d), seed=913, dtype="fp32"))
        args = (Qi.to(DEV), sq.to(DEV), Di.to(DEV), sd.to(DEV), off.to(DEV))
        score = lambda: m.maxsim_score_i8(*args)
    else:
        dt = "bf16" if kind == "bf16_scores_only" else "fp32"
        Q = workloads.normalized_tokens((32, d), seed=914, dtype=dt).to(DEV)
        D = workloads.normalized_tokens((B, 128, d), seed=915, dtype=dt).to(DEV)
        Ld = L.to(DEV)
        score = lambda: m.maxsim_score(Q, D, Ld)

    ref = score()
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    assert lib.maxsim_debug_set_faults(m.DEBUG_STALL_FWD_LOADER, 50_000_000) == 0
    try:
        score()
        st, flags = m.maxsim_device_status()
        assert st == TIMEOUT_STATUS and flags & m.DEVERR_TIMEOUT, (st, flags)
    finally:
        assert lib.maxsim_debug_set_faults(0, 0) == 0
    out = score()
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    assert torch.equal(out, ref)
