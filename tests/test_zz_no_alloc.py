"""maxsim_score_pq_noalloc: PQ scoring for callers that cannot allocate.

Callers such as host callbacks, hooks inside other libraries or plugins
without an allocator cannot create the table workspace that maxsim_score_pq
needs; this entry point keeps the table in the library's fixed device array
instead. The test calls it directly through the C ABI, twice in a row with
different table shapes (the second table is smaller, so entries left from
the first call must not leak into it), and compares each result with the
regular workspace entry point at the PQ tolerance of the other tests
(2e-4 * max(1, |score|)); argmax must be identical since both calls run the
same kernels on the same table values. It also checks that a table larger
than the fixed array is refused before anything runs.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
m = pytest.importorskip("maxsim_scoring_02_gb300")
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return m.load_library()


def _inputs(B, nq, d, M, K, seed):
    L = workloads.lognormal_lengths(B, math.log(70), 0.5, 1, 200, seed=seed)
    L[1] = 0
    off = workloads.csr_offsets(L)
    C, codes = workloads.pq_inputs(int(off[-1]), M, K, d, seed=seed + 1)
    Q = workloads.normalized_tokens((nq, d), seed=seed + 2, dtype="fp32")
    return Q.to(DEV), C.to(DEV), codes.to(DEV), off.to(DEV)


def _call_noalloc(lib, Q, C, codes, off):
    nq, d = Q.shape
    M, K, _ = C.shape
    B = off.numel() - 1
    out = torch.full((B,), float("nan"), device=DEV)
    am = torch.full((B, nq), -7, dtype=torch.int32, device=DEV)
    P = ctypes.c_void_p
    st = lib.maxsim_score_pq_noalloc(P(Q.data_ptr()), nq, d, P(C.data_ptr()), M, K, P(codes.data_ptr()),
                                     P(off.data_ptr()), B, codes.shape[0], P(out.data_ptr()), P(am.data_ptr()),
                                     P(torch.cuda.current_stream().cuda_stream))
    return st, out, am


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    for args in ((4000, 32, 128, 16, 256, 301), (1500, 20, 64, 8, 100, 311)):
        Q, C, codes, off = _inputs(*args)
        st, out, am = _call_noalloc(lib, Q, C, codes, off)
        assert st == 0, m.STATUS_NAMES.get(st, st)
        ref, ref_am = m.maxsim_score_pq(Q, C, codes, off, want_argmax=True)
        torch.cuda.synchronize()
        assert m.maxsim_device_status() == (0, 0)
        o, r = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(o).all()
        assert (np.abs(o - r) <= 2e-4 * np.maximum(1.0, np.abs(r))).all()
        assert torch.equal(am.cpu(), ref_am.cpu())


def test_noalloc_refuses_tables_beyond_its_capacity(lib):
    Q, C, codes, off = _inputs(10, 72, 128, 16, 256, 321)   # 9 groups x 128 KB > 1 MiB
    st, out, _ = _call_noalloc(lib, Q, C, codes, off)
    assert st == 5                                           # MAXSIM_ERR_WORKSPACE
    assert torch.isnan(out.cpu()).all()                      # nothing was launched
