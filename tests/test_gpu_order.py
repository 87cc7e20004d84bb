"""GPU: length-bucketed document order and ordered scoring.

maxsim_length_order must return exactly the stable ascending sort of the
documents by their 8-row granule count (bit-exact against numpy's stable
argsort of the same keys, an index computation). maxsim_score_ordered walks
the documents in that order; a document's result depends only on its own
rows, so scores and argmax must EQUAL those of maxsim_score, which is itself
checked against the fp64 oracle; one case here is also compared with the
oracle directly (TileMaxSim deep reading §5: length-sorted batching).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu
m = pytest.importorskip("maxsim_scoring_02_gb300")
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()


def _expected_order(L, cap=None):
    k = (L.astype(np.int64) + 7) // 8
    if cap is not None:
        k = np.minimum(k, cap)
    return np.argsort(k, kind="stable").astype(np.int32)


@pytest.mark.parametrize("B,lo,hi,nd", [(1, 0, 5, 8), (37, 0, 40, 40), (100_000, 32, 128, 128),
                                        (500_000, 0, 128, 128), (3000, 0, 1024, 1024)])
def test_length_order_is_the_stable_sort_by_granules(B, lo, hi, nd):
    L = workloads.uniform_lengths(B, lo, hi, seed=B + nd)
    order = m.maxsim_length_order(doc_len=L.to(DEV), nd=nd)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    np.testing.assert_array_equal(order.cpu().numpy(), _expected_order(L.numpy()))


def test_length_order_csr_and_long_documents():
    """CSR lengths; documents longer than 8176 tokens share the last bucket."""
    B = 5000
    L = workloads.lognormal_lengths(B, math.log(70), 0.5, 0, 256, seed=41)
    L[:20] = torch.tensor([9000, 0, 8184, 8183, 8191, 1, 7, 8, 9, 20000] * 2, dtype=torch.int32)
    off = workloads.csr_offsets(L)
    order = m.maxsim_length_order(offsets=off.to(DEV))
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    np.testing.assert_array_equal(order.cpu().numpy(), _expected_order(L.numpy(), cap=1023))


def test_bad_lengths_are_reported_and_bucketed_as_empty():
    L = torch.tensor([5, -3, 70, 64, 0, 2], dtype=torch.int32)
    order = m.maxsim_length_order(doc_len=L.to(DEV), nd=64)
    st, flags = m.maxsim_device_status()
    assert st == 1 and flags & m.DEVERR_BAD_INPUT
    np.testing.assert_array_equal(order.cpu().numpy(), _expected_order(np.array([5, 0, 0, 64, 0, 2])))


@pytest.mark.parametrize("n_queries,nq,d,B,nd", [(1, 32, 128, 3000, 128), (3, 40, 64, 1200, 200),
                                                 (2, 200, 256, 700, 96)])
def test_ordered_scoring_equals_index_order(n_queries, nq, d, B, nd):
    Q = workloads.normalized_tokens((n_queries, nq, d), seed=nq + d, dtype="bf16").to(DEV)
    D = workloads.normalized_tokens((B, nd, d), seed=B + nd, dtype="bf16").to(DEV)
    L = workloads.uniform_lengths(B, 0, nd, seed=d).to(DEV)
    order = m.maxsim_length_order(doc_len=L, nd=nd)
    out_o, am_o = m.maxsim_score_ordered(Q, D, order, L, want_argmax=True)
    out, am = m.maxsim_score(Q, D, L, want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    assert torch.equal(out_o, out) and torch.equal(am_o, am)
    # a reversed order as well: any permutation gives the same results
    out_r = m.maxsim_score_ordered(Q, D, torch.flip(order, [0]).contiguous(), L)
    assert torch.equal(out_r, out)


def test_ordered_scoring_against_oracle():
    B, nd, d = 900, 128, 128
    Q = workloads.normalized_tokens((32, d), seed=61, dtype="bf16")
    D = workloads.normalized_tokens((B, nd, d), seed=62, dtype="bf16")
    L = workloads.uniform_lengths(B, 32, nd, seed=63)
    workloads.zero_padding(D, L)
    Ld = L.to(DEV)
    order = m.maxsim_length_order(doc_len=Ld, nd=nd)
    out, am = m.maxsim_score_ordered(Q.to(DEV), D.to(DEV), order, Ld, want_argmax=True)
    torch.cuda.synchronize()
    Qn, Dn = Q[None].double().numpy(), D.double().numpy()
    ref, ref_am, gap = oracle.maxsim(Qn, Dn, L.numpy(), want_gap=True)
    P.check_scores(out.cpu().numpy(), ref, P.TOL_LOWP)
    P.check_argmax(am.cpu().numpy(), ref_am, gap, P.eps_rows(Qn, np.ones(B), d))
    P.check_topk(out.cpu().numpy()[0], ref[0])
