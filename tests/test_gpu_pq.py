"""GPU parity: fused PQ table-lookup scoring against the fp64 oracle.

Tolerance (the sources state none for PQ): |score - oracle| <= 2e-4 *
max(1, |oracle|); PQ scores are O(10-100) with N(0,1) codebooks. Argmax is
bit-exact wherever the oracle's top-2 gap exceeds the fp32 summation bound
of the 16 table terms.
"""
import json
import math
import os

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


def _case(B, nq, d, M, K, seed, lo=8, hi=256, empty=()):
    L = workloads.lognormal_lengths(B, math.log(70), 0.5, lo, hi, seed=seed)
    for e in empty:
        L[e] = 0
    off = workloads.csr_offsets(L)
    C, codes = workloads.pq_inputs(int(off[-1]), M, K, d, seed=seed + 1)
    Q = workloads.normalized_tokens((nq, d), seed=seed + 2, dtype="fp32")
    return Q, C, codes, off


def _check(Q, C, codes, off, want_argmax=True):
    out, am = m.maxsim_score_pq(Q.to(DEV), C.to(DEV), codes.to(DEV), off.to(DEV), want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    Qn, Cn, cn, offn = Q.double().numpy(), C.double().numpy(), codes.numpy(), off.numpy()
    T = oracle.pq_table(Qn, Cn)
    ref, ref_am = oracle.maxsim_pq(T, cn, offn)
    out = out.cpu().numpy().astype(np.float64)
    err = np.abs(out - ref) / np.maximum(1.0, np.abs(ref))
    assert err.max() <= 2e-4, err.max()
    # near-tie rule: gaps from the decode route (equal to the table route, pinned on CPU)
    _, _, gap = oracle.maxsim_varlen(Qn, oracle.pq_decode(Cn, cn), offn, want_gap=True)
    M = T.shape[1]
    eps = 8.0 * M * 2.0 ** -24 * np.abs(T).max(axis=2).sum(axis=1)          # [nq]
    sure = gap[0] >= eps[None, :]
    bad = (am.cpu().numpy() != ref_am) & sure
    assert not bad.any(), int(bad.sum())
    P.check_topk(out, ref)
    return out, am


def test_golden_case_embedded_in_four_subspaces(golden_dir):
    """The hand-derived PQ case (d=4, M=2) with two extra all-zero subspaces:
    their table entries are exactly 0, so score and argmax are the golden ones."""
    g = json.load(open(os.path.join(golden_dir, "pq_tiny.json")))
    Q = torch.zeros(1, 8)
    Q[0, :4] = torch.tensor(g["Q"][0], dtype=torch.float32)
    C = torch.zeros(4, 2, 2)
    C[:2] = torch.tensor(g["C"], dtype=torch.float32)
    codes = torch.zeros(2, 4, dtype=torch.uint8)
    codes[:, :2] = torch.tensor(g["codes"], dtype=torch.uint8)
    off = torch.tensor(g["offsets"], dtype=torch.int64)
    out, am = m.maxsim_score_pq(Q.to(DEV), C.to(DEV), codes.to(DEV), off.to(DEV), want_argmax=True)
    assert out.cpu().tolist() == [float(v) for v in g["score"]]
    assert am.cpu().tolist() == g["argmax"]


def test_config_shaped_pq():
    """M=16 subspaces of 8 dims, K=256 N(0,1) centroids, uniform uint8 codes,
    lognormal(ln 70, 0.5) lengths clipped to [8, 256], Q[32,128] fp32."""
    _check(*_case(3000, 32, 128, 16, 256, seed=101, empty=(5, 17)))


@pytest.mark.parametrize("nq,M,K,d", [(40, 8, 100, 64), (1, 4, 256, 32), (9, 32, 64, 128), (17, 64, 16, 256),
                                     (20, 16, 256, 128), (1, 16, 256, 64)])
def test_pq_shapes(nq, M, K, d):
    _check(*_case(400, nq, d, M, K, seed=nq + M, lo=1, hi=90, empty=(0, 399)))


def test_pq_many_docs_sampled():
    """B=100000 documents in the benchmark's launch shape; 400 sampled documents
    against the oracle."""
    Q, C, codes, off = _case(100_000, 32, 128, 16, 256, seed=111)
    out = m.maxsim_score_pq(Q.to(DEV), C.to(DEV), codes.to(DEV), off.to(DEV))
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    idx = np.sort(np.random.default_rng(3).choice(100_000, 400, replace=False))
    offn = off.numpy()
    T = oracle.pq_table(Q.double().numpy(), C.double().numpy())
    cn = codes.numpy()
    for b in idx:
        sub = cn[offn[b]:offn[b + 1]]
        ref, _ = oracle.maxsim_pq(T, sub, np.array([0, sub.shape[0]]))
        got = float(out[b].item())
        assert abs(got - ref[0]) <= 2e-4 * max(1.0, abs(ref[0])), (b, got, ref[0])


def test_out_of_range_codes_are_clamped_and_reported():
    """With K=10 a code of 200 is outside the codebook: the kernel clamps it to
    K-1 (never reading past the table) and sets the bad-input bit."""
    Q, C, codes, off = _case(50, 32, 64, 8, 10, seed=121, lo=4, hi=30)
    codes = codes % 10
    codes[3, 2] = 200
    m.maxsim_score_pq(Q.to(DEV), C.to(DEV), codes.to(DEV), off.to(DEV))
    st, flags = m.maxsim_device_status()
    assert st == 1 and flags & m.DEVERR_BAD_INPUT


def test_workspace_errors():
    Q, C, codes, off = _case(10, 32, 128, 16, 256, seed=131)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(m.MaxSimError) as ei:
        m.maxsim_score_pq(Q.to(DEV), C.to(DEV), codes.to(DEV), off.to(DEV), workspace=small)
    assert ei.value.status == 5
