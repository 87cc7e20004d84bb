"""GPU parity: the tcgen05 / FFMA forward kernels against the fp64 oracle.

Sizes span several 128-token tiles, several 64-wide d-slices and ragged
tails; edge cases cover empty documents, length-1 documents, B smaller than
the SM count, multi-query batches with long queries, and corrupt CSR
offsets (reported through the device status word, never a fault).
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
    yield
    st, flags = m.maxsim_device_status()
    assert flags & m.DEVERR_TIMEOUT == 0


def _np(t):
    return t.detach().cpu().to(torch.float64).numpy()


def _run_padded(Q, D, L, dtype_tol, argmax=True):
    out, am = m.maxsim_score(Q.to(DEV), D.to(DEV), None if L is None else L.to(DEV), want_argmax=True)
    torch.cuda.synchronize()
    st, flags = m.maxsim_device_status()
    assert st == 0 and flags == 0, (st, flags)
    Qn = _np(Q if Q.dim() == 3 else Q[None])
    Dn = _np(D)
    ref, ref_am, gap = oracle.maxsim(Qn, Dn, None if L is None else L.numpy(), want_gap=True)
    P.check_scores(out.cpu().numpy(), ref, dtype_tol)
    eps = P.eps_rows(Qn, np.linalg.norm(Dn, axis=-1).max(axis=1), Qn.shape[-1])
    P.check_argmax(am.cpu().numpy(), ref_am, gap, eps)
    P.check_argmax_attains(am.cpu().numpy(), Qn, lambda b: Dn[b], ref_am, eps)
    for q in range(ref.shape[0]):
        P.check_topk(out.cpu().numpy()[q], ref[q])
    return out, am, ref


def test_golden_cases_zero_padded_to_d64(golden_dir):
    """The hand-derived golden cases, with d padded by zeros to 64: integer
    inputs are exact in bf16 and every partial sum is exact, so the GPU must
    reproduce the golden values and argmax exactly."""
    g = json.load(open(os.path.join(golden_dir, "forward_tiny.json")))
    for c in g["cases"]:
        Q = np.array(c["Q"], float)
        D = np.array(c["D"], float)
        Qp = np.zeros(Q.shape[:-1] + (64,)); Qp[..., :Q.shape[-1]] = Q
        Dp = np.zeros(D.shape[:-1] + (64,)); Dp[..., :D.shape[-1]] = D
        L = None if c["doc_len"] is None else torch.tensor(c["doc_len"], dtype=torch.int32, device=DEV)
        for dt in (torch.bfloat16, torch.float16):
            out, am = m.maxsim_score(torch.tensor(Qp, dtype=dt, device=DEV), torch.tensor(Dp, dtype=dt, device=DEV),
                                     L, want_argmax=True)
            np.testing.assert_array_equal(out.cpu().numpy(), np.array(c["score"], np.float32), err_msg=c["name"])
            np.testing.assert_array_equal(am.cpu().numpy(), np.array(c["argmax"]), err_msg=c["name"])
    for c in g["varlen_cases"]:
        Q = np.array(c["Q"], float)
        D = np.array(c["D_packed"], float)
        Qp = np.zeros((Q.shape[0], 64)); Qp[:, :Q.shape[1]] = Q
        Dp = np.zeros((D.shape[0], 64)); Dp[:, :D.shape[1]] = D
        out, am = m.maxsim_score_varlen(torch.tensor(Qp, dtype=torch.bfloat16, device=DEV),
                                        torch.tensor(Dp, dtype=torch.bfloat16, device=DEV),
                                        torch.tensor(c["offsets"], dtype=torch.int64, device=DEV), want_argmax=True)
        np.testing.assert_array_equal(out.cpu().numpy()[0], np.array(c["score"], np.float32))
        np.testing.assert_array_equal(am.cpu().numpy()[0], np.array(c["argmax"]))


def test_pr1_reference_config():
    """Q[32,128], D[1000,128,128] bf16, L2-normalised Gaussian tokens, seed 0."""
    Q = workloads.normalized_tokens((32, 128), seed=0, dtype="bf16")
    D = workloads.normalized_tokens((1000, 128, 128), seed=1, dtype="bf16")
    _run_padded(Q, D, None, P.TOL_LOWP)


@pytest.mark.parametrize("d", [64, 128, 256, 768])
@pytest.mark.parametrize("nd", [32, 200])
def test_padded_ragged_dims(d, nd):
    """Length mask, partial last tiles, d-slices accumulated before the max."""
    B = 157
    Q = workloads.normalized_tokens((32, d), seed=d, dtype="bf16")
    D = workloads.normalized_tokens((B, nd, d), seed=d + nd, dtype="bf16")
    L = workloads.uniform_lengths(B, 0, nd, seed=3)
    L[0], L[1], L[2] = 0, 1, nd
    workloads.zero_padding(D, L)
    _run_padded(Q, D, L, P.TOL_LOWP)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_colbert_shaped_padded_lowp(dtype):
    Q = workloads.normalized_tokens((32, 128), seed=11, dtype=dtype)
    D = workloads.normalized_tokens((2000, 128, 128), seed=12, dtype=dtype)
    L = workloads.uniform_lengths(2000, 32, 128, seed=1)
    workloads.zero_padding(D, L)
    _run_padded(Q, D, L, P.TOL_LOWP)


def test_colbert_shaped_padded_fp32():
    Q = workloads.normalized_tokens((32, 128), seed=21, dtype="fp32")
    D = workloads.normalized_tokens((700, 128, 128), seed=22, dtype="fp32")
    L = workloads.uniform_lengths(700, 32, 128, seed=1)
    workloads.zero_padding(D, L)
    _run_padded(Q, D, L, P.TOL_FP32)


def test_fp32_odd_dims_and_lengths():
    Q = workloads.normalized_tokens((2, 45, 200), seed=23, dtype="fp32")
    D = workloads.normalized_tokens((50, 300, 200), seed=24, dtype="fp32")
    L = workloads.uniform_lengths(50, 0, 300, seed=25)
    _run_padded(Q, D, L, P.TOL_FP32)


@pytest.mark.parametrize("n_queries,nq,d,B,nd", [
    (1, 32, 4, 700, 40),       # d below one 32-dim slice
    (3, 33, 32, 2000, 64),     # one ring stage per (document, query chunk): many hand-offs per CTA
    (2, 64, 60, 300, 129),     # ragged d-slice and a 1-token second tile
    (1, 1, 1024, 20, 300),     # 32 d-slices, single query token, B below the SM count
    (4, 31, 128, 1000, 128),
])
def test_fp32_shapes(n_queries, nq, d, B, nd):
    """The FFMA path over query chunking, d-slicing, token tiles and lengths
    0, 1 and nd; NaN and Inf in the padding rows must never reach a score."""
    Q = workloads.normalized_tokens((n_queries, nq, d), seed=nq + d, dtype="fp32")
    D = workloads.normalized_tokens((B, nd, d), seed=B + nd, dtype="fp32")
    L = workloads.uniform_lengths(B, 0, nd, seed=d)
    L[0], L[1], L[-1] = 0, 1, nd
    Dg = D.clone()
    j = torch.arange(nd)[None, :, None]
    pad = j >= L.long()[:, None, None]
    Dg = torch.where(pad & (j % 2 == 0), torch.full_like(D, float("nan")), Dg)
    Dg = torch.where(pad & (j % 2 == 1), torch.full_like(D, float("inf")), Dg)
    out, am = m.maxsim_score(Q.to(DEV), Dg.to(DEV), L.to(DEV), want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    workloads.zero_padding(D, L)
    Qn, Dn = _np(Q), _np(D)
    ref, ref_am, gap = oracle.maxsim(Qn, Dn, L.numpy(), want_gap=True)
    P.check_scores(out.cpu().numpy(), ref, P.TOL_FP32)
    eps = P.eps_rows(Qn, np.linalg.norm(Dn, axis=-1).max(axis=1), d)
    P.check_argmax(am.cpu().numpy(), ref_am, gap, eps)
    P.check_argmax_attains(am.cpu().numpy(), Qn, lambda b: Dn[b], ref_am, eps)
    assert (out.cpu()[:, 0] == 0).all() and (am.cpu()[:, 0] == -1).all()


@pytest.mark.parametrize("nq", [1, 17, 40, 64, 100, 256, 300])
def test_query_lengths(nq):
    """Query chunking: NC in {32,64,128,256} plus multi-chunk queries."""
    Q = workloads.normalized_tokens((2, nq, 128), seed=nq, dtype="bf16")
    D = workloads.normalized_tokens((40, 150, 128), seed=nq + 1, dtype="bf16")
    L = workloads.uniform_lengths(40, 1, 150, seed=nq + 2)
    _run_padded(Q, D, L, P.TOL_LOWP)


def test_colpali_shaped_small():
    """Long queries and documents (Lq = Ld = 1024), several queries."""
    Q = workloads.normalized_tokens((3, 1024, 128), seed=31, dtype="bf16")
    D = workloads.normalized_tokens((6, 1024, 128), seed=32, dtype="bf16")
    _run_padded(Q, D, None, P.TOL_LOWP)


@pytest.mark.parametrize("nq,d,dtype", [(256, 128, "bf16"), (257, 128, "bf16"), (384, 64, "fp16"),
                                        (512, 128, "bf16"), (513, 128, "fp16"), (500, 192, "bf16"),
                                        (700, 128, "bf16"), (1000, 128, "bf16"), (1024, 64, "bf16"),
                                        (1100, 128, "bf16")])
def test_long_queries(nq, d, dtype):
    """Queries of 256..1100 tokens on CTA pairs: 1 to 4 block pairs (odd and
    even counts), the odd CTA's last block partly or wholly past nq; d=192 and
    1100 tokens take the chunked passes. Lengths cross tile edges (tiles of
    up to 256 columns split between the two CTAs), with empty and length-1
    documents."""
    Q = workloads.normalized_tokens((2, nq, d), seed=nq + d, dtype=dtype)
    D = workloads.normalized_tokens((30, 300, d), seed=nq + d + 1, dtype=dtype)
    L = workloads.uniform_lengths(30, 0, 300, seed=nq + d + 2)
    L[:6] = torch.tensor([0, 1, 128, 129, 256, 300], dtype=L.dtype)
    out, am, _ = _run_padded(Q, D, L, P.TOL_LOWP)
    assert (out[:, 0] == 0).all() and (am[:, 0] == -1).all() and (am[:, 1] == 0).all()
    out_only = m.maxsim_score(Q.to(DEV), D.to(DEV), L.to(DEV))   # no-argmax variant: same sums
    assert torch.equal(out_only.cpu(), out.cpu())


def test_long_queries_varlen_and_small_batches():
    """CSR documents with 700-token queries; batches smaller than the grid
    (1 and 5 documents) and one not divisible by it."""
    for B in (1, 5, 333):
        L = workloads.lognormal_lengths(B, math.log(200), 0.8, 1, 700, seed=B)
        off = workloads.csr_offsets(L)
        Q = workloads.normalized_tokens((3, 700, 128), seed=B + 1, dtype="bf16")
        Dp = workloads.normalized_tokens((int(off[-1]), 128), seed=B + 2, dtype="bf16")
        out, am = m.maxsim_score_varlen(Q.to(DEV), Dp.to(DEV), off.to(DEV), want_argmax=True)
        torch.cuda.synchronize()
        assert m.maxsim_device_status() == (0, 0)
        Qn, Dn, offn = _np(Q), _np(Dp), off.numpy()
        ref, ref_am, gap = oracle.maxsim_varlen(Qn, Dn, offn, want_gap=True)
        P.check_scores(out.cpu().numpy(), ref, P.TOL_LOWP)
        norms = np.array([np.linalg.norm(Dn[offn[b]:offn[b + 1]], axis=1).max() for b in range(B)])
        P.check_argmax(am.cpu().numpy(), ref_am, gap, P.eps_rows(Qn, norms, 128))


def test_long_queries_bad_csr_offsets_reported():
    Q = workloads.normalized_tokens((600, 128), seed=83, dtype="bf16").to(DEV)
    Dp = workloads.normalized_tokens((300, 128), seed=84, dtype="bf16").to(DEV)
    off = torch.tensor([0, 100, 50, 200, 10_000, 300], dtype=torch.int64, device=DEV)
    out, am = m.maxsim_score_varlen(Q, Dp, off, want_argmax=True)
    st, flags = m.maxsim_device_status()
    assert st == 1 and flags & m.DEVERR_BAD_INPUT and flags & m.DEVERR_TIMEOUT == 0
    ref, _, _ = oracle.maxsim_varlen(_np(Q)[None], _np(Dp), np.array([0, 100]))
    assert abs(out[0, 0].item() - ref[0, 0]) <= P.TOL_LOWP
    assert out[0, 1].item() == 0.0 and out[0, 3].item() == 0.0 and (am[0, 1] == -1).all()


def test_colpali_training_size_sampled():
    """ColPali training forward, Q[16,1024,128] x D[10000,1024,128] bf16, in the
    benchmark's launch shape: 6 sampled documents against the oracle."""
    nQ, nq, B, nd, d = 16, 1024, 10_000, 1024, 128
    Q = workloads.normalized_tokens((nQ, nq, d), seed=3, dtype="bf16", device=DEV)
    D = workloads.normalized_tokens((B, nd, d), seed=4, dtype="bf16", device=DEV)
    out, am = m.maxsim_score(Q, D, want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    idx = [0, 1, 4999, 5000, 8191, B - 1]
    _check_sampled(out.cpu().numpy(), am.cpu().numpy(), Q, lambda b: _np(D[b]), idx, P.TOL_LOWP)


def test_identity_scores_exactly_nq():
    """D := Q with exactly unit-norm sign-pattern tokens: score is exactly nq."""
    for nq, nnz in ((32, 16), (40, 64), (128, 4)):
        Qd = workloads.sign_pattern_tokens(nq, 128, nnz, seed=nq)
        Q = Qd.to(torch.bfloat16)
        D = torch.stack([Q, Q.flip(0)])                 # second doc: tokens reversed
        out, am = m.maxsim_score(Q.to(DEV), D.to(DEV), want_argmax=True)
        assert (out.cpu() == float(nq)).all(), out
        am = am.cpu().numpy()[0]
        assert (am[0] == np.arange(nq)).all() and (am[1] == np.arange(nq)[::-1]).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_varlen_csr(dtype):
    B = 600
    L = workloads.lognormal_lengths(B, math.log(70), 0.5, 8, 256, seed=5)
    L[3] = 0
    L[4] = 1
    off = workloads.csr_offsets(L)
    T = int(off[-1])
    Q = workloads.normalized_tokens((32, 128), seed=51, dtype=dtype)
    Dp = workloads.normalized_tokens((T, 128), seed=52, dtype=dtype)
    out, am = m.maxsim_score_varlen(Q.to(DEV), Dp.to(DEV), off.to(DEV), want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    Qn, Dn, offn = _np(Q)[None], _np(Dp), off.numpy()
    ref, ref_am, gap = oracle.maxsim_varlen(Qn, Dn, offn, want_gap=True)
    tol = P.TOL_FP32 if dtype == "fp32" else P.TOL_LOWP
    P.check_scores(out.cpu().numpy(), ref, tol)
    norms = np.array([np.linalg.norm(Dn[offn[b]:offn[b + 1]], axis=1).max() if offn[b + 1] > offn[b] else 1.0
                      for b in range(B)])
    eps = P.eps_rows(Qn, norms, 128)
    P.check_argmax(am.cpu().numpy(), ref_am, gap, eps)
    P.check_topk(out.cpu().numpy()[0], ref[0])
    assert out[0, 3].item() == 0.0 and (am[0, 3] == -1).all()


def test_padding_values_never_contribute():
    """Huge values in the padding rows (beyond L_b) leave scores unchanged."""
    B, nd = 64, 160
    Q = workloads.normalized_tokens((32, 128), seed=61, dtype="bf16").to(DEV)
    D = workloads.normalized_tokens((B, nd, 128), seed=62, dtype="bf16").to(DEV)
    L = workloads.uniform_lengths(B, 0, nd, seed=63).to(DEV)
    a = m.maxsim_score(Q, D, L).clone()
    j = torch.arange(nd, device=DEV)[None, :, None]
    D2 = torch.where(j >= L.long()[:, None, None], torch.full_like(D, 100.0), D)
    b = m.maxsim_score(Q, D2, L)
    assert torch.equal(a, b)


def test_small_batches_and_single_docs():
    for B in (1, 2, 151, 153):
        Q = workloads.normalized_tokens((32, 128), seed=B, dtype="bf16")
        D = workloads.normalized_tokens((B, 130, 128), seed=B + 1, dtype="bf16")
        _run_padded(Q, D, None, P.TOL_LOWP)


def test_empty_and_zero_length_inputs():
    Q = workloads.normalized_tokens((32, 128), seed=71, dtype="bf16").to(DEV)
    D = workloads.normalized_tokens((5, 64, 128), seed=72, dtype="bf16").to(DEV)
    L = torch.zeros(5, dtype=torch.int32, device=DEV)
    out, am = m.maxsim_score(Q, D, L, want_argmax=True)
    assert (out == 0).all() and (am == -1).all()
    out0 = m.maxsim_score(Q, D[:0])
    assert out0.shape == (1, 0)


def test_bad_csr_offsets_are_reported_not_faulted():
    """Offsets pointing outside the packed rows: the kernel's own checks score
    those documents as empty and set the bad-input bit; valid ones are scored."""
    Q = workloads.normalized_tokens((32, 128), seed=81, dtype="bf16").to(DEV)
    Dp = workloads.normalized_tokens((300, 128), seed=82, dtype="bf16").to(DEV)
    off = torch.tensor([0, 100, 50, 200, 10_000, 300], dtype=torch.int64, device=DEV)
    out = m.maxsim_score_varlen(Q, Dp, off)
    st, flags = m.maxsim_device_status()
    assert st == 1 and flags & m.DEVERR_BAD_INPUT
    ref, _, _ = oracle.maxsim_varlen(_np(Q)[None], _np(Dp), np.array([0, 100]))
    assert abs(out[0, 0].item() - ref[0, 0]) <= P.TOL_LOWP
    assert out[0, 1].item() == 0.0 and out[0, 3].item() == 0.0


def test_headline_size_sampled():
    """Q[32,128] x D[100000,128,128] bf16 in the benchmark's launch shape;
    512 sampled documents checked against the oracle one by one, and the
    scores of a permuted copy of a document slab match exactly."""
    B = 100_000
    Q = workloads.normalized_tokens((32, 128), seed=0, dtype="bf16", device=DEV)
    D = workloads.normalized_tokens((B, 128, 128), seed=1, dtype="bf16", device=DEV)
    out, am = m.maxsim_score(Q, D, want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    idx = torch.randperm(B, generator=torch.Generator().manual_seed(5))[:512]
    idx[0], idx[1] = 0, B - 1
    Qn = _np(Q)[None]
    Dn = _np(D[idx.to(DEV)])
    ref, ref_am, gap = oracle.maxsim(Qn, Dn, want_gap=True)
    P.check_scores(out.cpu().numpy()[:, idx.numpy()], ref, P.TOL_LOWP)
    eps = P.eps_rows(Qn, np.linalg.norm(Dn, axis=-1).max(axis=1), 128)
    P.check_argmax(am.cpu().numpy()[:, idx.numpy()], ref_am, gap, eps)
    # token permutation invariance at full size (exact: same products, same tiles)
    perm = torch.randperm(128, device=DEV)
    out2 = m.maxsim_score(Q, D[:2048][:, perm].contiguous())
    assert torch.allclose(out2, out[:, :2048], atol=2e-6, rtol=0)


def _check_sampled(out, am, Q, docs_of, idx, tol):
    """Oracle on a sample of documents; docs_of(b) -> fp64 [L_b, d]."""
    Qn = _np(Q if Q.dim() == 3 else Q[None])
    for b in idx:
        rows = docs_of(b)
        ref, ref_am, gap = oracle.maxsim(Qn, rows[None] if rows.shape[0] else np.zeros((1, 1, Qn.shape[-1])),
                                         None if rows.shape[0] else [0], want_gap=True)
        got = out[:, b]
        assert np.abs(got - ref[:, 0]).max() <= tol, (b, got, ref[:, 0])
        if am is not None:
            norms = np.linalg.norm(rows, axis=1).max() if rows.shape[0] else 1.0
            eps = P.eps_rows(Qn, np.array([norms]), Qn.shape[-1])
            P.check_argmax(am[:, b:b + 1], ref_am, gap, eps)


def test_long_documents_split_across_groups():
    """Single query: documents longer than one 256-chunk group (8192 tokens)
    continue across groups with their running maxima intact."""
    B, nd, d = 3, 9000, 64
    Q = workloads.normalized_tokens((32, d), seed=91, dtype="bf16")
    D = workloads.normalized_tokens((B, nd, d), seed=92, dtype="bf16")
    L = torch.tensor([9000, 8193, 300], dtype=torch.int32)
    _run_padded(Q, D, L, P.TOL_LOWP)


def test_many_short_csr_documents():
    """Thousands of 1..40-token documents: many groups per CTA, many documents
    per tile, empty documents interleaved."""
    B = 6000
    L = workloads.uniform_lengths(B, 0, 40, seed=93)
    off = workloads.csr_offsets(L)
    Q = workloads.normalized_tokens((32, 128), seed=94, dtype="bf16")
    Dp = workloads.normalized_tokens((int(off[-1]), 128), seed=95, dtype="bf16")
    out, am = m.maxsim_score_varlen(Q.to(DEV), Dp.to(DEV), off.to(DEV), want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    Qn, Dn, offn = _np(Q)[None], _np(Dp), off.numpy()
    ref, ref_am, gap = oracle.maxsim_varlen(Qn, Dn, offn, want_gap=True)
    P.check_scores(out.cpu().numpy(), ref, P.TOL_LOWP)
    norms = np.array([np.linalg.norm(Dn[offn[b]:offn[b + 1]], axis=1).max() if offn[b + 1] > offn[b] else 1.0
                      for b in range(B)])
    P.check_argmax(am.cpu().numpy(), ref_am, gap, P.eps_rows(Qn, norms, 128))


@pytest.mark.parametrize("nq", [32, 300])
def test_multi_query_many_groups(nq):
    """Several queries over CTA ranges of > 256 documents: several groups, each
    scored for every (query, query chunk) pass; sampled against the oracle."""
    B, nd = 50_000, 32
    Q = workloads.normalized_tokens((2, nq, 128), seed=96, dtype="bf16", device=DEV)
    D = workloads.normalized_tokens((B, nd, 128), seed=97, dtype="bf16", device=DEV)
    L = workloads.uniform_lengths(B, 0, nd, seed=98, device=DEV)
    out, am = m.maxsim_score(Q, D, L, want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    idx = torch.randperm(B, generator=torch.Generator().manual_seed(7))[:300].tolist() + [0, B - 1]
    Lc = L.cpu().numpy()
    _check_sampled(out.cpu().numpy(), am.cpu().numpy(), Q, lambda b: _np(D[b, :Lc[b]]), idx, P.TOL_LOWP)


@pytest.mark.parametrize("nq,d,B,nd,csr", [
    (32, 128, 500, 128, False),    # the configured shape: one 64-dim slice pair, four-slot tiles
    (1, 64, 300, 70, False),       # one query token, one slice, ragged tiles
    (20, 256, 200, 200, False),    # four slices, query rows past nq zero
    (33, 128, 400, 129, False),    # 64-column query chunk (N = 192), a 1-row second tile
    (64, 64, 157, 300, True),      # CSR, 64 query tokens
    (32, 128, 3000, 40, True),     # many short CSR documents sharing tiles
])
def test_fp32_tensor_core_split(nq, d, B, nd, csr):
    """fp32 inputs on the tensor cores: each value split into three bf16
    parts, all nine part products accumulated in fp32. Scores within the
    fp32 tolerance of the oracle, argmax by the near-tie rule; NaN and Inf in
    the padding rows never reach a score."""
    Q = workloads.normalized_tokens((nq, d), seed=nq * 7 + d, dtype="fp32")
    D = workloads.normalized_tokens((B, nd, d), seed=B + nd + d, dtype="fp32")
    L = workloads.uniform_lengths(B, 0, nd, seed=nq + d)
    L[0], L[1], L[-1] = 0, 1, nd
    if csr:
        off = workloads.csr_offsets(L)
        Dp = torch.cat([D[b, :L[b]] for b in range(B)])
        out, am = m.maxsim_score_varlen(Q.to(DEV), Dp.to(DEV), off.to(DEV), want_argmax=True)
    else:
        j = torch.arange(nd)[None, :, None]
        pad = j >= L.long()[:, None, None]
        Dg = torch.where(pad & (j % 2 == 0), torch.full_like(D, float("nan")), D)
        Dg = torch.where(pad & (j % 2 == 1), torch.full_like(D, float("inf")), Dg)
        out, am = m.maxsim_score(Q.to(DEV), Dg.to(DEV), L.to(DEV), want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    workloads.zero_padding(D, L)
    Qn, Dn = _np(Q)[None], _np(D)
    ref, ref_am, gap = oracle.maxsim(Qn, Dn, L.numpy(), want_gap=True)
    P.check_scores(out.cpu().numpy(), ref, P.TOL_FP32)
    eps = P.eps_rows(Qn, np.linalg.norm(Dn, axis=-1).max(axis=1), d)
    P.check_argmax(am.cpu().numpy(), ref_am, gap, eps)
    P.check_argmax_attains(am.cpu().numpy(), Qn, lambda b: Dn[b], ref_am, eps)
    assert (out.cpu()[:, 0] == 0).all() and (am.cpu()[:, 0] == -1).all()


@pytest.mark.parametrize("nq", [32, 256])
@pytest.mark.parametrize("K", [37, 200])
def test_argmax_exact_ties_pick_the_first_occurrence(nq, K):
    """Documents of 512 tokens built from K distinct tokens each: position t
    of document b holds base token (3t + 5b) mod K, so every token recurs
    across 32-row slots, 128-row tiles, 32-column chunks and rounds of four
    chunks, and positions 0 .. K-1 are exactly the first occurrences. Equal
    tokens give bit-identical similarities, so the argmax (lowest index among
    exact ties) must lie below K. Its token must be the oracle's best token of
    the base set wherever the best two differ by more than the fp32 bound.
    nq = 32 runs the short-query kernel, nq = 256 the long-query one."""
    d, nd, B = 128, 512, 64
    base = workloads.normalized_tokens((B, K, d), seed=1201 + K, dtype="bf16")
    pos = (3 * torch.arange(nd)[None, :] + 5 * torch.arange(B)[:, None]) % K       # [B, nd]
    D = torch.gather(base, 1, pos[:, :, None].expand(B, nd, d))
    Q = workloads.normalized_tokens((nq, d), seed=1202 + nq, dtype="bf16")
    _, am = m.maxsim_score(Q.to(DEV), D.to(DEV), want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    am = am.cpu().numpy()[0]                                                       # [B, nq]
    assert (am >= 0).all() and (am < K).all(), int((am >= K).sum())
    _, ref_tok, gap = oracle.maxsim(Q[None].double().numpy(), base.double().numpy(), want_gap=True)
    got_tok = np.take_along_axis(pos.numpy(), am, axis=1)
    eps = P.eps_rows(Q[None].double().numpy(), np.ones(B), d)
    sure = gap[0] >= eps[0]
    assert sure.mean() > 0.9
    assert (got_tok == ref_tok[0])[sure].all()
