"""GPU parity at the benchmarked sizes, in the benchmark's launch shape.

Every throughput row reported for the padded, length-masked, shape-sweep and
CSR workloads is measured on these exact inputs (same generators, same seeds
as ``bench.py`` for rank 0), so each is checked here at full size: the call
the benchmark times (scores only) and the argmax variant both run over all B
documents, and a seeded sample of documents -- plus the first and last, and
the shortest and longest -- is compared with the fp64 oracle under the rules
of ``tests/_parity.py``. The sample is gathered into one batch for a single
oracle call; scores of the two launches are also compared with each other.

Workloads (TileMaxSim deep reading §4: B, Nd and d scaling; §5: length mask
and padding; FLASH-MAXSIM Abstract: variable-length CSR scoring):
  * Q[32,128] x D[500000,128,128] bf16, lengths U{32..128}, zero padding;
  * the same at B = 100000 and 500000 in fp16 and in fp32 (tcgen05 on three
    bf16 parts of each fp32 value);
  * Q[32,768] x D[100000,512,768] bf16 and Q[32,64] x D[100000,32,64] bf16,
    full length (the corners of the d x Nd sweep);
  * Q[32,128] against 500000 CSR documents, lengths round(lognormal(ln 70,
    0.5)) clipped to [8, 256], bf16 and fp32.
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
N_SAMPLE = 300


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    yield
    torch.cuda.empty_cache()


@pytest.fixture(autouse=True)
def _release():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _np(t):
    return t.detach().cpu().to(torch.float64).numpy()


def _sample(B, lengths, seed):
    idx = torch.randperm(B, generator=torch.Generator().manual_seed(seed))[:N_SAMPLE].tolist()
    idx += [0, B - 1]
    if lengths is not None:
        L = lengths.cpu()
        idx += [int(torch.argmin(L)), int(torch.argmax(L))]
    return sorted(set(idx))


def _check(out_fast, out, am, Qn, docs, lens, idx, tol):
    """docs [S, n, d] fp64 (rows past lens[s] ignored by the oracle)."""
    ref, ref_am, gap = oracle.maxsim(Qn, docs, lens, want_gap=True)
    for o in (out_fast, out):
        P.check_scores(o.cpu().numpy()[:, idx], ref, tol)
    norms = np.array([np.linalg.norm(docs[s, :max(int(lens[s]) if lens is not None else docs.shape[1], 1)],
                                     axis=1).max() for s in range(len(idx))])
    eps = P.eps_rows(Qn, norms, Qn.shape[-1])
    a = am.cpu().numpy()[:, idx]
    P.check_argmax(a, ref_am, gap, eps)
    P.check_argmax_attains(a, Qn, lambda s: docs[s], ref_am, eps)
    P.check_topk(out.cpu().numpy()[0, idx], ref[0])
    assert torch.allclose(out_fast, out, atol=tol, rtol=0)


def _padded_case(B, nd, d, dtype, lenmask):
    """bench.py Headline workload, rank 0 (Q seed 0, D seed 1, lengths seed 2)."""
    Q = workloads.normalized_tokens((32, d), seed=0, dtype=dtype, device=DEV)
    D = workloads.normalized_tokens((B, nd, d), seed=1, dtype=dtype, device=DEV)
    L = None
    if lenmask:
        L = workloads.uniform_lengths(B, 32, nd, seed=2, device=DEV)
        workloads.zero_padding(D, L)
    out_fast = m.maxsim_score(Q, D, L)                 # the benchmark's call
    out, am = m.maxsim_score(Q, D, L, want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    idx = _sample(B, L, seed=B + nd + d)
    it = torch.tensor(idx, device=DEV)
    docs = _np(D[it])
    lens = None if L is None else L[it].cpu().numpy()
    tol = P.TOL_FP32 if dtype == "fp32" else P.TOL_LOWP
    _check(out_fast, out, am, _np(Q)[None], docs, lens, idx, tol)


def test_lenmask_b500k_bf16():
    _padded_case(500_000, 128, 128, "bf16", True)


@pytest.mark.parametrize("B", [100_000, 500_000])
@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_lenmask_fp16_fp32(dtype, B):
    _padded_case(B, 128, 128, dtype, True)


@pytest.mark.parametrize("nd,d", [(512, 768), (32, 64)])
def test_sweep_corners_b100k(nd, d):
    _padded_case(100_000, nd, d, "bf16", False)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_csr_b500k(dtype):
    """bench.py Varlen workload, rank 0 (lengths seed 50, Q seed 51, D seed 52)."""
    B = 500_000
    L = workloads.lognormal_lengths(B, math.log(70), 0.5, 8, 256, seed=50, device=DEV)
    off = workloads.csr_offsets(L)
    T = int(off[-1].item())
    Q = workloads.normalized_tokens((32, 128), seed=51, dtype=dtype, device=DEV)
    Dp = workloads.normalized_tokens((T, 128), seed=52, dtype=dtype, device=DEV)
    out_fast = m.maxsim_score_varlen(Q, Dp, off)
    out, am = m.maxsim_score_varlen(Q, Dp, off, want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    idx = _sample(B, L, seed=7)
    offc = off.cpu().numpy()
    Lc = L.cpu().numpy()
    docs = np.zeros((len(idx), int(Lc[idx].max()), 128))
    for s, b in enumerate(idx):
        docs[s, :Lc[b]] = _np(Dp[offc[b]:offc[b + 1]])
    _check(out_fast, out, am, _np(Q)[None], docs, Lc[idx], idx, P.TOL_FP32 if dtype == "fp32" else P.TOL_LOWP)
