"""GPU parity: INT8 x INT8 scoring against the oracle.

Both sides form sim = (float)dot * s_d[j] as one fp32 round-to-nearest
multiply of an exact integer dot, and compare in fp32 with the lowest index
winning ties; so the per-token maxima, their integer dots and their indices
must match BIT-EXACTLY. The score (a sum of nq fp32 products) is checked to
1e-5 * sum_i |s_q[i] * m_i|.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
m = pytest.importorskip("maxsim_scoring_02_gb300")
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()


def _inputs(B, nq, d, seed, lo=8, hi=256, empty=()):
    L = workloads.lognormal_lengths(B, math.log(70), 0.5, lo, hi, seed=seed)
    for e in empty:
        L[e] = 0
    off = workloads.csr_offsets(L)
    Qf = workloads.normalized_tokens((nq, d), seed=seed + 1, dtype="fp32")
    Df = workloads.normalized_tokens((int(off[-1]), d), seed=seed + 2, dtype="fp32")
    Qi, sq = workloads.quantize_int8(Qf)
    Di, sd = workloads.quantize_int8(Df)
    return Qi, sq, Di, sd, off


def _check(Qi, sq, Di, sd, off):
    out, mv, md, am = m.maxsim_score_i8(Qi.to(DEV), sq.to(DEV), Di.to(DEV), sd.to(DEV), off.to(DEV),
                                        want_details=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    ref, rmv, rmd, ram = oracle.maxsim_i8(Qi.numpy(), sq.numpy(), Di.numpy(), sd.numpy(), off.numpy())
    np.testing.assert_array_equal(md.cpu().numpy(), rmd)
    np.testing.assert_array_equal(mv.cpu().numpy(), rmv)
    np.testing.assert_array_equal(am.cpu().numpy(), ram)
    bound = 1e-5 * np.maximum(np.abs(sq.numpy()[None, :].astype(np.float64) * rmv).sum(axis=1), 1e-30)
    assert (np.abs(out.cpu().numpy() - ref) <= bound).all()
    return out


def test_golden_case_embedded_in_d64(golden_dir):
    """The hand-derived INT8 case with d padded by zeros to 64: same dots,
    same fp32 products, so every output equals the golden value exactly."""
    g = json.load(open(os.path.join(golden_dir, "i8_tiny.json")))
    Q = torch.zeros(2, 64, dtype=torch.int8)
    Q[:, :2] = torch.tensor(g["Q"], dtype=torch.int8)
    D = torch.zeros(3, 64, dtype=torch.int8)
    D[:, :2] = torch.tensor(g["D"], dtype=torch.int8)
    out, mv, md, am = m.maxsim_score_i8(Q.to(DEV), torch.tensor(g["s_q"], device=DEV), D.to(DEV),
                                        torch.tensor(g["s_d"], device=DEV),
                                        torch.tensor(g["offsets"], device=DEV), want_details=True)
    assert out.cpu().tolist() == g["score"]
    assert mv.cpu().tolist() == g["maxv"] and md.cpu().tolist() == g["maxdot"] and am.cpu().tolist() == g["argmax"]


def test_config_shaped_i8():
    """Per-token symmetric INT8 of L2-normalised Gaussian tokens, d=128,
    Q[32,128], lognormal(ln 70, 0.5) lengths clipped to [8, 256]."""
    _check(*_inputs(3000, 32, 128, seed=201, empty=(3, 2999)))


@pytest.mark.parametrize("nq,d", [(1, 64), (20, 128), (32, 192), (45, 256), (64, 512), (100, 768), (7, 1024)])
def test_i8_shapes(nq, d):
    _check(*_inputs(300, nq, d, seed=nq + d, lo=1, hi=100, empty=(0,)))


@pytest.mark.parametrize("d", [64, 128, 192])
def test_i8_tile_boundaries(d):
    """Runs of 0-3-token documents (up to 128 documents share one 128-row
    tile), documents of 127, 128, 129, 255, 256 and 257 tokens starting at
    shifting row alignments, and documents whose rows and scales are all
    equal, so every similarity ties and the argmax must be the first token."""
    rng = np.random.default_rng(d)
    L = []
    for _ in range(6):
        L += list(rng.integers(0, 4, size=150))
        L += [127, 128, 129, 255, 256, 257, 1, 0, 2, 5]
    L = torch.tensor(L, dtype=torch.int64)
    off = workloads.csr_offsets(L)
    Qf = workloads.normalized_tokens((32, d), seed=d + 1, dtype="fp32")
    Df = workloads.normalized_tokens((int(off[-1]), d), seed=d + 2, dtype="fp32")
    Qi, sq = workloads.quantize_int8(Qf)
    Di, sd = workloads.quantize_int8(Df)
    offn = off.numpy()
    for b in np.nonzero(L.numpy() >= 2)[0][::3]:
        s0, e0 = int(offn[b]), int(offn[b + 1])
        Di[s0:e0] = Di[s0]
        sd[s0:e0] = sd[s0]
    _check(Qi, sq, Di, sd, off)


def test_extreme_values_exact():
    """All +-127 inputs: dots reach 127^2 * d; every partial sum must stay exact."""
    d = 1024
    rng = np.random.default_rng(5)
    Q = torch.tensor(rng.choice([-127, 127], size=(8, d)), dtype=torch.int8)
    D = torch.tensor(rng.choice([-127, 127], size=(40, d)), dtype=torch.int8)
    D[7] = Q[3]                                   # dot = 127^2 * 1024 = 16516096 < 2^24
    sq = torch.full((8,), 1e-3)
    sd = torch.linspace(0.5, 2.0, 40)
    _check(Q, sq, D, sd, torch.tensor([0, 13, 40]))


def test_i8_many_docs_sampled():
    """B=500000 documents: 500 sampled documents checked bit-exactly."""
    Qi, sq, Di, sd, off = _inputs(500_000, 32, 128, seed=211)
    out, mv, md, am = m.maxsim_score_i8(Qi.to(DEV), sq.to(DEV), Di.to(DEV), sd.to(DEV), off.to(DEV),
                                        want_details=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    idx = np.sort(np.random.default_rng(9).choice(500_000, 500, replace=False))
    offn = off.numpy()
    for b in idx:
        o2 = np.array([0, offn[b + 1] - offn[b]])
        ref, rmv, rmd, ram = oracle.maxsim_i8(Qi.numpy(), sq.numpy(), Di.numpy()[offn[b]:offn[b + 1]],
                                              sd.numpy()[offn[b]:offn[b + 1]], o2)
        assert (md[b].cpu().numpy() == rmd[0]).all() and (am[b].cpu().numpy() == ram[0]).all()
        assert (mv[b].cpu().numpy() == rmv[0]).all()


def test_bad_offsets_are_reported_not_faulted():
    """Offsets beyond the packed rows: the kernel's own checks score those
    documents as empty and set the bad-input bit."""
    Qi, sq, Di, sd, _ = _inputs(4, 32, 128, seed=221)
    off = torch.tensor([0, 5, 3, 10_000_000, int(Di.shape[0])], dtype=torch.int64)
    out, mv, md, am = m.maxsim_score_i8(Qi.to(DEV), sq.to(DEV), Di.to(DEV), sd.to(DEV), off.to(DEV),
                                        want_details=True)
    st, flags = m.maxsim_device_status()
    assert st == 1 and flags & m.DEVERR_BAD_INPUT
    assert out[1].item() == 0.0 and (am[1] == -1).all() and out[2].item() == 0.0


# ---------------------------------------------------------------------------
# Scores only (no per-token outputs requested): the tcgen05 kernel with the
# documents on the MMA's M dimension (nq <= 64, d in {64, 128, 192}). Its
# per-token maxima are the same exact fp32 values; only the order of the
# q_scale-weighted sum differs, so the score is held to the same bound.

def _check_scores(Qi, sq, Di, sd, off):
    out = m.maxsim_score_i8(Qi.to(DEV), sq.to(DEV), Di.to(DEV), sd.to(DEV), off.to(DEV))
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    ref, rmv, _, _ = oracle.maxsim_i8(Qi.numpy(), sq.numpy(), Di.numpy(), sd.numpy(), off.numpy())
    bound = 1e-5 * np.maximum(np.abs(sq.numpy()[None, :].astype(np.float64) * rmv).sum(axis=1), 1e-30)
    err = np.abs(out.cpu().numpy() - ref)
    assert (err <= bound).all(), (err.max(), np.argmax(err - bound))
    return out


def test_scores_only_config_shaped():
    _check_scores(*_inputs(3000, 32, 128, seed=301, empty=(3, 2999)))


@pytest.mark.parametrize("nq,d", [(1, 64), (20, 128), (32, 192), (45, 128), (64, 64), (33, 192)])
def test_scores_only_shapes(nq, d):
    _check_scores(*_inputs(400, nq, d, seed=3 * nq + d, lo=1, hi=300, empty=(0, 7)))


@pytest.mark.parametrize("d", [64, 128, 192])
def test_scores_only_tile_boundaries(d):
    """Runs of 0-3-token documents, documents of 31-33, 127-129 and 255-257
    tokens at shifting row alignments (so documents share, fill and straddle
    128-row tiles), and documents whose rows are all equal (every similarity
    ties)."""
    rng = np.random.default_rng(d + 17)
    L = []
    for _ in range(6):
        L += list(rng.integers(0, 4, size=150))
        L += [31, 32, 33, 127, 128, 129, 255, 256, 257, 1, 0, 2, 5]
    L = torch.tensor(L, dtype=torch.int64)
    off = workloads.csr_offsets(L)
    Qf = workloads.normalized_tokens((32, d), seed=d + 3, dtype="fp32")
    Df = workloads.normalized_tokens((int(off[-1]), d), seed=d + 4, dtype="fp32")
    Qi, sq = workloads.quantize_int8(Qf)
    Di, sd = workloads.quantize_int8(Df)
    offn = off.numpy()
    for b in np.nonzero(L.numpy() >= 2)[0][::3]:
        s0, e0 = int(offn[b]), int(offn[b + 1])
        Di[s0:e0] = Di[s0]
        sd[s0:e0] = sd[s0]
    _check_scores(Qi, sq, Di, sd, off)


def test_scores_only_extreme_values():
    """All +-127 inputs at d=192: dots reach 127^2 * 192 < 2^22 and stay exact."""
    d = 192
    rng = np.random.default_rng(15)
    Q = torch.tensor(rng.choice([-127, 127], size=(32, d)), dtype=torch.int8)
    D = torch.tensor(rng.choice([-127, 127], size=(300, d)), dtype=torch.int8)
    D[7] = Q[3]
    D[200] = -Q[5]
    sq = torch.full((32,), 1e-3)
    sd = torch.linspace(0.5, 2.0, 300)
    _check_scores(Q, sq, D, sd, torch.tensor([0, 13, 140, 141, 300]))


def test_scores_only_match_detailed_call():
    """The scores-only call and the call with per-token outputs (another
    kernel) agree to the score bound on the same inputs."""
    Qi, sq, Di, sd, off = _inputs(5000, 32, 128, seed=311, empty=(10,))
    args = (Qi.to(DEV), sq.to(DEV), Di.to(DEV), sd.to(DEV), off.to(DEV))
    fast = m.maxsim_score_i8(*args)
    full, mv, _, _ = m.maxsim_score_i8(*args, want_details=True)
    torch.cuda.synchronize()
    bound = 1e-5 * (sq.to(DEV)[None, :] * mv).abs().sum(dim=1).clamp_min(1e-30)
    assert ((fast - full).abs() <= bound).all()


def test_scores_only_many_docs_sampled():
    """B=500000 documents in the benchmark's shape: 500 sampled scores
    against the oracle."""
    Qi, sq, Di, sd, off = _inputs(500_000, 32, 128, seed=321)
    out = m.maxsim_score_i8(Qi.to(DEV), sq.to(DEV), Di.to(DEV), sd.to(DEV), off.to(DEV))
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    idx = np.sort(np.random.default_rng(19).choice(500_000, 500, replace=False))
    offn = off.numpy()
    for b in idx:
        o2 = np.array([0, offn[b + 1] - offn[b]])
        ref, rmv, _, _ = oracle.maxsim_i8(Qi.numpy(), sq.numpy(), Di.numpy()[offn[b]:offn[b + 1]],
                                          sd.numpy()[offn[b]:offn[b + 1]], o2)
        bound = 1e-5 * max(float(np.abs(sq.numpy().astype(np.float64) * rmv[0]).sum()), 1e-30)
        assert abs(float(out[b]) - ref[0]) <= bound


def test_scores_only_bad_offsets_are_reported():
    Qi, sq, Di, sd, _ = _inputs(4, 32, 128, seed=331)
    off = torch.tensor([0, 5, 3, 10_000_000, int(Di.shape[0])], dtype=torch.int64)
    out = m.maxsim_score_i8(Qi.to(DEV), sq.to(DEV), Di.to(DEV), sd.to(DEV), off.to(DEV))
    st, flags = m.maxsim_device_status()
    assert st == 1 and flags & m.DEVERR_BAD_INPUT
    assert out[1].item() == 0.0 and out[2].item() == 0.0 and out[3].item() == 0.0
