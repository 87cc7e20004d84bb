"""Pins for the fp64 CPU oracle (no GPU needed).

Each oracle function is checked against something other than itself:
hand-derived golden cases (tests/golden/*.json, each citing the page and
section it follows), brute-force Python loops with exactly rounded sums,
numpy library routines on special cases, invariants of the operator, and
finite differences for the backward pass. The cases are chosen so that a
dropped term, a wrong index, a transposed operand, a sign error or a wrong
tie rule fails at least one test.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- golden cases

def test_golden_forward_padded(golden_dir):
    g = _load(golden_dir, "forward_tiny.json")
    for c in g["cases"]:
        s, a, _ = oracle.maxsim(np.array(c["Q"], float), np.array(c["D"], float), c["doc_len"])
        np.testing.assert_array_equal(s, np.array(c["score"], float), err_msg=c["name"])
        np.testing.assert_array_equal(a, np.array(c["argmax"]), err_msg=c["name"])


def test_golden_forward_varlen(golden_dir):
    g = _load(golden_dir, "forward_tiny.json")
    for c in g["varlen_cases"]:
        s, a, _ = oracle.maxsim_varlen(np.array(c["Q"], float), np.array(c["D_packed"], float),
                                       np.array(c["offsets"]))
        np.testing.assert_array_equal(s[0], np.array(c["score"], float), err_msg=c["name"])
        np.testing.assert_array_equal(a[0], np.array(c["argmax"]), err_msg=c["name"])


def test_golden_pq(golden_dir):
    g = _load(golden_dir, "pq_tiny.json")
    T = oracle.pq_table(np.array(g["Q"], float), np.array(g["C"], float))
    np.testing.assert_array_equal(T, np.array(g["T"], float))
    s, a = oracle.maxsim_pq(T, np.array(g["codes"], np.uint8), np.array(g["offsets"]))
    np.testing.assert_array_equal(s, np.array(g["score"], float))
    np.testing.assert_array_equal(a, np.array(g["argmax"]))


def test_golden_i8(golden_dir):
    g = _load(golden_dir, "i8_tiny.json")
    s, mv, md, a = oracle.maxsim_i8(np.array(g["Q"]), np.array(g["s_q"]), np.array(g["D"]),
                                    np.array(g["s_d"]), np.array(g["offsets"]))
    np.testing.assert_array_equal(s, np.array(g["score"]))
    np.testing.assert_array_equal(mv, np.array(g["maxv"], np.float32))
    np.testing.assert_array_equal(md, np.array(g["maxdot"]))
    np.testing.assert_array_equal(a, np.array(g["argmax"]))


def test_golden_backward(golden_dir):
    g = _load(golden_dir, "backward_tiny.json")
    Q, D = np.array(g["Q"], float), np.array(g["D"], float)
    _, a, _ = oracle.maxsim(Q, D)
    np.testing.assert_array_equal(a, np.array(g["argmax"]))
    dQ, dD = oracle.backward(Q, D, a, np.array(g["dS"], float))
    np.testing.assert_array_equal(dQ, np.array(g["dQ"], float))
    np.testing.assert_array_equal(dD, np.array(g["dD"], float))


# ------------------------------------------------------- brute force / library

def _brute_maxsim(Q, docs):
    """Pure-Python loops with exactly rounded dot products (math.fsum)."""
    out, arg = [], []
    for doc in docs:
        sc, ar = [], []
        for qi in Q:
            best, bj = -math.inf, -1
            for j, dj in enumerate(doc):
                s = math.fsum(float(x) * float(y) for x, y in zip(qi, dj))
                if s > best:
                    best, bj = s, j
            sc.append(best if bj >= 0 else 0.0)
            ar.append(bj)
        out.append(math.fsum(sc))
        arg.append(ar)
    return np.array(out), np.array(arg)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_forward_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    nq, nd, d, B = 5, 7, 9, 6
    Q = rng.standard_normal((nq, d))
    D = rng.standard_normal((B, nd, d))
    L = rng.integers(0, nd + 1, B)
    L[0], L[1] = 0, nd
    s, a, _ = oracle.maxsim(Q, D, L)
    bs, ba = _brute_maxsim(Q, [D[b, :L[b]] for b in range(B)])
    np.testing.assert_allclose(s[0], bs, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(a[0], ba)


@pytest.mark.parametrize("d", [16, 64, 128, 768])
def test_forward_matches_numpy_einsum(d):
    """Materialising reference (numpy einsum -> masked max -> sum) on small shapes."""
    Q = workloads.normalized_tokens((3, 8, d), seed=d, dtype="fp32").double().numpy()
    D = workloads.normalized_tokens((10, 33, d), seed=d + 1, dtype="fp32").double().numpy()
    L = workloads.uniform_lengths(10, 1, 33, seed=d + 2).numpy()
    S = np.einsum("qik,bjk->qbij", Q, D)
    mask = np.arange(33)[None, :] >= L[:, None]                 # [b, j]
    S = np.where(mask[None, :, None, :], -np.inf, S)
    ref = S.max(axis=-1).sum(axis=-1)
    s, a, _ = oracle.maxsim(Q, D, L)
    np.testing.assert_allclose(s, ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(a, S.argmax(axis=-1))


def test_dimension_chunked_partial_sums():
    """Chunked partial dot products over 128-wide slices of d, summed before the
    max, give the untiled score (TileMaxSim section 2(2))."""
    d = 384
    Q = workloads.normalized_tokens((6, d), seed=7, dtype="fp32").double().numpy()
    D = workloads.normalized_tokens((5, 20, d), seed=8, dtype="fp32").double().numpy()
    S = sum(np.einsum("ik,bjk->bij", Q[:, c:c + 128], D[:, :, c:c + 128]) for c in range(0, d, 128))
    ref = S.max(axis=-1).sum(axis=-1)
    s, _, _ = oracle.maxsim(Q, D)
    np.testing.assert_allclose(s[0], ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ invariants

@pytest.mark.parametrize("nnz", [4, 16, 64])
def test_identity_document_scores_exactly_nq(nnz):
    """D := Q with exactly unit-norm, pairwise distinct tokens: every query token
    finds itself (sim 1, others < 1), so the score is exactly Nq and argmax is i."""
    for nq in (1, 32, 40):
        Q = workloads.sign_pattern_tokens(nq, 128, nnz, seed=nq + nnz).numpy()
        s, a, gap = oracle.maxsim(Q, Q[None], want_gap=True)
        assert s[0, 0] == float(nq)
        np.testing.assert_array_equal(a[0, 0], np.arange(nq))
        if nq > 1:
            assert (gap[0, 0] > 0).all()


def test_token_permutation_invariance():
    rng = np.random.default_rng(3)
    Q = rng.standard_normal((6, 32))
    D = rng.standard_normal((4, 50, 32))
    s, a, _ = oracle.maxsim(Q, D)
    perm = rng.permutation(50)
    s2, a2, _ = oracle.maxsim(Q, D[:, perm])
    np.testing.assert_allclose(s2, s, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(perm[a2], a)      # argmax follows the tokens


def test_padding_and_csr_neighbours_do_not_contribute():
    rng = np.random.default_rng(4)
    Q = rng.standard_normal((5, 16))
    D = -np.abs(rng.standard_normal((6, 12, 16)))     # mostly negative similarities
    Q = np.abs(Q)
    L = np.array([1, 3, 5, 12, 7, 0])
    s, a, _ = oracle.maxsim(Q, D, L)
    Dbig = D.copy()
    for b in range(6):
        Dbig[b, L[b]:] = 1e3                          # huge values in the padding
    s2, a2, _ = oracle.maxsim(Q, Dbig, L)
    np.testing.assert_array_equal(s2, s)
    np.testing.assert_array_equal(a2, a)
    for b in range(6):                                # equals the truncated document
        sb, _, _ = oracle.maxsim(Q, D[b:b + 1, :max(L[b], 1)], [L[b]])
        assert sb[0, 0] == s[0, b]
    assert s[0, 5] == 0.0 and (a[0, 5] == -1).all()
    # CSR: the same documents packed back to back give the same scores
    packed = np.concatenate([Dbig[b, :L[b]] for b in range(6)])
    off = np.concatenate([[0], np.cumsum(L)])
    s3, a3, _ = oracle.maxsim_varlen(Q, packed, off)
    np.testing.assert_array_equal(s3, s)
    np.testing.assert_array_equal(a3, a)


def test_positive_scaling_and_query_additivity():
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((7, 24))
    D = rng.standard_normal((5, 9, 24))
    s, _, _ = oracle.maxsim(Q, D)
    s4, _, _ = oracle.maxsim(4.0 * Q, D)              # power of two: exact
    np.testing.assert_array_equal(s4, 4.0 * s)
    parts = [oracle.maxsim(Q[i:i + 1], D)[0] for i in range(7)]
    np.testing.assert_allclose(sum(parts), s, rtol=0, atol=1e-12)


def test_gap_is_top1_minus_top2():
    rng = np.random.default_rng(6)
    Q = rng.standard_normal((4, 8))
    D = rng.standard_normal((3, 10, 8))
    D[1, 7] = D[1, 2]                                 # exact duplicate -> ties possible
    _, a, gap = oracle.maxsim(Q, D, want_gap=True)
    S = np.einsum("ik,bjk->bij", Q, D)
    srt = np.sort(S, axis=-1)
    np.testing.assert_allclose(gap[0], srt[..., -1] - srt[..., -2], rtol=0, atol=1e-12)
    assert ((gap[0] == 0) == (srt[..., -1] == srt[..., -2])).all()


# ------------------------------------------------------------------------- PQ

def test_pq_table_matches_brute_force():
    rng = np.random.default_rng(7)
    nq, d, M, K = 3, 16, 4, 5
    Q = rng.standard_normal((nq, d))
    C = rng.standard_normal((M, K, d // M))
    T = oracle.pq_table(Q, C)
    ds = d // M
    for i in range(nq):
        for m in range(M):
            for k in range(K):
                ref = math.fsum(Q[i, m * ds + t] * C[m, k, t] for t in range(ds))
                assert abs(T[i, m, k] - ref) <= 1e-13


def test_pq_lookup_equals_exact_maxsim_on_decoded_vectors():
    """Route (ii) table lookup == route (i) decode to vectors then exact MaxSim."""
    Cg, codes = workloads.pq_inputs(300, 16, 256, 128, seed=9)
    C = Cg.double().numpy()
    codes = codes.numpy()
    Q = workloads.normalized_tokens((32, 128), seed=10, dtype="fp32").double().numpy()
    L = workloads.lognormal_lengths(6, math.log(40), 0.5, 8, 80, seed=11).numpy().astype(np.int64)
    L[-1] = 300 - L[:-1].sum() if L[:-1].sum() < 300 else 0
    off = np.concatenate([[0], np.cumsum(L)])
    codes = codes[:off[-1]]
    T = oracle.pq_table(Q, C)
    s_tab, a_tab = oracle.maxsim_pq(T, codes, off)
    Dhat = oracle.pq_decode(C, codes)
    s_dec, a_dec, _ = oracle.maxsim_varlen(Q, Dhat, off)
    np.testing.assert_allclose(s_tab, s_dec[0], rtol=0, atol=1e-9)
    np.testing.assert_array_equal(a_tab, a_dec[0])


# ----------------------------------------------------------------------- INT8

def test_i8_matches_python_integers_and_fp32_products():
    rng = np.random.default_rng(12)
    nq, d = 4, 40
    Q = rng.integers(-127, 128, (nq, d)).astype(np.int8)
    D = rng.integers(-127, 128, (17, d)).astype(np.int8)
    s_q = rng.uniform(1e-3, 1e-2, nq).astype(np.float32)
    s_d = rng.uniform(1e-3, 1e-2, 17).astype(np.float32)
    off = np.array([0, 5, 5, 17])
    s, mv, md, a = oracle.maxsim_i8(Q, s_q, D, s_d, off)
    for b in range(3):
        rows = range(off[b], off[b + 1])
        score = []
        for i in range(nq):
            if not len(rows):
                assert a[b, i] == -1 and md[b, i] == 0
                continue
            dots = [sum(int(x) * int(y) for x, y in zip(Q[i], D[r])) for r in rows]
            sims = [np.float32(dt) * s_d[r] for dt, r in zip(dots, rows)]   # numpy fp32 RN
            j = int(np.argmax(sims))                                      # first maximum
            assert a[b, i] == j and md[b, i] == dots[j] and mv[b, i] == sims[j]
            score.append(float(s_q[i]) * float(sims[j]))
        assert abs(s[b] - math.fsum(score)) <= 1e-12 * max(1.0, abs(s[b]))


def test_i8_quantiser_round_trip():
    x = workloads.normalized_tokens((50, 128), seed=13, dtype="fp32")
    q, s = workloads.quantize_int8(x)
    assert q.dtype.is_signed and int(q.abs().max()) == 127
    err = (q.float() * s[:, None] - x).abs().max(dim=1).values
    assert (err <= s / 2 * (1 + 1e-6)).all()


# ------------------------------------------------------------------- backward

def test_backward_matches_finite_differences():
    """Central differences of L = sum dS*score (oracle forward only) match the
    argmax-routed analytic gradient where every top-2 gap is >= 1e-3."""
    rng = np.random.default_rng(14)
    nQ, nq, nd, d, B = 2, 3, 4, 5, 3
    for _ in range(50):
        Q = rng.standard_normal((nQ, nq, d))
        D = rng.standard_normal((B, nd, d))
        _, a, gap = oracle.maxsim(Q, D, want_gap=True)
        if gap.min() >= 1e-3:
            break
    dS = rng.standard_normal((nQ, B))
    dQ, dD = oracle.backward(Q, D, a, dS)

    def loss(Qx, Dx):
        return float((oracle.maxsim(Qx, Dx)[0] * dS).sum())

    h = 1e-6
    for arr, grad in ((Q, dQ), (D, dD)):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = loss(Q, D)
            arr[idx] = old - h
            lm = loss(Q, D)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        rel = np.abs(num - grad).max() / np.abs(grad).max()
        assert rel <= 1e-6, rel


def test_backward_varlen_matches_padded():
    rng = np.random.default_rng(15)
    Q = rng.standard_normal((2, 4, 8))
    L = np.array([3, 0, 6, 1])
    D = rng.standard_normal((4, 6, 8))
    _, a, _ = oracle.maxsim(Q, D, L)
    dS = rng.standard_normal((2, 4))
    dQ, dD = oracle.backward(Q, D, a, dS, L)
    packed = np.concatenate([D[b, :L[b]] for b in range(4)])
    off = np.concatenate([[0], np.cumsum(L)])
    _, a2, _ = oracle.maxsim_varlen(Q, packed, off)
    np.testing.assert_array_equal(a2, a)
    dQ2, dD2 = oracle.backward_varlen(Q, packed, off, a2, dS)
    np.testing.assert_allclose(dQ2, dQ, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dD2, np.concatenate([dD[b, :L[b]] for b in range(4)]), rtol=0, atol=1e-12)
    for b in range(4):
        assert (dD[b, L[b]:] == 0).all()


@pytest.mark.parametrize("pattern", ["one_token", "heavy_tail", "even", "uniform"])
def test_skewed_argmax_generator(pattern):
    """The saved-argmax generator used by the backward parity tests: entries
    lie in [0, L_b) and are -1 exactly for empty documents; the patterns
    have their stated shapes."""
    L = np.array([0, 1, 2, 7, 64, 150, 33])
    a = workloads.skewed_argmax(3, len(L), 200, L, pattern, seed=41).numpy()
    assert a.shape == (3, len(L), 200) and a.dtype == np.int32
    for b, l in enumerate(L):
        if l == 0:
            assert (a[:, b] == -1).all()
        else:
            assert ((a[:, b] >= 0) & (a[:, b] < l)).all()
    live = a[:, L > 0]
    if pattern == "one_token":
        assert (live == 0).all()
    if pattern == "even":
        assert (live % 2 == 0).all()
    if pattern == "heavy_tail":   # floor(L u^4): median ~ L/16 (9.4 here), against L/2 for uniform draws
        assert np.median(a[:, 5]) <= 150 / 8


def test_backward_one_token_argmax_closed_form():
    """With every entry routed to token 0, dD[b, 0] = sum_q dS[q,b] sum_i
    Q[q,i], every other row of dD is zero, and dQ[q,i] = sum_b dS[q,b] D[b,0]."""
    rng = np.random.default_rng(43)
    nQ, nq, B, nd, d = 2, 5, 4, 6, 8
    Q = rng.standard_normal((nQ, nq, d))
    D = rng.standard_normal((B, nd, d))
    a = np.zeros((nQ, B, nq), dtype=np.int32)
    dS = rng.standard_normal((nQ, B))
    dQ, dD = oracle.backward(Q, D, a, dS)
    for b in range(B):
        np.testing.assert_allclose(dD[b, 0], sum(dS[q, b] * Q[q].sum(0) for q in range(nQ)), rtol=1e-12, atol=1e-12)
        assert (dD[b, 1:] == 0).all()
    for q in range(nQ):
        for i in range(nq):
            np.testing.assert_allclose(dQ[q, i], sum(dS[q, b] * D[b, 0] for b in range(B)), rtol=1e-12, atol=1e-12)
