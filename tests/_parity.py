"""Comparison rules between the CUDA path and the fp64 oracle.

Tolerances (written here once, used by every GPU parity test):
  * bf16 / fp16 inputs: max |score_gpu - score_oracle| <= 2e-4, and the
    top-100 ranking identical (ties by index) except between documents whose
    oracle scores lie within the observed score error of each other;
  * fp32 inputs: max |score diff| <= 1e-5;
  * argmax: bit-exact wherever the oracle's top-2 gap is at least the
    accumulation bound eps_i = 8 * d * 2^-24 * |q_i| * max_j |d_j| (the
    GPU accumulates fp32 in an order the oracle does not); rows under that
    bound may pick either token, and the pick must attain the maximum to
    within eps_i.
"""
import numpy as np

TOL_LOWP = 2e-4
TOL_FP32 = 1e-5


def eps_rows(Q, doc_norm_max, d):
    """Per (query, doc, token) accumulation bound; Q [nQ,nq,d] fp64, doc_norm_max [B]."""
    qn = np.linalg.norm(Q, axis=-1)                      # [nQ, nq]
    return 8.0 * d * 2.0 ** -24 * qn[:, None, :] * np.maximum(doc_norm_max, 1e-30)[None, :, None]


def check_scores(out, ref, tol):
    out = np.asarray(out, np.float64)
    err = np.abs(out - ref)
    assert err.max() <= tol, f"max |score diff| {err.max():.3e} > {tol:.1e}"
    return float(err.max())


def check_argmax(am, ref_am, gap, eps):
    am = np.asarray(am)
    sure = gap >= eps
    bad = (am != ref_am) & sure
    assert not bad.any(), f"{int(bad.sum())} argmax mismatches outside near-ties (of {am.size})"
    return int((~sure).sum())


def check_argmax_attains(am, Q, docs_rows, ref_am, eps):
    """For near-tie rows: the GPU's pick attains the oracle maximum within eps.
    docs_rows(q, b) -> fp64 token matrix of doc b."""
    am = np.asarray(am)
    diff = np.argwhere(am != ref_am)
    for q, b, i in diff:
        rows = docs_rows(b)
        j, jr = int(am[q, b, i]), int(ref_am[q, b, i])
        assert 0 <= j < rows.shape[0], (q, b, i, j)
        sj = float(rows[j] @ Q[q, i])
        sr = float(rows[jr] @ Q[q, i])
        assert sj >= sr - eps[q, b, i], (q, b, i, sj, sr)


def check_topk(out, ref, k=100):
    """Identical top-k ranking (ties by index) up to swaps between documents
    whose oracle scores differ by less than twice the observed score error."""
    out = np.asarray(out, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    k = min(k, out.size)
    tol = 2.0 * np.abs(out - ref).max() + 1e-12
    og = np.lexsort((np.arange(out.size), -out))[:k]
    orf = np.lexsort((np.arange(ref.size), -ref))[:k]
    if np.array_equal(og, orf):
        return 0
    swaps = 0
    for a, b in zip(og, orf):
        if a != b:
            swaps += 1
            assert abs(ref[a] - ref[b]) <= tol, f"top-{k} differs: doc {a} vs {b}, oracle gap {abs(ref[a]-ref[b]):.3e}"
    return swaps
