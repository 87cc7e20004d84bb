"""Plain fp64 CPU oracle for late-interaction MaxSim scoring.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library and
its Python binding never import, link or call it, and it shares no code with
them: the C part (``maxsim_oracle.c``) is compiled by gcc as a separate
shared object, and the numpy parts below are written straight from the
definitions.

Operator (TileMaxSim deep reading, §1; FLASH-MAXSIM, Abstract):
    score(Q, D_b) = sum_i max_{j in doc b} <q_i, d_j>

Every function takes numpy arrays and returns numpy arrays in fp64 (or the
integer types the definition fixes). Low-precision inputs (bf16, fp16) are
passed already up-converted to fp64, which is exact.

Pins: each function here is checked in ``tests/test_oracle.py`` against
hand-computed golden cases, brute-force Python loops, numpy library routines
on special cases, invariants (token permutation, padding, scale), or finite
differences. No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "maxsim_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_maxsim_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int, ctypes.c_int64
            lib.oracle_num_threads.restype = i32
            lib.oracle_set_num_threads.argtypes = [i32]
            lib.oracle_maxsim.argtypes = [P, i32, i32, i32, P, P, P, i64, P, P, P]
            lib.oracle_pq_table.argtypes = [P, i32, i32, P, i32, i32, P]
            lib.oracle_maxsim_pq.argtypes = [P, i32, i32, i32, P, P, i64, P, P]
            lib.oracle_maxsim_i8.argtypes = [P, P, i32, i32, P, P, P, i64, P, P, P, P]
            lib.oracle_backward.argtypes = [P, i32, i32, i32, P, P, i64, P, P, P, P]
            _lib = lib
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _ranges_padded(B, nd, doc_len):
    start = np.arange(B, dtype=np.int64) * nd
    if doc_len is None:
        length = np.full(B, nd, dtype=np.int64)
    else:
        length = np.asarray(doc_len, dtype=np.int64)
        assert length.shape == (B,) and (length >= 0).all() and (length <= nd).all()
    return start, length


def _ranges_csr(offsets):
    offsets = np.asarray(offsets, dtype=np.int64)
    assert offsets.ndim == 1 and offsets[0] == 0 and (np.diff(offsets) >= 0).all()
    return offsets[:-1].copy(), np.diff(offsets)


def _maxsim_ranges(Q, Drows, start, length, want_gap):
    Q = _c(Q, np.float64)
    if Q.ndim == 2:
        Q = Q[None]
    nQ, nq, d = Q.shape
    Drows = _c(Drows, np.float64).reshape(-1, d)
    assert np.isfinite(Q).all() and np.isfinite(Drows).all(), "oracle takes finite inputs"
    B = start.shape[0]
    if B:
        assert (start + length <= Drows.shape[0]).all()
    out = np.zeros((nQ, B), np.float64)
    arg = np.zeros((nQ, B, nq), np.int32)
    gap = np.zeros((nQ, B, nq), np.float64) if want_gap else None
    _load().oracle_maxsim(_p(Q), nQ, nq, d, _p(Drows), _p(_c(start, np.int64)),
                          _p(_c(length, np.int64)), B, _p(out), _p(arg), _p(gap))
    return out, arg, gap


def maxsim(Q, D, doc_len=None, want_gap=False):
    """Padded layout. Q [nq,d] or [nQ,nq,d]; D [B,Nd,d]; doc_len [B] or None.

    Returns (score [nQ,B], argmax [nQ,B,nq] int32, gap or None) in fp64.
    Tokens j >= doc_len[b] take no part in the maximum.
    """
    D = np.asarray(D)
    B, nd, d = D.shape
    start, length = _ranges_padded(B, nd, doc_len)
    return _maxsim_ranges(Q, D.reshape(B * nd, d), start, length, want_gap)


def maxsim_varlen(Q, D_packed, offsets, want_gap=False):
    """CSR layout: doc b owns packed rows offsets[b] .. offsets[b+1]-1."""
    start, length = _ranges_csr(offsets)
    return _maxsim_ranges(Q, D_packed, start, length, want_gap)


def pq_table(Q, C):
    """T[i,m,k] = q_i[subspace m] . C[m,k]  (TileMaxSim §2(3)); fp64."""
    Q = _c(Q, np.float64)
    C = _c(C, np.float64)
    nq, d = Q.shape
    M, K, ds = C.shape
    assert ds * M == d
    T = np.zeros((nq, M, K), np.float64)
    _load().oracle_pq_table(_p(Q), nq, d, _p(C), M, K, _p(T))
    return T


def maxsim_pq(T, codes, offsets):
    """Table-lookup PQ scoring: returns (score [B], argmax [B,nq])."""
    T = _c(T, np.float64)
    nq, M, K = T.shape
    codes = _c(codes, np.uint8).reshape(-1, M)
    offsets = _c(offsets, np.int64)
    B = offsets.shape[0] - 1
    out = np.zeros(B, np.float64)
    arg = np.zeros((B, nq), np.int32)
    _load().oracle_maxsim_pq(_p(T), nq, M, K, _p(codes), _p(offsets), B, _p(out), _p(arg))
    return out, arg


def pq_decode(C, codes):
    """Decoded vectors: row j = concat_m C[m, codes[j,m], :] (a plain gather)."""
    C = np.asarray(C, np.float64)
    M, K, ds = C.shape
    codes = np.asarray(codes).reshape(-1, M).astype(np.int64)
    return np.concatenate([C[m][codes[:, m]] for m in range(M)], axis=1)


def maxsim_i8(Qi8, s_q, Di8, s_d, offsets):
    """INT8 x INT8 scoring. Returns (score fp64 [B], maxv fp32 [B,nq],
    maxdot int32 [B,nq], argmax int32 [B,nq])."""
    Qi8 = _c(Qi8, np.int8)
    nq, d = Qi8.shape
    Di8 = _c(Di8, np.int8).reshape(-1, d)
    s_q = _c(s_q, np.float32)
    s_d = _c(s_d, np.float32)
    offsets = _c(offsets, np.int64)
    B = offsets.shape[0] - 1
    out = np.zeros(B, np.float64)
    maxv = np.zeros((B, nq), np.float32)
    maxdot = np.zeros((B, nq), np.int32)
    arg = np.zeros((B, nq), np.int32)
    _load().oracle_maxsim_i8(_p(Qi8), _p(s_q), nq, d, _p(Di8), _p(s_d), _p(offsets), B,
                             _p(out), _p(maxv), _p(maxdot), _p(arg))
    return out, maxv, maxdot, arg


def _backward_ranges(Q, Drows, start, argmax, dS):
    Q = _c(Q, np.float64)
    if Q.ndim == 2:
        Q = Q[None]
    nQ, nq, d = Q.shape
    Drows = _c(Drows, np.float64).reshape(-1, d)
    B = start.shape[0]
    argmax = _c(argmax, np.int32).reshape(nQ, B, nq)
    dS = _c(dS, np.float64).reshape(nQ, B)
    dQ = np.zeros((nQ, nq, d), np.float64)
    dD = np.zeros_like(Drows)
    _load().oracle_backward(_p(Q), nQ, nq, d, _p(Drows), _p(_c(start, np.int64)), B,
                            _p(argmax), _p(dS), _p(dQ), _p(dD))
    return dQ, dD


def backward(Q, D, argmax, dS, doc_len=None):
    """Gradients of sum_{q,b} dS[q,b]*score[q,b] through the given argmax.

    Padded layout: returns (dQ [nQ,nq,d], dD [B,Nd,d]) in fp64.
    """
    D = np.asarray(D)
    B, nd, d = D.shape
    start, _ = _ranges_padded(B, nd, doc_len)
    dQ, dD = _backward_ranges(Q, D.reshape(B * nd, d), start, argmax, dS)
    return dQ, dD.reshape(B, nd, d)


def backward_varlen(Q, D_packed, offsets, argmax, dS):
    start, _ = _ranges_csr(offsets)
    return _backward_ranges(Q, D_packed, start, argmax, dS)
