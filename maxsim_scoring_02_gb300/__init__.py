"""Late-interaction MaxSim scoring on NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI of ``libmaxsim.so`` (``include/maxsim.h``).
Every function here only checks and marshals arguments: it takes torch
tensors that already live on the GPU, passes their device pointers and the
current CUDA stream to the library, and allocates outputs with torch when the
caller did not pass them. Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and importing
this package fails loudly if the library has not been built.

Operator (TileMaxSim deep reading §1; FLASH-MAXSIM, Abstract):
    score(Q, D_b) = sum_i max_{j < L_b} <q_i, d_j>
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MaxSimError", "library_path", "load_library", "maxsim_score", "maxsim_score_varlen", "maxsim_length_order",
    "maxsim_score_ordered", "maxsim_length_order_workspace_size",
    "maxsim_score_streamed", "maxsim_score_streamed_workspace_size",
    "maxsim_score_pq", "maxsim_score_pq_workspace_size", "maxsim_score_i8", "maxsim_backward",
    "maxsim_backward_workspace_size", "maxsim_backward_dq", "maxsim_backward_dd", "maxsim_device_status",
    "maxsim_version", "allreduce_dq",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libmaxsim.so"

BF16, FP16, FP32 = 0, 1, 2
_DTYPE_CODE = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}

STATUS_NAMES = {0: "MAXSIM_OK", 1: "MAXSIM_ERR_INVALID_ARG", 2: "MAXSIM_ERR_UNSUPPORTED",
                3: "MAXSIM_ERR_CUDA", 4: "MAXSIM_ERR_TIMEOUT", 5: "MAXSIM_ERR_WORKSPACE"}
DEVERR_TIMEOUT = 0x1
DEVERR_BAD_INPUT = 0x2
DEBUG_STALL_FWD_LOADER = 0x1

# Every symbol the header declares (checked by the tests).
EXPORTS = (
    "maxsim_version", "maxsim_status_string", "maxsim_device_status", "maxsim_debug_set_faults",
    "maxsim_score",
    "maxsim_score_varlen", "maxsim_length_order_workspace_size", "maxsim_length_order", "maxsim_score_ordered",
    "maxsim_score_streamed_workspace_size", "maxsim_score_streamed",
    "maxsim_score_pq_workspace_size", "maxsim_score_pq", "maxsim_score_pq_noalloc",
    "maxsim_score_i8",
    "maxsim_backward_workspace_size", "maxsim_backward", "maxsim_backward_dq", "maxsim_backward_dd",
)


class MaxSimError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


_lib = None


def load_library():
    """Load libmaxsim.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build the CUDA library first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.maxsim_version.restype = I32
    lib.maxsim_status_string.restype = ctypes.c_char_p
    lib.maxsim_status_string.argtypes = [I32]
    lib.maxsim_device_status.restype = I32
    lib.maxsim_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
    lib.maxsim_debug_set_faults.restype = I32
    lib.maxsim_debug_set_faults.argtypes = [ctypes.c_uint, ctypes.c_uint64]
    lib.maxsim_score.restype = I32
    lib.maxsim_score.argtypes = [P, I32, I32, I32, P, I64, I32, P, I32, P, P, P]
    lib.maxsim_length_order_workspace_size.restype = SZ
    lib.maxsim_length_order_workspace_size.argtypes = [I64, I32, I32]
    lib.maxsim_length_order.restype = I32
    lib.maxsim_length_order.argtypes = [P, P, I64, I32, P, P, SZ, P]
    lib.maxsim_score_ordered.restype = I32
    lib.maxsim_score_ordered.argtypes = [P, I32, I32, I32, P, I64, I32, P, P, I32, P, P, P]
    lib.maxsim_score_varlen.restype = I32
    lib.maxsim_score_varlen.argtypes = [P, I32, I32, I32, P, P, I64, I64, I32, P, P, P]
    lib.maxsim_score_streamed_workspace_size.restype = SZ
    lib.maxsim_score_streamed_workspace_size.argtypes = [I32, I32, I32, I32, I32, I64]
    lib.maxsim_score_streamed.restype = I32
    lib.maxsim_score_streamed.argtypes = [P, I32, I32, I32, P, I64, I32, P, I32, P, P, P, SZ, I64, P]
    lib.maxsim_score_pq_workspace_size.restype = SZ
    lib.maxsim_score_pq_workspace_size.argtypes = [I32, I32, I32]
    lib.maxsim_score_pq.restype = I32
    lib.maxsim_score_pq.argtypes = [P, I32, I32, P, I32, I32, P, P, I64, I64, P, P, P, SZ, P]
    lib.maxsim_score_pq_noalloc.restype = I32
    lib.maxsim_score_pq_noalloc.argtypes = [P, I32, I32, P, I32, I32, P, P, I64, I64, P, P, P]
    lib.maxsim_score_i8.restype = I32
    lib.maxsim_score_i8.argtypes = [P, P, I32, I32, P, P, P, I64, I64, P, P, P, P, P]
    lib.maxsim_backward_workspace_size.restype = SZ
    lib.maxsim_backward_workspace_size.argtypes = [I32, I32, I32, I64, I32]
    lib.maxsim_backward.restype = I32
    lib.maxsim_backward.argtypes = [P, I32, I32, I32, P, I64, I32, P, I32, P, P, P, P, P, SZ, P]
    lib.maxsim_backward_dq.restype = I32
    lib.maxsim_backward_dq.argtypes = [I32, I32, I32, P, I64, I32, P, I32, P, P, P, P, SZ, P]
    lib.maxsim_backward_dd.restype = I32
    lib.maxsim_backward_dd.argtypes = [P, I32, I32, I32, I64, I32, P, I32, P, P, P, P]
    _lib = lib
    return lib


# ----------------------------------------------------------------- helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, name, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _check(status, what):
    if status != 0:
        raise MaxSimError(status, what)


def maxsim_version() -> int:
    return load_library().maxsim_version()


def maxsim_device_status(stream=None):
    """Synchronise ``stream`` and return (status, flags) of the device status word."""
    flags = ctypes.c_uint(0)
    st = load_library().maxsim_device_status(_stream(stream), ctypes.byref(flags))
    return st, flags.value


# ------------------------------------------------------------- entry points

def maxsim_score(Q, D, doc_len=None, out=None, argmax_out=None, want_argmax=False, stream=None):
    """Padded layout. Q [nq,d] or [n_queries,nq,d]; D [B,Nd,d] (bf16/fp16/fp32);
    doc_len [B] int32 or None. Returns out [n_queries,B] fp32 (and argmax
    [n_queries,B,nq] int32 when requested)."""
    lib = load_library()
    _dev(Q, "Q")
    _dev(D, "D", Q.dtype)
    Q3 = Q if Q.dim() == 3 else Q.unsqueeze(0)
    nQ, nq, d = Q3.shape
    B, nd, d2 = D.shape
    if d2 != d:
        raise ValueError("Q and D disagree on d")
    if doc_len is not None:
        _dev(doc_len, "doc_len", torch.int32)
    if out is None:
        out = torch.empty((nQ, B), dtype=torch.float32, device=Q.device)
    _dev(out, "out", torch.float32)
    if want_argmax and argmax_out is None:
        argmax_out = torch.empty((nQ, B, nq), dtype=torch.int32, device=Q.device)
    if argmax_out is not None:
        _dev(argmax_out, "argmax_out", torch.int32)
    st = lib.maxsim_score(_ptr(Q3), nQ, nq, d, _ptr(D), B, nd, _ptr(doc_len), _DTYPE_CODE[Q.dtype],
                          _ptr(out), _ptr(argmax_out), _stream(stream))
    _check(st, "maxsim_score")
    return (out, argmax_out) if argmax_out is not None else out


def maxsim_length_order_workspace_size(B, nd, csr=False):
    """Device bytes of the workspace of maxsim_length_order (no GPU needed)."""
    return int(load_library().maxsim_length_order_workspace_size(B, nd, 1 if csr else 0))


def maxsim_length_order(doc_len=None, offsets=None, B=None, nd=None, order=None, stream=None):
    """Length-bucketed document order: int32 [B] permutation sorting documents
    by ceil(L_b / 8), ascending and stable. Give doc_len [B] int32 with nd
    (padded layout) or offsets [B+1] int64 (CSR)."""
    lib = load_library()
    if (doc_len is None) == (offsets is None):
        raise ValueError("give exactly one of doc_len and offsets")
    ref = doc_len if doc_len is not None else offsets
    if doc_len is not None:
        _dev(doc_len, "doc_len", torch.int32)
        B = doc_len.numel()
        if nd is None:
            raise ValueError("nd is required with doc_len")
    else:
        _dev(offsets, "offsets", torch.int64)
        B = offsets.numel() - 1
        nd = 0
    if order is None:
        order = torch.empty(B, dtype=torch.int32, device=ref.device)
    _dev(order, "order", torch.int32)
    nb = lib.maxsim_length_order_workspace_size(B, nd, 0 if doc_len is not None else 1)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=ref.device)
    st = lib.maxsim_length_order(_ptr(doc_len), _ptr(offsets), B, nd, _ptr(order), _ptr(ws), ws.numel(),
                                 _stream(stream))
    _check(st, "maxsim_length_order")
    return order


def maxsim_score_ordered(Q, D, doc_order, doc_len=None, out=None, argmax_out=None, want_argmax=False, stream=None):
    """maxsim_score with the documents walked in doc_order (int32 [B]
    permutation); results land at the documents' own indices."""
    lib = load_library()
    _dev(Q, "Q")
    _dev(D, "D", Q.dtype)
    _dev(doc_order, "doc_order", torch.int32)
    Q3 = Q if Q.dim() == 3 else Q.unsqueeze(0)
    nQ, nq, d = Q3.shape
    B, nd, d2 = D.shape
    if d2 != d or doc_order.numel() != B:
        raise ValueError("Q, D and doc_order disagree")
    if doc_len is not None:
        _dev(doc_len, "doc_len", torch.int32)
    if out is None:
        out = torch.empty((nQ, B), dtype=torch.float32, device=Q.device)
    _dev(out, "out", torch.float32)
    if want_argmax and argmax_out is None:
        argmax_out = torch.empty((nQ, B, nq), dtype=torch.int32, device=Q.device)
    if argmax_out is not None:
        _dev(argmax_out, "argmax_out", torch.int32)
    st = lib.maxsim_score_ordered(_ptr(Q3), nQ, nq, d, _ptr(D), B, nd, _ptr(doc_len), _ptr(doc_order),
                                  _DTYPE_CODE[Q.dtype], _ptr(out), _ptr(argmax_out), _stream(stream))
    _check(st, "maxsim_score_ordered")
    return (out, argmax_out) if argmax_out is not None else out


def maxsim_score_streamed_workspace_size(n_queries, nq, nd, d, dtype, chunk_docs):
    """Device bytes of the workspace of maxsim_score_streamed (no GPU needed)."""
    return load_library().maxsim_score_streamed_workspace_size(n_queries, nq, nd, d, _DTYPE_CODE[dtype], chunk_docs)


def maxsim_score_streamed(Q, D_host, doc_len_host=None, chunk_docs=16384, out=None, argmax_out=None,
                          want_argmax=False, workspace=None, stream=None):
    """Padded layout with the documents in HOST memory: D_host [B,Nd,d] and
    doc_len_host [B] int32 (or None) are CPU tensors (page-locked, e.g.
    ``pin_memory()``, for copies that overlap scoring); Q is on the GPU.
    Chunks of ``chunk_docs`` documents are copied and scored in turn. Returns
    out [n_queries,B] fp32 (and argmax [n_queries,B,nq] int32 when requested).
    The host tensors must stay alive until the stream has completed."""
    lib = load_library()
    _dev(Q, "Q")
    if not isinstance(D_host, torch.Tensor) or D_host.is_cuda or not D_host.is_contiguous() or D_host.dtype != Q.dtype:
        raise ValueError("D_host must be a contiguous CPU tensor of Q's dtype")
    Q3 = Q if Q.dim() == 3 else Q.unsqueeze(0)
    nQ, nq, d = Q3.shape
    B, nd, d2 = D_host.shape
    if d2 != d:
        raise ValueError("Q and D_host disagree on d")
    if doc_len_host is not None and (doc_len_host.is_cuda or doc_len_host.dtype != torch.int32
                                     or not doc_len_host.is_contiguous()):
        raise ValueError("doc_len_host must be a contiguous CPU int32 tensor")
    if out is None:
        out = torch.empty((nQ, B), dtype=torch.float32, device=Q.device)
    _dev(out, "out", torch.float32)
    if want_argmax and argmax_out is None:
        argmax_out = torch.empty((nQ, B, nq), dtype=torch.int32, device=Q.device)
    if argmax_out is not None:
        _dev(argmax_out, "argmax_out", torch.int32)
    nbytes = lib.maxsim_score_streamed_workspace_size(nQ, nq, nd, d, _DTYPE_CODE[Q.dtype], chunk_docs)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=Q.device)
    _dev(workspace, "workspace", torch.uint8)
    st = lib.maxsim_score_streamed(_ptr(Q3), nQ, nq, d, ctypes.c_void_p(D_host.data_ptr()), B, nd,
                                   None if doc_len_host is None else ctypes.c_void_p(doc_len_host.data_ptr()),
                                   _DTYPE_CODE[Q.dtype], _ptr(out), _ptr(argmax_out), _ptr(workspace),
                                   workspace.numel(), chunk_docs, _stream(stream))
    _check(st, "maxsim_score_streamed")
    return (out, argmax_out) if argmax_out is not None else out


def maxsim_score_varlen(Q, D_packed, offsets, out=None, argmax_out=None, want_argmax=False, stream=None):
    """CSR layout: document b owns rows offsets[b]..offsets[b+1]-1 of D_packed [T,d]."""
    lib = load_library()
    _dev(Q, "Q")
    _dev(D_packed, "D_packed", Q.dtype)
    _dev(offsets, "offsets", torch.int64)
    Q3 = Q if Q.dim() == 3 else Q.unsqueeze(0)
    nQ, nq, d = Q3.shape
    T, d2 = D_packed.shape
    if d2 != d:
        raise ValueError("Q and D_packed disagree on d")
    B = offsets.numel() - 1
    if out is None:
        out = torch.empty((nQ, B), dtype=torch.float32, device=Q.device)
    if want_argmax and argmax_out is None:
        argmax_out = torch.empty((nQ, B, nq), dtype=torch.int32, device=Q.device)
    st = lib.maxsim_score_varlen(_ptr(Q3), nQ, nq, d, _ptr(D_packed), _ptr(offsets), B, T,
                                 _DTYPE_CODE[Q.dtype], _ptr(out), _ptr(argmax_out), _stream(stream))
    _check(st, "maxsim_score_varlen")
    return (out, argmax_out) if argmax_out is not None else out


def maxsim_score_pq_workspace_size(nq: int, M: int, K: int) -> int:
    return int(load_library().maxsim_score_pq_workspace_size(nq, M, K))


def maxsim_score_pq(Q, codebooks, codes, offsets, out=None, argmax_out=None, want_argmax=False,
                    workspace=None, stream=None):
    """PQ scoring: Q [nq,d] fp32, codebooks [M,K,d/M] fp32, codes [T,M] uint8, CSR offsets."""
    lib = load_library()
    _dev(Q, "Q", torch.float32)
    _dev(codebooks, "codebooks", torch.float32)
    _dev(codes, "codes", torch.uint8)
    _dev(offsets, "offsets", torch.int64)
    nq, d = Q.shape
    M, K, _ = codebooks.shape
    T = codes.shape[0]
    B = offsets.numel() - 1
    ws = maxsim_score_pq_workspace_size(nq, M, K)
    if workspace is None:
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=Q.device)
    if out is None:
        out = torch.empty(B, dtype=torch.float32, device=Q.device)
    if want_argmax and argmax_out is None:
        argmax_out = torch.empty((B, nq), dtype=torch.int32, device=Q.device)
    st = lib.maxsim_score_pq(_ptr(Q), nq, d, _ptr(codebooks), M, K, _ptr(codes), _ptr(offsets), B, T,
                             _ptr(out), _ptr(argmax_out), _ptr(workspace), workspace.numel(),
                             _stream(stream))
    _check(st, "maxsim_score_pq")
    return (out, argmax_out) if argmax_out is not None else out


def maxsim_score_pq_noalloc(Q, codebooks, codes, offsets, out=None, argmax_out=None, want_argmax=False,
                            stream=None):
    """PQ scoring with the table kept in the library's fixed device array, for
    callers that cannot allocate device memory themselves (see the header)."""
    lib = load_library()
    _dev(Q, "Q", torch.float32)
    _dev(codebooks, "codebooks", torch.float32)
    _dev(codes, "codes", torch.uint8)
    _dev(offsets, "offsets", torch.int64)
    nq, d = Q.shape
    M, K, _ = codebooks.shape
    T = codes.shape[0]
    B = offsets.numel() - 1
    if out is None:
        out = torch.empty(B, dtype=torch.float32, device=Q.device)
    if want_argmax and argmax_out is None:
        argmax_out = torch.empty((B, nq), dtype=torch.int32, device=Q.device)
    st = lib.maxsim_score_pq_noalloc(_ptr(Q), nq, d, _ptr(codebooks), M, K, _ptr(codes), _ptr(offsets), B, T,
                                     _ptr(out), _ptr(argmax_out), _stream(stream))
    _check(st, "maxsim_score_pq_noalloc")
    return (out, argmax_out) if argmax_out is not None else out


def maxsim_score_i8(Q, q_scale, D, d_scale, offsets, out=None, maxv_out=None, maxdot_out=None,
                    argmax_out=None, want_details=False, stream=None):
    """INT8 x INT8 scoring with per-token fp32 scales; CSR documents."""
    lib = load_library()
    _dev(Q, "Q", torch.int8)
    _dev(q_scale, "q_scale", torch.float32)
    _dev(D, "D", torch.int8)
    _dev(d_scale, "d_scale", torch.float32)
    _dev(offsets, "offsets", torch.int64)
    nq, d = Q.shape
    T = D.shape[0]
    B = offsets.numel() - 1
    if out is None:
        out = torch.empty(B, dtype=torch.float32, device=Q.device)
    if want_details:
        if maxv_out is None:
            maxv_out = torch.empty((B, nq), dtype=torch.float32, device=Q.device)
        if maxdot_out is None:
            maxdot_out = torch.empty((B, nq), dtype=torch.int32, device=Q.device)
        if argmax_out is None:
            argmax_out = torch.empty((B, nq), dtype=torch.int32, device=Q.device)
    st = lib.maxsim_score_i8(_ptr(Q), _ptr(q_scale), nq, d, _ptr(D), _ptr(d_scale), _ptr(offsets), B, T,
                             _ptr(out), _ptr(maxv_out), _ptr(maxdot_out), _ptr(argmax_out), _stream(stream))
    _check(st, "maxsim_score_i8")
    if want_details:
        return out, maxv_out, maxdot_out, argmax_out
    return out


def maxsim_backward_workspace_size(n_queries, nq, d, B, nd) -> int:
    return int(load_library().maxsim_backward_workspace_size(n_queries, nq, d, B, nd))


def maxsim_backward(Q, D, argmax, dS, doc_len=None, dQ=None, dD=None, workspace=None, stream=None):
    """Gradients of sum dS*score through the saved forward argmax (padded layout)."""
    lib = load_library()
    _dev(Q, "Q")
    _dev(D, "D", Q.dtype)
    _dev(argmax, "argmax", torch.int32)
    _dev(dS, "dS", torch.float32)
    Q3 = Q if Q.dim() == 3 else Q.unsqueeze(0)
    nQ, nq, d = Q3.shape
    B, nd, _ = D.shape
    if doc_len is not None:
        _dev(doc_len, "doc_len", torch.int32)
    if dQ is None:
        dQ = torch.empty((nQ, nq, d), dtype=torch.float32, device=Q.device)
    if dD is None:
        dD = torch.empty((B, nd, d), dtype=torch.float32, device=Q.device)
    ws = maxsim_backward_workspace_size(nQ, nq, d, B, nd)
    if workspace is None and ws > 0:
        workspace = torch.empty(ws, dtype=torch.uint8, device=Q.device)
    st = lib.maxsim_backward(_ptr(Q3), nQ, nq, d, _ptr(D), B, nd, _ptr(doc_len), _DTYPE_CODE[Q.dtype],
                             _ptr(argmax), _ptr(dS), _ptr(dQ), _ptr(dD), _ptr(workspace),
                             0 if workspace is None else workspace.numel(), _stream(stream))
    _check(st, "maxsim_backward")
    return dQ.view(Q.shape) if Q.dim() == 2 else dQ, dD


def maxsim_backward_dq(D, argmax, dS, nq=None, doc_len=None, dQ=None, workspace=None, stream=None):
    """dQ only (frozen document side). D [B,Nd,d]; argmax [n_queries,B,nq]
    int32; dS [n_queries,B] fp32. Returns dQ [n_queries,nq,d] fp32."""
    lib = load_library()
    _dev(D, "D")
    _dev(argmax, "argmax", torch.int32)
    _dev(dS, "dS", torch.float32)
    nQ, B2, nq_a = argmax.shape
    B, nd, d = D.shape
    if B2 != B or dS.shape != (nQ, B):
        raise ValueError("argmax / dS shapes do not match D")
    if doc_len is not None:
        _dev(doc_len, "doc_len", torch.int32)
    if dQ is None:
        dQ = torch.empty((nQ, nq_a, d), dtype=torch.float32, device=D.device)
    _dev(dQ, "dQ", torch.float32)
    ws = maxsim_backward_workspace_size(nQ, nq_a, d, B, nd)
    if workspace is None and ws > 0:
        workspace = torch.empty(ws, dtype=torch.uint8, device=D.device)
    st = lib.maxsim_backward_dq(nQ, nq_a, d, _ptr(D), B, nd, _ptr(doc_len), _DTYPE_CODE[D.dtype], _ptr(argmax),
                                _ptr(dS), _ptr(dQ), _ptr(workspace), 0 if workspace is None else workspace.numel(),
                                _stream(stream))
    _check(st, "maxsim_backward_dq")
    return dQ


def maxsim_backward_dd(Q, argmax, dS, nd, doc_len=None, dD=None, stream=None):
    """dD only (frozen query side). Q [nq,d] or [n_queries,nq,d]; argmax
    [n_queries,B,nq] int32; dS [n_queries,B] fp32. Returns dD [B,nd,d] fp32."""
    lib = load_library()
    _dev(Q, "Q")
    _dev(argmax, "argmax", torch.int32)
    _dev(dS, "dS", torch.float32)
    Q3 = Q if Q.dim() == 3 else Q.unsqueeze(0)
    nQ, nq, d = Q3.shape
    B = argmax.shape[1]
    if argmax.shape != (nQ, B, nq) or dS.shape != (nQ, B):
        raise ValueError("argmax / dS shapes do not match Q")
    if doc_len is not None:
        _dev(doc_len, "doc_len", torch.int32)
    if dD is None:
        dD = torch.empty((B, nd, d), dtype=torch.float32, device=Q.device)
    _dev(dD, "dD", torch.float32)
    st = lib.maxsim_backward_dd(_ptr(Q3), nQ, nq, d, B, nd, _ptr(doc_len), _DTYPE_CODE[Q.dtype], _ptr(argmax),
                                _ptr(dS), _ptr(dD), _stream(stream))
    _check(st, "maxsim_backward_dd")
    return dD


# ------------------------------------------------------------ sharded backward

def allreduce_dq(dQ, group=None):
    """Document-sharded training: every rank runs maxsim_backward on its own
    documents, so its dQ holds only those documents' terms of
    dQ[q,i,:] = sum_b dS[q,b] * D[b, argmax[q,b,i], :]; the sum over ranks is
    the full gradient. One in-place all-reduce (sum) over ``group`` (NCCL for
    CUDA tensors, gloo on CPU); dD rows belong to one rank's documents and
    need no exchange (FLASH-MAXSIM, Abstract: destination-owned reduction).
    A no-op without an initialised process group or with one rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return dQ
    dist.all_reduce(dQ, op=dist.ReduceOp.SUM, group=group)
    return dQ
