"""GPU: scoring documents held in host memory (maxsim_score_streamed).

Each chunk is scored by the same forward kernels as maxsim_score and every
document's result depends only on that document, so the streamed outputs
must EQUAL device-resident scoring exactly; the device-resident path is
itself checked against the fp64 oracle in test_gpu_forward.py, and one case
here is checked against the oracle directly.
"""
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


@pytest.mark.parametrize("dtype,n_queries,nq,nd,d,B,chunk,lengths", [
    ("bf16", 1, 32, 128, 128, 3000, 700, False),     # ragged last chunk, outputs in place
    ("bf16", 1, 32, 128, 128, 3000, 700, True),
    ("fp16", 3, 40, 96, 64, 1000, 333, True),        # several queries: strided scatter of scores and argmax
    ("fp32", 2, 17, 64, 60, 500, 128, True),         # FFMA path
    ("bf16", 1, 32, 64, 128, 100, 4096, False),      # one chunk larger than B
])
def test_streamed_equals_device_resident(dtype, n_queries, nq, nd, d, B, chunk, lengths):
    Q = workloads.normalized_tokens((n_queries, nq, d), seed=B + nd, dtype=dtype).to(DEV)
    D = workloads.normalized_tokens((B, nd, d), seed=B + nd + 1, dtype=dtype)
    L = workloads.uniform_lengths(B, 0, nd, seed=d) if lengths else None
    if L is not None:
        L[0], L[-1] = 0, nd
    Dh = D.pin_memory()
    Lh = L.pin_memory() if L is not None else None
    out_s, am_s = m.maxsim_score_streamed(Q, Dh, Lh, chunk_docs=chunk, want_argmax=True)
    out_d, am_d = m.maxsim_score(Q, D.to(DEV), None if L is None else L.to(DEV), want_argmax=True)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    assert torch.equal(out_s, out_d)
    assert torch.equal(am_s, am_d)


def test_streamed_against_oracle():
    Q = workloads.normalized_tokens((32, 128), seed=71, dtype="bf16")
    D = workloads.normalized_tokens((900, 128, 128), seed=72, dtype="bf16")
    L = workloads.uniform_lengths(900, 32, 128, seed=73)
    workloads.zero_padding(D, L)
    out = m.maxsim_score_streamed(Q.to(DEV), D.pin_memory(), L.pin_memory(), chunk_docs=256)
    torch.cuda.synchronize()
    ref, _, _ = oracle.maxsim(Q[None].double().numpy(), D.double().numpy(), L.numpy(), want_gap=True)
    P.check_scores(out.cpu().numpy(), ref, P.TOL_LOWP)


def test_streamed_short_workspace_is_rejected():
    Q = workloads.normalized_tokens((32, 128), seed=1, dtype="bf16").to(DEV)
    D = workloads.normalized_tokens((64, 128, 128), seed=2, dtype="bf16").pin_memory()
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    with pytest.raises(m.MaxSimError):
        m.maxsim_score_streamed(Q, D, chunk_docs=32, workspace=ws)


def test_back_to_back_calls_share_one_workspace():
    """Two streamed calls queued back to back on one stream and one workspace,
    with different documents and no synchronisation between them: the second
    call's first copies must wait for the first call's kernels still reading
    the same buffers. Each result equals device-resident scoring exactly."""
    B, nd, d, chunk = 12_000, 128, 128, 4096
    Q = workloads.normalized_tokens((32, d), seed=81, dtype="bf16").to(DEV)
    D1 = workloads.normalized_tokens((B, nd, d), seed=82, dtype="bf16")
    D2 = workloads.normalized_tokens((B, nd, d), seed=83, dtype="bf16")
    L2 = workloads.uniform_lengths(B, 1, nd, seed=84)
    nb = m.maxsim_score_streamed_workspace_size(1, 32, nd, d, torch.bfloat16, chunk)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    h1, h2, hl2 = D1.pin_memory(), D2.pin_memory(), L2.pin_memory()
    ref1 = m.maxsim_score(Q, D1.to(DEV))
    ref2 = m.maxsim_score(Q, D2.to(DEV), L2.to(DEV))
    torch.cuda.synchronize()
    for _ in range(3):
        out1 = m.maxsim_score_streamed(Q, h1, None, chunk_docs=chunk, workspace=ws)
        out2 = m.maxsim_score_streamed(Q, h2, hl2, chunk_docs=chunk, workspace=ws)
        torch.cuda.synchronize()
        assert m.maxsim_device_status() == (0, 0)
        assert torch.equal(out1, ref1)
        assert torch.equal(out2, ref2)
