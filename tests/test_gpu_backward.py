"""GPU parity: argmax-routed backward (inverse CSR dD, destination-owned dQ).

The backward is defined relative to the saved forward argmax, so each case
runs the GPU forward with argmax, then compares the GPU gradients with the
oracle's gradients for that same argmax. Tolerance (gradients): max |diff|
<= 1e-3 * max |oracle| per tensor; fp32 accumulation typically gives ~1e-6.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
m = pytest.importorskip("maxsim_scoring_02_gb300")
DEV = "cuda"
REL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()


def _np(t):
    return t.detach().cpu().to(torch.float64).numpy()


def _rel(got, ref):
    return np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)


def _run(Q, D, L, dS):
    Qd, Dd = Q.to(DEV), D.to(DEV)
    Ld = None if L is None else L.to(DEV)
    _, am = m.maxsim_score(Qd, Dd, Ld, want_argmax=True)
    dQ, dD = m.maxsim_backward(Qd, Dd, am, dS.to(DEV), doc_len=Ld)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    rQ, rD = oracle.backward(_np(Q if Q.dim() == 3 else Q[None]), _np(D), am.cpu().numpy(), dS.double().numpy(),
                             None if L is None else L.numpy())
    assert _rel(dQ.cpu().numpy().reshape(rQ.shape), rQ) <= REL
    assert _rel(dD.cpu().numpy(), rD) <= REL
    if L is not None:   # rows past each document's length are exactly zero
        for b, l in enumerate(L.tolist()):
            assert (dD[b, l:] == 0).all()
    return dQ, dD


def test_golden_backward_zero_padded_to_d64(golden_dir):
    """The hand-derived case with d padded by zeros to 64: all values are small
    integers or halves, exact in bf16 and fp32, so gradients match exactly."""
    g = json.load(open(os.path.join(golden_dir, "backward_tiny.json")))
    Q = torch.zeros(2, 2, 64, dtype=torch.bfloat16)
    Q[..., :2] = torch.tensor(g["Q"], dtype=torch.bfloat16)
    D = torch.zeros(2, 2, 64, dtype=torch.bfloat16)
    D[..., :2] = torch.tensor(g["D"], dtype=torch.bfloat16)
    _, am = m.maxsim_score(Q.to(DEV), D.to(DEV), want_argmax=True)
    assert am.cpu().tolist() == g["argmax"]
    dQ, dD = m.maxsim_backward(Q.to(DEV), D.to(DEV), am, torch.tensor(g["dS"], device=DEV))
    assert dQ.cpu()[..., :2].tolist() == g["dQ"] and (dQ.cpu()[..., 2:] == 0).all()
    assert dD.cpu()[..., :2].tolist() == g["dD"] and (dD.cpu()[..., 2:] == 0).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128, 192, 256, 512, 1024])
def test_backward_random_padded(dtype, d):
    nQ, nq, B, nd = 3, 40, 60, 150
    Q = workloads.normalized_tokens((nQ, nq, d), seed=d, dtype=dtype)
    D = workloads.normalized_tokens((B, nd, d), seed=d + 1, dtype=dtype)
    L = workloads.uniform_lengths(B, 0, nd, seed=d + 2)
    L[0], L[1] = 0, 1
    dS = workloads.normal((nQ, B), seed=d + 3)
    _run(Q, D, L, dS)


def test_backward_colpali_shaped_small():
    """Lq = Ld = 1024: 4096 argmax entries per document in the inverse CSR."""
    Q = workloads.normalized_tokens((4, 1024, 128), seed=401, dtype="bf16")
    D = workloads.normalized_tokens((20, 1024, 128), seed=402, dtype="bf16")
    dS = workloads.normal((4, 20), seed=403)
    _run(Q, D, None, dS)


def test_backward_colpali_training_size_sampled():
    """ColPali training step: Q[16,1024,128], D[10000,1024,128] bf16, dS ~ N(0,1).
    dD rows of 4 sampled documents and 24 sampled dQ rows against fp64 sums of
    the gathered inputs."""
    nQ, nq, B, nd, d = 16, 1024, 10_000, 1024, 128
    Q = workloads.normalized_tokens((nQ, nq, d), seed=3, dtype="bf16", device=DEV)
    D = workloads.normalized_tokens((B, nd, d), seed=4, dtype="bf16", device=DEV)
    dS = workloads.normal((nQ, B), seed=5, device=DEV)
    _, am = m.maxsim_score(Q, D, want_argmax=True)
    dQ, dD = m.maxsim_backward(Q, D, am, dS)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    Qn = _np(Q)
    for b in (0, 1234, 7777, B - 1):
        rQ, rD = oracle.backward(Qn, _np(D[b:b + 1]), am[:, b:b + 1].cpu().numpy(), _np(dS[:, b:b + 1]))
        assert _rel(dD[b:b + 1].cpu().numpy(), rD) <= REL
    rng = np.random.default_rng(11)
    for q, i in zip(rng.integers(0, nQ, 24), rng.integers(0, nq, 24)):
        a = am[q, :, i].long()                                    # [B]
        rows = D[torch.arange(B, device=DEV), a]                  # gathered inputs (torch indexing)
        ref = (dS[q].double()[:, None] * rows.double()).sum(0).cpu().numpy()
        got = dQ[q, i].cpu().numpy()
        assert np.abs(got - ref).max() <= REL * np.abs(ref).max()


def test_corrupt_argmax_is_reported_and_skipped():
    Q = workloads.normalized_tokens((1, 32, 128), seed=501, dtype="bf16").to(DEV)
    D = workloads.normalized_tokens((4, 64, 128), seed=502, dtype="bf16").to(DEV)
    L = torch.tensor([64, 10, 0, 64], dtype=torch.int32, device=DEV)
    _, am = m.maxsim_score(Q, D, L, want_argmax=True)
    am[0, 1, 3] = 50          # beyond L_1 = 10
    am[0, 3, 0] = -5
    dS = torch.ones(1, 4, device=DEV)
    dQ, dD = m.maxsim_backward(Q, D, am, dS, doc_len=L)
    st, flags = m.maxsim_device_status()
    assert st == 1 and flags & m.DEVERR_BAD_INPUT
    assert (dD[1, 10:] == 0).all() and (dD[2] == 0).all()


def test_backward_split_document_ranges():
    """B >= 2048 splits the dQ sweep into document ranges whose partials are
    added in range order from the workspace; the result must match the oracle."""
    nQ, nq, B, nd, d = 2, 64, 3000, 40, 128
    Q = workloads.normalized_tokens((nQ, nq, d), seed=601, dtype="bf16")
    D = workloads.normalized_tokens((B, nd, d), seed=602, dtype="bf16")
    L = workloads.uniform_lengths(B, 0, nd, seed=603)
    dS = workloads.normal((nQ, B), seed=604)
    assert m.maxsim_backward_workspace_size(nQ, nq, d, B, nd) > 0
    _run(Q, D, L, dS)


def test_backward_halves_equal_full_call():
    """maxsim_backward_dq and maxsim_backward_dd run the same kernels as the
    two halves of maxsim_backward: their outputs are identical to it."""
    nQ, nq, B, nd, d = 2, 48, 2500, 90, 128
    Q = workloads.normalized_tokens((nQ, nq, d), seed=701, dtype="bf16").to(DEV)
    D = workloads.normalized_tokens((B, nd, d), seed=702, dtype="bf16").to(DEV)
    L = workloads.uniform_lengths(B, 0, nd, seed=703).to(DEV)
    dS = workloads.normal((nQ, B), seed=704).to(DEV)
    _, am = m.maxsim_score(Q, D, L, want_argmax=True)
    dQ, dD = m.maxsim_backward(Q, D, am, dS, doc_len=L)
    dQ1 = m.maxsim_backward_dq(D, am, dS, doc_len=L)
    dD1 = m.maxsim_backward_dd(Q, am, dS, nd, doc_len=L)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    assert torch.equal(dQ1, dQ) and torch.equal(dD1, dD)


@pytest.mark.parametrize("pattern", ["one_token", "heavy_tail", "even"])
@pytest.mark.parametrize("d", [64, 128, 512])
def test_dd_skewed_argmax(pattern, d):
    """The inverse-CSR dD with skewed saved argmax: one token taking every
    entry of a document, a heavy-tailed token distribution, and even tokens
    only (odd rows get no entry), over empty, one-token and full-length
    documents. The row ranges of the entry groups are cut by entries + rows,
    so a single row can hold every entry of its document. dD matches the
    oracle's dD for the same argmax, and every row no entry points at is
    exactly zero."""
    nQ, nq, B, nd = 2, 300, 40, 150
    Q = workloads.normalized_tokens((nQ, nq, d), seed=801, dtype="bf16")
    L = workloads.uniform_lengths(B, 0, nd, seed=802)
    L[0], L[1], L[2] = 0, 1, nd
    am = workloads.skewed_argmax(nQ, B, nq, L, pattern, seed=803)
    dS = workloads.normal((nQ, B), seed=804)
    dD = m.maxsim_backward_dd(Q.to(DEV), am.to(DEV), dS.to(DEV), nd, doc_len=L.to(DEV))
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    _, rD = oracle.backward(_np(Q), np.zeros((B, nd, d)), am.numpy(), dS.double().numpy(), L.numpy())
    got = dD.cpu().numpy()
    assert _rel(got, rD) <= REL
    hit = np.zeros((B, nd), dtype=bool)
    a = am.numpy()
    for b in range(B):
        v = a[:, b].ravel()
        hit[b, v[v >= 0]] = True
    assert (got[~hit] == 0).all()
    assert hit[~(np.arange(nd)[None, :] < L.numpy()[:, None])].sum() == 0


def _allreduce_worker(rank, world, port, part, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = torch.from_numpy(part)
    m.allreduce_dq(t)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, t.numpy()))


def test_document_sharded_backward_sums_to_full_gradient():
    """Data-parallel sharding of the training step (TileMaxSim deep reading
    §5): each shard runs maxsim_backward on its own documents, with its slice
    of the forward argmax and of dS. The shards' dQ partials, summed as
    allreduce_dq sums them (here through a two-rank gloo group on host
    copies), equal the oracle's dQ over the whole batch, and every shard's
    dD equals the oracle's dD rows of its documents. The shards are uneven,
    so one runs the range-split dQ sweep (B >= 2048) and one does not."""
    import socket
    import torch.multiprocessing as mp
    nQ, nq, nd, d = 3, 40, 70, 128
    cuts = [0, 1900, 4200]
    B = cuts[-1]
    Q = workloads.normalized_tokens((nQ, nq, d), seed=801, dtype="bf16")
    D = workloads.normalized_tokens((B, nd, d), seed=802, dtype="bf16")
    L = workloads.uniform_lengths(B, 0, nd, seed=803)
    dS = workloads.normal((nQ, B), seed=804)
    Qd, Dd, Ld, dSd = Q.to(DEV), D.to(DEV), L.to(DEV), dS.to(DEV)
    _, am = m.maxsim_score(Qd, Dd, Ld, want_argmax=True)
    parts, dDs = [], []
    for b0, b1 in zip(cuts[:-1], cuts[1:]):
        dQp, dDp = m.maxsim_backward(Qd, Dd[b0:b1], am[:, b0:b1].contiguous(), dSd[:, b0:b1].contiguous(),
                                     doc_len=Ld[b0:b1])
        parts.append(dQp.cpu().numpy().astype(np.float64))
        dDs.append(dDp)
    torch.cuda.synchronize()
    assert m.maxsim_device_status() == (0, 0)
    rQ, rD = oracle.backward(_np(Q), _np(D), am.cpu().numpy(), dS.double().numpy(), L.numpy())
    assert _rel(parts[0] + parts[1], rQ) <= REL
    for (b0, b1), dDp in zip(zip(cuts[:-1], cuts[1:]), dDs):
        assert _rel(dDp.cpu().numpy(), rD[b0:b1]) <= REL
    # the same sum through the library's all-reduce on a two-rank gloo group
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    qu = ctx.Queue()
    procs = [ctx.Process(target=_allreduce_worker, args=(r, 2, port, parts[r], qu)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(qu.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        np.testing.assert_array_equal(res[r], parts[0] + parts[1])
        assert _rel(res[r], rQ) <= REL
