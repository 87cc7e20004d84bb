"""Seeded synthetic inputs shaped like the MaxSim workloads on the source pages.

This module holds input generation only: random draws, L2 normalisation of
the drawn tokens, length draws, CSR offset layout and the per-token INT8
quantisation that produces the library's INT8 inputs. It contains none of
the scoring arithmetic, and it is the one module both the oracle-side tests
and the CUDA-side tests/benchmark take their inputs from.

Shapes follow the pages' workloads (ColBERTv2-style d=128, Nq=32, Nd up to
512; ColPali-style Lq=Ld=1024) because the pages' datasets (MS MARCO, BEIR)
and model weights are not available; Gaussian tokens, L2-normalised, stand in
for the encoder's normalised embeddings.

All generation goes through ``torch.Generator`` seeded explicitly, on the
device asked for (CPU for oracle-sized cases, CUDA for benchmark-sized ones).
"""
from __future__ import annotations

import math

import torch

_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32,
       torch.bfloat16: torch.bfloat16, torch.float16: torch.float16,
       torch.float32: torch.float32}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normalized_tokens(shape, seed: int, dtype="bf16", device="cpu", chunk_rows=1 << 22):
    """i.i.d. N(0,1) entries, each token (last axis) scaled to unit L2 norm,
    then cast to ``dtype``. Drawn and normalised in fp32, in row chunks so
    that benchmark-sized tensors never need an fp32 copy of the whole array."""
    dtype = _DT[dtype]
    shape = tuple(int(s) for s in shape)
    d = shape[-1]
    rows = math.prod(shape[:-1]) if len(shape) > 1 else 1
    out = torch.empty((rows, d), dtype=dtype, device=device)
    g = _gen(seed, device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0, d), generator=g, device=device, dtype=torch.float32)
        x = x / x.norm(dim=1, keepdim=True).clamp_min(1e-30)
        out[r0:r1] = x.to(dtype)
    return out.reshape(shape)


def uniform_lengths(B: int, lo: int, hi: int, seed: int, device="cpu"):
    """Document lengths uniform on the integers lo..hi (inclusive), int32."""
    g = _gen(seed, device)
    return torch.randint(lo, hi + 1, (int(B),), generator=g, device=device, dtype=torch.int64).to(torch.int32)


def lognormal_lengths(B: int, mu: float, sigma: float, lo: int, hi: int, seed: int, device="cpu"):
    """round(exp(N(mu, sigma^2))) clipped to [lo, hi], int32."""
    g = _gen(seed, device)
    z = torch.randn((int(B),), generator=g, device=device, dtype=torch.float64)
    L = torch.exp(mu + sigma * z).round().clamp(lo, hi)
    return L.to(torch.int32)


def csr_offsets(lengths):
    """offsets[0] = 0, offsets[b+1] = offsets[b] + lengths[b]; int64."""
    lengths = lengths.to(torch.int64)
    off = torch.zeros(lengths.numel() + 1, dtype=torch.int64, device=lengths.device)
    off[1:] = torch.cumsum(lengths, 0)
    return off


def zero_padding(D, lengths):
    """Zero the rows j >= lengths[b] of a padded [B, Nd, d] tensor in place."""
    B, nd, _ = D.shape
    j = torch.arange(nd, device=D.device)[None, :]
    mask = j >= lengths.to(D.device).to(torch.int64)[:, None]
    D[mask] = 0
    return D


def quantize_int8(x):
    """Per-token symmetric INT8: s = max|x| / 127 (fp32), x_q = round-half-even(x / s)
    clamped to [-127, 127]. Returns (int8 tensor, fp32 scales over the leading axes)."""
    xf = x.to(torch.float32)
    s = xf.abs().amax(dim=-1) / 127.0
    s = torch.where(s > 0, s, torch.ones_like(s))
    q = torch.round(xf / s[..., None]).clamp(-127, 127).to(torch.int8)
    return q, s.contiguous()


def pq_inputs(n_tokens: int, M: int, K: int, d: int, seed: int, device="cpu"):
    """Codebooks C[M, K, d/M] ~ N(0,1) fp32 and codes[n_tokens, M] uniform uint8."""
    g = _gen(seed, device)
    C = torch.randn((M, K, d // M), generator=g, device=device, dtype=torch.float32)
    codes = torch.randint(0, K, (int(n_tokens), M), generator=g, device=device,
                          dtype=torch.int64).to(torch.uint8)
    return C, codes


def normal(shape, seed: int, device="cpu", dtype=torch.float32):
    """Plain i.i.d. N(0,1) draws (e.g. the upstream gradient dS)."""
    g = _gen(seed, device)
    return torch.randn(tuple(int(s) for s in shape), generator=g, device=device, dtype=dtype)


def sign_pattern_tokens(n: int, d: int, nnz: int, seed: int):
    """n distinct tokens with exactly ``nnz`` nonzero entries of value
    +-1/sqrt(nnz) (nnz a power of 4, so the value is a power of two and the
    token is exactly unit-norm in bf16/fp16/fp32). Two distinct tokens have
    dot product < 1, so a document equal to the query scores exactly n."""
    assert nnz in (4, 16, 64) and nnz <= d
    v = 1.0 / math.sqrt(nnz)
    g = _gen(seed, "cpu")
    seen = set()
    rows = []
    while len(rows) < n:
        idx = torch.randperm(d, generator=g)[:nnz]
        sgn = torch.randint(0, 2, (nnz,), generator=g) * 2 - 1
        key = tuple(sorted(zip(idx.tolist(), sgn.tolist())))
        if key in seen:
            continue
        seen.add(key)
        r = torch.zeros(d, dtype=torch.float64)
        r[idx] = sgn.to(torch.float64) * v
        rows.append(r)
    return torch.stack(rows)


def skewed_argmax(n_queries: int, B: int, nq: int, lengths, pattern: str, seed: int):
    """Argmax index tensors [n_queries, B, nq] (int32) with chosen token
    distributions, as saved-forward inputs for the backward: every entry lies
    in [0, L_b) for L_b > 0, and is -1 for empty documents.

    pattern: "one_token" (every entry is token 0), "heavy_tail" (token
    floor(L u^4), u ~ U[0,1): a few tokens take most entries), "even" (even
    tokens only), "uniform"."""
    g = _gen(seed, "cpu")
    L = torch.as_tensor(lengths, dtype=torch.int64).view(1, B, 1)
    u = torch.rand((n_queries, B, nq), generator=g, dtype=torch.float64)
    Lf = L.to(torch.float64)
    if pattern == "one_token":
        a = torch.zeros((n_queries, B, nq), dtype=torch.int64)
    elif pattern == "heavy_tail":
        a = torch.floor(Lf * u ** 4).to(torch.int64)
    elif pattern == "even":
        a = 2 * torch.floor(torch.floor((Lf + 1) / 2) * u).to(torch.int64)
    elif pattern == "uniform":
        a = torch.floor(Lf * u).to(torch.int64)
    else:
        raise ValueError(pattern)
    a = torch.minimum(a, (L - 1).clamp(min=0))
    a = torch.where(L > 0, a, torch.full_like(a, -1))
    return a.to(torch.int32)
