"""Seeded synthetic inputs for the KDA state path.

This module draws random numbers and shapes them; it holds none of the method's
arithmetic.  The same tensors feed both the CUDA library and the CPU oracle.

Distributions (for every workload): q, k ~ N(0, 1), each (token, head) vector scaled to unit
L2 norm; v ~ N(0, 1); beta = sigmoid(N(0, 1)) per token-head; alpha = sigmoid(N(3, 1)) per
token-head-channel; conv weights ~ N(0, 0.5^2), fp32, [H][3d][4].  Draws are fp32 and then
cast to the workload dtype.  Large workloads are drawn on the GPU in fixed token blocks so
that host memory stays small; the stream of numbers depends only on the seed, the device
and the block size.
"""
from __future__ import annotations

import dataclasses

import torch

BLOCK_TOKENS = 65536


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    H: int
    d: int
    dtype: str            # "f32" | "bf16"
    page_bytes: int
    stride: int = 1
    include_last: bool = False
    hash_block: int = 512
    nseq: int = 1
    T: int = 0            # tokens per sequence (fixed-length workloads)


WORKLOADS = {
    "tiny": Workload("tiny", 0, H=2, d=64, dtype="f32", page_bytes=65536, stride=1,
                     include_last=False, nseq=1, T=1024),
    "batched": Workload("batched", 1, H=16, d=128, dtype="bf16", page_bytes=65536, stride=4,
                        include_last=True, nseq=4, T=8192),
    "varlen_resume": Workload("varlen_resume", 2, H=32, d=128, dtype="bf16", page_bytes=65536,
                              stride=4, include_last=True, nseq=32),
    "decode": Workload("decode", 3, H=32, d=128, dtype="bf16", page_bytes=262144, nseq=256),
    "long": Workload("long", 4, H=32, d=128, dtype="bf16", page_bytes=65536, stride=4,
                     include_last=True, nseq=1, T=1048576),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.square().sum(-1, keepdim=True).sqrt()


def make_tokens(T_tot: int, H: int, d: int, dtype: str, seed: int, device="cpu"):
    """q, k, v, alpha [T_tot, H, d] and beta [T_tot, H] in the workload dtype, plus conv_w."""
    dt = TORCH_DTYPE[dtype]
    g = _gen(seed, device)
    conv_w = (torch.randn(H, 3 * d, 4, generator=g, device=device) * 0.5).contiguous()
    q = torch.empty(T_tot, H, d, dtype=dt, device=device)
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    alpha = torch.empty_like(q)
    beta = torch.empty(T_tot, H, dtype=dt, device=device)
    for t0 in range(0, T_tot, BLOCK_TOKENS):
        n = min(BLOCK_TOKENS, T_tot - t0)
        q[t0:t0 + n] = _unit(torch.randn(n, H, d, generator=g, device=device)).to(dt)
        k[t0:t0 + n] = _unit(torch.randn(n, H, d, generator=g, device=device)).to(dt)
        v[t0:t0 + n] = torch.randn(n, H, d, generator=g, device=device).to(dt)
        beta[t0:t0 + n] = torch.sigmoid(torch.randn(n, H, generator=g, device=device)).to(dt)
        alpha[t0:t0 + n] = torch.sigmoid(torch.randn(n, H, d, generator=g, device=device)
                                         + 3.0).to(dt)
    return {"q": q, "k": k, "v": v, "alpha": alpha, "beta": beta, "conv_w": conv_w}


def varlen_lengths(seed: int = 2, nseq: int = 32, lo: int = 512, hi: int = 32768) -> list[int]:
    """Sequence lengths uniform over the integers [lo, hi]."""
    g = _gen(seed, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (nseq,), generator=g)]


def resume_points(lengths: list[int], seed: int = 2, hash_block: int = 512) -> list[int]:
    """Per sequence, a resume boundary uniform over its stored checkpoints {512 j : j >= 1,
    512 j < L}; 0 (fresh start) when there is none."""
    g = _gen(seed + 1000, "cpu")
    out = []
    for L in lengths:
        n = (L - 1) // hash_block
        if n <= 0:
            out.append(0)
        else:
            out.append(hash_block * (1 + int(torch.randint(0, n, (1,), generator=g))))
    return out


def permuted_page_table(num_pages: int, nreq: int, pages_per_object: int, seed: int = 3):
    """First nreq * pages_per_object entries of a seeded permutation of 0..num_pages-1."""
    g = _gen(seed, "cpu")
    perm = torch.randperm(num_pages, generator=g)
    return perm[: nreq * pages_per_object].to(torch.int32).reshape(nreq, pages_per_object)


def decode_step_tokens(B: int, H: int, d: int, dtype: str, seed: int, step: int, device="cpu"):
    """Fresh q, k, v, alpha [B, H, d] and beta [B, H] for decode step `step`."""
    t = make_tokens(B, H, d, dtype, seed * 100003 + 7919 * (step + 1), device)
    del t["conv_w"]
    return t
