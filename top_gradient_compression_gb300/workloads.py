"""Seeded synthetic inputs shaped like the SparCML paper's workloads.

This module only draws random numbers. It holds none of the method's
arithmetic (no accumulation, selection, quantisation or reduction), so both
the CUDA path and the CPU oracle can be fed from it without sharing any of
the computation under test.

Workloads (SparCML: High-Performance Sparse Communication for Machine
Learning, §8.2-§8.4 and Appendix B.1 give the shapes they stand in for):

* ``tiny``      P=4,  N=65,536,      grad ~ N(0, 1) fresh per step.
* ``resnet50``  P=8,  N=25,557,032,  grad ~ N(0, sigma_b) with sigma_b
  log-uniform in [1e-4, 1e-1] per 100,000-element layer block (same sigma on
  every node and step); stands in for ResNet-50 layer-wise sparsification.
* ``sweep``     P in {2..64}, N=4,194,304, each node k = floor(d N) distinct
  uniform indices, values N(0, 1) (the uniform model of App. B.1).
* ``asr``       P=16, N=67,108,864, grad ~ Laplace(0, 1e-3) (LSTM/ASR-like).
* ``logreg``    P=32, N=4,194,304, 40,000 distinct indices per node from a
  Zipf(s=1.1) law over feature ranks 1..N (feature = rank - 1), values
  N(0, 1e-2) (naturally sparse logistic-regression gradients, URL task).

Dense gradients are drawn with a torch generator on the requested device so
that full-size inputs can be created directly in device memory; index sets
are drawn with numpy's PCG64 on the host.
"""
from __future__ import annotations

import numpy as np
import torch

BASE_SEED = 1802080

# Sizes of the named workloads.
TINY = dict(P=4, N=65_536, seg_len=65_536, k_num=1, k_den=100, steps=3)
RESNET50 = dict(P=8, N=25_557_032, seg_len=100_000, k_num=1, k_den=1000, steps=10)
SWEEP_N = 4_194_304
SWEEP_P = (2, 4, 8, 16, 32, 64)
SWEEP_D = ((1, 1000), (1, 100), (5, 100), (10, 100))  # 0.1%, 1%, 5%, 10%
ASR = dict(P=16, N=67_108_864, seg_len=67_108_864, k_num=1, k_den=100, steps=3,
           bucket=512, bits=4)
LOGREG = dict(P=32, N=4_194_304, nnz=40_000, zipf_s=1.1, std=1e-2)


def sub_seed(*parts: int) -> int:
    """Derive a 63-bit seed from the base seed and integer labels."""
    ss = np.random.SeedSequence([BASE_SEED] + [int(p) & 0xFFFFFFFF for p in parts])
    return int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1))


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_grad(P: int, N: int, std: float, seed: int, device="cpu") -> torch.Tensor:
    """[P, N] float32, i.i.d. N(0, std^2)."""
    g = _gen(device, seed)
    x = torch.randn((P, N), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def block_sigmas(N: int, block: int, seed: int, lo: float = 1e-4, hi: float = 1e-1) -> np.ndarray:
    """One sigma per block of ``block`` elements (last block shorter), log-uniform in [lo, hi]."""
    nb = (N + block - 1) // block
    rng = np.random.Generator(np.random.PCG64(seed))
    e = rng.uniform(np.log10(lo), np.log10(hi), size=nb)
    return (10.0 ** e).astype(np.float32)


def blocked_normal_grad(P: int, N: int, sigmas: np.ndarray, block: int, seed: int,
                        device="cpu") -> torch.Tensor:
    """[P, N] float32 with element i of every node ~ N(0, sigmas[i // block]^2)."""
    x = normal_grad(P, N, 1.0, seed, device)
    sig = torch.from_numpy(np.repeat(sigmas, block)[:N]).to(device)
    x.mul_(sig)
    return x


def laplace_grad(P: int, N: int, b: float, seed: int, device="cpu") -> torch.Tensor:
    """[P, N] float32 Laplace(0, b): exponential magnitude with a fair random sign."""
    g = _gen(device, seed)
    x = torch.empty((P, N), device=device, dtype=torch.float32)
    x.exponential_(1.0 / b, generator=g)
    s = torch.randint(0, 2, (P, N), generator=g, device=device, dtype=torch.int8)
    x.mul_(s.to(torch.float32).mul_(2.0).sub_(1.0))
    return x


def empty_streams(P: int, cap: int, device="cpu"):
    idx = torch.zeros((P, cap), dtype=torch.int32, device=device)
    val = torch.zeros((P, cap), dtype=torch.float32, device=device)
    nnz = torch.zeros((P,), dtype=torch.int32, device=device)
    return idx, val, nnz


def uniform_streams(P: int, N: int, k: int, seed: int, std: float = 1.0, cap: int | None = None):
    """Each node: k distinct indices drawn uniformly without replacement, sorted,
    values N(0, std^2). Returns host (idx int32 [P, cap], val float32 [P, cap], nnz int32 [P])."""
    cap = k if cap is None else cap
    assert cap >= k
    idx = np.zeros((P, cap), dtype=np.uint32)
    val = np.zeros((P, cap), dtype=np.float32)
    nnz = np.full((P,), k, dtype=np.uint32)
    for p in range(P):
        rng = np.random.Generator(np.random.PCG64(sub_seed(seed, p)))
        sel = np.sort(rng.choice(N, size=k, replace=False)).astype(np.uint32)
        idx[p, :k] = sel
        val[p, :k] = (rng.standard_normal(k) * std).astype(np.float32)
    return idx, val, nnz


def zipf_streams(P: int, N: int, nnz: int, s: float, std: float, seed: int, cap: int | None = None):
    """Each node: the first ``nnz`` distinct features met while drawing feature
    ranks r in 1..N with P(r) proportional to r^-s (feature index = r - 1),
    sorted ascending; values N(0, std^2)."""
    cap = nnz if cap is None else cap
    w = np.arange(1, N + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    idx = np.zeros((P, cap), dtype=np.uint32)
    val = np.zeros((P, cap), dtype=np.float32)
    nn = np.full((P,), nnz, dtype=np.uint32)
    for p in range(P):
        rng = np.random.Generator(np.random.PCG64(sub_seed(seed, p)))
        seen = np.empty(0, dtype=np.int64)
        order = np.empty(0, dtype=np.int64)
        batch = 4 * nnz
        while True:
            u = rng.random(batch)
            r = np.searchsorted(cdf, u, side="right").clip(0, N - 1)
            allr = np.concatenate([order, r]) if order.size else r
            uniq, first = np.unique(allr, return_index=True)
            if uniq.size >= nnz:
                firsts = np.sort(first)[:nnz]
                seen = allr[firsts]
                break
            order = allr
            batch *= 2
        sel = np.sort(seen).astype(np.uint32)
        idx[p, :nnz] = sel
        val[p, :nnz] = (rng.standard_normal(nnz) * std).astype(np.float32)
    return idx, val, nn


def tiny_grads(step: int, device="cpu") -> torch.Tensor:
    c = TINY
    return normal_grad(c["P"], c["N"], 1.0, sub_seed(1, step), device)


def resnet50_sigmas(N: int = RESNET50["N"], block: int = RESNET50["seg_len"]) -> np.ndarray:
    return block_sigmas(N, block, sub_seed(2, 0))


def resnet50_grads(step: int, P: int = RESNET50["P"], N: int = RESNET50["N"],
                   device="cpu") -> torch.Tensor:
    block = RESNET50["seg_len"]
    return blocked_normal_grad(P, N, resnet50_sigmas(N, block), block, sub_seed(2, 1 + step), device)


def asr_grads(step: int, P: int = ASR["P"], N: int = ASR["N"], device="cpu") -> torch.Tensor:
    return laplace_grad(P, N, 1e-3, sub_seed(4, step), device)


def sweep_streams(P: int, d_num: int, d_den: int, N: int = SWEEP_N, cap: int | None = None):
    k = N * d_num // d_den
    return uniform_streams(P, N, k, sub_seed(3, P, d_num, d_den), 1.0, cap)


def logreg_streams(P: int = LOGREG["P"], N: int = LOGREG["N"], nnz: int = LOGREG["nnz"]):
    return zipf_streams(P, N, nnz, LOGREG["zipf_s"], LOGREG["std"], sub_seed(5, P, N, nnz))


def asr_reduce_streams(device, P: int = ASR["P"], N: int = ASR["N"]):
    """The reduce input of the LSTM/ASR-like step, built on `device`: per node
    k = N * k_num / k_den sorted distinct uniform indices (the positions 1%
    Top-k of an i.i.d. gradient keeps are uniform) and Laplace(0, 1e-3)
    values. Returns int32 idx [P, k], float32 val [P, k], int32 nnz [P]."""
    k = N * ASR["k_num"] // ASR["k_den"]
    g = _gen(device, sub_seed(7, P, N, k))
    idx = torch.empty((P, k), dtype=torch.int32, device=device)
    for p in range(P):
        idx[p] = torch.randperm(N, generator=g, device=device)[:k].sort().values.to(torch.int32)
    val = laplace_grad(P, k, 1e-3, sub_seed(8, P, N, k), device)
    nnz = torch.full((P,), k, dtype=torch.int32, device=device)
    return idx, val, nnz


def quant_seed(step: int) -> int:
    """Per-step 64-bit key handed to the stochastic quantiser (the quantiser mixes
    it with the node and the index itself)."""
    return sub_seed(6, step)
