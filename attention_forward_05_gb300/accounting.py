"""Closed-form work and byte counts used by the benchmark's roofline figures.

Sources (web pages, cited by title and section):
  [T1] "FlashAttention 简化版：Tiling + Online Softmax" (forceinjection.github.io)
  [T2] "Flash Attention 代码填空 (Level 2-3)" (boots-coder.github.io, LLM-101-CN)
  [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com)
"""
from __future__ import annotations

ESIZE = {"fp32": 4, "bf16": 2}


def fwd_flops(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    """FLOPs of the two contractions S = Q K^T and O = P V: 2 * 2 * B*H*Nq*Nk*d ([T3] demo 3, 4 N^2 d)."""
    return 4 * B * H * Nq * Nk * d


def fwd_flops_causal(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    """FLOPs of the two contractions under a bottom-right causal mask: row i sees i + Nk - Nq + 1 keys."""
    visible = Nq * (Nk - Nq) + Nq * (Nq + 1) // 2
    return 4 * B * H * visible * d


def bwd_flops(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    """FLOPs of the backward's five contractions, S = Q K^T (recomputed), dP = dO V^T, dV = P^T dO,
    dQ = dS K and dK = dS^T Q: 5 * 2 * B*H*Nq*Nk*d (2.5x the forward).  The library recomputes S
    and dP once more for dQ; that extra work is not counted."""
    return 10 * B * H * Nq * Nk * d


def bwd_flops_causal(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    """bwd_flops over the (query, key) pairs a bottom-right causal mask leaves visible."""
    visible = Nq * (Nk - Nq) + Nq * (Nq + 1) // 2
    return 10 * B * H * visible * d


def fwd_min_bytes(B: int, H: int, Nq: int, Nk: int, d: int, dtype: str) -> int:
    """Smallest HBM traffic of one forward: read Q, K, V once, write O and the fp32 LSE."""
    e = ESIZE[dtype]
    return (B * H * Nq * d + 2 * B * H * Nk * d + B * H * Nq * d) * e + 4 * B * H * Nq


def decode_min_bytes(B: int, H: int, Nk: int, d: int, dtype: str = "bf16") -> int:
    """Algorithmic bytes of one split-KV decode: K and V once, q read and o written."""
    e = ESIZE[dtype]
    return 2 * B * H * Nk * d * e + 2 * B * H * d * e


def decode_gqa_min_bytes(B: int, H: int, Hkv: int, Nk: int, d: int, dtype: str = "bf16") -> int:
    """Algorithmic bytes of a grouped-query decode: each key/value head's K and V once, q read, o written."""
    e = ESIZE[dtype]
    return 2 * B * Hkv * Nk * d * e + 2 * B * H * d * e


def decode_workspace_traffic(B: int, H: int, d: int, splits: int) -> int:
    """Bytes of fp32 partial states (m, l, o[d]) written by the split kernel and read by the merge."""
    return 2 * B * H * splits * (d + 2) * 4


def standard_intermediate_bytes(N: int, esize: int = 4) -> int:
    """S and P of standard attention held at once: 2 N^2 elements ([T1] §1.1; [T2] Exercise 1)."""
    return 2 * N * N * esize


def nonmatmul_share(N: int, d: int, Bc: int, deferred: bool, cost_ratio: float = 16.0) -> float:
    """Time of the non-matmul work relative to the matmuls, at `cost_ratio` times the cost per op.

    Model of [T3] demo 3: matmul = 4 N^2 d; softmax work = 4 N^2 (max, subtract,
    exp, sum); per-step renormalisation of O costs 4 ops per element per KV
    block (N/Bc blocks), the deferred form 1 op per element per block plus one
    final division per element.
    """
    tc = N // Bc
    matmul = 4 * N * N * d
    softmax = 4 * N * N
    extra = tc * N * d * 1 + N * d if deferred else tc * N * d * 4
    return cost_ratio * (softmax + extra) / matmul
