"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds random-number generation only: no step of attention.  Both
the CUDA path and the float64 oracle are fed the very same bytes made here.

Workloads (the value recipe is normal draws in float32, optionally multiplied,
then rounded to the storage dtype with round-to-nearest-even):
  tiny_fp32       B=1  H=1  Nq=Nk=256    d=64  fp32, N(0,1)
  long_fp32       B=1  H=1  Nq=Nk=4096   d=64  fp32, N(0,1)
  mh_prefill      B=4  H=16 Nq=Nk=4096   d=64  bf16, N(0,1)
  peaked_d128     B=2  H=16 Nq=Nk=8192   d=128 bf16, Q,K ~ 3 N(0,1), V ~ N(0,1)
  decode          B=32 H=32 Nq=1 Nk=32768 d=64 bf16, N(0,1), 16 splits, seeded merge order
The decode merge order is numpy.random.default_rng(seed).permutation(splits).
The output gradient dO of a backward pass is N(0,1), rounded to the storage dtype (make_dout).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str            # "fp32" or "bf16"
    seed: int
    qk_mult: float = 1.0  # Q and K draws are multiplied by this before rounding
    splits: int = 0       # > 0 for split-KV decode
    order_seed: int = -1  # >= 0: seeded merge order for decode
    desc: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 1, 256, 256, 64, "fp32", 1001,
                          desc="tiny single-head attention, fp32"),
    "long_fp32": Workload("long_fp32", 1, 1, 4096, 4096, 64, "fp32", 1002,
                          desc="single-head long sequence, fp32 (TF32 MMA)"),
    "mh_prefill": Workload("mh_prefill", 4, 16, 4096, 4096, 64, "bf16", 1003,
                           desc="multi-head prefill, bf16"),
    "peaked_d128": Workload("peaked_d128", 2, 16, 8192, 8192, 128, "bf16", 1004, qk_mult=3.0,
                            desc="large-head-dim prefill with peaked scores, bf16"),
    "decode": Workload("decode", 32, 32, 1, 32768, 64, "bf16", 1005, splits=16, order_seed=2005,
                       desc="split-KV decode, one query per head, bf16"),
}


def _draw(shape, gen, device, mult: float, dtype) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    return x.to(dtype)  # round-to-nearest-even for bf16


def make_qkv(B: int, H: int, Nq: int, Nk: int, d: int, dtype="bf16", seed: int = 0,
             qk_mult: float = 1.0, v_mult: float = 1.0, device="cpu"):
    """q [B,H,Nq,d], k/v [B,H,Nk,d] contiguous, drawn from one generator seeded with `seed`."""
    tdt = dtype if isinstance(dtype, torch.dtype) else (torch.float32 if dtype == "fp32" else torch.bfloat16)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    q = _draw((B, H, Nq, d), gen, dev, qk_mult, tdt)
    k = _draw((B, H, Nk, d), gen, dev, qk_mult, tdt)
    v = _draw((B, H, Nk, d), gen, dev, v_mult, tdt)
    return q, k, v


def make_dout(B: int, H: int, Nq: int, d: int, dtype="bf16", seed: int = 0, device="cpu") -> torch.Tensor:
    """dO [B,H,Nq,d]: N(0,1) draws from a generator seeded with `seed`, rounded to the dtype."""
    tdt = dtype if isinstance(dtype, torch.dtype) else (torch.float32 if dtype == "fp32" else torch.bfloat16)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    return _draw((B, H, Nq, d), gen, dev, 1.0, tdt)


def workload_inputs(w: Workload, device="cpu"):
    """The q, k, v tensors of a named workload (decode q has Nq=1: [B,H,1,d])."""
    return make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, w.dtype, w.seed, w.qk_mult, device=device)


def merge_order(splits: int, seed: int) -> np.ndarray:
    """Seeded permutation of range(splits) (int32)."""
    return np.random.default_rng(int(seed)).permutation(int(splits)).astype(np.int32)
