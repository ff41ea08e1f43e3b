"""Seeded random sweep of the forward, backward and decode against the float64 oracle.

Each case draws its shape and options from a generator seeded by the case index: batch, query and
key/value heads (grouped or not), ragged query and key lengths, head dim, dtype, causal mask, key
splits, scale and the spread of the scores.  The fixed-shape tests pin known edge cases; this sweep
looks for combinations nobody thought of, with the same tolerances.
"""
import math

import numpy as np
import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import make_dout, make_qkv, merge_order
from parity import TOL_BWD, TOL_BWD_TF32_FWD, check_bwd, check_decode, check_fwd

pytestmark = pytest.mark.gpu


def _fwd_case(i):
    rng = np.random.default_rng(7000 + i)
    d = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["bf16", "fp32"]))
    B = int(rng.integers(1, 3))
    Hkv = int(rng.integers(1, 4))
    H = Hkv * int(rng.choice([1, 2, 4]))
    Nk = int(rng.integers(1, 1500))
    causal = bool(rng.random() < 0.4)
    Nq = int(rng.integers(1, Nk + 1)) if causal else int(rng.integers(1, 1500))
    splits = int(rng.choice([1, 0, 2, 3]))
    scale = float(rng.choice([1 / math.sqrt(d), 0.5 / math.sqrt(d), 1.0 / d]))
    mult = float(rng.choice([1.0, 1.0, 2.0]))
    if dtype == "fp32":  # the fp32 (tf32) bounds are derived for N(0,1) inputs; peaked scores are bf16's
        mult = 1.0
    return B, H, Hkv, Nq, Nk, d, dtype, causal, splits, scale, mult


@pytest.mark.parametrize("i", range(24))
def test_random_forward(cuda_device, i):
    B, H, Hkv, Nq, Nk, d, dtype, causal, splits, scale, mult = _fwd_case(i)
    tiles = (Nk + 127) // 128
    if splits > tiles:  # every split must own a key tile
        splits = 1
    q, _, _ = make_qkv(B, H, Nq, 1, d, dtype, seed=7100 + i, qk_mult=mult, device=cuda_device)
    _, k, v = make_qkv(B, Hkv, 1, Nk, d, dtype, seed=7200 + i, qk_mult=mult, device=cuda_device)
    o, lse = fa.fa_fwd(q, k, v, scale=scale, causal=causal, kv_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    check_fwd(q, k, v, o, lse, scale, causal=causal,
              name=f"random fwd {i}: B{B} H{H}/{Hkv} Nq{Nq} Nk{Nk} d{d} {dtype} causal={causal} splits={splits}")


@pytest.mark.parametrize("i", range(8))
def test_random_backward(cuda_device, i):
    rng = np.random.default_rng(7300 + i)
    d = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["bf16", "fp32"]))
    Hkv = int(rng.integers(1, 3))
    H = Hkv * int(rng.choice([1, 2]))
    Nk = int(rng.integers(1, 700))
    causal = bool(rng.random() < 0.5)
    Nq = int(rng.integers(1, Nk + 1)) if causal else int(rng.integers(1, 700))
    q, _, _ = make_qkv(1, H, Nq, 1, d, dtype, seed=7400 + i, device=cuda_device)
    _, k, v = make_qkv(1, Hkv, 1, Nk, d, dtype, seed=7500 + i, device=cuda_device)
    dout = make_dout(1, H, Nq, d, dtype, seed=7600 + i, device=cuda_device)
    sc = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q, k, v, scale=sc, causal=causal)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, dout, lse, scale=sc, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    # fp32 gradients here follow the library's fp32 forward (tf32 products), so they carry its rounding
    tol = TOL_BWD if dtype == "bf16" else TOL_BWD_TF32_FWD
    check_bwd(q, k, v, dout, dq, dk, dv, sc, causal=causal, tol=tol,
              name=f"random bwd {i}: H{H}/{Hkv} Nq{Nq} Nk{Nk} d{d} {dtype} causal={causal}")


@pytest.mark.parametrize("i", range(12))
def test_random_decode(cuda_device, i):
    rng = np.random.default_rng(7700 + i)
    d = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 4))
    Hkv = int(rng.integers(1, 5))
    group = int(rng.choice([1, 1, 2, 4, 8]))
    H = Hkv * group
    Nk = int(rng.integers(1, 6000))
    splits = int(rng.integers(1, min(Nk, 40) + 1))
    order = merge_order(splits, 7800 + i) if rng.random() < 0.5 else None
    q, _, _ = make_qkv(B, H, 1, 1, d, "bf16", seed=7900 + i, device=cuda_device)
    _, k, v = make_qkv(B, Hkv, 1, Nk, d, "bf16", seed=8000 + i, device=cuda_device)
    mo = torch.as_tensor(order, device=cuda_device) if order is not None else None
    sc = 1 / math.sqrt(d)
    if group == 1:
        o, lse = fa.fa_decode_splitkv_ex(q, k, v, splits, merge_order=mo, with_lse=True)
        kk, vv = k, v
    else:
        o, lse = fa.fa_decode_splitkv_gqa(q, k, v, splits, merge_order=mo, with_lse=True)
        kk, vv = (x.repeat_interleave(group, dim=1) for x in (k, v))  # the head each query head reads
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    check_decode(q, kk, vv, o, lse, sc, splits, order,
                 name=f"random decode {i}: B{B} H{H}/{Hkv} Nk{Nk} d{d} splits={splits} order={order is not None}")
