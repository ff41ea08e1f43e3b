"""GPU parity of the causal forward (fa_fwd_ex with causal = 1) against the float64 oracle.

The mask is aligned to the bottom-right corner: query row i sees keys 0 .. i + Nk - Nq (the
pages name causal masking as the next extension, "FlashAttention 简化版：Tiling + Online
Softmax" §7; the alignment is this library's reading).
"""
import math

import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import WORKLOADS, make_qkv, workload_inputs
from parity import check_fwd, sample_rows

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, Nq, Nk
    (1, 2, 200, 200),
    (2, 1, 128, 128),
    (1, 1, 300, 1000),   # queries are the last 300 positions of 1000
    (1, 2, 513, 513),
    (1, 1, 1, 77),       # one query: sees every key
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("kv_splits", [1, 0])
def test_causal_shapes(cuda_device, dtype, d, shape, kv_splits):
    B, H, Nq, Nk = shape
    q, _, _ = make_qkv(B, H, Nq, 1, d, dtype, seed=900 + Nq + d, device=cuda_device)
    _, k, v = make_qkv(B, H, 1, Nk, d, dtype, seed=901 + Nk + d, device=cuda_device)
    sc = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q, k, v, scale=sc, causal=True, kv_splits=kv_splits)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    check_fwd(q, k, v, o, lse, sc, causal=True, name=f"causal {dtype} d{d} {shape} splits={kv_splits}")


@pytest.mark.parametrize("kv_splits", [2, 7])
def test_causal_explicit_splits(cuda_device, kv_splits):
    """Split ranges above the diagonal of some query blocks hold no visible key (empty states)."""
    q, k, v = make_qkv(1, 2, 700, 700, 64, "bf16", seed=41, device=cuda_device)
    o, lse = fa.fa_fwd(q, k, v, causal=True, kv_splits=kv_splits)
    torch.cuda.synchronize()
    check_fwd(q, k, v, o, lse, 1 / 8, causal=True, name=f"causal splits={kv_splits}")


def test_causal_grouped_query_heads(cuda_device):
    q, _, _ = make_qkv(2, 8, 300, 1, 128, "bf16", seed=42, device=cuda_device)
    _, k, v = make_qkv(2, 2, 1, 400, 128, "bf16", seed=43, device=cuda_device)
    sc = 1 / math.sqrt(128)
    o, lse = fa.fa_fwd(q, k, v, scale=sc, causal=True)
    torch.cuda.synchronize()
    check_fwd(q, k, v, o, lse, sc, causal=True, name="causal gqa")


def test_causal_rejects_more_queries_than_keys(cuda_device):
    q, k, v = make_qkv(1, 1, 300, 200, 64, "bf16", seed=44, device=cuda_device)
    with pytest.raises(fa.FAError):
        fa.fa_fwd(q, k, v, causal=True)


@pytest.mark.parametrize("name", ["mh_prefill", "peaked_d128"])
def test_causal_full_size_sampled(cuda_device, name):
    """The full-size bf16 workloads with the causal mask: every head, sampled rows."""
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w, device=cuda_device)
    o, lse = fa.fa_fwd(q, k, v, scale=w.scale, causal=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rows = sample_rows(w.Nq, 32, seed=w.seed + 1)
    check_fwd(q, k, v, o, lse, w.scale, rows=rows, causal=True, name=f"causal {name}")
