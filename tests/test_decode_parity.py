"""GPU parity of the split-KV decode (split kernel + merge kernel) against the float64 oracle.

Page cited: [T3] "CS349E 第 11 讲 01_online_softmax.py", demo 2 (partial states
(m, l, o) merged in any order give the same result).
"""
import math

import numpy as np
import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import WORKLOADS, make_qkv, merge_order, workload_inputs
from parity import check_decode

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Nk, d, splits
    (2, 3, 100, 64, 7),     # ragged last chunk
    (1, 2, 17, 64, 16),     # chunks of 2 keys, the last seven empty
    (2, 2, 1000, 128, 5),
    (1, 1, 1, 64, 1),       # a single key
    (3, 1, 4096, 64, 16),
    (1, 4, 3000, 128, 12),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("ordered", [False, True])
def test_cases(cuda_device, case, ordered):
    B, H, Nk, d, splits = case
    q, k, v = make_qkv(B, H, 1, Nk, d, "bf16", seed=500 + CASES.index(case), device=cuda_device)
    order = merge_order(splits, 7) if ordered else None
    mo = torch.as_tensor(order, device=cuda_device) if ordered else None
    sc = 1 / math.sqrt(d)
    o, lse = fa.fa_decode_splitkv_ex(q, k, v, splits, scale=sc, merge_order=mo, with_lse=True)
    torch.cuda.synchronize()
    check_decode(q, k, v, o, lse, sc, splits, order, name=str(case))


def test_plain_entry_matches_ex(cuda_device):
    q, k, v = make_qkv(2, 2, 1, 777, 64, "bf16", seed=3, device=cuda_device)
    o1 = fa.fa_decode_splitkv(q, k, v, 6)
    o2, _ = fa.fa_decode_splitkv_ex(q, k, v, 6)
    ws = torch.empty(fa.fa_decode_workspace_bytes(2, 2, 64, 6) // 4, device=cuda_device, dtype=torch.float32)
    o3, _ = fa.fa_decode_splitkv_ex(q, k, v, 6, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(o1, o3)
    check_decode(q, k, v, o1, None, 1 / 8, 6, name="plain")


def test_merge_order_invariance(cuda_device):
    """Default and seeded merge orders agree to rounding: LSE within 1e-5, O within one bf16 step."""
    q, k, v = make_qkv(4, 4, 1, 8192, 64, "bf16", seed=11, device=cuda_device)
    o1, l1 = fa.fa_decode_splitkv_ex(q, k, v, 16, with_lse=True)
    mo = torch.as_tensor(merge_order(16, 2005), device=cuda_device)
    o2, l2 = fa.fa_decode_splitkv_ex(q, k, v, 16, merge_order=mo, with_lse=True)
    torch.cuda.synchronize()
    assert (l1 - l2).abs().max().item() <= 1e-5
    step = o1.float().abs().clamp_min(1e-3) * 2.0 ** -7
    assert ((o1.float() - o2.float()).abs() <= step).all()


def test_invalid_order_gives_nan(cuda_device):
    q, k, v = make_qkv(1, 2, 1, 64, 64, "bf16", seed=4, device=cuda_device)
    bad = torch.tensor([0, 1, 1, 3], dtype=torch.int32, device=cuda_device)
    o, lse = fa.fa_decode_splitkv_ex(q, k, v, 4, merge_order=bad, with_lse=True)
    torch.cuda.synchronize()
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()
    oob = torch.tensor([0, 1, 2, 9], dtype=torch.int32, device=cuda_device)
    o, _ = fa.fa_decode_splitkv_ex(q, k, v, 4, merge_order=oob)
    torch.cuda.synchronize()
    assert torch.isnan(o.float()).all()


def test_decode_workload_full_size(cuda_device):
    """B=32 H=32 Nk=32768 d=64, 16 splits, merge order seeded with 2005: 64 seeded heads against the
    oracle (same order), every output finite."""
    w = WORKLOADS["decode"]
    q, k, v = workload_inputs(w, device=cuda_device)
    order = merge_order(w.splits, w.order_seed)
    mo = torch.as_tensor(order, device=cuda_device)
    o, lse = fa.fa_decode_splitkv_ex(q, k, v, w.splits, merge_order=mo, with_lse=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    heads = np.sort(np.random.default_rng(w.seed).choice(w.B * w.H, size=64, replace=False))
    check_decode(q, k, v, o, lse, w.scale, w.splits, order, heads=heads, name=w.name)


def test_merge_stream_order(cuda_device):
    """The merge kernel is launched as a dependent of the split kernel; work enqueued after the call
    sees the merged output complete."""
    q, k, v = make_qkv(8, 16, 1, 16384, 64, "bf16", seed=1700, device=cuda_device)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o, lse = fa.fa_decode_splitkv_ex(q, k, v, 16, with_lse=True)
        early_o, early_lse = o.clone(), lse.clone()
    torch.cuda.synchronize()
    assert torch.equal(o, early_o) and torch.equal(lse, early_lse)
