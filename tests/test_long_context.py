"""Long contexts: index arithmetic past 2^31 elements of a K/V tensor and key loops of thousands of
tiles, checked against the oracle on sampled rows/heads."""
import math

import numpy as np
import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import make_dout, make_qkv, merge_order
from parity import check_bwd, check_decode, check_fwd, sample_rows

pytestmark = pytest.mark.gpu


def test_decode_million_keys(cuda_device):
    """B=1 H=4 Nk=2^20 d=128: each K and V tensor holds 2^29 elements (1 GiB), 64 splits."""
    B, H, Nk, d, splits = 1, 4, 1 << 20, 128, 64
    q, _, _ = make_qkv(B, H, 1, 1, d, "bf16", seed=4000, device=cuda_device)
    _, k, v = make_qkv(B, H, 1, Nk, d, "bf16", seed=4001, device=cuda_device)
    order = merge_order(splits, 4002)
    o, lse = fa.fa_decode_splitkv_ex(q, k, v, splits, with_lse=True,
                                     merge_order=torch.as_tensor(order, device=cuda_device))
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    check_decode(q.reshape(B, H, d), k, v, o, lse, 1 / math.sqrt(d), splits, order, heads=[0, 3],
                 name="decode Nk=2^20")


def test_forward_long_keys_causal(cuda_device):
    """Nq=512 queries at the end of Nk=131072 keys (causal, bottom-right), d=64, one head: CTAs walk
    about 2000 key tiles; the automatic key split runs too."""
    Nq, Nk, d = 512, 131072, 64
    q, _, _ = make_qkv(1, 1, Nq, 1, d, "bf16", seed=4010, device=cuda_device)
    _, k, v = make_qkv(1, 1, 1, Nk, d, "bf16", seed=4011, device=cuda_device)
    for splits in (1, 0):
        o, lse = fa.fa_fwd(q, k, v, causal=True, kv_splits=splits)
        torch.cuda.synchronize()
        assert fa.fa_check_device_error() == fa.FA_OK
        check_fwd(q, k, v, o, lse, 1 / 8, rows=sample_rows(Nq, 8, 4012), causal=True,
                  name=f"fwd Nk=131072 causal splits={splits}")


def test_backward_long_keys(cuda_device):
    """Backward with Nq=256 queries over Nk=32768 keys, d=128: the dQ kernel walks 512 key tiles, the
    dK/dV kernel 256 CTAs of 4 query steps."""
    Nq, Nk, d = 256, 32768, 128
    q, _, _ = make_qkv(1, 1, Nq, 1, d, "bf16", seed=4020, device=cuda_device)
    _, k, v = make_qkv(1, 1, 1, Nk, d, "bf16", seed=4021, device=cuda_device)
    dout = make_dout(1, 1, Nq, d, "bf16", seed=4022, device=cuda_device)
    sc = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q, k, v, scale=sc)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, dout, lse, scale=sc)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    check_bwd(q, k, v, dout, dq, dk, dv, sc, name="bwd Nk=32768")
