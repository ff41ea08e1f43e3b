"""Long contexts: K/V tensors of more than 2^31 elements (index arithmetic that must not wrap in 32
bits), a million keys in one head and key loops of thousands of tiles, checked against the oracle on
sampled rows/heads."""
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


# 17 heads x 2^21 keys x d=64: 2^31 + 2^27 elements in each of K and V (4.6 GB in bf16); the last
# head starts at element 2^31, so every address it reads is past the range of a 32-bit index.
BIG_H, BIG_NK, BIG_D = 17, 1 << 21, 64


@pytest.fixture(scope="module")
def big_kv(cuda_device):
    _, k, v = make_qkv(1, BIG_H, 1, BIG_NK, BIG_D, "bf16", seed=4031, device=cuda_device)
    assert k.numel() > 2**31 and (BIG_H - 1) * BIG_NK * BIG_D == 2**31
    yield k, v
    del k, v
    torch.cuda.empty_cache()


def test_forward_past_2_31_elements(cuda_device, big_kv):
    """128 queries per head over the 2^21 keys, with one key split (17 CTAs walk 32768 key tiles
    each) and with the automatic split; the last head is checked."""
    k, v = big_kv
    Nq, h = 128, BIG_H - 1
    q, _, _ = make_qkv(1, BIG_H, Nq, 1, BIG_D, "bf16", seed=4030, device=cuda_device)
    rows = sample_rows(Nq, 4, 4032)
    for splits in (1, 0):
        o, lse = fa.fa_fwd(q, k, v, kv_splits=splits)
        torch.cuda.synchronize()
        assert fa.fa_check_device_error() == fa.FA_OK
        check_fwd(q[:, h:], k[:, h:], v[:, h:], o[:, h:], lse[:, h:], 1 / 8, rows=rows,
                  name=f"fwd K/V past 2^31 elements, head {h}, splits={splits}")


def test_decode_past_2_31_elements(cuda_device, big_kv):
    """Split-KV decode (64 chunks, seeded merge order) over the same K/V; heads 0 and 16 checked."""
    k, v = big_kv
    splits = 64
    q, _, _ = make_qkv(1, BIG_H, 1, 1, BIG_D, "bf16", seed=4033, device=cuda_device)
    order = merge_order(splits, 4034)
    o, lse = fa.fa_decode_splitkv_ex(q, k, v, splits, with_lse=True,
                                     merge_order=torch.as_tensor(order, device=cuda_device))
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    check_decode(q.reshape(1, BIG_H, BIG_D), k, v, o, lse, 1 / 8, splits, order, heads=[0, BIG_H - 1],
                 name="decode K/V past 2^31 elements")


@pytest.mark.parametrize("group", [2, 4])
def test_gqa_decode_past_2_31_elements(cuda_device, big_kv, group):
    """Grouped-query decode over the same K/V (groups of 2 run on the CUDA cores, groups of 4 on the
    tensor cores); the query heads that read the last key/value head are checked."""
    k, v = big_kv
    splits, H = 64, BIG_H * group
    q, _, _ = make_qkv(1, H, 1, 1, BIG_D, "bf16", seed=4035 + group, device=cuda_device)
    o, lse = fa.fa_decode_splitkv_gqa(q, k, v, splits, with_lse=True)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    hs = slice(H - group, H)  # the query heads of key/value head BIG_H - 1
    kk, vv = (x[:, BIG_H - 1:].expand(1, group, BIG_NK, BIG_D) for x in (k, v))
    check_decode(q[:, hs], kk, vv, o[:, hs], lse[:, hs], 1 / 8, splits, None,
                 name=f"GQA decode (group {group}) K/V past 2^31 elements")


def test_backward_past_2_31_elements(cuda_device, big_kv):
    """Backward with 16 queries per head over the same K/V: the dK/dV kernel writes gradient rows past
    element 2^31 and the dQ kernel walks 32768 key tiles; the last head is checked."""
    k, v = big_kv
    Nq, h, sc = 16, BIG_H - 1, 1 / 8
    q, _, _ = make_qkv(1, BIG_H, Nq, 1, BIG_D, "bf16", seed=4040, device=cuda_device)
    dout = make_dout(1, BIG_H, Nq, BIG_D, "bf16", seed=4041, device=cuda_device)
    o, lse = fa.fa_fwd(q, k, v, scale=sc)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, dout, lse, scale=sc)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    check_bwd(q[:, h:], k[:, h:], v[:, h:], dout[:, h:], dq[:, h:], dk[:, h:], dv[:, h:], sc,
              name=f"bwd K/V past 2^31 elements, head {h}")
