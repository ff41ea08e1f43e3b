"""GPU parity of the grouped-query split-KV decode (fa_decode_splitkv_gqa) against the oracle.

Query head h reads key/value head h / (H / Hkv) ("FlashAttention 简化版：Tiling + Online Softmax" §7
names MQA/GQA); the oracle is the plain split-and-merge decode on K/V copied out per query head, in
the same merge order.
"""
import math

import numpy as np
import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import make_qkv, merge_order
from parity import check_decode

pytestmark = pytest.mark.gpu


def _per_query_head(x, group):
    return x.repeat_interleave(group, dim=1).contiguous()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(8, 8), (8, 4), (8, 2), (8, 1), (32, 2), (16, 1)],
                         ids=lambda x: str(x))
@pytest.mark.parametrize("Nk,splits", [(1000, 7), (4096, 16), (64, 1), (1, 1), (130, 3)])
def test_decode_gqa(cuda_device, d, H, Hkv, Nk, splits):
    B = 2
    q, _, _ = make_qkv(B, H, 1, 1, d, "bf16", seed=2100 + H + Hkv + d, device=cuda_device)
    _, k, v = make_qkv(B, Hkv, 1, Nk, d, "bf16", seed=2101 + Nk + splits, device=cuda_device)
    order = merge_order(splits, 2200 + splits)
    sc = 1 / math.sqrt(d)
    o, lse = fa.fa_decode_splitkv_gqa(q, k, v, splits, scale=sc, with_lse=True,
                                      merge_order=torch.as_tensor(order, device=cuda_device))
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    g = H // Hkv
    check_decode(q.reshape(B, H, d), _per_query_head(k, g), _per_query_head(v, g), o, lse, sc, splits, order,
                 name=f"decode gqa d{d} H{H} Hkv{Hkv} Nk{Nk} s{splits}")


def test_decode_gqa_one_wave_configuration(cuda_device):
    """A tensor-core decode grid that only a fourth CTA per SM starts in one wave (one key/value head,
    groups of 32; B from the SM count so that B*splits lies in (3*SMs, 4*SMs]) runs the 4-CTA d=64
    configuration.  One query head of every batch (each reads every CTA of its batch), plus the first
    and last, against the oracle."""
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    splits, H, Hkv, d = 16, 32, 1, 64
    B = (4 * sms) // splits
    assert 3 * sms < B * Hkv * splits <= 4 * sms
    Nk = 2 * 64 * splits  # chunks of two whole key tiles
    q, _, _ = make_qkv(B, H, 1, 1, d, "bf16", seed=2150, device=cuda_device)
    _, k, v = make_qkv(B, Hkv, 1, Nk, d, "bf16", seed=2151, device=cuda_device)
    order = merge_order(splits, 2152)
    sc = 1 / math.sqrt(d)
    o, lse = fa.fa_decode_splitkv_gqa(q, k, v, splits, scale=sc, with_lse=True,
                                      merge_order=torch.as_tensor(order, device=cuda_device))
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    heads = sorted({0, B * H - 1, *[b * H + (7 * b) % H for b in range(B)]})
    check_decode(q.reshape(B, H, d), _per_query_head(k, H), _per_query_head(v, H), o, lse, sc, splits, order,
                 heads=heads, name=f"decode gqa one wave B{B} Nk{Nk}")


def test_decode_gqa_matches_plain_decode_when_groups_are_one(cuda_device):
    """With Hkv = H the grouped kernel computes exactly what the per-head decode computes."""
    q, k, v = make_qkv(2, 4, 1, 777, 64, "bf16", seed=2300, device=cuda_device)
    a, la = fa.fa_decode_splitkv_gqa(q, k, v, 5, with_lse=True)
    b, lb = fa.fa_decode_splitkv_ex(q, k, v, 5, with_lse=True)
    torch.cuda.synchronize()
    assert (a.float() - b.float()).abs().max().item() <= 2 ** -7
    assert (la - lb).abs().max().item() <= 1e-5


def test_decode_gqa_full_size(cuda_device):
    """B=32, H=32 query heads on Hkv=8 key/value heads (groups of 4), Nk=32768, d=64, 16 splits:
    32 sampled query heads against the oracle."""
    B, H, Hkv, Nk, d, splits = 32, 32, 8, 32768, 64, 16
    q, _, _ = make_qkv(B, H, 1, 1, d, "bf16", seed=2400, device=cuda_device)
    _, k, v = make_qkv(B, Hkv, 1, Nk, d, "bf16", seed=2401, device=cuda_device)
    order = merge_order(splits, 2005)
    o, lse = fa.fa_decode_splitkv_gqa(q, k, v, splits, with_lse=True,
                                      merge_order=torch.as_tensor(order, device=cuda_device))
    torch.cuda.synchronize()
    rng = np.random.default_rng(2402)
    heads = sorted({0, B * H - 1, *rng.choice(B * H, 30, replace=False).tolist()})
    g = H // Hkv
    kk = torch.stack([k[h // H, (h % H) // g] for h in heads])[:, None]  # [n, 1, Nk, d]
    vv = torch.stack([v[h // H, (h % H) // g] for h in heads])[:, None]
    qq = q.reshape(B * H, d)[heads][:, None]
    check_decode(qq, kk, vv, o.reshape(B * H, d)[heads][:, None], lse.reshape(B * H)[heads][:, None],
                 1 / math.sqrt(d), splits, order, name="decode gqa full size (sampled heads)")


def test_decode_gqa_tensor_core_path_full_size(cuda_device):
    """Groups of 8 (32 query heads on 4 key/value heads) with chunks of whole key tiles go through the
    forward kernel in split mode: B=32, Nk=32768, d=64, 16 splits, sampled heads against the oracle."""
    B, H, Hkv, Nk, d, splits = 32, 32, 4, 32768, 64, 16
    q, _, _ = make_qkv(B, H, 1, 1, d, "bf16", seed=2500, device=cuda_device)
    _, k, v = make_qkv(B, Hkv, 1, Nk, d, "bf16", seed=2501, device=cuda_device)
    order = merge_order(splits, 2005)
    o, lse = fa.fa_decode_splitkv_gqa(q, k, v, splits, with_lse=True,
                                      merge_order=torch.as_tensor(order, device=cuda_device))
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    rng = np.random.default_rng(2502)
    heads = sorted({0, B * H - 1, *rng.choice(B * H, 30, replace=False).tolist()})
    g = H // Hkv
    kk = torch.stack([k[h // H, (h % H) // g] for h in heads])[:, None]
    vv = torch.stack([v[h // H, (h % H) // g] for h in heads])[:, None]
    qq = q.reshape(B * H, d)[heads][:, None]
    check_decode(qq, kk, vv, o.reshape(B * H, d)[heads][:, None], lse.reshape(B * H)[heads][:, None],
                 1 / math.sqrt(d), splits, order, name="decode gqa groups of 8, tensor-core path (sampled heads)")


@pytest.mark.parametrize("d", [64, 128])
def test_decode_gqa_bad_merge_order_gives_nan(cuda_device, d):
    """A merge order that is not a permutation makes both paths write NaN rather than read out of range."""
    for H, Hkv in ((8, 2), (16, 1)):  # groups of 4 (CUDA cores) and 16 (tensor cores)
        q, _, _ = make_qkv(1, H, 1, 1, d, "bf16", seed=2600, device=cuda_device)
        _, k, v = make_qkv(1, Hkv, 1, 1024, d, "bf16", seed=2601, device=cuda_device)
        bad = torch.tensor([0, 0, 1, 2], dtype=torch.int32, device=cuda_device)
        o, lse = fa.fa_decode_splitkv_gqa(q, k, v, 4, with_lse=True, merge_order=bad)
        torch.cuda.synchronize()
        assert torch.isnan(o.float()).all() and torch.isnan(lse).all()
