"""GPU checks of the d = 64 forward's key-split CTAs.

A d = 64 bf16 forward without the mask launches CTAs of 256 query rows, two per SM.  When they do not
fill whole waves and the last wave would leave each of its CTAs alone on an SM, the library gives that
wave's rows to key-split CTAs instead: one 128-row query tile each, whose two tile slots walk the two
halves of the keys and merge their partial states (m, l, unnormalised O) inside the CTA at the end
("CS349E 第 11 讲 01_online_softmax.py", demo 2: partial states over key segments merge exactly).
The shapes below take that path on a 152-SM GB300; each is checked against the oracle on every
head, with rows sampled at every 128-row tile boundary, and against the plain grid (kv_splits = 1).
"""
import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import WORKLOADS, make_qkv, workload_inputs
from parity import check_fwd, sample_rows

pytestmark = pytest.mark.gpu


def _fwd(q, k, v, sc, **kw):
    o, lse = fa.fa_fwd(q, k, v, scale=sc, **kw)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    return o, lse


def key_split_expected(B, H, Nq, Nk, sms):
    """Whether the library's plan gives the last wave to key-split CTAs (two 256-row CTAs per SM)."""
    units = B * H * -(-Nq // 256)
    slots = 2 * sms
    rest = units % slots
    return units >= slots and 0 < rest <= sms and -(-Nk // 64) >= 8


CASES = [
    # B, H, Hkv, Nq, Nk, Q/K multiplier
    (1, 20, 20, 4096, 4096, 1.0),   # 320 CTA units: 16 past the first wave (32 key-split CTAs)
    (2, 10, 10, 4000, 3000, 1.0),   # ragged query tiles; 47 key tiles: halves of 24 and 23
    (1, 20, 4, 4096, 2048, 1.0),    # grouped-query heads
    (2, 5, 5, 9000, 700, 3.0),      # the last wave starts inside a head; 11 key tiles; peaked scores
    (2, 20, 20, 2048, 1024, 10.0),  # 16 key tiles; maxima jump far past the lazy-rescale threshold
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}kv{}q{}k{}x{}".format(*c))
def test_key_split_matches_oracle(cuda_device, case):
    B, H, Hkv, Nq, Nk, mult = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert key_split_expected(B, H, Nq, Nk, sms), "the shape was chosen to take key-split CTAs"
    seed = 5000 + H + Nq + Nk
    q, _, _ = make_qkv(B, H, Nq, 1, 64, "bf16", seed=seed, qk_mult=mult, device=cuda_device)
    _, k, v = make_qkv(B, Hkv, 1, Nk, 64, "bf16", seed=seed + 1, qk_mult=mult, device=cuda_device)
    o, lse = _fwd(q, k, v, 0.125)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rows = sample_rows(Nq, 8, seed=seed + 2)
    check_fwd(q, k, v, o, lse, 0.125, rows=rows, name=f"key split {case}")
    # the plain grid agrees to within the two results' rounding: each is within the bf16 bound of the
    # exact value, so they may be two bf16 steps (2^-6 relative) apart, plus the absolute bound
    o1, lse1 = _fwd(q, k, v, 0.125, kv_splits=1)
    assert torch.allclose(o.float(), o1.float(), rtol=2.0 ** -6, atol=1.5e-2)
    assert (lse - lse1).abs().max().item() <= 1e-3


def test_key_split_every_row(cuda_device):
    """Every output row of the head whose rows the key-split CTAs take (B=1 H=20 N=4096: CTA units
    304 .. 319 are head 19), against the oracle."""
    B, H, N = 1, 20, 4096
    q, k, v = make_qkv(B, H, N, N, 64, "bf16", seed=5300, device=cuda_device)
    o, lse = _fwd(q, k, v, 0.125)
    h = slice(H - 1, H)
    check_fwd(q[:, h], k[:, h], v[:, h], o[:, h], lse[:, h], 0.125, name="key split every row of head 19")


def test_key_split_repeatable(cuda_device):
    """The merge runs in key order inside each CTA: repeated launches are bit-identical."""
    w = WORKLOADS["mh_prefill"]
    q, k, v = workload_inputs(w, device=cuda_device)
    o0, l0 = _fwd(q, k, v, w.scale)
    for _ in range(3):
        o, lse = _fwd(q, k, v, w.scale)
        assert torch.equal(o, o0) and torch.equal(lse, l0)


def test_key_split_without_lse_and_on_a_stream(cuda_device):
    """Key-split CTAs with no LSE output, into a caller's O, on a side stream: the same O as with the
    LSE on the default stream."""
    B, H, N = 1, 20, 4096
    q, k, v = make_qkv(B, H, N, N, 64, "bf16", seed=5400, device=cuda_device)
    o_ref, _ = _fwd(q, k, v, 0.125)
    o = torch.full_like(q, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _, lse = fa.fa_fwd(q, k, v, scale=0.125, o=o, with_lse=False, stream=s)
    s.synchronize()
    assert lse is None
    assert fa.fa_check_device_error() == fa.FA_OK
    assert torch.equal(o, o_ref)
