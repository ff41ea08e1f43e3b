"""The comparison helpers of the GPU parity tests, checked on the CPU.

The GPU-vs-oracle tests are only as strict as these helpers: rounding to bf16
must be round-to-nearest-even, the direct bf16 check must reject an output
that is off by more than the bound, and the fp32 LSE check must hold rows that
see many keys to the plain 1e-3.
"""
import numpy as np
import pytest
import torch

from parity import FEW_KEYS, TOL, bf16_step, check_bf16_output, check_fwd, rne_bf16


def test_rne_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-30, 30, 200000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(rne_bf16(x.astype(np.float64)), want)


def test_rne_bf16_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even neighbour is 1
    assert rne_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: the even neighbour is 1 + 2^-6
    assert rne_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert np.array_equal(bf16_step(np.array([1.0, 3.0, 4.0])), [2.0 ** -7, 2.0 ** -6, 2.0 ** -5])


def test_bf16_check_accepts_rounded_and_rejects_off_outputs():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((4, 64)) * 0.5
    got = rne_bf16(ref + rng.standard_normal(ref.shape) * 1e-4)
    check_bf16_output(got, ref, "rounded")
    bad = got.copy()
    small = np.argmin(np.abs(ref))  # an element below 2 in magnitude, where one step is under the bound
    bad.flat[small] = rne_bf16(np.array([ref.flat[small] + 2 * TOL["bf16"]["max_o"]]))[0]
    with pytest.raises(AssertionError):
        check_bf16_output(bad, ref, "planted")


def test_fp32_lse_bound_is_plain_for_rows_with_many_keys(monkeypatch):
    """A row that sees >= FEW_KEYS keys is held to 1e-3 even though its tf32 score bound is larger."""
    import parity
    B, H, Nq, Nk, d = 1, 1, 4, 64, 64
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn(1, 1, n, d, generator=g) * 4 for n in (Nq, Nk, Nk))
    o, lse = (torch.from_numpy(x) for x in parity.oracle.attention(q, k, v, 0.125))
    o, lse = o.float(), lse.float()
    assert parity.tf32_score_bound(q, k, 0.125).min() > 1e-3  # scores large enough that the widening matters
    check_fwd(q, k, v, o, lse, 0.125, name="exact")
    with pytest.raises(AssertionError):
        check_fwd(q, k, v, o, lse + 2e-3, 0.125, name="lse off by 2e-3")
    # under a causal mask the first rows see fewer than FEW_KEYS keys and get the wider bound
    q2, k2, v2 = q[:, :, :4], k[:, :, :4], v[:, :, :4]
    o2, l2 = (torch.from_numpy(x).float() for x in parity.oracle.attention(q2, k2, v2, 0.125, causal=True))
    check_fwd(q2, k2, v2, o2, l2 + 2e-3, 0.125, causal=True, name="few keys, wider bound")
    assert FEW_KEYS == 16
