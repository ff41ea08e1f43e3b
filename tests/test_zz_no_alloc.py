"""The allocation-free decode entry point, called through the C ABI.

fa_decode_splitkv_noalloc exists for callers that may not allocate device
memory during a call; its partial states live in a fixed device array of the
library.  It must give the same outputs as fa_decode_splitkv (the allocating
entry point) within the tests' bf16 tolerance, on consecutive calls that reuse
the array with different shapes, and it must refuse work that does not fit.
This file is collected last so a failure here leaves every other test run.
"""
import ctypes

import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import make_qkv
from parity import TOL, bf16_half_step

pytestmark = pytest.mark.gpu


def _c_fn():
    fn = fa.lib().fa_decode_splitkv_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    fn.restype = i
    return fn


def _noalloc(q, k, v, o, splits):
    B, H, Nk, d = k.shape
    return _c_fn()(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, Nk, d, splits,
                   torch.cuda.current_stream().cuda_stream)


def _assert_close(got, ref):
    g, r = got.float().cpu().double(), ref.float().cpu().double()
    err = (g - r).abs()
    beyond = (err.numpy() - bf16_half_step(r.numpy())).max()
    assert beyond <= TOL["bf16"]["max_o"]
    assert err.mean().item() <= TOL["bf16"]["mean_o"]


def test_noalloc_matches_allocating_entry_on_consecutive_calls(cuda_device):
    cases = [((4, 8, 4096, 64), 16, 31), ((2, 4, 3001, 128), 7, 32)]
    for (B, H, Nk, d), splits, seed in cases:  # second call reuses the array with another shape
        q, k, v = make_qkv(B, H, 1, Nk, d, "bf16", seed=seed, device=cuda_device)
        ref = fa.fa_decode_splitkv(q, k, v, splits)
        o = torch.full((B, H, d), float("nan"), device=cuda_device, dtype=torch.bfloat16)
        assert _noalloc(q, k, v, o, splits) == fa.FA_OK
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all()
        _assert_close(o, ref)


def test_noalloc_rejects_work_beyond_the_scratch(cuda_device):
    # B*H*splits*(d+2)*4 bytes of states: 64*64*64*130*4 = 136 MB > 8 MiB
    q, k, v = make_qkv(1, 1, 1, 64, 64, "bf16", seed=1, device=cuda_device)
    B, H, Nk, d, splits = 64, 64, 4096, 128, 64
    assert fa.lib().fa_decode_workspace_bytes(B, H, d, splits) > (8 << 20)
    st = _c_fn()(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(), B, H, Nk, d, splits, None)
    assert st == fa.FA_ERR_UNSUPPORTED
