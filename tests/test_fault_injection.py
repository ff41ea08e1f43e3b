"""Failure detection without a GPU fault: a bounded device-side wait that runs out.

The host arms a test-only fault that makes the forward kernel's TMA warp skip
its first key-tile copy.  The MMA thread's wait for that tile hits its limit
(about half a second), sets the CTA's abort flag and the library's error word;
every other role sees the flag, drains its own copies and MMAs, and the kernel
returns.  The host then reads FA_ERR_TIMEOUT, and the context stays usable.
"""
import math

import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import make_qkv
from parity import check_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
def test_skipped_copy_times_out_then_recovers(cuda_device, d):
    q, k, v = make_qkv(1, 1, 256, 512, d, "bf16", seed=91, device=cuda_device)  # one CTA
    sc = 1 / math.sqrt(d)
    assert fa.fa_check_device_error() == fa.FA_OK
    assert fa.fa_debug_set_fault(1) == fa.FA_OK
    fa.fa_fwd(q, k, v, scale=sc, kv_splits=1)         # enqueued fine; gives up on the device
    assert fa.fa_check_device_error() == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_error() == fa.FA_OK     # the word was cleared
    o, lse = fa.fa_fwd(q, k, v, scale=sc, kv_splits=1)  # the fault was one-shot
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    check_fwd(q, k, v, o, lse, sc, name=f"after fault d{d}")


@pytest.mark.parametrize("d", [64, 128])
def test_backward_skipped_copy_times_out_then_recovers(cuda_device, d):
    """The dK/dV kernel's load warp skips its key/value copy: both MMA warps' waits for it run out, the
    elementwise warps and the loader see the abort flag, and the host reads FA_ERR_TIMEOUT.  The next
    backward call is correct."""
    from attention_forward_05_gb300.inputs import make_dout
    from parity import check_bwd
    q, k, v = make_qkv(1, 1, 128, 256, d, "bf16", seed=92, device=cuda_device)  # two dK/dV CTAs
    dout = make_dout(1, 1, 128, d, "bf16", seed=93, device=cuda_device)
    sc = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q, k, v, scale=sc)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    assert fa.fa_debug_set_fault(1) == fa.FA_OK
    fa.fa_bwd(q, k, v, o, dout, lse, scale=sc)
    assert fa.fa_check_device_error() == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_error() == fa.FA_OK
    dq, dk, dv = fa.fa_bwd(q, k, v, o, dout, lse, scale=sc)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    check_bwd(q, k, v, dout, dq, dk, dv, sc, name=f"bwd after fault d{d}")
