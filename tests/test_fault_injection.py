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
