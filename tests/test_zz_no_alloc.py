"""The allocation-free decode entry point, called through the C ABI.

fa_decode_splitkv_noalloc exists for callers that may not allocate device
memory during a call; its partial states live in a fixed device array of the
library.  Both it and fa_decode_splitkv run the same split and merge kernels
and merge the chunks in index order, so their outputs must be identical bit
for bit, and both must match the oracle's split-and-merge.  The checks run on
consecutive calls that reuse the array with different shapes, on two calls
queued back to back on one stream with no synchronisation between them, and
on the device memory pool: a call must leave the pool's high-water mark where
it was (the allocating entry point, measured the same way, raises it).
This file is collected last so a failure here leaves every other test run.
"""
import ctypes
import math

import pytest
import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300.inputs import make_qkv
from parity import check_decode

pytestmark = pytest.mark.gpu

# CUmemPool_attribute values (cuda.h): bytes of the pool in use now, and their high-water mark.
_USED_MEM_CURRENT, _USED_MEM_HIGH = 7, 8


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


class _DefaultPool:
    """The current device's default memory pool (the one cudaMallocAsync draws from), read through
    the driver API."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def get(self, attr):
        val = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(val)) == 0
        return val.value

    def reset_high(self):
        zero = ctypes.c_uint64(0)  # the high-water mark can only be reset, to the current use
        assert self.cu.cuMemPoolSetAttribute(self.pool, _USED_MEM_HIGH, ctypes.byref(zero)) == 0


def _high_water_rise(pool, call):
    torch.cuda.synchronize()
    pool.reset_high()
    base = pool.get(_USED_MEM_CURRENT)
    call()
    torch.cuda.synchronize()
    return pool.get(_USED_MEM_HIGH) - base


def test_noalloc_matches_allocating_entry_and_oracle_on_consecutive_calls(cuda_device):
    cases = [((4, 8, 4096, 64), 16, 31), ((2, 4, 3001, 128), 7, 32)]
    for (B, H, Nk, d), splits, seed in cases:  # the second call reuses the array with another shape
        q, k, v = make_qkv(B, H, 1, Nk, d, "bf16", seed=seed, device=cuda_device)
        q = q.reshape(B, H, d)
        ref = fa.fa_decode_splitkv(q, k, v, splits)
        o = torch.full((B, H, d), float("nan"), device=cuda_device, dtype=torch.bfloat16)
        assert _noalloc(q, k, v, o, splits) == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.fa_check_device_error() == fa.FA_OK
        assert torch.equal(o, ref)
        check_decode(q, k, v, o, None, 1 / math.sqrt(d), splits, name=f"noalloc {(B, H, Nk, d)} splits={splits}")


def test_noalloc_back_to_back_on_one_stream(cuda_device):
    """Two calls queued on one stream with no synchronisation between them: the second reuses the
    array only after the first call's merge has read it (stream order), so both outputs are right."""
    B, H, Nk, d, splits = 8, 8, 2048, 64, 16
    qa, ka, va = make_qkv(B, H, 1, Nk, d, "bf16", seed=41, device=cuda_device)
    qb, kb, vb = make_qkv(B, H, 1, Nk, d, "bf16", seed=42, device=cuda_device)
    qa, qb = qa.reshape(B, H, d), qb.reshape(B, H, d)
    ref_a = fa.fa_decode_splitkv(qa, ka, va, splits)
    ref_b = fa.fa_decode_splitkv(qb, kb, vb, splits)
    torch.cuda.synchronize()
    oa = torch.full((B, H, d), float("nan"), device=cuda_device, dtype=torch.bfloat16)
    ob = torch.full_like(oa, float("nan"))
    assert _noalloc(qa, ka, va, oa, splits) == fa.FA_OK
    assert _noalloc(qb, kb, vb, ob, splits) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    assert torch.equal(oa, ref_a) and torch.equal(ob, ref_b)


def test_noalloc_takes_nothing_from_the_memory_pool(cuda_device):
    B, H, Nk, d, splits = 4, 8, 4096, 64, 16
    q, k, v = make_qkv(B, H, 1, Nk, d, "bf16", seed=43, device=cuda_device)
    q = q.reshape(B, H, d)
    o = torch.empty((B, H, d), device=cuda_device, dtype=torch.bfloat16)
    assert _noalloc(q, k, v, o, splits) == fa.FA_OK  # first call on the device: set-up done here
    pool = _DefaultPool()
    ws = fa.lib().fa_decode_workspace_bytes(B, H, d, splits)
    # the probe sees the allocating entry point's stream-ordered workspace ...
    assert _high_water_rise(pool, lambda: fa.fa_decode_splitkv(q, k, v, splits, o=o)) >= ws
    # ... and nothing from the allocation-free one
    assert _high_water_rise(pool, lambda: _noalloc(q, k, v, o, splits)) == 0


def test_noalloc_rejects_work_beyond_the_scratch(cuda_device):
    # B*H*splits*(d+2)*4 bytes of states: 64*64*64*130*4 = 136 MB > 8 MiB
    q, k, v = make_qkv(1, 1, 1, 64, 64, "bf16", seed=1, device=cuda_device)
    B, H, Nk, d, splits = 64, 64, 4096, 128, 64
    assert fa.lib().fa_decode_workspace_bytes(B, H, d, splits) > (8 << 20)
    st = _c_fn()(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(), B, H, Nk, d, splits, None)
    assert st == fa.FA_ERR_UNSUPPORTED
