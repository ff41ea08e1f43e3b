"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/fa.h declares, and rejects bad arguments
before anything is launched."""
import ctypes
import os
import re

import pytest

import attention_forward_05_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

# Fake device addresses: never dereferenced, because every call below carries at
# least one invalid argument and validation precedes any CUDA call.
P = 0x10000
P2 = 0x20000


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_function():
    L = fa.lib()
    names = declared_functions()
    assert {"fa_fwd", "fa_decode_splitkv"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
    out = os.popen(f"nm -D --defined-only {fa.lib_path()}").read()
    for n in names:
        assert re.search(rf"\bT {n}$", out, re.M), n


def test_status_strings():
    assert fa.status_string(0) == "FA_OK"
    assert fa.status_string(4) == "FA_ERR_TIMEOUT"
    assert fa.status_string(99) == "FA_ERR_UNKNOWN"


def _fwd(**kw):
    a = dict(q=P, k=P, v=P, o=P2, lse=None, B=1, H=1, Nq=16, Nk=16, d=64, scale=0.125, dtype=fa.FA_BF16)
    a.update(kw)
    return fa.lib().fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                           a["scale"], a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(k=P + 8), fa.FA_ERR_INVALID_ARG),
    (dict(lse=P + 2), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=-1), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=7), fa.FA_ERR_UNSUPPORTED),
    (dict(B=1 << 16, H=1 << 16), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 10, H=1 << 10, Nq=1 << 20), fa.FA_ERR_INVALID_ARG),
])
def test_fwd_rejects(kw, status):
    assert _fwd(**kw) == status


def _dec(**kw):
    a = dict(q=P, k=P, v=P, o=P2, B=2, H=2, Nk=64, d=64, splits=4, scale=0.125, ws=None, ws_bytes=0,
             order=None, lse=None)
    a.update(kw)
    return fa.lib().fa_decode_splitkv_ex(a["q"], a["k"], a["v"], a["o"], a["B"], a["H"], a["Nk"], a["d"],
                                         a["splits"], a["scale"], a["ws"], a["ws_bytes"], a["order"], a["lse"],
                                         None)


@pytest.mark.parametrize("kw,status", [
    (dict(v=None), fa.FA_ERR_INVALID_ARG),
    (dict(q=P + 4), fa.FA_ERR_INVALID_ARG),
    (dict(splits=0), fa.FA_ERR_INVALID_ARG),
    (dict(splits=65), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=1 << 30), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=8192, splits=5000), fa.FA_ERR_UNSUPPORTED),
    (dict(d=80), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(ws=P, ws_bytes=16), fa.FA_ERR_INVALID_ARG),
    (dict(ws=P + 8, ws_bytes=1 << 20), fa.FA_ERR_INVALID_ARG),
    (dict(order=P + 2), fa.FA_ERR_INVALID_ARG),
    (dict(lse=P + 1), fa.FA_ERR_INVALID_ARG),
])
def test_decode_rejects(kw, status):
    assert _dec(**kw) == status


def test_decode_plain_rejects():
    L = fa.lib()
    assert L.fa_decode_splitkv(None, P, P, P2, 1, 1, 16, 64, 2, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_decode_splitkv(P, P, P, P2, 1, 1, 16, 48, 2, None) == fa.FA_ERR_UNSUPPORTED
    assert L.fa_decode_splitkv(P, P, P, P2, 1, 1, 16, 64, 17, None) == fa.FA_ERR_INVALID_ARG


def test_workspace_bytes():
    L = fa.lib()
    assert L.fa_decode_workspace_bytes(32, 32, 64, 16) == 32 * 32 * 16 * 66 * 4
    assert L.fa_decode_workspace_bytes(1, 1, 128, 3) == 1792  # 3*130*4 = 1560 rounded up to 256
    assert L.fa_decode_workspace_bytes(0, 1, 64, 1) == 0
    assert L.fa_decode_workspace_bytes(1, 1, 100, 1) == 0


def test_debug_fault_arg():
    L = fa.lib()
    assert L.fa_debug_set_fault(2) == fa.FA_ERR_INVALID_ARG
    assert L.fa_debug_set_fault(-1) == fa.FA_ERR_INVALID_ARG
    assert L.fa_debug_set_fault(0) == fa.FA_OK


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(x, x, x)
    with pytest.raises(ValueError):
        fa.fa_decode_splitkv(x, x, x, 2)


def test_library_has_no_oracle_dependency():
    """The product library never links or names the oracle."""
    out = os.popen(f"nm -D {fa.lib_path()}").read()
    assert "fao_" not in out
    src_dir = os.path.join(ROOT, "attention_forward_05_gb300")
    for dirpath, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f


def _fwd_ex(**kw):
    a = dict(q=P, k=P, v=P, o=P2, lse=None, B=1, H=4, Hkv=2, Nq=16, Nk=256, d=64, scale=0.125, dtype=fa.FA_BF16,
             causal=0, kv_splits=1, ws=None, ws_bytes=0)
    a.update(kw)
    return fa.lib().fa_fwd_ex(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Hkv"], a["Nq"], a["Nk"],
                              a["d"], a["scale"], a["dtype"], a["causal"], a["kv_splits"], a["ws"], a["ws_bytes"],
                              None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hkv=3), fa.FA_ERR_INVALID_ARG),          # 4 query heads cannot share 3 key/value heads
    (dict(Hkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(causal=1, Nq=300, Nk=256), fa.FA_ERR_INVALID_ARG),  # rows 0..43 would see no key
    (dict(kv_splits=-1), fa.FA_ERR_INVALID_ARG),
    (dict(kv_splits=5), fa.FA_ERR_INVALID_ARG),    # 256 keys are 4 bf16 d=64 key tiles of 64
    (dict(ws=P + 4, kv_splits=2), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(v=None), fa.FA_ERR_INVALID_ARG),
])
def test_fwd_ex_rejects(kw, status):
    assert _fwd_ex(**kw) == status


def test_fwd_workspace_bytes_explicit_splits():
    L = fa.lib()
    # bf16, one split: no workspace
    assert L.fa_fwd_workspace_bytes(1, 4, 2, 100, 256, 64, fa.FA_BF16, 0, 1) == 0
    # bf16, 2 splits: fp32 O (2*4*100*64*4 = 204800) + (m, l) (2*4*100*2*4 = 6400, a multiple of 256)
    assert L.fa_fwd_workspace_bytes(1, 4, 2, 100, 256, 64, fa.FA_BF16, 0, 2) == 204800 + 6400
    # fp32, one split: rounded Q (1*4*100*64*4 = 102400), rounded K (1*2*256*64*4), V^T (1*2*64*256*4)
    assert L.fa_fwd_workspace_bytes(1, 4, 2, 100, 256, 64, fa.FA_FP32, 0, 1) == 102400 + 131072 + 131072
    assert L.fa_fwd_workspace_bytes(1, 4, 3, 100, 256, 64, fa.FA_BF16, 0, 1) == 0  # invalid heads


def _bwd(**kw):
    a = dict(q=P, k=P, v=P, o=P, do=P, lse=P, dq=P2, dk=P2, dv=P2, B=1, H=4, Hkv=2, Nq=100, Nk=256, d=64,
             scale=0.125, dtype=fa.FA_BF16, causal=0, ws=None, ws_bytes=0)
    a.update(kw)
    return fa.lib().fa_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"], a["B"],
                           a["H"], a["Hkv"], a["Nq"], a["Nk"], a["d"], a["scale"], a["dtype"], a["causal"], a["ws"],
                           a["ws_bytes"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(do=None), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(dk=P2 + 8), fa.FA_ERR_INVALID_ARG),
    (dict(lse=P + 2), fa.FA_ERR_INVALID_ARG),
    (dict(Hkv=3), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=1, Nq=300), fa.FA_ERR_INVALID_ARG),
    (dict(causal=3), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=7), fa.FA_ERR_UNSUPPORTED),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(ws=P, ws_bytes=16), fa.FA_ERR_INVALID_ARG),
    (dict(ws=P + 4, ws_bytes=1 << 20), fa.FA_ERR_INVALID_ARG),
])
def test_bwd_rejects(kw, status):
    assert _bwd(**kw) == status


def test_bwd_workspace_bytes():
    L = fa.lib()
    # D and -LSE log2(e), fp32, Nq rounded up to 64: 1*4*128*4 = 2048 bytes each
    assert L.fa_bwd_workspace_bytes(1, 4, 100, 64) == 2 * 2048
    assert L.fa_bwd_workspace_bytes(2, 3, 64, 128) == 2 * 1536
    assert L.fa_bwd_workspace_bytes(1, 1, 1, 64) == 2 * 256  # 256 bytes rounded to 256
    assert L.fa_bwd_workspace_bytes(1, 1, 64, 80) == 0
    assert L.fa_bwd_workspace_bytes(0, 1, 64, 64) == 0


def _dec_gqa(**kw):
    a = dict(q=P, k=P, v=P, o=P2, B=2, H=8, Hkv=2, Nk=64, d=64, splits=4, scale=0.125, ws=None, ws_bytes=0,
             order=None, lse=None)
    a.update(kw)
    return fa.lib().fa_decode_splitkv_gqa(a["q"], a["k"], a["v"], a["o"], a["B"], a["H"], a["Hkv"], a["Nk"], a["d"],
                                          a["splits"], a["scale"], a["ws"], a["ws_bytes"], a["order"], a["lse"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(k=None), fa.FA_ERR_INVALID_ARG),
    (dict(v=P + 8), fa.FA_ERR_INVALID_ARG),
    (dict(Hkv=3), fa.FA_ERR_INVALID_ARG),     # 8 query heads cannot share 3 key/value heads
    (dict(Hkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=6, Hkv=2), fa.FA_ERR_UNSUPPORTED),  # groups of 3
    (dict(H=24, Hkv=2), fa.FA_ERR_UNSUPPORTED),  # groups of 12
    (dict(splits=0), fa.FA_ERR_INVALID_ARG),
    (dict(splits=65), fa.FA_ERR_INVALID_ARG),
    (dict(d=80), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(ws=P, ws_bytes=16), fa.FA_ERR_INVALID_ARG),
    (dict(order=P + 2), fa.FA_ERR_INVALID_ARG),
])
def test_decode_gqa_rejects(kw, status):
    assert _dec_gqa(**kw) == status


def test_fwd_host_rejects_and_workspace():
    L = fa.lib()
    # argument errors come back before any device work
    assert L.fa_fwd_host(None, P, P, P2, None, 1, 4, 2, 64, 64, 64, 0.125, fa.FA_BF16, 0, None, 0, None) == \
        fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_host(P, P, P, P2, None, 1, 4, 3, 64, 64, 64, 0.125, fa.FA_BF16, 0, None, 0, None) == \
        fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_host(P, P, P, P2, None, 1, 4, 2, 64, 64, 96, 0.125, fa.FA_BF16, 0, None, 0, None) == \
        fa.FA_ERR_UNSUPPORTED
    assert L.fa_fwd_host(P, P, P, P2, None, 1, 4, 2, 64, 64, 64, 0.125, fa.FA_BF16, 0, P, 16, None) == \
        fa.FA_ERR_INVALID_ARG
    # q 1*4*100*64*2 = 51200, k/v 1*2*256*64*2 = 65536 each, o 51200, lse 1600 -> 1792 (256-rounded)
    assert L.fa_fwd_host_workspace_bytes(1, 4, 2, 100, 256, 64, fa.FA_BF16, 0) == 51200 + 65536 * 2 + 51200 + 1792
    assert L.fa_fwd_host_workspace_bytes(1, 4, 3, 100, 256, 64, fa.FA_BF16, 0) == 0


def test_binding_fwd_host_rejects_device_tensors():
    import torch
    if not torch.cuda.is_available():
        x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
        with pytest.raises(TypeError):
            fa.fa_fwd_host(x, x, x.float())
