"""attention_forward_05_gb300 -- Python binding of libfa (FlashAttention forward for GB300).

This module only marshals arguments: it checks tensors, takes their device
pointers and the current CUDA stream, and calls the C ABI of ``libfa.so``
(declared in ``include/fa.h``).  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.  If the library is missing or
fails to load, importing the binding's entry points raises.

Entry points (same names as the C ABI):
  fa_fwd(q, k, v, scale=None, o=None, lse=None, with_lse=True, kv_splits=0, causal=False, workspace=None)
      -> (o, lse)      (calls fa_fwd_ex; k/v may have fewer heads than q)
  fa_fwd_workspace_bytes(B, H, Hkv, Nq, Nk, d, dtype, causal, kv_splits)
  fa_fwd_host(q, k, v, scale=None, o=None, lse=None, with_lse=True, causal=False, workspace=None)
      -> (o, lse)      (host tensors in and out; copies overlap compute)
  fa_fwd_host_workspace_bytes(B, H, Hkv, Nq, Nk, d, dtype, causal)
  fa_decode_splitkv(q, k, v, splits, o=None) -> o
  fa_decode_splitkv_ex(q, k, v, splits, scale=None, workspace=None, merge_order=None, with_lse=False)
  fa_decode_workspace_bytes(B, H, d, splits)
  fa_decode_splitkv_gqa(q, k, v, splits, scale=None, workspace=None, merge_order=None, with_lse=False)
  fa_bwd(q, k, v, o, dout, lse, scale=None, causal=False, workspace=None) -> (dq, dk, dv)
  fa_bwd_workspace_bytes(B, H, Nq, d)
  fa_check_device_error()
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import _build

FA_FP32, FA_BF16 = 0, 1
FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)} ({status})"
        if status == FA_ERR_CUDA:
            L = lib()
            msg += f": {L.fa_last_cuda_error_string().decode()} [{L.fa_last_cuda_error()}]"
        super().__init__(msg)


def lib_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libfa.so (built first if stale).  Raises if it cannot be built or loaded."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if _build.is_stale() else _build.LIB
            L = ctypes.CDLL(path)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
            L.fa_fwd.restype = i
            L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, i, vp, sz, vp]
            L.fa_fwd_ex.restype = i
            L.fa_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i, i]
            L.fa_fwd_workspace_bytes.restype = sz
            L.fa_decode_splitkv.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
            L.fa_decode_splitkv.restype = i
            L.fa_decode_splitkv_ex.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp, vp, vp]
            L.fa_decode_splitkv_ex.restype = i
            L.fa_decode_splitkv_gqa.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, vp, sz, vp, vp, vp]
            L.fa_decode_splitkv_gqa.restype = i
            L.fa_decode_workspace_bytes.argtypes = [i, i, i, i]
            L.fa_decode_workspace_bytes.restype = sz
            L.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, sz, vp]
            L.fa_fwd_host.restype = i
            L.fa_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
            L.fa_fwd_host_workspace_bytes.restype = sz
            L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, sz, vp]
            L.fa_bwd.restype = i
            L.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
            L.fa_bwd_workspace_bytes.restype = sz
            L.fa_check_device_error.argtypes = []
            L.fa_check_device_error.restype = i
            L.fa_status_string.argtypes = [i]
            L.fa_status_string.restype = ctypes.c_char_p
            L.fa_debug_set_fault.argtypes = [i]
            L.fa_debug_set_fault.restype = i
            L.fa_last_cuda_error.argtypes = []
            L.fa_last_cuda_error.restype = i
            L.fa_last_cuda_error_string.argtypes = []
            L.fa_last_cuda_error_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FAError(status, where)


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32")


def _need_cuda_contig(name: str, t: torch.Tensor) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device and encodes its tensor maps there
        raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
           o: torch.Tensor | None = None, lse: torch.Tensor | None = None, with_lse: bool = True,
           stream=None, kv_splits: int = 0, causal: bool = False, workspace: torch.Tensor | None = None):
    """Exact attention softmax(q k^T * scale) v; returns (o, lse or None).

    q [B, H, Nq, d]; k, v [B, Hkv, Nk, d] with H a multiple of Hkv (grouped-query
    attention when Hkv < H).  kv_splits: 0 automatic, 1 none, n > 1 split keys.
    Calls fa_fwd_ex.
    """
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda_contig(n, t)
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Nq,d], k/v [B,Hkv,Nk,d] expected")
    if q.shape[1] % k.shape[1] != 0:
        raise ValueError("query heads must be a multiple of key/value heads")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    _need_cuda_contig("o", o)
    if o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("o must match q")
    if lse is None and with_lse:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    if lse is not None:
        _need_cuda_contig("lse", lse)
        if lse.shape != (B, H, Nq) or lse.dtype != torch.float32:
            raise ValueError("lse must be fp32 [B,H,Nq]")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need_cuda_contig("workspace", workspace)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib().fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                         lse.data_ptr() if lse is not None else None, B, H, Hkv, Nq, Nk, d, float(scale),
                         _dtype_code(q), int(bool(causal)), int(kv_splits), ws_ptr, ws_bytes,
                         _stream_handle(stream))
    _check(st, "fa_fwd_ex")
    return o, lse


def fa_fwd_workspace_bytes(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int, dtype=torch.bfloat16,
                           causal: bool = False, kv_splits: int = 0) -> int:
    code = FA_BF16 if dtype == torch.bfloat16 else FA_FP32
    return int(lib().fa_fwd_workspace_bytes(B, H, Hkv, Nq, Nk, d, code, int(bool(causal)), int(kv_splits)))


def _need_host_contig(name: str, t: torch.Tensor) -> None:
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fa_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
                o: torch.Tensor | None = None, lse: torch.Tensor | None = None, with_lse: bool = True,
                causal: bool = False, workspace: torch.Tensor | None = None, stream=None):
    """fa_fwd on host (CPU) tensors; returns host (o, lse or None), valid once `stream` (default: the
    current CUDA stream) has finished.  Pinned inputs and outputs let the copies overlap the compute."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need_host_contig(n, t)
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Nq,d], k/v [B,Hkv,Nk,d] expected")
    if q.shape[1] % k.shape[1] != 0:
        raise ValueError("query heads must be a multiple of key/value heads")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    _need_host_contig("o", o)
    if o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("o must match q")
    if lse is None and with_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=q.is_pinned())
    if lse is not None:
        _need_host_contig("lse", lse)
        if lse.shape != (B, H, Nq) or lse.dtype != torch.float32:
            raise ValueError("lse must be fp32 [B,H,Nq]")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need_cuda_contig("workspace", workspace)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib().fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr() if lse is not None else None, B, H, Hkv, Nq, Nk, d, float(scale),
                           _dtype_code(q), int(bool(causal)), ws_ptr, ws_bytes, _stream_handle(stream))
    _check(st, "fa_fwd_host")
    return o, lse


def fa_fwd_host_workspace_bytes(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int, dtype=torch.bfloat16,
                                causal: bool = False) -> int:
    code = FA_BF16 if dtype == torch.bfloat16 else FA_FP32
    return int(lib().fa_fwd_host_workspace_bytes(B, H, Hkv, Nq, Nk, d, code, int(bool(causal))))


def fa_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, dout: torch.Tensor,
           lse: torch.Tensor, scale: float | None = None, causal: bool = False,
           dq: torch.Tensor | None = None, dk: torch.Tensor | None = None, dv: torch.Tensor | None = None,
           workspace: torch.Tensor | None = None, stream=None):
    """Gradients (dq, dk, dv) of attention given the forward's o and lse and the output gradient dout.

    q, o, dout [B, H, Nq, d]; k, v [B, Hkv, Nk, d], all bf16 or all fp32; lse [B, H, Nq] fp32 from fa_fwd.
    """
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("lse", lse)):
        _need_cuda_contig(n, t)
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Nq,d], k/v [B,Hkv,Nk,d] expected")
    if o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("o and dout must match q")
    if q.shape[1] % k.shape[1] != 0:
        raise ValueError("query heads must be a multiple of key/value heads")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype):
        raise TypeError("q, k, v, o, dout must share a dtype")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32:
        raise ValueError("lse must be fp32 [B,H,Nq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for n, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _need_cuda_contig(n, t)
        if t.shape != ref.shape or t.dtype != ref.dtype:
            raise ValueError(f"{n} must match its input")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need_cuda_contig("workspace", workspace)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Hkv, Nq, Nk, d, float(scale),
                      _dtype_code(q), int(bool(causal)), ws_ptr, ws_bytes, _stream_handle(stream))
    _check(st, "fa_bwd")
    return dq, dk, dv


def fa_bwd_workspace_bytes(B: int, H: int, Nq: int, d: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, Nq, d))


def _decode_shapes(q, k, v):
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda_contig(n, t)
    if k.dim() != 4 or k.shape != v.shape:
        raise ValueError("k/v [B,H,Nk,d] expected")
    B, H, Nk, d = k.shape
    if q.numel() != B * H * d:
        raise ValueError("q must hold B*H*d elements ([B,H,d] or [B,H,1,d])")
    if not (q.dtype == k.dtype == v.dtype == torch.bfloat16):
        raise TypeError("decode takes bf16 q, k, v")
    return B, H, Nk, d


def fa_decode_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, splits: int,
                      o: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Split-KV decode with scale 1/sqrt(d); returns o [B, H, d] bf16."""
    B, H, Nk, d = _decode_shapes(q, k, v)
    if o is None:
        o = torch.empty((B, H, d), device=q.device, dtype=torch.bfloat16)
    _need_cuda_contig("o", o)
    st = lib().fa_decode_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, Nk, d,
                                 int(splits), _stream_handle(stream))
    _check(st, "fa_decode_splitkv")
    return o


def fa_decode_workspace_bytes(B: int, H: int, d: int, splits: int) -> int:
    return int(lib().fa_decode_workspace_bytes(B, H, d, splits))


def fa_decode_splitkv_ex(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, splits: int,
                         scale: float | None = None, workspace: torch.Tensor | None = None,
                         merge_order: torch.Tensor | None = None, with_lse: bool = False,
                         o: torch.Tensor | None = None, stream=None):
    """Split-KV decode with explicit scale, caller workspace, merge order and LSE; returns (o, lse)."""
    B, H, Nk, d = _decode_shapes(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty((B, H, d), device=q.device, dtype=torch.bfloat16)
    _need_cuda_contig("o", o)
    lse = torch.empty((B, H), device=q.device, dtype=torch.float32) if with_lse else None
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need_cuda_contig("workspace", workspace)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    ord_ptr = None
    if merge_order is not None:
        _need_cuda_contig("merge_order", merge_order)
        if merge_order.dtype != torch.int32 or merge_order.numel() != splits:
            raise ValueError("merge_order must be int32 [splits]")
        ord_ptr = merge_order.data_ptr()
    st = lib().fa_decode_splitkv_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, Nk, d,
                                    int(splits), float(scale), ws_ptr, ws_bytes, ord_ptr,
                                    lse.data_ptr() if lse is not None else None, _stream_handle(stream))
    _check(st, "fa_decode_splitkv_ex")
    return o, lse


def fa_decode_splitkv_gqa(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, splits: int,
                          scale: float | None = None, workspace: torch.Tensor | None = None,
                          merge_order: torch.Tensor | None = None, with_lse: bool = False,
                          o: torch.Tensor | None = None, stream=None):
    """Split-KV decode with Hkv = k.shape[1] key/value heads shared by q's H query heads; returns (o, lse).

    q [B, H, d] or [B, H, 1, d]; k, v [B, Hkv, Nk, d]; all bf16.
    """
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda_contig(n, t)
    if k.dim() != 4 or k.shape != v.shape:
        raise ValueError("k/v [B,Hkv,Nk,d] expected")
    B, Hkv, Nk, d = k.shape
    if q.dim() not in (3, 4) or q.shape[0] != B or q.shape[-1] != d or (q.dim() == 4 and q.shape[2] != 1):
        raise ValueError("q [B,H,d] or [B,H,1,d] expected")
    H = q.shape[1]
    if not (q.dtype == k.dtype == v.dtype == torch.bfloat16):
        raise TypeError("decode takes bf16 q, k, v")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty((B, H, d), device=q.device, dtype=torch.bfloat16)
    _need_cuda_contig("o", o)
    lse = torch.empty((B, H), device=q.device, dtype=torch.float32) if with_lse else None
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need_cuda_contig("workspace", workspace)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    ord_ptr = None
    if merge_order is not None:
        _need_cuda_contig("merge_order", merge_order)
        if merge_order.dtype != torch.int32 or merge_order.numel() != splits:
            raise ValueError("merge_order must be int32 [splits]")
        ord_ptr = merge_order.data_ptr()
    st = lib().fa_decode_splitkv_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, Hkv, Nk, d,
                                     int(splits), float(scale), ws_ptr, ws_bytes, ord_ptr,
                                     lse.data_ptr() if lse is not None else None, _stream_handle(stream))
    _check(st, "fa_decode_splitkv_gqa")
    return o, lse


def fa_decode_splitkv_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, splits: int,
                              o: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fa_decode_splitkv whose partial states use the library's fixed device scratch array.

    For callers that may not allocate device memory during a call; the C
    declaration in include/fa.h lists the size limit and the sharing rules
    (calls that overlap on the GPU race on the one array).
    """
    B, H, Nk, d = _decode_shapes(q, k, v)
    if o is None:
        o = torch.empty((B, H, d), device=q.device, dtype=torch.bfloat16)
    _need_cuda_contig("o", o)
    L = lib()
    fn = L.fa_decode_splitkv_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    fn.restype = i
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, Nk, d, int(splits),
            _stream_handle(stream))
    _check(st, "fa_decode_splitkv_noalloc")
    return o


def fa_check_device_error() -> int:
    """Synchronises the current device and returns (and clears) the library's device status."""
    return int(lib().fa_check_device_error())


def fa_debug_set_fault(mode: int) -> int:
    """Test only: arm (1) or disarm (0) the load-warp fault of the next fa_fwd launch."""
    return int(lib().fa_debug_set_fault(int(mode)))
