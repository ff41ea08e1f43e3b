"""Float64 CPU oracle for exact softmax attention and its split-KV form.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``attention_forward_05_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double, single thread, no
FMA contraction); this module compiles it with gcc and wraps it with ctypes.
``forms.py`` holds the pages' other, slower formulations (2-pass, 1-pass tiled,
KV-outer Algorithm 1, blocked-concatenation) written in numpy, used only as
cross-checks of the plain definition; ``brute.py`` holds an mpmath brute force.

Sources (web pages, cited by title and section):
  [T1] "FlashAttention 简化版：Tiling + Online Softmax" (forceinjection.github.io)
  [T2] "Flash Attention 代码填空 (Level 2-3)" (boots-coder.github.io, LLM-101-CN)
  [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com)
  [T4] "从零手写 FlashAttention（PyTorch实现 + 原理推导）" (mokono.cn)

Definition followed: S = Q K^T * scale, P = row-softmax(S) with the row maximum
subtracted, O = P V, LSE = m + ln(l) ([T1] §1.1, §2.1; [T2] Exercise 1;
[T3] attn_row_3pass and demo 2).  Partial states (m, l, o) with o unnormalised
and their merge follow [T3] demo 2.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def compile_c(src: str, out: str) -> str:
    """gcc build of a copy of the oracle's C source into a shared library at `out`.

    ``-ffp-contract=off`` keeps gcc from fusing multiply-adds (its default on
    aarch64), so the oracle rounds the same way on every host.
    """
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc; returns its path."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(_OUT_DIR, exist_ok=True)
    return compile_c(_SRC, _SO)


def source_path() -> str:
    return _SRC


@contextlib.contextmanager
def swapped_library(path: str):
    """Test support: the wrappers below call into the library at `path` (another build of oracle.c,
    e.g. one with a planted mistake) until the block exits."""
    global _lib
    other = _configure(ctypes.CDLL(path))
    with _lock:
        prev, _lib = _lib, other
    try:
        yield
    finally:
        with _lock:
            _lib = prev


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


def _configure(lib):
    """Declares the C signatures on a loaded oracle library."""
    lib.fao_attention_head.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_long,
                                       ctypes.c_long, ctypes.c_long, ctypes.c_double]
    lib.fao_attention_head.restype = ctypes.c_int
    lib.fao_attention.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                  ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_double]
    lib.fao_attention.restype = ctypes.c_int
    lib.fao_attention_head_limits.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                              ctypes.c_long, ctypes.c_double,
                                              ctypes.POINTER(ctypes.c_long)]
    lib.fao_attention_head_limits.restype = ctypes.c_int
    lib.fao_attention_bwd_head.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_long,
                                           ctypes.c_long, ctypes.c_long, ctypes.c_double]
    lib.fao_attention_bwd_head.restype = ctypes.c_int
    lib.fao_attention_bwd_head_limits.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_long,
                                                  ctypes.c_long, ctypes.c_long, ctypes.c_double,
                                                  ctypes.POINTER(ctypes.c_long)]
    lib.fao_attention_bwd_head_limits.restype = ctypes.c_int
    lib.fao_partial_state.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                      ctypes.c_double, _dp, _dp, _dp]
    lib.fao_partial_state.restype = ctypes.c_int
    lib.fao_merge_states.argtypes = [ctypes.c_double, ctypes.c_double, _dp, ctypes.c_double,
                                     ctypes.c_double, _dp, ctypes.c_long, _dp, _dp, _dp]
    lib.fao_merge_states.restype = None
    lib.fao_decode_splitkv.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                       ctypes.c_long, ctypes.c_long, ctypes.c_double, _ip]
    lib.fao_decode_splitkv.restype = ctypes.c_int
    return lib


def _f64(a) -> np.ndarray:
    """Exact up-cast of a numpy array or a (CPU or CUDA) torch tensor to C-contiguous float64."""
    if not isinstance(a, np.ndarray):  # torch tensor: go through float32, which holds bf16 exactly
        import torch  # local: only when a tensor is handed in
        t = a.detach()
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.float()
        a = t.cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def causal_limits(rows, nq_total: int, nk: int) -> np.ndarray:
    """Visible keys per query row under a causal mask aligned to the bottom-right corner.

    Query row i (of nq_total) sees keys 0 .. i + (nk - nq_total): the last query sees every key,
    and with nq_total == nk this is the usual lower triangle.  Requires nq_total <= nk.
    """
    if nq_total > nk:
        raise ValueError("causal attention needs Nq <= Nk")
    return np.asarray(rows, dtype=np.int64) + (nk - nq_total) + 1


def attention(q, k, v, scale: float, causal: bool = False, rows=None, nq_total=None):
    """Exact attention on [..., N, d] inputs; returns (O, LSE) as float64 arrays.

    Leading dimensions (batch, heads) must agree between q, k and v; each head
    is independent.  LSE has shape [..., Nq].  With 4-D inputs k and v may
    have fewer heads Hkv than q (grouped-query attention): query head h then
    uses key/value head h // (H / Hkv), i.e. consecutive query heads share one
    key/value head.

    causal: each query row only sees keys up to its causal limit (see
    causal_limits).  When q holds a subset of the query rows, `rows` gives
    their indices and `nq_total` the full query length.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if causal:
        return _attention_causal(q, k, v, scale, rows, nq_total)
    if q.ndim == 4 and k.ndim == 4 and k.shape[1] != q.shape[1]:
        if q.shape[1] % k.shape[1] != 0:
            raise ValueError("query heads must be a multiple of key/value heads")
        group = q.shape[1] // k.shape[1]
        k = np.ascontiguousarray(np.repeat(k, group, axis=1))
        v = np.ascontiguousarray(np.repeat(v, group, axis=1))
    if q.ndim < 2 or k.shape != v.shape or q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
        raise ValueError("shape mismatch")
    lead = q.shape[:-2]
    nq, d = q.shape[-2:]
    nk = k.shape[-2]
    bh = int(np.prod(lead)) if lead else 1
    o = np.empty_like(q)
    lse = np.empty(lead + (nq,), dtype=np.float64)
    _check(_load().fao_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), 1, bh, nq, nk, d,
                                 float(scale)), "attention")
    return o, lse


def _attention_causal(q, k, v, scale, rows, nq_total):
    if q.ndim == 4 and k.ndim == 4 and k.shape[1] != q.shape[1]:
        group = q.shape[1] // k.shape[1]
        k = np.ascontiguousarray(np.repeat(k, group, axis=1))
        v = np.ascontiguousarray(np.repeat(v, group, axis=1))
    lead = q.shape[:-2]
    nq, d = q.shape[-2:]
    nk = k.shape[-2]
    if rows is None:
        rows = np.arange(nq)
    limits = np.ascontiguousarray(causal_limits(rows, nq if nq_total is None else nq_total, nk), dtype=np.int64)
    lim_p = limits.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
    qf, kf, vf = q.reshape(-1, nq, d), k.reshape(-1, nk, d), v.reshape(-1, nk, d)
    o = np.empty_like(qf)
    lse = np.empty(qf.shape[:2], dtype=np.float64)
    L = _load()
    for h in range(qf.shape[0]):
        qh, kh, vh = (np.ascontiguousarray(x[h]) for x in (qf, kf, vf))
        oh = np.empty((nq, d))
        lh = np.empty(nq)
        _check(L.fao_attention_head_limits(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(oh), _ptr(lh), nq, nk, d,
                                           float(scale), lim_p), "attention (causal)")
        o[h], lse[h] = oh, lh
    return o.reshape(lead + (nq, d)), lse.reshape(lead + (nq,))


def attention_bwd(q, k, v, dout, scale: float, causal: bool = False):
    """Gradients (dQ, dK, dV) of exact attention for a loss whose gradient w.r.t. O is dout.

    q, dout [..., H, Nq, d]; k, v [..., Hkv, Nk, d] with H a multiple of Hkv: query head h reads
    key/value head h // (H // Hkv), and dK, dV of a shared head sum the contributions of its
    query heads.  causal: row i sees keys 0 .. i + Nk - Nq (bottom-right aligned).
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    nq, d = q.shape[-2:]
    nk = k.shape[-2]
    H, Hkv = (q.shape[-3], k.shape[-3]) if q.ndim >= 3 else (1, 1)
    group = H // Hkv
    if group > 1:
        k, v = np.repeat(k, group, axis=-3), np.repeat(v, group, axis=-3)
    lead = q.shape[:-2]
    qf, kf, vf, gf = q.reshape(-1, nq, d), k.reshape(-1, nk, d), v.reshape(-1, nk, d), dout.reshape(-1, nq, d)
    dq, dk, dv = np.empty_like(qf), np.empty_like(kf), np.empty_like(vf)
    lim = None
    if causal:
        lim = np.ascontiguousarray(causal_limits(np.arange(nq), nq, nk), dtype=np.int64)
        if (lim < 1).any():
            raise ValueError("causal mask needs Nq <= Nk")
    L = _load()
    for h in range(qf.shape[0]):
        a, b, c_, g = (np.ascontiguousarray(x[h]) for x in (qf, kf, vf, gf))
        oq, ok_, ov = np.empty((nq, d)), np.empty((nk, d)), np.empty((nk, d))
        if lim is None:
            rc = L.fao_attention_bwd_head(_ptr(a), _ptr(b), _ptr(c_), _ptr(g), _ptr(oq), _ptr(ok_), _ptr(ov), nq, nk,
                                          d, float(scale))
        else:
            rc = L.fao_attention_bwd_head_limits(_ptr(a), _ptr(b), _ptr(c_), _ptr(g), _ptr(oq), _ptr(ok_), _ptr(ov),
                                                 nq, nk, d, float(scale),
                                                 lim.ctypes.data_as(ctypes.POINTER(ctypes.c_long)))
        _check(rc, "attention_bwd")
        dq[h], dk[h], dv[h] = oq, ok_, ov
    dq = dq.reshape(lead + (nq, d))
    dk = dk.reshape(k.shape)
    dv = dv.reshape(v.shape)
    if group > 1:  # sum over the query heads that share a key/value head
        shp = dk.shape[:-3] + (Hkv, group, nk, d)
        dk, dv = dk.reshape(shp).sum(axis=-3), dv.reshape(shp).sum(axis=-3)
    return dq, dk, dv


def partial_state(q, k, v, scale: float):
    """(m, l, o) of one query q [d] over keys k/v [n, d] (n may be 0); o unnormalised."""
    q, k, v = _f64(q), _f64(k).reshape(-1, len(q)), _f64(v)
    n, d = k.shape[0], q.shape[0]
    if v.size != n * d:
        raise ValueError("v must be [n, d] like k")
    v = v.reshape(n, d)
    m, l = ctypes.c_double(), ctypes.c_double()
    o = np.empty(d, dtype=np.float64)
    _check(_load().fao_partial_state(_ptr(q), _ptr(k), _ptr(v), n, d, float(scale),
                                     ctypes.byref(m), ctypes.byref(l), _ptr(o)), "partial_state")
    return m.value, l.value, o


def merge_states(a, b):
    """Merge two partial states (m, l, o) -> (m, l, o)."""
    (ma, la, oa), (mb, lb, ob) = a, b
    oa, ob = _f64(oa), _f64(ob)
    d = oa.shape[0]
    m, l = ctypes.c_double(), ctypes.c_double()
    o = np.empty(d, dtype=np.float64)
    _load().fao_merge_states(float(ma), float(la), _ptr(oa), float(mb), float(lb), _ptr(ob), d,
                             ctypes.byref(m), ctypes.byref(l), _ptr(o))
    return m.value, l.value, o


def finish(state) -> np.ndarray:
    """Normalised output o / l of a partial state."""
    _, l, o = state
    return o / l


def decode_splitkv(q, k, v, splits: int, scale: float, order=None):
    """Split-KV attention of one query per head.

    q [..., d] (or [..., 1, d]), k/v [..., Nk, d].  Keys are cut into `splits`
    chunks of ceil(Nk/splits); chunk states are merged in `order` (a
    permutation; None = index order).  Returns (O [..., d], LSE [...]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead = k.shape[:-2]
    nk, d = k.shape[-2:]
    q = q.reshape(lead + (d,))
    bh = int(np.prod(lead)) if lead else 1
    o = np.empty(lead + (d,), dtype=np.float64)
    lse = np.empty(lead, dtype=np.float64)
    ordp = None
    if order is not None:
        order = np.ascontiguousarray(order, dtype=np.int32)
        if order.shape != (splits,):
            raise ValueError("order must be a permutation of range(splits)")
        ordp = order.ctypes.data_as(_ip)
    _check(_load().fao_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), bh, nk, d,
                                      int(splits), float(scale), ordp), "decode_splitkv")
    return o, lse
