"""The pages' alternative formulations of attention, in numpy float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Each function restates
one algorithm the pages describe, in the pages' loop order, so that tests can
check that every form reaches the same result as the plain definition in
``oracle.c``.  None of them is used by the CUDA library.

Sources (web pages, cited by title and section):
  [T1] "FlashAttention 简化版：Tiling + Online Softmax" (forceinjection.github.io)
  [T2] "Flash Attention 代码填空 (Level 2-3)" (boots-coder.github.io, LLM-101-CN)
  [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com)
  [T4] "从零手写 FlashAttention（PyTorch实现 + 原理推导）" (mokono.cn)
"""
from __future__ import annotations

import math

import numpy as np


# ----------------------------------------------------------------------------
# softmax of a matrix, row by row
# ----------------------------------------------------------------------------

def softmax_naive(x: np.ndarray) -> np.ndarray:
    """exp(x) / sum exp(x) without subtracting the maximum ([T2] Exercise 2, naive_softmax).

    Overflows once a score exceeds ~709 in float64; used only on small scores.
    """
    e = np.exp(x)
    return e / e.sum(axis=-1, keepdims=True)


def softmax_safe(x: np.ndarray) -> np.ndarray:
    """Two-pass stable softmax: subtract the row maximum first ([T1] §2.1; [T2] Exercise 2)."""
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def softmax_online(x: np.ndarray) -> np.ndarray:
    """Element-wise online softmax ([T2] Exercise 2 online_softmax).

    One sweep keeps the running maximum m and the running sum l, shrinking l by
    exp(m_old - m_new) whenever the maximum grows; a second sweep writes
    exp(x - m) / l.  Pure-Python loops: small inputs only.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    for i in range(x.shape[0]):
        m, l = -math.inf, 0.0
        for xj in x[i]:
            m_new = max(m, float(xj))
            l = l * math.exp(m - m_new) + math.exp(float(xj) - m_new)
            m = m_new
        for j, xj in enumerate(x[i]):
            out[i, j] = math.exp(float(xj) - m) / l
    return out


# ----------------------------------------------------------------------------
# one query row ([T3] demo 1)
# ----------------------------------------------------------------------------

def _key_ranges(n: int, width: int) -> list[tuple[int, int]]:
    """Half-open key ranges [lo, hi) of `width` keys (the last one shorter) covering 0 .. n."""
    return [(lo, min(n, lo + width)) for lo in range(0, n, width)]


def _block_scores(q: np.ndarray, K: np.ndarray, lo: int, hi: int, scale: float) -> np.ndarray:
    """Scaled scores of one query against keys lo .. hi-1."""
    return scale * (K[lo:hi] @ q)


def attn_row_2pass(q: np.ndarray, K: np.ndarray, V: np.ndarray, block: int, scale: float) -> np.ndarray:
    """Two sweeps over the keys of one query ([T3] demo 1, the two-pass form).

    The first sweep only gathers the softmax statistics block by block (running maximum, and the
    running sum re-based whenever the maximum moves); the second sweep recomputes each block's
    scores and accumulates their normalised weights times V.
    """
    ranges = _key_ranges(K.shape[0], block)
    stat_m, stat_l = -math.inf, 0.0
    for lo, hi in ranges:
        s = _block_scores(q, K, lo, hi, scale)
        top = max(stat_m, float(np.max(s)))
        stat_l = stat_l * math.exp(stat_m - top) + float(np.sum(np.exp(s - top)))
        stat_m = top
    weighted = [np.exp(_block_scores(q, K, lo, hi, scale) - stat_m) @ V[lo:hi] for lo, hi in ranges]
    return np.sum(weighted, axis=0) / stat_l


def attn_row_1pass(q: np.ndarray, K: np.ndarray, V: np.ndarray, block: int, scale: float,
                   trace: list | None = None) -> np.ndarray:
    """One sweep over keys and values of one query ([T3] demo 1, the one-pass form).

    The state (m, l, o) is the running maximum, the running sum and the unnormalised output.  A
    block with scores s moves the maximum to m' = max(m, max s); the old sum and output are
    re-based by alpha = exp(m - m') before the block's weights exp(s - m') are added.  The
    division by l comes once, after the last block.  If `trace` is a list, one record
    (block index, block max, m', alpha, l) is appended per block.
    """
    state_m, state_l, state_o = -math.inf, 0.0, np.zeros(V.shape[1])
    for idx, (lo, hi) in enumerate(_key_ranges(K.shape[0], block)):
        s = _block_scores(q, K, lo, hi, scale)
        blk_max = float(np.max(s))
        moved = max(state_m, blk_max)
        alpha = math.exp(state_m - moved)
        w = np.exp(s - moved)
        state_o = state_o * alpha + w @ V[lo:hi]
        state_l = state_l * alpha + float(np.sum(w))
        state_m = moved
        if trace is not None:
            trace.append((idx, blk_max, moved, alpha, state_l))
    return state_o / state_l


# ----------------------------------------------------------------------------
# whole heads
# ----------------------------------------------------------------------------

def attention_tiled(Q: np.ndarray, K: np.ndarray, V: np.ndarray, Br: int, Bc: int, scale: float):
    """Q-outer / KV-inner tiling with running (m, l, O) and normalisation deferred to the end.

    ([T1] §2.3 and §3.1 pseudocode; [T4] §4 recurrence.)  Tiles may be ragged
    at the ends.  Returns (O, LSE).
    """
    nq, d = Q.shape
    nk = K.shape[0]
    O = np.empty((nq, V.shape[1]))
    lse = np.empty(nq)
    for i0 in range(0, nq, Br):
        q = Q[i0:i0 + Br]
        m = np.full(q.shape[0], -np.inf)
        l = np.zeros(q.shape[0])
        o = np.zeros((q.shape[0], V.shape[1]))
        for j0 in range(0, nk, Bc):
            s = (q @ K[j0:j0 + Bc].T) * scale
            m_new = np.maximum(m, s.max(axis=1))
            corr = np.exp(m - m_new)  # exp(-inf) = 0 on the first tile
            p = np.exp(s - m_new[:, None])
            l = corr * l + p.sum(axis=1)
            o = corr[:, None] * o + p @ V[j0:j0 + Bc]
            m = m_new
        O[i0:i0 + Br] = o / l[:, None]
        lse[i0:i0 + Br] = m + np.log(l)
    return O, lse


def attention_kv_outer(Q: np.ndarray, K: np.ndarray, V: np.ndarray, B: int, scale: float) -> np.ndarray:
    """KV-outer / Q-inner order with O renormalised at every step ([T2] Exercise 4, Algorithm 1).

    O_i <- O_i * (l_i exp(m_i - m_new) / l_new) + P_ij V_j / l_new, so O_i is a
    normalised average after every KV block.
    """
    nq = Q.shape[0]
    nk = K.shape[0]
    O = np.zeros((nq, V.shape[1]))
    l = np.zeros(nq)
    m = np.full(nq, -np.inf)
    for j0 in range(0, nk, B):
        k, v = K[j0:j0 + B], V[j0:j0 + B]
        for i0 in range(0, nq, B):
            sl = slice(i0, i0 + B)
            s = (Q[sl] @ k.T) * scale
            m_new = np.maximum(m[sl], s.max(axis=1))
            p = np.exp(s - m_new[:, None])
            l_new = l[sl] * np.exp(m[sl] - m_new) + p.sum(axis=1)
            alpha = l[sl] * np.exp(m[sl] - m_new) / l_new
            beta = 1.0 / l_new
            O[sl] = alpha[:, None] * O[sl] + beta[:, None] * (p @ v)
            l[sl] = l_new
            m[sl] = m_new
    return O


def attention_blocked_concat(Q: np.ndarray, K: np.ndarray, V: np.ndarray, B: int, scale: float) -> np.ndarray:
    """Score blocks S_ij concatenated into whole rows, then one softmax and P_i V ([T2] Exercise 3)."""
    nq = Q.shape[0]
    nk = K.shape[0]
    O = np.empty((nq, V.shape[1]))
    for i0 in range(0, nq, B):
        q = Q[i0:i0 + B]
        row = np.concatenate([(q @ K[j0:j0 + B].T) * scale for j0 in range(0, nk, B)], axis=1)
        O[i0:i0 + B] = softmax_safe(row) @ V
    return O


def attention_chunked_batched(Q: np.ndarray, K: np.ndarray, V: np.ndarray, q_chunks: int, k_chunks: int,
                              scale: float = 1.0) -> np.ndarray:
    """Batched chunked form over [b, N, d] with q_chunks x k_chunks equal chunks ([T4] §5).

    [T4] applies no 1/sqrt(d) factor (its scores are plain q.k); pass scale=1
    to reproduce it.  N must divide evenly by both chunk counts.
    """
    b, nq, d = Q.shape
    nk = K.shape[1]
    qs, ks = nq // q_chunks, nk // k_chunks
    outs = []
    for i in range(q_chunks):
        q = Q[:, i * qs:(i + 1) * qs]
        m_prev = np.full((b, qs), -np.inf)
        l_prev = np.zeros((b, qs))
        o_prev = np.zeros((b, qs, V.shape[-1]))
        for j in range(k_chunks):
            k = K[:, j * ks:(j + 1) * ks]
            v = V[:, j * ks:(j + 1) * ks]
            logits = np.einsum("nqd,nkd->nqk", q, k) * scale
            m_cur = np.maximum(m_prev, logits.max(axis=-1))
            e = np.exp(logits - m_cur[..., None])
            l_cur = l_prev * np.exp(m_prev - m_cur) + e.sum(axis=-1)
            o_cur = o_prev * np.exp(m_prev - m_cur)[..., None] + np.einsum("nqk,nkd->nqd", e, v)
            m_prev, l_prev, o_prev = m_cur, l_cur, o_cur
        outs.append(o_prev / l_prev[..., None])
    return np.concatenate(outs, axis=1)


def merge_tree(states: list, merge) -> tuple:
    """Pairwise (tree) reduction of partial states, like a parallel reduction ([T3] demo 2)."""
    sts = list(states)
    while len(sts) > 1:
        sts = [merge(sts[i], sts[i + 1]) if i + 1 < len(sts) else sts[i] for i in range(0, len(sts), 2)]
    return sts[0]


def merge_sequential(states: list, merge) -> tuple:
    """Left-to-right merge of partial states ([T3] demo 2)."""
    acc = states[0]
    for s in states[1:]:
        acc = merge(acc, s)
    return acc
