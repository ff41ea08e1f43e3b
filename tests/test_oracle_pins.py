"""Pins of the float64 oracle against what the pages and mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a 50-digit
brute force, closed forms, invariants, library routines, or the set-ups the
pages use.  Page titles:
  [T1] "FlashAttention 简化版：Tiling + Online Softmax"
  [T2] "Flash Attention 代码填空 (Level 2-3)"
  [T3] "CS349E 第 11 讲 01_online_softmax.py"
  [T4] "从零手写 FlashAttention（PyTorch实现 + 原理推导）"
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import forms


def _rand(rng, *shape, mult=1.0):
    return rng.standard_normal(shape) * mult


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("nq,nk,d,scale", [
    (1, 1, 1, 1.0), (3, 5, 4, 0.5), (16, 16, 8, 1 / math.sqrt(8)), (7, 13, 3, 1.7), (16, 11, 16, 0.25),
])
def test_brute_force_mpmath(nq, nk, d, scale):
    """No-max-subtraction softmax at 50 digits agrees with the float64 3-pass oracle ([T2] Ex. 2)."""
    brute = pytest.importorskip("oracle.brute")
    pytest.importorskip("mpmath")
    rng = np.random.default_rng(100 + nq * 31 + nk)
    q, k, v = _rand(rng, nq, d), _rand(rng, nk, d), _rand(rng, nk, d)
    o, lse = oracle.attention(q, k, v, scale)
    ob, lb = brute.attention_mp(q, k, v, scale)
    assert np.abs(o - ob).max() <= 1e-14
    assert np.abs(lse - lb).max() <= 1e-13


def test_large_scores_need_max_subtraction():
    """Scores near 800 overflow exp() in double unless the maximum is subtracted ([T1] §2.1)."""
    brute = pytest.importorskip("oracle.brute")
    pytest.importorskip("mpmath")
    rng = np.random.default_rng(7)
    q, k, v = _rand(rng, 4, 8, mult=10), _rand(rng, 6, 8, mult=10), _rand(rng, 6, 8)
    scale = 3.0
    s = scale * q @ k.T
    assert s.max() > 710  # exp would overflow without the subtraction
    o, lse = oracle.attention(q, k, v, scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    ob, lb = brute.attention_mp(q, k, v, scale)
    assert np.abs(o - ob).max() <= 1e-13
    assert np.abs(lse - lb).max() <= 1e-12 * np.abs(lb).max()


# ------------------------------------------------------------ closed forms

def test_probabilities_exposed_by_identity_values():
    """With V = I (d = Nk) the output is P itself: rows sum to 1 and match a library softmax."""
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    nq, nk = 9, 12
    q, k = _rand(rng, nq, nk), _rand(rng, nk, nk)
    P, _ = oracle.attention(q, k, np.eye(nk), 0.4)
    assert (P >= 0).all()
    assert np.abs(P.sum(axis=1) - 1).max() <= 1e-15
    assert np.abs(P - scipy_special.softmax(0.4 * q @ k.T, axis=1)).max() <= 1e-15


def test_single_key():
    """Nk = 1: O = v_0 and LSE = s_00."""
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 5, 6), _rand(rng, 1, 6), _rand(rng, 1, 6)
    o, lse = oracle.attention(q, k, v, 0.3)
    assert np.array_equal(o, np.broadcast_to(v, o.shape))
    assert np.abs(lse - 0.3 * (q @ k[0])).max() <= 1e-15


@pytest.mark.parametrize("zero", ["keys", "scale"])
def test_uniform_scores_average_values(zero):
    """All scores equal (K = 0 or scale = 0): O = mean of the V rows, LSE = ln Nk."""
    rng = np.random.default_rng(5)
    nk = 37
    q, k, v = _rand(rng, 4, 8), _rand(rng, nk, 8), _rand(rng, nk, 8)
    scale = 0.5
    if zero == "keys":
        k = np.zeros_like(k)
    else:
        scale = 0.0
    o, lse = oracle.attention(q, k, v, scale)
    assert np.abs(o - v.mean(axis=0)).max() <= 1e-15
    assert np.abs(lse - math.log(nk)).max() <= 1e-14


def test_constant_values():
    """V rows all equal to c: O = c whatever the scores."""
    rng = np.random.default_rng(6)
    c = _rand(rng, 8)
    v = np.tile(c, (20, 1))
    o, _ = oracle.attention(_rand(rng, 3, 8, mult=4), _rand(rng, 20, 8, mult=4), v, 1.0)
    assert np.abs(o - c).max() <= 1e-14


def test_permutation_invariances():
    """Permuting K/V rows together leaves O unchanged; permuting Q rows permutes O."""
    rng = np.random.default_rng(8)
    q, k, v = _rand(rng, 10, 16), _rand(rng, 30, 16), _rand(rng, 30, 16)
    o, lse = oracle.attention(q, k, v, 0.25)
    pk = rng.permutation(30)
    o2, lse2 = oracle.attention(q, k[pk], v[pk], 0.25)
    assert np.abs(o - o2).max() <= 1e-14 and np.abs(lse - lse2).max() <= 1e-14
    pq = rng.permutation(10)
    o3, lse3 = oracle.attention(q[pq], k, v, 0.25)
    assert np.array_equal(o3, o[pq]) and np.array_equal(lse3, lse[pq])


def test_library_sdpa_rectangular():
    """Non-square shapes (Nq != Nk != d) against torch's float64 SDPA: catches transposed operands."""
    rng = np.random.default_rng(9)
    q, k, v = _rand(rng, 2, 3, 7, 5), _rand(rng, 2, 3, 11, 5), _rand(rng, 2, 3, 11, 5)
    o, lse = oracle.attention(q, k, v, 0.7)
    t = [torch.tensor(x) for x in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, scale=0.7).numpy()
    assert np.abs(o - ref).max() <= 1e-14
    ref_lse = torch.logsumexp(0.7 * t[0] @ t[1].transpose(-1, -2), dim=-1).numpy()
    assert np.abs(lse - ref_lse).max() <= 1e-14


# ---------------------------------------------------------- page set-ups

def test_page_softmax_setup():
    """[T2] Exercise 2 set-up: torch.manual_seed(42); x = randn(4, 8) * 10, against torch.softmax.

    The oracle sees scores x through identity keys (q_i = x_i, K = I, scale 1)
    and exposes P through identity values.
    """
    torch.manual_seed(42)
    x = (torch.randn(4, 8) * 10).double()
    P, lse = oracle.attention(x.numpy(), np.eye(8), np.eye(8), 1.0)
    ref = torch.softmax(x, dim=-1).numpy()
    assert np.abs(P - ref).max() <= 1e-15
    assert np.abs(lse - torch.logsumexp(x, -1).numpy()).max() <= 1e-14
    assert np.abs(forms.softmax_safe(x.numpy()) - ref).max() <= 1e-15
    assert np.abs(forms.softmax_online(x.numpy()) - ref).max() <= 1e-15


def test_page_einsum_chunked_setup():
    """[T4] §1 and §5-6: (1, 12, 10) inputs, no 1/sqrt(d), q_chunks = 4, k_chunks = 3."""
    g = torch.Generator().manual_seed(1204)
    query, key, value = (torch.randn(1, 12, 10, generator=g, dtype=torch.float64) for _ in range(3))
    ref = torch.einsum("bqk,bkd->bqd", torch.softmax(torch.einsum("bqd,bkd->bqk", query, key), -1), value)
    o, _ = oracle.attention(query.numpy(), key.numpy(), value.numpy(), 1.0)
    assert np.abs(o - ref.numpy()).max() <= 1e-14
    oc = forms.attention_chunked_batched(query.numpy(), key.numpy(), value.numpy(), 4, 3, scale=1.0)
    assert np.abs(oc - o).max() <= 1e-14


def test_three_two_one_pass_rows():
    """[T3] demo 1 set-up (default_rng(0), S = 4096 keys, d = 64, blocks of 256): the three forms agree."""
    rng = np.random.default_rng(0)
    S, d, blk = 4096, 64, 256
    q = rng.standard_normal(d)
    K = rng.standard_normal((S, d))
    V = rng.standard_normal((S, d))
    sc = 1 / math.sqrt(d)
    ref, _ = oracle.attention(q[None], K, V, sc)
    ref = ref[0]
    assert np.abs(forms.attn_row_2pass(q, K, V, blk, sc) - ref).max() <= 1e-14
    trace = []
    assert np.abs(forms.attn_row_1pass(q, K, V, blk, sc, trace) - ref).max() <= 1e-14
    # alpha of block 0 is exp(-inf) = 0; alpha is exactly 1 whenever the maximum does not grow
    assert trace[0][3] == 0.0
    prev_m = trace[0][2]
    for _, blk_max, m_new, alpha, _ in trace[1:]:
        if blk_max <= prev_m:
            assert alpha == 1.0 and m_new == prev_m
        else:
            assert alpha < 1.0
        prev_m = m_new


def test_merge_order_invariance():
    """[T3] demo 2 set-up: S = 3000 scores x ~ 3 N(0,1), d = 32, 12 random segments; sequential,
    tree and shuffled merges all equal the one-shot result."""
    rng = np.random.default_rng(1)
    S, d = 3000, 32
    x = rng.standard_normal(S) * 3
    V = rng.standard_normal((S, d))
    one = np.zeros(d)
    one[0] = 1.0
    K = np.zeros((S, d))
    K[:, 0] = x  # scores s_j = <e_0, x_j e_0> = x_j with scale 1
    full, _ = oracle.attention(one[None], K, V, 1.0)
    full = full[0]
    cuts = np.sort(rng.choice(np.arange(1, S), size=11, replace=False))
    segs = np.split(np.arange(S), cuts)
    states = [oracle.partial_state(one, K[s], V[s], 1.0) for s in segs]
    perm = rng.permutation(len(states))
    for st in (forms.merge_sequential(states, oracle.merge_states),
               forms.merge_tree(states, oracle.merge_states),
               forms.merge_sequential([states[i] for i in perm], oracle.merge_states)):
        assert np.abs(oracle.finish(st) - full).max() <= 1e-14
    # one segment is the plain definition
    m, l, o = oracle.partial_state(one, K, V, 1.0)
    assert np.abs(o / l - full).max() <= 1e-14
    assert m == x.max()


def test_empty_state_is_identity():
    rng = np.random.default_rng(11)
    st = oracle.partial_state(_rand(rng, 8), _rand(rng, 5, 8), _rand(rng, 5, 8), 0.5)
    empty = oracle.partial_state(np.ones(8), np.zeros((0, 8)), np.zeros((0, 8)), 0.5)
    assert empty[0] == -math.inf and empty[1] == 0.0 and not empty[2].any()
    for merged in (oracle.merge_states(st, empty), oracle.merge_states(empty, st)):
        assert merged[0] == st[0] and merged[1] == st[1] and np.array_equal(merged[2], st[2])
    both = oracle.merge_states(empty, empty)
    assert both[0] == -math.inf and both[1] == 0.0


@pytest.mark.parametrize("nk,splits", [(32768 // 64, 16), (17, 16), (100, 7), (5, 5), (1, 1)])
def test_decode_split_equals_full(nk, splits):
    """Split-KV decode (ragged and empty chunks, seeded merge orders) equals exact attention."""
    rng = np.random.default_rng(nk + splits)
    B, H, d = 2, 3, 16
    q, k, v = _rand(rng, B, H, 1, d), _rand(rng, B, H, nk, d), _rand(rng, B, H, nk, d)
    full, full_lse = oracle.attention(q, k, v, 0.25)
    for order in (None, rng.permutation(splits)):
        o, lse = oracle.decode_splitkv(q, k, v, splits, 0.25, order)
        assert np.abs(o - full[:, :, 0]).max() <= 1e-14
        assert np.abs(lse - full_lse[:, :, 0]).max() <= 1e-13


def test_decode_rejects_bad_order():
    rng = np.random.default_rng(12)
    q, k, v = _rand(rng, 1, 4), _rand(rng, 1, 8, 4), _rand(rng, 1, 8, 4)
    with pytest.raises(ValueError):
        oracle.decode_splitkv(q, k, v, 4, 0.5, np.array([0, 1, 1, 3]))


# ---------------------------------------------------------- tiled forms

@pytest.mark.parametrize("nq,nk,Br,Bc", [(256, 256, 64, 64), (200, 333, 64, 48), (1, 17, 128, 128)])
def test_tiled_forms_agree(nq, nk, Br, Bc):
    """[T1] §3.1 Q-outer tiling with deferred normalisation, incl. ragged tiles."""
    rng = np.random.default_rng(nq * 7 + nk)
    d = 64
    q, k, v = _rand(rng, nq, d), _rand(rng, nk, d), _rand(rng, nk, d)
    ref, ref_lse = oracle.attention(q, k, v, 1 / 8)
    o, lse = forms.attention_tiled(q, k, v, Br, Bc, 1 / 8)
    assert np.abs(o - ref).max() <= 1e-14
    assert np.abs(lse - ref_lse).max() <= 1e-13


def test_algorithm1_and_blocked_forms():
    """[T2] Exercise 3 (N = 128, block 32) and Exercise 4 (N = 256, block 32), seed 42 set-ups."""
    torch.manual_seed(42)
    Q, K, V = (torch.randn(128, 64).double().numpy() for _ in range(3))
    ref, _ = oracle.attention(Q, K, V, 1 / 8)
    assert np.abs(forms.attention_blocked_concat(Q, K, V, 32, 1 / 8) - ref).max() <= 1e-14
    torch.manual_seed(42)
    Q, K, V = (torch.randn(256, 64).double().numpy() for _ in range(3))
    ref, _ = oracle.attention(Q, K, V, 1 / 8)
    assert np.abs(forms.attention_kv_outer(Q, K, V, 32, 1 / 8) - ref).max() <= 1e-14


def test_peaked_scores_tiled():
    """x3 peaked scores (maxima move often) through the tiled form with 128 x 128 tiles."""
    rng = np.random.default_rng(13)
    d = 128
    q, k, v = _rand(rng, 300, d, mult=3), _rand(rng, 700, d, mult=3), _rand(rng, 700, d)
    sc = 1 / math.sqrt(d)
    ref, ref_lse = oracle.attention(q, k, v, sc)
    o, lse = forms.attention_tiled(q, k, v, 128, 128, sc)
    assert np.abs(o - ref).max() <= 1e-13
    assert np.abs(lse - ref_lse).max() <= 1e-12


def test_grouped_query_heads_library():
    """Grouped-query attention (query head h reads key/value head h // group) against torch's
    float64 SDPA with enable_gqa, and Hkv = H reduces to plain multi-head attention."""
    rng = np.random.default_rng(14)
    q, k, v = _rand(rng, 2, 6, 5, 8), _rand(rng, 2, 2, 9, 8), _rand(rng, 2, 2, 9, 8)
    o, lse = oracle.attention(q, k, v, 0.3)
    t = [torch.tensor(x) for x in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, scale=0.3, enable_gqa=True).numpy()
    assert np.abs(o - ref).max() <= 1e-14
    o1, _ = oracle.attention(q[:, :3], k[:, :1].repeat(3, axis=1), v[:, :1].repeat(3, axis=1), 0.3)
    assert np.array_equal(o1, o[:, :3])


@pytest.mark.parametrize("nq,nk", [(9, 9), (5, 12), (1, 7)])
def test_causal_brute_force(nq, nk):
    """Causal mask aligned to the bottom-right corner (row i sees keys 0 .. i + Nk - Nq) against the
    50-digit brute force restricted to the same keys."""
    brute = pytest.importorskip("oracle.brute")
    pytest.importorskip("mpmath")
    rng = np.random.default_rng(nq * 10 + nk)
    q, k, v = _rand(rng, nq, 6), _rand(rng, nk, 6), _rand(rng, nk, 6)
    o, lse = oracle.attention(q[None, None], k[None, None], v[None, None], 0.4, causal=True)
    lim = oracle.causal_limits(np.arange(nq), nq, nk)
    ob, lb = brute.attention_mp(q, k, v, 0.4, limits=lim)
    assert np.abs(o[0, 0] - ob).max() <= 1e-14
    assert np.abs(lse[0, 0] - lb).max() <= 1e-13


def test_causal_library_and_closed_forms():
    """torch's float64 SDPA with is_causal (square case) and with an explicit bottom-right mask;
    with Nq == Nk the first row is v_0 with LSE = s_00 and the last row is unmasked attention."""
    rng = np.random.default_rng(15)
    q, k, v = _rand(rng, 2, 3, 10, 8), _rand(rng, 2, 3, 10, 8), _rand(rng, 2, 3, 10, 8)
    o, lse = oracle.attention(q, k, v, 0.3, causal=True)
    t = [torch.tensor(x) for x in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, scale=0.3, is_causal=True).numpy()
    assert np.abs(o - ref).max() <= 1e-14
    assert np.array_equal(o[:, :, 0], v[:, :, 0])
    assert np.abs(lse[:, :, 0] - 0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])).max() <= 1e-14
    full, _ = oracle.attention(q, k, v, 0.3)
    assert np.abs(o[:, :, -1] - full[:, :, -1]).max() <= 1e-15
    # Nq < Nk: bottom-right alignment through an explicit boolean mask
    q2 = _rand(rng, 1, 2, 4, 8)
    o2, _ = oracle.attention(q2, k[:1, :2], v[:1, :2], 0.3, causal=True)
    mask = torch.tensor(np.arange(10)[None, :] <= np.arange(4)[:, None] + 6)
    ref2 = torch.nn.functional.scaled_dot_product_attention(torch.tensor(q2), t[1][:1, :2], t[2][:1, :2], scale=0.3,
                                                            attn_mask=mask).numpy()
    assert np.abs(o2 - ref2).max() <= 1e-14
    # a subset of rows with their absolute indices gives the same rows
    o3, _ = oracle.attention(q[:, :, [2, 7]], k, v, 0.3, causal=True, rows=[2, 7], nq_total=10)
    assert np.array_equal(o3, o[:, :, [2, 7]])


@pytest.mark.parametrize("causal,hkv", [(False, 2), (True, 2), (False, 1), (True, 1)])
def test_backward_finite_differences(causal, hkv):
    """dQ, dK, dV against central differences of the loss L = sum(dO * O) through the oracle's own
    forward (causal mask and shared key/value heads included): checks every gradient without using
    its formulas."""
    rng = np.random.default_rng(16 + hkv + 2 * causal)
    H, nq, nk, d, sc = 2, 4, 6, 3, 0.7
    q, k, v, g = _rand(rng, 1, H, nq, d), _rand(rng, 1, hkv, nk, d), _rand(rng, 1, hkv, nk, d), _rand(rng, 1, H, nq, d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, sc, causal=causal)
    assert dk.shape == k.shape and dv.shape == v.shape

    def loss(qq, kk, vv):
        return float((oracle.attention(qq, kk, vv, sc, causal=causal)[0] * g).sum())

    h = 1e-6
    args = {"q": q, "k": k, "v": v}
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            lp = loss(*(xp if n == name else args[n] for n in ("q", "k", "v")))
            lm = loss(*(xm if n == name else args[n] for n in ("q", "k", "v")))
            num[idx] = (lp - lm) / (2 * h)
        assert np.abs(num - grad).max() <= 1e-8, name
    if causal:  # the last key is seen by the last query row only
        assert np.abs(dk[..., nk - 1, :]).max() > 0


def test_backward_autograd_library():
    """torch float64 autograd through SDPA on rectangular shapes (Nq != Nk != d)."""
    rng = np.random.default_rng(17)
    q, k, v, g = _rand(rng, 2, 3, 7, 5), _rand(rng, 2, 3, 11, 5), _rand(rng, 2, 3, 11, 5), _rand(rng, 2, 3, 7, 5)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, 0.45)
    t = [torch.tensor(x, requires_grad=True) for x in (q, k, v)]
    out = torch.nn.functional.scaled_dot_product_attention(*t, scale=0.45)
    out.backward(torch.tensor(g))
    for mine, ref in zip((dq, dk, dv), t):
        assert np.abs(mine - ref.grad.numpy()).max() <= 1e-13


def test_backward_page_dv_setup():
    """[T2] Exercise 5 set-up (seed 42, N=64, d=32, blocks of 16): dV recomputed block by block from the
    saved row max m and sum l, P_ij = exp(S_ij - m_i) / l_i, dV_j += P_ij^T dO_i, equals the oracle's dV."""
    torch.manual_seed(42)
    N, d, B = 64, 32, 16
    Q, K, V = (torch.randn(N, d).double() for _ in range(3))
    S = Q @ K.T / math.sqrt(d)
    dO = torch.randn(N, d).double()
    m = S.max(dim=-1, keepdim=True).values
    l = torch.exp(S - m).sum(dim=-1, keepdim=True)
    dV = torch.zeros(N, d, dtype=torch.float64)
    for j in range(0, N, B):
        for i in range(0, N, B):
            s_ij = Q[i:i + B] @ K[j:j + B].T / math.sqrt(d)
            p_ij = torch.exp(s_ij - m[i:i + B]) / l[i:i + B]
            dV[j:j + B] += p_ij.T @ dO[i:i + B]
    _, _, dv = oracle.attention_bwd(Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), 1 / math.sqrt(d))
    assert np.abs(dv - dV.numpy()).max() <= 1e-13
