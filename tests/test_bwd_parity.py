"""GPU parity of the backward pass (fa_bwd) against the float64 oracle's gradients.

The pages give dV_j += P_ij^T dO_i with P rebuilt from the saved row statistics ("Flash Attention
代码填空 (Level 2-3)", Exercise 5); dQ and dK follow from the chain rule.  Every case runs the
library's forward first, so the backward sees the O and LSE it would see in training.
"""
import math

import numpy as np
import pytest
import torch

import attention_forward_05_gb300 as fa
import oracle
from attention_forward_05_gb300.inputs import WORKLOADS, make_dout, make_qkv, workload_inputs
from parity import TOL_BWD, TOL_BWD_FP32, TOL_BWD_TF32_FWD, check_bwd

pytestmark = pytest.mark.gpu


def _run(q, k, v, dout, causal=False, scale=None):
    d = q.shape[-1]
    sc = 1 / math.sqrt(d) if scale is None else scale
    o, lse = fa.fa_fwd(q, k, v, scale=sc, causal=causal)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, dout, lse, scale=sc, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    return sc, o, lse, dq, dk, dv


SHAPES = [
    # B, H, Nq, Nk
    (1, 2, 128, 128),
    (1, 1, 200, 300),    # ragged query and key tails
    (2, 1, 256, 256),
    (1, 1, 77, 1000),
    (1, 1, 1, 64),       # one query row
    (1, 2, 300, 65),     # one key past a tile
    (1, 1, 513, 129),
    (1, 3, 130, 17),     # fewer keys than one tile
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bwd_shapes(cuda_device, d, shape):
    B, H, Nq, Nk = shape
    q, _, _ = make_qkv(B, H, Nq, 1, d, "bf16", seed=1100 + Nq + d, device=cuda_device)
    _, k, v = make_qkv(B, H, 1, Nk, d, "bf16", seed=1101 + Nk + d, device=cuda_device)
    dout = make_dout(B, H, Nq, d, "bf16", seed=1102 + Nq, device=cuda_device)
    sc, _, _, dq, dk, dv = _run(q, k, v, dout)
    check_bwd(q, k, v, dout, dq, dk, dv, sc, name=f"bwd d{d} {shape}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_single_key(cuda_device, dtype, d):
    """One key: every P is 1, so dS = dP - D = 0 exactly, dQ = dK = 0 and dV_0 = sum_i dO_i.  The oracle
    gives those exactly.  On the GPU, D comes from the stored O (V itself in bf16; V rounded to tf32,
    relative error <= 2^-11, on the fp32 path) and dP from V, each summed in fp32 in its own order, so
    |dS_i| <= eps * sum_c |dO_ic v_c| with eps = 4 d 2^-24 (+ 2^-11 for fp32), and
    |dQ_ic| <= scale |dS_i| |k_c|, |dK_c| <= scale sum_i |dS_i| |q_ic| (twice that, for the roundings of
    dS and of the stored gradients).  dV_0 = sum_i P_i dO_i with |P_i - 1| <= 16 u (1 + s_i) in bf16 and
    another 2^-10 s_i on the fp32 path (the LSE comes from tf32 products), s_i = scale sum_c |q_ic k_c|,
    plus the rounding of the stored dV (2^-9 relative in bf16)."""
    B, H, Nq, Nk = 1, 3, 5, 1
    q, k, v = make_qkv(B, H, Nq, Nk, d, dtype, seed=1480 + d, device=cuda_device)
    dout = make_dout(B, H, Nq, d, dtype, seed=1481 + d, device=cuda_device)
    sc = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd(q, k, v, scale=sc)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, dout, lse, scale=sc)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    qh, kh, vh, gh = (x.double().cpu() for x in (q, k, v, dout))
    eps = 4 * d * 2.0 ** -24 + (2.0 ** -11 if dtype == "fp32" else 0.0)
    ds_bound = eps * (gh.abs() * vh.abs()).sum(dim=-1, keepdim=True)  # [B, H, Nq, 1]
    dq_bound = 2 * sc * ds_bound * kh.abs()                               # [B, H, Nq, d]
    dk_bound = 2 * sc * (ds_bound * qh.abs()).sum(dim=2, keepdim=True)    # [B, H, 1, d]
    assert (dq.double().cpu().abs() <= dq_bound + 1e-30).all()
    assert (dk.double().cpu().abs() <= dk_bound + 1e-30).all()
    s_abs = sc * (qh.abs() * kh.abs()).sum(dim=-1, keepdim=True)                    # [B, H, Nq, 1]
    p_err = 16 * 2.0 ** -24 * (1 + s_abs) + (2.0 ** -10 * s_abs if dtype == "fp32" else 0.0)
    ref_dv = gh.sum(dim=2, keepdim=True)
    dv_bound = (p_err * gh.abs()).sum(dim=2, keepdim=True) + (2.0 ** -8 if dtype == "bf16" else 2.0 ** -22) * ref_dv.abs()
    assert ((dv.double().cpu() - ref_dv).abs() <= dv_bound + 1e-30).all()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", [(1, 2, 200, 200), (1, 1, 300, 1000), (1, 2, 513, 513), (1, 1, 1, 77)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bwd_causal(cuda_device, d, shape):
    B, H, Nq, Nk = shape
    q, _, _ = make_qkv(B, H, Nq, 1, d, "bf16", seed=1200 + Nq + d, device=cuda_device)
    _, k, v = make_qkv(B, H, 1, Nk, d, "bf16", seed=1201 + Nk + d, device=cuda_device)
    dout = make_dout(B, H, Nq, d, "bf16", seed=1202 + Nq, device=cuda_device)
    sc, _, _, dq, dk, dv = _run(q, k, v, dout, causal=True)
    check_bwd(q, k, v, dout, dq, dk, dv, sc, causal=True, name=f"bwd causal d{d} {shape}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cfg", [(2, 8, 2, 300, 400, 128), (1, 4, 1, 256, 256, 64)],
                         ids=lambda c: "B%dH%dHkv%dNq%dNk%dd%d" % c)
def test_bwd_grouped_query_heads(cuda_device, cfg, causal):
    """dK, dV of a shared key/value head sum over the query heads that read it."""
    B, H, Hkv, Nq, Nk, d = cfg
    q, _, _ = make_qkv(B, H, Nq, 1, d, "bf16", seed=1300 + H, device=cuda_device)
    _, k, v = make_qkv(B, Hkv, 1, Nk, d, "bf16", seed=1301 + Hkv, device=cuda_device)
    dout = make_dout(B, H, Nq, d, "bf16", seed=1302, device=cuda_device)
    sc, _, _, dq, dk, dv = _run(q, k, v, dout, causal=causal)
    check_bwd(q, k, v, dout, dq, dk, dv, sc, causal=causal, name=f"bwd gqa {cfg} causal={causal}")


def test_bwd_scales_and_peaked_scores(cuda_device):
    """Unscaled scores (scale 1) and peaked Q, K: P close to one-hot, dS concentrated."""
    q, k, v = make_qkv(1, 2, 256, 384, 64, "bf16", seed=1400, qk_mult=3.0, device=cuda_device)
    dout = make_dout(1, 2, 256, 64, "bf16", seed=1401, device=cuda_device)
    sc, _, _, dq, dk, dv = _run(q, k, v, dout)
    check_bwd(q, k, v, dout, dq, dk, dv, sc, name="bwd peaked")
    q, k, v = make_qkv(1, 1, 128, 128, 64, "bf16", seed=1402, qk_mult=0.3, device=cuda_device)
    dout = make_dout(1, 1, 128, 64, "bf16", seed=1403, device=cuda_device)
    sc, _, _, dq, dk, dv = _run(q, k, v, dout, scale=1.0)
    check_bwd(q, k, v, dout, dq, dk, dv, sc, name="bwd scale=1")


def test_bwd_deterministic_and_caller_workspace(cuda_device):
    """No atomics: repeated calls are bit-identical, with the library's or the caller's workspace."""
    q, k, v = make_qkv(2, 4, 700, 900, 64, "bf16", seed=1500, device=cuda_device)
    dout = make_dout(2, 4, 700, 64, "bf16", seed=1501, device=cuda_device)
    o, lse = fa.fa_fwd(q, k, v)
    a = fa.fa_bwd(q, k, v, o, dout, lse)
    nbytes = fa.fa_bwd_workspace_bytes(2, 4, 700, 64)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=cuda_device)
    b = fa.fa_bwd(q, k, v, o, dout, lse, workspace=ws)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    with pytest.raises(fa.FAError):
        fa.fa_bwd(q, k, v, o, dout, lse, workspace=ws[: nbytes - 256])


# ----------------------------------------------------------------- fp32 tensors
# The pages' backward exercise is written for fp32 tensors ("Flash Attention 代码填空 (Level 2-3)",
# Exercise 5).  These cases give the fp32 backward the oracle's own O and LSE (rounded to fp32), so
# that its arithmetic alone is compared with the oracle's gradients at fp32 tolerances.

def _run_fp32_oracle_stats(q, k, v, dout, causal=False, scale=None):
    d = q.shape[-1]
    sc = 1 / math.sqrt(d) if scale is None else scale
    ref_o, ref_lse = oracle.attention(q, k, v, sc, causal=causal)
    o = torch.from_numpy(ref_o).float().to(q.device)
    lse = torch.from_numpy(ref_lse).float().to(q.device)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, dout, lse, scale=sc, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    return sc, dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bwd_fp32_shapes(cuda_device, d, shape):
    B, H, Nq, Nk = shape
    q, _, _ = make_qkv(B, H, Nq, 1, d, "fp32", seed=1800 + Nq + d, device=cuda_device)
    _, k, v = make_qkv(B, H, 1, Nk, d, "fp32", seed=1801 + Nk + d, device=cuda_device)
    dout = make_dout(B, H, Nq, d, "fp32", seed=1802 + Nq, device=cuda_device)
    sc, dq, dk, dv = _run_fp32_oracle_stats(q, k, v, dout)
    assert dq.dtype == torch.float32
    check_bwd(q, k, v, dout, dq, dk, dv, sc, name=f"bwd fp32 d{d} {shape}", tol=TOL_BWD_FP32)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_fp32_causal_and_grouped_heads(cuda_device, d, causal):
    B, H, Hkv, Nq, Nk = 2, 4, 2, 300, 400
    q, _, _ = make_qkv(B, H, Nq, 1, d, "fp32", seed=1900 + d, device=cuda_device)
    _, k, v = make_qkv(B, Hkv, 1, Nk, d, "fp32", seed=1901 + d, device=cuda_device)
    dout = make_dout(B, H, Nq, d, "fp32", seed=1902, device=cuda_device)
    sc, dq, dk, dv = _run_fp32_oracle_stats(q, k, v, dout, causal=causal)
    check_bwd(q, k, v, dout, dq, dk, dv, sc, causal=causal, name=f"bwd fp32 gqa d{d} causal={causal}",
              tol=TOL_BWD_FP32)


def test_bwd_fp32_peaked_and_scale_one(cuda_device):
    q, k, v = make_qkv(1, 2, 256, 384, 64, "fp32", seed=1950, qk_mult=3.0, device=cuda_device)
    dout = make_dout(1, 2, 256, 64, "fp32", seed=1951, device=cuda_device)
    sc, dq, dk, dv = _run_fp32_oracle_stats(q, k, v, dout)
    check_bwd(q, k, v, dout, dq, dk, dv, sc, name="bwd fp32 peaked", tol=TOL_BWD_FP32)
    q, k, v = make_qkv(1, 1, 130, 70, 64, "fp32", seed=1952, qk_mult=0.3, device=cuda_device)
    dout = make_dout(1, 1, 130, 64, "fp32", seed=1953, device=cuda_device)
    sc, dq, dk, dv = _run_fp32_oracle_stats(q, k, v, dout, scale=1.0)
    check_bwd(q, k, v, dout, dq, dk, dv, sc, name="bwd fp32 scale=1", tol=TOL_BWD_FP32)


def test_bwd_fp32_after_library_forward_and_deterministic(cuda_device):
    """The training-step pipeline on fp32 tensors: fa_fwd (tf32 products) then fa_bwd; the gradients
    carry the forward's tf32 rounding through O and LSE.  Repeated calls are bit-identical."""
    w = WORKLOADS["long_fp32"]
    q, k, v = workload_inputs(w, device=cuda_device)
    dout = make_dout(w.B, w.H, w.Nq, w.d, "fp32", seed=1960, device=cuda_device)
    o, lse = fa.fa_fwd(q, k, v, scale=w.scale)
    a = fa.fa_bwd(q, k, v, o, dout, lse, scale=w.scale)
    b = fa.fa_bwd(q, k, v, o, dout, lse, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    check_bwd(q, k, v, dout, *a, w.scale, name="bwd fp32 after fwd, N=4096", tol=TOL_BWD_TF32_FWD)


def test_bwd_full_size_d64(cuda_device):
    """B=4 H=16 N=4096 d=64 (the multi-head prefill shape): two whole heads, the first and the
    last, against the oracle."""
    B, H, N, d = 4, 16, 4096, 64
    q, k, v = make_qkv(B, H, N, N, d, "bf16", seed=1003, device=cuda_device)
    dout = make_dout(B, H, N, d, "bf16", seed=1700, device=cuda_device)
    sc, _, _, dq, dk, dv = _run(q, k, v, dout)
    for b, h in ((0, 0), (B - 1, H - 1)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        check_bwd(q[sl], k[sl], v[sl], dout[sl], dq[sl], dk[sl], dv[sl], sc, name=f"bwd full d64 head ({b},{h})")


def test_bwd_full_size_d128_properties(cuda_device):
    """B=2 H=16 N=8192 d=128 with peaked scores: dQ on sampled rows against the oracle (a row's dQ
    needs only that row and all keys), and two identities that hold at any size:
    sum_j dV_j = sum_i dO_i (rows of P sum to 1) and sum_j dK_j = 0 (sum_j dS_ij = 0 for every i)."""
    B, H, N, d = 2, 16, 8192, 128
    q, k, v = make_qkv(B, H, N, N, d, "bf16", seed=1004, qk_mult=3.0, device=cuda_device)
    dout = make_dout(B, H, N, d, "bf16", seed=1701, device=cuda_device)
    sc, _, _, dq, dk, dv = _run(q, k, v, dout)
    rng = np.random.default_rng(1702)
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.choice(N, 12, replace=False)]))
    idx = torch.as_tensor(rows, device=cuda_device)
    for b, h in ((0, 0), (B - 1, H - 1)):
        qs = q[b:b + 1, h:h + 1, idx]
        ref_dq, _, _ = oracle.attention_bwd(qs, k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                            dout[b:b + 1, h:h + 1, idx], sc)
        got = dq[b:b + 1, h:h + 1, idx].float().cpu().numpy()
        err = np.abs(got - ref_dq)
        rel = err.max() / np.abs(ref_dq).max()
        print(f"[parity] bwd full d128 dq rows head ({b},{h}): max_rel={rel:.3e}")
        assert rel <= TOL_BWD["max_rel"]
    dv64 = dv.double().sum(dim=2)
    do64 = dout.double().sum(dim=2)
    e_v = ((dv64 - do64).abs().max() / dout.double().abs().sum(dim=2).max()).item()
    dk64 = dk.double().sum(dim=2)
    e_k = (dk64.abs().max() / dk.double().abs().sum(dim=2).max()).item()
    print(f"[parity] bwd full d128 identities: sum dV vs sum dO {e_v:.3e}, |sum dK| {e_k:.3e}")
    # each sum has 8192 terms, each carrying a relative rounding of about u = 2^-8
    assert e_v <= 2.0 ** -8 and e_k <= 2.0 ** -8


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_stream_order(cuda_device, d):
    """The three backward kernels overlap one another (programmatic dependent launches), but work
    enqueued after fa_bwd on the same stream still sees all three gradients complete: copies taken
    right after the call, with no synchronisation in between, equal the gradients read later."""
    B, H, N = 4, 16, 2048  # several waves of the dK/dV grid, so its tail overlaps the dQ grid
    q, k, v = make_qkv(B, H, N, N, d, "bf16", seed=1600 + d, device=cuda_device)
    dout = make_dout(B, H, N, d, "bf16", seed=1601 + d, device=cuda_device)
    o, lse = fa.fa_fwd(q, k, v)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        grads = fa.fa_bwd(q, k, v, o, dout, lse)
        early = [g.clone() for g in grads]  # enqueued right behind the dQ kernel
    torch.cuda.synchronize()
    assert fa.fa_check_device_error() == fa.FA_OK
    for name, g, e in zip(("dq", "dk", "dv"), grads, early):
        assert torch.equal(g, e), name
