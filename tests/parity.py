"""Comparison helpers and tolerances for the GPU-vs-oracle parity tests.

Tolerances (absolute, on outputs of O(1) inputs), fixed by the build's target
and consistent with the pages' precision study ("CS349E 第 11 讲
01_online_softmax.py", demo 4: P in bf16 gives ~1e-3 relative error with
fp32 m, l and accumulators):
  fp32 inputs (TF32 products):  max |dO| <= 2e-3
  bf16 inputs:                  max |dO| <= 1.5e-2 and mean |dO| <= 2e-3
  LSE (both):                   max |dLSE| <= 1e-3
The oracle always runs on the exact bytes the GPU saw (bf16 up-cast exactly).

How the bf16 bound is applied.  O is stored in bf16, so even a correctly
rounded output sits up to half a bf16 step from the exact value: 0.0156 once
|O| >= 4, which is more than the 1.5e-2 bound itself (peaked scores put O close
to a single V row, and V rows reach |v| > 4).  Every bf16 check therefore
asserts two things, and reports the raw max |dO| beside them:
  * direct: |O_gpu - RNE_bf16(O_oracle)| <= 1.5e-2, the GPU's bf16 output
    against the oracle rounded to bf16 the way the kernel rounds.  Where one
    bf16 step is larger than 1.5e-2 (|O| >= 2) an output one step away from
    RNE_bf16(O_oracle) still passes: a kernel error of any size can put the
    two values on either side of a rounding boundary.
  * beyond the format: |O_gpu - O_oracle| - half_step(O_oracle) <= 1.5e-2.

How the fp32 LSE bound is applied.  Q and K are rounded to tf32 (unit
roundoff u = 2^-11) before the tensor core multiplies them, so one score is
off by about u |scale| sqrt(2/3 sum_i (q_i k_i)^2) (4e-4 for N(0,1) inputs at
d = 64 or 128 with scale 1/sqrt(d); at most 2u |scale| sum_i |q_i k_i|).  LSE
is a softmax-weighted mean of the scores, so these errors average out over the
keys a row sees: with n keys of similar weight the LSE error is about
4e-4 sqrt(e / n), and a bound of 1e-3 holds with a wide margin from n = 16 on.
Rows that see fewer than 16 keys (single-key shapes, the first rows under a
causal mask) are held to max(1e-3, the worst-case score bound); every other
row is held to 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {
    "fp32": dict(max_o=2e-3, mean_o=None, lse=1e-3),
    "bf16": dict(max_o=1.5e-2, mean_o=2e-3, lse=1e-3),
}


def dtype_name(t: torch.Tensor) -> str:
    return "bf16" if t.dtype == torch.bfloat16 else "fp32"


# Rows that see fewer keys than this are given the tf32 worst-case LSE bound (module docstring).
FEW_KEYS = 16


def sample_rows(Nq: int, n_random: int, seed: int, tile: int = 128) -> np.ndarray:
    """Seeded rows: the first and last row of every 128-row query tile (so every tile and CTA
    boundary), plus `n_random` random rows."""
    rng = np.random.default_rng(seed)
    n_t = (Nq + tile - 1) // tile
    tiles = range(n_t)
    rows = set()
    for t in tiles:
        rows.add(t * tile)
        rows.add(min(Nq - 1, t * tile + tile - 1))
    rows.update(rng.choice(Nq, size=min(n_random, Nq), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def check_fwd(q, k, v, o, lse, scale: float, rows=None, name: str = "", causal: bool = False) -> dict:
    """Compares GPU outputs (o, lse) with the oracle on all rows or on `rows`; asserts the tolerances."""
    dt = dtype_name(q)
    if rows is None:
        qs, og, lg = q, o, lse
    else:
        idx = torch.as_tensor(rows, device=q.device)
        qs, og = q[:, :, idx], o[:, :, idx]
        lg = lse[:, :, idx] if lse is not None else None
    ref_o, ref_lse = oracle.attention(qs, k, v, scale, causal=causal, rows=rows, nq_total=q.shape[2])
    got = og.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), f"{name}: non-finite output"
    tol = TOL[dt]
    if dt == "bf16":
        res = check_bf16_output(got, ref_o, name)
    else:
        err = np.abs(got - ref_o)
        res = dict(max_o=float(err.max()), mean_o=float(err.mean()))
        assert res["max_o"] <= tol["max_o"], f"{name}: max|dO| {res['max_o']:.3e} > {tol['max_o']}"
    if lg is not None:
        le = np.abs(lg.cpu().numpy().astype(np.float64) - ref_lse)
        res["lse"] = float(le.max())
        lse_tol = np.full(le.shape, tol["lse"])
        if dt == "fp32":
            row_ids = np.arange(q.shape[2]) if rows is None else np.asarray(rows)
            nk = k.shape[2]
            seen = np.minimum(nk, row_ids + 1 + nk - q.shape[2]) if causal else np.full(row_ids.shape, nk)
            few = (seen < FEW_KEYS)[None, None, :]
            lse_tol = np.where(few, np.maximum(lse_tol, tf32_score_bound(qs, k, scale)), lse_tol)
            res["lse_rows_few_keys"] = float(few.sum())
            rest = le[np.broadcast_to(~few, le.shape)]
            if rest.size:
                res["lse_many_keys"] = float(rest.max())
        assert (le <= lse_tol).all(), f"{name}: max|dLSE| {res['lse']:.3e} above its bound"
    print(f"[parity] {name}: " + " ".join(f"{k}={v:.3e}" for k, v in res.items()))
    return res


def rne_bf16(x: np.ndarray) -> np.ndarray:
    """float64 values rounded to the nearest bf16 value (8 significant bits), ties to even."""
    mant, ex = np.frexp(x)  # x = mant * 2^ex with 0.5 <= |mant| < 1
    step = np.exp2(np.maximum(ex, -125) - 8.0)
    return np.round(x / step) * step  # np.round rounds halves to even


def bf16_step(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x|: 2^(floor(log2|x|) - 7)."""
    return 2.0 * bf16_half_step(x)


def check_bf16_output(got: np.ndarray, ref: np.ndarray, name: str) -> dict:
    """bf16 outputs against float64 oracle values: the direct and the beyond-format bound of the module
    docstring, and the mean bound; returns the raw and direct figures."""
    tol = TOL["bf16"]
    err = np.abs(got - ref)
    direct = np.abs(got - rne_bf16(ref))
    beyond = err - bf16_half_step(ref)
    res = dict(max_o=float(err.max()), mean_o=float(err.mean()), max_o_vs_rne=float(direct.max()),
               max_o_beyond_format=float(beyond.max()))
    ok_direct = direct <= np.maximum(tol["max_o"], bf16_step(ref) * 1.0000001)
    assert ok_direct.all(), f"{name}: |O - RNE(O_ref)| up to {res['max_o_vs_rne']:.3e} above {tol['max_o']}"
    assert res["max_o_beyond_format"] <= tol["max_o"], \
        f"{name}: max|dO| {res['max_o']:.3e} ({res['max_o_beyond_format']:.3e} beyond bf16 rounding) > {tol['max_o']}"
    assert res["mean_o"] <= tol["mean_o"], f"{name}: mean|dO| {res['mean_o']:.3e} > {tol['mean_o']}"
    return res


def bf16_half_step(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits): 2^(floor(log2|x|) - 8)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 8)


def tf32_score_bound(q, k, scale: float) -> np.ndarray:
    """Per query row, max over keys of 2u |scale| sum_i |q_i k_i| with u = 2^-11 (tf32 rounding of q and k)."""
    qa = np.abs(q.float().cpu().numpy().astype(np.float64))
    ka = np.abs(k.float().cpu().numpy().astype(np.float64))
    if ka.shape[1] != qa.shape[1]:  # grouped-query heads
        ka = np.repeat(ka, qa.shape[1] // ka.shape[1], axis=1)
    per_key = np.einsum("bhqd,bhkd->bhqk", qa, ka)
    return 2.0 * 2.0 ** -11 * abs(scale) * per_key.max(axis=-1) * 1.001


def check_decode(q, k, v, o, lse, scale: float, splits: int, order=None, heads=None, name: str = "") -> dict:
    """Decode outputs o [B,H,d] (and lse [B,H]) against the oracle's split-and-merge in the same order.

    `heads` optionally restricts the check to a list of flat (b*H + h) indices.
    """
    B, H, Nk, d = k.shape
    qf = q.reshape(B * H, d)
    kf, vf = k.reshape(B * H, Nk, d), v.reshape(B * H, Nk, d)
    of = o.reshape(B * H, d)
    lf = lse.reshape(B * H) if lse is not None else None
    if heads is not None:
        idx = torch.as_tensor(heads, device=k.device)
        qf, kf, vf, of = qf[idx], kf[idx], vf[idx], of[idx]
        lf = lf[idx] if lf is not None else None
    ref_o, ref_lse = oracle.decode_splitkv(qf, kf, vf, splits, scale, order)
    got = of.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), f"{name}: non-finite output"
    tol = TOL["bf16"]
    res = check_bf16_output(got, ref_o, name)
    if lf is not None:
        le = np.abs(lf.cpu().numpy().astype(np.float64) - ref_lse)
        res["lse"] = float(le.max())
        assert res["lse"] <= tol["lse"], f"{name}: max|dLSE| {res['lse']:.3e}"
    print(f"[parity] {name}: " + " ".join(f"{k}={v:.3e}" for k, v in res.items()))
    return res


# Backward tolerances, relative to the size of each gradient tensor (no bound is fixed for the
# backward elsewhere, so these are derived from its arithmetic).  With bf16 unit roundoff
# u = 2^-8, every term of dV = P^T dO carries the rounding of P (u) and the output carries one more
# (u); dQ and dK add the rounding of dS (u) and the error of D = rowsum(dO * O), which is computed
# from the bf16-rounded forward output (u per term).  A term-wise worst case is therefore about
# 4u = 1.6e-2 of the largest |gradient| element.  The mean error is about 0.6u for diffuse P; when P
# is concentrated on one key, dP_ij - D_i cancels and the rounding of O in D dominates dS, which
# raises the mean error of dQ and dK to about 1.6u (a CPU emulation of the same roundings gives the
# same figure, and it falls back to 0.6u when O is not rounded).  The mean bound is 2u.
TOL_BWD = dict(max_rel=4 * 2.0 ** -8, mean_rel=2 * 2.0 ** -8)


# fp32 backward (fp32 products and sums on the CUDA cores), fed the oracle's own O and LSE so that
# only its arithmetic is measured.  With u = 2^-24, one score carries at most d u |scale| sum_c |q_c k_c|
# of rounding (the dot-product bound), 2e-5 at d = 64 and 5.5e-5 at d = 128 for N(0,1) inputs (about
# 1e-6 typically, the rounding errors being independent), and ex2.approx adds about 2^-22 relative
# to P.  Gradients inherit that relative error through P and dS; the bounds leave a margin of about 2
# over the worst case for the maximum and about 10 over the typical case for the mean.
TOL_BWD_FP32 = dict(max_rel=1e-4, mean_rel=1e-5)
# fp32 backward after the library's fp32-in forward: O and LSE then carry the forward's tf32 products
# (u = 2^-11), which P and D inherit; the bf16 reasoning above with u = 2^-11 gives these bounds.
TOL_BWD_TF32_FWD = dict(max_rel=4 * 2.0 ** -11, mean_rel=2 * 2.0 ** -11)


def check_bwd(q, k, v, dout, dq, dk, dv, scale: float, causal: bool = False, name: str = "", tol=None) -> dict:
    """GPU gradients against the oracle's float64 gradients on the same input bytes.

    For each of dQ, dK, dV: max|err| / max|ref| <= tol['max_rel'] and
    mean|err| / mean|ref| <= tol['mean_rel'] (tol defaults to TOL_BWD).
    """
    tol = TOL_BWD if tol is None else tol
    ref = oracle.attention_bwd(q, k, v, dout, scale, causal=causal)
    res = {}
    for nm, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = got.float().cpu().numpy().astype(np.float64)
        assert g.shape == r.shape, f"{name}: {nm} shape {g.shape} vs {r.shape}"
        assert np.isfinite(g).all(), f"{name}: non-finite {nm}"
        err = np.abs(g - r)
        res[nm + "_max_rel"] = float(err.max() / max(np.abs(r).max(), 1e-30))
        res[nm + "_mean_rel"] = float(err.mean() / max(np.abs(r).mean(), 1e-30))
    print(f"[parity] {name}: " + " ".join(f"{k}={v:.3e}" for k, v in res.items()))
    for nm in ("dq", "dk", "dv"):
        assert res[nm + "_max_rel"] <= tol["max_rel"], f"{name}: {nm} max rel err {res[nm + '_max_rel']:.3e}"
        assert res[nm + "_mean_rel"] <= tol["mean_rel"], f"{name}: {nm} mean rel err {res[nm + '_mean_rel']:.3e}"
    return res
