"""Shared test helpers: tolerance rules and running the GPU path / oracle on
the same seeded inputs.

Tolerances (derived from the arithmetic, and the bar the op is held to):
  * bf16 outputs pass per element when |gpu - oracle| <= 2 bf16 ulp of the
    oracle value, or <= 1e-2 * |oracle|, or <= floor + 1 ulp, where the floor
    bounds the error of that element before its final bf16 rounding (which can
    add one more ulp):
      - R'     : floor = 2^-19 * (sum_j |comb[j][i] R[j][h]| + |post[i] Y[h]|)
                 (five fp32 roundings are at most ~5 * 2^-24 of that sum)
      - layer_in: floor = rstd * |gamma[h]| * sum_i |pre[i]| (ulp(R'[i][h]) + 2^-16 |R'[i][h]|)
                 The first term carries over the allowed 1-ulp difference of the
                 bf16 R' (the GPU rounds an fp32 sum, the oracle an fp64 one, so
                 an element on a rounding boundary may land on either side)
                 into X = sum_i pre[i] R'[i]; the second bounds the fp32
                 combine, the fp32 square sum over H and the fp32 mixes (each at
                 most ~1e-6 relative to that scale).
    The floor only matters where X is smaller than its terms.
  * fp32 mixes (pre, post, comb_res_mix) pass when |gpu - oracle| <= 1e-4.
"""
from __future__ import annotations

import numpy as np

from manifold_constrained_hyper_mhc_gb300 import synth

F = synth.bf16_bits_to_f32
MIX_ATOL = 1e-4


def ulp_bf16(w: np.ndarray) -> np.ndarray:
    a = np.abs(w)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    u = 2.0 ** (e - 7)
    return np.where(a > 0, u, 2.0 ** -133)


def bf16_check(got_bits, want_bits, floor):
    """Returns (n_bad, max_ulp, n_floor_only)."""
    g = F(got_bits).astype(np.float64)
    w = F(want_bits).astype(np.float64)
    d = np.abs(g - w)
    u = ulp_bf16(w)
    rel_ok = (d <= 2 * u) | (d <= 1e-2 * np.abs(w))
    ok = rel_ok | (d <= floor + u)
    return int((~ok).sum()), float((d / u).max()) if d.size else 0.0, int((ok & ~rel_ok).sum())


def residual_floor(R_bits, Y_bits, prev_post, prev_comb):
    R = np.abs(F(R_bits).astype(np.float64))            # [n,4,H]
    Y = np.abs(F(Y_bits).astype(np.float64))            # [n,H]
    S = np.einsum("nji,njh->nih", np.abs(prev_comb.astype(np.float64)), R)
    S += np.abs(prev_post.astype(np.float64))[:, :, None] * Y[:, None, :]
    return 2.0 ** -19 * S


def layer_in_floor(Rp_bits, pre, rstd, gamma_bits):
    Rp = np.abs(F(Rp_bits).astype(np.float64))
    S = np.einsum("ni,nih->nh", np.abs(pre), ulp_bf16(Rp) + 2.0 ** -16 * Rp)
    return rstd[:, None] * np.abs(F(gamma_bits).astype(np.float64))[None, :] * S


def compare_fused(gpu: dict, ref: dict, inputs, gamma, t0=0, label=""):
    """gpu: numpy outputs of the GPU call for tokens [t0, t0+n); ref: oracle dict
    (debug=True) for the same tokens; inputs = (R, Y, prev_post, prev_comb) of them."""
    R, Y, pp, pc = inputs
    msgs = []
    if "R" in ref and ref["R"] is not None and "residual_out" in gpu:
        nb, mu, nf = bf16_check(gpu["residual_out"], ref["R"], residual_floor(R, Y, pp, pc))
        if nb:
            msgs.append(f"{label} residual_out: {nb} elements out of tolerance (max {mu:.1f} ulp)")
    Rp = ref["R"] if ref.get("R") is not None else R
    nb, mu, nf = bf16_check(gpu["layer_in"], ref["X"], layer_in_floor(Rp, ref["pre"], ref["rstd"], gamma))
    if nb:
        msgs.append(f"{label} layer_in: {nb} elements out of tolerance (max {mu:.1f} ulp)")
    for k, rk in (("pre_mix", "pre"), ("post_mix", "post"), ("comb_res_mix", "res")):
        d = np.abs(gpu[k].astype(np.float64) - ref[rk]).max()
        if not d <= MIX_ATOL:
            msgs.append(f"{label} {k}: max abs error {d:.3g} > {MIX_ATOL}")
    return msgs
