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
The full-size parity tests report, per output, the largest error in ulp, the 99.99th
percentile and the number of elements that pass by the floor alone (summarize()); with the
environment variable MHC_PARITY_REPORT set to a directory they also write it there as JSON.
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


def bf16_check(got_bits, want_bits, floor, stats=None):
    """Returns (n_bad, max_ulp, n_floor_only).  With a dict `stats`, also accumulates into it
    (over several calls, e.g. token chunks): n, n_bad, n_floor_only, max_ulp and a histogram of
    the error in ulp from which p9999_ulp() reads the 99.99th percentile."""
    g = F(got_bits).astype(np.float64)
    w = F(want_bits).astype(np.float64)
    d = np.abs(g - w)
    u = ulp_bf16(w)
    rel_ok = (d <= 2 * u) | (d <= 1e-2 * np.abs(w))
    ok = rel_ok | (d <= floor + u)
    n_bad, n_floor = int((~ok).sum()), int((ok & ~rel_ok).sum())
    e = d / u
    max_ulp = float(e.max()) if d.size else 0.0
    if stats is not None:
        stats["n"] = stats.get("n", 0) + int(d.size)
        stats["n_bad"] = stats.get("n_bad", 0) + n_bad
        stats["n_floor_only"] = stats.get("n_floor_only", 0) + n_floor
        stats["max_ulp"] = max(stats.get("max_ulp", 0.0), max_ulp)
        hist = stats.setdefault("hist", np.zeros(len(_ULP_EDGES) + 1, np.int64))
        hist += np.bincount(np.searchsorted(_ULP_EDGES, e.ravel(), side="right"), minlength=len(_ULP_EDGES) + 1)
    return n_bad, max_ulp, n_floor


# bins of the error histogram, in bf16 ulp of the oracle value
_ULP_EDGES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 8.0, 16.0, 64.0, 256.0, 4096.0])


def p9999_ulp(stats):
    """Upper edge of the histogram bin that holds the 99.99th percentile of the error (ulp)."""
    hist = stats["hist"]
    k = int(np.searchsorted(np.cumsum(hist), 0.9999 * hist.sum()))
    return float(_ULP_EDGES[k]) if k < len(_ULP_EDGES) else float("inf")


def summarize(report):
    """One line per output of a compare_fused report."""
    out = []
    for k, st in report.items():
        if "hist" in st:
            out.append(f"{k}: {st['n']} elements, max {st['max_ulp']:.2f} ulp, 99.99th pct <= "
                       f"{p9999_ulp(st):g} ulp, {st['n_floor_only']} pass by the floor only, {st['n_bad']} bad")
        else:
            out.append(f"{k}: max abs error {st['max_abs']:.3g}")
    return out


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


def compare_fused(gpu: dict, ref: dict, inputs, gamma, t0=0, label="", report=None):
    """gpu: numpy outputs of the GPU call for tokens [t0, t0+n); ref: oracle dict
    (debug=True) for the same tokens; inputs = (R, Y, prev_post, prev_comb) of them.
    With a dict `report`, per-output statistics accumulate into it (see bf16_check)."""
    R, Y, pp, pc = inputs
    msgs = []
    rep = report if report is not None else {}
    if "R" in ref and ref["R"] is not None and "residual_out" in gpu:
        nb, mu, nf = bf16_check(gpu["residual_out"], ref["R"], residual_floor(R, Y, pp, pc),
                                rep.setdefault("residual_out", {}))
        if nb:
            msgs.append(f"{label} residual_out: {nb} elements out of tolerance (max {mu:.1f} ulp)")
    Rp = ref["R"] if ref.get("R") is not None else R
    nb, mu, nf = bf16_check(gpu["layer_in"], ref["X"], layer_in_floor(Rp, ref["pre"], ref["rstd"], gamma),
                            rep.setdefault("layer_in", {}))
    if nb:
        msgs.append(f"{label} layer_in: {nb} elements out of tolerance (max {mu:.1f} ulp)")
    for k, rk in (("pre_mix", "pre"), ("post_mix", "post"), ("comb_res_mix", "res")):
        d = float(np.abs(gpu[k].astype(np.float64) - ref[rk]).max())
        st = rep.setdefault(k, {"max_abs": 0.0})
        st["max_abs"] = max(st["max_abs"], d)
        if not d <= MIX_ATOL:
            msgs.append(f"{label} {k}: max abs error {d:.3g} > {MIX_ATOL}")
    return msgs


def write_report(name, report):
    """Prints the summary and, if MHC_PARITY_REPORT names a directory, writes it as JSON."""
    import json
    import os
    lines = summarize(report)
    print(f"parity report {name}:\n  " + "\n  ".join(lines))
    d = os.environ.get("MHC_PARITY_REPORT")
    if d:
        os.makedirs(d, exist_ok=True)
        rec = {k: {kk: (p9999_ulp(v) if kk == "hist" else vv) for kk, vv in v.items()} for k, v in report.items()}
        for v in rec.values():
            if "hist" in v:
                v["p9999_ulp_at_most"] = v.pop("hist")
        with open(os.path.join(d, f"{name}.json"), "w") as f:
            json.dump(rec, f, indent=1)
    return lines
