"""Pins for the CPU oracle: closed forms, invariants, hand-derived worked
examples and special cases that reduce to a library routine.

Each test is chosen so that a plausible slip in the oracle (a transposed
operand, a wrong flattening, a dropped or misplaced eps, the wrong bias or
alpha slice, rows and columns swapped in Sinkhorn, a sum where a mean belongs)
makes it fail.  None of these tests re-types the oracle's own loop.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from manifold_constrained_hyper_mhc_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SC = synth.scalars()
B = synth.f32_to_bf16_bits
F = synth.bf16_bits_to_f32


def bf(x):
    return B(np.asarray(x, np.float32))


def _zeros_weights(H):
    return (np.zeros((4 * H, 24), np.float32), np.zeros(24, np.float32),
            np.array([0.01, 0.01, 0.01], np.float32), bf(np.ones(H)))


def _identity_comb(T):
    return np.broadcast_to(np.eye(4, dtype=np.float32), (T, 4, 4)).copy()


# ---------------------------------------------------------------- bf16 rounding

@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80), (-1.0, 0xBF80), (0.0, 0x0000), (-0.0, 0x8000),
    (1 + 2**-7, 0x3F81),            # exactly representable
    (1 + 2**-8, 0x3F80),            # tie -> even (down)
    (1 + 3 * 2**-8, 0x3F82),        # tie -> even (up)
    (1 + 2**-8 + 2**-30, 0x3F81),   # just above the tie -> up
    (2.0**-133, 0x0001),            # smallest subnormal
    (2.0**-134, 0x0000),            # tie between 0 and the smallest subnormal -> even (0)
    (3 * 2.0**-134, 0x0002),        # tie between 1 and 2 subnormal quanta -> even (2)
    (2.0**-126, 0x0080),            # smallest normal
    (3.3895313892515355e38, 0x7F7F),  # largest finite bf16
    (3.4e38, 0x7F80),               # rounds past the largest finite -> inf
    (math.inf, 0x7F80), (-math.inf, 0xFF80),
])
def test_bf16_rounding_bit_patterns(x, bits):
    assert oracle.double_to_bf16(x) == bits


def test_bf16_rounding_matches_torch_on_fp32_values():
    """For inputs that are fp32 values, the direct fp64->bf16 rounding must
    equal torch's fp32->bf16 round-to-nearest-even conversion."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10) ** rng.integers(-30, 30, 20000).astype(np.float32),
        (np.float32(1) + np.arange(4096, dtype=np.float32) * np.float32(2**-16)),
    ]).astype(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.double_to_bf16(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_bf16_widening_is_exact():
    for b in (0x3F80, 0x0001, 0x7F7F, 0xC2F7, 0x0080):
        u = np.array([b << 16], np.uint32).view(np.float32)[0]
        assert oracle.bf16_to_double(b) == float(u)


# ---------------------------------------------------------------- step (1): post

def test_post_permutation_comb_moves_streams():
    """comb[j][i] = 1 iff i = sigma(j) (a 4-cycle, not an involution) and post = 0:
    R'[sigma(j)] = R[j] bit for bit.  A transposed comb would apply sigma^-1."""
    rng = np.random.default_rng(1)
    T, H = 3, 40
    R = bf(rng.standard_normal((T, 4, H)))
    Y = bf(rng.standard_normal((T, H)))
    sigma = [1, 2, 3, 0]
    comb = np.zeros((T, 4, 4), np.float32)
    for j in range(4):
        comb[:, j, sigma[j]] = 1.0
    out = oracle.post(R, Y, np.zeros((T, 4), np.float32), comb)
    for j in range(4):
        np.testing.assert_array_equal(out[:, sigma[j]], R[:, j])


def test_post_layer_output_goes_to_the_indexed_stream():
    """comb = 0, post = 2 * e_i: R'[i] = 2 Y exactly and the other streams are 0."""
    rng = np.random.default_rng(2)
    T, H = 4, 24
    R = bf(rng.standard_normal((T, 4, H)))
    Y = bf(rng.standard_normal((T, H)))
    post = np.zeros((T, 4), np.float32)
    for t in range(T):
        post[t, t % 4] = 2.0
    out = oracle.post(R, Y, post, np.zeros((T, 4, 4), np.float32))
    for t in range(T):
        for i in range(4):
            if i == t % 4:
                np.testing.assert_array_equal(out[t, i], bf(2.0 * F(Y[t])))
            else:  # 0 * (negative) is -0: compare values, not bits
                np.testing.assert_array_equal(F(out[t, i]), 0.0)


def test_post_zero_layer_output_is_pure_residual_mix():
    """Y = 0: R' = comb^T R, the pure residual mix.  With small-integer streams and
    quarter-step weights the sums are exact in bf16, so a library einsum is the
    exact answer."""
    rng = np.random.default_rng(3)
    T, H = 5, 16
    Rf = rng.integers(-4, 5, (T, 4, H)).astype(np.float32)
    comb = rng.integers(0, 5, (T, 4, 4)).astype(np.float32) / 4
    post = rng.integers(0, 9, (T, 4)).astype(np.float32) / 4
    out = oracle.post(bf(Rf), np.zeros((T, H), np.uint16), post, comb)
    want = np.einsum("tji,tjh->tih", comb.astype(np.float64), Rf.astype(np.float64))
    np.testing.assert_array_equal(F(out).astype(np.float64), want)


# ---------------------------------------------------------------- step (3): Sinkhorn

def _golden_sinkhorn():
    with open(os.path.join(GOLDEN, "sinkhorn_worked_examples.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_sinkhorn(), ids=lambda c: c["name"])
def test_sinkhorn_hand_worked_examples(case):
    got = oracle.sinkhorn(case["M"], case["iters"], case["eps"])
    want = np.array([[float(Fraction(v)) for v in row] for row in case["expected"]])
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)


def test_sinkhorn_uniform_converges_to_closed_form():
    """Uniform logits with eps: the fixed point of x -> x / (4x + eps) is (1 - eps)/4."""
    eps = SC["sinkhorn_eps"]
    got = oracle.sinkhorn(np.full((4, 4), 7.5), 20, eps)
    np.testing.assert_allclose(got, (1 - eps) / 4, rtol=1e-14)


def test_sinkhorn_eps_enters_the_denominator():
    """One iteration on the all-ones matrix: rows give 1/(4+eps), then columns give
    1/(4 + 4 eps + eps^2)."""
    eps = 0.01
    got = oracle.sinkhorn(np.ones((4, 4)), 1, eps)
    np.testing.assert_allclose(got, 1.0 / (4 + 4 * eps + eps * eps), rtol=1e-15)


def test_sinkhorn_rank_one_is_exact_after_one_iteration():
    """eps = 0, M = u v^T: one row step leaves v / sum(v) in every row, one column
    step then leaves exactly 1/4 everywhere."""
    u = np.array([0.5, 2.0, 3.0, 7.0])
    v = np.array([1.0, 0.25, 4.0, 9.0])
    got = oracle.sinkhorn(np.outer(u, v), 1, 0.0)
    np.testing.assert_allclose(got, 0.25, rtol=1e-15)


def test_sinkhorn_invariants_on_random_matrices():
    """After the last column step the columns sum to S/(S+eps) < 1, the rows are within
    1e-3 of 1, all entries are positive; with eps = 0 columns sum to 1 exactly-ish."""
    rng = np.random.default_rng(4)
    eps = SC["sinkhorn_eps"]
    for _ in range(200):
        M = np.exp(rng.normal(0, 1.0, (4, 4)))
        out = oracle.sinkhorn(M, 20, eps)
        cs, rs = out.sum(0), out.sum(1)
        assert np.all(out > 0)
        assert np.all(cs < 1) and np.all(cs > 1 - 2 * eps)
        assert np.all(np.abs(rs - 1) < 1e-3)
        out0 = oracle.sinkhorn(M, 20, 0.0)
        np.testing.assert_allclose(out0.sum(0), 1.0, rtol=1e-14)


# ---------------------------------------------------------------- steps (2)-(3): RMS, projection, heads

def test_rms_and_projection_closed_form():
    """One token, comb = I, post = 0 so R' = R.  R' = a everywhere except
    R'[2][5] = v; phi has a single 1 at row k0 = 2*H + 5 (stream-major flattening),
    column 7.  Then r = 1/sqrt(((4H-1) a^2 + v^2)/(4H) + hc_norm_eps), z[7] = r v and
    every other logit is 0.  A stream/hidden-swapped flattening reads a instead of
    v, a sum instead of a mean or a misplaced eps changes r."""
    H = 8
    a, v = 2.0**-8, 0.5
    R = np.full((1, 4, H), a, np.float32)
    R[0, 2, 5] = v
    phi, bias, ms, gamma = _zeros_weights(H)
    phi[2 * H + 5, 7] = 1.0
    o = oracle.shifted_post_pre(bf(R), bf(np.zeros((1, H))), np.zeros((1, 4), np.float32),
                                _identity_comb(1), phi, bias, ms, gamma, **SC, debug=True)
    np.testing.assert_array_equal(o["R"], bf(R))
    K = 4 * H
    r = 1.0 / math.sqrt(((K - 1) * a * a + v * v) / K + SC["hc_norm_eps"])
    assert o["r"][0] == pytest.approx(r, rel=1e-15)
    want = np.zeros(24)
    want[7] = r * v
    np.testing.assert_allclose(o["z"][0], want, rtol=1e-15, atol=0)


def test_heads_and_alpha_slices_closed_form():
    """With z[1] = z[5] = z[9] = s known in closed form and distinct alphas
    (0.5, 2, 3): pre[1] = sigmoid(0.5 s + b1), post[1] = 1.25 sigmoid(2 s + b5),
    and the residual logit M[0][1] = 3 s (others 0) gives, after one eps-free
    Sinkhorn iteration, res[0][1] = q / (q + 3/4) with q = m/(3+m), m = exp(3 s)."""
    H = 8
    R = np.zeros((1, 4, H), np.float32)
    R[0, 0, 0] = 1.0
    phi, bias, _, gamma = _zeros_weights(H)
    for n in (1, 5, 9):
        phi[0, n] = 1.0
    bias[1], bias[5] = 0.3, -0.2
    ms = np.array([0.5, 2.0, 3.0], np.float32)
    sc = dict(SC, sinkhorn_iters=1, sinkhorn_eps=0.0)
    o = oracle.shifted_post_pre(bf(R), bf(np.zeros((1, H))), np.zeros((1, 4), np.float32),
                                _identity_comb(1), phi, bias, ms, gamma, **sc, debug=True)
    K = 4 * H
    s = 1.0 / math.sqrt(1.0 / K + SC["hc_norm_eps"])
    sig = lambda x: 1 / (1 + math.exp(-x))
    assert o["pre"][0, 1] == pytest.approx(sig(0.5 * s + float(np.float32(0.3))), rel=1e-14)
    assert o["pre"][0, 0] == pytest.approx(0.5, rel=1e-15)
    assert o["post"][0, 1] == pytest.approx(1.25 * sig(2.0 * s + float(np.float32(-0.2))), rel=1e-14)
    assert o["post"][0, 0] == pytest.approx(0.625, rel=1e-15)
    m = math.exp(3.0 * s)
    q = m / (3 + m)
    assert o["res"][0, 0, 1] == pytest.approx(q / (q + 0.75), rel=1e-13)
    assert o["res"][0, 1, 0] == pytest.approx(0.25 / (1 / (3 + m) + 0.75), rel=1e-13)


def test_zero_projection_gives_bias_only_heads():
    """phi = 0 so z = 0: pre = sigmoid(b[0:4]) and post = 1.25 sigmoid(b[4:8]) in
    closed form (b = ln 3 -> 3/4, b = -ln 3 -> 1/4, b = 0 -> 1/2), and the residual
    mix is Sinkhorn(exp(b[8:24])) reshaped row-major: with exp(b[8:24]) = M01 of
    the worked examples and one eps-free iteration the result is that example."""
    H = 16
    rng = np.random.default_rng(5)
    R = bf(rng.standard_normal((1, 4, H)))
    phi, _, ms, gamma = _zeros_weights(H)
    bias = np.zeros(24, np.float32)
    bias[0], bias[1], bias[4], bias[7] = math.log(3), -math.log(3), math.log(3), -math.log(3)
    bias[8 + 1] = math.log(3)   # M[0][1] = 3 in a row-major reshape
    sc = dict(SC, sinkhorn_iters=1, sinkhorn_eps=0.0)
    o = oracle.shifted_post_pre(R, bf(np.zeros((1, H))), np.zeros((1, 4), np.float32),
                                _identity_comb(1), phi, bias, ms, gamma, **sc)
    b32 = lambda x: float(np.float32(x))
    sig = lambda x: 1 / (1 + math.exp(-x))
    np.testing.assert_allclose(o["pre"][0], [sig(b32(math.log(3))), sig(b32(-math.log(3))), 0.5, 0.5], rtol=1e-15)
    np.testing.assert_allclose(o["post"][0], [1.25 * sig(b32(math.log(3))), 0.625, 0.625,
                                              1.25 * sig(b32(-math.log(3)))], rtol=1e-15)
    ex = {c["name"]: c for c in _golden_sinkhorn()}["M01_one_iteration"]
    want = np.array([[float(Fraction(v)) for v in row] for row in ex["expected"]])
    # exp(float32(ln 3)) is 3 up to float32 rounding of ln 3
    np.testing.assert_allclose(o["res"][0], want, rtol=1e-6)


def test_projection_matches_library_matmul():
    """The 24 logits are a plain matrix product of the flattened bf16 row with phi,
    scaled by r: check against numpy's fp64 matmul on random data."""
    rng = np.random.default_rng(6)
    T, H = 7, 72
    R = bf(rng.standard_normal((T, 4, H)))
    phi = (rng.standard_normal((4 * H, 24)) * 0.02).astype(np.float32)
    _, bias, ms, gamma = _zeros_weights(H)
    o = oracle.pre(R, phi, bias, ms, gamma, **SC, debug=True)
    flat = F(R).reshape(T, 4 * H).astype(np.float64)
    r = 1 / np.sqrt((flat ** 2).mean(1) + SC["hc_norm_eps"])
    np.testing.assert_allclose(o["r"], r, rtol=1e-13)
    np.testing.assert_allclose(o["z"], r[:, None] * (flat @ phi.astype(np.float64)), rtol=1e-11, atol=1e-14)


# ---------------------------------------------------------------- step (4): combine + RMSNorm

def test_identical_constant_streams_closed_form():
    """R' = a in every stream, phi = 0 so pre = sigmoid(b): X = a S with
    S = sum(pre), out = a S / sqrt(a^2 S^2 + rmsnorm_eps) * gamma (eps matters: a^2 S^2 ~ eps)."""
    H = 32
    a = 2.0**-10
    rng = np.random.default_rng(8)
    phi, _, ms, _ = _zeros_weights(H)
    bias = (rng.standard_normal(24) * 0.5).astype(np.float32)
    gamma = bf(1 + 0.1 * rng.standard_normal(H))
    R = bf(np.full((1, 4, H), a))
    o = oracle.pre(R, phi, bias, ms, gamma, **SC)
    S = sum(1 / (1 + math.exp(-float(bias[i]))) for i in range(4))
    want = a * S / math.sqrt((a * S) ** 2 + SC["rmsnorm_eps"]) * F(gamma).astype(np.float64)
    np.testing.assert_array_equal(o["X"][0], np.array([oracle.double_to_bf16(w) for w in want], np.uint16))


def test_combine_uses_the_indexed_pre_weight():
    """Stream 0 = 1 on even h, stream 1 = 1 on odd h, streams 2-3 = 0, phi = 0 with
    pre0 = 3/4 and pre1 = 1/2 (from the biases): X[even] = 3/4, X[odd] = 1/2 and
    mean X^2 = (9/16 + 1/4)/2.  Swapping pre indices swaps even and odd."""
    H = 16
    R = np.zeros((1, 4, H), np.float32)
    R[0, 0, 0::2] = 1.0
    R[0, 1, 1::2] = 1.0
    phi, _, ms, gamma = _zeros_weights(H)
    bias = np.zeros(24, np.float32)
    bias[0] = np.float32(math.log(3))
    o = oracle.pre(bf(R), phi, bias, ms, gamma, **SC)
    p0 = 1 / (1 + math.exp(-float(bias[0])))
    ms2 = (p0 ** 2 + 0.25) / 2
    want = np.where(np.arange(H) % 2 == 0, p0, 0.5) / math.sqrt(ms2 + SC["rmsnorm_eps"])
    np.testing.assert_array_equal(o["X"][0], np.array([oracle.double_to_bf16(w) for w in want], np.uint16))


def test_rmsnorm_matches_library_rms_norm():
    """With phi = 0 the pre weights are known (sigmoid of the biases), so the combine
    reduces to X = sum_i pre_i R'_i and the output to torch's fp64 rms_norm(X) * gamma."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    T, H = 6, 256
    R = bf(rng.standard_normal((T, 4, H)) * 3)
    phi, _, ms, _ = _zeros_weights(H)
    bias = (rng.standard_normal(24) * 0.5).astype(np.float32)
    gamma = bf(1 + 0.1 * rng.standard_normal(H))
    o = oracle.pre(R, phi, bias, ms, gamma, **SC)
    pre = torch.sigmoid(torch.from_numpy(bias[:4].astype(np.float64)))
    X = torch.einsum("i,tih->th", pre, torch.from_numpy(F(R).astype(np.float64)))
    want = torch.nn.functional.rms_norm(X, (H,), torch.from_numpy(F(gamma).astype(np.float64)),
                                        eps=SC["rmsnorm_eps"]).numpy()
    got = F(o["X"]).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(want))) - 7)
    assert np.all(np.abs(got - want) <= 0.5 * ulp * (1 + 1e-9))
    np.testing.assert_allclose(o["pre"], np.broadcast_to(pre.numpy(), (T, 4)), rtol=1e-15)


def test_zero_row():
    """R = Y = 0: R' = 0, z = 0, r = 1/sqrt(hc_norm_eps), X_out = 0, mixes from the biases."""
    H = 24
    rng = np.random.default_rng(10)
    phi = (rng.standard_normal((4 * H, 24)) * 0.02).astype(np.float32)
    _, _, ms, gamma = _zeros_weights(H)
    bias = np.zeros(24, np.float32)
    o = oracle.shifted_post_pre(np.zeros((2, 4, H), np.uint16), np.zeros((2, H), np.uint16),
                                np.ones((2, 4), np.float32), _identity_comb(2), phi, bias, ms,
                                gamma, **SC, debug=True)
    assert not o["R"].any() and not o["X"].any()
    np.testing.assert_array_equal(o["z"], 0.0)
    np.testing.assert_allclose(o["r"], 1 / math.sqrt(SC["hc_norm_eps"]), rtol=1e-15)
    np.testing.assert_allclose(o["pre"], 0.5, rtol=0)
    np.testing.assert_allclose(o["res"], (1 - SC["sinkhorn_eps"]) / 4, rtol=1e-14)


# ---------------------------------------------------------------- whole step

def test_scale_equivariance_exact():
    """With both eps set to 0, scaling R and Y by 2^5 scales R' by 2^5 bit for bit
    and leaves z, every mix and X_out bit-identical (powers of two are exact
    through sums, square roots and products)."""
    w = synth.Workload("pin", 3, 64, 11)
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)
    sc = dict(SC, hc_norm_eps=0.0, rmsnorm_eps=0.0)
    o1 = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **sc, debug=True)
    o2 = oracle.shifted_post_pre(bf(F(R) * 32), bf(F(Y) * 32), pp, pc, phi, bias, ms, gamma,
                                 **sc, debug=True)
    np.testing.assert_array_equal(F(o2["R"]), F(o1["R"]) * 32)
    for k in ("z", "pre", "post", "res", "X"):
        np.testing.assert_array_equal(o2[k], o1[k])


def test_fused_equals_post_then_pre():
    w = synth.WORKLOADS["tiny"]
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)
    o = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC)
    Rp = oracle.post(R, Y, pp, pc)
    q = oracle.pre(Rp, phi, bias, ms, gamma, **SC)
    np.testing.assert_array_equal(o["R"], Rp)
    for k in ("X", "pre", "post", "res"):
        np.testing.assert_array_equal(o[k], q[k])


def test_thread_split_does_not_change_results():
    w = synth.Workload("pin", 13, 128, 12)
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)
    o1 = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC, nthreads=1)
    o5 = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC, nthreads=5)
    for k in ("R", "X", "pre", "post", "res"):
        np.testing.assert_array_equal(o1[k], o5[k])


@pytest.mark.parametrize("a,b", [("hc_norm_eps", "rmsnorm_eps"), ("hc_norm_eps", "sinkhorn_eps"),
                                 ("hc_norm_eps", "hc_post_scale"), ("rmsnorm_eps", "sinkhorn_eps"),
                                 ("rmsnorm_eps", "hc_post_scale"), ("sinkhorn_eps", "hc_post_scale")])
def test_scalar_swap_changes_results(a, b):
    """The four scalars are pairwise distinct; swapping any two must change an output
    (each one is used where it belongs, and only there)."""
    w = synth.Workload("pin", 4, 64, 13, token_scale=True)
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)
    R = bf(F(R) * np.float32(0.003))  # small rows so both eps values matter
    Y = bf(F(Y) * np.float32(0.003))
    o = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC)
    sw = dict(SC)
    sw[a], sw[b] = SC[b], SC[a]
    q = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **sw)
    assert any(not np.array_equal(o[k], q[k]) for k in ("X", "pre", "post", "res"))


def test_synthetic_inputs_are_reproducible_by_block():
    w = synth.WORKLOADS["mid_batch"]
    R, Y, pp, pc = synth.tokens(w)
    R2, Y2, pp2, pc2 = synth.tokens(w, 37, 101)
    np.testing.assert_array_equal(R[37:101], R2)
    np.testing.assert_array_equal(pc[37:101], pc2)
    # Sinkhorn outputs (eps = 3e-4): columns sum to S / (S + eps), rows to 1 within 1e-3
    np.testing.assert_allclose(pc.sum(1), 1 - 3e-4, atol=1e-5)
    np.testing.assert_allclose(pc.sum(2), 1, atol=1e-3)
    assert np.all(pc > 0) and np.all((pp > 0) & (pp < 2))


# ---------------------------------------------------------------- MXFP8 quantize
# E4M3 facts from the format definition (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
# no infinities, S.1111.111 is NaN): largest finite S.1111.110 = 448, smallest normal
# S.0001.000 = 2^-6, largest subnormal S.0000.111 = 7/8 * 2^-6, smallest subnormal 2^-9.

E4M3_SPEC = [(448.0, 0x7E), (-448.0, 0xFE), (1.0, 0x38), (-1.0, 0xB8), (0.5, 0x30),
             (2.0 ** -6, 0x08), (7 * 2.0 ** -9, 0x07), (2.0 ** -9, 0x01), (256.0, 0x78),
             (1.125, 0x39), (240.0, 0x77), (0.0, 0x00), (-0.0, 0x80)]


@pytest.mark.parametrize("v,code", E4M3_SPEC)
def test_e4m3_spec_values(v, code):
    assert oracle.e4m3_encode(v) == code
    assert oracle.e4m3_decode(code) == v and math.copysign(1, oracle.e4m3_decode(code)) == math.copysign(1, v)


def test_e4m3_rounding_saturation_and_nan():
    # ties to even at the subnormal end: 2^-10 is half of the smallest subnormal
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(-(2.0 ** -10)) == 0x80
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02      # 1.5 quanta -> 2 (even)
    assert oracle.e4m3_encode(5 * 2.0 ** -10) == 0x02      # 2.5 quanta -> 2 (even)
    assert oracle.e4m3_encode(1.0625) == 0x38               # halfway 1 and 1.125 -> even (1)
    assert oracle.e4m3_encode(1.1875) == 0x3A               # halfway 1.125 and 1.25 -> 1.25
    # beyond the largest finite value: saturate, never NaN
    for v in (448.0001, 464.0, 480.0, 1e9, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E and oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_round_trip_and_nearest_even_brute_force():
    finite = [b for b in range(256) if b not in (0x7F, 0xFF)]
    for b in finite:
        assert oracle.e4m3_encode(oracle.e4m3_decode(b)) == b
    pos = sorted((oracle.e4m3_decode(b), b) for b in range(0x00, 0x7F))
    for (va, ba), (vb, bb) in zip(pos, pos[1:]):
        mid = (va + vb) / 2
        assert oracle.e4m3_encode(mid) == (ba if ba % 2 == 0 else bb)     # tie -> even code
        assert oracle.e4m3_encode(va + (vb - va) * 0.25) == ba
        assert oracle.e4m3_encode(va + (vb - va) * 0.75) == bb


@pytest.mark.parametrize("amax,e_floor,e_ceil", [
    (1.0, -8, -8), (1.75, -8, -8), (1.875, -8, -7), (448.0, 0, 0), (449.0, 0, 1),
    (2.0 ** -20, -28, -28), (3 * 2.0 ** 100, 93, 93), (3.75 * 2.0 ** 100, 93, 94)])
def test_mx_scale_exponent(amax, e_floor, e_ceil):
    # mode 0: E = floor(log2 amax) - 8; mode 1: smallest E with amax <= 448 * 2^E
    assert oracle.mx_scale_exp(amax, 0) == e_floor
    assert oracle.mx_scale_exp(amax, 1) == e_ceil
    assert amax <= 448 * 2.0 ** e_ceil and amax > 448 * 2.0 ** (e_ceil - 1)
    assert 2.0 ** (e_floor + 8) <= amax < 2.0 ** (e_floor + 9)


def test_mx_scale_exponent_zero_and_clamp():
    assert oracle.mx_scale_exp(0.0, 0) == -127 and oracle.mx_scale_exp(0.0, 1) == -127
    assert oracle.mx_scale_exp(2.0 ** -133, 0) == -127     # bf16's smallest subnormal


def test_mx_scale_tile_layout_is_a_bijection_with_contiguous_rows():
    T, H = 300, 7168 + 32 * 5                    # ragged rows and block columns
    rows, cols = oracle.mx_scale_shape(T, H)
    assert rows == 384 and cols == (H // 32 + 3) // 4 * 4
    seen = np.zeros(rows * cols, np.int32)
    for m in range(rows):
        for k in range(cols):
            seen[oracle.mx_scale_offset(m, k, H)] += 1
    assert np.all(seen == 1)
    # four consecutive blocks of one token are four consecutive bytes; tokens m and m + 32 of a
    # 128-row tile sit 4 bytes apart; each 128 x 4 tile is 512 contiguous bytes
    for m in (0, 37, 127, 255):
        base = oracle.mx_scale_offset(m, 8, H)
        assert [oracle.mx_scale_offset(m, 8 + j, H) for j in range(4)] == [base + j for j in range(4)]
    assert oracle.mx_scale_offset(32, 0, H) - oracle.mx_scale_offset(0, 0, H) == 4
    assert oracle.mx_scale_offset(1, 0, H) - oracle.mx_scale_offset(0, 0, H) == 16
    assert oracle.mx_scale_offset(0, 4, H) - oracle.mx_scale_offset(0, 0, H) == 512


@pytest.mark.parametrize("mode", [0, 1])
def test_mxfp8_quantize_decodes_back_within_half_a_quantum(mode):
    rng = np.random.default_rng(11)
    T, H = 5, 256
    mag = 10.0 ** rng.uniform(-3, 3, size=(T, H // 32, 1))
    X = bf(rng.standard_normal((T, H // 32, 32)) * mag).reshape(T, H)
    q, sc = oracle.mxfp8_quantize(X, mode)
    x = F(X).astype(np.float64)
    for t in range(T):
        for k in range(H // 32):
            blk = x[t, 32 * k:32 * k + 32]
            E = int(sc[oracle.mx_scale_offset(t, k, H)]) - 127
            assert E == oracle.mx_scale_exp(np.abs(blk).max(), mode)
            scaled = np.abs(blk) / 2.0 ** E
            if mode == 1:
                assert scaled.max() <= 448
            else:
                assert 256 <= scaled.max() < 512
            dec = np.array([oracle.e4m3_decode(b) for b in q[t, 32 * k:32 * k + 32]]) * 2.0 ** E
            for xv, dv, sv in zip(blk, dec, scaled):
                if sv > 448:
                    assert dv == math.copysign(448 * 2.0 ** E, xv)     # saturated
                    continue
                be = max(math.floor(math.log2(sv)) if sv > 0 else -6, -6)
                assert abs(dv - xv) <= 2.0 ** (E + be - 4) * (1 + 1e-12)   # half a quantum


# ---------------------------------------------------------------- post with int8 Y and square sum

def _post_inputs(T, H, seed):
    rng = np.random.default_rng(seed)
    R = bf(rng.standard_normal((T, 4, H)))
    pp = (2.0 / (1.0 + np.exp(-rng.standard_normal((T, 4))))).astype(np.float32)
    pc = rng.uniform(0.0, 0.5, (T, 4, 4)).astype(np.float32)
    return rng, R, pp, pc


def test_post_int8_reduces_to_the_bf16_post_when_q_times_scale_is_a_bf16_value():
    # x_scale a power of two and |q| < 128: q * s has at most 7 significant bits, so it is a bf16
    # value and the int8 post must equal the (pinned) bf16 post on Y = q * s bit for bit
    T, H = 5, 96
    rng, R, pp, pc = _post_inputs(T, H, 3)
    q = rng.integers(-127, 128, (T, H)).astype(np.int8)
    xs = (2.0 ** rng.integers(-12, 3, T)).astype(np.float32)
    Y = bf(q.astype(np.float64) * xs[:, None])
    assert np.array_equal(F(Y).astype(np.float64), q * xs[:, None].astype(np.float64))
    got, _ = oracle.post_ex(R, pp, pc, Yq=q, x_scales=xs)
    assert np.array_equal(got, oracle.post(R, Y, pp, pc))
    got_b, _ = oracle.post_ex(R, pp, pc, Y=Y)
    assert np.array_equal(got_b, got)


def test_post_square_sum_closed_forms():
    T, H = 4, 64
    rng, R, pp, pc = _post_inputs(T, H, 4)
    q = rng.integers(-127, 128, (T, H)).astype(np.int8)
    xs = rng.uniform(0.001, 0.1, T).astype(np.float32)
    # identity mix, zero post: R' = R, the square sum is that of R itself
    eye = _identity_comb(T)
    Rp, ss = oracle.post_ex(R, np.zeros((T, 4), np.float32), eye, Yq=q, x_scales=xs)
    assert np.array_equal(Rp, R)
    np.testing.assert_allclose(ss, (F(R).astype(np.float64) ** 2).sum(axis=(1, 2)), rtol=1e-13)
    # zero mix, unit post: every stream is bf16(q * s); the sum is 4 * sum_h bf16(q * s)^2
    Rp, ss = oracle.post_ex(R, np.ones((T, 4), np.float32), np.zeros((T, 4, 4), np.float32), Yq=q, x_scales=xs)
    y = F(bf(q.astype(np.float64) * xs[:, None].astype(np.float64))).astype(np.float64)
    for i in range(4):
        assert np.array_equal(F(Rp[:, i, :]).astype(np.float64), y)
    np.testing.assert_allclose(ss, 4 * (y ** 2).sum(axis=1), rtol=1e-13)


def test_post_square_sum_matches_the_pre_step_rms():
    # the pre step's r = 1/sqrt(ss/(4H) + eps) of the same R' (an independently pinned function)
    T, H = 3, 128
    rng, R, pp, pc = _post_inputs(T, H, 5)
    Y = bf(rng.standard_normal((T, H)))
    Rp, ss = oracle.post_ex(R, pp, pc, Y=Y)
    phi, bias, ms, gamma = _zeros_weights(H)
    out = oracle.pre(Rp, phi, bias, ms, gamma, **SC, debug=True)
    np.testing.assert_allclose(out["r"], 1.0 / np.sqrt(ss / (4 * H) + SC["hc_norm_eps"]), rtol=1e-13)


# ---------------------------------------------------------------- first-layer broadcast pre

def test_pre_broadcast_closed_forms():
    """Four copies of x: the mean of the 4H squares is the mean over H, and the flattened
    projection is x against the sum of phi's four row blocks, z = r * x @ (phi_0 + .. + phi_3).
    X = (sum_i pre_i) x, so the layer input is x * s / sqrt(mean (s x)^2 + eps) * gamma."""
    rng = np.random.default_rng(21)
    T, H = 4, 96
    x = bf(rng.standard_normal((T, H)))
    phi = (rng.standard_normal((4 * H, 24)) * 0.05).astype(np.float32)
    bias = (rng.standard_normal(24) * 0.1).astype(np.float32)
    ms = np.array([0.7, 0.4, 0.3], np.float32)
    gamma = bf(1.0 + 0.1 * rng.standard_normal(H))
    out = oracle.pre_broadcast(x, phi, bias, ms, gamma, **SC, debug=True)
    xd = F(x).astype(np.float64)
    r = 1.0 / np.sqrt((xd ** 2).mean(axis=1) + SC["hc_norm_eps"])
    np.testing.assert_allclose(out["r"], r, rtol=1e-13)
    phisum = phi.astype(np.float64).reshape(4, H, 24).sum(axis=0)
    np.testing.assert_allclose(out["z"], r[:, None] * (xd @ phisum), rtol=1e-10, atol=1e-13)
    s = out["pre"].sum(axis=1)
    X = s[:, None] * xd
    want = X / np.sqrt((X ** 2).mean(axis=1, keepdims=True) + SC["rmsnorm_eps"]) * F(gamma).astype(np.float64)
    got = F(out["X"]).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(want), 1e-30))) - 7)
    assert np.all(np.abs(got - want) <= ulp)     # one bf16 rounding of the same value
    assert np.array_equal(out["R"], np.repeat(x[:, None, :], 4, axis=1))


def test_prev_comb_table_is_the_scripts_output():
    """The generator's table of previous residual mixes is exactly what the committed script
    writes with the oracle's Sinkhorn (20 iterations of exp(N(0, 0.5)), eps 3e-4), and each
    matrix has the Sinkhorn invariants: positive, columns summing to S / (S + eps), rows to 1
    within 1e-3."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("mk", os.path.join(GOLDEN, "make_prev_comb_table.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    stored = synth.prev_comb_table()
    assert stored.shape == (1024, 4, 4) and stored.dtype == np.float32
    assert np.array_equal(stored, mk.table())
    assert (stored > 0).all()
    assert np.abs(stored.sum(axis=1) - (1 - 3e-4)).max() < 1e-5
    assert np.abs(stored.sum(axis=2) - 1).max() < 1e-3
    # the generator draws from it
    w = synth.WORKLOADS["tiny"]
    _, _, _, pc = synth.tokens(w)
    assert all(any(np.array_equal(m, t) for t in stored) for m in pc)


# ---------------------------------------------------------------- brute force, whole step

def _mp_round_bf16(mp, x):
    """x rounded to the nearest bf16 value (ties to even), computed in mpmath; also whether x
    lies so close to a midpoint that a correctly rounded fp64 intermediate could round the other
    way (such elements are left out of the exact comparison)."""
    if x == 0:
        return mp.mpf(0), False
    a = abs(x)
    e = int(mp.floor(mp.log(a, 2)))
    while a >= mp.mpf(2) ** (e + 1):
        e += 1
    while a < mp.mpf(2) ** e:
        e -= 1
    assert -126 <= e <= 127, "normal bf16 range only"
    ulp = mp.mpf(2) ** (e - 7)
    q = x / ulp
    n = mp.floor(q)
    frac = q - n
    if frac > mp.mpf(1) / 2 or (frac == mp.mpf(1) / 2 and int(n) % 2 == 1):
        n += 1
    near_tie = abs(frac - mp.mpf(1) / 2) < mp.mpf(10) ** -9
    return n * ulp, near_tie


def _mp_step(mp, R, Y, pp, pc, phi, bias, ms, gamma, sc):
    """The definition's four steps for one token, term by term at 50 digits: bf16 inputs widened
    exactly, R' and the layer input rounded to bf16, everything else unrounded."""
    H = Y.shape[0]
    f = lambda v: mp.mpf(float(v))
    Rm = [[f(F(np.uint16(R[j, h]))) for h in range(H)] for j in range(4)]
    Ym = [f(F(np.uint16(Y[h]))) for h in range(H)]
    Rp, Rp_tie = [[None] * H for _ in range(4)], [[False] * H for _ in range(4)]
    for i in range(4):
        for h in range(H):
            v = f(pp[i]) * Ym[h]
            for j in range(4):
                v += f(pc[j, i]) * Rm[j][h]
            Rp[i][h], Rp_tie[i][h] = _mp_round_bf16(mp, v)
    ss = mp.fsum(Rp[i][h] ** 2 for i in range(4) for h in range(H))
    r = 1 / mp.sqrt(ss / (4 * H) + f(sc["hc_norm_eps"]))
    z = [r * mp.fsum(Rp[i][h] * f(phi[i * H + h, n]) for i in range(4) for h in range(H)) for n in range(24)]
    pre = [1 / (1 + mp.exp(-(f(ms[0]) * z[i] + f(bias[i])))) for i in range(4)]
    post = [f(sc["hc_post_scale"]) / (1 + mp.exp(-(f(ms[1]) * z[4 + i] + f(bias[4 + i])))) for i in range(4)]
    M = [[mp.exp(f(ms[2]) * z[8 + 4 * a + c] + f(bias[8 + 4 * a + c])) for c in range(4)] for a in range(4)]
    eps = f(sc["sinkhorn_eps"])
    for _ in range(sc["sinkhorn_iters"]):
        for a in range(4):
            s = mp.fsum(M[a]) + eps
            M[a] = [m / s for m in M[a]]
        for c in range(4):
            s = mp.fsum(M[a][c] for a in range(4)) + eps
            for a in range(4):
                M[a][c] /= s
    X = [mp.fsum(pre[i] * Rp[i][h] for i in range(4)) for h in range(H)]
    rstd = 1 / mp.sqrt(mp.fsum(x * x for x in X) / H + f(sc["rmsnorm_eps"]))
    out, out_tie = zip(*[_mp_round_bf16(mp, X[h] * rstd * f(F(np.uint16(gamma[h])))) for h in range(H)])
    return dict(Rp=Rp, Rp_tie=Rp_tie, r=r, pre=pre, post=post, res=M, X=list(out), X_tie=list(out_tie), rstd=rstd)


@pytest.mark.parametrize("H,seed", [(8, 1), (8, 2), (16, 3), (16, 4)])
def test_whole_step_matches_a_50_digit_brute_force(H, seed):
    """The fp64 oracle against the step recomputed term by term in 50-digit arithmetic (mpmath),
    with its own bf16 rounding: R' and the layer input equal bit for bit (barring values within
    1e-9 of a bf16 midpoint, where the fp64 sum may round the other way), r, rstd and the mixes
    within 1e-12.  Nothing of the oracle's code is reused; the inputs have larger alphas than the
    workloads so that every logit moves its head."""
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 50
    rng = np.random.default_rng([seed, 99])
    R = bf(rng.standard_normal((1, 4, H)))
    Y = bf(rng.standard_normal((1, H)))
    pp = (2.0 / (1.0 + np.exp(-rng.standard_normal((1, 4))))).astype(np.float32)
    pc = synth.prev_comb_table()[rng.integers(0, 1024, size=1)]
    phi = (rng.standard_normal((4 * H, 24)) * 0.3).astype(np.float32)
    bias = (rng.standard_normal(24) * 0.1).astype(np.float32)
    ms = np.array([0.7, 0.5, 0.3], np.float32)
    gamma = bf(1.0 + 0.1 * rng.standard_normal(H))
    got = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC, debug=True)
    ref = _mp_step(mp, R[0], Y[0], pp[0], pc[0], phi, bias, ms, gamma, SC)
    ties = 0
    for i in range(4):
        for h in range(H):
            if ref["Rp_tie"][i][h]:
                ties += 1
                continue
            assert got["R"][0, i, h] == bf(float(ref["Rp"][i][h])), (i, h)
    for h in range(H):
        if ref["X_tie"][h]:
            ties += 1
            continue
        assert got["X"][0, h] == bf(float(ref["X"][h])), h
    assert ties <= 2
    assert abs(got["r"][0] - float(ref["r"])) <= 1e-12 * float(ref["r"])
    assert abs(got["rstd"][0] - float(ref["rstd"])) <= 1e-12 * float(ref["rstd"])
    assert np.abs(got["pre"][0] - np.array([float(v) for v in ref["pre"]])).max() <= 1e-12
    assert np.abs(got["post"][0] - np.array([float(v) for v in ref["post"]])).max() <= 1e-12
    assert np.abs(got["res"][0] - np.array([[float(v) for v in row] for row in ref["res"]])).max() <= 1e-12
