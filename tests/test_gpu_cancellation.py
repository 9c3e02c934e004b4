"""Streams that cancel in the combined row X = sum_i pre_i R'_i.

The fused schedules take sum_h X^2 (the RMSNorm statistic of the combine, "[DSV4.1] Four BS=1
critical-path fixes for DSpark decode", "What changed" item 3) from the Gram matrix of the four
streams, pre^T G pre.  For anti-correlated streams with equal pre weights that is a small
difference of large terms, so the schedules flag such tokens and sum X^2 directly.  These inputs
(synth.cancellation_case) make pre_1 = pre_0 and pre_3 = pre_2 exactly and pair each stream
with a near negative of another, from exact cancellation down to independent streams.

Two checks per call: the oracle parity of the other tests, and -- since the layer-input floor
there grows with rstd, exactly where a wrong rstd would hide -- the RMS of layer_in / gamma per
token against the oracle's sqrt(ms / (ms + rmsnorm_eps)), ms = mean_h X^2, within 1e-2 (on
every token but those whose X is zero up to rounding).
"""
import numpy as np
import pytest

import oracle
from manifold_constrained_hyper_mhc_gb300 import synth

from _helpers import F, compare_fused

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
SC = synth.scalars()


@pytest.fixture(scope="module")
def mhc(mhc_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return mhc_lib


def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.cpu().numpy()


def unit_rms_errors(layer_in_bits, gamma_bits, rstd):
    """|RMS(layer_in / gamma) - sqrt(ms / (ms + eps))| per token, ms from the oracle's rstd."""
    x = F(layer_in_bits).astype(np.float64) / F(gamma_bits).astype(np.float64)[None, :]
    got = np.sqrt((x * x).mean(axis=1))
    want = np.sqrt(np.clip(1.0 - SC["rmsnorm_eps"] * rstd * rstd, 0.0, 1.0))
    return np.abs(got - want)


def run(mhc, T, H, schedule, via_pre=False, seed=0):
    R, Y, pp, pc, phi, bias, ms, gamma = synth.cancellation_case(T, H, 500 + seed + T + H)
    wd = (dev_f32(phi), dev_f32(bias), dev_f32(ms), dev_bf16(gamma))
    mhc.set_schedule(schedule)
    try:
        if via_pre:
            o = mhc.pre(dev_bf16(R), *wd, **SC)
        else:
            o = mhc.shifted_post_pre(dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd, **SC)
        torch.cuda.synchronize()
    finally:
        mhc.set_schedule("auto")
    got = {k: host(v) for k, v in o.items()}
    ref = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC, debug=True)
    if via_pre:
        ref["R"] = None  # the pre's residual is R itself (R' = R for these mixes)
    # R' = R exactly for these mixes (as values: an input -0 comes out +0, since 0 * Y is added)
    if not via_pre:
        assert np.array_equal(F(got["residual_out"]), F(R))
    msgs = compare_fused(got, ref, (R, Y, pp, pc), gamma, label=f"cancel {schedule} {T}x{H}")
    err = unit_rms_errors(got["layer_in"], gamma, ref["rstd"])
    # "exact" tokens: X is rounding noise of its terms on both sides, so their RMS is ~0 only
    # up to that noise; every other kind has X well above it
    err[np.arange(T) % len(synth.CANCEL_KINDS) == synth.CANCEL_KINDS.index("exact")] = 0.0
    worst = int(np.argmax(err))
    if err[worst] > 1e-2:
        msgs.append(f"unit RMS of layer_in/gamma off by {err[worst]:.3g} at token {worst} "
                    f"({synth.CANCEL_KINDS[worst % len(synth.CANCEL_KINDS)]})")
    assert not msgs, "\n".join(msgs)
    # the equal-weight construction holds on the GPU as well (equal phi columns and biases)
    pre = got["pre_mix"]
    assert np.abs(pre[:, 0] - pre[:, 1]).max() <= 1e-6 and np.abs(pre[:, 2] - pre[:, 3]).max() <= 1e-6


@pytest.mark.parametrize("schedule,T,H", [
    ("auto", 20, 7168), ("small", 20, 7168), ("small", 32, 1024), ("small", 96, 4096),
    ("ws", 20, 7168), ("ws", 200, 7168), ("ws", 130, 4096), ("ws", 45, 2056), ("auto", 300, 1024),
    ("split", 40, 7168), ("split", 17, 1000), ("tile", 40, 7168), ("tile", 33, 1088), ("auto", 2048, 7168)])
def test_cancelling_streams_fused(mhc, schedule, T, H):
    run(mhc, T, H, schedule)


@pytest.mark.parametrize("schedule,T,H", [("small", 15, 7168), ("ws", 64, 7168), ("split", 10, 4096), ("tile", 50, 4096),
                                          ("auto", 2100, 4096)])
def test_cancelling_streams_pre(mhc, schedule, T, H):
    run(mhc, T, H, schedule, via_pre=True)


def test_cancelling_streams_split_variant(mhc):
    """The side-stream variant: same bits as the fused call on the same inputs."""
    T, H = 16, 7168
    R, Y, pp, pc, phi, bias, ms, gamma = synth.cancellation_case(T, H, 77)
    args = (dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), dev_f32(phi), dev_f32(bias), dev_f32(ms),
            dev_bf16(gamma))
    side = torch.cuda.Stream()
    fork, join = torch.cuda.Event(), torch.cuda.Event()
    fork.record()
    join.record()
    a = mhc.shifted_post_pre(*args, **SC)
    b = mhc.shifted_post_pre_split(*args, **SC, side_stream=side, fork_event=fork, join_event=join)
    torch.cuda.current_stream().wait_event(join)
    torch.cuda.synchronize()
    for k in a:
        x, y = a[k], b[k]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), k


@pytest.mark.parametrize("schedule,T", [("ws", 100), ("small", 20)])
@pytest.mark.parametrize("want_bf16", [True, False])
def test_cancelling_streams_mxfp8(mhc, schedule, T, want_bf16):
    """The MXFP8 layer input of redone tokens: the codes and scales equal the oracle's quantize
    of the GPU's bf16 layer input of the plain call (with and without the bf16 output)."""
    H = 7168
    R, Y, pp, pc, phi, bias, ms, gamma = synth.cancellation_case(T, H, 88)
    args = (dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), dev_f32(phi), dev_f32(bias), dev_f32(ms),
            dev_bf16(gamma))
    mhc.set_schedule(schedule)
    try:
        plain = mhc.shifted_post_pre(*args, **SC)
        nsb = mhc.mxfp8_scale_bytes(T, H)
        mx = mhc.shifted_post_pre_mxfp8(*args, **SC, scale_mode=0, want_bf16=want_bf16,
                                        out={"layer_in_scales": torch.zeros(nsb, dtype=torch.uint8, device="cuda")})
        torch.cuda.synchronize()
    finally:
        mhc.set_schedule("auto")
    X = host(plain["layer_in"])
    q_ref, s_ref = oracle.mxfp8_quantize(X, 0)
    assert np.array_equal(mx["layer_in_fp8"].cpu().numpy(), q_ref)
    assert np.array_equal(mx["layer_in_scales"].cpu().numpy(), s_ref)
    if want_bf16:
        assert np.array_equal(host(mx["layer_in"]), X)


def test_cancelling_streams_repeat_on_one_workspace(mhc):
    """The redo flags are cleared by the call that set them: a second call on the same workspace
    with independent streams is as correct as on a fresh one."""
    T, H = 150, 7168
    ws = mhc.new_workspace(T, H)
    R, Y, pp, pc, phi, bias, ms, gamma = synth.cancellation_case(T, H, 99)
    args = (dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), dev_f32(phi), dev_f32(bias), dev_f32(ms),
            dev_bf16(gamma))
    mhc.shifted_post_pre(*args, **SC, workspace=ws)
    mhc.check_status(ws)
    w = synth.Workload("after_cancel", T, H, 98)
    phi2, bias2, ms2, gamma2 = synth.weights(w)
    R2, Y2, pp2, pc2 = synth.tokens(w)
    a2 = (dev_bf16(R2), dev_bf16(Y2), dev_f32(pp2), dev_f32(pc2), dev_f32(phi2), dev_f32(bias2), dev_f32(ms2),
          dev_bf16(gamma2))
    o_reused = mhc.shifted_post_pre(*a2, **SC, workspace=ws)
    o_fresh = mhc.shifted_post_pre(*a2, **SC)
    mhc.check_status(ws)
    torch.cuda.synchronize()
    for k in o_fresh:
        x, y = o_fresh[k], o_reused[k]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), k
