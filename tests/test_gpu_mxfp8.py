"""GPU parity of the MXFP8 layer-input epilogue (mhc_shifted_post_pre_mxfp8).

The pages' test compares the fused epilogue with the bf16 output followed by the separate
quantize: bf16 output, E4M3 values and swizzled UE8M0 scales all equal.  Here the oracle's
quantize of the GPU's own bf16 layer input must match the GPU's E4M3 codes and scale bytes
bit for bit; the bf16 output and the mixes must equal the plain call's on the same
schedule bit for bit (and the plain call is held to the oracle by test_gpu_parity)."""
import numpy as np
import pytest

import oracle
from manifold_constrained_hyper_mhc_gb300 import synth

from _helpers import compare_fused

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


def host_bf16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def decade_gamma(H, seed):
    """gamma with a magnitude of 10^U(-2.5, 2.5) per block of 32: the blocks' scales span five
    decades, as in the pages' test."""
    rng = np.random.default_rng(seed)
    mag = 10.0 ** rng.uniform(-2.5, 2.5, size=H // 32)
    g = np.repeat(mag, 32) * (1.0 + 0.1 * rng.standard_normal(H))
    return synth.f32_to_bf16_bits(g.astype(np.float32))


def run_case(mhc, w, schedule, mode, gamma_decades=True, check_oracle=True):
    phi, bias, ms, gamma = synth.weights(w)
    if gamma_decades:
        gamma = decade_gamma(w.H, w.seed + 77)
    R, Y, pp, pc = synth.tokens(w)
    args = (dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), dev_f32(phi), dev_f32(bias), dev_f32(ms),
            dev_bf16(gamma))
    mhc.set_schedule(schedule)
    try:
        nsb = mhc.mxfp8_scale_bytes(w.T, w.H)
        zeros = lambda: {"layer_in_scales": torch.zeros(nsb, dtype=torch.uint8, device="cuda")}  # padding stays 0
        plain = mhc.shifted_post_pre(*args, **SC)
        mx = mhc.shifted_post_pre_mxfp8(*args, **SC, scale_mode=mode, out=zeros())
        mx_only = mhc.shifted_post_pre_mxfp8(*args, **SC, scale_mode=mode, want_bf16=False, out=zeros())
        torch.cuda.synchronize()
    finally:
        mhc.set_schedule("auto")
    for k in ("residual_out", "layer_in", "pre_mix", "post_mix", "comb_res_mix"):
        a, b = plain[k], mx[k]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), k
    X = host_bf16(mx["layer_in"])
    q_ref, s_ref = oracle.mxfp8_quantize(X, mode)
    q = mx["layer_in_fp8"].cpu().numpy()
    s = mx["layer_in_scales"].cpu().numpy()
    assert s.shape == s_ref.shape
    bad_q = int((q != q_ref).sum())
    bad_s = int((s != s_ref).sum())
    assert bad_q == 0 and bad_s == 0, f"{bad_q} E4M3 codes and {bad_s} scale bytes differ"
    assert np.array_equal(mx_only["layer_in_fp8"].cpu().numpy(), q)
    assert np.array_equal(mx_only["layer_in_scales"].cpu().numpy(), s)
    if not check_oracle:
        return
    # the bf16 output itself against the oracle
    ref = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC, debug=True)
    got = {"residual_out": host_bf16(mx["residual_out"]), "layer_in": X,
           "pre_mix": mx["pre_mix"].cpu().numpy(), "post_mix": mx["post_mix"].cpu().numpy(),
           "comb_res_mix": mx["comb_res_mix"].cpu().numpy()}
    msgs = compare_fused(got, ref, (R, Y, pp, pc), gamma, label=w.name)
    assert not msgs, "\n".join(msgs)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("schedule,T,H", [
    ("small", 6, 7168), ("small", 37, 1024), ("small", 1, 4096),
    ("ws", 6, 7168), ("ws", 130, 4096), ("ws", 300, 7168), ("ws", 9, 2080),
    ("tile", 40, 7168), ("tile", 300, 4096), ("tile", 7, 1088),
    ("split", 40, 7168), ("split", 17, 1088),
    ("auto", 6, 7168), ("auto", 1000, 7168), ("auto", 2500, 7168), ("auto", 40, 7232), ("auto", 500, 7232)])
def test_mxfp8_epilogue_matches_separate_quantize(mhc, schedule, T, H, mode):
    run_case(mhc, synth.Workload(f"mx_{schedule}_{T}x{H}", T, H, 300 + T, token_scale=True), schedule, mode)


def test_mxfp8_prefill_chunk(mhc):
    """T=8192, H=7168 (the bench's workload), ws, every block checked."""
    run_case(mhc, synth.WORKLOADS["prefill_chunk"], "auto", 0, gamma_decades=False, check_oracle=False)


def test_mxfp8_rejects_bad_shapes_and_schedules(mhc):
    w = synth.Workload("mx_bad", 4, 1000, 5)     # H % 32 != 0
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)
    args = (dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), dev_f32(phi), dev_f32(bias), dev_f32(ms),
            dev_bf16(gamma))
    with pytest.raises(mhc.MhcError) as ei:
        mhc.shifted_post_pre_mxfp8(*args, **SC)
    assert ei.value.status == -1
    # a forced split call with the MXFP8 form only writes its bf16 layer input to the workspace
    # first; where AUTO would not take split (H <= 7168 here) the workspace has no room for it
    w = synth.Workload("mx_split", 600, 7168, 6)
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)
    args = (dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), dev_f32(phi), dev_f32(bias), dev_f32(ms),
            dev_bf16(gamma))
    out = {"layer_in_fp8": torch.full((600, 7168), 7, dtype=torch.uint8, device="cuda")}
    mhc.set_schedule("split")
    try:
        with pytest.raises(mhc.MhcError) as ei:
            mhc.shifted_post_pre_mxfp8(*args, **SC, want_bf16=False, out=out)
    finally:
        mhc.set_schedule("auto")
    assert ei.value.status == -3
    with pytest.raises(mhc.MhcError) as ei:
        mhc.shifted_post_pre_mxfp8(*args, **SC, scale_mode=2, out=out)
    assert ei.value.status == -1
    torch.cuda.synchronize()
    assert bool((out["layer_in_fp8"] == 7).all())
