"""GPU parity of the first layer's broadcast pre (mhc_pre_broadcast) against the oracle, and
its equality with mhc_pre on the materialised four-copy residual."""
import numpy as np
import pytest

import oracle
from manifold_constrained_hyper_mhc_gb300 import synth

from _helpers import MIX_ATOL, bf16_check, layer_in_floor

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
SC = synth.scalars()


@pytest.fixture(scope="module")
def mhc(mhc_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return mhc_lib


def dev(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bf16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("schedule", ["auto", "small", "ws", "split"])
@pytest.mark.parametrize("T,H", [(1, 1024), (6, 7168), (37, 2048), (300, 7168)])
def test_pre_broadcast_parity(mhc, schedule, T, H):
    if schedule == "small" and T > 64:
        pytest.skip("the small schedule takes T <= 64")
    w = synth.Workload(f"bcast_{T}x{H}", T, H, 700 + T, token_scale=True)
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, _, _ = synth.tokens(w)
    x = Y                                     # a seeded (T, H) bf16 input
    wd = (dev(phi), dev(bias), dev(ms), dev(gamma))
    mhc.set_schedule(schedule)
    try:
        o = mhc.pre_broadcast(dev(x), *wd, **SC)
        Rb = o["residual_out"].clone()
        q = mhc.pre(Rb, *wd, **SC)
        torch.cuda.synchronize()
    finally:
        mhc.set_schedule("auto")
    ref = oracle.pre_broadcast(x, phi, bias, ms, gamma, **SC, debug=True)
    assert np.array_equal(host_bf16(o["residual_out"]), ref["R"])
    for k in ("layer_in", "pre_mix", "post_mix", "comb_res_mix"):   # equal to mhc_pre on the residual
        a, b = o[k], q[k]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), k
    nb, mu, _ = bf16_check(host_bf16(o["layer_in"]), ref["X"], layer_in_floor(ref["R"], ref["pre"], ref["rstd"], gamma))
    assert nb == 0, f"layer_in: {nb} bad, max {mu} ulp"
    for k, rk in (("pre_mix", "pre"), ("post_mix", "post"), ("comb_res_mix", "res")):
        d = np.abs(o[k].cpu().numpy().astype(np.float64) - ref[rk]).max()
        assert d <= MIX_ATOL, (k, d)


def test_pre_broadcast_rejects_overlap_before_launching(mhc):
    T, H = 4, 1024
    w = synth.Workload("bcast_bad", T, H, 9)
    phi, bias, ms, gamma = synth.weights(w)
    _, Y, _, _ = synth.tokens(w)
    big = torch.full((T, 4, H), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    x = big[:, 0, :].contiguous()
    with pytest.raises(mhc.MhcError):
        # the layer input aliases the residual output: refused, and nothing is written
        mhc.pre_broadcast(dev(Y), dev(phi), dev(bias), dev(ms), dev(gamma), **SC,
                          out={"residual_out": big, "layer_in": big.view(-1)[:T * H].view(T, H)})
    torch.cuda.synchronize()
    assert bool((big.view(torch.int16) == 7).all())
