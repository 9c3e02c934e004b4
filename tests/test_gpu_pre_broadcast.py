"""GPU parity of the first layer's broadcast pre (mhc_pre_broadcast) against the oracle.  The
path that materialises the four-copy residual and runs the pre on it must equal mhc_pre on that
residual bit for bit; the fused kernel that works from x alone (schedule "bcast", and AUTO for
T > 32 with H % 64 == 0) sums in another order and is held to the oracle's tolerances."""
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


def fused_path(schedule, T, H):
    return schedule == "bcast" or (schedule == "auto" and T > 32 and H % 64 == 0)


@pytest.mark.parametrize("schedule", ["auto", "small", "ws", "split", "bcast"])
@pytest.mark.parametrize("T,H", [(1, 1024), (6, 7168), (37, 2048), (300, 7168), (9, 1088), (2001, 1088)])
def test_pre_broadcast_parity(mhc, schedule, T, H):
    if schedule == "small" and T > 128:
        pytest.skip("the small schedule takes T <= 128")
    if schedule in ("small", "ws", "split") and T > 300:
        pytest.skip("the materialised path is covered at the smaller sizes")
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
    if not fused_path(schedule, T, H):
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


@pytest.mark.parametrize("T,H", [(8, 64), (41, 64), (16, 512), (152 * 8 + 3, 192)])
def test_pre_broadcast_fused_edges(mhc, T, H):
    """The fused kernel at its edges: H = 64 (one chunk mostly outside the tensor, zero-filled
    loads and clipped stores), whole and ragged 8-token tiles, exactly one chunk, and more
    tiles than CTAs with a ragged last tile."""
    w = synth.Workload(f"bcast_edge_{T}x{H}", T, H, 900 + T, token_scale=True)
    phi, bias, ms, gamma = synth.weights(w)
    _, x, _, _ = synth.tokens(w)
    mhc.set_schedule("bcast")
    try:
        ws = mhc.new_workspace(T, H)
        o = mhc.pre_broadcast(dev(x), dev(phi), dev(bias), dev(ms), dev(gamma), **SC, workspace=ws)
        mhc.check_status(ws)
    finally:
        mhc.set_schedule("auto")
    ref = oracle.pre_broadcast(x, phi, bias, ms, gamma, **SC, debug=True)
    assert np.array_equal(host_bf16(o["residual_out"]), ref["R"])
    nb, mu, _ = bf16_check(host_bf16(o["layer_in"]), ref["X"], layer_in_floor(ref["R"], ref["pre"], ref["rstd"], gamma))
    assert nb == 0, f"layer_in: {nb} bad, max {mu} ulp"
    for k, rk in (("pre_mix", "pre"), ("post_mix", "post"), ("comb_res_mix", "res")):
        d = np.abs(o[k].cpu().numpy().astype(np.float64) - ref[rk]).max()
        assert d <= MIX_ATOL, (k, d)


def test_pre_broadcast_fused_prefill_chunk_sampled(mhc):
    """The fused kernel at the prefill chunk's size (T = 8192, H = 7168), as the bench runs it:
    the residual is checked whole on the GPU, the other outputs on sampled tokens (the first and
    last tiles, and tiles spread over every CTA's share) against the oracle on those tokens."""
    w = synth.WORKLOADS["prefill_chunk"]
    T, H = w.T, w.H
    phi, bias, ms, gamma = synth.weights(w)
    _, x, _, _ = synth.tokens(w)
    wd = (dev(phi), dev(bias), dev(ms), dev(gamma))
    xd = dev(x)
    ws = mhc.new_workspace(T, H)
    o = mhc.pre_broadcast(xd, *wd, **SC, workspace=ws)
    mhc.check_status(ws)   # no bounded device wait gave up
    rv = o["residual_out"].view(torch.int16)
    assert torch.equal(rv, xd.view(torch.int16)[:, None, :].expand(T, 4, H))
    rng = np.random.default_rng(11)
    idx = np.unique(np.concatenate([np.arange(8), np.arange(T - 8, T), rng.choice(T, 48, replace=False)]))
    ref = oracle.pre_broadcast(x[idx], phi, bias, ms, gamma, **SC, debug=True)
    nb, mu, _ = bf16_check(host_bf16(o["layer_in"])[idx], ref["X"],
                           layer_in_floor(ref["R"], ref["pre"], ref["rstd"], gamma))
    assert nb == 0, f"layer_in: {nb} bad, max {mu} ulp"
    for k, rk in (("pre_mix", "pre"), ("post_mix", "post"), ("comb_res_mix", "res")):
        d = np.abs(o[k].cpu().numpy()[idx].astype(np.float64) - ref[rk]).max()
        assert d <= MIX_ATOL, (k, d)


@pytest.mark.parametrize("T", [33, 1217])
def test_pre_broadcast_auto_picks_fused_above_32(mhc, T):
    """AUTO takes the fused kernel for T > 32 (two launches: the phi_sum packing and the kernel)."""
    H = 1024
    w = synth.Workload(f"bcast_auto_{T}", T, H, 40 + T)
    phi, bias, ms, gamma = synth.weights(w)
    _, x, _, _ = synth.tokens(w)
    mhc.pre_broadcast(dev(x), dev(phi), dev(bias), dev(ms), dev(gamma), **SC)
    torch.cuda.synchronize()
    assert mhc.last_launch_count() == 2


def test_pre_broadcast_fused_in_graph_capture_on_fresh_stream(mhc):
    """The fused path (a packing launch, then the kernel under programmatic dependent launch)
    captured into a CUDA graph on a new stream: the replay gives the eager result bit for bit."""
    T, H = 300, 2048
    w = synth.Workload("bcast_graph", T, H, 77)
    phi, bias, ms, gamma = synth.weights(w)
    _, x, _, _ = synth.tokens(w)
    args = (dev(x), dev(phi), dev(bias), dev(ms), dev(gamma))
    eager = mhc.pre_broadcast(*args, **SC)
    torch.cuda.synchronize()
    outs = {k: torch.empty_like(v) for k, v in eager.items()}
    ws = mhc.new_workspace(T, H)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mhc.pre_broadcast(*args, **SC, out=outs, workspace=ws, stream=s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for k in eager:
        a, b = eager[k], outs[k]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), k
    mhc.check_status(ws)
