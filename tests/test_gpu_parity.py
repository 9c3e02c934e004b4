"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, element by element, with the tolerances in _helpers."""
import numpy as np
import pytest

import oracle
from manifold_constrained_hyper_mhc_gb300 import synth

from _helpers import F, MIX_ATOL, bf16_check, compare_fused, write_report

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


def host(t):
    return t.cpu().numpy()


def weights_dev(w):
    phi, bias, ms, gamma = synth.weights(w)
    return (phi, bias, ms, gamma), (dev_f32(phi), dev_f32(bias), dev_f32(ms), dev_bf16(gamma))


def gpu_fused(mhc, R, Y, pp, pc, wd, sc=SC, **kw):
    o = mhc.shifted_post_pre(dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd, **sc, **kw)
    torch.cuda.synchronize()
    return {k: (host_bf16(v) if v.dtype == torch.bfloat16 else host(v)) for k, v in o.items()}


SMALL_MAX_T = 128  # the small-T schedule takes T <= 128 (while its shared memory fits) and refuses larger calls


def check_workload(mhc, w, schedule="auto"):
    if schedule == "small" and (w.T > SMALL_MAX_T or (w.T > 96 and w.H > 4096)):
        pytest.skip("the small schedule takes T <= 128, and at H = 7168 T <= 96 (shared memory)")
    if schedule == "tile" and (w.H % 64 != 0 or w.H <= 256):
        pytest.skip("the tile schedule needs H % 64 == 0 and H > 256")
    (phi, bias, ms, gamma), wd = weights_dev(w)
    R, Y, pp, pc = synth.tokens(w)
    mhc.set_schedule(schedule)
    try:
        got = gpu_fused(mhc, R, Y, pp, pc, wd)
    finally:
        mhc.set_schedule("auto")
    ref = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC, debug=True)
    msgs = compare_fused(got, ref, (R, Y, pp, pc), gamma, label=w.name)
    assert not msgs, "\n".join(msgs)


ALL_SCHEDULES = ["auto", "split", "ws", "small", "tile"]


@pytest.mark.parametrize("name", ["tiny", "decode_verify", "mid_batch"])
@pytest.mark.parametrize("schedule", ALL_SCHEDULES)
def test_workload_parity(mhc, name, schedule):
    check_workload(mhc, synth.WORKLOADS[name], schedule)


@pytest.mark.parametrize("T,H", [(1, 8), (3, 24), (5, 264), (17, 1000), (33, 2056), (130, 520)])
@pytest.mark.parametrize("schedule", ALL_SCHEDULES)
def test_ragged_shapes(mhc, T, H, schedule):
    check_workload(mhc, synth.Workload(f"ragged_{T}x{H}", T, H, 100 + T, token_scale=True), schedule)


@pytest.mark.parametrize("T,H", [(1, 320), (17, 1088), (37, 2112), (130, 7168), (300, 4096), (1000, 7168)])
def test_tile_schedule_shapes(mhc, T, H):
    """The token-tile kernel alone on every SM: a single token, ragged tiles (T % 18 != 0) and
    ragged chunks (H % 256 != 0), more tiles than SMs."""
    check_workload(mhc, synth.Workload(f"tile_{T}x{H}", T, H, 200 + T, token_scale=True), "tile")


@pytest.mark.parametrize("T,H", [(500, 7232), (600, 8192), (100, 7232), (40, 8256)])
def test_auto_beyond_ws_hidden_size(mhc, T, H):
    """H > 7168, where ws's 16-CTA slice no longer fits: AUTO takes the token-tile kernel alone
    from 448 tokens on and the split schedule below; every token against the oracle."""
    want = "tile" if T >= 448 else "split"
    assert mhc.auto_schedule(T, H) == mhc.SCHEDULES[want]
    check_workload(mhc, synth.Workload(f"wide_{T}x{H}", T, H, 400 + T, token_scale=True))


def test_auto_side_share_query(mhc):
    """mhc_auto_side_tokens: no side share below 2048 tokens or off the ws schedule; above, ws
    keeps a whole number of 8-token groups and the tile kernel the rest."""
    assert mhc.auto_side_tokens(1024, 7168) == 0
    assert mhc.auto_side_tokens(6, 7168) == 0
    assert mhc.auto_side_tokens(8192, 8192) == 0           # H > 7168: tile alone, not beside ws
    side = mhc.auto_side_tokens(8192, 7168)
    assert 0 < side < 8192 and (8192 - side) % 8 == 0
    assert mhc.auto_side_tokens(-1, 7168) == -1


@pytest.mark.parametrize("T,H", [(2048, 7168), (4096, 4096), (2500, 7168)])
def test_ws_with_tile_beside(mhc, T, H):
    """AUTO from 2048 tokens on: ws on the leading tokens, the token-tile kernel beside it on the
    SMs ws's clusters leave idle; every token against the oracle, and the same results in place."""
    w = synth.Workload(f"beside_{T}x{H}", T, H, 300 + T, token_scale=True)
    check_workload(mhc, w)
    (phi, bias, ms, gamma), wd = weights_dev(w)
    R, Y, pp, pc = synth.tokens(w)
    Rd = dev_bf16(R)
    a = mhc.shifted_post_pre(dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd, **SC)
    b = mhc.shifted_post_pre(Rd, dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd, **SC, out={"residual_out": Rd})
    torch.cuda.synchronize()
    for k in a:
        x, y = a[k], b[k]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), k


def _full_parity(mhc, w, step=1024):
    """Every token of workload w against the oracle (compared in token chunks to bound host
    memory).  Returns the GPU outputs (on the device) and the parity report."""
    (phi, bias, ms, gamma), wd = weights_dev(w)
    R, Y, pp, pc = synth.tokens(w)
    o = mhc.shifted_post_pre(dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd, **SC)
    torch.cuda.synchronize()
    msgs, report = [], {}
    for t0 in range(0, w.T, step):
        s = slice(t0, t0 + step)
        got = {k: (host_bf16(v[s]) if v.dtype == torch.bfloat16 else host(v[s])) for k, v in o.items()}
        ref = oracle.shifted_post_pre(R[s], Y[s], pp[s], pc[s], phi, bias, ms, gamma, **SC, debug=True)
        msgs += compare_fused(got, ref, (R[s], Y[s], pp[s], pc[s]), gamma, label=f"tokens {t0}+", report=report)
    write_report(w.name, report)
    assert not msgs, "\n".join(msgs[:20])
    return o, gamma, report


def test_prefill_chunk_full_parity(mhc):
    """T=8192, H=7168, the bench's workload and launch configuration: every token
    against the oracle."""
    _full_parity(mhc, synth.WORKLOADS["prefill_chunk"])


@pytest.mark.slow
def test_long_prefill_full_parity_and_invariants(mhc):
    """T=65536, H=7168 with 1% zero-Y and 1% identical-stream tokens: every token against
    the oracle, and properties that hold at any size on every token."""
    w = synth.WORKLOADS["long_prefill"]
    o, gamma, _ = _full_parity(mhc, w, step=2048)
    res = o["comb_res_mix"]
    cs, rs = res.sum(1), res.sum(2)
    eps = SC["sinkhorn_eps"]
    assert bool((res > 0).all())
    assert bool(((cs < 1 + 1e-6) & (cs > 1 - 2 * eps)).all())
    assert bool(((rs - 1).abs() < 1e-3).all())
    assert bool(((o["pre_mix"] > 0) & (o["pre_mix"] < 1)).all())
    assert bool(((o["post_mix"] > 0) & (o["post_mix"] < SC["hc_post_scale"])).all())
    x = o["layer_in"].float() / dev_bf16(gamma).float()[None, :]
    ms2 = (x * x).mean(1)
    assert bool(((ms2 - 1).abs() < 2e-2).all()), float((ms2 - 1).abs().max())


@pytest.mark.parametrize("schedule", ALL_SCHEDULES[1:])
def test_fused_equals_post_then_pre_bitwise(mhc, schedule):
    mhc.set_schedule(schedule)
    try:
        _fused_vs_composed(mhc, SMALL_MAX_T if schedule == "small" else None)
    finally:
        mhc.set_schedule("auto")


def _fused_vs_composed(mhc, max_t=None):
    for name in ("tiny", "mid_batch"):
        w = synth.WORKLOADS[name]
        if max_t is not None and w.T > max_t:
            continue
        _, wd = weights_dev(w)
        R, Y, pp, pc = synth.tokens(w)
        Rd, Yd, ppd, pcd = dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc)
        f = mhc.shifted_post_pre(Rd, Yd, ppd, pcd, *wd, **SC)
        rp = mhc.post(Rd, Yd, ppd, pcd)
        q = mhc.pre(rp, *wd, **SC)
        torch.cuda.synchronize()
        assert torch.equal(f["residual_out"].view(torch.int16), rp.view(torch.int16))
        for k in ("layer_in", "pre_mix", "post_mix", "comb_res_mix"):
            a, b = f[k], q[k]
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), k


def test_post_alone_matches_oracle(mhc):
    w = synth.Workload("post", 37, 776, 7, token_scale=True)
    R, Y, pp, pc = synth.tokens(w)
    got = host_bf16(mhc.post(dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc)))
    ref = oracle.post(R, Y, pp, pc)
    from _helpers import residual_floor
    nb, mu, _ = bf16_check(got, ref, residual_floor(R, Y, pp, pc))
    assert nb == 0, f"{nb} bad, max {mu} ulp"


def test_pre_identical_streams_property(mhc):
    """mhc_pre on four identical streams s: X = s * sum(pre), so the output is
    RMSNorm(s) * gamma whatever pre is (up to rmsnorm_eps)."""
    w = synth.Workload("same", 9, 1024, 21)
    (phi, bias, ms, gamma), wd = weights_dev(w)
    R, _, _, _ = synth.tokens(w)
    R[:, 1:, :] = R[:, :1, :]
    o = mhc.pre(dev_bf16(R), *wd, **SC)
    ref = oracle.pre(R, phi, bias, ms, gamma, **SC, debug=True)
    got = host_bf16(o["layer_in"])
    s = F(R[:, 0, :]).astype(np.float64)
    want = s / np.sqrt((s * s).mean(1, keepdims=True)) * F(gamma).astype(np.float64)[None, :]
    g = F(got).astype(np.float64)
    assert np.all(np.abs(g - want) <= 3 * 2.0 ** (np.floor(np.log2(np.abs(want) + 1e-30)) - 7) + 1e-6)
    np.testing.assert_array_less(np.abs(host(o["pre_mix"]) - ref["pre"]), MIX_ATOL)


def test_in_place_residual_update(mhc):
    w = synth.WORKLOADS["tiny"]
    _, wd = weights_dev(w)
    R, Y, pp, pc = synth.tokens(w)
    Rd = dev_bf16(R)
    ref = mhc.shifted_post_pre(dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd, **SC)
    out = mhc.shifted_post_pre(Rd, dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd, **SC,
                               out={"residual_out": Rd})
    torch.cuda.synchronize()
    assert out["residual_out"].data_ptr() == Rd.data_ptr()
    assert torch.equal(Rd.view(torch.int16), ref["residual_out"].view(torch.int16))
    assert torch.equal(out["layer_in"].view(torch.int16), ref["layer_in"].view(torch.int16))


def test_repeatable_bit_for_bit(mhc):
    w = synth.WORKLOADS["mid_batch"]
    _, wd = weights_dev(w)
    R, Y, pp, pc = synth.tokens(w)
    args = (dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd)
    a = mhc.shifted_post_pre(*args, **SC)
    b = mhc.shifted_post_pre(*args, **SC)
    torch.cuda.synchronize()
    for k in a:
        x, y = a[k], b[k]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), k


def test_first_call_inside_graph_capture_on_fresh_stream(mhc):
    """No lazy per-stream state: the very first call on a new stream may be
    captured into a CUDA graph, and replay gives the eager result."""
    w = synth.WORKLOADS["decode_verify"]
    _, wd = weights_dev(w)
    R, Y, pp, pc = synth.tokens(w)
    args = (dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd)
    eager = mhc.shifted_post_pre(*args, **SC)
    torch.cuda.synchronize()
    outs = {k: torch.empty_like(v) for k, v in eager.items()}
    ws = mhc.new_workspace(w.T, w.H)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mhc.shifted_post_pre(*args, **SC, out=outs, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    for k in eager:
        x, y = eager[k], outs[k]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), k
    mhc.check_status(ws)


def test_bad_arguments_launch_nothing(mhc):
    w = synth.WORKLOADS["tiny"]
    _, wd = weights_dev(w)
    R, Y, pp, pc = synth.tokens(w)
    Rd, Yd, ppd, pcd = dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc)
    outs = {"layer_in": torch.full((w.T, w.H), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)}
    with pytest.raises(mhc.MhcError):
        mhc.shifted_post_pre(Rd, Yd, ppd, pcd, *wd, **dict(SC, sinkhorn_iters=-3), out=outs)
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(mhc.MhcError):
        mhc.shifted_post_pre(Rd, Yd, ppd, pcd, *wd, **SC, out=outs, workspace=small)
    torch.cuda.synchronize()
    assert bool((outs["layer_in"].view(torch.int16) == 7).all())


def test_zero_tokens(mhc):
    H = 1024
    w = synth.Workload("z", 1, H, 0)
    _, wd = weights_dev(w)
    e = torch.empty((0, 4, H), dtype=torch.bfloat16, device="cuda")
    o = mhc.shifted_post_pre(e, torch.empty((0, H), dtype=torch.bfloat16, device="cuda"),
                             torch.empty((0, 4), device="cuda"), torch.empty((0, 4, 4), device="cuda"),
                             *wd, **SC)
    assert o["layer_in"].shape == (0, H)


@pytest.mark.parametrize("T,H", [(96, 7168), (SMALL_MAX_T, 4096), (SMALL_MAX_T, 1024)])
def test_small_schedule_largest_T(mhc, T, H):
    """The small-T schedule at its largest token counts (eight 16-token tiles; at H = 7168 the
    shared memory allows 96 tokens), against the oracle."""
    check_workload(mhc, synth.Workload(f"small_{T}x{H}", T, H, 40, token_scale=True), "small")


def test_small_schedule_refuses_large_T(mhc):
    w = synth.Workload("small_too_many", SMALL_MAX_T + 1, 1024, 41)
    _, wd = weights_dev(w)
    R, Y, pp, pc = synth.tokens(w)
    outs = {"layer_in": torch.full((w.T, w.H), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)}
    mhc.set_schedule("small")
    try:
        with pytest.raises(mhc.MhcError) as ei:
            mhc.shifted_post_pre(dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd, **SC, out=outs)
    finally:
        mhc.set_schedule("auto")
    assert ei.value.status == -2
    torch.cuda.synchronize()
    assert bool((outs["layer_in"].view(torch.int16) == 7).all())


def test_small_schedule_barrier_timeout_is_reported(mhc):
    """The grid barrier's wait is bounded: with its arrival counter preset so that
    it can never complete, every CTA gives up after its time limit, the call
    leaves the status word set, mhc_check_status reports MHC_ERR_DEVICE_TIMEOUT
    and clears the control block, and the next call on the same workspace is
    correct again."""
    w = synth.WORKLOADS["decode_verify"]
    (phi, bias, ms, gamma), wd = weights_dev(w)
    R, Y, pp, pc = synth.tokens(w)
    args = (dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd)
    ws = mhc.new_workspace(w.T, w.H)
    words = ws.view(torch.int32)
    mhc.set_schedule("small")
    try:
        words[16] = 0x40000000  # arrival counter far from the CTA count: the barrier never opens
        mhc.shifted_post_pre(*args, **SC, workspace=ws)
        with pytest.raises(mhc.MhcError) as ei:
            mhc.check_status(ws)
        assert ei.value.status == -5
        assert int(words[:64].abs().sum()) == 0
        o = mhc.shifted_post_pre(*args, **SC, workspace=ws)
        mhc.check_status(ws)
    finally:
        mhc.set_schedule("auto")
    got = {k: (host_bf16(v) if v.dtype == torch.bfloat16 else host(v)) for k, v in o.items()}
    ref = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC, debug=True)
    msgs = compare_fused(got, ref, (R, Y, pp, pc), gamma, label="after timeout")
    assert not msgs, "\n".join(msgs)


def test_small_schedule_one_workspace_across_hidden_sizes(mhc):
    """The small schedule's CTA count follows H (112 CTAs at H = 7168, 64 at 4096, 16 at 1024)
    and its grid barrier keeps its word in the workspace's control block: calls with those
    sizes and the first again, in a row on one workspace, each against the oracle, with the
    status word checked after each."""
    cases = [synth.Workload("seq_7168", 6, 7168, 61), synth.Workload("seq_4096", 17, 4096, 62),
             synth.Workload("seq_1024", 32, 1024, 63), synth.Workload("seq_7168b", 5, 7168, 64)]
    ws = mhc.new_workspace(max(w.T for w in cases), 7168)
    assert ws.numel() >= max(mhc.workspace_size(w.T, w.H) for w in cases)
    mhc.set_schedule("small")
    try:
        for w in cases:
            (phi, bias, ms, gamma), wd = weights_dev(w)
            R, Y, pp, pc = synth.tokens(w)
            o = mhc.shifted_post_pre(dev_bf16(R), dev_bf16(Y), dev_f32(pp), dev_f32(pc), *wd, **SC, workspace=ws)
            mhc.check_status(ws)
            got = {k: (host_bf16(v) if v.dtype == torch.bfloat16 else host(v)) for k, v in o.items()}
            ref = oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **SC, debug=True)
            msgs = compare_fused(got, ref, (R, Y, pp, pc), gamma, label=w.name)
            assert not msgs, "\n".join(msgs)
    finally:
        mhc.set_schedule("auto")
