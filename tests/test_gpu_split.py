"""The split fused step (mhc_shifted_post_pre_split): the post and residual mixes on a side
stream.  Outputs must equal mhc_shifted_post_pre's on the same schedule bit for bit, eagerly
and under CUDA-graph capture, and the events must order the side work."""
import numpy as np
import pytest

from manifold_constrained_hyper_mhc_gb300 import synth

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


def inputs(T, H, seed):
    w = synth.Workload(f"split_{T}x{H}", T, H, seed, token_scale=True)
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)
    return (dev(R), dev(Y), dev(pp), dev(pc), dev(phi), dev(bias), dev(ms), dev(gamma))


def events():
    f, j = torch.cuda.Event(), torch.cuda.Event()
    f.record(); j.record()  # torch creates the CUDA events on first record
    return f, j


def same(a, b):
    for k in a:
        x, y = a[k], b[k]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), k


@pytest.mark.parametrize("schedule", ["auto", "small", "ws"])
@pytest.mark.parametrize("T,H", [(1, 1024), (6, 7168), (16, 7168), (32, 4096)])
def test_split_equals_fused(mhc, schedule, T, H):
    args = inputs(T, H, 800 + T)
    side = torch.cuda.Stream()
    f, j = events()
    mhc.set_schedule(schedule)
    try:
        ref = mhc.shifted_post_pre(*args, **SC)
        o = mhc.shifted_post_pre_split(*args, **SC, side_stream=side, fork_event=f, join_event=j)
        launches = mhc.last_launch_count()
        torch.cuda.current_stream().wait_event(j)
        torch.cuda.synchronize()
    finally:
        mhc.set_schedule("auto")
    if schedule != "ws":
        assert launches == 2      # the main kernel and the side kernel
    same(ref, o)


def test_split_under_graph_capture_with_two_workspaces(mhc):
    """The pattern a decoder uses: call i waits on the join of call i-2 (same workspace) so that
    the side kernel of call i overlaps the main kernel of call i+1."""
    T, H = 6, 7168
    args = inputs(T, H, 900)
    ref = mhc.shifted_post_pre(*args, **SC)
    torch.cuda.synchronize()
    s, side = torch.cuda.Stream(), torch.cuda.Stream()
    wss = [mhc.new_workspace(T, H), mhc.new_workspace(T, H)]
    evs = [events(), events()]
    outs = [{k: torch.empty_like(v) for k, v in ref.items()} for _ in range(4)]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(4):
            f, j = evs[i % 2]
            if i >= 2:
                s.wait_event(j)
            mhc.shifted_post_pre_split(*args, **SC, side_stream=side, fork_event=f, join_event=j,
                                       out=outs[i], workspace=wss[i % 2], stream=s)
        for f, j in evs:
            s.wait_event(j)
    g.replay()
    torch.cuda.synchronize()
    for o in outs:
        same(ref, o)
    for w in wss:
        mhc.check_status(w)


def test_split_rejects_missing_events(mhc):
    T, H = 2, 1024
    args = inputs(T, H, 901)
    side = torch.cuda.Stream()
    lib = mhc.lib()
    import ctypes
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    o = {"layer_in": torch.full((T, H), 7, dtype=torch.int16, device="cuda")}
    rc = lib.mhc_shifted_post_pre_split(*[P(a) for a in args], T, H, *[float(SC[k]) for k in
                                        ("hc_norm_eps", "rmsnorm_eps", "hc_post_scale", "sinkhorn_eps")],
                                        int(SC["sinkhorn_iters"]), P(torch.empty((T, 4, H), dtype=torch.bfloat16, device="cuda")),
                                        P(o["layer_in"]), P(torch.empty((T, 4), device="cuda")),
                                        P(torch.empty((T, 4), device="cuda")), P(torch.empty((T, 4, 4), device="cuda")),
                                        P(mhc.new_workspace(T, H)), mhc.workspace_size(T, H), None,
                                        ctypes.c_void_p(side.cuda_stream), None, None)
    assert rc == -1
    torch.cuda.synchronize()
    assert bool((o["layer_in"] == 7).all())


def test_split_with_no_tokens_still_records_the_events(mhc):
    H = 1024
    args = inputs(1, H, 902)
    e = lambda *shape: torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    z = (e(0, 4, H), e(0, H), torch.empty((0, 4), device="cuda"), torch.empty((0, 4, 4), device="cuda"), *args[4:])
    side = torch.cuda.Stream()
    f, j = events()
    o = mhc.shifted_post_pre_split(*z, **SC, side_stream=side, fork_event=f, join_event=j)
    torch.cuda.current_stream().wait_event(j)
    torch.cuda.synchronize()
    assert o["layer_in"].shape == (0, H) and j.query()
