"""phi packed once (mhc_pack_phi) and the _prepacked calls: bit-identical to the plain calls on
every schedule, one launch fewer on ws, and the packed bytes equal to what a plain call builds in
its workspace."""
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


def _args(w):
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    return (bf(R), bf(Y), f(pp), f(pc)), (f(phi), f(bias), f(ms), bf(gamma))


def _same(a, b):
    for k in a:
        x, y = a[k], b[k]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), k


@pytest.mark.parametrize("schedule,T,H", [("auto", 300, 7168), ("ws", 130, 4096), ("ws", 45, 2056),
                                          ("auto", 6, 7168), ("split", 40, 7168), ("ws", 8192, 7168),
                                          ("auto", 8192, 7168), ("tile", 300, 4096)])
def test_prepacked_equals_plain(mhc, schedule, T, H):
    w = synth.Workload(f"pk_{T}x{H}", T, H, 700 + T)
    toks, wts = _args(w)
    packed = mhc.pack_phi(wts[0])
    assert packed.numel() >= mhc.packed_phi_bytes(H)
    mhc.set_schedule(schedule)
    try:
        a = mhc.shifted_post_pre(*toks, *wts, **SC)
        na = mhc.last_launch_count()
        b = mhc.shifted_post_pre(*toks, *wts, **SC, packed_phi=packed)
        nb = mhc.last_launch_count()
        c = mhc.pre(toks[0], *wts, **SC)
        d = mhc.pre(toks[0], *wts, **SC, packed_phi=packed)
        torch.cuda.synchronize()
        ran = mhc.auto_schedule(T, H) if schedule == "auto" else mhc.SCHEDULES[schedule]
    finally:
        mhc.set_schedule("auto")
    _same(a, b)
    _same(c, d)
    if ran in (mhc.SCHEDULES["ws"], mhc.SCHEDULES["tile"]):
        assert nb == na - 1  # no packing launch


def test_pack_phi_equals_the_workspace_packing(mhc):
    """The plain ws call packs phi into its workspace right after the 256-byte control block;
    mhc_pack_phi writes the same bytes."""
    w = synth.Workload("pk_ws", 64, 7168, 5)
    toks, wts = _args(w)
    ws = mhc.new_workspace(w.T, w.H)
    mhc.set_schedule("ws")
    try:
        mhc.shifted_post_pre(*toks, *wts, **SC, workspace=ws)
    finally:
        mhc.set_schedule("auto")
    packed = mhc.pack_phi(wts[0])
    n = mhc.packed_phi_bytes(w.H)
    torch.cuda.synchronize()
    assert torch.equal(ws[256:256 + n], packed[:n])


@pytest.mark.parametrize("schedule,T,H,want_bf16", [("auto", 8192, 7168, True), ("auto", 8192, 7168, False),
                                                    ("auto", 6, 7168, True), ("ws", 130, 4096, False),
                                                    ("tile", 300, 4096, True)])
def test_mxfp8_prepacked_equals_plain(mhc, schedule, T, H, want_bf16):
    """mhc_shifted_post_pre_mxfp8_prepacked: every output bit-identical to the plain MXFP8 call."""
    w = synth.Workload(f"mxpk_{T}x{H}", T, H, 77)
    tok, wts = _args(w)
    mhc.set_schedule(schedule)
    try:
        nsb = mhc.mxfp8_scale_bytes(T, H)
        zeros = lambda: {"layer_in_scales": torch.zeros(nsb, dtype=torch.uint8, device="cuda")}
        a = mhc.shifted_post_pre_mxfp8(*tok, *wts, **SC, want_bf16=want_bf16, out=zeros())
        b = mhc.shifted_post_pre_mxfp8(*tok, *wts, **SC, want_bf16=want_bf16, out=zeros(),
                                       packed_phi=mhc.pack_phi(wts[0]))
        torch.cuda.synchronize()
    finally:
        mhc.set_schedule("auto")
    _same({k: v for k, v in a.items() if v is not None}, {k: v for k, v in b.items() if v is not None})
