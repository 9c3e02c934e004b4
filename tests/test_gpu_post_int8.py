"""GPU parity of the post with an int8 layer output (mhc_post_int8) and of the fused square
sum (mhc_post_sqrsum), against the oracle's post_ex on the same seeded inputs."""
import numpy as np
import pytest

import oracle
from manifold_constrained_hyper_mhc_gb300 import synth

from _helpers import F, bf16_check, residual_floor

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
SQ_RTOL = 1e-4   # fp32 accumulation of 4H squares against the fp64 sum


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


def int8_layer_out(T, H, seed):
    """A symmetric per-token int8 quantization of a N(0, 1) layer output, with a few tokens
    scaled over decades and one all-zero token when T > 2."""
    rng = np.random.default_rng([seed, 8])
    y = rng.standard_normal((T, H)) * 10.0 ** rng.uniform(-2, 2, (T, 1))
    if T > 2:
        y[1] = 0.0
    amax = np.abs(y).max(axis=1)
    xs = np.where(amax > 0, amax / 127.0, 1.0).astype(np.float32)
    q = np.clip(np.rint(y / xs[:, None]), -127, 127).astype(np.int8)
    return q, xs


def int8_floor(R, q, xs, pp, pc):
    Ra = np.abs(F(R).astype(np.float64))
    S = np.einsum("nji,njh->nih", np.abs(pc.astype(np.float64)), Ra)
    S += np.abs(pp.astype(np.float64))[:, :, None] * np.abs(q.astype(np.float64) * xs[:, None])[:, None, :]
    return 2.0 ** -19 * S


@pytest.mark.parametrize("T,H", [(1, 8), (3, 1000), (6, 7168), (37, 1024), (130, 4096), (2048, 7168)])
def test_post_int8_parity(mhc, T, H):
    w = synth.Workload(f"post_int8_{T}x{H}", T, H, 500 + T, token_scale=True)
    R, _, pp, pc = synth.tokens(w)
    q, xs = int8_layer_out(T, H, w.seed)
    got, ss = mhc.post_int8(dev(R), dev(q), dev(xs), dev(pp), dev(pc))
    torch.cuda.synchronize()
    ref, ss_ref = oracle.post_ex(R, pp, pc, Yq=q, x_scales=xs)
    nb, mu, _ = bf16_check(host_bf16(got), ref, int8_floor(R, q, xs, pp, pc))
    assert nb == 0, f"{nb} bad, max {mu} ulp"
    np.testing.assert_allclose(ss.cpu().numpy(), ss_ref, rtol=SQ_RTOL)
    # deterministic, and the square sum is optional
    got2, ss2 = mhc.post_int8(dev(R), dev(q), dev(xs), dev(pp), dev(pc))
    got3, none = mhc.post_int8(dev(R), dev(q), dev(xs), dev(pp), dev(pc), sqrsum=False)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(got.view(torch.int16), got2.view(torch.int16)) and torch.equal(ss, ss2)
    assert torch.equal(got.view(torch.int16), got3.view(torch.int16))


@pytest.mark.parametrize("T,H", [(1, 8), (6, 7168), (130, 4096)])
def test_post_sqrsum_parity_and_equal_to_post(mhc, T, H):
    w = synth.Workload(f"post_sq_{T}x{H}", T, H, 600 + T, token_scale=True)
    R, Y, pp, pc = synth.tokens(w)
    got, ss = mhc.post_sqrsum(dev(R), dev(Y), dev(pp), dev(pc))
    plain = mhc.post(dev(R), dev(Y), dev(pp), dev(pc))
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), plain.view(torch.int16))
    ref, ss_ref = oracle.post_ex(R, pp, pc, Y=Y)
    nb, mu, _ = bf16_check(host_bf16(got), ref, residual_floor(R, Y, pp, pc))
    assert nb == 0, f"{nb} bad, max {mu} ulp"
    np.testing.assert_allclose(ss.cpu().numpy(), ss_ref, rtol=SQ_RTOL)


def test_post_int8_in_place_and_bad_arguments(mhc):
    T, H = 4, 1024
    w = synth.Workload("post_int8_ip", T, H, 7)
    R, _, pp, pc = synth.tokens(w)
    q, xs = int8_layer_out(T, H, 7)
    ref, _ = mhc.post_int8(dev(R), dev(q), dev(xs), dev(pp), dev(pc))
    Rd = dev(R)
    mhc.post_int8(Rd, dev(q), dev(xs), dev(pp), dev(pc), out=Rd)
    torch.cuda.synchronize()
    assert torch.equal(Rd.view(torch.int16), ref.view(torch.int16))
    out = torch.full((T, 4, H), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    lib = mhc.lib()
    P = lambda t: None if t is None else __import__("ctypes").c_void_p(t.data_ptr())
    rc = lib.mhc_post_int8(P(dev(R)), P(dev(q)), None, P(dev(pp)), P(dev(pc)), T, H, P(out), None, None)
    assert rc == -1
    torch.cuda.synchronize()
    assert bool((out.view(torch.int16) == 7).all())
