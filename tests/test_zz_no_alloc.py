"""mhc_shifted_post_pre_noalloc: the fused call for callers that cannot
allocate device memory (a host framework that owns all device memory, a
plugin that must not grow the footprint, a hot path where an allocation would
synchronise).  Its scratch is a fixed static array inside the library, so the
caller passes only inputs and outputs.

Called here through the C ABI (ctypes) and checked against the regular
mhc_shifted_post_pre on calls in a row with different inputs and sizes, with
the tolerances of the parity tests; mhc_noalloc_check_status reads the static
scratch's status word after each.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from manifold_constrained_hyper_mhc_gb300 import synth

from _helpers import MIX_ATOL, bf16_check

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
SC = synth.scalars()


@pytest.fixture(scope="module")
def lib(mhc_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = mhc_lib.lib()
    P, I64, F, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    L.mhc_shifted_post_pre_noalloc.argtypes = [P, P, P, P, P, P, P, P, I64, I64, F, F, F, F, I,
                                               P, P, P, P, P, P]
    L.mhc_shifted_post_pre_noalloc.restype = I
    L.mhc_noalloc_check_status.argtypes = [P]
    L.mhc_noalloc_check_status.restype = I
    return L


def _inputs(w):
    phi, bias, ms, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)
    bf = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    return (bf(R), bf(Y), f(pp), f(pc), f(phi), f(bias), f(ms), bf(gamma))


def _outs(T, H):
    return {"residual_out": torch.empty((T, 4, H), dtype=torch.bfloat16, device="cuda"),
            "layer_in": torch.empty((T, H), dtype=torch.bfloat16, device="cuda"),
            "pre_mix": torch.empty((T, 4), device="cuda"), "post_mix": torch.empty((T, 4), device="cuda"),
            "comb_res_mix": torch.empty((T, 4, 4), device="cuda")}


def _noalloc(L, ins, T, H, o):
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return L.mhc_shifted_post_pre_noalloc(
        *[p(t) for t in ins], T, H, SC["hc_norm_eps"], SC["rmsnorm_eps"], SC["hc_post_scale"],
        SC["sinkhorn_eps"], SC["sinkhorn_iters"], p(o["residual_out"]), p(o["layer_in"]), p(o["pre_mix"]),
        p(o["post_mix"]), p(o["comb_res_mix"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_noalloc_matches_fused_on_two_calls_in_a_row(lib, mhc_lib):
    cases = [synth.WORKLOADS["decode_verify"], synth.WORKLOADS["mid_batch"]]
    ins = [_inputs(w) for w in cases]
    got = [_outs(w.T, w.H) for w in cases]
    for w, i, o in zip(cases, ins, got):          # two no-alloc calls back to back
        assert _noalloc(lib, i, w.T, w.H, o) == 0, lib.mhc_last_error().decode()
    assert lib.mhc_noalloc_check_status(_stream()) == 0, lib.mhc_last_error().decode()
    want = [mhc_lib.shifted_post_pre(*i, **SC) for i in ins]
    torch.cuda.synchronize()
    for w, g, r in zip(cases, got, want):
        for k in ("residual_out", "layer_in"):
            nbad, max_ulp, _ = bf16_check(_bits(g[k]), _bits(r[k]), 0.0)
            assert nbad == 0, f"{w.name} {k}: {nbad} elements beyond tolerance (max {max_ulp} ulp)"
        for k in ("pre_mix", "post_mix", "comb_res_mix"):
            assert float((g[k] - r[k]).abs().max()) <= MIX_ATOL, (w.name, k)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_noalloc_calls_of_different_hidden_sizes_in_a_row(lib, mhc_lib):
    """Calls of at most 32 tokens run on the small schedule, whose CTA count follows H (112 at
    H = 7168, 64 at 4096, 16 at 1024) and whose grid barrier keeps its word in the shared static
    scratch.  H = 7168, 4096, 1024 and 7168 again in a row: each against mhc_shifted_post_pre
    on a fresh workspace, and the scratch's status word clear after each."""
    cases = [synth.Workload("na_7168", 6, 7168, 61), synth.Workload("na_4096", 17, 4096, 62),
             synth.Workload("na_1024", 32, 1024, 63), synth.Workload("na_7168b", 5, 7168, 64)]
    for w in cases:
        assert mhc_lib.auto_schedule(w.T, w.H) == mhc_lib.SCHEDULES["small"]
        ins = _inputs(w)
        o = _outs(w.T, w.H)
        assert _noalloc(lib, ins, w.T, w.H, o) == 0, lib.mhc_last_error().decode()
        assert lib.mhc_noalloc_check_status(_stream()) == 0, lib.mhc_last_error().decode()
        r = mhc_lib.shifted_post_pre(*ins, **SC)
        torch.cuda.synchronize()
        for k in ("residual_out", "layer_in"):
            nbad, max_ulp, _ = bf16_check(_bits(o[k]), _bits(r[k]), 0.0)
            assert nbad == 0, f"{w.name} {k}: {nbad} elements beyond tolerance (max {max_ulp} ulp)"
        for k in ("pre_mix", "post_mix", "comb_res_mix"):
            assert float((o[k] - r[k]).abs().max()) <= MIX_ATOL, (w.name, k)


def test_noalloc_rejects_calls_beyond_its_scratch(lib):
    w = synth.Workload("big", 2048, 7168, 0)
    ins = _inputs(synth.Workload("one", 1, 7168, 0))
    o = _outs(1, 7168)
    o["layer_in"].view(torch.int16).fill_(7)
    torch.cuda.synchronize()
    # pointers of a 1-token call with T claiming 2048 tokens: rejected before any launch
    rc = _noalloc(lib, ins, w.T, w.H, o)
    assert rc == -1
    assert "static scratch" in lib.mhc_last_error().decode()
    torch.cuda.synchronize()
    assert bool((o["layer_in"].view(torch.int16) == 7).all())
