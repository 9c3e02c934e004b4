"""CPU-only checks of the variant entry points (MXFP8 epilogue, int8 post, square-sum post,
broadcast pre, side-stream split): their argument checks reject bad calls before touching
CUDA, and the host-side size helpers hold their closed forms.  Pointers are fake aligned
addresses: nothing is dereferenced before validation."""
import ctypes

import pytest

import oracle

SC = (2e-5, 2e-6, 1.25, 3e-4, 20)


def P(a):
    return ctypes.c_void_p(a)


def ins(n, base=0x100000000):
    return [P(base + i * (1 << 36)) for i in range(n)]


def test_mxfp8_scale_bytes_matches_the_oracle_layout(mhc_lib):
    L = mhc_lib.lib()
    for T, H in [(1, 7168), (6, 7168), (128, 4096), (300, 7168 + 160), (8192, 7168)]:
        rows, cols = oracle.mx_scale_shape(T, H)
        assert L.mhc_mxfp8_scale_bytes(T, H) == rows * cols
    assert L.mhc_mxfp8_scale_bytes(4, 1000) == 0      # H % 32 != 0


def _mx_call(L, T, H, q, s, mode, X=True):
    p = ins(8)
    outs = ins(5, 0x200000000000)
    return L.mhc_shifted_post_pre_mxfp8(*p, T, H, *SC[:4], SC[4], outs[0], outs[1] if X else None, q, s, mode,
                                        outs[2], outs[3], outs[4], P(0x7000000000), 1 << 30, None)


def test_mxfp8_argument_checks(mhc_lib):
    L = mhc_lib.lib()
    q, s = P(0x300000000000), P(0x310000000000)
    assert _mx_call(L, 4, 1000, q, s, 0) == -1          # H % 32 != 0
    assert _mx_call(L, 4, 1024, q, s, 2) == -1          # unknown scale rule
    assert _mx_call(L, 4, 1024, None, s, 0) == -1       # no E4M3 buffer
    assert _mx_call(L, 4, 1024, q, None, 0) == -1       # no scale buffer
    assert _mx_call(L, 4, 1024, P(0x300000000004), s, 0) == -1   # misaligned E4M3 buffer
    assert _mx_call(L, 0, 1024, q, s, 0) == 0           # T == 0: nothing to do


def test_post_variant_argument_checks(mhc_lib):
    L = mhc_lib.lib()
    R, q, xs, pp, pc = ins(5)
    out, ss = P(0x200000000000), P(0x210000000000)
    assert L.mhc_post_int8(R, None, xs, pp, pc, 4, 1024, out, ss, None) == -1
    assert L.mhc_post_int8(R, q, None, pp, pc, 4, 1024, out, ss, None) == -1
    assert L.mhc_post_int8(R, q, xs, pp, pc, 4, 1020, out, ss, None) == -1       # H % 8
    assert L.mhc_post_int8(R, q, xs, pp, pc, 4, 1024, out, R, None) == -1        # sqrsum overlaps R
    assert L.mhc_post_sqrsum(R, q, pp, pc, 4, 1024, out, None, None) == -1       # sqrsum required
    assert L.mhc_post_int8(R, q, xs, pp, pc, 0, 1024, out, ss, None) == 0


def test_pre_broadcast_argument_checks(mhc_lib):
    L = mhc_lib.lib()
    x, phi, bias, ms, g = ins(5)
    Ro, X, pre, post, res = ins(5, 0x200000000000)
    ws = P(0x7000000000)
    assert L.mhc_pre_broadcast(x, phi, bias, ms, g, 4, 1024, *SC[:4], SC[4], None, X, pre, post, res, ws,
                               1 << 30, None) == -1                                # residual_out required
    assert L.mhc_pre_broadcast(x, phi, bias, ms, g, 4, 1024, *SC[:4], SC[4], x, X, pre, post, res, ws,
                               1 << 30, None) == -1                                # output overlaps x
    assert L.mhc_pre_broadcast(x, phi, bias, ms, g, 4, 1024, *SC[:4], SC[4], Ro, Ro, pre, post, res, ws,
                               1 << 30, None) == -1                                # outputs overlap
    assert L.mhc_pre_broadcast(x, phi, bias, ms, g, 4, 1024, *SC[:4], SC[4], Ro, X, pre, post, res, ws,
                               16, None) == -3                                     # workspace too small


def test_broadcast_schedule_is_refused_where_it_cannot_run(mhc_lib):
    """The fused broadcast schedule needs H % 64 == 0: forced on another H, mhc_pre_broadcast
    refuses the call (MHC_ERR_UNSUPPORTED) before it touches the device.  The schedule id is
    accepted, and the other calls treat it as AUTO."""
    L = mhc_lib.lib()
    x, phi, bias, ms, g = ins(5)
    Ro, X, pre, post, res = ins(5, 0x200000000000)
    ws = P(0x7000000000)
    assert L.mhc_set_schedule(10) == 0
    try:
        assert L.mhc_pre_broadcast(x, phi, bias, ms, g, 40, 1032, *SC[:4], SC[4], Ro, X, pre, post, res, ws,
                                   1 << 30, None) == -2
    finally:
        assert L.mhc_set_schedule(0) == 0
    assert L.mhc_set_schedule(12) == -1                                           # unknown schedule


def test_workspace_covers_the_broadcast_kernel(mhc_lib):
    """The workspace holds the packed phi_sum fragments (96 bytes per hidden value, in 16-value
    steps) and the residual-mix logits (64 bytes per token) after the 256-byte control block."""
    L = mhc_lib.lib()
    L.mhc_workspace_size.restype = ctypes.c_size_t
    for T, H in [(33, 1024), (8192, 7168), (65536, 7168), (300, 1088)]:
        need = 256 + (((H + 15) // 16 * 1536 + 255) // 256 * 256) + T * 64
        assert L.mhc_workspace_size(T, H) >= need


def test_split_argument_checks(mhc_lib):
    L = mhc_lib.lib()
    p = ins(8)
    outs = ins(5, 0x200000000000)
    ws = P(0x7000000000)
    side, f, j = P(0x1234), P(0x5678), P(0x9abc)
    common = (*p, 4, 1024, *SC[:4], SC[4], *outs, ws, 1 << 30)
    assert L.mhc_shifted_post_pre_split(*common, None, side, None, j) == -1       # no fork event
    assert L.mhc_shifted_post_pre_split(*common, None, side, f, None) == -1       # no join event
    assert L.mhc_shifted_post_pre_split(*common, side, side, f, j) == -1          # side == main stream


def test_bench_byte_counts_match_the_scope_table():
    """The per-call algorithmic bytes: 20H + 176 per token plus phi (fp32 [4H, 24]), gamma and
    the scalars per call: 3.63 MB for T=6 and 1.1786 GB for T=8192 at H=7168."""
    import importlib.util
    import os
    spec = importlib.util.spec_from_file_location(
        "bench", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.algorithmic_bytes(6, 7168) == 6 * 143536 + 4 * 7168 * 24 * 4 + 2 * 7168 + 108
    assert abs(bench.algorithmic_bytes(6, 7168) / 1e6 - 3.63) < 0.005
    assert abs(bench.algorithmic_bytes(8192, 7168) / 1e9 - 1.1786) < 0.0001
    assert bench.algorithmic_bytes(8192, 7168, True) - bench.algorithmic_bytes(8192, 7168) == 8192 * (7168 + 224)


def test_removed_schedule_ids_are_refused(mhc_lib):
    """Ids 2-7 named the cluster and pipelined schedules that ws superseded; they are gone."""
    L = mhc_lib.lib()
    for sid in range(2, 8):
        assert L.mhc_set_schedule(sid) == -1
    for sid in (0, 1, 8, 9, 10, 11):
        assert L.mhc_set_schedule(sid) == 0
    assert L.mhc_set_schedule(0) == 0


def test_noalloc_negative_sizes_are_refused_with_a_message(mhc_lib):
    L = mhc_lib.lib()
    P_, I64, F_, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    L.mhc_shifted_post_pre_noalloc.argtypes = [P_] * 8 + [I64, I64, F_, F_, F_, F_, I] + [P_] * 6
    L.mhc_shifted_post_pre_noalloc.restype = I
    p = ins(8)
    outs = ins(5, 0x200000000000)
    assert L.mhc_set_schedule(999) == -1  # leaves an unrelated message behind
    for T, H in ((-1, 1024), (4, -8)):
        assert L.mhc_shifted_post_pre_noalloc(*p, T, H, *SC[:4], SC[4], *outs, None) == -1
        assert b"must not be negative" in L.mhc_last_error()


def test_pack_phi_argument_checks_and_size(mhc_lib):
    """mhc_packed_phi_bytes: 16 CTA slices of ceil(H / 1024) * 64 hidden values, each 4 * slice / 16
    k16 steps of three 512-byte fragment tiles (hi and lo bf16 of phi^T); bad calls are refused
    before any device work."""
    L = mhc_lib.lib()
    Z, I64 = ctypes.c_size_t, ctypes.c_int64
    L.mhc_packed_phi_bytes.argtypes = [I64]
    L.mhc_packed_phi_bytes.restype = Z
    L.mhc_pack_phi.argtypes = [ctypes.c_void_p, I64, ctypes.c_void_p, Z, ctypes.c_void_p]
    for H in (1024, 4096, 7168, 2056):
        hs = (H + 1023) // 1024 * 64
        assert L.mhc_packed_phi_bytes(H) == 16 * (4 * hs // 16) * 3 * 512
    assert L.mhc_packed_phi_bytes(1020) == 0 and L.mhc_packed_phi_bytes(0) == 0
    phi, out = P(0x100000000), P(0x200000000000)
    n = L.mhc_packed_phi_bytes(7168)
    assert L.mhc_pack_phi(phi, 7168, out, n - 16, None) == -1       # too small
    assert L.mhc_pack_phi(None, 7168, out, n, None) == -1            # no phi
    assert L.mhc_pack_phi(phi, 7168, None, n, None) == -1            # no output
    assert L.mhc_pack_phi(phi, 7168, P(0x100000010), n, None) == -1  # overlaps phi
    assert L.mhc_pack_phi(phi, 1020, out, n, None) == -1             # H % 8
