"""CPU-only checks of the C-ABI library: it builds, loads, exports every symbol
include/mhc.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    txt = open(os.path.join(ROOT, "include", "mhc.h")).read()
    return sorted(set(re.findall(r"MHC_API\s+[\w\s\*]*?\b(mhc_\w+)\s*\(", txt)))


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for n in ("mhc_shifted_post_pre", "mhc_post", "mhc_pre", "mhc_workspace_size",
              "mhc_status_string", "mhc_check_status", "mhc_set_schedule", "mhc_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(mhc_lib):
    L = mhc_lib.lib()
    for n in _declared_symbols():
        assert hasattr(L, n), n


def test_status_strings(mhc_lib):
    L = mhc_lib.lib()
    for code, name in mhc_lib.STATUS.items():
        assert L.mhc_status_string(code).decode().startswith(name)
    assert L.mhc_status_string(12345) is not None


def test_workspace_size_grows_with_tokens(mhc_lib):
    a = mhc_lib.workspace_size(1, 1024)
    b = mhc_lib.workspace_size(1000, 1024)
    assert a >= 256 and b > a and a % 256 == 0 and b % 256 == 0
    assert mhc_lib.workspace_size(-1, 8) == 0


def _fake(addr):
    return ctypes.c_void_p(addr)


def _call_fused(L, T, H, ptrs=None, scal=(2e-5, 2e-6, 1.25, 3e-4, 20), ws_bytes=1 << 30, ws=0x7000000000):
    base = 0x100000000
    p = [_fake(base + i * (1 << 36)) for i in range(8)] if ptrs is None else ptrs
    outs = [_fake(0x200000000000 + i * (1 << 36)) for i in range(5)]
    return L.mhc_shifted_post_pre(*p, T, H, *scal[:4], scal[4], *outs, _fake(ws), ws_bytes, None)


@pytest.mark.parametrize("T,H", [(-1, 1024), ((1 << 20) + 1, 1024), (1 << 23, 1024), (4, 0), (4, 12), (4, 65544), (4, 4)])
def test_bad_sizes_are_rejected(mhc_lib, T, H):
    assert _call_fused(mhc_lib.lib(), T, H) == -1


@pytest.mark.parametrize("scal", [(-1e-5, 2e-6, 1.25, 3e-4, 20), (2e-5, float("nan"), 1.25, 3e-4, 20),
                                  (2e-5, 2e-6, float("inf"), 3e-4, 20), (2e-5, 2e-6, 1.25, -3e-4, 20),
                                  (2e-5, 2e-6, 1.25, 3e-4, -1), (2e-5, 2e-6, 1.25, 3e-4, 65)])
def test_bad_scalars_are_rejected(mhc_lib, scal):
    assert _call_fused(mhc_lib.lib(), 4, 1024, scal=scal) == -1


def test_empty_input_is_a_no_op(mhc_lib):
    L = mhc_lib.lib()
    nulls = [None] * 8
    assert L.mhc_shifted_post_pre(*nulls, 0, 1024, 2e-5, 2e-6, 1.25, 3e-4, 20,
                                  None, None, None, None, None, None, 0, None) == 0
    assert L.mhc_post(None, None, None, None, 0, 64, None, None) == 0


def test_null_and_misaligned_pointers_are_rejected(mhc_lib):
    L = mhc_lib.lib()
    base = [_fake(0x100000000 + i * (1 << 36)) for i in range(8)]
    for k in range(8):
        p = list(base)
        p[k] = None
        assert _call_fused(L, 4, 1024, ptrs=p) == -1
        p[k] = _fake(base[k].value + 8)
        assert _call_fused(L, 4, 1024, ptrs=p) == -1
    assert "aligned" in L.mhc_last_error().decode()


def test_workspace_errors(mhc_lib):
    L = mhc_lib.lib()
    assert _call_fused(L, 4, 1024, ws=0) == -3
    assert _call_fused(L, 4, 1024, ws=0x7000000010) == -3
    assert _call_fused(L, 4096, 7168, ws_bytes=1024) == -3


def test_overlapping_output_is_rejected(mhc_lib):
    L = mhc_lib.lib()
    base = [_fake(0x100000000 + i * (1 << 36)) for i in range(8)]
    outs = [_fake(0x200000000000 + i * (1 << 36)) for i in range(5)]
    outs[1] = _fake(base[1].value + 64)   # layer_in_out inside layer_out
    rc = L.mhc_shifted_post_pre(*base, 4, 1024, 2e-5, 2e-6, 1.25, 3e-4, 20, *outs,
                                _fake(0x7000000000), 1 << 30, None)
    assert rc == -1 and "overlap" in L.mhc_last_error().decode()


def test_unknown_schedule_is_rejected(mhc_lib):
    L = mhc_lib.lib()
    assert L.mhc_set_schedule(999) == -1
    assert L.mhc_set_schedule(0) == 0


def test_binding_fails_loudly_without_cuda(mhc_lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    x = torch.zeros((2, 4, 64), dtype=torch.bfloat16)
    with pytest.raises((ValueError, RuntimeError)):
        mhc_lib.post(x, torch.zeros((2, 64), dtype=torch.bfloat16), torch.zeros((2, 4)),
                     torch.zeros((2, 4, 4)))


def test_planning_queries_without_a_device(mhc_lib):
    """The AUTO planning queries need a current CUDA device; without one (this CPU machine) they say so
    instead of guessing: the side share is -1, and bad sizes are -1 as well."""
    L = mhc_lib.lib()
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a CUDA device is present")
    except ImportError:
        pass
    assert mhc_lib.auto_side_tokens(8192, 7168) == -1
    assert L.mhc_auto_side_tokens(-1, 7168, 1) == -1
