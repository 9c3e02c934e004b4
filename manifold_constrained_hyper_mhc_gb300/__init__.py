"""Python binding of libmhc.so, the GB300 fused mHC post+pre library.

Argument marshalling only: every step of the op runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  The library must be
built (``_build.build()``); importing the binding without it, or calling it
without a CUDA device, raises -- there is no CPU fallback.

Names follow the C ABI in ``include/mhc.h`` (mhc_shifted_post_pre, mhc_post,
mhc_pre), which follows "[DSv4.1] Integrate Mega-mHC from DeepGEMM".
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "MhcError", "lib", "workspace_size", "new_workspace", "shifted_post_pre", "post", "pre",
    "set_schedule", "auto_schedule", "auto_side_tokens", "check_status", "last_launch_count", "SCHEDULES",
    "post_int8", "post_sqrsum", "pre_broadcast", "shifted_post_pre_split", "shifted_post_pre_mxfp8", "mxfp8_scale_bytes", "MX_SCALE_FLOOR", "MX_SCALE_CEIL", "set_main_kernel_events",
    "packed_phi_bytes", "pack_phi",
]
MX_SCALE_FLOOR, MX_SCALE_CEIL = 0, 1

OK = 0
STATUS = {0: "MHC_OK", -1: "MHC_ERR_INVALID_ARG", -2: "MHC_ERR_UNSUPPORTED", -3: "MHC_ERR_WORKSPACE",
          -4: "MHC_ERR_CUDA", -5: "MHC_ERR_DEVICE_TIMEOUT"}
SCHEDULES = {"auto": 0, "split": 1, "ws": 8, "small": 9, "bcast": 10, "tile": 11}


class MhcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = lib().mhc_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS.get(status, status)} ({detail})")


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded C library (ctypes).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise ImportError(f"libmhc.so not built at {path}; run manifold_constrained_hyper_mhc_gb300._build.build()")
            L = ctypes.CDLL(path)
            P, I64, F, I, Z = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
            L.mhc_workspace_size.argtypes = [I64, I64]
            L.mhc_workspace_size.restype = Z
            L.mhc_shifted_post_pre.argtypes = [P, P, P, P, P, P, P, P, I64, I64, F, F, F, F, I,
                                               P, P, P, P, P, P, Z, P]
            L.mhc_shifted_post_pre.restype = I
            L.mhc_shifted_post_pre_mxfp8.argtypes = [P, P, P, P, P, P, P, P, I64, I64, F, F, F, F, I,
                                                     P, P, P, P, I, P, P, P, P, Z, P]
            L.mhc_shifted_post_pre_mxfp8.restype = I
            L.mhc_mxfp8_scale_bytes.argtypes = [I64, I64]
            L.mhc_mxfp8_scale_bytes.restype = Z
            L.mhc_post_int8.argtypes = [P, P, P, P, P, I64, I64, P, P, P]
            L.mhc_post_int8.restype = I
            L.mhc_post_sqrsum.argtypes = [P, P, P, P, I64, I64, P, P, P]
            L.mhc_post_sqrsum.restype = I
            L.mhc_pre_broadcast.argtypes = [P, P, P, P, P, I64, I64, F, F, F, F, I, P, P, P, P, P, P, Z, P]
            L.mhc_pre_broadcast.restype = I
            L.mhc_shifted_post_pre_split.argtypes = [P, P, P, P, P, P, P, P, I64, I64, F, F, F, F, I,
                                                     P, P, P, P, P, P, Z, P, P, P, P]
            L.mhc_shifted_post_pre_split.restype = I
            L.mhc_packed_phi_bytes.argtypes = [I64]
            L.mhc_packed_phi_bytes.restype = Z
            L.mhc_pack_phi.argtypes = [P, I64, P, Z, P]
            L.mhc_pack_phi.restype = I
            L.mhc_shifted_post_pre_prepacked.argtypes = [P, P, P, P, P, P, P, P, P, I64, I64, F, F, F, F, I,
                                                         P, P, P, P, P, P, Z, P]
            L.mhc_shifted_post_pre_prepacked.restype = I
            L.mhc_pre_prepacked.argtypes = [P, P, P, P, P, P, I64, I64, F, F, F, F, I, P, P, P, P, P, Z, P]
            L.mhc_pre_prepacked.restype = I
            L.mhc_shifted_post_pre_mxfp8_prepacked.argtypes = [P, P, P, P, P, P, P, P, P, I64, I64, F, F, F, F, I,
                                                               P, P, P, P, I, P, P, P, P, Z, P]
            L.mhc_shifted_post_pre_mxfp8_prepacked.restype = I
            L.mhc_post.argtypes = [P, P, P, P, I64, I64, P, P]
            L.mhc_post.restype = I
            L.mhc_pre.argtypes = [P, P, P, P, P, I64, I64, F, F, F, F, I, P, P, P, P, P, Z, P]
            L.mhc_pre.restype = I
            L.mhc_set_schedule.argtypes = [I]
            L.mhc_set_schedule.restype = I
            L.mhc_auto_schedule.argtypes = [I64, I64]
            L.mhc_auto_schedule.restype = I
            L.mhc_auto_side_tokens.argtypes = [I64, I64, I]
            L.mhc_auto_side_tokens.restype = I64
            L.mhc_check_status.argtypes = [P, P]
            L.mhc_check_status.restype = I
            L.mhc_status_string.argtypes = [I]
            L.mhc_status_string.restype = ctypes.c_char_p
            L.mhc_last_launch_count.argtypes = []
            L.mhc_last_launch_count.restype = I
            L.mhc_set_main_kernel_events.argtypes = [P, P]
            L.mhc_set_main_kernel_events.restype = None
            L.mhc_last_error.argtypes = []
            L.mhc_last_error.restype = ctypes.c_char_p
            _lib = L
    return _lib


_torch_mod = None


def _torch():
    global _torch_mod
    if _torch_mod is None:
        import torch
        _torch_mod = torch
    return _torch_mod


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc, where):
    if rc != OK:
        raise MhcError(rc, where)


def workspace_size(T: int, H: int) -> int:
    return int(lib().mhc_workspace_size(int(T), int(H)))


def new_workspace(T: int, H: int, device=None):
    """A zero-filled workspace (uint8 tensor) for calls with up to T tokens of size H."""
    torch = _torch()
    return torch.zeros(max(workspace_size(T, H), 256), dtype=torch.uint8, device=device or "cuda")


# The checks below run on every call, so they stay cheap: a torch.Size compares equal to a tuple.
def _bf16(t, name, shape):
    torch = _torch()
    if t.dtype != torch.bfloat16 and t.dtype != torch.int16 and t.dtype != torch.uint16:
        raise TypeError(f"{name} must be bfloat16 (or its 16-bit bit pattern), got {t.dtype}")
    if t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


def _f32(t, name, shape):
    torch = _torch()
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


def _outputs(T, H, device, out, with_residual):
    """The output dict: the caller's tensors, and new ones only for the keys it left out."""
    torch = _torch()
    out = dict(out or {})
    shapes = ((("residual_out", (T, 4, H), torch.bfloat16),) if with_residual else ()) + (
        ("layer_in", (T, H), torch.bfloat16), ("pre_mix", (T, 4), torch.float32),
        ("post_mix", (T, 4), torch.float32), ("comb_res_mix", (T, 4, 4), torch.float32))
    for k, shape, dtype in shapes:
        if k not in out:
            out[k] = torch.empty(shape, dtype=dtype, device=device)
    return out


def packed_phi_bytes(H: int) -> int:
    return int(lib().mhc_packed_phi_bytes(int(H)))


def pack_phi(phi, *, out=None, stream=None):
    """mhc_pack_phi: phi [4H, 24] fp32 in the packed form the fused kernels read (a uint8 tensor of
    packed_phi_bytes(H) bytes), for the packed_phi argument of shifted_post_pre and pre."""
    torch = _torch()
    H = phi.shape[0] // 4
    _f32(phi, "phi", (4 * H, 24))
    n = packed_phi_bytes(H)
    o = out if out is not None else torch.empty(max(n, 16), dtype=torch.uint8, device=phi.device)
    _check(lib().mhc_pack_phi(_ptr(phi), H, _ptr(o), o.numel() * o.element_size(), _stream(stream, phi.device)),
           "mhc_pack_phi")
    return o


def shifted_post_pre(residual, layer_out, prev_post_mix, prev_comb_res_mix, phi, bias, mix_scales,
                     rmsnorm_weight, *, hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps,
                     sinkhorn_iters=20, out=None, workspace=None, stream=None, packed_phi=None):
    """mhc_shifted_post_pre: the fused post+pre step.  Returns a dict with
    residual_out [T,4,H] bf16, layer_in [T,H] bf16, pre_mix [T,4], post_mix [T,4],
    comb_res_mix [T,4,4] (fp32).  ``out`` may supply preallocated outputs; with ``packed_phi``
    (pack_phi(phi)) it calls mhc_shifted_post_pre_prepacked (same results, no packing launch)."""
    T, _, H = residual.shape
    _bf16(residual, "residual", (T, 4, H)); _bf16(layer_out, "layer_out", (T, H))
    _f32(prev_post_mix, "prev_post_mix", (T, 4)); _f32(prev_comb_res_mix, "prev_comb_res_mix", (T, 4, 4))
    _f32(phi, "phi", (4 * H, 24)); _f32(bias, "bias", (24,)); _f32(mix_scales, "mix_scales", (3,))
    _bf16(rmsnorm_weight, "rmsnorm_weight", (H,))
    dev = residual.device
    o = _outputs(T, H, dev, out, True)
    ws = workspace if workspace is not None else new_workspace(T, H, dev)
    if packed_phi is not None:
        rc = lib().mhc_shifted_post_pre_prepacked(
            _ptr(residual), _ptr(layer_out), _ptr(prev_post_mix), _ptr(prev_comb_res_mix), _ptr(phi),
            _ptr(packed_phi), _ptr(bias), _ptr(mix_scales), _ptr(rmsnorm_weight), T, H, hc_norm_eps, rmsnorm_eps,
            hc_post_scale, sinkhorn_eps, int(sinkhorn_iters), _ptr(o["residual_out"]), _ptr(o["layer_in"]),
            _ptr(o["pre_mix"]), _ptr(o["post_mix"]), _ptr(o["comb_res_mix"]), _ptr(ws),
            ws.numel() * ws.element_size(), _stream(stream, dev))
        _check(rc, "mhc_shifted_post_pre_prepacked")
        return o
    rc = lib().mhc_shifted_post_pre(
        _ptr(residual), _ptr(layer_out), _ptr(prev_post_mix), _ptr(prev_comb_res_mix), _ptr(phi),
        _ptr(bias), _ptr(mix_scales), _ptr(rmsnorm_weight), T, H, hc_norm_eps, rmsnorm_eps,
        hc_post_scale, sinkhorn_eps, int(sinkhorn_iters), _ptr(o["residual_out"]), _ptr(o["layer_in"]),
        _ptr(o["pre_mix"]), _ptr(o["post_mix"]), _ptr(o["comb_res_mix"]), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream, dev))
    _check(rc, "mhc_shifted_post_pre")
    return o


def shifted_post_pre_split(residual, layer_out, prev_post_mix, prev_comb_res_mix, phi, bias, mix_scales,
                           rmsnorm_weight, *, side_stream, fork_event, join_event, hc_norm_eps, rmsnorm_eps,
                           hc_post_scale, sinkhorn_eps, sinkhorn_iters=20, out=None, workspace=None, stream=None):
    """mhc_shifted_post_pre_split: the fused step with the post and residual mixes computed on
    side_stream (torch.cuda.Stream); fork_event / join_event are torch.cuda.Event objects (already
    created, e.g. recorded once).  Wait on join_event before reading post_mix / comb_res_mix or
    reusing the workspace."""
    T, _, H = residual.shape
    _bf16(residual, "residual", (T, 4, H)); _bf16(layer_out, "layer_out", (T, H))
    _f32(prev_post_mix, "prev_post_mix", (T, 4)); _f32(prev_comb_res_mix, "prev_comb_res_mix", (T, 4, 4))
    _f32(phi, "phi", (4 * H, 24)); _f32(bias, "bias", (24,)); _f32(mix_scales, "mix_scales", (3,))
    _bf16(rmsnorm_weight, "rmsnorm_weight", (H,))
    dev = residual.device
    o = _outputs(T, H, dev, out, True)
    ws = workspace if workspace is not None else new_workspace(T, H, dev)
    rc = lib().mhc_shifted_post_pre_split(
        _ptr(residual), _ptr(layer_out), _ptr(prev_post_mix), _ptr(prev_comb_res_mix), _ptr(phi),
        _ptr(bias), _ptr(mix_scales), _ptr(rmsnorm_weight), T, H, hc_norm_eps, rmsnorm_eps,
        hc_post_scale, sinkhorn_eps, int(sinkhorn_iters), _ptr(o["residual_out"]), _ptr(o["layer_in"]),
        _ptr(o["pre_mix"]), _ptr(o["post_mix"]), _ptr(o["comb_res_mix"]), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream, dev), ctypes.c_void_p(side_stream.cuda_stream),
        ctypes.c_void_p(fork_event.cuda_event), ctypes.c_void_p(join_event.cuda_event))
    _check(rc, "mhc_shifted_post_pre_split")
    return o


def mxfp8_scale_bytes(T: int, H: int) -> int:
    return int(lib().mhc_mxfp8_scale_bytes(int(T), int(H)))


def shifted_post_pre_mxfp8(residual, layer_out, prev_post_mix, prev_comb_res_mix, phi, bias, mix_scales,
                           rmsnorm_weight, *, hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps,
                           sinkhorn_iters=20, scale_mode=MX_SCALE_FLOOR, want_bf16=True, out=None,
                           workspace=None, stream=None, packed_phi=None):
    """mhc_shifted_post_pre_mxfp8: the fused step with the layer input also as MXFP8.  Returns the
    dict of shifted_post_pre (layer_in only if want_bf16) plus layer_in_fp8 [T,H] uint8 (E4M3
    codes) and layer_in_scales (uint8, mxfp8_scale_bytes(T, H), 128x4 tile layout).  With
    packed_phi (pack_phi's output for this phi) it calls mhc_shifted_post_pre_mxfp8_prepacked."""
    torch = _torch()
    T, _, H = residual.shape
    _bf16(residual, "residual", (T, 4, H)); _bf16(layer_out, "layer_out", (T, H))
    _f32(prev_post_mix, "prev_post_mix", (T, 4)); _f32(prev_comb_res_mix, "prev_comb_res_mix", (T, 4, 4))
    _f32(phi, "phi", (4 * H, 24)); _f32(bias, "bias", (24,)); _f32(mix_scales, "mix_scales", (3,))
    _bf16(rmsnorm_weight, "rmsnorm_weight", (H,))
    dev = residual.device
    o = dict(out or {})
    if not want_bf16:
        o.setdefault("layer_in", None)
    o = _outputs(T, H, dev, o, True)
    if "layer_in_fp8" not in o:
        o["layer_in_fp8"] = torch.empty((T, H), dtype=torch.uint8, device=dev)
    if "layer_in_scales" not in o:
        o["layer_in_scales"] = torch.empty(max(mxfp8_scale_bytes(T, H), 1), dtype=torch.uint8, device=dev)
    ws = workspace if workspace is not None else new_workspace(T, H, dev)
    head = (_ptr(residual), _ptr(layer_out), _ptr(prev_post_mix), _ptr(prev_comb_res_mix), _ptr(phi))
    tail = (_ptr(bias), _ptr(mix_scales), _ptr(rmsnorm_weight), T, H, hc_norm_eps, rmsnorm_eps,
            hc_post_scale, sinkhorn_eps, int(sinkhorn_iters), _ptr(o["residual_out"]), _ptr(o["layer_in"]),
            _ptr(o["layer_in_fp8"]), _ptr(o["layer_in_scales"]), int(scale_mode), _ptr(o["pre_mix"]),
            _ptr(o["post_mix"]), _ptr(o["comb_res_mix"]), _ptr(ws), ws.numel() * ws.element_size(),
            _stream(stream, dev))
    if packed_phi is None:
        rc = lib().mhc_shifted_post_pre_mxfp8(*head, *tail)
        _check(rc, "mhc_shifted_post_pre_mxfp8")
    else:
        rc = lib().mhc_shifted_post_pre_mxfp8_prepacked(*head, _ptr(packed_phi), *tail)
        _check(rc, "mhc_shifted_post_pre_mxfp8_prepacked")
    return o


def post(residual, layer_out, prev_post_mix, prev_comb_res_mix, *, out=None, stream=None):
    """mhc_post: step (1) only.  Returns residual_out [T,4,H] bf16."""
    torch = _torch()
    T, _, H = residual.shape
    _bf16(residual, "residual", (T, 4, H)); _bf16(layer_out, "layer_out", (T, H))
    _f32(prev_post_mix, "prev_post_mix", (T, 4)); _f32(prev_comb_res_mix, "prev_comb_res_mix", (T, 4, 4))
    o = out if out is not None else torch.empty((T, 4, H), dtype=torch.bfloat16, device=residual.device)
    rc = lib().mhc_post(_ptr(residual), _ptr(layer_out), _ptr(prev_post_mix), _ptr(prev_comb_res_mix),
                        T, H, _ptr(o), _stream(stream, residual.device))
    _check(rc, "mhc_post")
    return o


def post_int8(residual, layer_out_q, x_scales, prev_post_mix, prev_comb_res_mix, *, sqrsum=True, out=None,
              stream=None):
    """mhc_post_int8: step (1) from an int8 layer output (codes [T,H] int8, x_scales [T] fp32).
    Returns (residual_out [T,4,H] bf16, sqrsum [T] fp32 or None)."""
    torch = _torch()
    T, _, H = residual.shape
    _bf16(residual, "residual", (T, 4, H))
    if layer_out_q.dtype != torch.int8 or tuple(layer_out_q.shape) != (T, H) or not layer_out_q.is_contiguous():
        raise TypeError("layer_out_q must be a contiguous int8 [T, H] tensor")
    _f32(x_scales, "x_scales", (T,))
    _f32(prev_post_mix, "prev_post_mix", (T, 4)); _f32(prev_comb_res_mix, "prev_comb_res_mix", (T, 4, 4))
    o = out if out is not None else torch.empty((T, 4, H), dtype=torch.bfloat16, device=residual.device)
    ss = torch.empty(T, dtype=torch.float32, device=residual.device) if sqrsum else None
    rc = lib().mhc_post_int8(_ptr(residual), _ptr(layer_out_q), _ptr(x_scales), _ptr(prev_post_mix),
                             _ptr(prev_comb_res_mix), T, H, _ptr(o), _ptr(ss), _stream(stream, residual.device))
    _check(rc, "mhc_post_int8")
    return o, ss


def post_sqrsum(residual, layer_out, prev_post_mix, prev_comb_res_mix, *, out=None, stream=None):
    """mhc_post_sqrsum: mhc_post plus the square sum of R' per token.  Returns (residual_out, sqrsum)."""
    torch = _torch()
    T, _, H = residual.shape
    _bf16(residual, "residual", (T, 4, H)); _bf16(layer_out, "layer_out", (T, H))
    _f32(prev_post_mix, "prev_post_mix", (T, 4)); _f32(prev_comb_res_mix, "prev_comb_res_mix", (T, 4, 4))
    o = out if out is not None else torch.empty((T, 4, H), dtype=torch.bfloat16, device=residual.device)
    ss = torch.empty(max(T, 1), dtype=torch.float32, device=residual.device)[:T]
    rc = lib().mhc_post_sqrsum(_ptr(residual), _ptr(layer_out), _ptr(prev_post_mix), _ptr(prev_comb_res_mix),
                               T, H, _ptr(o), _ptr(ss), _stream(stream, residual.device))
    _check(rc, "mhc_post_sqrsum")
    return o, ss


def pre(residual, phi, bias, mix_scales, rmsnorm_weight, *, hc_norm_eps, rmsnorm_eps, hc_post_scale,
        sinkhorn_eps, sinkhorn_iters=20, out=None, workspace=None, stream=None, packed_phi=None):
    """mhc_pre: steps (2)-(4) from post-updated streams.  Returns the fused call's
    outputs without residual_out.  With ``packed_phi`` it calls mhc_pre_prepacked."""
    T, _, H = residual.shape
    _bf16(residual, "residual", (T, 4, H))
    _f32(phi, "phi", (4 * H, 24)); _f32(bias, "bias", (24,)); _f32(mix_scales, "mix_scales", (3,))
    _bf16(rmsnorm_weight, "rmsnorm_weight", (H,))
    dev = residual.device
    o = _outputs(T, H, dev, out, False)
    ws = workspace if workspace is not None else new_workspace(T, H, dev)
    if packed_phi is not None:
        rc = lib().mhc_pre_prepacked(_ptr(residual), _ptr(phi), _ptr(packed_phi), _ptr(bias), _ptr(mix_scales),
                                     _ptr(rmsnorm_weight), T, H, hc_norm_eps, rmsnorm_eps, hc_post_scale,
                                     sinkhorn_eps, int(sinkhorn_iters), _ptr(o["layer_in"]), _ptr(o["pre_mix"]),
                                     _ptr(o["post_mix"]), _ptr(o["comb_res_mix"]), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream, dev))
        _check(rc, "mhc_pre_prepacked")
        return o
    rc = lib().mhc_pre(_ptr(residual), _ptr(phi), _ptr(bias), _ptr(mix_scales), _ptr(rmsnorm_weight),
                       T, H, hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, int(sinkhorn_iters),
                       _ptr(o["layer_in"]), _ptr(o["pre_mix"]), _ptr(o["post_mix"]),
                       _ptr(o["comb_res_mix"]), _ptr(ws), ws.numel() * ws.element_size(),
                       _stream(stream, dev))
    _check(rc, "mhc_pre")
    return o


def pre_broadcast(x, phi, bias, mix_scales, rmsnorm_weight, *, hc_norm_eps, rmsnorm_eps, hc_post_scale,
                  sinkhorn_eps, sinkhorn_iters=20, out=None, workspace=None, stream=None):
    """mhc_pre_broadcast: the first layer's pre from the (T, H) input x.  Returns the dict of
    pre() plus residual_out [T,4,H] (four copies of x).  For T > 32 with H % 64 == 0 (or the
    "bcast" schedule forced) one kernel works from x alone; otherwise the residual is written
    and pre() runs on it."""
    T, H = x.shape
    _bf16(x, "x", (T, H))
    _f32(phi, "phi", (4 * H, 24)); _f32(bias, "bias", (24,)); _f32(mix_scales, "mix_scales", (3,))
    _bf16(rmsnorm_weight, "rmsnorm_weight", (H,))
    dev = x.device
    o = _outputs(T, H, dev, out, True)
    ws = workspace if workspace is not None else new_workspace(T, H, dev)
    rc = lib().mhc_pre_broadcast(_ptr(x), _ptr(phi), _ptr(bias), _ptr(mix_scales), _ptr(rmsnorm_weight), T, H,
                                 hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, int(sinkhorn_iters),
                                 _ptr(o["residual_out"]), _ptr(o["layer_in"]), _ptr(o["pre_mix"]),
                                 _ptr(o["post_mix"]), _ptr(o["comb_res_mix"]), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream, dev))
    _check(rc, "mhc_pre_broadcast")
    return o


def set_schedule(name_or_id):
    sid = SCHEDULES[name_or_id] if isinstance(name_or_id, str) else int(name_or_id)
    _check(lib().mhc_set_schedule(sid), "mhc_set_schedule")


def auto_schedule(T: int, H: int) -> int:
    return int(lib().mhc_auto_schedule(int(T), int(H)))


def auto_side_tokens(T: int, H: int, fused: bool = True) -> int:
    """How many trailing tokens of an AUTO call (fused: shifted_post_pre; else pre) the token-tile
    kernel takes beside ws (0: ws alone or another schedule); -1 without a CUDA device."""
    return int(lib().mhc_auto_side_tokens(int(T), int(H), 1 if fused else 0))


def last_launch_count() -> int:
    """Kernels launched by the last library call on this thread."""
    return int(lib().mhc_last_launch_count())


def set_main_kernel_events(start=None, stop=None):
    """Measurement hook: record these torch.cuda.Event objects around each call's main kernel
    (None, None turns it off)."""
    lib().mhc_set_main_kernel_events(None if start is None else ctypes.c_void_p(start.cuda_event),
                                     None if stop is None else ctypes.c_void_p(stop.cuda_event))


def check_status(workspace, stream=None):
    """Synchronises the stream and raises MhcError if a device-side wait timed out."""
    _check(lib().mhc_check_status(_ptr(workspace), _stream(stream, workspace.device)), "mhc_check_status")
