"""ctypes shim over the CPU oracle (``mhc_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline / reference leg load this; the library never does.  It shares no
code with the CUDA path; the only thing both sides share is the seeded input
generator, which holds none of the op's arithmetic.

Parity pins: every oracle function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, invariants, special cases that
reduce to a library routine, hand-derived worked examples under
``tests/golden/``).  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mhc_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmhc_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math) into oracle/_build/."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64, D, I = ctypes.c_int64, ctypes.c_double, ctypes.c_int
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = D
            lib.oracle_double_to_bf16.argtypes = [D]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            lib.oracle_sinkhorn.argtypes = [P, I, D]
            lib.oracle_sinkhorn.restype = None
            lib.oracle_post.argtypes = [P, P, P, P, I64, I64, P, I]
            lib.oracle_post.restype = I
            lib.oracle_pre.argtypes = [P, P, P, P, P, I64, I64, D, D, D, D, I,
                                       P, P, P, P, P, P, P, I]
            lib.oracle_pre.restype = I
            lib.oracle_shifted_post_pre.argtypes = [P, P, P, P, P, P, P, P, I64, I64,
                                                    D, D, D, D, I, P, P, P, P, P, P, P, P, I]
            lib.oracle_shifted_post_pre.restype = I
            lib.oracle_e4m3_encode.argtypes = [D]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = D
            lib.oracle_mx_scale_exp.argtypes = [D, I]
            lib.oracle_mx_scale_exp.restype = I
            lib.oracle_mx_scale_offset.argtypes = [I64, I64, I64]
            lib.oracle_mx_scale_offset.restype = I64
            lib.oracle_mxfp8_quantize.argtypes = [P, I64, I64, I, P, P]
            lib.oracle_mxfp8_quantize.restype = I
            lib.oracle_post_ex.argtypes = [P, P, P, P, P, P, I64, I64, P, P]
            lib.oracle_post_ex.restype = I
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def default_threads() -> int:
    return os.cpu_count() or 1


def bf16_to_double(b: int) -> float:
    return _load().oracle_bf16_to_double(int(b))


def double_to_bf16(x: float) -> int:
    return int(_load().oracle_double_to_bf16(float(x)))


def sinkhorn(M, iters: int, eps: float) -> np.ndarray:
    m = np.array(M, dtype=np.float64).reshape(16).copy()
    _load().oracle_sinkhorn(_p(m), int(iters), float(eps))
    return m.reshape(4, 4)


def post(R, Y, prev_post, prev_comb, nthreads: int | None = None):
    R = _c(R, np.uint16); Y = _c(Y, np.uint16)
    T, _, H = R.shape
    pp = _c(prev_post, np.float32); pc = _c(prev_comb, np.float32)
    out = np.empty_like(R)
    rc = _load().oracle_post(_p(R), _p(Y), _p(pp), _p(pc), T, H, _p(out),
                             nthreads or default_threads())
    assert rc == 0
    return out


def _sc(kw):
    return (float(kw["hc_norm_eps"]), float(kw["rmsnorm_eps"]), float(kw["hc_post_scale"]),
            float(kw["sinkhorn_eps"]), int(kw["sinkhorn_iters"]))


def pre(Rp, phi, bias, mix_scales, gamma, *, hc_norm_eps, rmsnorm_eps, hc_post_scale,
        sinkhorn_eps, sinkhorn_iters, nthreads: int | None = None, debug: bool = False):
    """Steps (2)-(4).  Returns dict with X (bf16 bits), pre, post, res (fp64) [+ z, r, rstd]."""
    Rp = _c(Rp, np.uint16)
    T, _, H = Rp.shape
    phi = _c(phi, np.float32); bias = _c(bias, np.float32)
    ms = _c(mix_scales, np.float32); g = _c(gamma, np.uint16)
    X = np.empty((T, H), np.uint16)
    pre_ = np.empty((T, 4)); post_ = np.empty((T, 4)); res = np.empty((T, 4, 4))
    z = np.empty((T, 24)) if debug else None
    r = np.empty(T) if debug else None
    rstd = np.empty(T) if debug else None
    rc = _load().oracle_pre(_p(Rp), _p(phi), _p(bias), _p(ms), _p(g), T, H,
                            *_sc(dict(hc_norm_eps=hc_norm_eps, rmsnorm_eps=rmsnorm_eps,
                                      hc_post_scale=hc_post_scale, sinkhorn_eps=sinkhorn_eps,
                                      sinkhorn_iters=sinkhorn_iters)),
                            _p(X), _p(pre_), _p(post_), _p(res), _p(z), _p(r), _p(rstd),
                            nthreads or default_threads())
    assert rc == 0
    out = dict(X=X, pre=pre_, post=post_, res=res)
    if debug:
        out.update(z=z, r=r, rstd=rstd)
    return out


def shifted_post_pre(R, Y, prev_post, prev_comb, phi, bias, mix_scales, gamma, *,
                     hc_norm_eps, rmsnorm_eps, hc_post_scale, sinkhorn_eps, sinkhorn_iters,
                     nthreads: int | None = None, debug: bool = False, want_R: bool = True):
    """The whole step.  Returns dict with R (bf16 bits), X, pre, post, res [+ z, r, rstd]."""
    R = _c(R, np.uint16); Y = _c(Y, np.uint16)
    T, _, H = R.shape
    pp = _c(prev_post, np.float32); pc = _c(prev_comb, np.float32)
    phi = _c(phi, np.float32); bias = _c(bias, np.float32)
    ms = _c(mix_scales, np.float32); g = _c(gamma, np.uint16)
    Rout = np.empty_like(R) if want_R else None
    X = np.empty((T, H), np.uint16)
    pre_ = np.empty((T, 4)); post_ = np.empty((T, 4)); res = np.empty((T, 4, 4))
    z = np.empty((T, 24)) if debug else None
    r = np.empty(T) if debug else None
    rstd = np.empty(T) if debug else None
    rc = _load().oracle_shifted_post_pre(
        _p(R), _p(Y), _p(pp), _p(pc), _p(phi), _p(bias), _p(ms), _p(g), T, H,
        *_sc(dict(hc_norm_eps=hc_norm_eps, rmsnorm_eps=rmsnorm_eps, hc_post_scale=hc_post_scale,
                  sinkhorn_eps=sinkhorn_eps, sinkhorn_iters=sinkhorn_iters)),
        _p(Rout), _p(X), _p(pre_), _p(post_), _p(res), _p(z), _p(r), _p(rstd),
        nthreads or default_threads())
    assert rc == 0
    out = dict(R=Rout, X=X, pre=pre_, post=post_, res=res)
    if debug:
        out.update(z=z, r=r, rstd=rstd)
    return out


# ---- MXFP8 quantize of the layer input (see mhc_oracle.c for the readings) ----

def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def e4m3_decode(b: int) -> float:
    return float(_load().oracle_e4m3_decode(int(b)))


def mx_scale_exp(amax: float, mode: int) -> int:
    return int(_load().oracle_mx_scale_exp(float(amax), int(mode)))


def mx_scale_offset(m: int, k: int, H: int) -> int:
    return int(_load().oracle_mx_scale_offset(int(m), int(k), int(H)))


def mx_scale_shape(T: int, H: int):
    """Padded (rows, block columns) of the 128 x 4 tile layout; bytes = rows * cols."""
    return (T + 127) // 128 * 128, (H // 32 + 3) // 4 * 4


def mxfp8_quantize(X, mode: int):
    """X: [T, H] bf16 bits.  Returns (q [T, H] uint8 E4M3 codes, scales flat uint8 in the
    tile layout, padding zero)."""
    X = _c(X, np.uint16)
    T, H = X.shape
    rows, cols = mx_scale_shape(T, H)
    q = np.zeros((T, H), np.uint8)
    sc = np.zeros(rows * cols, np.uint8)
    rc = _load().oracle_mxfp8_quantize(_p(X), T, H, int(mode), _p(q), _p(sc))
    assert rc == 0
    return q, sc


# ---- the post with an int8 layer output (x_scales) and the fused square sum ----

def post_ex(R, prev_post, prev_comb, *, Y=None, Yq=None, x_scales=None):
    """Step (1) with Y given as bf16 bits (Y) or as int8 codes Yq [T,H] with one fp32 scale per
    token (x_scales [T]).  Returns (R' [T,4,H] bf16 bits, square sum of R' per token [T] fp64)."""
    R = _c(R, np.uint16)
    T, _, H = R.shape
    pp = _c(prev_post, np.float32); pc = _c(prev_comb, np.float32)
    Yb = None if Y is None else _c(Y, np.uint16)
    Yi = None if Yq is None else _c(Yq, np.int8)
    xs = None if x_scales is None else _c(x_scales, np.float32)
    assert (Yb is None) != (Yi is None) and (Yi is None or xs is not None)
    out = np.empty_like(R)
    ss = np.empty(T)
    rc = _load().oracle_post_ex(_p(R), _p(Yb), _p(Yi), _p(xs), _p(pp), _p(pc), T, H, _p(out), _p(ss))
    assert rc == 0
    return out, ss


# ---- the first layer's pre: one (T, H) input broadcast to the 4 streams ----

def pre_broadcast(x, phi, bias, mix_scales, gamma, **kw):
    """Steps (2)-(4) on the residual made of 4 identical copies of x [T, H] (bf16 bits), the
    first layer's case ("[DSv4.1] Integrate Mega-mHC from DeepGEMM": the (T, H) broadcast input
    of mhc_pre_broadcast; the carried pre mix is None there).  Returns pre()'s dict plus
    R = the broadcast residual [T, 4, H]."""
    x = _c(x, np.uint16)
    R = np.ascontiguousarray(np.repeat(x[:, None, :], 4, axis=1))
    out = pre(R, phi, bias, mix_scales, gamma, **kw)
    out["R"] = R
    return out
