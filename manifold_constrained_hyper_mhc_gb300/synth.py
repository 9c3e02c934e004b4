"""Seeded synthetic inputs for the fused mHC post+pre step.

This module only draws random numbers and packs them into the buffers the op
consumes.  It holds none of the op's arithmetic (no post mix, no RMS, no
projection, no sigmoid heads, no Sinkhorn, no RMSNorm), so that both the CUDA
path and the CPU oracle can be fed from it without sharing any computation.

Shapes follow the interface of the Mega-mHC integration ("[DSv4.1] Integrate
Mega-mHC from DeepGEMM", review section "Verified OK": hc_mult = 4 streams,
fp32 mixes of shape [T, hc]); the flattened residual row is [hc_mult * H]
(same page, "Paths on current main that still call DeepGEMM on SM12x", item 1:
x.shape[1] == hc_mult * hidden_size).

Layouts (all row-major, contiguous):
  residual      R        [T, 4, H]   bf16 bits (uint16)
  layer output  Y        [T, H]      bf16 bits
  prev post mix          [T, 4]      fp32
  prev comb_res_mix      [T, 4, 4]   fp32, entry [j, i] weights stream j into i
  phi                    [4H, 24]    fp32
  bias                   [24]        fp32
  mix_scales             [3]         fp32 (alpha_pre, alpha_post, alpha_res)
  rmsnorm weight gamma   [H]         bf16 bits

Tokens are drawn in blocks of ``BLOCK`` tokens, each from its own generator
seeded with (seed, 1, block index), so any token range can be regenerated on
its own (sampled parity checks at full size need this).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
from dataclasses import dataclass, field

import numpy as np

BLOCK = 256
HC = 4
NMIX = 24  # 4 pre + 4 post + 16 residual-mix logits

# The scalar tail used by every workload.  The four values are pairwise
# distinct so that an argument-order swap anywhere shows up as a mismatch
# ("[DSv4.1] Integrate Mega-mHC from DeepGEMM", "Verified OK", item 1).
HC_NORM_EPS = 2e-5
RMSNORM_EPS = 2e-6
SINKHORN_EPS = 3e-4
HC_POST_SCALE = 1.25
SINKHORN_ITERS = 20
MIX_SCALES = (0.01, 0.01, 0.01)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    seed: int
    token_scale: bool = False      # per-token residual scale 10**U(-2, 2)
    special_tokens: bool = False   # 1% zero-Y tokens, 1% identical-stream tokens
    note: str = field(default="", compare=False)


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny", 6, 1024, 0, note="tiny post+pre, T=6 H=1024"),
        Workload("decode_verify", 6, 7168, 1,
                 note="BS=1 speculative verify block of 5 tokens plus 1"),
        Workload("mid_batch", 128, 4096, 2, token_scale=True,
                 note="mid-batch decode, residual scale spread over 4 decades"),
        Workload("prefill_chunk", 8192, 7168, 3, note="prefill chunk"),
        Workload("long_prefill", 65536, 7168, 4, special_tokens=True,
                 note="long prefill with 1% zero-Y and 1% identical-stream tokens"),
    )
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); returns uint16 bits.

    Random draws are finite, so no NaN handling is needed here.
    """
    u = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    u += (u >> np.uint32(16)) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# The previous layer's residual mixes: 1024 seeded matrices, each the 20-iteration Sinkhorn
# normalisation of exp(N(0, 0.5)) as the workload definition states, written once by
# tests/golden/make_prev_comb_table.py (with the CPU oracle's Sinkhorn, so that no arithmetic of
# the op lives here); every token takes one of them by a seeded index.
_PREV_COMB_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tests", "golden",
                               "prev_comb_sinkhorn20.npy")
_prev_comb_table = None


def prev_comb_table() -> np.ndarray:
    global _prev_comb_table
    if _prev_comb_table is None:
        _prev_comb_table = np.load(_PREV_COMB_PATH)
    return _prev_comb_table


def weights(w: Workload):
    """phi [4H,24] f32, bias [24] f32, mix_scales [3] f32, gamma [H] bf16 bits."""
    rng = np.random.default_rng([w.seed, 0])
    phi = rng.standard_normal((HC * w.H, NMIX), dtype=np.float32) * np.float32(0.02)
    bias = rng.standard_normal(NMIX, dtype=np.float32) * np.float32(0.1)
    gamma = f32_to_bf16_bits(1.0 + 0.1 * rng.standard_normal(w.H, dtype=np.float32))
    mix_scales = np.array(MIX_SCALES, dtype=np.float32)
    return phi, bias, mix_scales, gamma


def _block(w: Workload, b: int):
    """All inputs of token block b (tokens [b*BLOCK, min(T, (b+1)*BLOCK)))."""
    t0 = b * BLOCK
    n = min(w.T, t0 + BLOCK) - t0
    rng = np.random.default_rng([w.seed, 1, b])
    R = rng.standard_normal((n, HC, w.H), dtype=np.float32)
    Y = rng.standard_normal((n, w.H), dtype=np.float32)
    # prev post mix: 2 * logistic(N(0,1)), i.e. a scaled logit-normal draw
    prev_post = (2.0 / (1.0 + np.exp(-rng.standard_normal((n, HC))))).astype(np.float32)
    prev_comb = prev_comb_table()[rng.integers(0, len(prev_comb_table()), size=n)]
    if w.token_scale:
        s = (10.0 ** rng.uniform(-2.0, 2.0, size=n)).astype(np.float32)
        R *= s[:, None, None]
    if w.special_tokens:
        t = np.arange(t0, t0 + n)
        Y[t % 100 == 0] = 0.0
        same = t % 100 == 50
        R[same, 1:, :] = R[same, :1, :]
    return f32_to_bf16_bits(R), f32_to_bf16_bits(Y), prev_post, prev_comb


def tokens(w: Workload, t0: int = 0, t1: int | None = None):
    """R [n,4,H] u16, Y [n,H] u16, prev_post [n,4] f32, prev_comb [n,4,4] f32 for tokens [t0,t1)."""
    t1 = w.T if t1 is None else t1
    assert 0 <= t0 <= t1 <= w.T
    n = t1 - t0
    R = np.empty((n, HC, w.H), np.uint16)
    Y = np.empty((n, w.H), np.uint16)
    post = np.empty((n, HC), np.float32)
    comb = np.empty((n, HC, HC), np.float32)

    def fill(b):
        Rb, Yb, pb, cb = _block(w, b)
        lo = max(t0, b * BLOCK)
        hi = min(t1, b * BLOCK + len(Yb))
        s = slice(lo - b * BLOCK, hi - b * BLOCK)
        d = slice(lo - t0, hi - t0)
        R[d], Y[d], post[d], comb[d] = Rb[s], Yb[s], pb[s], cb[s]

    blocks = range(t0 // BLOCK, (t1 + BLOCK - 1) // BLOCK) if n else range(0)
    # numpy's generators release the GIL while filling, so blocks run in parallel
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(blocks), os.cpu_count() or 1))) as ex:
        list(ex.map(fill, blocks))
    return R, Y, post, comb


CANCEL_KINDS = ("exact", "mild", "severe", "partial", "independent")


def cancellation_case(T: int, H: int, seed: int):
    """Inputs whose streams cancel in the combined row X = sum_i pre_i R'_i (an adversarial case
    for any shortcut that forms sum_h X^2 from per-stream sums).

    The previous mixes are the identity residual mix and a zero post mix, so R' = R exactly.
    phi's logit columns 1 and 3 repeat columns 0 and 2, and the matching biases repeat too,
    so pre_1 = pre_0 and pre_3 = pre_2 whatever the streams are.  Token t of kind
    CANCEL_KINDS[t % 5], with A, B ~ N(0,1) * 10**U(0, 2) per token and d ~ N(0, s^2):
      exact       R = [A, -A, B, -B]                 (X is zero up to rounding)
      mild        R = [A, -A + d, B, -B + d'], s = 2^-6 |scale|
      severe      R = [A, -A + d, B, -B + d'], s = 2^-10 |scale|
      partial     R = [A, -A + d, B, C],       s = 2^-10 |scale|, C ~ N(0,1) * scale
      independent R = [A, B, C, D]
    Returns (R, Y, prev_post, prev_comb, phi, bias, mix_scales, gamma) like tokens() and
    weights()."""
    rng = np.random.default_rng([seed, 7])
    phi = rng.standard_normal((HC * H, NMIX), dtype=np.float32) * np.float32(0.02)
    phi[:, 1] = phi[:, 0]
    phi[:, 3] = phi[:, 2]
    bias = rng.standard_normal(NMIX, dtype=np.float32) * np.float32(0.1)
    bias[1] = bias[0]
    bias[3] = bias[2]
    gamma = f32_to_bf16_bits(1.0 + 0.1 * rng.standard_normal(H, dtype=np.float32))
    mix_scales = np.array(MIX_SCALES, dtype=np.float32)
    scale = (10.0 ** rng.uniform(0.0, 2.0, size=T)).astype(np.float32)
    Z = rng.standard_normal((T, HC, H), dtype=np.float32) * scale[:, None, None]
    D = rng.standard_normal((T, 2, H), dtype=np.float32) * scale[:, None, None]
    R = Z.copy()
    kind = np.arange(T) % len(CANCEL_KINDS)
    for k, name in enumerate(CANCEL_KINDS):
        m = kind == k
        if name == "exact":
            R[m, 1] = -Z[m, 0]
            R[m, 3] = -Z[m, 2]
        elif name in ("mild", "severe"):
            s_ = np.float32(2.0 ** -6 if name == "mild" else 2.0 ** -10)
            R[m, 1] = -Z[m, 0] + s_ * D[m, 0]
            R[m, 3] = -Z[m, 2] + s_ * D[m, 1]
        elif name == "partial":
            R[m, 1] = -Z[m, 0] + np.float32(2.0 ** -10) * D[m, 0]
    Y = f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    prev_post = np.zeros((T, HC), np.float32)
    prev_comb = np.broadcast_to(np.eye(HC, dtype=np.float32), (T, HC, HC)).copy()
    return f32_to_bf16_bits(R), Y, prev_post, prev_comb, phi, bias, mix_scales, gamma


def scalars():
    return dict(hc_norm_eps=HC_NORM_EPS, rmsnorm_eps=RMSNORM_EPS,
                hc_post_scale=HC_POST_SCALE, sinkhorn_eps=SINKHORN_EPS,
                sinkhorn_iters=SINKHORN_ITERS)
