"""Element-wise tolerances for comparing a GPU step with the float64 oracle.

TEST INFRASTRUCTURE ONLY (see oracle/forge_oracle.py).

Corollary 1 of the FORGE paper (Appendix A) says the fused step differs
from "materialise G, then step" only through the summation order of G,
plus the float32 rounding of the element-wise update. The float32 sum of
BT exact products differs from the exact G by a multiple of
A = |dY|^T |X| (not of |G|: cancellation makes |G| much smaller than A),
and each float32 operation of the update adds a relative 2^-24.

The tolerance of an output x is therefore "how far x moves when every
input of the step is perturbed by a relative rtol", with the gradient's
perturbation taken as rtol * A:

  |x_gpu - x_ref| <= tol_x = rtol * (|x_ref| + sum_i |dx/d in_i| * scale_i)

computed here in float64, with the non-smooth pieces (the square root
near v = 0, Lion's sign near c = 0) bounded by explicit evaluation at the
perturbed corners instead of derivatives. rtol = 1e-5 is the bound the
fp32 path is held to; the measured worst case is reported beside it.
"""

from __future__ import annotations

import numpy as np

from .forge_oracle import Hyper


def _u_adamw(m1, v1, h: Hyper, t: int):
    return (m1 / (1.0 - h.beta1 ** t)) / (np.sqrt(np.maximum(v1, 0.0) / (1.0 - h.beta2 ** t)) + h.eps)


def adamw_tol(W, m, v, G, A, h: Hyper, t: int, rtol: float = 1e-5):
    """(tol_W, tol_m, tol_v) for one AdamW step from stored (W, m, v)."""
    W = np.asarray(W, np.float64); m = np.asarray(m, np.float64); v = np.asarray(v, np.float64)
    G = np.asarray(G, np.float64); A = np.asarray(A, np.float64)
    b1, b2 = h.beta1, h.beta2
    m1 = b1 * m + (1 - b1) * G
    v1 = b2 * v + (1 - b2) * G * G
    dG = rtol * A
    sm = rtol * (np.abs(m1) + b1 * np.abs(m)) + (1 - b1) * dG
    sv = rtol * (np.abs(v1) + b2 * np.abs(v)) + (1 - b2) * (2 * np.abs(G) * dG + dG * dG)
    u0 = _u_adamw(m1, v1, h, t)
    du = np.zeros_like(u0)
    for sgm in (-1.0, 1.0):
        for sgv in (-1.0, 1.0):
            du = np.maximum(du, np.abs(_u_adamw(m1 + sgm * sm, v1 + sgv * sv, h, t) - u0))
    du += rtol * np.abs(u0)
    decay = 1 - h.lr * h.weight_decay
    W1 = decay * W - h.lr * u0
    tw = rtol * (np.abs(W1) + abs(decay) * np.abs(W) + h.lr * np.abs(u0)) + h.lr * du
    return tw, sm, sv


def sgdm_tol(W, m, G, A, h: Hyper, t: int, rtol: float = 1e-5):
    W = np.asarray(W, np.float64); m = np.asarray(m, np.float64)
    G = np.asarray(G, np.float64); A = np.asarray(A, np.float64)
    gt = G + h.weight_decay * W
    m1 = h.beta1 * m + gt
    sm = rtol * (np.abs(m1) + h.beta1 * np.abs(m) + A + abs(h.weight_decay) * np.abs(W))
    W1 = W - h.lr * m1
    tw = rtol * (np.abs(W1) + np.abs(W)) + h.lr * sm
    return tw, sm


def lion_tol(W, m, G, A, h: Hyper, t: int, rtol: float = 1e-5):
    W = np.asarray(W, np.float64); m = np.asarray(m, np.float64)
    G = np.asarray(G, np.float64); A = np.asarray(A, np.float64)
    c = h.beta1 * m + (1 - h.beta1) * G
    sc = rtol * (np.abs(c) + h.beta1 * np.abs(m)) + (1 - h.beta1) * rtol * A
    undetermined = np.abs(c) <= sc          # sign(c) may legitimately differ
    decay = 1 - h.lr * h.weight_decay
    W1 = decay * W - h.lr * np.sign(c)
    tw = rtol * (np.abs(W1) + abs(decay) * np.abs(W) + h.lr) + np.where(undetermined, 2 * h.lr, 0.0)
    m1 = h.beta2 * m + (1 - h.beta2) * G
    sm = rtol * (np.abs(m1) + h.beta2 * np.abs(m)) + (1 - h.beta2) * rtol * A
    return tw, sm


def rel_violation(x_gpu, x_ref, tol):
    """max |x_gpu - x_ref| / tol (<= 1 passes)."""
    d = np.abs(np.asarray(x_gpu, np.float64) - np.asarray(x_ref, np.float64))
    return float(np.max(d / np.maximum(tol, 1e-300))) if d.size else 0.0


def bf16_ulp(x_bits: np.ndarray) -> np.ndarray:
    """Spacing of the bf16 grid at each bf16 value (for ulp distances)."""
    e = (np.asarray(x_bits).astype(np.int64) >> 7) & 0xFF
    return np.ldexp(1.0, np.maximum(e, 1) - 127 - 7)


def bf16_ulp_distance(a_bits, b_bits) -> np.ndarray:
    """Distance in bf16 ulps between two bf16 bit arrays of the same sign class."""
    def key(b):
        b = np.asarray(b).astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(key(a_bits) - key(b_bits))


def generic_tol(opt: str, W, s0, s1, G, A, h: Hyper, t: int, rtol: float = 1e-5):
    """Tolerances (W', s0', s1') of any element-wise rule by explicit perturbation.

    Every input of the step is moved by a relative rtol (the gradient by
    rtol * A) at each of the 16 sign corners; the tolerance of an output is
    its largest move plus rtol of its own magnitude. The rules are
    element-wise, so all elements are perturbed at once.
    """
    from . import forge_oracle as O

    def run(Wp, a, b, Gp):
        if opt == "adamw":
            return O.adamw_f64(Wp, a, b, Gp, h, t)
        if opt == "sgdm":
            return (*O.sgdm_f64(Wp, a, Gp, h, t), None)
        if opt == "lion":
            return (*O.lion_f64(Wp, a, Gp, h, t), None)
        if opt == "sgd":
            return O.sgd_f64(Wp, Gp, h, t), None, None
        if opt == "rmsprop":
            return (*O.rmsprop_f64(Wp, a, Gp, h, t), None)
        if opt == "adagrad":
            return (*O.adagrad_f64(Wp, a, Gp, h, t), None)
        if opt == "nadam":
            return O.nadam_f64(Wp, a, b, Gp, h, t)
        return O.radam_f64(Wp, a, b, Gp, h, t)

    W = np.asarray(W, np.float64); G = np.asarray(G, np.float64); A = np.asarray(A, np.float64)
    z = np.zeros_like(W)
    s0 = z if s0 is None else np.asarray(s0, np.float64)
    s1 = z if s1 is None else np.asarray(s1, np.float64)
    base = run(W, s0, s1, G)
    dev = [np.zeros_like(W) if x is not None else None for x in base]
    for sw in (-1, 1):
        for sa in (-1, 1):
            for sb in (-1, 1):
                for sg in (-1, 1):
                    out = run(W * (1 + sw * rtol), s0 * (1 + sa * rtol), s1 * (1 + sb * rtol), G + sg * rtol * A)
                    for i, (o, b) in enumerate(zip(out, base)):
                        if o is not None:
                            dev[i] = np.maximum(dev[i], np.abs(o - b))
    return tuple(None if d is None else d + rtol * np.abs(b) for d, b in zip(dev, base))
