"""CPU oracle for the fused weight-gradient + optimizer step (FORGE).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or
executes this module: only the test-suite, the smoke check and the
benchmark's CPU-baseline leg do. It shares no code, header, table or
helper with the CUDA implementation.

What it computes. FORGE ("Fused On-Register Gradient Elimination",
arXiv 2606.22932) forms the weight gradient of a linear layer
G = dY^T X (section 2.1, Eq. 3) tile by tile (Eq. 5) and applies an
element-wise optimizer to each accumulator tile before anything is
written (Algorithm 1). Proposition 1 (Appendix A) proves that the tiled
schedule lands on exactly the weights that "materialise G, then step
once" produces. The oracle is therefore that plain definition:

  1. G = dY^T X in float64 (a library matmul of the exactly upcast inputs);
  2. the textbook optimizer step per element, in float64;
  3. the storage rule of each output (fp32 round-to-nearest-even, bf16
     round-to-nearest-even, bf16 stochastic rounding, 8-bit block codes).

A second mode, ``mode="f32emu"``, evaluates step 2 as an explicit
sequence of correctly rounded float32 operations (no fused multiply-add)
on float32 operands. It is used where a result must be bit-exact: when
the gradient is exact (integer-valued inputs) a correct implementation
of the same op sequence reproduces it bit for bit, including every
stochastic-rounding decision and every 8-bit code.

Readings of points the paper leaves open (each is also listed with the
design notes of this library):

* step t is 1-based (Algorithm 1's bias correction uses 1 - beta^t);
* SGD-momentum, which Appendix N only names ("single moment"), is the
  common library rule with coupled L2 decay, no dampening, no Nesterov:
  g~ = g + lambda W; m' = mu m + g~; W' = W - eta m';
* Lion, which Appendix N only names ("sign of momentum, single buffer"),
  follows Chen et al. 2023: c = b1 m + (1-b1) g;
  W' = (1 - eta lambda) W - eta sign(c); m' = b2 m + (1-b2) g; sign(0)=0;
* the update uses the unquantised new moments; quantisation applies to
  what is stored (Proposition 4's model, Appendix B);
* stochastic rounding (Appendix C, Proposition 5) of an fp32 value x:
  add a uniform 16-bit integer to the bit pattern of x and keep the high
  16 bits; NaN becomes a quiet NaN of the same sign;
* the random 16-bit draws come from Philox4x32-10 (Salmon et al.,
  SC'11) with key (seed lo, seed hi) and counter
  (idx/8 lo, idx/8 hi, step, site), idx = p * D_in + q the row-major
  element index, site 0 = W, 1 = m, 2 = v; element idx takes the 16 bits
  at half (idx % 2) of output word (idx % 8) / 2, low half first;
* 8-bit moments (Section 2.3 and Appendix B, block of 128 along D_in):
  first moment: s = absmax / 127, code = clamp(rint(m / s), -127, 127),
  a nonzero m never gets code 0 (it gets sign(m)); second moment:
  u = sqrt(v), s = absmax(u) / 255, code = clamp(rint(u / s), 1, 255)
  for v != 0 and 0 for v == 0; an all-zero block has scale 0. The stored
  scale is s. Dequantisation: m = code * s, v = (code * s)^2. Each code
  is round(x / s) of the stored float32 x and s, rounded exactly (ties to
  even), the paper's q(x) = s * round(x / s);
* a NaN stored as bf16 with round-to-nearest-even becomes 0x7FFF.
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

import numpy as np

F32 = np.float32
U32_MASK = np.uint64(0xFFFFFFFF)

# --------------------------------------------------------------------------
# Hyper-parameters
# --------------------------------------------------------------------------


@dataclasses.dataclass
class Hyper:
    """(eta, beta1, beta2, eps, lambda) of Algorithm 1.

    For SGD-momentum ``beta1`` is the momentum mu; Lion uses beta1 for the
    interpolation and beta2 for the moment decay.
    """

    lr: float
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    momentum_decay: float = 4e-3   # NAdam psi


# --------------------------------------------------------------------------
# Phase 1: the weight gradient (Eq. 3 / Eq. 5)
# --------------------------------------------------------------------------


def wgrad_f64(dY: np.ndarray, X: np.ndarray) -> np.ndarray:
    """G = dY^T X in float64 (Eq. 3). dY: [BT, D_out], X: [BT, D_in]."""
    return np.asarray(dY, dtype=np.float64).T @ np.asarray(X, dtype=np.float64)


def abs_wgrad_f64(dY: np.ndarray, X: np.ndarray) -> np.ndarray:
    """A = |dY|^T |X|: the magnitude every term of G is formed from.

    Used only to scale tolerances (the rounding error of any summation
    order of G is bounded by a multiple of A).
    """
    return np.abs(np.asarray(dY, dtype=np.float64)).T @ np.abs(np.asarray(X, dtype=np.float64))


# --------------------------------------------------------------------------
# Phase 2 in float64: the textbook element-wise rules
# --------------------------------------------------------------------------


def adamw_f64(W, m, v, G, h: Hyper, t: int):
    """AdamW, Algorithm 1 phase 2 (decoupled decay on the old W)."""
    assert t >= 1
    W = np.asarray(W, np.float64); m = np.asarray(m, np.float64)
    v = np.asarray(v, np.float64); G = np.asarray(G, np.float64)
    m1 = h.beta1 * m + (1.0 - h.beta1) * G
    v1 = h.beta2 * v + (1.0 - h.beta2) * G * G
    mhat = m1 / (1.0 - h.beta1 ** t)
    vhat = v1 / (1.0 - h.beta2 ** t)
    W1 = (1.0 - h.lr * h.weight_decay) * W - h.lr * mhat / (np.sqrt(vhat) + h.eps)
    return W1, m1, v1


def sgdm_f64(W, m, G, h: Hyper, t: int):
    """SGD with momentum (Appendix N (i).8; coupled L2 decay, no dampening)."""
    assert t >= 1
    W = np.asarray(W, np.float64); m = np.asarray(m, np.float64); G = np.asarray(G, np.float64)
    gt = G + h.weight_decay * W
    m1 = h.beta1 * m + gt
    W1 = W - h.lr * m1
    return W1, m1


def lion_f64(W, m, G, h: Hyper, t: int):
    """Lion (Appendix N (i).4; Chen et al. 2023), sign(0) = 0."""
    assert t >= 1
    W = np.asarray(W, np.float64); m = np.asarray(m, np.float64); G = np.asarray(G, np.float64)
    c = h.beta1 * m + (1.0 - h.beta1) * G
    sg = np.where(c > 0, 1.0, np.where(c < 0, -1.0, 0.0))
    W1 = (1.0 - h.lr * h.weight_decay) * W - h.lr * sg
    m1 = h.beta2 * m + (1.0 - h.beta2) * G
    return W1, m1


# The remaining element-wise families of Appendix N (i), read as the PyTorch
# optimizers of the same name with their defaults (coupled L2 decay
# g~ = g + lambda W; RMSprop without momentum or centring, alpha = beta2;
# AdaGrad without lr decay, initial accumulator 0). The one state tensor of
# RMSprop and AdaGrad is their second moment.


def sgd_f64(W, G, h: Hyper, t: int):
    """Plain SGD (Appendix N (i).7)."""
    W = np.asarray(W, np.float64); G = np.asarray(G, np.float64)
    return W - h.lr * (G + h.weight_decay * W)


def rmsprop_f64(W, v, G, h: Hyper, t: int):
    """RMSprop (Appendix N (i).5): second moment only."""
    W = np.asarray(W, np.float64); v = np.asarray(v, np.float64); G = np.asarray(G, np.float64)
    gt = G + h.weight_decay * W
    v1 = h.beta2 * v + (1.0 - h.beta2) * gt * gt
    return W - h.lr * gt / (np.sqrt(v1) + h.eps), v1


def adagrad_f64(W, v, G, h: Hyper, t: int):
    """AdaGrad (Appendix N (i).6): cumulative squared gradient."""
    W = np.asarray(W, np.float64); v = np.asarray(v, np.float64); G = np.asarray(G, np.float64)
    gt = G + h.weight_decay * W
    v1 = v + gt * gt
    return W - h.lr * gt / (np.sqrt(v1) + h.eps), v1


def nadam_mu(h: Hyper, i: float) -> float:
    """NAdam's momentum schedule mu_i = beta1 (1 - 0.5 * 0.96^(i psi))."""
    return h.beta1 * (1.0 - 0.5 * 0.96 ** (i * h.momentum_decay))


def nadam_f64(W, m, v, G, h: Hyper, t: int):
    """NAdam (Appendix N (i).2): Nesterov-corrected Adam."""
    W = np.asarray(W, np.float64); m = np.asarray(m, np.float64)
    v = np.asarray(v, np.float64); G = np.asarray(G, np.float64)
    gt = G + h.weight_decay * W
    m1 = h.beta1 * m + (1.0 - h.beta1) * gt
    v1 = h.beta2 * v + (1.0 - h.beta2) * gt * gt
    prod = 1.0
    for i in range(1, t + 1):
        prod *= nadam_mu(h, i)
    mu_t, mu_n = nadam_mu(h, t), nadam_mu(h, t + 1)
    denom = np.sqrt(v1 / (1.0 - h.beta2 ** t)) + h.eps
    W1 = W - h.lr * (1.0 - mu_t) / (1.0 - prod) * gt / denom - h.lr * mu_n / (1.0 - prod * mu_n) * m1 / denom
    return W1, m1, v1


def radam_rect(h: Hyper, t: int):
    """(rectified?, r_t) of RAdam at step t."""
    rho_inf = 2.0 / (1.0 - h.beta2) - 1.0
    rho_t = rho_inf - 2.0 * t * h.beta2 ** t / (1.0 - h.beta2 ** t)
    if rho_t > 5.0:
        return True, np.sqrt((rho_t - 4) * (rho_t - 2) * rho_inf / ((rho_inf - 4) * (rho_inf - 2) * rho_t))
    return False, 1.0


def radam_f64(W, m, v, G, h: Hyper, t: int):
    """RAdam (Appendix N (i).3): Adam with the variance rectification."""
    W = np.asarray(W, np.float64); m = np.asarray(m, np.float64)
    v = np.asarray(v, np.float64); G = np.asarray(G, np.float64)
    gt = G + h.weight_decay * W
    m1 = h.beta1 * m + (1.0 - h.beta1) * gt
    v1 = h.beta2 * v + (1.0 - h.beta2) * gt * gt
    mhat = m1 / (1.0 - h.beta1 ** t)
    rect, r = radam_rect(h, t)
    if rect:
        W1 = W - h.lr * mhat * r * np.sqrt(1.0 - h.beta2 ** t) / (np.sqrt(v1) + h.eps)
    else:
        W1 = W - h.lr * mhat
    return W1, m1, v1


# --------------------------------------------------------------------------
# Phase 2 as a float32 op sequence
# --------------------------------------------------------------------------


def fold_scalars(opt: str, h: Hyper, t: int) -> dict:
    """The per-step float32 scalars of each rule, folded in float64 first.

    Every scalar that does not depend on the element is computed once in
    float64 from the hyper-parameters and the step, then rounded to
    float32: 1 - beta, 1 - eta*lambda, eta / (1 - beta1^t) and
    1 / sqrt(1 - beta2^t).
    """
    if opt == "adamw":
        return dict(
            b1=F32(h.beta1), omb1=F32(1.0 - h.beta1),
            b2=F32(h.beta2), omb2=F32(1.0 - h.beta2),
            decay=F32(1.0 - h.lr * h.weight_decay),
            step_size=F32(h.lr / (1.0 - h.beta1 ** t)),
            inv_sqrt_bc2=F32(1.0 / np.sqrt(1.0 - h.beta2 ** t)),
            eps=F32(h.eps))
    if opt == "sgdm":
        return dict(mu=F32(h.beta1), wd=F32(h.weight_decay), lr=F32(h.lr))
    if opt == "lion":
        return dict(
            b1=F32(h.beta1), omb1=F32(1.0 - h.beta1),
            b2=F32(h.beta2), omb2=F32(1.0 - h.beta2),
            decay=F32(1.0 - h.lr * h.weight_decay), lr=F32(h.lr))
    if opt in ("sgd", "adagrad"):
        return dict(wd=F32(h.weight_decay), lr=F32(h.lr), eps=F32(h.eps))
    if opt == "rmsprop":
        return dict(wd=F32(h.weight_decay), lr=F32(h.lr), eps=F32(h.eps),
                    a=F32(h.beta2), oma=F32(1.0 - h.beta2))
    if opt == "nadam":
        prod = 1.0
        for i in range(1, t + 1):
            prod *= nadam_mu(h, i)
        mu_t, mu_n = nadam_mu(h, t), nadam_mu(h, t + 1)
        return dict(wd=F32(h.weight_decay), b1=F32(h.beta1), omb1=F32(1.0 - h.beta1),
                    b2=F32(h.beta2), omb2=F32(1.0 - h.beta2), eps=F32(h.eps),
                    inv_sqrt_bc2=F32(1.0 / np.sqrt(1.0 - h.beta2 ** t)),
                    c1=F32(h.lr * (1.0 - mu_t) / (1.0 - prod)),
                    c2=F32(h.lr * mu_n / (1.0 - prod * mu_n)))
    if opt == "radam":
        rect, r = radam_rect(h, t)
        bc1, bc2 = 1.0 - h.beta1 ** t, 1.0 - h.beta2 ** t
        c = h.lr * r * np.sqrt(bc2) / bc1 if rect else h.lr / bc1
        return dict(wd=F32(h.weight_decay), b1=F32(h.beta1), omb1=F32(1.0 - h.beta1),
                    b2=F32(h.beta2), omb2=F32(1.0 - h.beta2), eps=F32(h.eps), rect=rect, c=F32(c))
    raise ValueError(opt)


def _f32(a):
    a = np.asarray(a)
    assert a.dtype == np.float32, a.dtype
    return a


def adamw_f32(W, m, v, G, s: dict):
    """AdamW as the float32 sequence
    m' = b1*m + omb1*g;  v' = b2*v + omb2*(g*g);
    d  = sqrt(v')*inv_sqrt_bc2 + eps;  u = m'/d;
    W' = decay*W - step_size*u
    (each operation rounded to float32; no fused multiply-add)."""
    W, m, v, G = _f32(W), _f32(m), _f32(v), _f32(G)
    m1 = s["b1"] * m + s["omb1"] * G
    v1 = s["b2"] * v + s["omb2"] * (G * G)
    d = np.sqrt(v1) * s["inv_sqrt_bc2"] + s["eps"]
    u = m1 / d
    W1 = s["decay"] * W - s["step_size"] * u
    return W1, m1, v1


def sgdm_f32(W, m, G, s: dict):
    """SGD-momentum as g~ = g + wd*W; m' = mu*m + g~; W' = W - lr*m'."""
    W, m, G = _f32(W), _f32(m), _f32(G)
    gt = G + s["wd"] * W
    m1 = s["mu"] * m + gt
    W1 = W - s["lr"] * m1
    return W1, m1


def lion_f32(W, m, G, s: dict):
    """Lion as c = b1*m + omb1*g; W' = decay*W - lr*sign(c);
    m' = b2*m + omb2*g."""
    W, m, G = _f32(W), _f32(m), _f32(G)
    c = s["b1"] * m + s["omb1"] * G
    # sign with sign(+-0) = +0
    sg = np.where(c > 0, F32(1.0), np.where(c < 0, F32(-1.0), F32(0.0))).astype(np.float32)
    W1 = s["decay"] * W - s["lr"] * sg
    m1 = s["b2"] * m + s["omb2"] * G
    return W1, m1


def sgd_f32(W, G, s: dict):
    """g~ = g + wd*W; W' = W - lr*g~."""
    W, G = _f32(W), _f32(G)
    return W - s["lr"] * (G + s["wd"] * W)


def rmsprop_f32(W, v, G, s: dict):
    """g~ = g + wd*W; v' = a*v + (1-a)*(g~*g~); W' = W - lr*(g~/(sqrt(v') + eps))."""
    W, v, G = _f32(W), _f32(v), _f32(G)
    gt = G + s["wd"] * W
    v1 = s["a"] * v + s["oma"] * (gt * gt)
    return W - s["lr"] * (gt / (np.sqrt(v1) + s["eps"])), v1


def adagrad_f32(W, v, G, s: dict):
    """g~ = g + wd*W; v' = v + g~*g~; W' = W - lr*(g~/(sqrt(v') + eps))."""
    W, v, G = _f32(W), _f32(v), _f32(G)
    gt = G + s["wd"] * W
    v1 = v + gt * gt
    return W - s["lr"] * (gt / (np.sqrt(v1) + s["eps"])), v1


def nadam_f32(W, m, v, G, s: dict):
    """g~; m' = b1*m + (1-b1)*g~; v' = b2*v + (1-b2)*(g~*g~);
    d = sqrt(v')*inv_sqrt_bc2 + eps; W' = W - (c1*g~ + c2*m')/d."""
    W, m, v, G = _f32(W), _f32(m), _f32(v), _f32(G)
    gt = G + s["wd"] * W
    m1 = s["b1"] * m + s["omb1"] * gt
    v1 = s["b2"] * v + s["omb2"] * (gt * gt)
    d = np.sqrt(v1) * s["inv_sqrt_bc2"] + s["eps"]
    return W - (s["c1"] * gt + s["c2"] * m1) / d, m1, v1


def radam_f32(W, m, v, G, s: dict):
    """g~; m', v' as NAdam; rectified: W' = W - c*(m'/(sqrt(v') + eps)); else W' = W - c*m'."""
    W, m, v, G = _f32(W), _f32(m), _f32(v), _f32(G)
    gt = G + s["wd"] * W
    m1 = s["b1"] * m + s["omb1"] * gt
    v1 = s["b2"] * v + s["omb2"] * (gt * gt)
    if s["rect"]:
        return W - s["c"] * (m1 / (np.sqrt(v1) + s["eps"])), m1, v1
    return W - s["c"] * m1, m1, v1


# Number of state tensors per rule (RMSprop / AdaGrad: their one state is
# held in State.m).
NSTATE = {"adamw": 2, "nadam": 2, "radam": 2, "sgdm": 1, "lion": 1, "rmsprop": 1, "adagrad": 1, "sgd": 0}


# --------------------------------------------------------------------------
# Storage rules
# --------------------------------------------------------------------------


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values (exact)."""
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_rne(x) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest, ties to even; NaN -> 0x7FFF."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = np.uint64(0x7FFF)
    return r.astype(np.uint16)


def f64_to_bf16_rne(x) -> np.ndarray:
    """float64 -> bf16 bits, correctly rounded (ties to even) from the exact value.

    The bf16 grid is a subset of the float64 grid, so rounding float64 to
    the nearest bf16 is done here directly: the two neighbours of x on the
    bf16 grid are found by truncating the float32 bit pattern of a value
    that brackets x, and the nearer (ties: even mantissa) is returned.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_x = x.reshape(-1)
    flat_o = out.reshape(-1)
    # Truncation of the float32 rounding toward zero gives the bf16 value
    # below |x|; the next bf16 value above is one bf16 ulp further.
    ax = np.abs(flat_x)
    with np.errstate(over="ignore", invalid="ignore"):
        f = ax.astype(np.float32)  # RNE to float32, may round up
        # Step f down to the float32 value <= ax (round toward zero).
        fb = f.view(np.uint32).copy()
        too_big = f.astype(np.float64) > ax
        fb[too_big] -= np.uint32(1)
        lo_bits = fb & np.uint32(0xFFFF0000)          # bf16 value <= |x|
        hi_bits = lo_bits + np.uint32(0x00010000)     # next bf16 value
        lo = lo_bits.view(np.float32).astype(np.float64)
        hi = hi_bits.view(np.float32).astype(np.float64)
        d_lo = ax - lo
        d_hi = hi - ax
        pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (((lo_bits >> np.uint32(16)) & np.uint32(1)) == 1))
        mag = np.where(pick_hi, hi_bits, lo_bits) >> np.uint32(16)
    sign = np.where(np.signbit(flat_x), np.uint32(0x8000), np.uint32(0))
    res = (mag | sign).astype(np.uint32)
    nan = np.isnan(flat_x)
    res[nan] = np.uint32(0x7FFF)
    inf = np.isinf(flat_x)
    res[inf] = np.where(np.signbit(flat_x[inf]), np.uint32(0xFF80), np.uint32(0x7F80))
    flat_o[:] = res.astype(np.uint16)
    return out


def f32_to_bf16_sr(x, r16) -> np.ndarray:
    """Stochastic rounding of float32 x to bf16 (Appendix C, Proposition 5).

    bits(x) + r16 with r16 uniform in [0, 2^16), then keep the high 16
    bits: the magnitude rounds up with probability (discarded low bits) /
    2^16, so the store is unbiased for either sign. NaN -> quiet NaN.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    r = (b + (np.asarray(r16).astype(np.uint64) & np.uint64(0xFFFF))) >> np.uint64(16)
    r &= np.uint64(0xFFFF)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((b[nan] >> np.uint64(16)) | np.uint64(0x0040)) & np.uint64(0xFFFF)
    return r.astype(np.uint16)


# --------------------------------------------------------------------------
# Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11, "Parallel Random
# Numbers: As Easy as 1, 2, 3", section 5: the Philox S-box construction)
# --------------------------------------------------------------------------

PHILOX_M0 = np.uint64(0xD2511F53)   # multiplier applied to counter word 0
PHILOX_M1 = np.uint64(0xCD9E8D57)   # multiplier applied to counter word 2
PHILOX_W0 = np.uint64(0x9E3779B9)   # key schedule increment, key word 0
PHILOX_W1 = np.uint64(0xBB67AE85)   # key schedule increment, key word 1


def philox4x32_10(ctr: np.ndarray, key: Tuple[int, int]) -> np.ndarray:
    """Philox4x32 with 10 rounds. ctr: [N, 4] uint32-valued; returns [N, 4] uint32.

    One round maps (c0, c1, c2, c3) with key (k0, k1) to
    (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)),
    and the key is bumped by (W0, W1) between rounds.
    """
    c = np.asarray(ctr, dtype=np.uint64).reshape(-1, 4)
    c0, c1, c2, c3 = (c[:, i].copy() for i in range(4))
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    for rnd in range(10):
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        n0 = ((p1 >> np.uint64(32)) ^ c1 ^ k0) & U32_MASK
        n1 = p1 & U32_MASK
        n2 = ((p0 >> np.uint64(32)) ^ c3 ^ k1) & U32_MASK
        n3 = p0 & U32_MASK
        c0, c1, c2, c3 = n0, n1, n2, n3
        k0 = (k0 + PHILOX_W0) & U32_MASK
        k1 = (k1 + PHILOX_W1) & U32_MASK
    return np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32)


SITE_W, SITE_M, SITE_V = 0, 1, 2


def sr_draws(seed: int, step: int, site: int, rows: int, cols: int,
             row0: int = 0, col0: int = 0, total_cols: Optional[int] = None) -> np.ndarray:
    """The 16-bit draws r16 for a [rows, cols] block of a D_out x D_in tensor.

    Element (p, q) (global row p = row0 + i, column q = col0 + j) has
    idx = p * D_in + q; its draw is half (idx % 2) of word (idx % 8) / 2 of
    Philox4x32-10(counter = (idx/8 lo, idx/8 hi, step, site),
    key = (seed lo, seed hi)).
    """
    D_in = cols if total_cols is None else total_cols
    p = (np.arange(rows, dtype=np.uint64) + np.uint64(row0))[:, None]
    q = (np.arange(cols, dtype=np.uint64) + np.uint64(col0))[None, :]
    idx = (p * np.uint64(D_in) + q).reshape(-1)
    blk = idx >> np.uint64(3)
    # One Philox call per distinct counter value over the covered range.
    b_lo = blk.min()
    ublk = np.arange(b_lo, blk.max() + np.uint64(1), dtype=np.uint64)
    inv = (blk - b_lo).astype(np.int64)
    ctr = np.zeros((ublk.size, 4), dtype=np.uint64)
    ctr[:, 0] = ublk & U32_MASK
    ctr[:, 1] = ublk >> np.uint64(32)
    ctr[:, 2] = np.uint64(step & 0xFFFFFFFF)
    ctr[:, 3] = np.uint64(site)
    out = philox4x32_10(ctr, (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    lane = (idx & np.uint64(7)).astype(np.int64)
    word = out[inv, lane // 2].astype(np.uint32)
    r16 = (word >> (16 * (lane % 2)).astype(np.uint32)) & np.uint32(0xFFFF)
    return r16.reshape(rows, cols)


# --------------------------------------------------------------------------
# 8-bit block moments (Section 2.3, Appendix B), block = 128 along D_in
# --------------------------------------------------------------------------

QBLOCK = 128


def _blocks(a: np.ndarray) -> np.ndarray:
    rows, cols = a.shape
    assert cols % QBLOCK == 0
    return a.reshape(rows, cols // QBLOCK, QBLOCK)


def round_quotient(x, s) -> np.ndarray:
    """round(x / s) with ties to even, for float32 x and float32 s > 0.

    This is the rounding of the paper's quantiser q(x) = s * round(x / s)
    (Section 2.3; Appendix B, Proposition 4), decided on the exact quotient
    of the two float32 numbers. The quotient is formed in float64, which
    decides that rounding exactly for float32 operands with |x / s| < 2^9:

    * an exact tie x / s = k + 1/2 is representable, so the correctly
      rounded float64 quotient is that tie and ``rint`` sends it to the
      even neighbour;
    * otherwise 2x - (2k + 1) s is a nonzero multiple of the last-bit
      value of the smaller-exponent operand, which puts x / s at least
      2^-27 away from k + 1/2, far more than the float64 division's
      error of at most 2^9 * 2^-53.

    The brute-force check of this against exact rational arithmetic is in
    the oracle's pin tests.
    """
    x64 = np.asarray(x, np.float32).astype(np.float64)
    s64 = np.asarray(s, np.float32).astype(np.float64)
    return np.rint(x64 / s64)


def quant_m(m1) -> Tuple[np.ndarray, np.ndarray]:
    """First moment -> (int8 codes [rows, cols], scales [cols/128, rows]).

    s = absmax / 127 (float32 division); code = clamp(round(m / s), -127, 127)
    with round the exact ties-to-even rounding of ``round_quotient``; a
    nonzero m whose code rounds to 0 gets sign(m); a block whose scale is 0
    (all zero) gets codes 0.
    """
    m1 = _f32(m1)
    b = _blocks(m1)
    amax = np.max(np.abs(b), axis=2)                    # [rows, nb] f32
    s = (amax / F32(127.0)).astype(np.float32)
    pos = (s > 0)[:, :, None]
    q = round_quotient(b, np.where(pos, s[:, :, None], F32(1.0)))
    q = np.clip(q, -127, 127)
    bump = (b != 0) & (q == 0)
    q = np.where(bump, np.sign(b), q)
    q = np.where(pos, q, 0)
    codes = q.astype(np.int8).reshape(m1.shape)
    return codes, np.ascontiguousarray(s.T)


def quant_v(v1) -> Tuple[np.ndarray, np.ndarray]:
    """Second moment -> (uint8 codes of sqrt(v), scales [cols/128, rows]).

    u = sqrt(v) (float32); s = absmax(u) / 255; code = 0 for v == 0 and
    clamp(round(u / s), 1, 255) otherwise, with the exact ties-to-even
    rounding of ``round_quotient`` (zero code only for exact zero, which
    floors a nonzero v away from zero).
    """
    v1 = _f32(v1)
    u = np.sqrt(v1)
    b = _blocks(u)
    amax = np.max(b, axis=2)
    s = (amax / F32(255.0)).astype(np.float32)
    pos = (s > 0)[:, :, None]
    q = np.clip(round_quotient(b, np.where(pos, s[:, :, None], F32(1.0))), 1, 255)
    q = np.where(_blocks(v1) == 0, 0, q)
    q = np.where(pos, q, 0)
    codes = q.astype(np.uint8).reshape(v1.shape)
    return codes, np.ascontiguousarray(s.T)


def dequant_m(codes, scales) -> np.ndarray:
    """m = code * s in float32. scales: [cols/128, rows]."""
    c = np.asarray(codes).astype(np.float32)
    s = np.ascontiguousarray(np.asarray(scales, np.float32).T)     # [rows, nb]
    return (_blocks(c) * s[:, :, None]).reshape(c.shape).astype(np.float32)


def dequant_v(codes, scales) -> np.ndarray:
    """v = (code * s)^2 in float32 (two float32 multiplications)."""
    c = np.asarray(codes).astype(np.float32)
    s = np.ascontiguousarray(np.asarray(scales, np.float32).T)
    u = (_blocks(c) * s[:, :, None]).astype(np.float32)
    return (u * u).reshape(c.shape).astype(np.float32)


# --------------------------------------------------------------------------
# The whole step: read stored state, Phase 1, Phase 2, Phase 3
# --------------------------------------------------------------------------


@dataclasses.dataclass
class State:
    """Stored optimizer state of one linear layer.

    W: float32 values, or uint16 bf16 bit patterns when w_dtype == "bf16".
    m, v: float32 values ("f32"), uint16 bf16 bits ("bf16") or 8-bit codes
    ("q8", int8 for m and uint8 for v) with scales [D_in/128, D_out].
    """

    W: np.ndarray
    m: Optional[np.ndarray]
    v: Optional[np.ndarray] = None
    m_scale: Optional[np.ndarray] = None
    v_scale: Optional[np.ndarray] = None
    w_dtype: str = "f32"
    state: str = "f32"


def load_w(st: State) -> np.ndarray:
    return bf16_bits_to_f32(st.W) if st.w_dtype == "bf16" else _f32(st.W)


def load_m(st: State) -> np.ndarray:
    if st.state == "q8":
        return dequant_m(st.m, st.m_scale)
    return bf16_bits_to_f32(st.m) if st.state == "bf16" else _f32(st.m)


def load_v(st: State) -> np.ndarray:
    if st.state == "q8":
        return dequant_v(st.v, st.v_scale)
    return bf16_bits_to_f32(st.v) if st.state == "bf16" else _f32(st.v)


def row_draws(seed: int, t: int, site: int, shape, rows=None) -> np.ndarray:
    """The stochastic-rounding draws of a [r, c] array of whole rows: rows
    0 .. r-1 of the tensor, or the global rows ``rows`` of a tensor whose
    rows have c elements (a sample of rows of a larger layer)."""
    r, c = shape
    if rows is None:
        return sr_draws(seed, t, site, r, c)
    return np.stack([sr_draws(seed, t, site, 1, c, row0=int(p), total_cols=c)[0] for p in rows])


def _store_w(W1, st: State, mode: str, sr: bool, seed: int, t: int, rows=None):
    if st.w_dtype == "f32":
        return np.asarray(W1).astype(np.float32)
    if sr:
        w32 = np.asarray(W1).astype(np.float32)
        return f32_to_bf16_sr(w32, row_draws(seed, t, SITE_W, w32.shape, rows))
    if mode == "f64":
        return f64_to_bf16_rne(W1)
    return f32_to_bf16_rne(W1)


def _store_moment(x1, which: str, st: State, mode: str, sr: bool, seed: int, t: int, rows=None):
    """Returns (stored array, scale or None)."""
    if st.state == "f32":
        return np.asarray(x1).astype(np.float32), None
    if st.state == "bf16":
        if sr:
            x32 = np.asarray(x1).astype(np.float32)
            site = SITE_M if which == "m" else SITE_V
            return f32_to_bf16_sr(x32, row_draws(seed, t, site, x32.shape, rows)), None
        if mode == "f64":
            return f64_to_bf16_rne(x1), None
        return f32_to_bf16_rne(x1), None
    if st.state == "q8":
        x32 = np.asarray(x1).astype(np.float32)
        return quant_m(x32) if which == "m" else quant_v(x32)
    raise ValueError(st.state)


def step(opt: str, X, dY, st: State, h: Hyper, t: int, *, seed: int = 0,
         sr_w: bool = False, sr_moments: bool = False, mode: str = "f64",
         G: Optional[np.ndarray] = None, rows: Optional[np.ndarray] = None) -> State:
    """One fused step of ``opt`` ("adamw", "sgdm", "lion"); returns the new stored state.

    mode "f64": Phase 2 in float64 from the exactly upcast stored state,
    then each output rounded by its storage rule.
    mode "f32emu": G rounded to float32, Phase 2 as the float32 op
    sequence of ``adamw_f32`` / ``sgdm_f32`` / ``lion_f32``.
    ``G`` may be given to skip Phase 1 (it must equal dY^T X).
    ``rows``: when the state holds a sample of whole rows of a larger layer,
    their global row indices (the stochastic-rounding streams are keyed on
    the element's index in the whole layer).
    """
    if G is None:
        G = wgrad_f64(dY, X)
    ns = NSTATE[opt]
    W0 = load_w(st)
    m0 = load_m(st) if ns >= 1 else None
    v0 = load_v(st) if ns == 2 else None
    m1 = v1 = None
    if mode == "f64":
        if opt == "adamw":
            W1, m1, v1 = adamw_f64(W0, m0, v0, G, h, t)
        elif opt == "sgdm":
            W1, m1 = sgdm_f64(W0, m0, G, h, t)
        elif opt == "lion":
            W1, m1 = lion_f64(W0, m0, G, h, t)
        elif opt == "sgd":
            W1 = sgd_f64(W0, G, h, t)
        elif opt == "rmsprop":
            W1, m1 = rmsprop_f64(W0, m0, G, h, t)
        elif opt == "adagrad":
            W1, m1 = adagrad_f64(W0, m0, G, h, t)
        elif opt == "nadam":
            W1, m1, v1 = nadam_f64(W0, m0, v0, G, h, t)
        elif opt == "radam":
            W1, m1, v1 = radam_f64(W0, m0, v0, G, h, t)
        else:
            raise ValueError(opt)
    elif mode == "f32emu":
        s = fold_scalars(opt, h, t)
        g32 = np.asarray(G).astype(np.float32)
        if opt == "adamw":
            W1, m1, v1 = adamw_f32(W0, m0, v0, g32, s)
        elif opt == "sgdm":
            W1, m1 = sgdm_f32(W0, m0, g32, s)
        elif opt == "lion":
            W1, m1 = lion_f32(W0, m0, g32, s)
        elif opt == "sgd":
            W1 = sgd_f32(W0, g32, s)
        elif opt == "rmsprop":
            W1, m1 = rmsprop_f32(W0, m0, g32, s)
        elif opt == "adagrad":
            W1, m1 = adagrad_f32(W0, m0, g32, s)
        elif opt == "nadam":
            W1, m1, v1 = nadam_f32(W0, m0, v0, g32, s)
        elif opt == "radam":
            W1, m1, v1 = radam_f32(W0, m0, v0, g32, s)
        else:
            raise ValueError(opt)
    else:
        raise ValueError(mode)

    Wn = _store_w(W1, st, mode, sr_w, seed, t, rows)
    mn = msn = vn = vsn = None
    if m1 is not None:
        mn, msn = _store_moment(m1, "m", st, mode, sr_moments, seed, t, rows)
    if v1 is not None:
        vn, vsn = _store_moment(v1, "v", st, mode, sr_moments, seed, t, rows)
    return State(W=Wn, m=mn, v=vn, m_scale=msn, v_scale=vsn, w_dtype=st.w_dtype, state=st.state)


def step_values(opt: str, X, dY, st: State, h: Hyper, t: int, G: Optional[np.ndarray] = None):
    """Unrounded float64 outputs of Phase 2 (W', m', v') and G; for tolerances."""
    if G is None:
        G = wgrad_f64(dY, X)
    ns = NSTATE[opt]
    W0 = load_w(st)
    m0 = load_m(st) if ns >= 1 else None
    v0 = load_v(st) if ns == 2 else None
    m1 = v1 = None
    if opt == "adamw":
        W1, m1, v1 = adamw_f64(W0, m0, v0, G, h, t)
    elif opt == "sgdm":
        W1, m1 = sgdm_f64(W0, m0, G, h, t)
    elif opt == "lion":
        W1, m1 = lion_f64(W0, m0, G, h, t)
    elif opt == "sgd":
        W1 = sgd_f64(W0, G, h, t)
    elif opt == "rmsprop":
        W1, m1 = rmsprop_f64(W0, m0, G, h, t)
    elif opt == "adagrad":
        W1, m1 = adagrad_f64(W0, m0, G, h, t)
    elif opt == "nadam":
        W1, m1, v1 = nadam_f64(W0, m0, v0, G, h, t)
    else:
        W1, m1, v1 = radam_f64(W0, m0, v0, G, h, t)
    return W1, m1, v1, G


# --------------------------------------------------------------------------
# Input gradient (Remark 1): dX = dY W, read before W is overwritten
# --------------------------------------------------------------------------


def accumulated_gradient_f64(micro_batches) -> np.ndarray:
    """G = sum_i dY_i^T X_i over the micro-batches [(X_i, dY_i), ...], in
    float64 (FORGE, Appendix L: exact gradient accumulation; the micro-step
    GEMMs add into one accumulator and the step fires once, at the end)."""
    G = None
    for X, dY in micro_batches:
        g = wgrad_f64(dY, X)
        G = g if G is None else G + g
    return G


def accumulated_step(opt: str, micro_batches, st: "State", h: Hyper, t: int, **kw) -> "State":
    """The step of ``opt`` fired once on the accumulated gradient of the window
    (Appendix L); keyword arguments as for ``step``."""
    return step(opt, None, None, st, h, t, G=accumulated_gradient_f64(micro_batches), **kw)


def dgrad_f64(dY, W) -> np.ndarray:
    """dX = dY W in float64 (Remark 1, Appendix A). dY: [BT, D_out], W: [D_out, D_in]."""
    return np.asarray(dY, np.float64) @ np.asarray(W, np.float64)


def backward_step(opt: str, X, dY, st: "State", h: Hyper, t: int, **kw):
    """The layer's whole backward pass: (dX, new stored state).

    Remark 1 (Appendix A): the input gradient must be formed from the
    weights the forward pass used, so dX = dY W_old is taken from the
    stored W before the fused step overwrites it. Keyword arguments as for
    ``step``.
    """
    dX = dgrad_f64(dY, load_w(st))
    return dX, step(opt, X, dY, st, h, t, **kw)
