"""Seeded synthetic inputs for the fused weight-gradient + optimizer step.

This module only draws numbers. It holds none of the method's arithmetic
(no gradient, no optimizer rule, no rounding or quantisation rule of the
step), so that both the CUDA path and the CPU oracle can be fed from it
without sharing any of the computation they are compared on.

Every tensor is drawn from numpy's PCG64 generator keyed on
``(seed, stream_id)`` so that each tensor of a problem has its own
independent, reproducible stream. Tensors come back as torch CPU tensors
in the dtype the caller asked for; bf16 tensors are obtained by torch's
own fp32 -> bf16 cast of the fp32 draw.

Shapes follow the FORGE paper's notation (FORGE, "Fused On-Register
Gradient Elimination", section 2.1, Eq. 2-3): ``X`` is ``BT x D_in``,
``dY`` is ``BT x D_out`` and ``W`` (with its moments) is ``D_out x D_in``.
The distributions are those of the Llama-3.1-8B workloads: activations
and upstream gradients ~ N(0, 1), weights ~ N(0, 0.02), first moment
~ N(0, 1e-3), second moment = |N(0, 1e-6)| (N(0, s) has standard
deviation s).
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch

# Stream ids: one independent generator stream per tensor of a problem.
STREAM_X = 1
STREAM_DY = 2
STREAM_W = 3
STREAM_M = 4
STREAM_V = 5
STREAM_ZERO_ROWS = 6
STREAM_M_CODES = 7
STREAM_V_CODES = 8

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}

# Llama-3.1-8B linear shapes (D_out, D_in) per transformer layer.
LLAMA31_8B_LINEARS = (
    ("q_proj", 4096, 4096),
    ("k_proj", 1024, 4096),
    ("v_proj", 1024, 4096),
    ("o_proj", 4096, 4096),
    ("gate_proj", 14336, 4096),
    ("up_proj", 14336, 4096),
    ("down_proj", 4096, 14336),
)
LLAMA31_8B_LAYERS = 32


def rng(seed: int, stream_id: int) -> np.random.Generator:
    """Independent generator for tensor ``stream_id`` of problem ``seed``."""
    return np.random.Generator(np.random.PCG64([int(seed), int(stream_id)]))


def normal(shape, std: float, seed: int, stream_id: int, dtype: str = "f32") -> torch.Tensor:
    """N(0, std) draw as a CPU tensor of ``dtype`` ("f32" or "bf16")."""
    a = rng(seed, stream_id).standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(std)
    return torch.from_numpy(a).to(_TORCH_DTYPES[dtype])


def abs_normal(shape, std: float, seed: int, stream_id: int, dtype: str = "f32") -> torch.Tensor:
    """|N(0, std)| draw (the second-moment initialisation)."""
    a = rng(seed, stream_id).standard_normal(size=shape, dtype=np.float32)
    np.abs(a, out=a)
    a *= np.float32(std)
    return torch.from_numpy(a).to(_TORCH_DTYPES[dtype])


def small_integers(shape, lo: int, hi: int, seed: int, stream_id: int, dtype: str = "f32") -> torch.Tensor:
    """Integers drawn uniformly from [lo, hi], stored as ``dtype``.

    With |X|, |dY| <= 3 every product is <= 9 and every partial sum over
    fewer than 2**24 / 9 tokens is an integer exactly representable in
    fp32, so the gradient is exact in any summation order.
    """
    a = rng(seed, stream_id).integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.float32)
    return torch.from_numpy(a).to(_TORCH_DTYPES[dtype])


def zero_row_mask(d_out: int, fraction: float, seed: int) -> np.ndarray:
    """Boolean mask of ``round(fraction * d_out)`` rows chosen by a seeded permutation."""
    n_zero = int(round(fraction * d_out))
    perm = rng(seed, STREAM_ZERO_ROWS).permutation(d_out)
    mask = np.zeros(d_out, dtype=bool)
    mask[perm[:n_zero]] = True
    return mask


def q8_state(d_out: int, d_in: int, seed: int, zero_rows: Optional[np.ndarray] = None,
             m_scale: float = 3e-3 / 127.0, v_scale: float = 2e-3 / 255.0):
    """Random 8-bit block-quantised moment state.

    The codes are drawn directly (they are not produced by quantising
    anything): first-moment codes are a clipped discretised normal in
    [-127, 127], second-moment codes are uniform in [1, 255]. Every
    128-element row block gets the same scale, chosen so that the
    dequantised magnitudes are those of the fp32 initialisation
    (|m| up to ~3e-3, sqrt(v) up to ~2e-3). Rows in ``zero_rows`` get
    code 0 and scale 0 (an exactly zero moment).

    Returns (m_codes int8 [d_out, d_in], m_scales f32 [d_in/128, d_out],
             v_codes uint8 [d_out, d_in], v_scales f32 [d_in/128, d_out]).
    """
    assert d_in % 128 == 0, "8-bit block state needs D_in to be a multiple of 128"
    nb = d_in // 128
    z = rng(seed, STREAM_M_CODES).standard_normal(size=(d_out, d_in), dtype=np.float32)
    mc = np.clip(np.rint(z * np.float32(42.0)), -127, 127).astype(np.int8)
    vc = rng(seed, STREAM_V_CODES).integers(1, 256, size=(d_out, d_in), dtype=np.int64).astype(np.uint8)
    ms = np.full((nb, d_out), m_scale, dtype=np.float32)
    vs = np.full((nb, d_out), v_scale, dtype=np.float32)
    if zero_rows is not None:
        mc[zero_rows, :] = 0
        vc[zero_rows, :] = 0
        ms[:, zero_rows] = 0.0
        vs[:, zero_rows] = 0.0
    return (torch.from_numpy(mc), torch.from_numpy(ms), torch.from_numpy(vc), torch.from_numpy(vs))


@dataclasses.dataclass
class LinearProblem:
    """One linear layer's step inputs (CPU tensors)."""

    X: torch.Tensor            # [BT, D_in]
    dY: torch.Tensor           # [BT, D_out]
    W: torch.Tensor            # [D_out, D_in]
    m: Optional[torch.Tensor]  # [D_out, D_in] (f32/bf16) or int8 codes
    v: Optional[torch.Tensor]  # [D_out, D_in] (f32/bf16) or uint8 codes
    m_scale: Optional[torch.Tensor] = None  # [D_in/128, D_out] f32 (8-bit state)
    v_scale: Optional[torch.Tensor] = None
    zero_rows: Optional[np.ndarray] = None

    def tensors(self) -> Dict[str, torch.Tensor]:
        out = {"X": self.X, "dY": self.dY, "W": self.W}
        for k in ("m", "v", "m_scale", "v_scale"):
            t = getattr(self, k)
            if t is not None:
                out[k] = t
        return out


def linear_problem(d_out: int, d_in: int, bt: int, *, seed: int = 0,
                   x_dtype: str = "bf16", w_dtype: str = "f32", state: str = "f32",
                   two_moments: bool = True, exact: bool = False,
                   zero_row_fraction: float = 0.0, fresh_moments: bool = False,
                   w_bf16_representable: bool = True) -> LinearProblem:
    """Draw one linear layer's inputs and optimizer state.

    x_dtype: dtype of X and dY ("bf16" or "f32").
    w_dtype: storage of W ("f32" master or "bf16").
    state: moment storage ("f32", "bf16" or "q8").
    exact: integer-valued X, dY in [-3, 3] (exact gradient in fp32).
    zero_row_fraction: that share of W rows gets an exactly zero gradient
        (the matching dY columns are zeroed) and exactly zero moments.
    fresh_moments: m = v = 0 (a first step).
    w_bf16_representable: an fp32 master W is initialised to
        bf16-representable values (the bf16 N(0, 0.02) draw, upcast).
    """
    if exact:
        X = small_integers((bt, d_in), -3, 3, seed, STREAM_X, x_dtype)
        dY = small_integers((bt, d_out), -3, 3, seed, STREAM_DY, x_dtype)
    else:
        X = normal((bt, d_in), 1.0, seed, STREAM_X, x_dtype)
        dY = normal((bt, d_out), 1.0, seed, STREAM_DY, x_dtype)
    zero_rows = None
    if zero_row_fraction > 0.0:
        zero_rows = zero_row_mask(d_out, zero_row_fraction, seed)
        dY[:, torch.from_numpy(zero_rows)] = 0

    if w_dtype == "bf16" or w_bf16_representable:
        W = normal((d_out, d_in), 0.02, seed, STREAM_W, "bf16")
        if w_dtype == "f32":
            W = W.to(torch.float32)
    else:
        W = normal((d_out, d_in), 0.02, seed, STREAM_W, "f32")

    m = v = ms = vs = None
    if state == "q8":
        m, ms, v, vs = q8_state(d_out, d_in, seed, zero_rows)
        if fresh_moments:
            m.zero_(); v.zero_(); ms.zero_(); vs.zero_()
        if not two_moments:
            v = vs = None
    else:
        if fresh_moments:
            m = torch.zeros((d_out, d_in), dtype=_TORCH_DTYPES[state])
            v = torch.zeros((d_out, d_in), dtype=_TORCH_DTYPES[state])
        else:
            m = normal((d_out, d_in), 1e-3, seed, STREAM_M, state)
            v = abs_normal((d_out, d_in), 1e-6, seed, STREAM_V, state)
        if zero_rows is not None:
            zr = torch.from_numpy(zero_rows)
            m[zr, :] = 0
            v[zr, :] = 0
        if not two_moments:
            v = None
    return LinearProblem(X=X, dY=dY, W=W, m=m, v=v, m_scale=ms, v_scale=vs, zero_rows=zero_rows)


def step_inputs(d_out: int, d_in: int, bt: int, seed: int, step: int, x_dtype: str = "f32"):
    """Fresh (X, dY) for step ``step`` of a multi-step run.

    Each step draws its own activations and upstream gradients from the
    streams keyed on (seed, step, tensor).
    """
    X = normal((bt, d_in), 1.0, seed * 1000003 + step, STREAM_X, x_dtype)
    dY = normal((bt, d_out), 1.0, seed * 1000003 + step, STREAM_DY, x_dtype)
    return X, dY


def device_normal_(t: torch.Tensor, std: float, seed: int, stream_id: int, absolute: bool = False) -> torch.Tensor:
    """Fill a device tensor with N(0, std) (or |N(0, std)|) from torch's seeded
    device generator keyed on (seed, stream_id). Used where host generation
    would be too slow (the 7-billion-parameter linear stack)."""
    g = torch.Generator(device=t.device)
    g.manual_seed(int(seed) * 1000003 + int(stream_id))
    if t.dtype == torch.float32:
        t.normal_(0.0, std, generator=g)
    else:
        tmp = torch.empty(t.shape, dtype=torch.float32, device=t.device)
        tmp.normal_(0.0, std, generator=g)
        t.copy_(tmp)
    if absolute:
        t.abs_()
    return t
