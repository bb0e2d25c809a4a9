"""GPU parity of exact gradient accumulation (FORGE, Appendix L): the
micro-batch GEMMs add into an fp32 accumulator G_acc (forge_wgrad_accumulate)
and the fused step fires once, at the last micro-batch, on G_acc + that
micro-batch's tiles (forge_wgrad_step_accumulated).

Exact cases use integer-valued X, dY (every partial gradient and every
running sum is an integer well inside fp32's exact range), so the
accumulator must equal the float64 sum and the final state must match the
oracle's float32 op-sequence mode bit for bit -- and equal, bit for bit, one
fused step on the concatenated batch. Random cases hold the final state to
the element-wise tolerance of oracle/tolerance.py with |dY|^T |X| summed over
the micro-batches.
"""

import numpy as np
import pytest
import torch

import backward_gemm_optimizer_gb300 as F
from backward_gemm_optimizer_gb300 import synthetic as S
import oracle.forge_oracle as O

from forge_cases import HYPER, NSTATE, assert_bit_exact, check_tolerance, oracle_state, state_tensors, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
RULES = ["adamw", "sgdm", "lion", "sgd", "rmsprop", "adagrad", "nadam", "radam"]
VARIANTS = [("f32", "f32"), ("f32", "bf16"), ("bf16", "bf16"), ("bf16", "f32")]
TOKENS = (200, 70, 129)  # micro-batch sizes: ragged token tails


def _hkw(rule):
    hp = dict(HYPER[rule])
    return dict(lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"], weight_decay=hp["weight_decay"],
                momentum_decay=hp.get("momentum_decay", 4e-3))


def micro_batches(d_out, d_in, tokens, seed, exact):
    """[(X_i, dY_i)] bf16 CPU tensors, one independent draw per micro-batch."""
    out = []
    for i, n in enumerate(tokens):
        s = seed * 1000 + i
        if exact:
            out.append((S.small_integers((n, d_in), -3, 3, s, S.STREAM_X, "bf16"),
                        S.small_integers((n, d_out), -3, 3, s, S.STREAM_DY, "bf16")))
        else:
            out.append((S.normal((n, d_in), 1.0, s, S.STREAM_X, "bf16"), S.normal((n, d_out), 1.0, s, S.STREAM_DY, "bf16")))
    return out


def run_accumulated(rule, prob, mbs, t, *, seed=0, sr_w=False, sr_moments=False, last_empty=False):
    """Accumulate every micro-batch but the last, then the accumulated step with the last."""
    d_out, d_in = prob.W.shape
    W = prob.W.to(DEV)
    s0, s1 = state_tensors(rule, prob)
    s0 = s0.to(DEV) if s0 is not None else None
    s1 = s1.to(DEV) if s1 is not None else None
    G = torch.full((d_out, d_in), float("nan"), dtype=torch.float32, device=DEV)   # overwritten by the first
    body = mbs if last_empty else mbs[:-1]
    for i, (X, dY) in enumerate(body):
        F.wgrad_accumulate(X.to(DEV), dY.to(DEV), G, overwrite=(i == 0))
    if last_empty:
        Xl = torch.empty((0, d_in), dtype=torch.bfloat16, device=DEV)
        dYl = torch.empty((0, d_out), dtype=torch.bfloat16, device=DEV)
    else:
        Xl, dYl = mbs[-1][0].to(DEV), mbs[-1][1].to(DEV)
    G_before = G.clone()
    F.wgrad_step_accumulated(rule, Xl, dYl, G, W, s0, s1, step=t, seed=seed, sr_w=sr_w, sr_moments=sr_moments,
                             **_hkw(rule))
    F.sync_status()
    assert torch.equal(G, G_before), "the accumulated step must not write G_acc"
    return O.State(W=to_np(W), m=to_np(s0) if s0 is not None else None, v=to_np(s1) if s1 is not None else None)


def _np(mbs):
    return [(x.float().numpy().astype(np.float64), d.float().numpy().astype(np.float64)) for x, d in mbs]


def test_accumulator_equals_the_exact_sum():
    d_out, d_in = 384, 264
    mbs = micro_batches(d_out, d_in, TOKENS, 1, exact=True)
    G = torch.empty((d_out, d_in), dtype=torch.float32, device=DEV)
    for k in range(len(mbs)):
        F.wgrad_accumulate(mbs[k][0].to(DEV), mbs[k][1].to(DEV), G, overwrite=(k == 0))
        F.sync_status()
        ref = O.accumulated_gradient_f64(_np(mbs[:k + 1]))
        assert np.array_equal(G.cpu().numpy(), ref.astype(np.float32)), f"after micro-batch {k}"


@pytest.mark.parametrize("shape", [(136, 200), (2048, 1280)], ids=lambda s: "x".join(map(str, s)))
def test_accumulator_random_inputs_within_tolerance(shape):
    d_out, d_in = shape
    mbs = micro_batches(d_out, d_in, TOKENS, 2, exact=False)
    G = torch.empty((d_out, d_in), dtype=torch.float32, device=DEV)
    for k, (X, dY) in enumerate(mbs):
        F.wgrad_accumulate(X.to(DEV), dY.to(DEV), G, overwrite=(k == 0))
    F.sync_status()
    ref = O.accumulated_gradient_f64(_np(mbs))
    A = sum(np.abs(d).T @ np.abs(x) for x, d in _np(mbs))
    # fp32 sums inside each tile, plus one rounding per micro-batch
    assert np.all(np.abs(G.cpu().numpy() - ref) <= 1e-5 * A)


@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: f"W{v[0]}-m{v[1]}")
def test_accumulated_step_exact(rule, variant):
    w, st = variant
    d_out, d_in = 256, 384
    prob = S.linear_problem(d_out, d_in, 8, seed=3, x_dtype="bf16", w_dtype=w, state=st)
    mbs = micro_batches(d_out, d_in, TOKENS, 3, exact=True)
    sr, srm = w == "bf16", st == "bf16" and NSTATE[rule] > 0
    for t in (1, 5):
        got = run_accumulated(rule, prob, mbs, t, seed=99, sr_w=sr, sr_moments=srm)
        ref = O.accumulated_step(rule, _np(mbs), oracle_state(prob, w, st, rule), O.Hyper(**HYPER[rule]), t,
                                 seed=99, sr_w=sr, sr_moments=srm, mode="f32emu")
        assert_bit_exact(got, ref, rule)


@pytest.mark.parametrize("shape", [(256, 384), (2048, 1280)], ids=lambda s: "x".join(map(str, s)))
def test_accumulated_step_equals_the_concatenated_batch(shape):
    # Appendix L: identical to one step on the whole effective batch (exact
    # inputs, so no summation-order difference is possible).
    d_out, d_in = shape
    prob = S.linear_problem(d_out, d_in, 8, seed=4, x_dtype="bf16", w_dtype="f32", state="f32")
    mbs = micro_batches(d_out, d_in, TOKENS, 4, exact=True)
    a = run_accumulated("adamw", prob, mbs, 2)
    X = torch.cat([x for x, _ in mbs]).to(DEV); dY = torch.cat([d for _, d in mbs]).to(DEV)
    W, m, v = prob.W.to(DEV), prob.m.to(DEV), prob.v.to(DEV)
    F.wgrad_step_adamw(X, dY, W, m, v, step=2, **HYPER["adamw"])
    F.sync_status()
    assert_bit_exact(a, O.State(W=to_np(W), m=to_np(m), v=to_np(v)), "adamw")


@pytest.mark.parametrize("rule", ["adamw", "lion", "nadam"])
def test_accumulated_step_random_within_tolerance(rule):
    d_out, d_in = 512, 640
    prob = S.linear_problem(d_out, d_in, 8, seed=5, x_dtype="bf16", w_dtype="f32", state="f32",
                            w_bf16_representable=False)
    mbs = micro_batches(d_out, d_in, TOKENS, 5, exact=False)
    got = run_accumulated(rule, prob, mbs, 3)
    # check_tolerance takes one (X, dY): the concatenated batch has the same G
    # and the same |dY|^T |X|.
    cat = S.LinearProblem(**{**prob.__dict__, "X": torch.cat([x for x, _ in mbs]),
                             "dY": torch.cat([d for _, d in mbs])})
    check_tolerance(rule, cat, "f32", "f32", 3, got)


def test_accumulated_step_with_an_empty_last_micro_batch():
    d_out, d_in = 256, 384
    prob = S.linear_problem(d_out, d_in, 8, seed=6, x_dtype="bf16", w_dtype="f32", state="f32")
    mbs = micro_batches(d_out, d_in, TOKENS, 6, exact=True)
    got = run_accumulated("adamw", prob, mbs, 1, last_empty=True)
    ref = O.accumulated_step("adamw", _np(mbs), oracle_state(prob, "f32", "f32"), O.Hyper(**HYPER["adamw"]), 1,
                             mode="f32emu")
    assert_bit_exact(got, ref, "adamw")


def test_accumulation_rejects_what_it_does_not_support():
    d_out, d_in = 128, 128
    X = torch.zeros((16, d_in), dtype=torch.bfloat16, device=DEV)
    dY = torch.zeros((16, d_out), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(F.ForgeError) as ei:           # the accumulator is fp32
        F.wgrad_accumulate(X, dY, torch.zeros((d_out, d_in), dtype=torch.bfloat16, device=DEV))
    assert ei.value.status == 2
    with pytest.raises(F.ForgeError) as ei:           # fp32 inputs: tensor-core path only
        F.wgrad_accumulate(X.float(), dY.float(), torch.zeros((d_out, d_in), device=DEV))
    assert ei.value.status == 2
    prob = S.linear_problem(d_out, d_in, 16, seed=7, x_dtype="bf16", w_dtype="f32", state="q8")
    G = torch.zeros((d_out, d_in), device=DEV)
    import ctypes
    from backward_gemm_optimizer_gb300 import _lib
    tX, tdY, tG, tW = (F.tensor_desc(t) for t in (X, dY, G, prob.W.to(DEV)))
    m, ms = prob.m.to(DEV), prob.m_scale.to(DEV)
    v, vs = prob.v.to(DEV), prob.v_scale.to(DEV)
    tm, tv = F.tensor_desc(m, ms), F.tensor_desc(v, vs)
    h = _lib._hyper(1e-3, 0.9, 0.999, 1e-8, 0.0, False, False, 0)
    st = F.lib().forge_wgrad_step_accumulated(0, ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tG),
                                              ctypes.byref(tW), ctypes.byref(tm), ctypes.byref(tv), ctypes.byref(h),
                                              1, 0, _lib._stream(None))
    assert st == 2                                     # no 8-bit state variant
    F.sync_status()
