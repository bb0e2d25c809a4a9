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

forge_backward_accumulate also forms each micro-batch's input gradient
dX = dY W: with integer W as well, dX is exact and must equal the float64
product bit for bit (rounded once for a bf16 dX), on the fused pass and on
the split one; random cases hold it to |dX - dY W16| <= 1e-5 |dY| |W16|.
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


# ---------------------------------------------------------------------------
# forge_backward_accumulate: the micro-batch's dX and the accumulation in one
# pass over the tiles (or dgrad + accumulate on the split path)
# ---------------------------------------------------------------------------

def _weights(d_out, d_in, w, seed, exact):
    if exact:   # small integers: exact in bf16, so dX = dY W is exact in fp32
        return S.small_integers((d_out, d_in), -3, 3, seed, S.STREAM_W, w)
    return S.normal((d_out, d_in), 0.02, seed, S.STREAM_W, w)


def run_backward_window(mbs, W, *, path, dx_dtype="bf16"):
    """forge_backward_accumulate over every micro-batch; (G_acc, [dX_i]) on the CPU."""
    d_out, d_in = W.shape
    Wd = W.to(DEV)
    G = torch.full((d_out, d_in), float("nan"), dtype=torch.float32, device=DEV)
    flags = {"fused": F.FLAG_BACKWARD_FUSED, "split": F.FLAG_BACKWARD_SPLIT, "auto": 0}[path]
    dxs = []
    for i, (X, dY) in enumerate(mbs):
        bt = X.shape[0]
        ws = torch.empty(max(16, F.workspace_bytes(d_out, d_in, bt)), dtype=torch.uint8, device=DEV)
        dX = torch.full((bt, d_in), float("nan"), device=DEV,
                        dtype=torch.bfloat16 if dx_dtype == "bf16" else torch.float32)
        F.backward_accumulate(X.to(DEV), dY.to(DEV), Wd, G, dX, overwrite=(i == 0), workspace=ws, flags=flags)
        dxs.append(dX)
    F.sync_status()
    assert torch.equal(Wd.cpu(), W), "the weights are read only"
    return G.cpu().numpy(), [d.float().cpu().numpy() for d in dxs]


def _dx_reference(dY, W):
    w16 = O.bf16_bits_to_f32(O.f32_to_bf16_rne(W.float().numpy())).astype(np.float64)
    dYn = dY.float().numpy().astype(np.float64)
    return O.dgrad_f64(dYn, w16), np.abs(dYn) @ np.abs(w16)


@pytest.mark.parametrize("path", ["fused", "split"])
@pytest.mark.parametrize("w", ["f32", "bf16"])
@pytest.mark.parametrize("dx_dtype", ["bf16", "f32"])
def test_backward_accumulate_exact(path, w, dx_dtype):
    d_out, d_in = 384, 264
    mbs = micro_batches(d_out, d_in, TOKENS, 11, exact=True)
    W = _weights(d_out, d_in, w, 11, exact=True)
    G, dxs = run_backward_window(mbs, W, path=path, dx_dtype=dx_dtype)
    assert np.array_equal(G, O.accumulated_gradient_f64(_np(mbs)).astype(np.float32))
    for i, ((_, dY), got) in enumerate(zip(mbs, dxs)):
        ref, _ = _dx_reference(dY, W)
        want = ref.astype(np.float32) if dx_dtype == "f32" else O.bf16_bits_to_f32(O.f64_to_bf16_rne(ref))
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"micro-batch {i}: {len(bad)} dX elements differ, first {bad[:3].tolist()}"


@pytest.mark.parametrize("shape", [(136, 200), (2048, 1280)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("w", ["f32", "bf16"])
def test_backward_accumulate_random_within_tolerance(shape, w):
    d_out, d_in = shape
    mbs = micro_batches(d_out, d_in, TOKENS, 12, exact=False)
    W = _weights(d_out, d_in, w, 12, exact=False)
    G, dxs = run_backward_window(mbs, W, path="fused", dx_dtype="f32")
    ref = O.accumulated_gradient_f64(_np(mbs))
    A = sum(np.abs(d).T @ np.abs(x) for x, d in _np(mbs))
    assert np.all(np.abs(G - ref) <= 1e-5 * A)
    for i, ((_, dY), got) in enumerate(zip(mbs, dxs)):
        dref, dA = _dx_reference(dY, W)
        viol = float(np.max(np.abs(got - dref) / np.maximum(1e-5 * dA, 1e-300)))
        assert viol <= 1.0, f"micro-batch {i}: dX at {viol:.3f} of the tolerance"


def test_backward_accumulate_paths_agree():
    # Random inputs: both paths add each micro-batch's fp32 tile sums to G_acc;
    # dX sums the same products in another order.
    d_out, d_in = 1024, 768
    mbs = micro_batches(d_out, d_in, TOKENS, 13, exact=False)
    W = _weights(d_out, d_in, "f32", 13, exact=False)
    Gf, dxf = run_backward_window(mbs, W, path="fused", dx_dtype="f32")
    Gs, dxs = run_backward_window(mbs, W, path="split", dx_dtype="f32")
    A = sum(np.abs(d).T @ np.abs(x) for x, d in _np(mbs))
    assert np.all(np.abs(Gf - Gs) <= 2e-5 * A)
    for (_, dY), a, b in zip(mbs, dxf, dxs):
        _, dA = _dx_reference(dY, W)
        assert np.all(np.abs(a - b) <= 2e-5 * dA)
    # The library's own choice with a workspace: the fused pass, run to run identical.
    Ga, dxa = run_backward_window(mbs, W, path="auto", dx_dtype="f32")
    assert np.array_equal(Ga, Gf) and all(np.array_equal(a, b) for a, b in zip(dxa, dxf))


def test_backward_accumulate_window_equals_concatenated_step():
    # A whole window on the fused passes (dX of the last micro-batch by
    # forge_dgrad before the accumulated step) against one backward pass on
    # the concatenated batch: exact inputs, so both are exact.
    d_out, d_in = 256, 384
    prob = S.linear_problem(d_out, d_in, 8, seed=14, x_dtype="bf16", w_dtype="f32", state="f32")
    prob.W = _weights(d_out, d_in, "f32", 14, exact=True)
    mbs = micro_batches(d_out, d_in, TOKENS, 14, exact=True)
    W, m, v = prob.W.to(DEV), prob.m.to(DEV), prob.v.to(DEV)
    G, dxs = run_backward_window(mbs[:-1], prob.W, path="fused", dx_dtype="f32")
    G = torch.from_numpy(G).to(DEV)
    Xl, dYl = mbs[-1][0].to(DEV), mbs[-1][1].to(DEV)
    dX_last = torch.empty((Xl.shape[0], d_in), device=DEV)
    F.dgrad(dYl, W, dX_last)
    F.wgrad_step_accumulated("adamw", Xl, dYl, G, W, m, v, step=3, **_hkw("adamw"))
    F.sync_status()
    Wc, mc, vc = prob.W.to(DEV), prob.m.to(DEV), prob.v.to(DEV)
    X = torch.cat([x for x, _ in mbs]).to(DEV); dY = torch.cat([d for _, d in mbs]).to(DEV)
    dX_cat = torch.empty((X.shape[0], d_in), device=DEV)
    ws = torch.empty(F.workspace_bytes(d_out, d_in, X.shape[0]), dtype=torch.uint8, device=DEV)
    F.backward_step("adamw", X, dY, Wc, mc, vc, dX_cat, step=3, workspace=ws, flags=F.FLAG_BACKWARD_SPLIT,
                    **_hkw("adamw"))
    F.sync_status()
    assert_bit_exact(O.State(W=to_np(W), m=to_np(m), v=to_np(v)), O.State(W=to_np(Wc), m=to_np(mc), v=to_np(vc)),
                     "adamw")
    got = np.concatenate(dxs + [dX_last.cpu().numpy()])
    assert np.array_equal(got, dX_cat.cpu().numpy())


def test_backward_accumulate_long_token_axis_takes_the_split_path():
    d_out, d_in = 256, 384
    mbs = micro_batches(d_out, d_in, (800, 130), 15, exact=True)
    W = _weights(d_out, d_in, "bf16", 15, exact=True)
    G, dxs = run_backward_window(mbs, W, path="auto", dx_dtype="f32")
    assert np.array_equal(G, O.accumulated_gradient_f64(_np(mbs)).astype(np.float32))
    for (_, dY), got in zip(mbs, dxs):
        assert np.array_equal(got, _dx_reference(dY, W)[0].astype(np.float32))


def test_backward_accumulate_rejects_what_it_cannot_do():
    d_out, d_in = 128, 128
    W = torch.zeros((d_out, d_in), device=DEV)
    G = torch.zeros((d_out, d_in), device=DEV)
    X = torch.zeros((800, d_in), dtype=torch.bfloat16, device=DEV)
    dY = torch.zeros((800, d_out), dtype=torch.bfloat16, device=DEV)
    dX = torch.empty((800, d_in), device=DEV)
    with pytest.raises(F.ForgeError) as ei:            # more tokens than tensor memory holds
        F.backward_accumulate(X, dY, W, G, dX, flags=F.FLAG_BACKWARD_FUSED)
    assert ei.value.status == 2
    X, dY, dX = X[:64], dY[:64], dX[:64]
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(F.ForgeError) as ei:            # forced fused pass, workspace too small
        F.backward_accumulate(X, dY, W, G, dX, workspace=small, flags=F.FLAG_BACKWARD_FUSED)
    assert ei.value.status == 1
    F.sync_status()


def test_backward_accumulate_with_no_tokens():
    # An empty micro-batch: the first of a window sets G_acc to zero, a later
    # one leaves it as it is; dX is empty.
    d_out, d_in = 256, 384
    W = torch.zeros((d_out, d_in), device=DEV)
    G = torch.full((d_out, d_in), 3.0, device=DEV)
    X = torch.empty((0, d_in), dtype=torch.bfloat16, device=DEV)
    dY = torch.empty((0, d_out), dtype=torch.bfloat16, device=DEV)
    dX = torch.empty((0, d_in), dtype=torch.bfloat16, device=DEV)
    F.backward_accumulate(X, dY, W, G, dX, overwrite=False)
    F.sync_status()
    assert torch.all(G == 3.0)
    F.backward_accumulate(X, dY, W, G, dX, overwrite=True)
    F.sync_status()
    assert torch.all(G == 0.0)
